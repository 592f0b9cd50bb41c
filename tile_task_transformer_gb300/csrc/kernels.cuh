// Launchers of the memory-bound tile kernels (implemented in kernels.cu).
//
// Each launcher enqueues on `st` and returns NNT_OK, INVALID_ARG for sizes the
// kernel does not support, or CUDA if the launch failed. Row-wise kernels work
// on a contiguous block of rows; the tile executor passes one token tile at a
// time, the stand-alone op API passes the whole matrix.
#pragma once
#include "common.cuh"

namespace nnt {

// ---- embedding (review page "What carries the argument": embedding tile tasks)
nnt_status launch_embedding_fwd(const uint16_t* ids, int64_t ids_stride, const float* wte,
                                const float* wpe, float* x, int d, int vocab, TokMap tm, int b0,
                                int nb, int s0, int ns, cudaStream_t st);
// Tokens per batch*seq window the embedding backward handles, and the block
// of consecutive tokens one CTA of the token sort orders in shared memory.
constexpr int kMaxTokens = 1 << 20;
constexpr int kTokenSortBlock = 16384;
// Sort keys of the T = B*S tokens, T <= kMaxTokens (keys_out: T entries):
// blocks of min(T, kTokenSortBlock) tokens, each sorted by (id, token) in one
// CTA; key id*Bs + j for token j of its block.
nnt_status launch_token_sort(const uint16_t* ids, int64_t ids_stride, int B, int S,
                             uint32_t* keys_out, cudaStream_t st);
// dwte[id] += dx rows of that id in token order (keys from launch_token_sort)
nnt_status launch_embedding_scatter(const uint32_t* keys, int T, const float* dx, TokMap tm,
                                    int S, float* dwte, int d, int vocab, cudaStream_t st);
// dwpe[s] (+)= sum_b dx[b, s] in b order, for s in [s0, s0+ns)
nnt_status launch_wpe_grad(const float* dx, TokMap tm, int B, int s0, int ns, int d, float* dwpe,
                           int accumulate, cudaStream_t st);

// ---- layer norm
nnt_status launch_layernorm_fwd(const float* x, const float* g, const float* b, void* y,
                                float* mean, float* rstd, int64_t rows, int cols, float eps,
                                int act_dtype, cudaStream_t st);
nnt_status launch_layernorm_bwd(const float* dy, const float* x, const float* mean,
                                const float* rstd, const float* g, const float* resid, float* dx,
                                void* dx_act, int64_t rows, int cols, int act_dtype,
                                cudaStream_t st);
// dg (+)= sum_rows dy*xhat, db (+)= sum_rows dy and (out != NULL) dbias (+)=
// sum_rows out, in a fixed order; part: scratch of ln_colsum_chunks(rows) * 3 *
// cols floats
int64_t ln_colsum_chunks(int64_t rows);
nnt_status launch_ln_bwd_colsums(const float* dy, const float* x, const float* mean,
                                 const float* rstd, const float* out, int64_t rows, int cols,
                                 float* part, float* dg, float* db, float* dbias, int accumulate,
                                 cudaStream_t st);
nnt_status launch_sum_parts3(const float* part, int64_t nparts, int64_t cols, float* o0, float* o1,
                             float* o2, int accumulate, cudaStream_t st);
// Layer-norm backward (as launch_layernorm_bwd) that also writes the column
// sums sum dy*xhat, sum dy and (want_out) sum dx of its rows as
// ln_bwd_fused_ctas(rows) partial rows part[p][3][cols] (cols <= 1024; add
// them with launch_sum_parts3). dy, x and dx are read or written once.
int ln_bwd_fused_ctas(int64_t rows, int cols);
nnt_status launch_ln_bwd_fused(const float* dy, const float* x, const float* mean, const float* rstd,
                               const float* g, const float* resid, float* dx, void* dx_act,
                               int64_t rows, int cols, int act_dtype, float* part, int want_out,
                               cudaStream_t st);

// out[c] (=|+=) sum over p of part[p][c], p in increasing order
nnt_status launch_sum_parts(const float* part, int64_t nparts, int64_t cols, int64_t ld,
                            float* out, int accumulate, cudaStream_t st);
// column sums of an act or fp32 matrix [rows, cols] (ld) into out (fp32 [cols]);
// part: scratch of colsum_nparts(rows) * cols floats
int64_t colsum_nparts(int64_t rows);
nnt_status launch_colsum(const void* a, int a_dtype, int64_t rows, int64_t cols, int64_t ld,
                         float* part, float* out, int accumulate, cudaStream_t st);

// ---- causal softmax on score rows [z][q][k], z = zm.z(i) for i < nz, q in [q0, q0+nq)
nnt_status launch_softmax_fwd(const float* s, void* p, int64_t S, ZMap zm, int nz, int q0, int nq,
                              int act_dtype, cudaStream_t st);
nnt_status launch_softmax_bwd(const void* p, const float* dp, void* ds, int64_t S, ZMap zm, int nz,
                              int q0, int nq, float scale, int act_dtype, cudaStream_t st);

// ---- GELU
nnt_status launch_gelu_fwd(const float* u, void* g, int64_t n, int act_dtype, cudaStream_t st);
nnt_status launch_gelu_bwd(const void* dg, const float* u, void* du, int64_t n, int act_dtype,
                           cudaStream_t st);

// ---- cross-entropy + dlogits over rows [r0, r0+nrows) of z
// targets: tok_ids != NULL -> id of row r is tok_ids[b*(S+1) + s + 1] with (b,s) = tm.bs(r);
//          else tgt[r * tgt_stride]
nnt_status launch_cross_entropy(const float* z, int64_t ldz, int64_t r0, int64_t nrows,
                                int64_t cols, const uint16_t* tok_ids, TokMap tm,
                                const uint16_t* tgt, int64_t tgt_stride, void* dz, int64_t lddz,
                                float* row_loss, float inv_rows, int act_dtype, cudaStream_t st);
// The same with the row held in shared memory, half a row per CTA of a
// two-CTA cluster (one HBM read of the logits); rows of 1 to 55296 logits
// (ldz, lddz multiples of 4, z 16-byte aligned).
bool cross_entropy_smem_fits(int64_t cols);
nnt_status launch_cross_entropy_smem(const float* z, int64_t ldz, int64_t r0, int64_t nrows,
                                     int64_t cols, const uint16_t* tok_ids, TokMap tm,
                                     const uint16_t* tgt, int64_t tgt_stride, void* dz, int64_t lddz,
                                     float* row_loss, float inv_rows, int act_dtype, int sms,
                                     cudaStream_t st);
nnt_status launch_mean_loss(const float* row_loss, int64_t rows, float* loss, cudaStream_t st);

// ---- AdamW
nnt_status launch_adamw(float* w, const float* g, float* m, float* v, bf16* w_bf16, int64_t n,
                        float lr, float b1, float b2, float eps, float wd, float bc1, float bc2,
                        cudaStream_t st);

// same, hyper-parameters read on the device from hyper_dev[0..7] =
// (lr, beta1, beta2, eps, weight_decay, 1-beta1^t, 1-beta2^t, gradient scale)
// max_ctas > 0 caps the grid (moments in host memory: a few CTAs keep NVLink-C2C
// busy without taking SMs from concurrent tasks)
nnt_status launch_adamw_dev(float* w, const float* g, float* m, float* v, bf16* w_bf16, int64_t n,
                            const float* hyper_dev, cudaStream_t st, int max_ctas = 0);

// ---- init / casts
// std in double: the default 0.02 is the double 0.02, as in the host generator
nnt_status launch_init_normal(float* w, int64_t n, uint64_t seed, uint64_t stream_id, double std,
                              cudaStream_t st);
nnt_status launch_fill(float* w, int64_t n, float value, cudaStream_t st);
nnt_status launch_cast_bf16(const float* src, bf16* dst, int64_t n, cudaStream_t st);
nnt_status launch_check_tokens(const uint16_t* ids, int64_t n, int vocab, cudaStream_t st);

}  // namespace nnt
