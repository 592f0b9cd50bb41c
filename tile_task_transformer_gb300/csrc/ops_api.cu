// Stand-alone tile tasks of nnt.h ("single tile tasks" section): each call
// validates its arguments and enqueues the same kernel the step's executor
// runs, on caller buffers.
#include <mutex>

#include "common.cuh"
#include "flash.cuh"
#include "gemm.cuh"
#include "kernels.cuh"

using namespace nnt;

namespace {

// Library-owned device scratch for the calls that need temporaries (partial
// sums, sort keys). Grown on demand with cudaMalloc, per device, kept until
// exit; calls on different streams that need scratch are serialised by the
// device-wide synchronisation below when the buffer has to grow.
struct Scratch {
  std::mutex mu;
  void* ptr[64] = {};
  size_t bytes[64] = {};
};
Scratch g_scratch;

nnt_status scratch(size_t bytes, void** out) {
  int dev = 0;
  NNT_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return NNT_ERR_INTERNAL;
  std::lock_guard<std::mutex> lk(g_scratch.mu);
  if (g_scratch.bytes[dev] < bytes) {
    if (g_scratch.ptr[dev]) {
      NNT_CUDA_TRY(cudaDeviceSynchronize());
      cudaFree(g_scratch.ptr[dev]);
      g_scratch.ptr[dev] = nullptr;
      g_scratch.bytes[dev] = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
      cudaGetLastError();
      set_thread_error("scratch allocation of %zu bytes failed", bytes);
      return NNT_ERR_OOM;
    }
    g_scratch.ptr[dev] = p;
    g_scratch.bytes[dev] = bytes;
  }
  *out = g_scratch.ptr[dev];
  return NNT_OK;
}

bool dtype_ok(int d) { return d == NNT_F32 || d == NNT_BF16; }

}  // namespace

extern "C" {

nnt_status nnt_op_layernorm_fwd(const float* x_dev, const float* g_dev, const float* b_dev,
                                void* y_dev, float* mean_dev, float* rstd_dev, int64_t rows,
                                int64_t cols, float eps, int32_t dtype, void* stream) {
  NNT_CHECK_ARG(x_dev && g_dev && b_dev && y_dev && mean_dev && rstd_dev, "NULL pointer");
  NNT_CHECK_ARG(rows >= 0 && cols > 0 && cols <= 32768 && dtype_ok(dtype), "bad size or dtype");
  return launch_layernorm_fwd(x_dev, g_dev, b_dev, y_dev, mean_dev, rstd_dev, rows, (int)cols, eps,
                              dtype, (cudaStream_t)stream);
}

nnt_status nnt_op_layernorm_bwd(const float* dy_dev, const float* x_dev, const float* mean_dev,
                                const float* rstd_dev, const float* g_dev, const float* resid_dev,
                                float* dx_dev, void* dx_act_dev, float* dg_dev, float* db_dev,
                                int64_t rows, int64_t cols, int32_t dtype, void* stream) {
  NNT_CHECK_ARG(dy_dev && x_dev && mean_dev && rstd_dev && g_dev && dx_dev, "NULL pointer");
  NNT_CHECK_ARG((dg_dev == nullptr) == (db_dev == nullptr), "dg and db must both be given or both NULL");
  NNT_CHECK_ARG(rows >= 0 && cols > 0 && cols <= 32768 && dtype_ok(dtype), "bad size or dtype");
  cudaStream_t st = (cudaStream_t)stream;
  if (dg_dev && rows > 0 && cols <= 1024) {  // one pass: rows and their column sums
    const int64_t np = ln_bwd_fused_ctas(rows, (int)cols);
    void* part = nullptr;
    NNT_TRY(scratch((size_t)np * 3 * cols * 4, &part));
    NNT_TRY(launch_ln_bwd_fused(dy_dev, x_dev, mean_dev, rstd_dev, g_dev, resid_dev, dx_dev, dx_act_dev,
                                rows, (int)cols, dtype, (float*)part, 0, st));
    return launch_sum_parts3((const float*)part, np, cols, dg_dev, db_dev, nullptr, 0, st);
  }
  NNT_TRY(launch_layernorm_bwd(dy_dev, x_dev, mean_dev, rstd_dev, g_dev, resid_dev, dx_dev,
                               dx_act_dev, rows, (int)cols, dtype, st));
  if (dg_dev) {
    if (rows == 0) {
      NNT_CUDA_TRY(cudaMemsetAsync(dg_dev, 0, cols * 4, st));
      NNT_CUDA_TRY(cudaMemsetAsync(db_dev, 0, cols * 4, st));
      return NNT_OK;
    }
    void* part = nullptr;
    NNT_TRY(scratch((size_t)ln_colsum_chunks(rows) * 3 * cols * 4, &part));
    NNT_TRY(launch_ln_bwd_colsums(dy_dev, x_dev, mean_dev, rstd_dev, nullptr, rows, (int)cols,
                                  (float*)part, dg_dev, db_dev, nullptr, 0, st));
  }
  return NNT_OK;
}

nnt_status nnt_op_softmax_causal_fwd(const float* s_dev, void* p_dev, int64_t nmat, int64_t seq,
                                     int32_t dtype, void* stream) {
  NNT_CHECK_ARG(s_dev && p_dev, "NULL pointer");
  NNT_CHECK_ARG(nmat >= 0 && nmat < (1ll << 31) && seq > 0 && dtype_ok(dtype), "bad size or dtype");
  ZMap zm{0, 0, 1, 1};
  return launch_softmax_fwd(s_dev, p_dev, seq, zm, (int)nmat, 0, (int)seq, dtype,
                            (cudaStream_t)stream);
}

nnt_status nnt_op_softmax_causal_bwd(const void* p_dev, const float* dp_dev, void* ds_dev,
                                     int64_t nmat, int64_t seq, float scale, int32_t dtype,
                                     void* stream) {
  NNT_CHECK_ARG(p_dev && dp_dev && ds_dev, "NULL pointer");
  NNT_CHECK_ARG(nmat >= 0 && nmat < (1ll << 31) && seq > 0 && dtype_ok(dtype), "bad size or dtype");
  ZMap zm{0, 0, 1, 1};
  return launch_softmax_bwd(p_dev, dp_dev, ds_dev, seq, zm, (int)nmat, 0, (int)seq, scale, dtype,
                            (cudaStream_t)stream);
}

namespace {
// FlashArgs of the op-level calls: plain [Z][S][hd] buffers (one head per item).
FlashArgs plain_flash(int64_t Z, int64_t S, int64_t hd) {
  FlashArgs a;
  a.S = (int)S;
  a.hd = (int)hd;
  a.nz = (int)Z;
  a.zm = ZMap{0, 0, 1, 1};
  a.z_total = Z;
  a.tm = TokMap{(int)S, (int)Z, (int)S, 1};
  a.ldo = hd;
  a.ldd = hd;
  return a;
}
}  // namespace

nnt_status nnt_op_flash_attention_fwd(const void* q_dev, const void* k_dev, const void* v_dev,
                                      void* o_dev, float* lse_dev, int64_t Z, int64_t S,
                                      int64_t hd, void* stream) {
  NNT_CHECK_ARG(q_dev && k_dev && v_dev && o_dev && lse_dev, "NULL pointer");
  NNT_CHECK_ARG(Z > 0 && S > 0 && Z * S < (1ll << 31) && flash_supported((int)hd),
                "bad size (Z, S >= 1, Z*S < 2^31, hd 64 or 128)");
  FlashArgs a = plain_flash(Z, S, hd);
  a.o = static_cast<bf16*>(o_dev);
  a.lse = lse_dev;
  return launch_flash_fwd(static_cast<const bf16*>(q_dev), static_cast<const bf16*>(k_dev),
                          static_cast<const bf16*>(v_dev), a, (cudaStream_t)stream);
}

nnt_status nnt_op_flash_attention_bwd(const void* q_dev, const void* k_dev, const void* v_dev,
                                      const void* o_dev, const void* do_dev, const float* lse_dev,
                                      void* dq_dev, void* dk_dev, void* dv_dev, int64_t Z,
                                      int64_t S, int64_t hd, void* stream) {
  NNT_CHECK_ARG(q_dev && k_dev && v_dev && o_dev && do_dev && lse_dev && dq_dev && dk_dev && dv_dev,
                "NULL pointer");
  NNT_CHECK_ARG(Z > 0 && S > 0 && Z * S < (1ll << 31) && flash_supported((int)hd),
                "bad size (Z, S >= 1, Z*S < 2^31, hd 64 or 128)");
  // scratch: D [Z][S] fp32, then (S a multiple of 8) dS^T [Z][S][S] bf16
  const size_t d_bytes = ((size_t)(Z * S) * sizeof(float) + 255) / 256 * 256;
  const bool with_ds = S % 8 == 0;
  void* D = nullptr;
  NNT_TRY(scratch(d_bytes + (with_ds ? (size_t)Z * S * S * 2 : 0), &D));
  FlashArgs a = plain_flash(Z, S, hd);
  if (with_ds) a.ds = reinterpret_cast<bf16*>(static_cast<char*>(D) + d_bytes);
  a.o = const_cast<bf16*>(static_cast<const bf16*>(o_dev));
  a.lse = const_cast<float*>(lse_dev);
  a.D = static_cast<float*>(D);
  a.dq = static_cast<bf16*>(dq_dev);
  a.dk = static_cast<bf16*>(dk_dev);
  a.dv = static_cast<bf16*>(dv_dev);
  return launch_flash_bwd(static_cast<const bf16*>(q_dev), static_cast<const bf16*>(k_dev),
                          static_cast<const bf16*>(v_dev), static_cast<const bf16*>(do_dev), a,
                          (cudaStream_t)stream);
}

nnt_status nnt_op_gelu_fwd(const float* u_dev, void* g_dev, int64_t n, int32_t dtype, void* stream) {
  NNT_CHECK_ARG(u_dev && g_dev && n >= 0 && dtype_ok(dtype), "bad argument");
  return launch_gelu_fwd(u_dev, g_dev, n, dtype, (cudaStream_t)stream);
}

nnt_status nnt_op_gelu_bwd(const void* dg_dev, const float* u_dev, void* du_dev, int64_t n,
                           int32_t dtype, void* stream) {
  NNT_CHECK_ARG(dg_dev && u_dev && du_dev && n >= 0 && dtype_ok(dtype), "bad argument");
  return launch_gelu_bwd(dg_dev, u_dev, du_dev, n, dtype, (cudaStream_t)stream);
}

nnt_status nnt_op_cross_entropy(const float* z_dev, int64_t rows, int64_t cols, int64_t ldz,
                                const uint16_t* tgt_dev, int64_t tgt_stride, void* dz_dev,
                                int64_t lddz, float* row_loss_dev, float* loss_dev,
                                int32_t dtype, void* stream) {
  NNT_CHECK_ARG(z_dev && tgt_dev && dz_dev && row_loss_dev && loss_dev, "NULL pointer");
  NNT_CHECK_ARG(rows > 0 && rows < (1ll << 31) && cols > 0 && dtype_ok(dtype), "bad size or dtype");
  cudaStream_t st = (cudaStream_t)stream;
  TokMap tm{1, 1, 1, 1};
  NNT_TRY(launch_cross_entropy(z_dev, ldz, 0, rows, cols, nullptr, tm, tgt_dev, tgt_stride, dz_dev,
                               lddz, row_loss_dev, 1.0f / (float)rows, dtype, st));
  return launch_mean_loss(row_loss_dev, rows, loss_dev, st);
}

nnt_status nnt_op_adamw(float* w_dev, const float* g_dev, float* m_dev, float* v_dev,
                        void* w_bf16_dev, int64_t n, float lr, float beta1, float beta2, float eps,
                        float weight_decay, float bc1, float bc2, void* stream) {
  NNT_CHECK_ARG(w_dev && g_dev && m_dev && v_dev && n >= 0, "bad argument");
  NNT_CHECK_ARG(bc1 > 0 && bc2 > 0 && eps > 0, "bias corrections and eps must be positive");
  return launch_adamw(w_dev, g_dev, m_dev, v_dev, (bf16*)w_bf16_dev, n, lr, beta1, beta2, eps,
                      weight_decay, bc1, bc2, (cudaStream_t)stream);
}

nnt_status nnt_op_embedding_fwd(const uint16_t* ids_dev, int64_t ids_stride, const float* wte_dev,
                                const float* wpe_dev, float* x_dev, int64_t batch, int64_t seq,
                                int64_t d, int64_t vocab, void* stream) {
  NNT_CHECK_ARG(ids_dev && wte_dev && wpe_dev && x_dev, "NULL pointer");
  NNT_CHECK_ARG(batch > 0 && seq > 0 && d > 0 && vocab > 0 && vocab <= 65536 && ids_stride >= seq,
                "bad size");
  TokMap tm{(int)seq, (int)batch, (int)seq, 1};
  return launch_embedding_fwd(ids_dev, ids_stride, wte_dev, wpe_dev, x_dev, (int)d, (int)vocab, tm, 0,
                              (int)batch, 0, (int)seq, (cudaStream_t)stream);
}

nnt_status nnt_op_embedding_bwd(const uint16_t* ids_dev, int64_t ids_stride, const float* dx_dev,
                                float* dwte_dev, float* dwpe_dev, int64_t batch, int64_t seq,
                                int64_t d, int64_t vocab, void* stream) {
  NNT_CHECK_ARG(ids_dev && dx_dev && dwte_dev && dwpe_dev, "NULL pointer");
  NNT_CHECK_ARG(batch > 0 && seq > 0 && batch * seq <= kMaxTokens && d > 0 && vocab > 0 &&
                    vocab <= 65536 && ids_stride >= seq,
                "bad size (batch*seq must be <= %d)", kMaxTokens);
  cudaStream_t st = (cudaStream_t)stream;
  const int T = (int)(batch * seq);
  void* keys = nullptr;
  NNT_TRY(scratch((size_t)T * 4, &keys));
  TokMap tm{(int)seq, (int)batch, (int)seq, 1};
  NNT_TRY(launch_token_sort(ids_dev, ids_stride, (int)batch, (int)seq, (uint32_t*)keys, st));
  NNT_TRY(launch_embedding_scatter((const uint32_t*)keys, T, dx_dev, tm, (int)seq, dwte_dev, (int)d,
                                   (int)vocab, st));
  return launch_wpe_grad(dx_dev, tm, (int)batch, 0, (int)seq, (int)d, dwpe_dev, 1, st);
}

nnt_status nnt_op_gemm(const void* a_dev, int64_t lda, int32_t a_trans, const void* b_dev,
                       int64_t ldb, int32_t b_trans, void* c_dev, int64_t ldc, int32_t c_dtype,
                       int64_t M, int64_t N, int64_t K, float alpha, float beta, int32_t dtype,
                       int32_t backend, void* stream) {
  NNT_CHECK_ARG(a_dev && b_dev && c_dev, "NULL pointer");
  NNT_CHECK_ARG(M >= 0 && N >= 0 && K >= 0 && M < (1ll << 31) && N < (1ll << 31) && K < (1ll << 31),
                "bad size");
  NNT_CHECK_ARG(dtype_ok(dtype) && dtype_ok(c_dtype), "bad dtype");
  NNT_CHECK_ARG(beta == 0.f || (beta == 1.f && c_dtype == NNT_F32), "beta must be 0, or 1 with fp32 C");
  NNT_CHECK_ARG(lda >= (a_trans ? M : K) && ldb >= (b_trans ? N : K) && ldc >= N, "leading dimension too small");
  GemmArgs g;
  g.M = (int)M; g.N = (int)N; g.K = (int)K;
  g.m0 = 0; g.mt = (int)M; g.n0 = 0; g.nt = (int)N;
  g.A = a_dev; g.lda = lda; g.a_trans = a_trans ? 1 : 0;
  g.B = b_dev; g.ldb = ldb; g.b_trans = b_trans ? 1 : 0;
  g.op_dtype = dtype;
  g.C = c_dev; g.ldc = ldc; g.c_dtype = c_dtype;
  g.alpha = alpha;
  g.beta = beta != 0.f;
  if (M == 0 || N == 0) return NNT_OK;
  return gemm(g, backend, (cudaStream_t)stream);
}

nnt_status nnt_op_wait_selftest(int64_t limit_ns, int32_t arrive, void* stream) {
  NNT_CHECK_ARG(limit_ns >= 1000 && limit_ns <= 1000000000, "limit_ns must be in [1 us, 1 s]");
  return launch_wait_selftest((uint64_t)limit_ns, arrive != 0, (cudaStream_t)stream);
}

nnt_status nnt_op_read_error(uint32_t* code_out, void* stream) {
  NNT_CHECK_ARG(code_out, "NULL pointer");
  return read_and_clear_device_error(code_out, (cudaStream_t)stream);
}

}  // extern "C"
