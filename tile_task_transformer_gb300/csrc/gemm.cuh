// Tile GEMM interface shared by the tensor-core (tcgen05) and CUDA-core
// kernels: C = alpha * op(A) op(B) over a window of the output, with the
// step's fused epilogues (bias, residual add, GELU and its derivative, head
// split/merge of attention layouts) and the causal tile rules of the
// attention products.
#pragma once
#include "common.cuh"

namespace nnt {

enum EpiKind : int {
  EPI_STORE = 0,     // C = alpha*acc (+ bias[n]) (+ resid[m, n]) (+ C if beta)
  EPI_GELU = 1,      // u = alpha*acc + bias[n]; C = gelu(u), aux = gelu'(u) (aux_dtype)
  EPI_GELU_BWD = 2,  // C = alpha*acc * aux[m, n] (aux = gelu'(u) from the EPI_GELU launch)
};

enum OutMode : int {
  OUT_PLAIN = 0,      // C[z*c_zs + m*ldc + n], z = zm.z(batch item)
  OUT_HEADSPLIT = 1,  // m = token storage row, n in [0, parts*d): -> [parts][B][H][S][hd]
  OUT_HEADMERGE = 2,  // batch item z=(b,h), m = position s, n < hd: -> C[row(b,s)*ldc + h*hd + n]
};

enum CausalMode : int {
  CAUSAL_NONE = 0,
  CAUSAL_TILES = 1,    // only output tiles with n_start < round_up(m_end, kCausalBlock)
  CAUSAL_K_UPPER = 2,  // k in [0, round_up(m_end, kCausalBlock))
  CAUSAL_K_LOWER = 3,  // k in [round_down(m_start, kCausalBlock), K)
};

struct GemmArgs {
  int M = 0, N = 0, K = 0;
  int nbatch = 1;
  ZMap zm{0, 0, 1, 1};          // batch item i -> z = zm.z(i)
  int m0 = 0, mt = 0, n0 = 0, nt = 0;  // output window (global coordinates)
  // operands (op_dtype: NNT_F32 or NNT_BF16)
  const void* A = nullptr;
  int64_t lda = 0, a_zs = 0;  // a_zs, b_zs, c_zs: element strides per z = zm.z(i)
  int a_trans = 0;  // 0: A[m*lda + k]; 1: A[k*lda + m]
  const void* B = nullptr;
  int64_t ldb = 0, b_zs = 0;
  int b_trans = 0;  // 0: B[n*ldb + k]; 1: B[k*ldb + n]
  int op_dtype = NNT_BF16;
  // output
  void* C = nullptr;
  int64_t ldc = 0, c_zs = 0;
  int c_dtype = NNT_F32;
  int out_mode = OUT_PLAIN;
  TokMap tm{1, 1, 1, 1};
  int hs_B = 1, hs_H = 1, hs_S = 1, hs_hd = 1, hs_d = 1;  // head split/merge geometry
  int64_t c_col_off = 0;                                   // OUT_HEADMERGE column offset
  int64_t c_row0 = 0;  // OUT_PLAIN: row m is stored at (m - c_row0) * ldc (C holds rows from c_row0)
  float alpha = 1.f;
  int beta = 0;
  int epi = EPI_STORE;
  // fp32 workspace for splitting K across CTAs (plain fp32 stores only; see
  // gemm_split_k): partial products go here, then a fixed-order sum into C
  float* ws = nullptr;
  int64_t ws_elems = 0;
  const float* bias = nullptr;
  const float* resid = nullptr;
  int64_t ld_resid = 0;
  void* aux = nullptr;  // GELU derivative gelu'(u): written by EPI_GELU, read by EPI_GELU_BWD
  int64_t ld_aux = 0;
  int aux_dtype = NNT_F32;  // NNT_F32 or NNT_BF16
  int causal = CAUSAL_NONE;
  // limit of every mbarrier wait of the tensor-core kernel (%globaltimer ns);
  // on expiry it sets the device error word and returns
  uint64_t wait_ns = 5000000000ull;
};

__device__ __forceinline__ float gelu_fwd_dev(float u) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  return 0.5f * u * (1.0f + tanhf(c * (u + a * u * u * u)));
}
__device__ __forceinline__ float gelu_grad_dev(float u) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  const float t = tanhf(c * (u + a * u * u * u));
  return 0.5f * (1.0f + t) + 0.5f * u * (1.0f - t * t) * c * (1.0f + 3.0f * a * u * u);
}

__device__ __forceinline__ float aux_load(const GemmArgs& g, int64_t idx) {
  return g.aux_dtype == NNT_BF16 ? __bfloat162float(static_cast<const bf16*>(g.aux)[idx])
                                 : static_cast<const float*>(g.aux)[idx];
}
__device__ __forceinline__ void aux_store(const GemmArgs& g, int64_t idx, float v) {
  if (g.aux_dtype == NNT_BF16)
    static_cast<bf16*>(g.aux)[idx] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(g.aux)[idx] = v;
}

// Element offset of output (i, m, n) in C.
__device__ __forceinline__ int64_t out_offset(const GemmArgs& g, int i, int m, int n) {
  if (g.out_mode == OUT_PLAIN) return g.zm.z(i) * g.c_zs + (int64_t)(m - g.c_row0) * g.ldc + n;
  if (g.out_mode == OUT_HEADSPLIT) {
    int b, s;
    g.tm.bs(m, b, s);
    const int part = n / g.hs_d, r = n - part * g.hs_d;
    const int h = r / g.hs_hd, j = r - h * g.hs_hd;
    return ((((int64_t)part * g.hs_B + b) * g.hs_H + h) * g.hs_S + s) * g.hs_hd + j;
  }
  // OUT_HEADMERGE
  const int b = g.zm.b(i), h = g.zm.h(i);
  return g.tm.row(b, m) * g.ldc + g.c_col_off + (int64_t)h * g.hs_hd + n;
}

// Apply the epilogue to one accumulator value.
__device__ __forceinline__ void epilogue_one(const GemmArgs& g, int i, int m, int n, float acc) {
  const int64_t o = out_offset(g, i, m, n);
  float v = g.alpha * acc;
  if (g.epi == EPI_STORE) {
    if (g.bias) v += g.bias[n];
    if (g.resid) v += g.resid[(int64_t)m * g.ld_resid + n];
    if (g.beta) v += static_cast<const float*>(g.C)[o];
  } else if (g.epi == EPI_GELU) {
    if (g.bias) v += g.bias[n];
    aux_store(g, (int64_t)m * g.ld_aux + n, gelu_grad_dev(v));
    v = gelu_fwd_dev(v);
  } else {  // EPI_GELU_BWD
    v *= aux_load(g, (int64_t)m * g.ld_aux + n);
  }
  if (g.c_dtype == NNT_BF16)
    static_cast<bf16*>(g.C)[o] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(g.C)[o] = v;
}

// K range [k_lo, k_hi) of an output tile starting at row m_start (m_end exclusive).
__host__ __device__ __forceinline__ void causal_k_range(const GemmArgs& g, int m_start, int m_end,
                                                        int& k_lo, int& k_hi) {
  k_lo = 0;
  k_hi = g.K;
  if (g.causal == CAUSAL_K_UPPER) {
    int64_t e = round_up(m_end, kCausalBlock);
    k_hi = (int)(e < g.K ? e : g.K);
  } else if (g.causal == CAUSAL_K_LOWER) {
    k_lo = m_start / kCausalBlock * kCausalBlock;
  }
}
__host__ __device__ __forceinline__ bool causal_tile_needed(const GemmArgs& g, int m_start,
                                                            int m_end, int n_start) {
  if (g.causal != CAUSAL_TILES) return true;
  return n_start < round_up(m_end, kCausalBlock);
}

// Validate and run. backend 0: tcgen05 for bf16 operands when the shape allows,
// else CUDA cores; backend 1: CUDA cores.
nnt_status gemm(const GemmArgs& g, int backend, cudaStream_t st);
nnt_status gemm_simt(const GemmArgs& g, cudaStream_t st);
nnt_status gemm_tc(const GemmArgs& g, cudaStream_t st);  // NNT_ERR_INVALID_ARG if unsupported
bool gemm_tc_supported(const GemmArgs& g);
// Number of K slices the tensor-core path uses for g when a workspace of
// ws_elems floats is available (1 = no split). A split GEMM computes the
// slices as a batch of products into the workspace and sums them in slice
// order into C, so the result does not depend on scheduling. Only plain fp32
// outputs without bias, residual or activation, one batch item, alpha 1, and
// few output tiles for the SM count qualify.
int gemm_split_k(const GemmArgs& g, int64_t ws_elems);

// One bounded mbarrier wait (the tensor-core kernels' wait) on a phase that
// nothing completes (arrive false) or that is completed first (arrive true);
// on giving up after limit_ns it sets DEVERR_WAIT_TIMEOUT and returns.
nnt_status launch_wait_selftest(uint64_t limit_ns, bool arrive, cudaStream_t st);

}  // namespace nnt
