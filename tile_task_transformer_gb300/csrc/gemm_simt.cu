// CUDA-core tile GEMM: the fp32 path (the NNTile experiments' own precision
// class, fp32/TF32) and a debug cross-check for the tensor-core kernel. Any
// operand layout, fp32 or bf16 operands, fp32 accumulation, 64x64 output tile
// per CTA, 4x4 outputs per thread, K staged 16 at a time in shared memory.
#include "gemm.cuh"

namespace nnt {

namespace {
constexpr int BM = 64, BN = 64, BK = 16;

template <typename T>
__device__ __forceinline__ float ld_op(const T* p, int64_t i) { return to_f(p[i]); }

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  // tiles sit on absolute multiples of BM/BN (so no tile straddles a causal block)
  const int i = blockIdx.z;
  const int m_box = (g.m0 / BM + (int)blockIdx.y) * BM;
  const int n_box = (g.n0 / BN + (int)blockIdx.x) * BN;
  const int m_start = max(g.m0, m_box), n_start = max(g.n0, n_box);
  const int m_end = min(g.m0 + g.mt, m_box + BM);
  const int n_end = min(g.n0 + g.nt, n_box + BN);
  if (!causal_tile_needed(g, m_start, m_end, n_start)) return;
  int k_lo, k_hi;
  causal_k_range(g, m_start, m_end, k_lo, k_hi);
  const int64_t z = g.zm.z(i);
  const T* A = static_cast<const T*>(g.A) + z * g.a_zs;
  const T* B = static_cast<const T*>(g.B) + z * g.b_zs;
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  float acc[4][4] = {};
  for (int k0 = k_lo; k0 < k_hi; k0 += BK) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int e = tid + r * 256;
      int mm, kk;
      if (g.a_trans) { mm = e % BM; kk = e / BM; } else { mm = e / BK; kk = e % BK; }
      const int m = m_box + mm, k = k0 + kk;
      float v = 0.f;
      if (m >= m_start && m < m_end && k < k_hi)
        v = ld_op(A, g.a_trans ? (int64_t)k * g.lda + m : (int64_t)m * g.lda + k);
      As[kk][mm] = v;
      int nn;
      if (g.b_trans) { nn = e % BN; kk = e / BN; } else { nn = e / BK; kk = e % BK; }
      const int n = n_box + nn, k2 = k0 + kk;
      float w = 0.f;
      if (n >= n_start && n < n_end && k2 < k_hi)
        w = ld_op(B, g.b_trans ? (int64_t)k2 * g.ldb + n : (int64_t)n * g.ldb + k2);
      Bs[kk][nn] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        a[r] = As[kk][ty * 4 + r];
        b[r] = Bs[kk][tx * 4 + r];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int m = m_box + ty * 4 + r, n = n_box + tx * 4 + c;
      if (m >= m_start && m < m_end && n >= n_start && n < n_end) epilogue_one(g, i, m, n, acc[r][c]);
    }
}
}  // namespace

nnt_status gemm_simt(const GemmArgs& g, cudaStream_t st) {
  if (g.mt <= 0 || g.nt <= 0 || g.nbatch <= 0) return NNT_OK;
  dim3 grid((unsigned)((g.n0 + g.nt - 1) / BN - g.n0 / BN + 1),
            (unsigned)((g.m0 + g.mt - 1) / BM - g.m0 / BM + 1), (unsigned)g.nbatch);
  NNT_CHECK_ARG(grid.y < 65536 && grid.z < 65536, "gemm: grid too large");
  if (g.op_dtype == NNT_BF16)
    launch_pdl(gemm_simt_kernel<bf16>, grid, 256, 0, st, g);
  else
    launch_pdl(gemm_simt_kernel<float>, grid, 256, 0, st, g);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_thread_error("gemm_simt launch: %s", cudaGetErrorString(e));
    return NNT_ERR_CUDA;
  }
  return NNT_OK;
}

nnt_status gemm(const GemmArgs& g, int backend, cudaStream_t st) {
  NNT_CHECK_ARG(g.A && g.B && g.C, "gemm: NULL operand");
  NNT_CHECK_ARG(g.m0 >= 0 && g.n0 >= 0 && g.m0 + g.mt <= g.M && g.n0 + g.nt <= g.N,
                "gemm: window [%d,+%d)x[%d,+%d) outside %dx%d", g.m0, g.mt, g.n0, g.nt, g.M, g.N);
  NNT_CHECK_ARG(g.epi == EPI_STORE || g.aux, "gemm: GELU epilogue needs aux");
  NNT_CHECK_ARG(!g.beta || g.c_dtype == NNT_F32, "gemm: beta needs fp32 C");
  if (backend == 0 && g.op_dtype == NNT_BF16 && gemm_tc_supported(g)) return gemm_tc(g, st);
  return gemm_simt(g, st);
}

}  // namespace nnt
