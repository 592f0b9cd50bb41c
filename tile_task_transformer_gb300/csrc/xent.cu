// Mean cross-entropy and dlogits with the logit row held in shared memory.
//
// Loss per row: lse(z) - z[target]; dz = (softmax(z) - onehot(target)) / rows
// (the mean over all tokens; README "--loss-reduction=mean").
//
// A cluster of two CTAs takes one row at a time, each CTA one half of it, and
// two CTAs share an SM, so one CTA's loads stream while the other computes. A
// CTA brings its half (up to 27648 fp32 logits) into shared memory with four
// bulk copies (cp.async.bulk, completion counted on one mbarrier per copy);
// pass 1 (running max and sum of exponentials) starts on each quarter as it
// lands. The two halves' (max, sum) are exchanged through distributed shared
// memory (st.async into the peer's slot, counted on the peer's mbarrier), both
// CTAs combine them in the same order into the same lse, and pass 2 writes dz
// from shared memory, handing each quarter back to the next row's copy as soon
// as every thread is done with it. Each logit is read from HBM once.
// Every mbarrier wait is bounded; on expiry the kernel records the device
// error word, tells the peer, waits (bounded) for its copies in flight and
// returns after a final cluster barrier that both CTAs always reach.
#include "kernels.cuh"
#include "ptx_math.cuh"
#include "tc_ptx.cuh"

namespace nnt {
namespace {

constexpr int kCeChunks = 4;  // bulk copies per half row
constexpr int kCeThreads = 512;
constexpr float kLog2eX = 1.4426950408889634f;
constexpr int kCeMaxSmem = 108 * 1024;  // dynamic shared memory for one half row (two CTAs per SM)

__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// two floats into a peer CTA's shared memory, counted on the peer's mbarrier
__device__ __forceinline__ void st_async_f32x2(uint32_t raddr, float a, float b, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                   raddr),
               "f"(a), "f"(b), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// CTA `rank` of a cluster holds columns [rank * half, rank * half + n_cols) of
// the current row in shared memory, brought in as kCeChunks copies of cf
// floats (the last shorter).
template <typename T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kCeThreads, 2) cross_entropy_pair_kernel(
    const float* __restrict__ z, int64_t ldz, int64_t r0, int64_t nrows, int64_t cols,
    const uint16_t* __restrict__ tok_ids, TokMap tm, const uint16_t* __restrict__ tgt,
    int64_t tgt_stride, T* __restrict__ dz, int64_t lddz, float* __restrict__ row_loss,
    float inv_rows, int half, int cf, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) float rowbuf[];  // this CTA's half row
  __shared__ __align__(8) uint64_t full[kCeChunks];
  __shared__ __align__(8) uint64_t xbar[2];         // the peer's (max, sum) landed, by row parity
  __shared__ __align__(8) float peer_ms[2][2];      // the peer's (max, sum), by row parity
  __shared__ float red_m[kCeThreads / 32], red_s[kCeThreads / 32];
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const int ncol = (int)cols;
  const int L = (ncol + 3) / 4 * 4;  // columns brought in (a multiple of 4)
  const int c_lo = (int)rank * half;
  const int n_cols = max(0, min(half, L - c_lo));
  auto cbytes = [&](int k) -> uint32_t {
    const int b = (n_cols - k * cf) * 4;
    return (uint32_t)(b <= 0 ? 0 : (b < cf * 4 ? b : cf * 4));
  };
  int issued[kCeChunks] = {0, 0, 0, 0};  // thread 0's copies per chunk (for the abort path)
  auto issue = [&](int k, int64_t rr) {
    const uint32_t nb = cbytes(k);
    if (nb == 0) return;
    mbar_arrive_expect_tx(&full[k], nb);
    bulk_load_1d(rowbuf + k * cf, z + (r0 + rr) * ldz + c_lo + k * cf, nb, &full[k]);
    ++issued[k];
  };
  if (tid == 0) {
    for (int k = 0; k < kCeChunks; ++k) mbar_init(&full[k], 1);
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    mbar_fence_init();
  }
  cluster_sync_all();  // both CTAs' barriers exist before any remote signal
  const int64_t cl = cluster_id_x(), ncl = cluster_count_x();
  if (tid == 0 && cl < nrows)
    for (int k = 0; k < kCeChunks; ++k) issue(k, cl);
  const int tail0 = ncol & ~3;  // first column of the scalar tail
  const float2 l2 = make_float2(kLog2eX, kLog2eX);
  const float log2_inv_rows = log2f(inv_rows);
  bool aborted = false;
  int it = 0;
  for (int64_t rr = cl; rr < nrows; rr += ncl, ++it) {
    const int64_t r = r0 + rr;
    const int slot = it & 1;
    if (tid == 0) mbar_arrive_expect_tx(&xbar[slot], 8);
    // the target, loaded now so that its latency hides behind pass 1
    int y;
    if (tok_ids) {
      int b, sq;
      tm.bs(r, b, sq);
      y = tok_ids[(int64_t)b * (tm.S + 1) + sq + 1];
    } else {
      y = tgt[r * tgt_stride];
    }
    // ---- pass 1: running (max, sum of exp) over each quarter as it lands
    float m = -INFINITY;
    float2 s2 = make_float2(0.f, 0.f);
    bool ok = true;
    for (int k = 0; k < kCeChunks; ++k) {
      if (cbytes(k) == 0) continue;
      if (ok) ok = mbar_wait(&full[k], (uint32_t)(it & 1));
      if (!ok) continue;
      const int g0 = c_lo + k * cf, g1 = c_lo + min((k + 1) * cf, n_cols);
      const int jend = max(min(g1, tail0) - c_lo, 0) >> 2;
      for (int j = (k * cf >> 2) + tid; j < jend; j += kCeThreads) {
        const float4 v = reinterpret_cast<const float4*>(rowbuf)[j];
        const float lm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
        if (lm > m) {
          const float f = ex2f((m - lm) * kLog2eX);
          s2 = mul2(s2, make_float2(f, f));
          m = lm;
        }
        const float2 nm = make_float2(-m * kLog2eX, -m * kLog2eX);
        const float2 a = fma2(make_float2(v.x, v.y), l2, nm);
        const float2 b = fma2(make_float2(v.z, v.w), l2, nm);
        s2 = add2(s2, add2(make_float2(ex2f(a.x), ex2f(a.y)), make_float2(ex2f(b.x), ex2f(b.y))));
      }
      if (g0 <= ncol - 1 && ncol - 1 < g1) {  // the scalar tail of the row
        for (int c = tail0 + tid; c < ncol; c += kCeThreads) {
          const float v = rowbuf[c - c_lo];
          if (v > m) {
            const float f = ex2f((m - v) * kLog2eX);
            s2 = mul2(s2, make_float2(f, f));
            m = v;
          }
          s2.x += ex2f((v - m) * kLog2eX);
        }
      }
    }
    float s = s2.x + s2.y;
    // ---- merge (m, s) over the CTA, in warp order
    const float wm = warp_max(m);
    s = (m == -INFINITY) ? 0.f : s * ex2f((m - wm) * kLog2eX);
    s = warp_sum(s);
    const int w = tid >> 5;
    if ((tid & 31) == 0) {
      red_m[w] = wm;
      red_s[w] = s;
    }
    const bool bad = __syncthreads_or(!ok);
    float M = -INFINITY;
    for (int i = 0; i < kCeThreads / 32; ++i) M = fmaxf(M, red_m[i]);
    float SUM = 0.f;
    for (int i = 0; i < kCeThreads / 32; ++i)
      if (red_m[i] != -INFINITY) SUM += red_s[i] * ex2f((red_m[i] - M) * kLog2eX);
    // ---- exchange the halves' (max, sum); a negative sum tells the peer to stop
    if (tid == 0)
      st_async_f32x2(peer_addr(&peer_ms[slot][0], rank ^ 1u), M, bad ? -1.f : SUM,
                     peer_addr(&xbar[slot], rank ^ 1u));
    const bool got = mbar_wait(&xbar[slot], (uint32_t)((it >> 1) & 1));
    const float pM = peer_ms[slot][0], pS = peer_ms[slot][1];
    if (__syncthreads_or(bad || !got || pS < 0.f)) {
      aborted = true;
      break;
    }
    // both CTAs combine (half 0, half 1) in this order, so both get the same lse
    const float M0 = rank == 0 ? M : pM, S0 = rank == 0 ? SUM : pS;
    const float M1 = rank == 0 ? pM : M, S1 = rank == 0 ? pS : SUM;
    const float MM = fmaxf(M0, M1);
    const float tot = (M0 == -INFINITY ? 0.f : S0 * ex2f((M0 - MM) * kLog2eX)) +
                      (M1 == -INFINITY ? 0.f : S1 * ex2f((M1 - MM) * kLog2eX));
    const float lse = MM + logf(tot);
    if (y >= ncol) {
      if (tid == 0 && rank == 0) atomicOr(err, DEVERR_TOKEN_RANGE);
      y = 0;
    }
    // the CTA holding the target's logit writes the row's loss
    if (tid == 0 && y >= c_lo && y < c_lo + n_cols) row_loss[r] = lse - rowbuf[y - c_lo];
    // ---- pass 2: dz per quarter; each quarter then takes the next row's copy.
    // dz = exp2(z log2 e - lse log2 e + log2(1/rows)) - onehot / rows
    const float ls = lse * kLog2eX - log2_inv_rows;
    const float2 nls = make_float2(-ls, -ls);
    T* dr = dz + r * lddz;
    const int64_t rn = rr + ncl;
    for (int k = 0; k < kCeChunks; ++k) {
      if (cbytes(k) == 0) continue;
      const int g0 = c_lo + k * cf, g1 = c_lo + min((k + 1) * cf, n_cols);
      const int jend = max(min(g1, tail0) - c_lo, 0) >> 2;
      for (int j = (k * cf >> 2) + tid; j < jend; j += kCeThreads) {
        const float4 v = reinterpret_cast<const float4*>(rowbuf)[j];
        const float2 a = fma2(make_float2(v.x, v.y), l2, nls);
        const float2 b = fma2(make_float2(v.z, v.w), l2, nls);
        float4 o = make_float4(ex2f(a.x), ex2f(a.y), ex2f(b.x), ex2f(b.y));
        const int c0 = c_lo + 4 * j;
        const unsigned d = (unsigned)(y - c0);
        if (d < 4u) {
          if (d == 0) o.x -= inv_rows;
          else if (d == 1) o.y -= inv_rows;
          else if (d == 2) o.z -= inv_rows;
          else o.w -= inv_rows;
        }
        store4(dr + c0, o);
      }
      if (g0 <= ncol - 1 && ncol - 1 < g1) {  // scalar tail, then the padding columns as zeros
        for (int64_t c = tail0 + tid; c < lddz; c += kCeThreads) {
          float o = 0.f;
          if (c < ncol) o = ex2f(rowbuf[c - c_lo] * kLog2eX - ls) - (c == y ? inv_rows : 0.f);
          dr[c] = from_f<T>(o);
        }
      }
      __syncthreads();  // every thread is done with this quarter
      if (tid == 0 && rn < nrows) issue(k, rn);
    }
    __syncthreads();  // red_m / red_s are rewritten by the next row
  }
  if (aborted && tid == 0) {
    atomicOr(err, DEVERR_WAIT_TIMEOUT);
    // bounded waits for the copies still in flight before shared memory is released
    for (int k = 0; k < kCeChunks; ++k)
      for (int ph = it; ph < issued[k]; ++ph) mbar_wait(&full[k], (uint32_t)(ph & 1));
  }
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the peer may still address its shared memory
}

// floats per CTA (the half row) and per bulk copy, both multiples of 4
int64_t ce_half(int64_t cols) { return ((cols + 3) / 4 * 4 + 7) / 8 * 4; }
int ce_chunk(int half) { return (half + kCeChunks * 4 - 1) / (kCeChunks * 4) * 4; }

template <typename T>
nnt_status launch_pair(const float* z, int64_t ldz, int64_t r0, int64_t nrows, int64_t cols,
                       const uint16_t* tok_ids, TokMap tm, const uint16_t* tgt, int64_t tgt_stride,
                       T* dz, int64_t lddz, float* row_loss, float inv_rows, int sms, uint32_t* err,
                       cudaStream_t st) {
  auto kern = cross_entropy_pair_kernel<T>;
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCeMaxSmem);
  NNT_CUDA_TRY(attr);
  const int half = (int)ce_half(cols), cf = ce_chunk(half);
  const unsigned clusters = (unsigned)std::min<int64_t>(nrows, sms);
  launch_pdl(kern, 2 * clusters, kCeThreads, (size_t)half * 4, st, z, ldz, r0, nrows, cols, tok_ids, tm, tgt,
                                                          tgt_stride, dz, lddz, row_loss, inv_rows,
                                                          half, cf, err);
  return launch_check("cross_entropy_pair");
}

}  // namespace

bool cross_entropy_smem_fits(int64_t cols) { return cols > 0 && ce_half(cols) * 4 <= kCeMaxSmem; }

nnt_status launch_cross_entropy_smem(const float* z, int64_t ldz, int64_t r0, int64_t nrows,
                                     int64_t cols, const uint16_t* tok_ids, TokMap tm,
                                     const uint16_t* tgt, int64_t tgt_stride, void* dz, int64_t lddz,
                                     float* row_loss, float inv_rows, int act_dtype, int sms,
                                     cudaStream_t st) {
  NNT_CHECK_ARG(cross_entropy_smem_fits(cols) && ldz % 4 == 0 && lddz % 4 == 0 && ldz >= cols &&
                    lddz >= cols,
                "cross entropy: unsupported row length or leading dimensions");
  NNT_CHECK_ARG(reinterpret_cast<uintptr_t>(z) % 16 == 0, "cross entropy: logits must be 16-byte aligned");
  if (nrows == 0) return NNT_OK;
  uint32_t* err = device_error_word();
  NNT_CHECK_ARG(err != nullptr, "device error word unavailable");
  if (act_dtype == NNT_BF16)
    return launch_pair<bf16>(z, ldz, r0, nrows, cols, tok_ids, tm, tgt, tgt_stride, (bf16*)dz, lddz,
                             row_loss, inv_rows, sms, err, st);
  return launch_pair<float>(z, ldz, r0, nrows, cols, tok_ids, tm, tgt, tgt_stride, (float*)dz, lddz,
                            row_loss, inv_rows, sms, err, st);
}

}  // namespace nnt
