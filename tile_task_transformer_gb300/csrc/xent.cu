// Mean cross-entropy and dlogits with the logit row held in shared memory.
//
// Loss per row: lse(z) - z[target]; dz = (softmax(z) - onehot(target)) / rows
// (the mean over all tokens; README "--loss-reduction=mean"). One CTA per SM
// walks the rows. A row (up to ~56K fp32 logits) is brought into shared memory
// by four bulk copies (cp.async.bulk, completion counted on one mbarrier per
// copy); pass 1 (running max and sum of exponentials) starts on each quarter
// as it lands, and pass 2 writes dz from shared memory, handing each quarter
// back to the next row's copy as soon as every thread is done with it. Each
// logit is read from HBM once and the next row streams in during pass 2.
// Every mbarrier wait is bounded; on expiry the kernel records the device
// error word, waits (bounded) for its copies in flight and returns.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace nnt {
namespace {

constexpr int kCeChunks = 4;
constexpr int kCeThreads = 512;
constexpr float kLog2eX = 1.4426950408889634f;
constexpr int kCeMaxSmem = 220 * 1024;  // dynamic shared memory bound for one row

__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kCeThreads, 1) cross_entropy_smem_kernel(
    const float* __restrict__ z, int64_t ldz, int64_t r0, int64_t nrows, int64_t cols,
    const uint16_t* __restrict__ tok_ids, TokMap tm, const uint16_t* __restrict__ tgt,
    int64_t tgt_stride, T* __restrict__ dz, int64_t lddz, float* __restrict__ row_loss,
    float inv_rows, int64_t cf, uint32_t* err) {
  extern __shared__ __align__(128) float rowbuf[];  // ldz floats
  __shared__ __align__(8) uint64_t full[kCeChunks];
  __shared__ float red_m[32], red_s[32];
  const int tid = threadIdx.x;
  const int64_t row_bytes = ldz * 4;
  auto cbytes = [&](int k) -> uint32_t {
    const int64_t b = row_bytes - (int64_t)k * cf * 4;
    return (uint32_t)(b <= 0 ? 0 : (b < cf * 4 ? b : cf * 4));
  };
  int issued[kCeChunks] = {0, 0, 0, 0};  // thread 0's copies per chunk (for the abort path)
  auto issue = [&](int k, int64_t rr) {
    const uint32_t nb = cbytes(k);
    if (nb == 0) return;
    mbar_arrive_expect_tx(&full[k], nb);
    bulk_load_1d(rowbuf + k * cf, z + (r0 + rr) * ldz + k * cf, nb, &full[k]);
    ++issued[k];
  };
  if (tid == 0) {
    for (int k = 0; k < kCeChunks; ++k) mbar_init(&full[k], 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0 && (int64_t)blockIdx.x < nrows)
    for (int k = 0; k < kCeChunks; ++k) issue(k, blockIdx.x);
  const int64_t n4 = cols >> 2;
  bool aborted = false;
  int it = 0;
  for (int64_t rr = blockIdx.x; rr < nrows; rr += gridDim.x, ++it) {
    const int64_t r = r0 + rr;
    // ---- pass 1: running (max, sum of exp) over each quarter as it lands
    float m = -INFINITY, s = 0.f;
    bool ok = true;
    for (int k = 0; k < kCeChunks; ++k) {
      if (cbytes(k) == 0) continue;
      if (ok) ok = mbar_wait(&full[k], (uint32_t)(it & 1));
      if (!ok) continue;
      const int64_t e0 = k * cf, e1 = std::min<int64_t>((k + 1) * cf, cols);
      for (int64_t i = e0 / 4 + tid; i < e1 / 4 && i < n4; i += kCeThreads) {
        const float4 v = *reinterpret_cast<const float4*>(rowbuf + 4 * i);
        const float lm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
        if (lm > m) {
          s *= exp2f((m - lm) * kLog2eX);
          m = lm;
        }
        const float ms = m * kLog2eX;
        s += exp2f(v.x * kLog2eX - ms) + exp2f(v.y * kLog2eX - ms) + exp2f(v.z * kLog2eX - ms) +
             exp2f(v.w * kLog2eX - ms);
      }
      if (e0 < cols && e1 == cols) {  // the scalar tail of the row
        for (int64_t c = 4 * n4 + tid; c < cols; c += kCeThreads) {
          const float v = rowbuf[c];
          if (v > m) {
            s *= exp2f((m - v) * kLog2eX);
            m = v;
          }
          s += exp2f((v - m) * kLog2eX);
        }
      }
    }
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    // ---- merge (m, s) over the CTA, in warp order
    const float wm = warp_max(m);
    s = (m == -INFINITY) ? 0.f : s * exp2f((m - wm) * kLog2eX);
    s = warp_sum(s);
    const int w = tid >> 5;
    if ((tid & 31) == 0) {
      red_m[w] = wm;
      red_s[w] = s;
    }
    __syncthreads();
    float M = -INFINITY;
    for (int i = 0; i < kCeThreads / 32; ++i) M = fmaxf(M, red_m[i]);
    float SUM = 0.f;
    for (int i = 0; i < kCeThreads / 32; ++i) SUM += red_s[i] * exp2f((red_m[i] - M) * kLog2eX);
    const float lse = M + logf(SUM);
    int y;
    if (tok_ids) {
      int b, sq;
      tm.bs(r, b, sq);
      y = tok_ids[(int64_t)b * (tm.S + 1) + sq + 1];
    } else {
      y = tgt[r * tgt_stride];
    }
    if (y >= cols) {
      if (tid == 0) atomicOr(err, DEVERR_TOKEN_RANGE);
      y = 0;
    }
    if (tid == 0) row_loss[r] = lse - rowbuf[y];
    // ---- pass 2: dz per quarter; each quarter then takes the next row's copy
    const float ls = lse * kLog2eX;
    T* dr = dz + r * lddz;
    const int64_t rn = rr + gridDim.x;
    for (int k = 0; k < kCeChunks; ++k) {
      if (cbytes(k) == 0) continue;
      const int64_t e0 = k * cf, e1 = std::min<int64_t>((k + 1) * cf, cols);
      for (int64_t i = e0 / 4 + tid; i < e1 / 4 && i < n4; i += kCeThreads) {
        const float4 v = *reinterpret_cast<const float4*>(rowbuf + 4 * i);
        float4 o;
        o.x = exp2f(v.x * kLog2eX - ls);
        o.y = exp2f(v.y * kLog2eX - ls);
        o.z = exp2f(v.z * kLog2eX - ls);
        o.w = exp2f(v.w * kLog2eX - ls);
        const int64_t c0 = 4 * i;
        if (y >= c0 && y < c0 + 4) {
          const int kk = (int)(y - c0);
          if (kk == 0) o.x -= 1.f;
          else if (kk == 1) o.y -= 1.f;
          else if (kk == 2) o.z -= 1.f;
          else o.w -= 1.f;
        }
        o.x *= inv_rows;
        o.y *= inv_rows;
        o.z *= inv_rows;
        o.w *= inv_rows;
        store4(dr + c0, o);
      }
      if (e0 < cols && e1 == cols) {  // scalar tail, then the padding columns as zeros
        for (int64_t c = 4 * n4 + tid; c < lddz; c += kCeThreads) {
          float o = 0.f;
          if (c < cols) o = (exp2f(rowbuf[c] * kLog2eX - ls) - (c == y ? 1.f : 0.f)) * inv_rows;
          dr[c] = from_f<T>(o);
        }
      }
      __syncthreads();  // every thread is done with this quarter
      if (tid == 0 && rn < nrows) issue(k, rn);
    }
  }
  if (aborted && tid == 0) {
    atomicOr(err, DEVERR_WAIT_TIMEOUT);
    // bounded waits for the copies still in flight before shared memory is released
    for (int k = 0; k < kCeChunks; ++k)
      for (int ph = it; ph < issued[k]; ++ph) mbar_wait(&full[k], (uint32_t)(ph & 1));
  }
}

}  // namespace

bool cross_entropy_smem_fits(int64_t ldz) { return ldz * 4 <= kCeMaxSmem; }

nnt_status launch_cross_entropy_smem(const float* z, int64_t ldz, int64_t r0, int64_t nrows,
                                     int64_t cols, const uint16_t* tok_ids, TokMap tm,
                                     const uint16_t* tgt, int64_t tgt_stride, void* dz, int64_t lddz,
                                     float* row_loss, float inv_rows, int act_dtype, int sms,
                                     cudaStream_t st) {
  NNT_CHECK_ARG(cross_entropy_smem_fits(ldz) && ldz % 4 == 0, "cross entropy: row too long for shared memory");
  NNT_CHECK_ARG(reinterpret_cast<uintptr_t>(z) % 16 == 0, "cross entropy: logits must be 16-byte aligned");
  uint32_t* err = device_error_word();
  NNT_CHECK_ARG(err != nullptr, "device error word unavailable");
  const int64_t cf = (ldz + kCeChunks * 4 - 1) / (kCeChunks * 4) * 4;  // floats per quarter (x4)
  const int smem = (int)(ldz * 4);
  const unsigned grid = (unsigned)std::min<int64_t>(nrows, sms);
  if (act_dtype == NNT_BF16) {
    auto k = cross_entropy_smem_kernel<bf16>;
    static const cudaError_t attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kCeMaxSmem);
    NNT_CUDA_TRY(attr);
    k<<<grid, kCeThreads, smem, st>>>(z, ldz, r0, nrows, cols, tok_ids, tm, tgt, tgt_stride, (bf16*)dz,
                                      lddz, row_loss, inv_rows, cf, err);
  } else {
    auto k = cross_entropy_smem_kernel<float>;
    static const cudaError_t attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kCeMaxSmem);
    NNT_CUDA_TRY(attr);
    k<<<grid, kCeThreads, smem, st>>>(z, ldz, r0, nrows, cols, tok_ids, tm, tgt, tgt_stride,
                                      (float*)dz, lddz, row_loss, inv_rows, cf, err);
  }
  return launch_check("cross_entropy_smem");
}

}  // namespace nnt
