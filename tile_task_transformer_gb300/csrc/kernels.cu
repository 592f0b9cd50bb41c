// Memory-bound tile kernels of the GPT2 step: embedding gather/scatter, layer
// norm, causal softmax, GELU, cross-entropy, AdamW, column sums, init.
//
// The operations are the tile-wise layers the NNTile review page lists
// (pith.science, "What carries the argument": embedding, layer norm, softmax,
// attention, cross-entropy, Adam). All of them stream HBM once: rows are held
// in registers between the reduction and the write, loads and stores are
// 16-byte vectors, and reductions use warp shuffles. Reductions that produce
// parameter gradients write per-CTA partials that a second kernel sums in a
// fixed order, so results do not depend on scheduling.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "kernels.cuh"

namespace nnt {

static __device__ uint32_t g_device_error = 0;

uint32_t* device_error_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<uint32_t*>(p);
}

// Copies the word to pinned-free host memory; synchronises `st`.
nnt_status read_and_clear_device_error(uint32_t* code_host, cudaStream_t st) {
  uint32_t zero = 0;
  NNT_CUDA_TRY(cudaMemcpyFromSymbolAsync(code_host, g_device_error, 4, 0, cudaMemcpyDeviceToHost, st));
  NNT_CUDA_TRY(cudaMemcpyToSymbolAsync(g_device_error, &zero, 4, 0, cudaMemcpyHostToDevice, st));
  NNT_CUDA_TRY(cudaStreamSynchronize(st));
  return NNT_OK;
}

static thread_local char t_err[512] = "";
void set_thread_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof t_err, fmt, ap);
  va_end(ap);
}
const char* thread_error() { return t_err; }

static constexpr float kLog2e = 1.4426950408889634f;

// =====================================================================
// embedding
// =====================================================================

// x[row(b,s), :] = wte[id(b,s), :] + wpe[s, :]; one thread per 4 columns.
__global__ void embedding_fwd_kernel(const uint16_t* __restrict__ ids, int64_t ids_stride,
                                     const float* __restrict__ wte, const float* __restrict__ wpe,
                                     float* __restrict__ x, int d, int vocab, TokMap tm, int b0,
                                     int nb, int s0, int ns) {
  pdl_wait();
  pdl_trigger();
  const int nv = d >> 2;
  const int64_t total = (int64_t)nb * ns * nv;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % nv);
    const int64_t tok = i / nv;
    const int b = b0 + (int)(tok / ns), s = s0 + (int)(tok % ns);
    const int id = ids[(int64_t)b * ids_stride + s];
    float4 out;
    if (id < vocab) {
      float4 e = load4(wte + (int64_t)id * d + 4 * c);
      float4 p = load4(wpe + (int64_t)s * d + 4 * c);
      out = make_float4(e.x + p.x, e.y + p.y, e.z + p.z, e.w + p.w);
    } else {
      if (c == 0) atomicOr(&g_device_error, DEVERR_TOKEN_RANGE);
      out = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    store4(x + tm.row(b, s) * d + 4 * c, out);
  }
}

nnt_status launch_embedding_fwd(const uint16_t* ids, int64_t ids_stride, const float* wte,
                                const float* wpe, float* x, int d, int vocab, TokMap tm, int b0,
                                int nb, int s0, int ns, cudaStream_t st) {
  NNT_CHECK_ARG(d % 4 == 0 && d > 0, "embedding: d must be a positive multiple of 4");
  int64_t total = (int64_t)nb * ns * (d / 4);
  if (total == 0) return NNT_OK;
  int grid = (int)std::min<int64_t>(ceil_div(total, 256), 152 * 16);
  launch_pdl(embedding_fwd_kernel, grid, 256, 0, st, ids, ids_stride, wte, wpe, x, d, vocab, tm, b0, nb, s0,
                                             ns);
  return launch_check("embedding_fwd");
}

// Token sort for the embedding scatter-add. The T tokens are cut into blocks
// of Bs = min(T, kTokenSortBlock) consecutive tokens; CTA b sorts the keys
// id*Bs + j (j = local index of token t = b*Bs + j) of block b with a bitonic
// network in shared memory and writes them to keys_out[b*Bs ...]. Keys are
// unique, so inside a block the tokens that share an id stay in token order;
// the blocks themselves are in token order.
__global__ void token_sort_kernel(const uint16_t* __restrict__ ids, int64_t ids_stride, int B,
                                  int S, uint32_t* __restrict__ keys_out, int Bs, int npow2) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t sk[];
  const int T = B * S;
  const int t0 = blockIdx.x * Bs;
  const int n = min(Bs, T - t0);
  for (int i = threadIdx.x; i < npow2; i += blockDim.x) {
    uint32_t k = 0xFFFFFFFFu;
    if (i < n) {
      const int t = t0 + i;
      const int b = t / S, s = t % S;
      k = (uint32_t)ids[(int64_t)b * ids_stride + s] * (uint32_t)Bs + (uint32_t)i;
    }
    sk[i] = k;
  }
  __syncthreads();
  for (int size = 2; size <= npow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < npow2 / 2; i += blockDim.x) {
        int lo = 2 * i - (i & (stride - 1));
        int hi = lo + stride;
        bool up = ((lo & size) == 0);
        uint32_t a = sk[lo], c = sk[hi];
        if ((a > c) == up) {
          sk[lo] = c;
          sk[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) keys_out[t0 + i] = sk[i];
}

int token_sort_block(int T) { return T < kTokenSortBlock ? T : kTokenSortBlock; }

nnt_status launch_token_sort(const uint16_t* ids, int64_t ids_stride, int B, int S,
                             uint32_t* keys_out, cudaStream_t st) {
  const int64_t T64 = (int64_t)B * S;
  NNT_CHECK_ARG(T64 > 0 && T64 <= kMaxTokens, "token sort: batch*seq must be in [1, %d] (got %lld)",
                kMaxTokens, (long long)T64);
  const int T = (int)T64;
  const int Bs = token_sort_block(T);
  int npow2 = 1;
  while (npow2 < Bs) npow2 <<= 1;
  size_t smem = (size_t)npow2 * 4;
  if (smem > 48 * 1024)
    NNT_CUDA_TRY(cudaFuncSetAttribute(token_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem));
  launch_pdl(token_sort_kernel, (T + Bs - 1) / Bs, 1024, smem, st, ids, ids_stride, B, S, keys_out, Bs, npow2);
  return launch_check("token_sort");
}

// First position in keys[0, n) whose key is >= v (keys ascending).
__device__ __forceinline__ int lower_bound_u32(const uint32_t* keys, int n, uint32_t v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (keys[mid] < v) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// CTA p looks at sorted position p (block b = p / Bs). It works only when p
// starts the run of its id inside block b and no earlier block holds that id;
// it then adds the dx rows of every token with that id -- block by block from
// b on, each block's run in token order, so in increasing token order -- onto
// dwte[id].
constexpr int kScatterMaxBlocks = kMaxTokens / kTokenSortBlock;
__global__ void embedding_scatter_kernel(const uint32_t* __restrict__ keys, int T, int Bs,
                                         const float* __restrict__ dx, TokMap tm, int S,
                                         float* __restrict__ dwte, int d, int vocab) {
  pdl_wait();
  pdl_trigger();
  __shared__ int run_lo[kScatterMaxBlocks], run_hi[kScatterMaxBlocks];
  __shared__ int in_earlier;
  const int p = blockIdx.x;
  const int blk = p / Bs;
  const uint32_t id = keys[p] / (uint32_t)Bs;
  if (p > blk * Bs && keys[p - 1] / (uint32_t)Bs == id) return;  // uniform over the CTA
  if (id >= (uint32_t)vocab) return;
  const int nblk = (T + Bs - 1) / Bs;
  if (threadIdx.x == 0) in_earlier = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
    const int n = min(Bs, T - b * Bs);
    const uint32_t* kb = keys + (int64_t)b * Bs;
    const int lo = b == blk ? p - blk * Bs : lower_bound_u32(kb, n, id * (uint32_t)Bs);
    const int hi = lower_bound_u32(kb, n, (id + 1) * (uint32_t)Bs);
    run_lo[b] = lo;
    run_hi[b] = hi;
    if (b < blk && hi > lo) in_earlier = 1;
  }
  __syncthreads();
  if (in_earlier) return;  // that block's CTA covers this id
  const int nv = d >> 2;
  for (int c = threadIdx.x; c < nv; c += blockDim.x) {
    float4 acc = load4(dwte + (int64_t)id * d + 4 * c);
    for (int b = blk; b < nblk; ++b) {
      const uint32_t* kb = keys + (int64_t)b * Bs;
      for (int j = run_lo[b]; j < run_hi[b]; ++j) {
        const int t = b * Bs + (int)(kb[j] % (uint32_t)Bs);
        float4 g = load4(dx + tm.row(t / S, t % S) * d + 4 * c);
        acc.x += g.x;
        acc.y += g.y;
        acc.z += g.z;
        acc.w += g.w;
      }
    }
    store4(dwte + (int64_t)id * d + 4 * c, acc);
  }
}

nnt_status launch_embedding_scatter(const uint32_t* keys, int T, const float* dx, TokMap tm, int S,
                                    float* dwte, int d, int vocab, cudaStream_t st) {
  NNT_CHECK_ARG(d % 4 == 0, "embedding scatter: d must be a multiple of 4");
  NNT_CHECK_ARG(T >= 0 && T <= kMaxTokens, "embedding scatter: too many tokens (%d)", T);
  if (T == 0) return NNT_OK;
  int threads = std::min(256, std::max(32, (d / 4 + 31) / 32 * 32));
  launch_pdl(embedding_scatter_kernel, T, threads, 0, st, keys, T, token_sort_block(T), dx, tm, S, dwte, d,
                                                  vocab);
  return launch_check("embedding_scatter");
}

__global__ void wpe_grad_kernel(const float* __restrict__ dx, TokMap tm, int B, int s0, int ns,
                                int d, float* __restrict__ dwpe, int accumulate) {
  pdl_wait();
  pdl_trigger();
  const int nv = d >> 2;
  const int64_t total = (int64_t)ns * nv;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int s = s0 + (int)(i / nv), c = (int)(i % nv);
    float4 acc = accumulate ? load4(dwpe + (int64_t)s * d + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int b = 0; b < B; ++b) {
      float4 g = load4(dx + tm.row(b, s) * d + 4 * c);
      acc.x += g.x;
      acc.y += g.y;
      acc.z += g.z;
      acc.w += g.w;
    }
    store4(dwpe + (int64_t)s * d + 4 * c, acc);
  }
}

nnt_status launch_wpe_grad(const float* dx, TokMap tm, int B, int s0, int ns, int d, float* dwpe,
                           int accumulate, cudaStream_t st) {
  int64_t total = (int64_t)ns * (d / 4);
  if (total == 0) return NNT_OK;
  int grid = (int)std::min<int64_t>(ceil_div(total, 256), 152 * 8);
  launch_pdl(wpe_grad_kernel, grid, 256, 0, st, dx, tm, B, s0, ns, d, dwpe, accumulate);
  return launch_check("wpe_grad");
}

// =====================================================================
// layer norm (reference "Layer Normalization"; pre-LN blocks)
// =====================================================================

// TPR threads per row, each holding up to MAXV float4 of the row in registers.
template <int TPR, int MAXV, typename T>
__global__ void ln_fwd_kernel(const float* __restrict__ x, const float* __restrict__ g,
                              const float* __restrict__ b, T* __restrict__ y,
                              float* __restrict__ mean, float* __restrict__ rstd, int64_t rows,
                              int cols, float eps) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  const int rpc = blockDim.x / TPR;
  const int lane = threadIdx.x % TPR;
  const int64_t row = (int64_t)blockIdx.x * rpc + threadIdx.x / TPR;
  const bool active = row < rows;
  const int nv = cols >> 2;
  const float* xr = x + (active ? row : 0) * cols;
  float4 v[MAXV];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + i * TPR;
    if (active && c < nv) {
      v[i] = load4(xr + 4 * c);
      s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    } else {
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  s = group_sum<TPR>(s, red);
  const float mu = s / (float)cols;
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + i * TPR;
    if (active && c < nv) {
      float a = v[i].x - mu, bb = v[i].y - mu, cc = v[i].z - mu, dd = v[i].w - mu;
      ss += (a * a + bb * bb) + (cc * cc + dd * dd);
    }
  }
  ss = group_sum<TPR>(ss, red);
  const float rs = 1.0f / sqrtf(ss / (float)cols + eps);
  if (!active) return;
  T* yr = y + row * cols;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + i * TPR;
    if (c < nv) {
      float4 gv = load4(g + 4 * c), bv = load4(b + 4 * c);
      float4 o;
      o.x = (v[i].x - mu) * rs * gv.x + bv.x;
      o.y = (v[i].y - mu) * rs * gv.y + bv.y;
      o.z = (v[i].z - mu) * rs * gv.z + bv.z;
      o.w = (v[i].w - mu) * rs * gv.w + bv.w;
      store4(yr + 4 * c, o);
    }
  }
  if (lane == 0) {
    mean[row] = mu;
    rstd[row] = rs;
  }
}

// Pick threads-per-row so that a row fits in <= 8 float4 per thread.
static int row_tpr(int cols) {
  int nv = cols / 4;
  int tpr = 32;
  while (tpr * 8 < nv && tpr < 1024) tpr <<= 1;
  return tpr;
}

// float4 groups per thread actually needed (1, 2, 4, 6 or 8), so register
// arrays are no larger than the row.
static int row_maxv(int cols, int tpr) {
  const int need = (int)ceil_div(cols / 4, tpr);
  return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 6 ? 6 : 8;
}

#define NNT_MAXV_DISPATCH(mv, ...)                               \
  switch (mv) {                                                  \
    case 1: { constexpr int MV = 1; __VA_ARGS__; } break;        \
    case 2: { constexpr int MV = 2; __VA_ARGS__; } break;        \
    case 4: { constexpr int MV = 4; __VA_ARGS__; } break;        \
    case 6: { constexpr int MV = 6; __VA_ARGS__; } break;        \
    default: { constexpr int MV = 8; __VA_ARGS__; } break;       \
  }

#define NNT_TPR_DISPATCH(tpr, ...)                          \
  switch (tpr) {                                            \
    case 32: { constexpr int TPR = 32; __VA_ARGS__; } break;     \
    case 64: { constexpr int TPR = 64; __VA_ARGS__; } break;     \
    case 128: { constexpr int TPR = 128; __VA_ARGS__; } break;   \
    case 256: { constexpr int TPR = 256; __VA_ARGS__; } break;   \
    case 512: { constexpr int TPR = 512; __VA_ARGS__; } break;   \
    default: { constexpr int TPR = 1024; __VA_ARGS__; } break;   \
  }

nnt_status launch_layernorm_fwd(const float* x, const float* g, const float* b, void* y,
                                float* mean, float* rstd, int64_t rows, int cols, float eps,
                                int act_dtype, cudaStream_t st) {
  NNT_CHECK_ARG(cols % 4 == 0 && cols > 0 && cols <= 32768,
                "layernorm: cols must be a multiple of 4 in [4, 32768] (got %d)", cols);
  if (rows == 0) return NNT_OK;
  const int tpr = row_tpr(cols);
  const int block = std::max(256, tpr);
  const int rpc = block / tpr;
  const int64_t grid = ceil_div(rows, rpc);
  const int mv = row_maxv(cols, tpr);
  NNT_TPR_DISPATCH(tpr, NNT_MAXV_DISPATCH(mv, {
    if (act_dtype == NNT_BF16)
      launch_pdl(ln_fwd_kernel<TPR, MV, bf16>, grid, block, 0, st, x, g, b, (bf16*)y, mean, rstd, rows, cols, eps);
    else
      launch_pdl(ln_fwd_kernel<TPR, MV, float>, grid, block, 0, st, x, g, b, (float*)y, mean, rstd, rows, cols, eps);
  }));
  return launch_check("layernorm_fwd");
}

// dx = rstd*(gdy - mean(gdy) - xhat*mean(gdy*xhat)) (+ resid), gdy = g*dy; the
// parameter gradients come from ln_bwd_colsums_kernel.
template <int TPR, int MAXV, typename T>
__global__ void ln_bwd_kernel(const float* __restrict__ dy, const float* __restrict__ x,
                              const float* __restrict__ mean, const float* __restrict__ rstd,
                              const float* __restrict__ g, const float* resid, float* dx,
                              T* __restrict__ dx_act, int64_t rows, int cols) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  const int rpc = blockDim.x / TPR;
  const int lane = threadIdx.x % TPR;
  const int64_t row = (int64_t)blockIdx.x * rpc + threadIdx.x / TPR;
  const bool active = row < rows;
  const int64_t r = active ? row : 0;
  const int nv = cols >> 2;
  const float mu = mean[r], rs = rstd[r];
  float4 xh[MAXV], gd[MAXV];
  float s1 = 0.f, s2 = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + i * TPR;
    if (active && c < nv) {
      const float4 dv = load4(dy + r * cols + 4 * c);
      const float4 xv = load4(x + r * cols + 4 * c);
      const float4 gm = load4(g + 4 * c);
      xh[i] = make_float4((xv.x - mu) * rs, (xv.y - mu) * rs, (xv.z - mu) * rs, (xv.w - mu) * rs);
      gd[i] = make_float4(gm.x * dv.x, gm.y * dv.y, gm.z * dv.z, gm.w * dv.w);
      s1 += (gd[i].x + gd[i].y) + (gd[i].z + gd[i].w);
      s2 += (gd[i].x * xh[i].x + gd[i].y * xh[i].y) + (gd[i].z * xh[i].z + gd[i].w * xh[i].w);
    } else {
      xh[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      gd[i] = xh[i];
    }
  }
  const float inv_n = 1.0f / (float)cols;
  s1 = group_sum<TPR>(s1, red) * inv_n;
  s2 = group_sum<TPR>(s2, red) * inv_n;
  if (!active) return;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + i * TPR;
    if (c < nv) {
      float4 o;
      o.x = rs * (gd[i].x - s1 - xh[i].x * s2);
      o.y = rs * (gd[i].y - s1 - xh[i].y * s2);
      o.z = rs * (gd[i].z - s1 - xh[i].z * s2);
      o.w = rs * (gd[i].w - s1 - xh[i].w * s2);
      if (resid) {
        const float4 q = load4(resid + r * cols + 4 * c);
        o.x += q.x;
        o.y += q.y;
        o.z += q.z;
        o.w += q.w;
      }
      store4(dx + r * cols + 4 * c, o);
      if (dx_act) store4(dx_act + r * cols + 4 * c, o);
    }
  }
}

nnt_status launch_layernorm_bwd(const float* dy, const float* x, const float* mean,
                                const float* rstd, const float* g, const float* resid, float* dx,
                                void* dx_act, int64_t rows, int cols, int act_dtype,
                                cudaStream_t st) {
  NNT_CHECK_ARG(cols % 4 == 0 && cols > 0 && cols <= 32768,
                "layernorm bwd: cols must be a multiple of 4 in [4, 32768] (got %d)", cols);
  if (rows == 0) return NNT_OK;
  const int tpr = row_tpr(cols);
  const int block = std::max(256, tpr);
  const int64_t grid = ceil_div(rows, block / tpr);
  const int mv = row_maxv(cols, tpr);
  NNT_TPR_DISPATCH(tpr, NNT_MAXV_DISPATCH(mv, {
    if (act_dtype == NNT_BF16)
      launch_pdl(ln_bwd_kernel<TPR, MV, bf16>, grid, block, 0, st, dy, x, mean, rstd, g, resid, dx, (bf16*)dx_act, rows, cols);
    else
      launch_pdl(ln_bwd_kernel<TPR, MV, float>, grid, block, 0, st, dy, x, mean, rstd, g, resid, dx, (float*)dx_act, rows, cols);
  }));
  return launch_check("layernorm_bwd");
}

// Layer-norm backward with its column sums in the same pass, for rows of at
// most 1024 columns. A row belongs to a group of RW warps (RW = 1 or 2; each
// lane holds MAXV float4 groups of the row: dy, x and the residual are all
// loaded before the row statistics are reduced, so a row costs one memory
// round trip); the two warps of a pair swap their partial sums through shared
// memory with a 64-thread named barrier. Row groups take rows blockIdx*G + g,
// then every gridDim*G-th (G = 8 / RW). Besides dx it accumulates, per column,
// sum dy*xhat, sum dy and (want_out) sum dx; the row groups' sums are added in
// group order through shared memory and the CTA writes part[blockIdx][3][cols]
// (sum_parts3 adds the CTAs in order). dy, x and the residual are read once.
template <int RW, int MAXV, typename T>
__global__ void __launch_bounds__(256, 2) ln_bwd_fused_kernel(
    const float* __restrict__ dy, const float* __restrict__ x, const float* __restrict__ mean,
    const float* __restrict__ rstd, const float* __restrict__ g, const float* resid, float* dx,
    T* __restrict__ dx_act, int64_t rows, int cols, float* __restrict__ part, int want_out) {
  pdl_wait();
  pdl_trigger();
  constexpr int G = 8 / RW;  // row groups per CTA
  extern __shared__ float red[];  // [G][3][cols]
  __shared__ float xch[2][8][2];  // pair exchange: [parity][warp][s1, s2]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int grp = w / RW, half = w % RW;
  const int nv = cols >> 2;
  const float inv_n = 1.0f / (float)cols;
  float4 ag[MAXV], ab[MAXV], ao[MAXV];
#pragma unroll
  for (int i = 0; i < MAXV; ++i) ag[i] = ab[i] = ao[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  int parity = 0;
  for (int64_t row = (int64_t)blockIdx.x * G + grp; row < rows; row += (int64_t)gridDim.x * G) {
    const float mu = mean[row], rs = rstd[row];
    float4 dv[MAXV], xh[MAXV], q[MAXV];
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int c = half * 32 + lane + 32 * RW * i;
      if (c < nv) {
        dv[i] = load4(dy + row * cols + 4 * c);
        xh[i] = load4(x + row * cols + 4 * c);
        q[i] = resid ? load4(resid + row * cols + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        dv[i] = xh[i] = q[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int c = half * 32 + lane + 32 * RW * i;
      if (c < nv) {
        const float4 gm = __ldg(reinterpret_cast<const float4*>(g) + c);
        xh[i] = make_float4((xh[i].x - mu) * rs, (xh[i].y - mu) * rs, (xh[i].z - mu) * rs, (xh[i].w - mu) * rs);
        const float4 gd = make_float4(gm.x * dv[i].x, gm.y * dv[i].y, gm.z * dv[i].z, gm.w * dv[i].w);
        s1 += (gd.x + gd.y) + (gd.z + gd.w);
        s2 += (gd.x * xh[i].x + gd.y * xh[i].y) + (gd.z * xh[i].z + gd.w * xh[i].w);
      }
    }
    s1 = warp_sum(s1);
    s2 = warp_sum(s2);
    if constexpr (RW == 2) {
      if (lane == 0) {
        xch[parity][w][0] = s1;
        xch[parity][w][1] = s2;
      }
      asm volatile("bar.sync %0, 64;" ::"r"(1 + grp) : "memory");
      const int p0 = grp * 2;  // the pair's sums in warp order
      s1 = xch[parity][p0][0] + xch[parity][p0 + 1][0];
      s2 = xch[parity][p0][1] + xch[parity][p0 + 1][1];
      parity ^= 1;  // the next row writes the other slot, so no second barrier is needed
    }
    s1 *= inv_n;
    s2 *= inv_n;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int c = half * 32 + lane + 32 * RW * i;
      if (c < nv) {
        const float4 gm = __ldg(reinterpret_cast<const float4*>(g) + c);
        float4 o;
        o.x = rs * (gm.x * dv[i].x - s1 - xh[i].x * s2) + q[i].x;
        o.y = rs * (gm.y * dv[i].y - s1 - xh[i].y * s2) + q[i].y;
        o.z = rs * (gm.z * dv[i].z - s1 - xh[i].z * s2) + q[i].z;
        o.w = rs * (gm.w * dv[i].w - s1 - xh[i].w * s2) + q[i].w;
        store4(dx + row * cols + 4 * c, o);
        if (dx_act) store4(dx_act + row * cols + 4 * c, o);
        ag[i].x += dv[i].x * xh[i].x; ag[i].y += dv[i].y * xh[i].y;
        ag[i].z += dv[i].z * xh[i].z; ag[i].w += dv[i].w * xh[i].w;
        ab[i].x += dv[i].x; ab[i].y += dv[i].y; ab[i].z += dv[i].z; ab[i].w += dv[i].w;
        ao[i].x += o.x; ao[i].y += o.y; ao[i].z += o.z; ao[i].w += o.w;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = half * 32 + lane + 32 * RW * i;
    if (c < nv) {
      float* r0 = red + (grp * 3) * cols + 4 * c;
      *reinterpret_cast<float4*>(r0) = ag[i];
      *reinterpret_cast<float4*>(r0 + cols) = ab[i];
      *reinterpret_cast<float4*>(r0 + 2 * cols) = ao[i];
    }
  }
  __syncthreads();
  const int nsum = (want_out ? 3 : 2) * cols;
  for (int k = threadIdx.x; k < nsum; k += blockDim.x) {
    float t = 0.f;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) t += red[gg * 3 * cols + k];
    part[(int64_t)blockIdx.x * 3 * cols + k] = t;
  }
}

static int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// rows of more than 512 columns: two warps per row
static int ln_rw(int cols) { return cols > 512 ? 2 : 1; }

int ln_bwd_fused_ctas(int64_t rows, int cols) {
  const int G = 8 / ln_rw(cols);
  return (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(rows, G), 2 * sm_count()));
}

nnt_status launch_ln_bwd_fused(const float* dy, const float* x, const float* mean, const float* rstd,
                               const float* g, const float* resid, float* dx, void* dx_act,
                               int64_t rows, int cols, int act_dtype, float* part, int want_out,
                               cudaStream_t st) {
  NNT_CHECK_ARG(cols % 4 == 0 && cols > 0 && cols <= 1024,
                "fused layernorm bwd: cols must be a multiple of 4 in [4, 1024] (got %d)", cols);
  if (rows == 0) return NNT_OK;
  const int rw = ln_rw(cols);
  const int grid = ln_bwd_fused_ctas(rows, cols);
  const size_t smem = (size_t)(8 / rw) * 3 * cols * 4;
  const int mv = row_maxv(cols, 32 * rw);
  // the largest dynamic smem any call needs (1024 columns), allowed once per instantiation
#define NNT_LN_FUSED_LAUNCH(RWV)                                                                   \
  NNT_MAXV_DISPATCH(mv, {                                                                        \
    if (act_dtype == NNT_BF16) {                                                                 \
      auto k = ln_bwd_fused_kernel<RWV, MV, bf16>;                                              \
      static const cudaError_t attr =                                                            \
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 8 / RWV * 3 * 1024 * 4); \
      NNT_CUDA_TRY(attr);                                                                        \
      launch_pdl(k, grid, 256, smem, st, dy, x, mean, rstd, g, resid, dx, (bf16*)dx_act, rows, cols, part, \
                                 want_out);                                                      \
    } else {                                                                                     \
      auto k = ln_bwd_fused_kernel<RWV, MV, float>;                                             \
      static const cudaError_t attr =                                                            \
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 8 / RWV * 3 * 1024 * 4); \
      NNT_CUDA_TRY(attr);                                                                        \
      launch_pdl(k, grid, 256, smem, st, dy, x, mean, rstd, g, resid, dx, (float*)dx_act, rows, cols,      \
                                 part, want_out);                                                \
    }                                                                                            \
  })
  if (rw == 2) {
    NNT_LN_FUSED_LAUNCH(2);
  } else {
    NNT_LN_FUSED_LAUNCH(1);
  }
#undef NNT_LN_FUSED_LAUNCH
  return launch_check("layernorm_bwd_fused");
}

// Column sums of the layer-norm backward over a chunk of rows: sum dy*xhat
// (gain gradient), sum dy (shift gradient) and, when `out` is given, sum out
// (the bias gradient of the linear layer whose output gradient `out` is).
// CTA (strip of 128 columns, row chunk): each lane owns 4 columns (16-byte
// loads), warp w takes rows w, w+8, ...; the 8 warp sums are added in warp
// order. part: [nchunks][3][cols].
__global__ void ln_bwd_colsums_kernel(const float* __restrict__ dy, const float* __restrict__ x,
                                      const float* __restrict__ mean,
                                      const float* __restrict__ rstd, const float* __restrict__ out,
                                      int64_t rows, int cols, int64_t rows_per_chunk,
                                      float* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  __shared__ float4 red[3][8][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = (blockIdx.x * 32 + lane) * 4;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_chunk;
  const int64_t r1 = r0 + rows_per_chunk < rows ? r0 + rows_per_chunk : rows;
  float4 sg = make_float4(0.f, 0.f, 0.f, 0.f), sb = sg, so = sg;
  if (c < cols) {
#pragma unroll 2
    for (int64_t r = r0 + w; r < r1; r += 8) {
      const float4 d = load4(dy + r * cols + c);
      const float4 xv = load4(x + r * cols + c);
      const float mu = mean[r], rs = rstd[r];
      sg.x += d.x * ((xv.x - mu) * rs);
      sg.y += d.y * ((xv.y - mu) * rs);
      sg.z += d.z * ((xv.z - mu) * rs);
      sg.w += d.w * ((xv.w - mu) * rs);
      sb.x += d.x; sb.y += d.y; sb.z += d.z; sb.w += d.w;
      if (out) {
        const float4 o = load4(out + r * cols + c);
        so.x += o.x; so.y += o.y; so.z += o.z; so.w += o.w;
      }
    }
  }
  red[0][w][lane] = sg;
  red[1][w][lane] = sb;
  red[2][w][lane] = so;
  __syncthreads();
  if (w < 3 && c < cols) {
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = red[w][i][lane];
      t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
    }
    store4(part + ((int64_t)blockIdx.y * 3 + w) * cols + c, t);
  }
}

int64_t ln_colsum_chunks(int64_t rows) { return std::min<int64_t>(128, std::max<int64_t>(1, ceil_div(rows, 32))); }

nnt_status launch_ln_bwd_colsums(const float* dy, const float* x, const float* mean,
                                 const float* rstd, const float* out, int64_t rows, int cols,
                                 float* part, float* dg, float* db, float* dbias, int accumulate,
                                 cudaStream_t st) {
  NNT_CHECK_ARG(cols % 4 == 0, "layernorm colsums: cols must be a multiple of 4");
  const int64_t nch = ln_colsum_chunks(rows);
  const int64_t rpc = ceil_div(rows, nch);
  dim3 grid((unsigned)ceil_div(cols, 128), (unsigned)nch);
  launch_pdl(ln_bwd_colsums_kernel, grid, 256, 0, st, dy, x, mean, rstd, out, rows, cols, rpc, part);
  NNT_TRY(launch_check("ln_bwd_colsums"));
  return launch_sum_parts3(part, nch, cols, dg, db, out ? dbias : nullptr, accumulate, st);
}

// out[c] (+)= sum_p part[p*ld + c]. A CTA owns 32 columns; its kSumWarps warps
// take every kSumWarps-th partial row (lane = column, so each row read is one
// coalesced 128-byte segment; four rows in flight per warp) and the warp sums
// are added in warp order: a fixed summation order, independent of scheduling.
constexpr int kSumWarps = 32;

__global__ void __launch_bounds__(32 * kSumWarps) sum_parts_kernel(const float* __restrict__ part, int64_t nparts, int64_t cols,
                                 int64_t ld, float* __restrict__ out, int accumulate) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[kSumWarps][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = blockIdx.x * 32ll + lane;
  float s = 0.f;
  if (c < cols) {
    int64_t p = w;
    for (; p + 3 * kSumWarps < nparts; p += 4 * kSumWarps) {
      const float a0 = part[p * ld + c], a1 = part[(p + kSumWarps) * ld + c];
      const float a2 = part[(p + 2 * kSumWarps) * ld + c], a3 = part[(p + 3 * kSumWarps) * ld + c];
      s += a0;
      s += a1;
      s += a2;
      s += a3;
    }
    for (; p < nparts; p += kSumWarps) s += part[p * ld + c];
  }
  red[w][lane] = s;
  __syncthreads();
  if (w == 0 && c < cols) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < kSumWarps; ++i) t += red[i][lane];
    out[c] = accumulate ? out[c] + t : t;
  }
}

__global__ void __launch_bounds__(32 * kSumWarps) sum_parts3_kernel(const float* __restrict__ part, int64_t nparts, int64_t cols,
                                  float* o0, float* o1, float* o2, int accumulate) {
  pdl_wait();
  pdl_trigger();
  float* outs[3] = {o0, o1, o2};
  float* out = outs[blockIdx.y];
  if (!out) return;
  __shared__ float red[kSumWarps][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = blockIdx.x * 32ll + lane;
  const int64_t ld = 3 * cols;
  const float* p0 = part + blockIdx.y * cols;
  float s = 0.f;
  if (c < cols) {
    // four loads in flight per warp; each warp still adds its rows in a fixed order
    int64_t p = w;
    for (; p + 3 * kSumWarps < nparts; p += 4 * kSumWarps) {
      const float a0 = p0[p * ld + c], a1 = p0[(p + kSumWarps) * ld + c];
      const float a2 = p0[(p + 2 * kSumWarps) * ld + c], a3 = p0[(p + 3 * kSumWarps) * ld + c];
      s += a0;
      s += a1;
      s += a2;
      s += a3;
    }
    for (; p < nparts; p += kSumWarps) s += p0[p * ld + c];
  }
  red[w][lane] = s;
  __syncthreads();
  if (w == 0 && c < cols) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < kSumWarps; ++i) t += red[i][lane];
    out[c] = accumulate ? out[c] + t : t;
  }
}

nnt_status launch_sum_parts3(const float* part, int64_t nparts, int64_t cols, float* o0, float* o1,
                             float* o2, int accumulate, cudaStream_t st) {
  if (cols == 0) return NNT_OK;
  dim3 grid((unsigned)ceil_div(cols, 32), 3);
  launch_pdl(sum_parts3_kernel, grid, 32 * kSumWarps, 0, st, part, nparts, cols, o0, o1, o2, accumulate);
  return launch_check("sum_parts3");
}

nnt_status launch_sum_parts(const float* part, int64_t nparts, int64_t cols, int64_t ld,
                            float* out, int accumulate, cudaStream_t st) {
  if (cols == 0) return NNT_OK;
  launch_pdl(sum_parts_kernel, (unsigned)ceil_div(cols, 32), 32 * kSumWarps, 0, st, part, nparts, cols, ld, out,
                                                                  accumulate);
  return launch_check("sum_parts");
}

// Column sums in two fixed-order stages: CTA (strip of 128 columns, chunk of
// kColRows rows) adds its rows with 4 columns per lane and 8 warps in warp
// order into part[chunk][c]; launch_sum_parts adds the chunks.
static constexpr int kColRows = 64;
int64_t colsum_nparts(int64_t rows) { return ceil_div(rows, kColRows); }

template <typename T>
__global__ void colsum_part_kernel(const T* __restrict__ a, int64_t rows, int64_t cols, int64_t ld,
                                   float* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  __shared__ float4 red[8][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = ((int64_t)blockIdx.x * 32 + lane) * 4;
  const int64_t r0 = (int64_t)blockIdx.y * kColRows;
  const int64_t r1 = r0 + kColRows < rows ? r0 + kColRows : rows;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < cols) {
#pragma unroll 4
    for (int64_t r = r0 + w; r < r1; r += 8) {
      const float4 v = load4(a + r * ld + c);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
  }
  red[w][lane] = s;
  __syncthreads();
  if (w == 0 && c < cols) {
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = red[i][lane];
      t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
    }
    store4(part + (int64_t)blockIdx.y * cols + c, t);
  }
}

nnt_status launch_colsum(const void* a, int a_dtype, int64_t rows, int64_t cols, int64_t ld,
                         float* part, float* out, int accumulate, cudaStream_t st) {
  if (cols == 0) return NNT_OK;
  NNT_CHECK_ARG(cols % 4 == 0 && ld % 4 == 0, "colsum: cols and ld must be multiples of 4");
  const int64_t np = colsum_nparts(rows);
  NNT_CHECK_ARG(np < 65536, "colsum: too many rows");
  dim3 grid((unsigned)ceil_div(cols, 128), (unsigned)np);
  if (a_dtype == NNT_BF16)
    launch_pdl(colsum_part_kernel<bf16>, grid, 256, 0, st, (const bf16*)a, rows, cols, ld, part);
  else
    launch_pdl(colsum_part_kernel<float>, grid, 256, 0, st, (const float*)a, rows, cols, ld, part);
  NNT_TRY(launch_check("colsum_part"));
  return launch_sum_parts(part, np, cols, cols, out, accumulate, st);
}

// =====================================================================
// causal softmax over score rows (scores already scaled by 1/sqrt(hd))
// =====================================================================

// One warp per score row. Rows of up to 1024 causal entries stay in registers
// (8 float4 per lane); longer rows are swept in 1024-entry segments with an
// online (max, sum) and re-read (from L2) for the output. Only the q+1 valid
// entries are loaded and exponentiated; entries past q up to the 128-key block
// boundary are written as 0. No block-level barriers.
template <typename T>
__global__ void __launch_bounds__(256) softmax_fwd_kernel(const float* __restrict__ s,
                                                          T* __restrict__ p, int64_t S, ZMap zm,
                                                          int nz, int q0, int nq) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= (int64_t)nz * nq) return;
  const int q = q0 + (int)(r % nq);
  const int64_t z = zm.z((int)(r / nq));
  const float* sr = s + (z * S + q) * S;
  T* pr = p + (z * S + q) * S;
  const int valid = q + 1;
  const int wend = (int)std::min<int64_t>(S, round_up(valid, kCausalBlock));
  const int nvv = (valid + 3) >> 2;  // float4 groups holding valid entries
  const int nw = wend >> 2;
  if (nvv <= 256) {
    float4 v[8];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < nvv) {
        v[i] = load4_stream(sr + 4 * c);
        if (4 * c + 1 > q) v[i].y = -INFINITY;
        if (4 * c + 2 > q) v[i].z = -INFINITY;
        if (4 * c + 3 > q) v[i].w = -INFINITY;
        mx = fmaxf(mx, fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w)));
      }
    }
    mx = warp_max(mx);
    const float ms = mx * kLog2e;
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < nvv) {
        v[i].x = exp2f(v[i].x * kLog2e - ms);
        v[i].y = exp2f(v[i].y * kLog2e - ms);
        v[i].z = exp2f(v[i].z * kLog2e - ms);
        v[i].w = exp2f(v[i].w * kLog2e - ms);
        sum += (v[i].x + v[i].y) + (v[i].z + v[i].w);
      }
    }
    const float inv = 1.0f / warp_sum(sum);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < nvv) store4(pr + 4 * c, make_float4(v[i].x * inv, v[i].y * inv, v[i].z * inv, v[i].w * inv));
      else if (c < nw) store4(pr + 4 * c, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    return;
  }
  // long rows: online max/sum over the valid entries, then a second sweep
  float mx = -INFINITY, sum = 0.f;
  for (int c = lane; c < nvv; c += 32) {
    float4 v = load4(sr + 4 * c);
    if (4 * c + 1 > q) v.y = -INFINITY;
    if (4 * c + 2 > q) v.z = -INFINITY;
    if (4 * c + 3 > q) v.w = -INFINITY;
    const float lm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (lm > mx) {
      sum *= exp2f((mx - lm) * kLog2e);
      mx = lm;
    }
    sum += exp2f((v.x - mx) * kLog2e) + exp2f((v.y - mx) * kLog2e) + exp2f((v.z - mx) * kLog2e) +
           exp2f((v.w - mx) * kLog2e);
  }
  const float M = warp_max(mx);
  sum = (mx == -INFINITY) ? 0.f : sum * exp2f((mx - M) * kLog2e);
  const float inv = 1.0f / warp_sum(sum);
  const float ms = M * kLog2e;
  for (int c = lane; c < nw; c += 32) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < nvv) {
      const float4 v = load4(sr + 4 * c);
      o.x = exp2f(v.x * kLog2e - ms) * inv;
      o.y = 4 * c + 1 > q ? 0.f : exp2f(v.y * kLog2e - ms) * inv;
      o.z = 4 * c + 2 > q ? 0.f : exp2f(v.z * kLog2e - ms) * inv;
      o.w = 4 * c + 3 > q ? 0.f : exp2f(v.w * kLog2e - ms) * inv;
    }
    store4(pr + 4 * c, o);
  }
}

// Four entries of a probability row kept in their storage type (bf16 rows
// stay packed in two registers) and widened when used.
template <typename T> struct Raw4;
template <> struct Raw4<float> {
  float4 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ float4 get() const { return v; }
};
template <> struct Raw4<bf16> {
  uint2 u;
  __device__ __forceinline__ void load(const bf16* p) { u = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ float4 get() const {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
};

// dS = scale * P * (dP - rowsum(dP * P)) over the valid entries, 0 beyond q up
// to the block boundary; one warp per row, as the forward. The register path
// keeps P (in its storage type) and P*dP, so dS = scale * (P*dP - P*dot).
template <typename T>
__global__ void __launch_bounds__(256, 3) softmax_bwd_kernel(const T* __restrict__ p,
                                                             const float* __restrict__ dp,
                                                             T* __restrict__ ds, int64_t S, ZMap zm,
                                                             int nz, int q0, int nq, float scale) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= (int64_t)nz * nq) return;
  const int q = q0 + (int)(r % nq);
  const int64_t z = zm.z((int)(r / nq));
  const int64_t off = (z * S + q) * S;
  const int valid = q + 1;
  const int wend = (int)std::min<int64_t>(S, round_up(valid, kCausalBlock));
  const int nvv = (valid + 3) >> 2;
  const int nw = wend >> 2;
  auto masked = [q](float4& a, int c) {
    if (4 * c + 1 > q) a.y = 0.f;
    if (4 * c + 2 > q) a.z = 0.f;
    if (4 * c + 3 > q) a.w = 0.f;
  };
  if (nvv <= 256) {
    Raw4<T> pr[8];
    float4 pd[8];
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < nvv) {
        pr[i].load(p + off + 4 * c);
        pd[i] = load4_stream(dp + off + 4 * c);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < nvv) {
        float4 a = pr[i].get();
        masked(a, c);
        masked(pd[i], c);  // P is 0 past q; clear dP there too so 0*garbage cannot leak in
        pd[i] = make_float4(a.x * pd[i].x, a.y * pd[i].y, a.z * pd[i].z, a.w * pd[i].w);
        dot += (pd[i].x + pd[i].y) + (pd[i].z + pd[i].w);
      }
    }
    dot = warp_sum(dot);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i;
      if (c < nvv) {
        float4 a = pr[i].get();
        masked(a, c);
        store4(ds + off + 4 * c, make_float4(scale * (pd[i].x - a.x * dot), scale * (pd[i].y - a.y * dot),
                                             scale * (pd[i].z - a.z * dot), scale * (pd[i].w - a.w * dot)));
      } else if (c < nw) {
        store4(ds + off + 4 * c, make_float4(0.f, 0.f, 0.f, 0.f));
      }
    }
    return;
  }
  float dot = 0.f;
  for (int c = lane; c < nvv; c += 32) {
    float4 a = load4(p + off + 4 * c), b = load4(dp + off + 4 * c);
    masked(a, c);
    masked(b, c);
    dot += (a.x * b.x + a.y * b.y) + (a.z * b.z + a.w * b.w);
  }
  dot = warp_sum(dot);
  for (int c = lane; c < nw; c += 32) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < nvv) {
      float4 a = load4(p + off + 4 * c), b = load4(dp + off + 4 * c);
      masked(a, c);
      masked(b, c);
      o = make_float4(scale * a.x * (b.x - dot), scale * a.y * (b.y - dot), scale * a.z * (b.z - dot),
                      scale * a.w * (b.w - dot));
    }
    store4(ds + off + 4 * c, o);
  }
}

nnt_status launch_softmax_fwd(const float* s, void* p, int64_t S, ZMap zm, int nz, int q0, int nq,
                              int act_dtype, cudaStream_t st) {
  NNT_CHECK_ARG(S % 4 == 0 && S > 0, "softmax: seq must be a positive multiple of 4");
  const int64_t rows = (int64_t)nz * nq;
  if (rows == 0) return NNT_OK;
  const int64_t grid = ceil_div(rows, 8);
  if (act_dtype == NNT_BF16)
    launch_pdl(softmax_fwd_kernel<bf16>, grid, 256, 0, st, s, (bf16*)p, S, zm, nz, q0, nq);
  else
    launch_pdl(softmax_fwd_kernel<float>, grid, 256, 0, st, s, (float*)p, S, zm, nz, q0, nq);
  return launch_check("softmax_fwd");
}

nnt_status launch_softmax_bwd(const void* p, const float* dp, void* ds, int64_t S, ZMap zm, int nz,
                              int q0, int nq, float scale, int act_dtype, cudaStream_t st) {
  NNT_CHECK_ARG(S % 4 == 0 && S > 0, "softmax bwd: seq must be a positive multiple of 4");
  const int64_t rows = (int64_t)nz * nq;
  if (rows == 0) return NNT_OK;
  const int64_t grid = ceil_div(rows, 8);
  if (act_dtype == NNT_BF16)
    launch_pdl(softmax_bwd_kernel<bf16>, grid, 256, 0, st, (const bf16*)p, dp, (bf16*)ds, S, zm, nz, q0, nq, scale);
  else
    launch_pdl(softmax_bwd_kernel<float>, grid, 256, 0, st, (const float*)p, dp, (float*)ds, S, zm, nz, q0, nq, scale);
  return launch_check("softmax_bwd");
}

// =====================================================================
// GELU (tanh form)
// =====================================================================

__device__ __forceinline__ float gelu_f(float u) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  return 0.5f * u * (1.0f + tanhf(c * (u + a * u * u * u)));
}
__device__ __forceinline__ float gelu_grad_f(float u) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  const float t = tanhf(c * (u + a * u * u * u));
  return 0.5f * (1.0f + t) + 0.5f * u * (1.0f - t * t) * c * (1.0f + 3.0f * a * u * u);
}

template <typename T>
__global__ void gelu_fwd_kernel(const float* __restrict__ u, T* __restrict__ g, int64_t n4) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 x = load4_stream(u + 4 * i);
    store4(g + 4 * i, make_float4(gelu_f(x.x), gelu_f(x.y), gelu_f(x.z), gelu_f(x.w)));
  }
}
template <typename T>
__global__ void gelu_bwd_kernel(const T* __restrict__ dg, const float* __restrict__ u,
                                T* __restrict__ du, int64_t n4) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 x = load4_stream(u + 4 * i);
    float4 d = load4(dg + 4 * i);
    store4(du + 4 * i, make_float4(d.x * gelu_grad_f(x.x), d.y * gelu_grad_f(x.y),
                                   d.z * gelu_grad_f(x.z), d.w * gelu_grad_f(x.w)));
  }
}

static int elementwise_grid(int64_t n4) {
  return (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n4, 256), 152 * 8));
}

nnt_status launch_gelu_fwd(const float* u, void* g, int64_t n, int act_dtype, cudaStream_t st) {
  NNT_CHECK_ARG(n % 4 == 0, "gelu: n must be a multiple of 4");
  if (n == 0) return NNT_OK;
  if (act_dtype == NNT_BF16)
    launch_pdl(gelu_fwd_kernel<bf16>, elementwise_grid(n / 4), 256, 0, st, u, (bf16*)g, n / 4);
  else
    launch_pdl(gelu_fwd_kernel<float>, elementwise_grid(n / 4), 256, 0, st, u, (float*)g, n / 4);
  return launch_check("gelu_fwd");
}
nnt_status launch_gelu_bwd(const void* dg, const float* u, void* du, int64_t n, int act_dtype,
                           cudaStream_t st) {
  NNT_CHECK_ARG(n % 4 == 0, "gelu bwd: n must be a multiple of 4");
  if (n == 0) return NNT_OK;
  if (act_dtype == NNT_BF16)
    launch_pdl(gelu_bwd_kernel<bf16>, elementwise_grid(n / 4), 256, 0, st, (const bf16*)dg, u, (bf16*)du, n / 4);
  else
    launch_pdl(gelu_bwd_kernel<float>, elementwise_grid(n / 4), 256, 0, st, (const float*)dg, u, (float*)du, n / 4);
  return launch_check("gelu_bwd");
}

// =====================================================================
// cross-entropy (mean over tokens) + dlogits
// =====================================================================

// Each CTA takes rows in turn: pass 1 keeps a running (max, sum of exp) per
// thread and merges them across the CTA; pass 2 re-reads the row (from L2) and
// writes dz = (exp(z - lse) - onehot) * inv_rows, zero in the padding columns.
template <typename T>
__global__ void __launch_bounds__(512) cross_entropy_kernel(
    const float* __restrict__ z, int64_t ldz, int64_t r0, int64_t nrows, int64_t cols,
    const uint16_t* __restrict__ tok_ids, TokMap tm, const uint16_t* __restrict__ tgt,
    int64_t tgt_stride, T* __restrict__ dz, int64_t lddz, float* __restrict__ row_loss,
    float inv_rows) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red_m[32], red_s[32];
  for (int64_t rr = blockIdx.x; rr < nrows; rr += gridDim.x) {
  const int64_t r = r0 + rr;
  const float* zr = z + r * ldz;
  const int64_t n4 = cols >> 2;  // full float4s
  float m = -INFINITY, s = 0.f;
  // four float4 per thread in flight per iteration, then the online update
  const int64_t bs = blockDim.x;
  for (int64_t i0 = threadIdx.x; i0 < n4; i0 += 4 * bs) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = (i0 + u * bs < n4) ? load4(zr + 4 * (i0 + u * bs))
                                : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float lm = m;
#pragma unroll
    for (int u = 0; u < 4; ++u) lm = fmaxf(lm, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
    if (lm > m) {
      s *= exp2f((m - lm) * kLog2e);
      m = lm;
    }
    const float ms = m * kLog2e;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      s += exp2f(v[u].x * kLog2e - ms) + exp2f(v[u].y * kLog2e - ms) + exp2f(v[u].z * kLog2e - ms) +
           exp2f(v[u].w * kLog2e - ms);
  }
  for (int64_t c = 4 * n4 + threadIdx.x; c < cols; c += blockDim.x) {
    float v = zr[c];
    if (v > m) {
      s *= exp2f((m - v) * kLog2e);
      m = v;
    }
    s += exp2f((v - m) * kLog2e);
  }
  // merge (m, s) over the CTA
  float wm = warp_max(m);
  s = (m == -INFINITY) ? 0.f : s * exp2f((m - wm) * kLog2e);
  s = warp_sum(s);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red_m[w] = wm;
    red_s[w] = s;
  }
  __syncthreads();
  float M = -INFINITY;
  for (int i = 0; i < nw; ++i) M = fmaxf(M, red_m[i]);
  float SUM = 0.f;
  for (int i = 0; i < nw; ++i) SUM += red_s[i] * exp2f((red_m[i] - M) * kLog2e);
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
    if (threadIdx.x == 0) atomicOr(&g_device_error, DEVERR_TOKEN_RANGE);
    y = 0;
  }
  if (threadIdx.x == 0) row_loss[r] = lse - zr[y];
  const float ls = lse * kLog2e;
  T* dr = dz + r * lddz;
#pragma unroll 4
  for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
    float4 v = load4(zr + 4 * i);
    float4 o;
    o.x = exp2f(v.x * kLog2e - ls);
    o.y = exp2f(v.y * kLog2e - ls);
    o.z = exp2f(v.z * kLog2e - ls);
    o.w = exp2f(v.w * kLog2e - ls);
    const int64_t c0 = 4 * i;
    if (y >= c0 && y < c0 + 4) {
      const int k = (int)(y - c0);
      if (k == 0) o.x -= 1.f;
      else if (k == 1) o.y -= 1.f;
      else if (k == 2) o.z -= 1.f;
      else o.w -= 1.f;
    }
    o.x *= inv_rows;
    o.y *= inv_rows;
    o.z *= inv_rows;
    o.w *= inv_rows;
    store4(dr + c0, o);
  }
  for (int64_t c = 4 * n4 + threadIdx.x; c < lddz; c += blockDim.x) {
    float o = 0.f;
    if (c < cols) o = (exp2f(zr[c] * kLog2e - ls) - (c == y ? 1.f : 0.f)) * inv_rows;
    dr[c] = from_f<T>(o);
  }
  __syncthreads();  // red_m / red_s are reused by the next row
  }
}

nnt_status launch_cross_entropy(const float* z, int64_t ldz, int64_t r0, int64_t nrows,
                                int64_t cols, const uint16_t* tok_ids, TokMap tm,
                                const uint16_t* tgt, int64_t tgt_stride, void* dz, int64_t lddz,
                                float* row_loss, float inv_rows, int act_dtype, cudaStream_t st) {
  NNT_CHECK_ARG(ldz % 4 == 0 && lddz % 4 == 0 && ldz >= cols && lddz >= cols,
                "cross entropy: leading dimensions must be multiples of 4 and >= cols");
  if (nrows == 0) return NNT_OK;
  // Rows from 32768 logits up to what shared memory holds take the cluster-pair
  // kernel (one HBM read); shorter rows stay in L2 between the two passes here,
  // which measured faster. NNT_CE_KERNEL=pair or twopass forces one of them.
  const char* force_env = getenv("NNT_CE_KERNEL");
  const char* force = force_env ? force_env : "";
  const bool pair_ok = cross_entropy_smem_fits(cols) && reinterpret_cast<uintptr_t>(z) % 16 == 0;
  const bool pair = pair_ok && (strcmp(force, "pair") == 0 ||
                                (strcmp(force, "twopass") != 0 && cols >= 32768));
  if (pair)
    return launch_cross_entropy_smem(z, ldz, r0, nrows, cols, tok_ids, tm, tgt, tgt_stride, dz, lddz,
                                     row_loss, inv_rows, act_dtype, sm_count(), st);
  // two CTAs per SM walk the rows, so the rows being re-read (pass 2) stay in L2
  const unsigned grid = (unsigned)std::min<int64_t>(nrows, 2 * 152);
  if (act_dtype == NNT_BF16)
    launch_pdl(cross_entropy_kernel<bf16>, grid, 512, 0, st, 
        z, ldz, r0, nrows, cols, tok_ids, tm, tgt, tgt_stride, (bf16*)dz, lddz, row_loss, inv_rows);
  else
    launch_pdl(cross_entropy_kernel<float>, grid, 512, 0, st, 
        z, ldz, r0, nrows, cols, tok_ids, tm, tgt, tgt_stride, (float*)dz, lddz, row_loss, inv_rows);
  return launch_check("cross_entropy");
}

// loss = (sum of row losses in a fixed order, in double) / rows
__global__ void mean_loss_kernel(const float* __restrict__ row_loss, int64_t rows,
                                 float* __restrict__ loss) {
  pdl_wait();
  pdl_trigger();
  __shared__ double red[1024];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < rows; i += blockDim.x) s += (double)row_loss[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = (float)(red[0] / (double)rows);
}

nnt_status launch_mean_loss(const float* row_loss, int64_t rows, float* loss, cudaStream_t st) {
  launch_pdl(mean_loss_kernel, 1, 1024, 0, st, row_loss, rows, loss);
  return launch_check("mean_loss");
}

// =====================================================================
// AdamW (decoupled weight decay), fp32 state, optional bf16 copy out
// =====================================================================

// Every operation is rounded explicitly (no contraction left to the compiler),
// so each instantiation of the kernel below -- and thus the device-moment and
// host-moment paths -- produces the same bits for the same inputs.
__device__ __forceinline__ void adamw_one(float& w, float g, float& m, float& v, float lr, float b1,
                                          float b2, float eps, float wd, float bc1, float bc2) {
  m = __fmaf_rn(b1, m, __fmul_rn(1.f - b1, g));
  v = __fmaf_rn(b2, v, __fmul_rn(__fmul_rn(1.f - b2, g), g));
  const float mhat = __fdiv_rn(m, bc1);
  const float vhat = __fdiv_rn(v, bc2);
  const float decay = __fmul_rn(__fmul_rn(lr, wd), w);
  const float step = __fdiv_rn(__fmul_rn(lr, mhat), __fadd_rn(__fsqrt_rn(vhat), eps));
  w = __fsub_rn(__fsub_rn(w, decay), step);
}

// hyper (optional, device): lr, beta1, beta2, eps, wd, bc1, bc2, gscale --
// overrides the by-value arguments so a captured graph can be replayed with new
// values. The gradient used is g * gscale (1 for a single backward; 1/k for the
// sum of k accumulated minibatch gradients, i.e. their mean).
// UNROLL float4 groups per thread per iteration: all their loads are issued
// before any math, which keeps enough bytes in flight when m and v sit behind
// the slower host link.
template <int UNROLL>
__global__ void adamw_kernel(float* __restrict__ w, const float* __restrict__ g,
                             float* __restrict__ m, float* __restrict__ v, bf16* __restrict__ wb,
                             int64_t n, float lr, float b1, float b2, float eps, float wd,
                             float bc1, float bc2, const float* __restrict__ hyper) {
  pdl_wait();
  pdl_trigger();
  float gs = 1.f;
  if (hyper) {
    lr = hyper[0]; b1 = hyper[1]; b2 = hyper[2]; eps = hyper[3]; wd = hyper[4];
    bc1 = hyper[5]; bc2 = hyper[6]; gs = hyper[7];
  }
  const int64_t n4 = n >> 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i0 < n4; i0 += stride * UNROLL) {
    float4 W[UNROLL], G[UNROLL], M[UNROLL], V[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n4) {
        W[u] = load4_stream(w + 4 * i);
        G[u] = load4_stream(g + 4 * i);
        M[u] = load4_stream(m + 4 * i);
        V[u] = load4_stream(v + 4 * i);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n4) {
        adamw_one(W[u].x, __fmul_rn(G[u].x, gs), M[u].x, V[u].x, lr, b1, b2, eps, wd, bc1, bc2);
        adamw_one(W[u].y, __fmul_rn(G[u].y, gs), M[u].y, V[u].y, lr, b1, b2, eps, wd, bc1, bc2);
        adamw_one(W[u].z, __fmul_rn(G[u].z, gs), M[u].z, V[u].z, lr, b1, b2, eps, wd, bc1, bc2);
        adamw_one(W[u].w, __fmul_rn(G[u].w, gs), M[u].w, V[u].w, lr, b1, b2, eps, wd, bc1, bc2);
        store4_stream(w + 4 * i, W[u]);
        store4_stream(m + 4 * i, M[u]);
        store4_stream(v + 4 * i, V[u]);
        if (wb) store4(wb + 4 * i, W[u]);
      }
    }
  }
  // tail
  const int64_t t = 4 * n4 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t < n) {
    float W = w[t], M = m[t], V = v[t];
    adamw_one(W, __fmul_rn(g[t], gs), M, V, lr, b1, b2, eps, wd, bc1, bc2);
    w[t] = W;
    m[t] = M;
    v[t] = V;
    if (wb) wb[t] = __float2bfloat16_rn(W);
  }
}

nnt_status launch_adamw(float* w, const float* g, float* m, float* v, bf16* w_bf16, int64_t n,
                        float lr, float b1, float b2, float eps, float wd, float bc1, float bc2,
                        cudaStream_t st) {
  if (n == 0) return NNT_OK;
  NNT_CHECK_ARG(((uintptr_t)w | (uintptr_t)g | (uintptr_t)m | (uintptr_t)v) % 16 == 0 &&
                    ((uintptr_t)w_bf16) % 8 == 0,
                "adamw: buffers must be 16-byte aligned (bf16 copy 8-byte)");
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n / 4 + 1, 256), 152 * 8));
  launch_pdl(adamw_kernel<1>, grid, 256, 0, st, w, g, m, v, w_bf16, n, lr, b1, b2, eps, wd, bc1, bc2, nullptr);
  return launch_check("adamw");
}

nnt_status launch_adamw_dev(float* w, const float* g, float* m, float* v, bf16* w_bf16, int64_t n,
                            const float* hyper_dev, cudaStream_t st, int max_ctas) {
  if (n == 0) return NNT_OK;
  if (max_ctas > 0) {
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n / 4 + 1, 256 * 4), max_ctas));
    launch_pdl(adamw_kernel<4>, grid, 256, 0, st, w, g, m, v, w_bf16, n, 0, 0, 0, 0, 0, 1, 1, hyper_dev);
  } else {
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n / 4 + 1, 256), 152 * 8));
    launch_pdl(adamw_kernel<1>, grid, 256, 0, st, w, g, m, v, w_bf16, n, 0, 0, 0, 0, 0, 1, 1, hyper_dev);
  }
  return launch_check("adamw");
}

// =====================================================================
// init: splitmix64 counter stream + Box-Muller (same recipe as the host
// generator: key = sm(sm(seed) ^ stream), bits_i = sm(key + i),
// u = ((bits >> 11) + 0.5) * 2^-53, pairs (2j, 2j+1) -> cos / sin branch)
// =====================================================================

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void init_normal_kernel(float* __restrict__ w, int64_t n, uint64_t key, double std) {
  pdl_wait();
  pdl_trigger();
  const int64_t npairs = (n + 1) / 2;
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < npairs;
       j += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t b1 = splitmix64(key + (uint64_t)(2 * j));
    const uint64_t b2 = splitmix64(key + (uint64_t)(2 * j + 1));
    const double u1 = ((double)(b1 >> 11) + 0.5) * 0x1.0p-53;
    const double u2 = ((double)(b2 >> 11) + 0.5) * 0x1.0p-53;
    const double r = sqrt(-2.0 * log(u1));
    const double th = 6.283185307179586 * u2;
    double sn, cs;
    sincos(th, &sn, &cs);
    w[2 * j] = (float)(r * cs * std);
    if (2 * j + 1 < n) w[2 * j + 1] = (float)(r * sn * std);
  }
}

static uint64_t host_splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

nnt_status launch_init_normal(float* w, int64_t n, uint64_t seed, uint64_t stream_id, double std,
                              cudaStream_t st) {
  if (n == 0) return NNT_OK;
  const uint64_t key = host_splitmix64(host_splitmix64(seed) ^ stream_id);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div((n + 1) / 2, 256), 152 * 16));
  launch_pdl(init_normal_kernel, grid, 256, 0, st, w, n, key, std);
  return launch_check("init_normal");
}

__global__ void fill_kernel(float* __restrict__ w, int64_t n, float value) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    w[i] = value;
}
nnt_status launch_fill(float* w, int64_t n, float value, cudaStream_t st) {
  if (n == 0) return NNT_OK;
  launch_pdl(fill_kernel, (int)std::min<int64_t>(ceil_div(n, 256), 152 * 16), 256, 0, st, w, n, value);
  return launch_check("fill");
}

__global__ void cast_bf16_kernel(const float* __restrict__ s, bf16* __restrict__ d, int64_t n) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    d[i] = __float2bfloat16_rn(s[i]);
}
nnt_status launch_cast_bf16(const float* src, bf16* dst, int64_t n, cudaStream_t st) {
  if (n == 0) return NNT_OK;
  launch_pdl(cast_bf16_kernel, (int)std::min<int64_t>(ceil_div(n, 256), 152 * 16), 256, 0, st, src, dst, n);
  return launch_check("cast_bf16");
}

__global__ void check_tokens_kernel(const uint16_t* __restrict__ ids, int64_t n, int vocab) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    if (ids[i] >= vocab) atomicOr(&g_device_error, DEVERR_TOKEN_RANGE);
}
nnt_status launch_check_tokens(const uint16_t* ids, int64_t n, int vocab, cudaStream_t st) {
  if (n == 0) return NNT_OK;
  launch_pdl(check_tokens_kernel, (int)std::min<int64_t>(ceil_div(n, 256), 152), 256, 0, st, ids, n, vocab);
  return launch_check("check_tokens");
}

}  // namespace nnt
