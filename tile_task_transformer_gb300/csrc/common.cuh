// Shared device/host helpers of libnnt (no torch, no oracle code).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nnt.h"

namespace nnt {

// ---------------------------------------------------------------- errors
// Device error word: kernels OR a code in, the host reads and clears it.
enum DeviceError : uint32_t {
  DEVERR_TOKEN_RANGE = 1u << 0,   // token id >= vocab
  DEVERR_WAIT_TIMEOUT = 1u << 1,  // a bounded mbarrier wait ran out
  DEVERR_BAD_TILE = 1u << 2,      // a tile index out of range (checks build)
  DEVERR_SMEM_ALIGN = 1u << 3,    // dynamic shared memory not at the alignment a kernel needs
};
// Device address of the error word on the current device (for kernels in other
// translation units), and a stream-ordered read-and-clear of it.
uint32_t* device_error_word();
nnt_status read_and_clear_device_error(uint32_t* code_host, cudaStream_t st);

// Host-side fault injection (nnt_set_fault_injection): counts one call of
// `kind`; true for the call that the armed count designates.
enum FaultKind : int {
  FAULT_DEVICE_ALLOC = NNT_FAULT_DEVICE_ALLOC,
  FAULT_HOST_ALLOC = NNT_FAULT_HOST_ALLOC,
  FAULT_COPY = NNT_FAULT_COPY,
  FAULT_EVENT_WAIT = NNT_FAULT_EVENT_WAIT,
  FAULT_KINDS = 4
};
bool fault_hit(FaultKind kind);

const char* status_name(nnt_status s);
void set_thread_error(const char* fmt, ...);
// Status of the last kernel launch on this thread (error text set on failure).
inline nnt_status launch_check(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_thread_error("launch of %s failed: %s", what, cudaGetErrorString(e));
    return NNT_ERR_CUDA;
  }
  return NNT_OK;
}
const char* thread_error();

#define NNT_CUDA_TRY(expr)                                                        \
  do {                                                                            \
    cudaError_t e_ = (expr);                                                      \
    if (e_ != cudaSuccess) {                                                      \
      ::nnt::set_thread_error("%s failed: %s (%s:%d)", #expr, cudaGetErrorString(e_), \
                              __FILE__, __LINE__);                                \
      return NNT_ERR_CUDA;                                                        \
    }                                                                             \
  } while (0)

#define NNT_TRY(expr)                      \
  do {                                     \
    nnt_status s_ = (expr);                \
    if (s_ != NNT_OK) return s_;           \
  } while (0)

#define NNT_CHECK_ARG(cond, ...)                  \
  do {                                            \
    if (!(cond)) {                                \
      ::nnt::set_thread_error(__VA_ARGS__);       \
      return NNT_ERR_INVALID_ARG;                 \
    }                                             \
  } while (0)

// ---------------------------------------------------------------- launches
// Programmatic dependent launch: the library's kernels are launched with
// launch_pdl, which lets a kernel start (and run its prologue) while the
// previous kernel on its stream finishes. Each kernel calls pdl_wait() before
// its first access to global memory -- griddepcontrol.wait returns once the
// preceding grids have completed and their writes are visible -- and then
// pdl_trigger(), after which the next kernel may launch. NNT_PDL=0 in the
// environment launches without the attribute (the waits are then no-ops).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
bool pdl_enabled();

template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- types
typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// 4-element vector load/store of an activation type (float: 16 B, bf16: 8 B).
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const bf16* p) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// streaming (evict-first) variants for data read or written exactly once
__device__ __forceinline__ float4 load4_stream(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void store4_stream(float* p, float4 v) {
  __stcs(reinterpret_cast<float4*>(p), v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over a group of TPR consecutive threads (TPR a power of two, 1..1024).
// Groups of more than 32 threads use `red` (TPR/32 floats per group, in shared
// memory) and a barrier, so every thread of the CTA must call it.
template <int TPR>
__device__ __forceinline__ float group_sum(float v, float* red) {
  v = warp_sum(v);
  if constexpr (TPR > 32) {
    const int nw = TPR / 32;
    const int grp = threadIdx.x / TPR;
    const int w = (threadIdx.x % TPR) / 32;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[grp * nw + w] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < nw; ++i) s += red[grp * nw + i];
    v = s;
  }
  return v;
}
template <int TPR>
__device__ __forceinline__ float group_max(float v, float* red) {
  v = warp_max(v);
  if constexpr (TPR > 32) {
    const int nw = TPR / 32;
    const int grp = threadIdx.x / TPR;
    const int w = (threadIdx.x % TPR) / 32;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[grp * nw + w] = v;
    __syncthreads();
    float s = -INFINITY;
#pragma unroll
    for (int i = 0; i < nw; ++i) s = fmaxf(s, red[grp * nw + i]);
    v = s;
  }
  return v;
}

// ---------------------------------------------------------------- token tiles
// Token (b, s) -> storage row. Token tiles (batch_tile x seq_tile) are stored
// as contiguous row blocks, tile-major: tile (bt, st) occupies rows
// [(bt*n_st + st) * tb*ts, +tb*ts), inside it row bl*ts + sl.
struct TokMap {
  int S, tb, ts, n_st;
  __host__ __device__ __forceinline__ int64_t row(int b, int s) const {
    int bt = b / tb, bl = b - bt * tb, st = s / ts, sl = s - st * ts;
    return ((int64_t)(bt * n_st + st) * tb + bl) * ts + sl;
  }
  // inverse: storage row -> (b, s)
  __host__ __device__ __forceinline__ void bs(int64_t r, int& b, int& s) const {
    int64_t tile = r / (tb * ts);
    int in = (int)(r - tile * tb * ts);
    int bt = (int)(tile / n_st), st = (int)(tile - (int64_t)bt * n_st);
    b = bt * tb + in / ts;
    s = st * ts + in % ts;
  }
};

constexpr int kCausalBlock = 128;  // key-block granularity of the causal score tiles

__host__ __device__ __forceinline__ int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace nnt

namespace nnt {
// Batch index i of a batched attention task -> (sequence b, head h); the task
// covers sequences [b0, b0 + i/nh ...) and heads [h0, h0 + nh) of H heads.
struct ZMap {
  int b0, h0, nh, H;
  __host__ __device__ __forceinline__ int b(int i) const { return b0 + i / nh; }
  __host__ __device__ __forceinline__ int h(int i) const { return h0 + i % nh; }
  __host__ __device__ __forceinline__ int64_t z(int i) const { return (int64_t)b(i) * H + h(i); }
};
}  // namespace nnt
