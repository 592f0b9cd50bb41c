// Allocation-free variant of the embedding scatter-add (nnt_op_embedding_bwd).
//
// Some callers cannot allocate device memory while they run: hosts that own
// all device memory through their own allocator or a fixed budget (a library
// allocation would bypass it or fail), and latency-critical loops where the
// implicit device synchronisation of cudaMalloc/cudaFree is not acceptable.
// nnt_op_embedding_bwd takes its scratch
// (the token sort keys) from a library-owned buffer that it grows with
// cudaMalloc; this variant instead uses a fixed array compiled into the
// library, so it never calls cudaMalloc, cudaFree or any allocating routine.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

using namespace nnt;

namespace {

// Largest batch*seq the fixed scratch serves: one 32-bit sort key per token,
// as many tokens as one CTA of the token sort orders (64 KiB of keys).
constexpr int kNoAllocMaxTokens = kTokenSortBlock;

// The scratch itself: 64 KiB in every device's global memory for as long as
// the library is loaded. In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint32_t g_noalloc_sort_keys[kNoAllocMaxTokens];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
std::atomic<uint32_t*> g_keys_dev[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on each device does this set-up). Later calls
// read it without taking the lock.
nnt_status keys_on_current_device(uint32_t** out) {
  int dev = 0;
  NNT_CUDA_TRY(cudaGetDevice(&dev));
  NNT_CHECK_ARG(dev >= 0 && dev < kMaxDevices, "device ordinal %d out of range", dev);
  uint32_t* k = g_keys_dev[dev].load(std::memory_order_acquire);
  if (!k) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    k = g_keys_dev[dev].load(std::memory_order_relaxed);
    if (!k) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_sort_keys);
      if (e != cudaSuccess || !p) {
        set_thread_error("cudaGetSymbolAddress of the fixed scratch failed: %s", cudaGetErrorString(e));
        return NNT_ERR_CUDA;
      }
      k = static_cast<uint32_t*>(p);
      g_keys_dev[dev].store(k, std::memory_order_release);
    }
  }
  *out = k;
  return NNT_OK;
}

}  // namespace

extern "C" nnt_status nnt_op_embedding_bwd_noalloc(const uint16_t* ids_dev, int64_t ids_stride,
                                                   const float* dx_dev, float* dwte_dev,
                                                   float* dwpe_dev, int64_t batch, int64_t seq,
                                                   int64_t d, int64_t vocab, void* stream) {
  NNT_CHECK_ARG(ids_dev && dx_dev && dwte_dev && dwpe_dev, "NULL pointer");
  NNT_CHECK_ARG(batch > 0 && seq > 0 && d > 0 && vocab > 0 && vocab <= 65536 && ids_stride >= seq,
                "bad size");
  NNT_CHECK_ARG(batch * seq <= kNoAllocMaxTokens,
                "batch*seq = %lld exceeds the fixed scratch of the allocation-free call (%d tokens)",
                (long long)(batch * seq), kNoAllocMaxTokens);
  uint32_t* keys = nullptr;
  NNT_TRY(keys_on_current_device(&keys));
  cudaStream_t st = (cudaStream_t)stream;
  const int T = (int)(batch * seq);
  // the sort overwrites keys[0, T) before the scatter reads them, so nothing
  // left by an earlier call needs clearing
  TokMap tm{(int)seq, (int)batch, (int)seq, 1};
  NNT_TRY(launch_token_sort(ids_dev, ids_stride, (int)batch, (int)seq, keys, st));
  NNT_TRY(launch_embedding_scatter(keys, T, dx_dev, tm, (int)seq, dwte_dev, (int)d, (int)vocab, st));
  return launch_wpe_grad(dx_dev, tm, (int)batch, 0, (int)seq, (int)d, dwpe_dev, 1, st);
}
