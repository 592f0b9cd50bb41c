// Host-side fault injection for the failure-detection tests: an armed kind
// makes its Nth call from now fail as the real failure would (the allocation
// returns OOM, the copy submission or the wait returns its error), without
// touching the GPU. Off by default; nothing on the device is ever faulted.
#include <stdlib.h>

#include <atomic>

#include "common.cuh"

namespace nnt {
namespace {
std::atomic<int64_t> g_fault_left[FAULT_KINDS];
}  // namespace

bool fault_hit(FaultKind kind) {
  std::atomic<int64_t>& c = g_fault_left[kind];
  int64_t v = c.load(std::memory_order_relaxed);
  while (v > 0) {
    if (c.compare_exchange_weak(v, v - 1, std::memory_order_relaxed)) return v == 1;
  }
  return false;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("NNT_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

}  // namespace nnt

extern "C" nnt_status nnt_set_fault_injection(int32_t kind, int64_t nth) {
  NNT_CHECK_ARG(kind >= 0 && kind < nnt::FAULT_KINDS, "fault kind %d out of range", kind);
  NNT_CHECK_ARG(nth >= 0, "nth must be >= 0");
  nnt::g_fault_left[kind].store(nth, std::memory_order_relaxed);
  return NNT_OK;
}
