// Fused causal attention tile task (flash attention): launch interface.
#pragma once

#include "common.cuh"

namespace nnt {

// One launch covers nz (sequence, head) items, item i -> z = zm.z(i), each over
// all S queries. q, k, v (and dO) are bf16 [Zall][S][hd] (head-major, as the
// QKV projection writes them); the outputs go to token rows: element (z, s, j)
// of O is stored at o[tm.row(b, s) * ldo + o_col + h * hd + j] with
// (b, h) = (zm.b(i), zm.h(i)); a plain [Z][S][hd] output is the case H = 1,
// tm = {S, Z, S, 1}, ldo = hd, o_col = 0.
struct FlashArgs {
  int S = 0, hd = 0, nz = 0;
  ZMap zm{0, 0, 1, 1};
  int64_t z_total = 0;  // Zall: items in the q/k/v buffers
  TokMap tm{1, 1, 1, 1};
  // forward output / backward input O
  bf16* o = nullptr;
  int64_t ldo = 0, o_col = 0;
  // per-row log-sum-exp of the scaled scores, base 2, [Zall][S]
  float* lse = nullptr;
  // backward: D = rowsum(dO * O) scratch [Zall][S]; gradient outputs in the
  // same token-row layout (ldd, columns dq_col / dk_col / dv_col + h * hd)
  float* D = nullptr;
  // optional [Zall][S][S] bf16 scratch (S a multiple of 8): the dK/dV pass then
  // also stores dS^T (row = key, column = query) and dQ = dS K runs as a
  // tensor-core GEMM instead of a second recomputing pass
  bf16* ds = nullptr;
  bf16* dq = nullptr;
  bf16* dk = nullptr;
  bf16* dv = nullptr;
  int64_t ldd = 0, dq_col = 0, dk_col = 0, dv_col = 0;
};

// true when the fused kernels serve this head size (64 or 128)
bool flash_supported(int hd);

// O and lse from q, k, v (scores scaled by 1/sqrt(hd), causal mask).
nnt_status launch_flash_fwd(const bf16* q, const bf16* k, const bf16* v, const FlashArgs& a,
                            cudaStream_t st);
// dq, dk, dv from q, k, v, O, dO and lse (three kernels: D, dK/dV, dQ).
nnt_status launch_flash_bwd(const bf16* q, const bf16* k, const bf16* v, const bf16* dO,
                            const FlashArgs& a, cudaStream_t st);

}  // namespace nnt
