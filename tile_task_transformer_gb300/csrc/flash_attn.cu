// Fused causal attention tile task ("flash attention") for sm_103a.
//
// The README's example command turns on --flashattention, which the pages list
// as a memory-saving option whose kernel NNTile does not have yet (README
// "Minimal working GPT example", flag list). Here it is a tile task of its
// own: the score tile S = Q K^T / sqrt(hd) of one (sequence, head) and 128
// queries lives in tensor memory, the causal softmax is taken row by row with
// a running maximum and sum (online softmax), P reaches P V through tensor
// memory (the product's A operand), and nothing of size S x S is written to HBM. The backward pass
// recomputes P from the per-row log-sum-exp saved by the forward.
//
// The forward and the head-size-128 backward kernels are block-synchronous:
// threads t, t+128, ... own row t of the current tile, which is TMEM lane t
// (warp w reads lanes 32(w%4)..32(w%4)+31), each taking a share of the row's
// columns; thread 0 also issues the TMA copies and the tcgen05.mma
// instructions. The head-size-64 dK/dV kernel is warp-specialised (one issuing
// warp, sixteen compute warps, mbarrier hand-offs). Tiles are [128 rows][hd]
// bf16 loaded by TMA with a 128-byte swizzle as hd/64 chunks of 16 KB; the same
// smem tile serves
// as a K-major operand (rows = M or N, K = hd) or an MN-major one (N = hd,
// K = rows) through its descriptor. P and dS tiles written by the threads use
// the K-major layout TMA would produce.
//
//   flash_fwd_kernel     item x query block: O and the log-sum-exp
//   flash_bwd_d_kernel   D = rowsum(dO * O)
//   flash_bwd_kv_ws_kernel / flash_bwd_kv_kernel (head size 64 / 128)
//                        item x key block: dK, dV over the query blocks at or after it,
//                        and (given a dS^T buffer) each dS^T tile stored by TMA, after
//                        which dQ = dS K is the causal tensor-core GEMM
//   flash_bwd_q_kernel   item x query block: dQ over the key blocks at or before it
//                        (recomputing S and dP; used without a dS^T buffer)
// dK/dV and dQ come from separate passes, so every sum has a fixed order (no
// atomics). Every mbarrier wait is bounded: on expiry the kernel records the
// device error word, waits (bounded) for its own copies and MMAs in flight,
// frees its TMEM and returns.
#include <math.h>

#include <mutex>

#include "flash.cuh"
#include "gemm.cuh"
#include "ptx_math.cuh"
#include "tc_ptx.cuh"

namespace nnt {
namespace {

constexpr int FB = 128;              // queries or keys per block
constexpr int kThreads = 256;     // forward: two threads per row, one per half of the columns
constexpr int kBwdThreads = 256;  // backward dQ kernel: the same split
constexpr int kKvThreads = 512;   // backward dK/dV kernel: four threads per key row, 32 columns each
constexpr int CHUNK = FB * 128;      // one [128 rows][64 bf16] swizzled chunk: 16 KB

// Descriptor of K step kk (16 elements) of a [128][*] tile used K-major.
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk) {
  return make_sdesc(base + (uint32_t)((kk >> 2) * CHUNK + (kk & 3) * 32), 16, 1024);
}
// Descriptor of K step kk (16 rows) of a [128][hd] tile used MN-major (N = hd).
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int kk) {
  return make_sdesc(base + (uint32_t)(kk * 2048), CHUNK, 1024);
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Columns 8g..8g+7 of row r of a [128][128] bf16 K-major tile (two chunks).
__device__ __forceinline__ void put8(uint8_t* tile, int r, int g, const float* v) {
  uint4 pk;
  pk.x = pack_bf2(v[0], v[1]);
  pk.y = pack_bf2(v[2], v[3]);
  pk.z = pack_bf2(v[4], v[5]);
  pk.w = pack_bf2(v[6], v[7]);
  *reinterpret_cast<uint4*>(tile + (g >> 3) * CHUNK + r * 128 + (((g & 7) ^ (r & 7)) << 4)) = pk;
}

// One [128][HD] tile starting at sequence row `row` of item z.
template <int HD>
__device__ __forceinline__ void load_tile(const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int row,
                                          int z) {
#pragma unroll
  for (int c = 0; c < HD / 64; ++c) tma_load_3d(dst + c * CHUNK, map, bar, 64 * c, row, z);
}

// NCOL (a multiple of 32) TMEM columns of this thread's row, scaled, to bf16 at dst.
template <int NCOL>
__device__ __forceinline__ void store_row(uint32_t taddr, bool row_ok, bf16* dst, float scale) {
#pragma unroll
  for (int c = 0; c < NCOL / 32; ++c) {
    uint32_t o[32];
    tmem_ld32_nw(taddr + 32 * c, o);
    tmem_wait_ld();
    if (row_ok) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 pk;
        pk.x = pack_bf2(__uint_as_float(o[8 * k + 0]) * scale, __uint_as_float(o[8 * k + 1]) * scale);
        pk.y = pack_bf2(__uint_as_float(o[8 * k + 2]) * scale, __uint_as_float(o[8 * k + 3]) * scale);
        pk.z = pack_bf2(__uint_as_float(o[8 * k + 4]) * scale, __uint_as_float(o[8 * k + 5]) * scale);
        pk.w = pack_bf2(__uint_as_float(o[8 * k + 6]) * scale, __uint_as_float(o[8 * k + 7]) * scale);
        *reinterpret_cast<uint4*>(dst + 32 * c + 8 * k) = pk;
      }
    }
  }
}

// Bounded waits for every copy a barrier still owes (n issued, *w waited).
__device__ __forceinline__ void drain(uint64_t* bar, int n, int* w) {
  for (; *w < n; ++*w) mbar_wait(bar, (uint32_t)(*w & 1));
}

// ================================================================ forward

template <int HD>
struct FwdCfg {
  static constexpr int TILE = FB * HD * 2;
  // Q, K (two stages), V (two stages), and scratch for the halves' row maxima
  // and sums ([2][128] floats).
  static constexpr int OFF_Q = 0, OFF_K = TILE, OFF_V = 3 * TILE, OFF_P = 5 * TILE;
  static constexpr int OFF_RED = OFF_P;
  static constexpr int OFF_BAR = OFF_P + 2 * CHUNK;
  // head size 64: no room to re-align the base by hand if two CTAs are to fit
  // on an SM; the kernel then requires a 1024-byte aligned dynamic base
  static constexpr bool FIXED_BASE = HD <= 64;
  static constexpr int SMEM = OFF_BAR + 128 + (FIXED_BASE ? 0 : 1024);
  // S: 128 columns, O: HD, P (bf16 pairs, the A operand of P V): 64
  static constexpr uint32_t T_O = FB, T_P = FB + HD;
  static constexpr uint32_t TMEM_COLS = FB + HD + FB / 2 <= 256 ? 256 : 512;
};

// Per CTA: item blockIdx % nz, query block nqb-1 - blockIdx / nz (largest
// first). Key blocks 0..qb in order; K and V are double-buffered: once S_j is
// done (and with it P V_{j-1}), K_{j+2} and V_{j+1} load into the freed
// stages.
//
// Two threads per row, one per half of the columns (256 threads; warps w and
// w+4 share TMEM lanes 32(w%4)..). Softmax of row r at key block j: m =
// running maximum of the scaled scores in base 2 (the halves' maxima meet in
// shared memory), l = running sum of 2^(s*c2 - m), kept per half and added at
// the end. The maximum actually used is raised only when a row's new maximum
// exceeds it by more than 8 (P stays below 2^8, exact in fp32 and in bf16's
// range); then l and the row of O are multiplied by 2^(m_old - m_new), each
// thread rescaling its half of O through TMEM.
template <int HD>
__global__ void __launch_bounds__(kThreads, HD <= 64 ? 2 : 1)
    flash_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const FlashArgs a, int nqb, float c2,
                     uint32_t* err) {
  using C = FwdCfg<HD>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (C::FIXED_BASE && sm != smem_raw) {  // 128-byte swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicOr(err, DEVERR_SMEM_ALIGN);
    return;
  }
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* bar_k = bar_q + 1;  // two stages
  uint64_t* bar_v = bar_q + 3;  // two stages
  uint64_t* bar_s = bar_q + 5;
  uint64_t* bar_o = bar_q + 6;
  uint64_t* bar_x = bar_q + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_q + 8);
  float* red = reinterpret_cast<float*>(sm + C::OFF_RED);  // [2][FB]: row maxima, then row sums

  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = tid & (FB - 1), hf = tid >> 7;  // row of the tile, column half
  const int qb = nqb - 1 - (int)(blockIdx.x / a.nz);
  const int item = (int)(blockIdx.x % a.nz);
  const int z = (int)a.zm.z(item);
  const int q0 = qb * FB, nkb = qb + 1;
  const int q = q0 + r;

  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(bar_q + i, 1);
    mbar_fence_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the prologue above overlaps the previous kernel
  pdl_trigger();
  const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const uint32_t s_q = smem_u32(sm + C::OFF_Q), s_v = smem_u32(sm + C::OFF_V);
  constexpr int HC = FB / 2;  // score columns per thread
  constexpr int HO = HD / 2;  // O columns per thread

  int n_k[2] = {0, 0}, w_k[2] = {0, 0}, n_v[2] = {0, 0}, w_v[2] = {0, 0}, w_q = 0;
  auto load_kv = [&](const CUtensorMap* map, int off, uint64_t* bar, int blk) {
    mbar_arrive_expect_tx(bar, C::TILE);
    load_tile<HD>(map, sm + off + (blk & 1) * C::TILE, bar, blk * FB, z);
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_q, C::TILE);
    load_tile<HD>(&tmQ, sm + C::OFF_Q, bar_q, q0, z);
    for (int blk = 0; blk < 2 && blk < nkb; ++blk) {
      load_kv(&tmK, C::OFF_K, &bar_k[blk], blk);
      load_kv(&tmV, C::OFF_V, &bar_v[blk], blk);
      n_k[blk] = n_v[blk] = 1;
    }
  }

  float m_used = -INFINITY, l = 0.f;
  bool ok = true, aborted = false;
  for (int j = 0; j < nkb; ++j) {
    const int st = j & 1;
    if (tid == 0) {
      if (j == 0) {
        ok = mbar_wait(bar_q, 0);
        w_q = ok ? 1 : 0;
      }
      if (ok) {
        ok = mbar_wait(&bar_k[st], (uint32_t)((j >> 1) & 1));
        if (ok) ++w_k[st];
      }
      if (ok) {
        tc_fence_after();
        const uint32_t s_k = smem_u32(sm + C::OFF_K + st * C::TILE);
        constexpr uint32_t idesc = make_idesc(FB, FB, false, false);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16(tmem, desc_k(s_q, kk), desc_k(s_k, kk), idesc, kk > 0 ? 1u : 0u);
        umma_commit(bar_s);
      }
    }
    if (ok) ok = mbar_wait(bar_s, (uint32_t)(j & 1));
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    tc_fence_after();
    if (tid == 0) {  // S_j done, and with it P V_{j-1}: K stage j&1 and V stage (j+1)&1 are free
      if (j + 2 < nkb) {
        load_kv(&tmK, C::OFF_K, &bar_k[st], j + 2);
        ++n_k[st];
      }
      if (j >= 1 && j + 1 < nkb) {
        load_kv(&tmV, C::OFF_V, &bar_v[st ^ 1], j + 1);
        ++n_v[st ^ 1];
      }
    }
    // ---- softmax of row r over keys [j*128, j*128 + 128), columns [hf*64, hf*64 + 64)
    uint32_t u[HC];
#pragma unroll
    for (int c = 0; c < HC / 32; ++c) tmem_ld32_nw(t_row + hf * HC + 32 * c, u + 32 * c);
    tmem_wait_ld();
    const bool diag = j == nkb - 1;  // keys past the query only in the last block
    float mx = -INFINITY;
    if (diag) {
#pragma unroll
      for (int c = 0; c < HC; ++c) {
        float x = __uint_as_float(u[c]);
        if (hf * HC + c > r) x = -INFINITY;
        u[c] = __float_as_uint(x);
        mx = fmaxf(mx, x);
      }
    } else {
      float m2 = -INFINITY;  // two chains
#pragma unroll
      for (int c = 0; c < HC; c += 2) {
        mx = fmaxf(mx, __uint_as_float(u[c]));
        m2 = fmaxf(m2, __uint_as_float(u[c + 1]));
      }
      mx = fmaxf(mx, m2);
    }
    red[hf * FB + r] = mx;
    __syncthreads();
    mx = fmaxf(mx, red[(hf ^ 1) * FB + r]);
    __syncthreads();  // the scratch lies in P, written below
    const float m_new = fmaxf(m_used, mx * c2);
    if (j == 0) {
      m_used = m_new;
    } else {
      const bool need = m_new > m_used + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2f(m_used - m_new) : 1.f;
        if (need) {
          l *= alpha;
          m_used = m_new;
        }
#pragma unroll
        for (int c = 0; c < HO / 32; ++c) {
          uint32_t o[32];
          const uint32_t ta = t_row + FB + hf * HO + 32 * c;
          tmem_ld32_nw(ta, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(ta, o);
        }
        tmem_wait_st();
      }
    }
    float2 sum2 = make_float2(0.f, 0.f);
    const float2 c22 = make_float2(c2, c2), mm = make_float2(-m_used, -m_used);
    // P in bf16 pairs into tensor memory (this thread: keys hf*HC.., columns T_P + hf*HC/2..)
    uint32_t pk[HC / 2];
#pragma unroll
    for (int e = 0; e < HC; e += 2) {
      const float2 t = fma2(make_float2(__uint_as_float(u[e]), __uint_as_float(u[e + 1])), c22, mm);
      const float2 pv = make_float2(ex2f(t.x), ex2f(t.y));
      sum2 = add2(sum2, pv);
      pk[e / 2] = pack_bf2(pv.x, pv.y);
    }
    tmem_st32(t_row + C::T_P + hf * (HC / 2), pk);
    l += sum2.x + sum2.y;
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
      ok = mbar_wait(&bar_v[st], (uint32_t)((j >> 1) & 1));
      if (ok) {
        ++w_v[st];
        tc_fence_after();
        const uint32_t s_vt = s_v + (uint32_t)(st * C::TILE);
        constexpr uint32_t idesc = make_idesc(FB, HD, false, true);
#pragma unroll
        for (int kk = 0; kk < FB / 16; ++kk)
          umma_bf16_ta(tmem + C::T_O, tmem + C::T_P + 8 * kk, desc_mn(s_vt, kk), idesc, (j > 0 || kk > 0) ? 1u : 0u);
      }
    }
  }
  if (!aborted) {
    if (tid == 0 && ok) umma_commit(bar_o);
    if (ok) ok = mbar_wait(bar_o, 0);
    if (__syncthreads_or(!ok)) aborted = true;
  }
  if (!aborted) {
    red[hf * FB + r] = l;  // P's last reader (the final P V) is done
    __syncthreads();
    l += red[(hf ^ 1) * FB + r];
    tc_fence_after();
    const int b = a.zm.b(item), h = a.zm.h(item);
    const bool row_ok = q < a.S;
    bf16* orow = a.o + (row_ok ? a.tm.row(b, q) * a.ldo + a.o_col + (int64_t)h * HD + hf * HO : 0);
    store_row<HO>(t_row + FB + hf * HO, row_ok, orow, 1.f / l);
    if (row_ok && hf == 0) a.lse[(int64_t)z * a.S + q] = m_used + log2f(l);
  } else if (tid == 0) {
    atomicOr(err, DEVERR_WAIT_TIMEOUT);
    drain(bar_q, 1, &w_q);
    drain(&bar_k[0], n_k[0], &w_k[0]);
    drain(&bar_k[1], n_k[1], &w_k[1]);
    drain(&bar_v[0], n_v[0], &w_v[0]);
    drain(&bar_v[1], n_v[1], &w_v[1]);
    umma_commit(bar_x);
    mbar_wait(bar_x, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ================================================================ backward

__device__ __forceinline__ float dot8_bf16(uint4 x, uint4 y) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[i]));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[i]));
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
  }
  return acc;
}

// D[z][s] = sum_j dO[z][s][j] * O(z, s, j). CTA: 32 rows of item blockIdx.y;
// eight lanes per row, 16 bytes of dO and of O each per step.
__global__ void __launch_bounds__(256) flash_bwd_d_kernel(const bf16* __restrict__ dO, const FlashArgs a) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int item = blockIdx.y;
  const int s = blockIdx.x * 32 + warp * 4 + (lane >> 3);
  const int sub = lane & 7;
  const int64_t z = a.zm.z(item);
  float acc = 0.f;
  if (s < a.S) {
    const bf16* dr = dO + (z * a.S + s) * a.hd;
    const bf16* orow = a.o + a.tm.row(a.zm.b(item), s) * a.ldo + a.o_col + (int64_t)a.zm.h(item) * a.hd;
    for (int j = 8 * sub; j < a.hd; j += 64)
      acc += dot8_bf16(*reinterpret_cast<const uint4*>(dr + j), *reinterpret_cast<const uint4*>(orow + j));
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  if (sub == 0 && s < a.S) a.D[z * a.S + s] = acc;
}

template <int HD>
struct KvCfg {
  static constexpr int TILE = FB * HD * 2;
  // head size 128 (64 takes the warp-specialised kernel): one (Q, dO) stage,
  // tensor memory full with S^T, dP^T, dV and dK
  static constexpr int NS = 1;
  static constexpr int OFF_K = 0, OFF_V = TILE, OFF_ST = 2 * TILE;  // stage s: Q, then dO
  static constexpr int OFF_PT = OFF_ST + NS * 2 * TILE, OFF_DS = OFF_PT + 2 * CHUNK;
  static constexpr int OFF_ROW = OFF_DS + 2 * CHUNK;  // lse and D of the current query block
  static constexpr int OFF_BAR = OFF_ROW + 2 * FB * 4;
  static constexpr int SMEM = OFF_BAR + 128 + 1024;
};

// Per CTA: key block kb = blockIdx / nz (the first ones have the most query
// blocks), item blockIdx % nz. For each query block i >= kb:
//   S^T = K Q_i^T, dP^T = V dO_i^T            (TMEM columns 0..127, 128..255)
//   P^T = 2^(S^T c2 - lse), dS^T = scale * P^T (dP^T - D)   (rows = keys, in smem)
//   dV += P^T dO_i, dK += dS^T Q_i              (TMEM columns 256.., 256+HD..)
template <int HD>
__global__ void __launch_bounds__(kKvThreads, 1)
    flash_bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                        const __grid_constant__ CUtensorMap tmDS, int store_ds, const FlashArgs a,
                        int nqb, float c2, float scale, uint32_t* err) {
  using C = KvCfg<HD>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_kv = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* bar_ld = bar_kv + 1;    // [3]
  uint64_t* bar_free = bar_kv + 4;  // [3]
  uint64_t* bar_s = bar_kv + 7;
  uint64_t* bar_o = bar_kv + 8;
  uint64_t* bar_x = bar_kv + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_kv + 10);
  float* lse_s = reinterpret_cast<float*>(sm + C::OFF_ROW);
  float* d_s = lse_s + FB;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = tid & (FB - 1), hf = tid >> 7;  // row of the tile, column quarter
  const int kb = (int)(blockIdx.x / a.nz);
  const int item = (int)(blockIdx.x % a.nz);
  const int z = (int)a.zm.z(item);
  const int n = nqb - kb;
  const int key = kb * FB + r;

  if (tid == 0) {
    for (int i = 0; i < 10; ++i) mbar_init(bar_kv + i, 1);
    mbar_fence_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
    tma_prefetch_map(&tmdO);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the prologue above overlaps the previous kernel
  pdl_trigger();
  const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const uint32_t s_k = smem_u32(sm + C::OFF_K), s_v = smem_u32(sm + C::OFF_V);
  const uint32_t s_pt = smem_u32(sm + C::OFF_PT), s_ds = smem_u32(sm + C::OFF_DS);

  auto load_qdo = [&](int s, int i) {
    uint8_t* dst = sm + C::OFF_ST + s * 2 * C::TILE;
    mbar_arrive_expect_tx(&bar_ld[s], 2 * C::TILE);
    load_tile<HD>(&tmQ, dst, &bar_ld[s], i * FB, z);
    load_tile<HD>(&tmdO, dst + C::TILE, &bar_ld[s], i * FB, z);
  };
  int n_ld[3] = {0, 0, 0}, w_ld[3] = {0, 0, 0}, w_kv = 0;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_kv, 2 * C::TILE);
    load_tile<HD>(&tmK, sm + C::OFF_K, bar_kv, kb * FB, z);
    load_tile<HD>(&tmV, sm + C::OFF_V, bar_kv, kb * FB, z);
    for (int it = 0; it < NS && it < n; ++it) {
      load_qdo(it, kb + it);
      n_ld[it] = 1;
    }
  }

  bool ok = true, aborted = false;
  // column r of query block i: lse (first half of the threads) or D (second);
  // the next block's value is loaded one iteration ahead
  const float* rowsrc = hf == 1 ? a.D : a.lse;  // quarters 0 and 1 stage lse and D
  auto row_val = [&](int i) {
    const int qc = i * FB + r;
    return hf < 2 && qc < a.S ? rowsrc[(int64_t)z * a.S + qc] : 0.f;
  };
  // refill the stage freed by iteration it-1 with the operands of iteration it+NS-1
  auto refill = [&](int it) {
    if (ok && it >= 1 && it + NS - 1 < n) {
      const int s2 = (it + NS - 1) % NS;
      ok = mbar_wait(&bar_free[s2], (uint32_t)(((it - 1) / NS) & 1));
      if (ok) {
        load_qdo(s2, kb + it + NS - 1);
        ++n_ld[s2];
      }
    }
  };
  // S^T = K Q_i^T and dP^T = V dO_i^T of iteration it_ into TMEM columns 0..255
  // (thread 0; the operands' stage must have landed)
  auto issue_s = [&](int it_) {
    const int st_ = it_ % NS;
    if (ok) {
      ok = mbar_wait(&bar_ld[st_], (uint32_t)((it_ / NS) & 1));
      if (ok) ++w_ld[st_];
    }
    if (ok) {
      tc_fence_after();
      const uint32_t s_qt = smem_u32(sm + C::OFF_ST + st_ * 2 * C::TILE), s_do = s_qt + C::TILE;
      constexpr uint32_t idesc = make_idesc(FB, FB, false, false);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        umma_bf16(tmem, desc_k(s_k, kk), desc_k(s_qt, kk), idesc, kk > 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        umma_bf16(tmem + FB, desc_k(s_v, kk), desc_k(s_do, kk), idesc, kk > 0 ? 1u : 0u);
      umma_commit(bar_s);
    }
  };
  float row_next = row_val(kb);
  for (int it = 0; it < n; ++it) {
    const int i = kb + it, st = it % NS;
    const float row_c = row_next;
    if (it + 1 < n) row_next = row_val(i + 1);
    // the previous dS^T tile must have left shared memory before it is rewritten
    if (store_ds && tid == 32 && it > 0) bulk_wait_read();
    if (tid == 0) {
      if (it == 0) {
        ok = mbar_wait(bar_kv, 0);
        w_kv = ok ? 1 : 0;
      }
      refill(it);  // single stage: the operands of this iteration
      issue_s(it);
    }
    if (hf < 2) (hf ? d_s : lse_s)[r] = row_c;
    if (ok) ok = mbar_wait(bar_s, (uint32_t)(it & 1));
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    tc_fence_after();
    const bool diag = i == kb;
    uint8_t* pt = sm + C::OFF_PT;
    uint8_t* dst = sm + C::OFF_DS;
    // this thread's 32 query columns
    uint32_t sv[32], dv[32];
    tmem_ld32_nw(t_row + 32 * hf, sv);
    tmem_ld32_nw(t_row + FB + 32 * hf, dv);
    tmem_wait_ld();
    {
      const int c = hf;
      // the chunk's lse and D values are read from shared memory as they are
      // needed (the same addresses across the warp: broadcast); P^T and dS^T
      // overwrite the registers that held S^T and dP^T
      const float* lsr = lse_s + 32 * c;
      const float* ddr = d_s + 32 * c;
      float* p = reinterpret_cast<float*>(sv);
      float* ds = reinterpret_cast<float*>(dv);
      if (!diag && i * FB + 32 * c + 32 <= a.S) {  // every entry of the chunk is causal and in range
        const float2 c22 = make_float2(c2, c2), sc2 = make_float2(scale, scale);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 ls2 = *reinterpret_cast<const float2*>(lsr + e);
          const float2 dd2 = *reinterpret_cast<const float2*>(ddr + e);
          const float2 t = fma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c22,
                                make_float2(-ls2.x, -ls2.y));
          const float2 pv = make_float2(ex2f(t.x), ex2f(t.y));
          const float2 dq = add2(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                 make_float2(-dd2.x, -dd2.y));
          const float2 d2 = mul2(mul2(pv, sc2), dq);
          p[e] = pv.x; p[e + 1] = pv.y;
          ds[e] = d2.x; ds[e + 1] = d2.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int qq = 32 * c + e;
          const bool valid = i * FB + qq < a.S && (!diag || qq >= r);
          const float pv = valid ? ex2f(fmaf(__uint_as_float(sv[e]), c2, -lsr[e])) : 0.f;
          const float dsv = pv * scale * (__uint_as_float(dv[e]) - ddr[e]);
          p[e] = pv;
          ds[e] = dsv;
        }
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        put8(pt, r, 4 * c + g, p + 8 * g);
        put8(dst, r, 4 * c + g, ds + 8 * g);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (store_ds && tid == 32) {  // dS^T tile to global: rows kb*128.., columns i*128..
#pragma unroll
      for (int c = 0; c < 2; ++c) tma_store_3d(&tmDS, dst + c * CHUNK, i * FB + 64 * c, kb * FB, z);
      bulk_commit();
    }
    if (tid == 0 && ok) {
      tc_fence_after();
      const uint32_t s_qt = smem_u32(sm + C::OFF_ST + st * 2 * C::TILE), s_do = s_qt + C::TILE;
      constexpr uint32_t idesc = make_idesc(FB, HD, false, true);
#pragma unroll
      for (int kk = 0; kk < FB / 16; ++kk)
        umma_bf16(tmem + 2 * FB, desc_k(s_pt, kk), desc_mn(s_do, kk), idesc, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < FB / 16; ++kk)
        umma_bf16(tmem + 2 * FB + HD, desc_k(s_ds, kk), desc_mn(s_qt, kk), idesc,
                  (it > 0 || kk > 0) ? 1u : 0u);
      umma_commit(&bar_free[st]);
    }
  }
  if (!aborted) {
    if (tid == 0 && ok) umma_commit(bar_o);
    if (ok) ok = mbar_wait(bar_o, 0);
    if (__syncthreads_or(!ok)) aborted = true;
  }
  if (!aborted) {
    tc_fence_after();
    const int b = a.zm.b(item), h = a.zm.h(item);
    const bool row_ok = key < a.S;
    const int64_t row = row_ok ? a.tm.row(b, key) * a.ldd : 0;
    // quarters 0, 1: the two halves of dV; quarters 2, 3: of dK
    const int c0 = (hf & 1) * (HD / 2);
    if (hf < 2)
      store_row<HD / 2>(t_row + 2 * FB + c0, row_ok, a.dv + row + a.dv_col + (int64_t)h * HD + c0, 1.f);
    else
      store_row<HD / 2>(t_row + 2 * FB + HD + c0, row_ok, a.dk + row + a.dk_col + (int64_t)h * HD + c0, 1.f);
  } else if (tid == 0) {
    atomicOr(err, DEVERR_WAIT_TIMEOUT);
    drain(bar_kv, 1, &w_kv);
    for (int s2 = 0; s2 < NS; ++s2) drain(&bar_ld[s2], n_ld[s2], &w_ld[s2]);
    umma_commit(bar_x);
    mbar_wait(bar_x, 0);
  }
  if (store_ds && tid == 32) bulk_wait_all();  // stores finished before shared memory goes
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- dK/dV, warp-specialised (head size 64)

// Sixteen compute warps (four threads per key row, 32 query columns each) and one
// warp whose lane 0 issues every TMA copy and tensor-core product, handing off
// through mbarriers instead of block-wide barriers, so the products of one
// query block run while the next block's arithmetic runs:
//
//   issuer, block it:  S^T, dP^T of block it+1 once the compute warps hold
//                      block it's in registers; the (Q, dO) stage of block
//                      it-1 refilled with block it+2 once dV, dK of it-1 are
//                      done; dV += P^T dO and dK += dS^T Q of block it once
//                      P^T (tensor memory) and dS^T (shared memory) are
//                      written; dS^T of block it stored to global by TMA.
//   compute, block it: block it+1's -lse and -scale D staged in shared memory
//                      (three buffers, so no block-wide barrier); S^T, dP^T
//                      to registers; P^T and dS^T computed, then written
//                      once the products of block it-1 (and the store of
//                      block it-2's dS^T buffer) are done.
//
// The products are bound by shared-memory bandwidth at these sizes (N of 64
// or 128), so the operands that can live in tensor memory do: K and V (the A
// operands of S^T and dP^T, copied there once) and P^T (the A operand of dV).
// Tensor memory (512 columns): S^T 0..127, dP^T 128..255, dV 256..319,
// dK 320..383, P^T 384..447, K 448..479, V 480..511 (16-bit pairs).
struct KvWsCfg {
  static constexpr int HD = 64;
  static constexpr int TILE = FB * HD * 2;
  static constexpr int NS = 3;  // (Q, dO) stages
  static constexpr int OFF_K = 0, OFF_V = TILE, OFF_ST = 2 * TILE;
  static constexpr int OFF_DS = OFF_ST + NS * 2 * TILE;  // two [128][128] bf16 dS^T tiles
  static constexpr int OFF_ROW = OFF_DS + 2 * 2 * CHUNK;  // [3][-lse, -scale D][FB] floats
  static constexpr int OFF_BAR = OFF_ROW + 3 * 2 * FB * 4;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr uint32_t T_DV = 2 * FB, T_DK = 2 * FB + HD, T_P = 2 * FB + 2 * HD;
  static constexpr uint32_t T_K = T_P + FB / 2, T_V = T_K + HD / 2;
};
constexpr int kKvWsCompute = 512;
constexpr int kKvWsThreads = kKvWsCompute + 32;

__global__ void __launch_bounds__(kKvWsThreads, 1)
    flash_bwd_kv_ws_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                           const __grid_constant__ CUtensorMap tmDS, int store_ds, const FlashArgs a,
                           int nqb, float c2, float scale, uint32_t* err) {
  using C = KvWsCfg;
  constexpr int HD = C::HD, NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_kv = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* bar_ld = bar_kv + 1;      // [NS] (Q, dO) stage landed
  uint64_t* bar_s = bar_kv + 4;       // S^T, dP^T of the current block done
  uint64_t* bar_sfree = bar_kv + 5;   // compute warps hold S^T, dP^T in registers (16 arrivals)
  uint64_t* bar_pready = bar_kv + 6;  // [2] P^T, dS^T of block it written (16 arrivals), by it % 2
  uint64_t* bar_free = bar_kv + 8;    // [NS] dV, dK of a block done: its stage and buffers are free
  uint64_t* bar_dsread = bar_kv + 11; // [2] the store of dS^T buffer b has read it
  uint64_t* bar_o = bar_kv + 13;
  uint64_t* bar_x = bar_kv + 14;
  uint64_t* bar_kvt = bar_kv + 15;    // K and V copied into tensor memory (16 arrivals)
  uint64_t* bar_rows = bar_kv + 16;   // [3] -lse, -scale D of a query block staged (16 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_kv + 19);
  float* rows = reinterpret_cast<float*>(sm + C::OFF_ROW);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kb = (int)(blockIdx.x / a.nz);
  const int item = (int)(blockIdx.x % a.nz);
  const int z = (int)a.zm.z(item);
  const int n = nqb - kb;

  if (tid == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_ld[s], 1);
      mbar_init(&bar_free[s], 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_sfree, kKvWsCompute / 32);
    mbar_init(&bar_pready[0], kKvWsCompute / 32);
    mbar_init(&bar_pready[1], kKvWsCompute / 32);
    mbar_init(&bar_dsread[0], 1);
    mbar_init(&bar_dsread[1], 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_x, 1);
    mbar_init(bar_kvt, kKvWsCompute / 32);
    for (int q = 0; q < 3; ++q) mbar_init(&bar_rows[q], kKvWsCompute / 32);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the prologue above overlaps the previous kernel
  pdl_trigger();

  bool ok = true;
  int n_ld[NS] = {0, 0, 0}, w_ld[NS] = {0, 0, 0}, w_kv = 0;  // issuer: copies issued / waited per stage
  const bool issuer = warp == kKvWsCompute / 32;
  const int r = tid & (FB - 1), h = (tid >> 7) & 3;  // compute warps: key row, quarter of the columns
  const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  if (issuer) {
    // ------------------------------------------------ TMA / MMA issue (lane 0)
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmdO);
      auto load_qdo = [&](int s, int i) {
        uint8_t* dst = sm + C::OFF_ST + s * 2 * C::TILE;
        mbar_arrive_expect_tx(&bar_ld[s], 2 * C::TILE);
        load_tile<HD>(&tmQ, dst, &bar_ld[s], i * FB, z);
        load_tile<HD>(&tmdO, dst + C::TILE, &bar_ld[s], i * FB, z);
        ++n_ld[s];
      };
      mbar_arrive_expect_tx(bar_kv, 2 * C::TILE);
      load_tile<HD>(&tmK, sm + C::OFF_K, bar_kv, kb * FB, z);
      load_tile<HD>(&tmV, sm + C::OFF_V, bar_kv, kb * FB, z);
      for (int it = 0; it < NS && it < n; ++it) load_qdo(it, kb + it);
      // S^T = K Q^T and dP^T = V dO^T of block it_ into columns 0..255 (K, V from tensor memory)
      auto issue_s = [&](int it_) {
        const int s = it_ % NS;
        ok = ok && mbar_wait(&bar_ld[s], (uint32_t)((it_ / NS) & 1));
        if (!ok) return;
        ++w_ld[s];
        tc_fence_after();
        const uint32_t s_qt = smem_u32(sm + C::OFF_ST + s * 2 * C::TILE), s_do = s_qt + C::TILE;
        constexpr uint32_t idesc = make_idesc(FB, FB, false, false);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16_ta(tmem, tmem + C::T_K + 8 * kk, desc_k(s_qt, kk), idesc, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16_ta(tmem + FB, tmem + C::T_V + 8 * kk, desc_k(s_do, kk), idesc, kk > 0 ? 1u : 0u);
        umma_commit(bar_s);
      };
      ok = mbar_wait(bar_kvt, 0);
      issue_s(0);
      for (int it = 0; it < n && ok; ++it) {
        const int st = it % NS, b = it & 1;
        if (it + 1 < n) {
          ok = mbar_wait(bar_sfree, (uint32_t)(it & 1));
          if (ok) {
            tc_fence_after();
            issue_s(it + 1);
          }
        }
        if (ok && it >= 1 && it + 2 < n) {  // stage of block it-1 <- operands of block it+2
          ok = mbar_wait(&bar_free[(it - 1) % NS], (uint32_t)(((it - 1) / NS) & 1));
          if (ok) load_qdo((it + 2) % NS, kb + it + 2);
        }
        if (ok && store_ds && it >= 1) {  // the store of dS^T(it-1) has read its buffer
          bulk_wait_read();
          mbar_arrive(&bar_dsread[(it - 1) & 1]);
        }
        if (ok) ok = mbar_wait(&bar_pready[b], (uint32_t)((it >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_qt = smem_u32(sm + C::OFF_ST + st * 2 * C::TILE), s_do = s_qt + C::TILE;
        const uint32_t s_ds = smem_u32(sm + C::OFF_DS + b * 2 * CHUNK);
        constexpr uint32_t idesc = make_idesc(FB, HD, false, true);
#pragma unroll
        for (int kk = 0; kk < FB / 16; ++kk)
          umma_bf16_ta(tmem + C::T_DV, tmem + C::T_P + 8 * kk, desc_mn(s_do, kk), idesc,
                       (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < FB / 16; ++kk)
          umma_bf16(tmem + C::T_DK, desc_k(s_ds, kk), desc_mn(s_qt, kk), idesc, (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bar_free[st]);
        if (store_ds) {  // dS^T tile to global: rows kb*128.., columns (kb+it)*128..
          uint8_t* dsb = sm + C::OFF_DS + b * 2 * CHUNK;
#pragma unroll
          for (int c = 0; c < 2; ++c) tma_store_3d(&tmDS, dsb + c * CHUNK, (kb + it) * FB + 64 * c, kb * FB, z);
          bulk_commit();
        }
      }
      if (ok) umma_commit(bar_o);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ compute warps
    // K and V rows into tensor memory (quarters 0, 1: head columns 32h.. of K's
    // row r; quarters 2, 3: of V's)
    ok = mbar_wait(bar_kv, 0);
    __syncwarp();
    {
      uint32_t w[16];
      const int half = h & 1;
      const uint8_t* src = sm + (h < 2 ? C::OFF_K : C::OFF_V) + r * 128;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int piece = (4 * half + k) ^ (r & 7);  // 128-byte swizzle of the TMA tile
        const uint4 x = *reinterpret_cast<const uint4*>(src + (piece << 4));
        w[4 * k] = x.x; w[4 * k + 1] = x.y; w[4 * k + 2] = x.z; w[4 * k + 3] = x.w;
      }
      tmem_st16(t_row + (h < 2 ? C::T_K : C::T_V) + 16 * half, w);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_kvt);
    }
    // -lse (quarter 0) or -scale * D (quarter 1) of query column r of block i
    auto row_val = [&](int i) {
      const int qc = i * FB + r;
      if (qc >= a.S || h > 1) return 0.f;
      const int64_t o = (int64_t)z * a.S + qc;
      return h ? -scale * a.D[o] : -a.lse[o];
    };
    const float2 c22 = make_float2(c2, c2), sc2 = make_float2(scale, scale);
    if (h < 2) rows[(2 * 0 + h) * FB + r] = row_val(kb);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar_rows[0]);
    float row_next = n > 1 ? row_val(kb + 1) : 0.f;
    for (int it = 0; it < n; ++it) {
      const int i = kb + it, b = it % 3;
      if (it + 1 < n) {  // block it+1's values into buffer (it+1) % 3 (last read in block it-2)
        if (h < 2) rows[(2 * ((it + 1) % 3) + h) * FB + r] = row_next;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_rows[(it + 1) % 3]);
        if (it + 2 < n) row_next = row_val(i + 2);
      }
      ok = ok && mbar_wait(&bar_rows[b], (uint32_t)((it / 3) & 1));
      uint32_t sv[32], dv[32];
      ok = ok && mbar_wait(bar_s, (uint32_t)(it & 1));
      __syncwarp();
      tc_fence_after();
      tmem_ld32_nw(t_row + 32 * h, sv);
      tmem_ld32_nw(t_row + FB + 32 * h, dv);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sfree);
      // P^T = 2^(S^T c2 - lse), dS^T = P^T (scale dP^T - scale D), in place
      const float* nls = rows + (2 * b) * FB + 32 * h;
      const float* nds = rows + (2 * b + 1) * FB + 32 * h;
      const int bd = it & 1;
      float* p = reinterpret_cast<float*>(sv);
      float* ds = reinterpret_cast<float*>(dv);
      if (i != kb && i * FB + 32 * h + 32 <= a.S) {  // every entry causal and in range
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(nls + e);
          const float4 d4 = *reinterpret_cast<const float4*>(nds + e);
          const float2 t0 = fma2(make_float2(p[e], p[e + 1]), c22, make_float2(l4.x, l4.y));
          const float2 t1 = fma2(make_float2(p[e + 2], p[e + 3]), c22, make_float2(l4.z, l4.w));
          const float2 p0 = make_float2(ex2f(t0.x), ex2f(t0.y)), p1 = make_float2(ex2f(t1.x), ex2f(t1.y));
          const float2 q0 = fma2(make_float2(ds[e], ds[e + 1]), sc2, make_float2(d4.x, d4.y));
          const float2 q1 = fma2(make_float2(ds[e + 2], ds[e + 3]), sc2, make_float2(d4.z, d4.w));
          const float2 g0 = mul2(p0, q0), g1 = mul2(p1, q1);
          p[e] = p0.x; p[e + 1] = p0.y; p[e + 2] = p1.x; p[e + 3] = p1.y;
          ds[e] = g0.x; ds[e + 1] = g0.y; ds[e + 2] = g1.x; ds[e + 3] = g1.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int qq = 32 * h + e;
          const bool valid = i * FB + qq < a.S && (i != kb || qq >= r);
          const float pv = valid ? ex2f(fmaf(p[e], c2, nls[e])) : 0.f;
          p[e] = pv;
          ds[e] = pv * fmaf(ds[e], scale, nds[e]);
        }
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = pack_bf2(p[2 * e], p[2 * e + 1]);
      // P^T's buffer was read by dV of block it-1; dS^T buffer b by dK and the store of block it-2
      if (it >= 1) ok = ok && mbar_wait(&bar_free[(it - 1) % NS], (uint32_t)(((it - 1) / NS) & 1));
      if (it >= 2 && store_ds) ok = ok && mbar_wait(&bar_dsread[bd], (uint32_t)(((it - 2) >> 1) & 1));
      __syncwarp();
      tc_fence_after();
      tmem_st16(t_row + C::T_P + 16 * h, pk);
      uint8_t* dsb = sm + C::OFF_DS + bd * 2 * CHUNK;
#pragma unroll
      for (int g = 0; g < 4; ++g) put8(dsb, r, 4 * h + g, ds + 8 * g);
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pready[bd]);
    }
    ok = ok && mbar_wait(bar_o, 0);
    __syncwarp();
  }
  if (__syncthreads_or(!ok)) {
    if (issuer && lane == 0) {
      atomicOr(err, DEVERR_WAIT_TIMEOUT);
      drain(bar_kv, 1, &w_kv);
      for (int s = 0; s < NS; ++s) drain(&bar_ld[s], n_ld[s], &w_ld[s]);
      umma_commit(bar_x);
      mbar_wait(bar_x, 0);
    }
  } else if (!issuer) {
    tc_fence_after();
    const int key = kb * FB + r;
    const int bb = a.zm.b(item), hh = a.zm.h(item);
    const bool row_ok = key < a.S;
    const int64_t row = row_ok ? a.tm.row(bb, key) * a.ldd : 0;
    // quarters 0, 1: the two halves of dV; quarters 2, 3: of dK
    const int c0 = (h & 1) * (HD / 2);
    if (h < 2)
      store_row<HD / 2>(t_row + C::T_DV + c0, row_ok, a.dv + row + a.dv_col + (int64_t)hh * HD + c0, 1.f);
    else
      store_row<HD / 2>(t_row + C::T_DK + c0, row_ok, a.dk + row + a.dk_col + (int64_t)hh * HD + c0, 1.f);
  }
  if (issuer && lane == 0 && store_ds) bulk_wait_all();  // stores finished before shared memory goes
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD>
struct QCfg {
  static constexpr int TILE = FB * HD * 2;
  static constexpr int NS = 2;  // stages of (K, V)
  static constexpr int OFF_Q = 0, OFF_DO = TILE, OFF_ST = 2 * TILE;  // stage s: K, then V
  static constexpr int OFF_DS = OFF_ST + NS * 2 * TILE;
  static constexpr int OFF_BAR = OFF_DS + 2 * CHUNK;
  static constexpr int SMEM = OFF_BAR + 128 + 1024;
};

// Per CTA: query block qb = nqb-1 - blockIdx / nz, item blockIdx % nz. For
// each key block j <= qb:
//   S = Q K_j^T, dP = dO V_j^T                  (TMEM columns 0..127, 128..255)
//   dS = scale * P (dP - D), P = 2^(S c2 - lse)  (rows = queries, in smem)
//   dQ += dS K_j                                (TMEM columns 256..)
template <int HD>
__global__ void __launch_bounds__(kBwdThreads, 1)
    flash_bwd_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const FlashArgs a, int nqb, float c2, float scale, uint32_t* err) {
  using C = QCfg<HD>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_qd = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* bar_ld = bar_qd + 1;    // [2]
  uint64_t* bar_free = bar_qd + 3;  // [2]
  uint64_t* bar_s = bar_qd + 5;
  uint64_t* bar_o = bar_qd + 6;
  uint64_t* bar_x = bar_qd + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_qd + 8);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = tid & (FB - 1), hf = tid >> 7;  // row of the tile, column half
  const int qb = nqb - 1 - (int)(blockIdx.x / a.nz);
  const int item = (int)(blockIdx.x % a.nz);
  const int z = (int)a.zm.z(item);
  const int n = qb + 1;
  const int q = qb * FB + r;
  const float lse_r = q < a.S ? a.lse[(int64_t)z * a.S + q] : 0.f;
  const float d_r = q < a.S ? a.D[(int64_t)z * a.S + q] : 0.f;

  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(bar_qd + i, 1);
    mbar_fence_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
    tma_prefetch_map(&tmdO);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the prologue above overlaps the previous kernel
  pdl_trigger();
  const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const uint32_t s_q = smem_u32(sm + C::OFF_Q), s_do = smem_u32(sm + C::OFF_DO);
  const uint32_t s_ds = smem_u32(sm + C::OFF_DS);

  auto load_kv = [&](int s, int j) {
    uint8_t* dst = sm + C::OFF_ST + s * 2 * C::TILE;
    mbar_arrive_expect_tx(&bar_ld[s], 2 * C::TILE);
    load_tile<HD>(&tmK, dst, &bar_ld[s], j * FB, z);
    load_tile<HD>(&tmV, dst + C::TILE, &bar_ld[s], j * FB, z);
  };
  int n_ld[2] = {0, 0}, w_ld[2] = {0, 0}, w_qd = 0;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_qd, 2 * C::TILE);
    load_tile<HD>(&tmQ, sm + C::OFF_Q, bar_qd, qb * FB, z);
    load_tile<HD>(&tmdO, sm + C::OFF_DO, bar_qd, qb * FB, z);
    for (int it = 0; it < NS && it < n; ++it) {
      load_kv(it, it);
      n_ld[it] = 1;
    }
  }

  bool ok = true, aborted = false;
  for (int j = 0; j < n; ++j) {
    const int st = j % NS;
    if (tid == 0) {
      if (j == 0) {
        ok = mbar_wait(bar_qd, 0);
        w_qd = ok ? 1 : 0;
      }
      if (ok) {
        ok = mbar_wait(&bar_ld[st], (uint32_t)((j / NS) & 1));
        if (ok) ++w_ld[st];
      }
      if (ok) {
        tc_fence_after();
        const uint32_t s_kt = smem_u32(sm + C::OFF_ST + st * 2 * C::TILE), s_vt = s_kt + C::TILE;
        constexpr uint32_t idesc = make_idesc(FB, FB, false, false);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16(tmem, desc_k(s_q, kk), desc_k(s_kt, kk), idesc, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16(tmem + FB, desc_k(s_do, kk), desc_k(s_vt, kk), idesc, kk > 0 ? 1u : 0u);
        umma_commit(bar_s);
      }
      // refill the stage freed by iteration j-1 (after the issue, so the MMAs
      // queue back to back)
      if (ok && j >= 1 && j + NS - 1 < n) {
        const int s2 = (j + NS - 1) % NS;
        ok = mbar_wait(&bar_free[s2], (uint32_t)(((j - 1) / NS) & 1));
        if (ok) {
          load_kv(s2, j + NS - 1);
          ++n_ld[s2];
        }
      }
    }
    if (ok) ok = mbar_wait(bar_s, (uint32_t)(j & 1));
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    tc_fence_after();
    const bool diag = j == qb;
    uint8_t* dst = sm + C::OFF_DS;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {  // this thread's 64 key columns
      const int c = 2 * hf + cc;
      uint32_t sv[32], dv[32];
      tmem_ld32_nw(t_row + 32 * c, sv);
      tmem_ld32_nw(t_row + FB + 32 * c, dv);
      tmem_wait_ld();
      float ds[32];
      if (!diag) {
        const float2 c22 = make_float2(c2, c2), ml = make_float2(-lse_r, -lse_r);
        const float2 sc2 = make_float2(scale, scale), md = make_float2(-d_r, -d_r);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 t = fma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c22, ml);
          const float2 pv = make_float2(ex2f(t.x), ex2f(t.y));
          const float2 dq = add2(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), md);
          const float2 d2 = mul2(mul2(pv, sc2), dq);
          ds[e] = d2.x; ds[e + 1] = d2.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const bool valid = 32 * c + e <= r;
          const float pv = valid ? ex2f(fmaf(__uint_as_float(sv[e]), c2, -lse_r)) : 0.f;
          ds[e] = pv * scale * (__uint_as_float(dv[e]) - d_r);
        }
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) put8(dst, r, 4 * c + g, ds + 8 * g);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
      tc_fence_after();
      const uint32_t s_kt = smem_u32(sm + C::OFF_ST + st * 2 * C::TILE);
      constexpr uint32_t idesc = make_idesc(FB, HD, false, true);
#pragma unroll
      for (int kk = 0; kk < FB / 16; ++kk)
        umma_bf16(tmem + 2 * FB, desc_k(s_ds, kk), desc_mn(s_kt, kk), idesc, (j > 0 || kk > 0) ? 1u : 0u);
      umma_commit(&bar_free[st]);
    }
  }
  if (!aborted) {
    if (tid == 0 && ok) umma_commit(bar_o);
    if (ok) ok = mbar_wait(bar_o, 0);
    if (__syncthreads_or(!ok)) aborted = true;
  }
  if (!aborted) {
    tc_fence_after();
    const int b = a.zm.b(item), h = a.zm.h(item);
    const bool row_ok = q < a.S;
    const int64_t row = row_ok ? a.tm.row(b, q) * a.ldd : 0;
    const int c0 = hf * (HD / 2);
    store_row<HD / 2>(t_row + 2 * FB + c0, row_ok, a.dq + row + a.dq_col + (int64_t)h * HD + c0, 1.f);
  } else if (tid == 0) {
    atomicOr(err, DEVERR_WAIT_TIMEOUT);
    drain(bar_qd, 1, &w_qd);
    drain(&bar_ld[0], n_ld[0], &w_ld[0]);
    drain(&bar_ld[1], n_ld[1], &w_ld[1]);
    umma_commit(bar_x);
    mbar_wait(bar_x, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side

// Opt a kernel into `bytes` of dynamic shared memory, once per kernel: each
// caller passes its own once_flag and result slot (kernels of one signature
// share a function-pointer type, so a static inside a template on that type
// would be shared between them).
template <typename K>
nnt_status allow_smem(K kern, int bytes, std::once_flag& once, cudaError_t& e) {
  std::call_once(once, [&] { e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes); });
  if (e != cudaSuccess) {
    set_thread_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return NNT_ERR_CUDA;
  }
  return NNT_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

nnt_status check_args(const FlashArgs& a, const void* q, const void* k, const void* v) {
  NNT_CHECK_ARG(flash_supported(a.hd), "flash attention: head size %d (supported: 64, 128)", a.hd);
  NNT_CHECK_ARG(a.S > 0 && a.nz > 0 && a.z_total > 0, "flash attention: empty problem");
  NNT_CHECK_ARG(a.nz <= 65535, "flash attention: more than 65535 (sequence, head) items in one launch");
  NNT_CHECK_ARG(a.zm.z(a.nz - 1) < a.z_total && a.zm.z(0) >= 0, "flash attention: item out of range");
  NNT_CHECK_ARG(q && k && v && aligned16(q) && aligned16(k) && aligned16(v),
                "flash attention: q, k, v must be 16-byte aligned device pointers");
  NNT_CHECK_ARG(a.o && aligned16(a.o) && a.ldo % 8 == 0 && a.o_col % 8 == 0 && a.lse,
                "flash attention: O must be 16-byte aligned with ldo, o_col multiples of 8; lse needed");
  return NNT_OK;
}

nnt_status qkv_maps(const FlashArgs& a, const bf16* q, const bf16* k, const bf16* v, CUtensorMap* mq,
                    CUtensorMap* mk, CUtensorMap* mv) {
  const int64_t hd = a.hd, S = a.S;
  NNT_TRY(make_map(mq, q, hd, S, hd, S * hd, a.z_total, 64, FB));
  NNT_TRY(make_map(mk, k, hd, S, hd, S * hd, a.z_total, 64, FB));
  return make_map(mv, v, hd, S, hd, S * hd, a.z_total, 64, FB);
}

template <int HD>
nnt_status fwd_hd(const bf16* q, const bf16* k, const bf16* v, const FlashArgs& a, cudaStream_t st) {
  auto kern = flash_fwd_kernel<HD>;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  NNT_TRY(allow_smem(kern, FwdCfg<HD>::SMEM, once, attr));
  CUtensorMap mq, mk, mv;
  NNT_TRY(qkv_maps(a, q, k, v, &mq, &mk, &mv));
  uint32_t* err = device_error_word();
  NNT_CHECK_ARG(err != nullptr, "device error word unavailable");
  const int nqb = (int)ceil_div(a.S, FB);
  const float c2 = (float)(1.4426950408889634 / sqrt((double)HD));
  launch_pdl(kern, (unsigned)(nqb * a.nz), kThreads, FwdCfg<HD>::SMEM, st, mq, mk, mv, a, nqb, c2, err);
  return launch_check("flash_fwd");
}

template <int HD>
nnt_status bwd_hd(const bf16* q, const bf16* k, const bf16* v, const bf16* dO, const FlashArgs& a,
                  cudaStream_t st) {
  // head size 64: the warp-specialised dK/dV kernel; 128 leaves no tensor
  // memory for K, V and P^T and takes the block-synchronous one
  void (*kv)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, int, FlashArgs, int, float,
             float, uint32_t*);
  int kv_smem, kv_threads;
  if constexpr (HD == 64) {
    kv = flash_bwd_kv_ws_kernel;
    kv_smem = KvWsCfg::SMEM;
    kv_threads = kKvWsThreads;
  } else {
    kv = flash_bwd_kv_kernel<HD>;
    kv_smem = KvCfg<HD>::SMEM;
    kv_threads = kKvThreads;
  }
  auto qk = flash_bwd_q_kernel<HD>;
  static std::once_flag once_kv, once_q;
  static cudaError_t attr_kv = cudaSuccess, attr_q = cudaSuccess;
  NNT_TRY(allow_smem(kv, kv_smem, once_kv, attr_kv));
  NNT_TRY(allow_smem(qk, QCfg<HD>::SMEM, once_q, attr_q));
  CUtensorMap mq, mk, mv, mdo;
  NNT_TRY(qkv_maps(a, q, k, v, &mq, &mk, &mv));
  NNT_TRY(make_map(&mdo, dO, a.hd, a.S, a.hd, (int64_t)a.S * a.hd, a.z_total, 64, FB));
  uint32_t* err = device_error_word();
  NNT_CHECK_ARG(err != nullptr, "device error word unavailable");
  const int nqb = (int)ceil_div(a.S, FB);
  const double scale = 1.0 / sqrt((double)HD);
  const float c2 = (float)(1.4426950408889634 * scale);
  launch_pdl(flash_bwd_d_kernel, dim3((unsigned)ceil_div(a.S, 32), (unsigned)a.nz), 256, 0, st, dO, a);
  NNT_TRY(launch_check("flash_bwd_d"));
  const bool via_gemm = a.ds && a.S % 8 == 0;
  CUtensorMap mds = mq;  // unused unless via_gemm
  if (via_gemm) NNT_TRY(make_map(&mds, a.ds, a.S, a.S, a.S, (int64_t)a.S * a.S, a.z_total, 64, FB));
  launch_pdl(kv, (unsigned)(nqb * a.nz), kv_threads, kv_smem, st, mq, mk, mv, mdo, mds, via_gemm ? 1 : 0, a, nqb,
             c2, (float)scale, err);
  NNT_TRY(launch_check("flash_bwd_kv"));
  if (!via_gemm) {
    launch_pdl(qk, (unsigned)(nqb * a.nz), kBwdThreads, QCfg<HD>::SMEM, st, mq, mk, mv, mdo, a, nqb, c2, (float)scale, err);
    return launch_check("flash_bwd_q");
  }
  // dQ[q] = sum_{k <= q} dS[q][k] K[k]: A = dS^T read MN-major, causal key range per query tile
  GemmArgs g;
  g.M = a.S; g.N = HD; g.K = a.S;
  g.nbatch = a.nz; g.zm = a.zm;
  g.m0 = 0; g.mt = a.S; g.n0 = 0; g.nt = HD;
  g.A = a.ds; g.lda = a.S; g.a_zs = (int64_t)a.S * a.S; g.a_trans = 1;
  g.B = k; g.ldb = HD; g.b_zs = (int64_t)a.S * HD; g.b_trans = 1;
  g.op_dtype = NNT_BF16;
  g.C = a.dq; g.ldc = a.ldd; g.c_dtype = NNT_BF16; g.out_mode = OUT_HEADMERGE;
  g.c_col_off = a.dq_col; g.hs_hd = HD; g.hs_H = a.zm.H; g.hs_B = (int)(a.z_total / a.zm.H); g.hs_S = a.S;
  g.tm = a.tm;
  g.causal = CAUSAL_K_UPPER;
  return gemm(g, 0, st);
}

}  // namespace

bool flash_supported(int hd) { return hd == 64 || hd == 128; }

nnt_status launch_flash_fwd(const bf16* q, const bf16* k, const bf16* v, const FlashArgs& a,
                            cudaStream_t st) {
  NNT_TRY(check_args(a, q, k, v));
  return a.hd == 64 ? fwd_hd<64>(q, k, v, a, st) : fwd_hd<128>(q, k, v, a, st);
}

nnt_status launch_flash_bwd(const bf16* q, const bf16* k, const bf16* v, const bf16* dO,
                            const FlashArgs& a, cudaStream_t st) {
  NNT_TRY(check_args(a, q, k, v));
  NNT_CHECK_ARG(dO && aligned16(dO) && a.D && a.dq && a.dk && a.dv && aligned16(a.dq) &&
                    aligned16(a.dk) && aligned16(a.dv) && a.ldd % 8 == 0 && a.dq_col % 8 == 0 &&
                    a.dk_col % 8 == 0 && a.dv_col % 8 == 0,
                "flash attention backward: dO, D and 16-byte aligned dq, dk, dv (ldd and column "
                "offsets multiples of 8) needed");
  return a.hd == 64 ? bwd_hd<64>(q, k, v, dO, a, st) : bwd_hd<128>(q, k, v, dO, a, st);
}

}  // namespace nnt
