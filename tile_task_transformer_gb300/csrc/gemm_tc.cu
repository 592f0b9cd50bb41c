// Tensor-core tile GEMM for sm_103a: tcgen05.mma (kind::f16, bf16 in, fp32
// accumulate in TMEM) fed by TMA, with the step's fused epilogues.
//
// The linear layers and the attention products QK^T, PV and their backward
// products are the dense contractions of the step (review page "What carries
// the argument": linear and attention tile tasks). One kernel covers all of
// them: operands may be K-major or MN-major (weights [out, in] used as-is for
// x W^T, dY W and dY^T X without transposes), batched over (sequence, head),
// with the causal tile rules of gemm.cuh.
//
// Structure (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: 128x64 A box and BNx64 B box per k-block into a
//               ring of shared-memory stages (128-byte swizzle), signalled by
//               mbarrier transaction counts;
//   warp 1      allocates 2*BN TMEM columns (two accumulators) and issues the
//               MMAs (128 x BN x 16 each, four per k-block) from one thread;
//               tcgen05.commit frees a stage / publishes an accumulator;
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time from their TMEM lane
//               quarter, apply bias / residual / GELU / layout, store; the
//               accumulator is handed back so the next tile's MMAs overlap.
// Every mbarrier wait is bounded: on expiry the kernel sets the device error
// word, stops issuing work, waits (bounded) for its own copies in flight,
// frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "gemm.cuh"
#include "ptx_math.cuh"
#include "tc_ptx.cuh"

namespace nnt {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Operand stored [Z][outer][ld] with `inner` contiguous elements per row.
nnt_status make_map(CUtensorMap* map, const void* base, int64_t inner, int64_t outer, int64_t ld,
                    int64_t zs, int64_t Z, int box_inner, int box_outer) {
  auto fn = encode_fn();
  if (!fn) {
    set_thread_error("cuTensorMapEncodeTiled is unavailable");
    return NNT_ERR_CUDA;
  }
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)Z};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)zs * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_thread_error("cuTensorMapEncodeTiled failed (%d): dims %lld x %lld x %lld, ld %lld, zs %lld",
                     (int)r, (long long)inner, (long long)outer, (long long)Z, (long long)ld,
                     (long long)zs);
    return NNT_ERR_INVALID_ARG;
  }
  return NNT_OK;
}

namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = 128 bytes: one swizzle row
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each on half of the tile's columns
constexpr int kThreads = 64 + 32 * kEpiWarps;

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN >= 192 ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int TMEM_COLS = BN == 192 ? 512 : 2 * BN;  // two accumulators, power of two
  static constexpr int BAR_BYTES = 256;
  // per epilogue warp: one 4 KB buffer -- a 32x32 fp32 output chunk, or a
  // 32x32 bf16 output chunk plus its 32x32 bf16 GELU input chunk
  static constexpr int STAGING_BYTES = kEpiWarps * 4096;
  static constexpr int SMEM = STAGES * STAGE + STAGING_BYTES + BAR_BYTES + 1024;
};

// Output-tile space of one launch (host-computed).
struct TileSpace {
  int mt0, n_mt, nt0, n_nt;
  int total;
  int c_mode;   // 0: direct stores; 1: TMA store, window map; 2: TMA head split; 3: TMA head merge
  int aux_tma;  // 1: GELU input u written by TMA store (window map)
};

struct TileCoord {
  int i, m_box, m_start, m_end, n_box, n_start, n_end, kb_lo, kb_hi;
  bool needed;
};

// Tile order: batch item, then groups of kGroupM m-tiles; inside a group the m
// index runs fastest. CTAs working at the same time then share a band of A rows
// and a band of B rows, which stay in L2.
constexpr int kGroupM = 16;

template <int BN>
__device__ __forceinline__ TileCoord tile_at(const GemmArgs& g, const TileSpace& ts, int t) {
  TileCoord c;
  const int per_batch = ts.n_mt * ts.n_nt;
  c.i = t / per_batch;
  const int r = t - c.i * per_batch;
  const int grp = r / (kGroupM * ts.n_nt);
  const int m_base = grp * kGroupM;
  const int gs = min(kGroupM, ts.n_mt - m_base);
  const int rr = r - grp * kGroupM * ts.n_nt;
  const int im = m_base + rr % gs;
  const int in = rr / gs;
  c.m_box = (ts.mt0 + im) * BM;
  c.m_start = max(g.m0, c.m_box);
  c.m_end = min(g.m0 + g.mt, c.m_box + BM);
  c.n_box = (ts.nt0 + in) * BN;
  c.n_start = max(g.n0, c.n_box);
  c.n_end = min(g.n0 + g.nt, c.n_box + BN);
  c.needed = causal_tile_needed(g, c.m_start, c.m_end, c.n_start);
  int k_lo, k_hi;
  causal_k_range(g, c.m_start, c.m_end, k_lo, k_hi);
  c.kb_lo = k_lo / BK;
  c.kb_hi = (k_hi + BK - 1) / BK;
  return c;
}

// tanh-form GELU and its derivative through the logistic function:
// (1 + tanh(x)) / 2 = 1 / (1 + e^(-2x)), so with x = c (u + a u^3) and
// s = 1 / (1 + 2^(-2x log2 e)):  gelu(u) = u s,  gelu'(u) = s + 2 u s (1 - s) x'
// (x' = c (1 + 3 a u^2)). Nothing cancels in the negative tail (where 1 + tanh
// would), and the error is that of ex2.approx (2^-22 relative) and one fast
// division: fp32-accurate.
__device__ __forceinline__ float gelu_sig_fast(float u) {
  const float c2l = 2.0f * 0.7978845608028654f * 1.4426950408889634f, a = 0.044715f;
  // the exponent is capped at 64 (s ~ 5e-20 there) so the division stays in its normal range
  return __fdividef(1.0f, 1.0f + ex2f(fminf(-c2l * (u + a * u * u * u), 64.0f)));
}
__device__ __forceinline__ float gelu_grad_from_sig(float u, float s) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  return s + 2.0f * u * s * (1.0f - s) * c * (1.0f + 3.0f * a * u * u);
}

// Elementwise epilogue of one 32-column chunk of row m held in registers
// (columns nb..nb+31; `full`: all of them inside the window). Bias loads are
// the same address across the warp (broadcast). `pre` holds this row's 32
// residual (EPI_STORE) or GELU-derivative (EPI_GELU_BWD) values when the chunk lies
// wholly inside the window (loaded coalesced and transposed through shared
// memory by the caller); otherwise they are read here element by element.
__device__ __forceinline__ void epi_chunk(const GemmArgs& g, int i, int m, bool row_ok, int nb,
                                          int n_lo, int n_hi, bool full, float* v, float* u_out,
                                          const float* pre) {
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] *= g.alpha;
  if (g.bias) {
    if (full) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(g.bias + nb) + k);
        v[4 * k] += b.x; v[4 * k + 1] += b.y; v[4 * k + 2] += b.z; v[4 * k + 3] += b.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (nb + j >= n_lo && nb + j < n_hi) v[j] += g.bias[nb + j];
    }
  }
  if (g.epi == EPI_STORE) {
    if (g.resid && row_ok) {
      if (pre) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += pre[j];
      } else {
        const float* add = g.resid + (int64_t)m * g.ld_resid;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (nb + j >= n_lo && nb + j < n_hi) v[j] += add[nb + j];
      }
    }
    if (g.beta && row_ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (nb + j >= n_lo && nb + j < n_hi) v[j] += static_cast<const float*>(g.C)[out_offset(g, i, m, nb + j)];
    }
  } else if (g.epi == EPI_GELU) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float s = gelu_sig_fast(v[j]);
      u_out[j] = gelu_grad_from_sig(v[j], s);  // aux: gelu'(u) for the backward
      v[j] *= s;
    }
  } else if (row_ok) {  // EPI_GELU_BWD: times the stored gelu'(u)
    if (pre) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= pre[j];
    } else {
      const int64_t ub = (int64_t)m * g.ld_aux;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (nb + j >= n_lo && nb + j < n_hi) v[j] *= aux_load(g, ub + nb + j);
    }
  }
}

// Row `lane` of a 32x32 chunk into shared memory in the TMA 128-byte (fp32) or
// 64-byte (bf16) swizzled box layout: 16-byte piece k of row r goes to
// position k ^ (r & 7) (fp32) or k ^ ((r >> 1) & 3) (bf16), so the eight lanes
// of a quarter-warp hit different banks.
__device__ __forceinline__ void stage_f32(uint8_t* st, int lane, const float* v) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    *reinterpret_cast<float4*>(st + lane * 128 + ((k ^ (lane & 7)) << 4)) =
        make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}
__device__ __forceinline__ void stage_bf16(uint8_t* st, int lane, const float* v) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4 pk;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * k], v[8 * k + 1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * k + 2], v[8 * k + 3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * k + 4], v[8 * k + 5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * k + 6], v[8 * k + 7]);
    pk.x = *reinterpret_cast<uint32_t*>(&h0);
    pk.y = *reinterpret_cast<uint32_t*>(&h1);
    pk.z = *reinterpret_cast<uint32_t*>(&h2);
    pk.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(st + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) = pk;
  }
}

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmU,
                   const GemmArgs g, const TileSpace ts, uint32_t* err) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE + C::STAGING_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 32 * kEpiWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the prologue above (barriers, TMEM, descriptor prefetch) overlaps the
  // previous kernel; from here on global memory is read and written
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      for (int t = blockIdx.x; t < ts.total && !*abort_flag; t += gridDim.x) {
        const TileCoord c = tile_at<BN>(g, ts, t);
        if (!c.needed) continue;
        const int z = (int)g.zm.z(c.i);
        for (int kb = c.kb_lo; kb < c.kb_hi; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, g.wait_ns)) {
            atomicOr(err, DEVERR_WAIT_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          uint8_t* sa = smem + s * C::STAGE;
          uint8_t* sb = sa + C::A_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE);
          const int k = kb * BK;
          if (A_MN) {
            tma_load_3d(sa, &tmA, &full[s], c.m_box, k, z);
            tma_load_3d(sa + 8192, &tmA, &full[s], c.m_box + 64, k, z);
          } else {
            tma_load_3d(sa, &tmA, &full[s], k, c.m_box, z);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_3d(sb + j * 8192, &tmB, &full[s], c.n_box + 64 * j, k, z);
          } else {
            tma_load_3d(sb, &tmB, &full[s], k, c.n_box, z);
          }
          ++issued;
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // wait (bounded) until every copy issued into the ring has landed
      int outstanding = issued < C::STAGES ? issued : C::STAGES;
      int ss = s;
      uint32_t pp = ph;
      for (int j = 0; j < outstanding; ++j) {
        if (--ss < 0) {
          ss = C::STAGES - 1;
          pp ^= 1;
        }
        if (!mbar_wait(&full[ss], pp, g.wait_ns)) atomicOr(err, DEVERR_WAIT_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = make_idesc(BM, BN, A_MN, B_MN);
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      for (int t = blockIdx.x; t < ts.total && !*abort_flag; t += gridDim.x) {
        const TileCoord c = tile_at<BN>(g, ts, t);
        if (!c.needed) continue;
        if (!mbar_wait(&tempty[acc], aph ^ 1, g.wait_ns)) {
          atomicOr(err, DEVERR_WAIT_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = c.kb_lo; kb < c.kb_hi; ++kb) {
          if (!mbar_wait(&full[s], ph, g.wait_ns)) {
            atomicOr(err, DEVERR_WAIT_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::STAGE);
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? make_sdesc(sa + kk * 2048, 8192, 1024)
                                     : make_sdesc(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? make_sdesc(sb + kk * 2048, 8192, 1024)
                                     : make_sdesc(sb + kk * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb > c.kb_lo || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
          if (++s == C::STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          aph ^= 1;
        }
      }
    }
  } else {
    // ---------------- epilogue: warps 2..9; warp w drains TMEM lane quarter
    // w % 4 (the quarter a warp may access) and half (w - 2) / 4 of the tile's
    // 32-column chunks
    const int q = warp & 3;
    const int nch = BN / 64;  // chunks per warp
    const int ch0 = ((warp - 2) >> 2) * nch;
    // Staging: one 4 KB buffer per warp (an fp32 chunk, or a bf16 chunk and
    // its bf16 GELU-input chunk), reused once the previous bulk store has
    // read it; the other warps' work covers that wait. A GELU epilogue with
    // an fp32 output or fp32 u stores directly.
    uint8_t* stage_base = smem + C::STAGES * C::STAGE + (warp - 2) * 4096;
    const bool cbf = g.c_dtype == NNT_BF16;
    const bool gelu = g.epi == EPI_GELU;
    const bool ubf = g.aux_dtype == NNT_BF16;
    const bool gelu_direct = gelu && !(cbf && ubf);
    // residual (EPI_STORE) or GELU derivative (EPI_GELU_BWD): each chunk's 32x32
    // block is read coalesced one chunk ahead and turned into one row per lane
    // through the chunk's (free) output staging buffer
    const void* src = g.epi == EPI_GELU_BWD ? g.aux : (g.epi == EPI_STORE ? g.resid : nullptr);
    const bool src_bf = g.epi == EPI_GELU_BWD && ubf;
    const int64_t ld_src = g.epi == EPI_GELU_BWD ? g.ld_aux : g.ld_resid;
    int issued = 0;  // bulk store groups of this warp so far
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < ts.total && !*abort_flag; t += gridDim.x) {
      const TileCoord c = tile_at<BN>(g, ts, t);
      if (!c.needed) continue;
      const int row0 = c.m_box + q * 32;
      const int m = row0 + lane;
      const bool row_ok = m >= c.m_start && m < c.m_end;
      const bool rows_full = row0 >= c.m_start && row0 + 32 <= c.m_end;
      // fp32: lane reads rows 4*rr + lane/8 of the block, 16 bytes at column
      // 4*(lane%8); bf16: rows 8*rr + lane/4, 16 bytes at column 8*(lane%4)
      uint4 pf[8];
      auto prefetch = [&](int nb_) {
        const bool whole = src && rows_full && nb_ >= c.n_start && nb_ + 32 <= c.n_end;
        if (whole) {
          if (src_bf) {
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
              pf[rr] = __ldg(reinterpret_cast<const uint4*>(static_cast<const bf16*>(src) +
                                                            (int64_t)(row0 + 8 * rr + (lane >> 2)) * ld_src +
                                                            nb_ + 8 * (lane & 3)));
          } else {
#pragma unroll
            for (int rr = 0; rr < 8; ++rr)
              pf[rr] = __ldg(reinterpret_cast<const uint4*>(static_cast<const float*>(src) +
                                                            (int64_t)(row0 + 4 * rr + (lane >> 3)) * ld_src +
                                                            nb_ + 4 * (lane & 7)));
          }
        }
        return whole;
      };
      // the first chunk's residual / GELU-derivative block does not depend on
      // the accumulator: its loads are in flight while the MMAs finish
      bool have = prefetch(c.n_box + ch0 * 32);
      if (!mbar_wait(&tfull[acc], aph, g.wait_ns)) {
        atomicOr(err, DEVERR_WAIT_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int ch = ch0; ch < ch0 + nch; ++ch) {
        const int nb = c.n_box + ch * 32;
        if (nb >= c.n_end) break;  // uniform across the warp
        float v[32], u[32], pre[32];
        tmem_ld32(tbase + ch * 32, v);
        if (row0 >= c.m_end) continue;  // no row of this warp in the window (uniform)
        const bool cols_full = nb >= c.n_start && nb + 32 <= c.n_end;
        bool tma;
        if (ts.c_mode == 1) tma = row0 >= c.m_start && nb >= c.n_start;
        else tma = ts.c_mode > 1 && rows_full && cols_full;
        if (tma && gelu && (!ts.aux_tma || gelu_direct)) tma = false;
        uint8_t* stage_c = stage_base;
        uint8_t* stage_u = stage_base + 2048;
        const bool have_cur = have;
        if ((tma || have_cur) && issued >= 1) {
          // the group that last used the buffer must have finished reading it
          if (lane == 0) bulk_wait_read();
          __syncwarp();
        }
        if (have_cur) {
          if (src_bf) {
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int rl = 8 * rr + (lane >> 2);
              *reinterpret_cast<uint4*>(stage_c + rl * 64 + (((lane & 3) ^ ((rl >> 1) & 3)) << 4)) = pf[rr];
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 x = *reinterpret_cast<const uint4*>(stage_c + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4));
              const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
                pre[8 * k + 2 * e] = f2.x;
                pre[8 * k + 2 * e + 1] = f2.y;
              }
            }
          } else {
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
              const int rl = 4 * rr + (lane >> 3);
              *reinterpret_cast<uint4*>(stage_c + rl * 128 + (((lane & 7) ^ (rl & 7)) << 4)) = pf[rr];
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float4 x = *reinterpret_cast<const float4*>(stage_c + lane * 128 + ((k ^ (lane & 7)) << 4));
              pre[4 * k] = x.x; pre[4 * k + 1] = x.y; pre[4 * k + 2] = x.z; pre[4 * k + 3] = x.w;
            }
          }
          __syncwarp();
        }
        have = ch + 1 < ch0 + nch && prefetch(nb + 32);  // next chunk's block, in flight meanwhile
        epi_chunk(g, c.i, m, row_ok, nb, c.n_start, c.n_end, cols_full, v, u, have_cur ? pre : nullptr);
        if (!tma) {
          if (row_ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int n = nb + j;
              if (n < c.n_start || n >= c.n_end) continue;
              if (g.epi == EPI_GELU) aux_store(g, (int64_t)m * g.ld_aux + n, u[j]);
              const int64_t o = out_offset(g, c.i, m, n);
              if (cbf) static_cast<bf16*>(g.C)[o] = __float2bfloat16_rn(v[j]);
              else static_cast<float*>(g.C)[o] = v[j];
            }
          }
          continue;
        }
        if (cbf) stage_bf16(stage_c, lane, v);
        else stage_f32(stage_c, lane, v);
        if (gelu) {
          if (ubf) stage_bf16(stage_u, lane, u);
          else stage_f32(stage_u, lane, u);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (ts.c_mode == 1) {
            tma_store_3d(&tmC, stage_c, nb - g.n0, row0 - g.m0, (int)g.zm.z(c.i));
          } else if (ts.c_mode == 2) {
            int b, sq;
            g.tm.bs(row0, b, sq);
            const int part = nb / g.hs_d, r = nb - part * g.hs_d;
            const int h = r / g.hs_hd;
            tma_store_5d(&tmC, stage_c, r - h * g.hs_hd, sq, h, b, part);
          } else {
            const int b = g.zm.b(c.i), h = g.zm.h(c.i);
            tma_store_2d(&tmC, stage_c, (int)(g.c_col_off + (int64_t)h * g.hs_hd + nb),
                         (int)g.tm.row(b, row0));
          }
          if (gelu) tma_store_2d(&tmU, stage_u, nb - g.n0, row0 - g.m0);
          bulk_commit();
        }
        ++issued;
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        aph ^= 1;
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// General tiled map (rank 2..5) for the epilogue's bulk stores.
nnt_status make_store_map(CUtensorMap* map, const void* base, bool bf, int rank, const cuuint64_t* dims,
                          const cuuint64_t* stride_bytes) {
  auto fn = encode_fn();
  if (!fn) {
    set_thread_error("cuTensorMapEncodeTiled is unavailable");
    return NNT_ERR_CUDA;
  }
  cuuint32_t box[5] = {32, 32, 1, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank,
                  const_cast<void*>(base), dims, stride_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  bf ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_thread_error("cuTensorMapEncodeTiled (store map) failed (%d)", (int)r);
    return NNT_ERR_INVALID_ARG;
  }
  return NNT_OK;
}

bool al16(int64_t bytes) { return (bytes & 15) == 0; }

// Epilogue store maps and mode for one launch (see TileSpace::c_mode).
nnt_status store_maps(const GemmArgs& g, int64_t zmax, CUtensorMap* mc, CUtensorMap* mu, int& c_mode,
                      int& aux_tma) {
  memset(mc, 0, sizeof *mc);
  memset(mu, 0, sizeof *mu);
  c_mode = 0;
  aux_tma = 0;
  const bool bf = g.c_dtype == NNT_BF16;
  const int64_t es = bf ? 2 : 4;
  const char* C = static_cast<const char*>(g.C);
  if (g.out_mode == OUT_PLAIN) {
    const char* base = C + ((int64_t)(g.m0 - g.c_row0) * g.ldc + g.n0) * es;
    const int64_t zs = g.c_zs > 0 ? g.c_zs : (int64_t)g.M * g.ldc;
    if (al16((int64_t)(uintptr_t)base) && al16(g.ldc * es) && al16(zs * es)) {
      cuuint64_t dims[3] = {(cuuint64_t)g.nt, (cuuint64_t)g.mt, (cuuint64_t)zmax};
      cuuint64_t str[2] = {(cuuint64_t)(g.ldc * es), (cuuint64_t)(zs * es)};
      NNT_TRY(make_store_map(mc, base, bf, 3, dims, str));
      c_mode = 1;
    }
  } else if (g.hs_hd % 32 == 0 && g.tm.ts % 32 == 0 && al16((int64_t)(uintptr_t)C)) {
    if (g.out_mode == OUT_HEADSPLIT) {
      const int64_t hd = g.hs_hd, S = g.hs_S, H = g.hs_H, B = g.hs_B;
      cuuint64_t dims[5] = {(cuuint64_t)hd, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B,
                            (cuuint64_t)(g.N / g.hs_d)};
      cuuint64_t str[4] = {(cuuint64_t)(hd * es), (cuuint64_t)(S * hd * es), (cuuint64_t)(H * S * hd * es),
                           (cuuint64_t)(B * H * S * hd * es)};
      if (g.hs_d % 32 == 0 && al16(hd * es)) {
        NNT_TRY(make_store_map(mc, C, bf, 5, dims, str));
        c_mode = 2;
      }
    } else if (al16(g.ldc * es) && g.c_col_off % 8 == 0) {
      cuuint64_t dims[2] = {(cuuint64_t)g.ldc, (cuuint64_t)((int64_t)g.hs_B * g.hs_S)};
      cuuint64_t str[1] = {(cuuint64_t)(g.ldc * es)};
      NNT_TRY(make_store_map(mc, C, bf, 2, dims, str));
      c_mode = 3;
    }
  }
  if (g.epi == EPI_GELU && c_mode == 1) {
    const bool ub = g.aux_dtype == NNT_BF16;
    const int64_t ues = ub ? 2 : 4;
    const char* base = reinterpret_cast<const char*>(g.aux) + ((int64_t)g.m0 * g.ld_aux + g.n0) * ues;
    if (al16((int64_t)(uintptr_t)base) && al16(g.ld_aux * ues)) {
      cuuint64_t dims[2] = {(cuuint64_t)g.nt, (cuuint64_t)g.mt};
      cuuint64_t str[1] = {(cuuint64_t)(g.ld_aux * ues)};
      NNT_TRY(make_store_map(mu, base, ub, 2, dims, str));
      aux_tma = 1;
    }
  }
  return NNT_OK;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

TileSpace tile_space(const GemmArgs& g, int BN) {
  TileSpace t;
  t.mt0 = g.m0 / BM;
  t.n_mt = (g.m0 + g.mt - 1) / BM - t.mt0 + 1;
  t.nt0 = g.n0 / BN;
  t.n_nt = (g.n0 + g.nt - 1) / BN - t.nt0 + 1;
  t.total = g.nbatch * t.n_mt * t.n_nt;
  t.c_mode = 0;
  t.aux_tma = 0;
  return t;
}

template <int BN, bool A_MN, bool B_MN>
nnt_status launch_tc(const GemmArgs& g, cudaStream_t st) {
  using C = Cfg<BN>;
  auto kern = gemm_tc_kernel<BN, A_MN, B_MN>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (attr_err != cudaSuccess) {
    set_thread_error("cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));
    return NNT_ERR_CUDA;
  }
  const int64_t zmax = g.zm.z(g.nbatch - 1) + 1;
  CUtensorMap ma, mb;
  if (A_MN)
    NNT_TRY(make_map(&ma, g.A, g.M, g.K, g.lda, g.a_zs > 0 ? g.a_zs : (int64_t)g.K * g.lda, zmax, 64, 64));
  else
    NNT_TRY(make_map(&ma, g.A, g.K, g.M, g.lda, g.a_zs > 0 ? g.a_zs : (int64_t)g.M * g.lda, zmax, 64, BM));
  if (B_MN)
    NNT_TRY(make_map(&mb, g.B, g.N, g.K, g.ldb, g.b_zs > 0 ? g.b_zs : (int64_t)g.K * g.ldb, zmax, 64, 64));
  else
    NNT_TRY(make_map(&mb, g.B, g.K, g.N, g.ldb, g.b_zs > 0 ? g.b_zs : (int64_t)g.N * g.ldb, zmax, 64, BN));
  TileSpace ts = tile_space(g, BN);
  CUtensorMap mc, mu;
  NNT_TRY(store_maps(g, zmax, &mc, &mu, ts.c_mode, ts.aux_tma));
  const int grid = std::min(ts.total, num_sms());
  uint32_t* err = device_error_word();
  if (!err) {
    set_thread_error("device error word unavailable");
    return NNT_ERR_CUDA;
  }
  launch_pdl(gemm_tc_kernel<BN, A_MN, B_MN>, grid, kThreads, C::SMEM, st, ma, mb, mc, mu, g, ts, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_thread_error("gemm_tc launch: %s", cudaGetErrorString(e));
    return NNT_ERR_CUDA;
  }
  return NNT_OK;
}

template <int BN>
nnt_status launch_bn(const GemmArgs& g, cudaStream_t st) {
  if (g.a_trans) {
    if (g.b_trans) return launch_tc<BN, true, true>(g, st);
    return launch_tc<BN, true, false>(g, st);
  }
  if (g.b_trans) return launch_tc<BN, false, true>(g, st);
  return launch_tc<BN, false, false>(g, st);
}

// NNT_GEMM_BN=64|128|192|256 forces the tile width (for measurement).
int bn_override() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("NNT_GEMM_BN");
    v = e ? atoi(e) : 0;
    if (v != 64 && v != 128 && v != 192 && v != 256) v = 0;
  }
  return v;
}

// Tile width BN of the 128 x BN output tiles: the one with the best product of
// wave efficiency (tiles over whole waves of one tile per SM) and the relative
// tensor-pipe efficiency of a 128 x BN tile (shared-memory operand traffic per
// MMA grows as BN shrinks), measured on GB300 for K >= 768.
int choose_bn(const GemmArgs& g) {
  if (bn_override()) return bn_override();
  if (g.nt <= 64) return 64;
  const int sms = num_sms();
  double best = 0;
  int best_bn = 64;
  for (int bn : {256, 192, 128, 64}) {
    if (bn > 64 && g.nt <= bn / 2) continue;
    const TileSpace t = tile_space(g, bn);
    const double waves = std::ceil((double)t.total / sms);
    const double eff = (double)t.total / (waves * sms) *
                       (bn == 256 ? 1.0 : bn == 192 ? 0.95 : bn == 128 ? 0.8 : 0.35);
    if (eff > best + 1e-9) {
      best = eff;
      best_bn = bn;
    }
  }
  return best_bn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool gemm_tc_supported(const GemmArgs& g) {
  if (g.op_dtype != NNT_BF16) return false;
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.mt <= 0 || g.nt <= 0 || g.nbatch <= 0) return false;
  if (!aligned16(g.A) || !aligned16(g.B) || !aligned16(g.C)) return false;
  if (g.lda % 8 || g.ldb % 8) return false;
  if (g.a_zs % 8 || g.b_zs % 8) return false;
  if (g.m0 % 8 || g.n0 % 8) return false;
  if (g.c_dtype == NNT_BF16 ? (g.ldc % 8) : (g.ldc % 4)) return false;
  if (g.out_mode == OUT_PLAIN && g.nbatch > 1 && (g.c_dtype == NNT_BF16 ? g.c_zs % 8 : g.c_zs % 4)) return false;
  if (g.out_mode != OUT_PLAIN && (g.hs_hd % 8 || g.c_col_off % 8)) return false;
  if (g.bias && !aligned16(g.bias)) return false;
  if (g.resid && (!aligned16(g.resid) || g.ld_resid % 4)) return false;
  if (g.aux && (!aligned16(g.aux) || g.ld_aux % (g.aux_dtype == NNT_BF16 ? 8 : 4))) return false;
  return true;
}

nnt_status gemm_tc_one(const GemmArgs& g, cudaStream_t st) {
  switch (choose_bn(g)) {
    case 256: return launch_bn<256>(g, st);
    case 192: return launch_bn<192>(g, st);
    case 128: return launch_bn<128>(g, st);
    default: return launch_bn<64>(g, st);
  }
}

// out[(m - c_row0) * ldc + n] (+)= sum over slices s in order of
// ws[s][m - m0][n - n0], for the window rows m and columns n.
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int split, int64_t mt, int nt,
                                     float* C, int64_t ldc, int accumulate) {
  pdl_wait();
  pdl_trigger();
  const int64_t n4 = (int64_t)mt * (nt / 4);
  const int64_t win = (int64_t)mt * nt;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / (nt / 4);
    const int c = (int)(i - r * (nt / 4)) * 4;
    float4 t = *reinterpret_cast<const float4*>(ws + r * nt + c);
    for (int s = 1; s < split; ++s) {
      const float4 u = *reinterpret_cast<const float4*>(ws + s * win + r * nt + c);
      t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
    }
    float4* o = reinterpret_cast<float4*>(C + r * ldc + c);
    if (accumulate) {
      const float4 p = *o;
      t.x += p.x; t.y += p.y; t.z += p.z; t.w += p.w;
    }
    *o = t;
  }
}

// K split into `split` equal slices run as batch items of one launch (operand
// offsets of i*K/split along K, outputs to workspace slice i), then summed.
nnt_status gemm_tc_split(const GemmArgs& g, int split, cudaStream_t st) {
  NNT_CHECK_ARG(g.nt % 4 == 0 && g.ldc % 4 == 0, "split GEMM: output width and ldc must be multiples of 4");
  const int ks = g.K / split;
  GemmArgs b = g;
  b.K = ks;
  b.nbatch = split;
  b.zm = ZMap{0, 0, 1, 1};
  b.a_zs = g.a_trans ? (int64_t)ks * g.lda : ks;
  b.b_zs = g.b_trans ? (int64_t)ks * g.ldb : ks;
  b.C = g.ws - g.n0;  // slice z row m, column n at ws[z * mt*nt + (m - m0) * nt + (n - n0)]
  b.c_row0 = g.m0;
  b.ldc = g.nt;
  b.c_zs = (int64_t)g.mt * g.nt;
  b.beta = 0;
  b.ws = nullptr;
  NNT_TRY(gemm_tc_one(b, st));
  float* out = static_cast<float*>(g.C) + (int64_t)(g.m0 - g.c_row0) * g.ldc + g.n0;
  const int64_t n4 = (int64_t)g.mt * (g.nt / 4);
  const int grid = (int)std::min<int64_t>((n4 + 255) / 256, 4 * num_sms());
  launch_pdl(splitk_reduce_kernel, grid, 256, 0, st, g.ws, split, g.mt, g.nt, out, g.ldc, g.beta);
  return launch_check("splitk_reduce");
}

nnt_status gemm_tc(const GemmArgs& g, cudaStream_t st) {
  if (!gemm_tc_supported(g)) {
    set_thread_error("gemm_tc: unsupported shape/layout");
    return NNT_ERR_INVALID_ARG;
  }
  const int split = gemm_split_k(g, g.ws ? g.ws_elems : 0);
  if (split > 1) return gemm_tc_split(g, split, st);
  return gemm_tc_one(g, st);
}

namespace {
__global__ void wait_selftest_kernel(uint64_t limit_ns, int arrive, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  mbar_fence_init();
  if (arrive) mbar_arrive(&bar);
  if (!mbar_wait(&bar, 0, limit_ns)) atomicOr(err, DEVERR_WAIT_TIMEOUT);
}
}  // namespace

nnt_status launch_wait_selftest(uint64_t limit_ns, bool arrive, cudaStream_t st) {
  uint32_t* err = device_error_word();
  if (!err) {
    set_thread_error("device error word unavailable");
    return NNT_ERR_CUDA;
  }
  launch_pdl(wait_selftest_kernel, 1, 32, 0, st, limit_ns, arrive ? 1 : 0, err);
  return launch_check("wait_selftest");
}

int gemm_split_k(const GemmArgs& g, int64_t ws_elems) {
  if (ws_elems <= 0 || g.out_mode != OUT_PLAIN || g.epi != EPI_STORE || g.c_dtype != NNT_F32 ||
      g.bias || g.resid || g.aux || g.nbatch != 1 || g.alpha != 1.f || g.causal != CAUSAL_NONE)
    return 1;
  const int sms = num_sms();
  const int tiles = tile_space(g, choose_bn(g)).total;
  if (2 * tiles > sms) return 1;
  // the most slices that fill the SMs once, each at least 8 k-blocks deep and
  // an exact share of K (the slices are batch items of one launch)
  int best = 1;
  for (int s = 2; s <= 8; s *= 2) {
    if (tiles * s > sms || g.K % (s * BK) != 0 || g.K / (s * BK) < 8) break;
    if ((int64_t)s * g.mt * g.nt > ws_elems) break;
    best = s;
  }
  return best;
}

}  // namespace nnt
