// GPT2 training step as a static tile-task program, behind the C ABI of nnt.h.
//
// Model: GPT2 with pre-LN blocks, causal multi-head attention, tanh-GELU MLP,
// final LayerNorm and a tied LM head, mean next-token cross-entropy, AdamW
// with decoupled weight decay (first page: title and "Builds on" references
// -- Attention Is All You Need, Layer Normalization, On Layer Normalization in
// the Transformer Architecture, Decoupled Weight Decay Regularization; README
// "Minimal working GPT example": GPT2 config, tile flags, fusedadamw flags,
// --loss-reduction=mean).
//
// Tiling (README flag descriptions): tokens are tiled by batch_tile x
// seq_tile, features by embd_tile / inner_tile, heads by head_tile, the
// vocabulary by vocab_tile. Every layer is emitted as tasks over those tiles
// that declare the tiles they read and write; the executor derives the
// dependency graph and the stream schedule once, at creation.
#include <math.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <string>
#include <thread>
#include <vector>

#include "common.cuh"
#include "executor.h"
#include "flash.cuh"
#include "gemm.cuh"
#include "kernels.cuh"

using namespace nnt;

namespace {

enum TaskType : int {
  TT_EMBED = 0, TT_LN_FWD, TT_GEMM_QKV, TT_GEMM_QK, TT_SOFTMAX_FWD, TT_GEMM_PV, TT_GEMM_ATTN_O,
  TT_GEMM_FC, TT_GEMM_MLP_PROJ, TT_GEMM_LM_HEAD, TT_XENT, TT_LOSS,
  TT_GEMM_LM_DX, TT_GEMM_LM_DW, TT_LN_BWD, TT_LN_PARTS, TT_GEMM_DX, TT_GEMM_DW, TT_COLSUM,
  TT_GEMM_ATTN_BWD, TT_SOFTMAX_BWD, TT_EMB_SORT, TT_EMB_SCATTER, TT_WPE_GRAD, TT_ADAMW,
  TT_ADAMW_HOST, TT_FLASH_FWD, TT_FLASH_BWD, TT_COUNT
};
const char* kTaskNames[TT_COUNT] = {
    "embedding_fwd", "layernorm_fwd", "gemm_qkv", "gemm_qk", "softmax_fwd", "gemm_pv",
    "gemm_attn_out", "gemm_fc_gelu", "gemm_mlp_proj", "gemm_lm_head", "cross_entropy",
    "mean_loss", "gemm_lm_dx", "gemm_lm_dw", "layernorm_bwd", "layernorm_param_grads",
    "gemm_dx", "gemm_dw", "bias_grads", "gemm_attn_bwd", "softmax_bwd", "token_sort",
    "embedding_scatter", "wpe_grad", "adamw", "adamw_host_moments", "flash_attn_fwd",
    "flash_attn_bwd"};


struct ParamInfo {
  std::string name;
  int64_t shape0, shape1;  // shape1 = 0 for vectors
  int64_t off, n;
  int64_t goff = -1;  // gradient offset in the gradient buffer (-1: streamed through the ring)
  int kind;  // 0 weight (normal), 1 bias (normal or 0), 2 ln gain (1), 3 ln bias (0)
};

// A tensor's tile grid: up to 4 tile axes, tile id = base + linear index.
struct TGrid {
  int64_t base = 0;
  int g[4] = {1, 1, 1, 1};
};

// A contiguous run of rows of one parameter that AdamW updates as one task.
struct Chunk {
  int param = 0;
  int64_t r0 = 0, r1 = 1;  // rows (a vector is one row)
  int64_t e0 = 0, n = 0;   // element offset inside the parameter and count
  int t0 = 0, t1 = 1;      // rows of the parameter's gradient tile grid it covers
  bool ring = false;       // gradient streamed through a ring slot
  int slot = -1;           // ring slot, or staging slot for host-resident moments
  int64_t goff = -1;       // offset of the gradient in the gradient buffer
  bool host = false;       // AdamW moments in pinned host memory
  int64_t mv_off = -1;     // offset in the device or host moment pool
};

// graph slot of the accumulating backward (0-3: forward, backward, AdamW, fused)
constexpr int kSlotBwdAcc = 8;

struct AdamHyperDev {
  float lr, b1, b2, eps, wd, bc1, bc2, gscale;
};

thread_local std::string t_model_err;

}  // namespace

struct nnt_model {
  nnt_gpt2_config cfg;
  nnt_tiles tiles;
  nnt_options opts;
  int act = NNT_BF16;
  size_t act_size = 2;
  int L, d, H, hd, f, V, S, B, T;
  int tb, ts, te, ti, th, tv;
  int n_bt, n_st, n_ht, n_tok, TT, nce, ncf, ncv;
  TokMap tm;
  int64_t ldz, lddz;
  int backend = 0;
  int gemm_min_cols = 2048;
  std::string err;

  // memory
  std::vector<void*> dev_allocs;
  uint64_t device_bytes = 0, host_bytes = 0;
  // dry run: plan the allocations (count bytes, allocate nothing)
  bool dry = false;
  uint64_t free_device = 0;  // free device memory the plan assumes

  // parameters (flat fp32 buffers + bf16 copy, same offsets)
  std::vector<ParamInfo> params;
  int64_t n_flat = 0, n_scalar = 0;
  float *master = nullptr, *grad = nullptr, *mom1 = nullptr, *mom2 = nullptr;
  bf16* wbf = nullptr;
  AdamHyperDev* hyper_dev = nullptr;
  AdamHyperDev hyper_host{};

  // activations
  uint16_t* tokens_dev = nullptr;
  std::vector<float*> x, xmid, mu1, r1, mu2, r2;
  std::vector<void*> h1, qkvh, P, O, h2, g;
  // gelu'(u) of the FC pre-activation u (activation dtype), written by the FC
  // epilogue for the GELU backward
  std::vector<void*> u;
  float* scores = nullptr;  // [B*H][S][S] fp32, reused by every layer (fwd scores, bwd dP)
  // fused attention (flash): per-layer row log-sum-exp [B*H][S] and the
  // backward's D = rowsum(dO * O) scratch [B*H][S]; no P or scores buffers
  bool flash = false;
  std::vector<float*> lse;
  float* attn_d = nullptr;
  bf16* attn_ds = nullptr;  // [B*H][S][S] dS^T of the backward (its dQ is then a GEMM)
  void* y = nullptr;
  float *muf = nullptr, *rf = nullptr;
  float* z = nullptr;
  void* dz = nullptr;
  float *row_loss = nullptr, *loss_dev = nullptr;
  float* loss_host = nullptr;  // pinned
  // backward scratch
  float* dres = nullptr;
  void* dres_act = nullptr;
  float* dtmp = nullptr;
  void* du = nullptr;
  void* dOh = nullptr;
  void* dqkv = nullptr;
  float *ln_part_g = nullptr, *ln_part_b = nullptr;
  float* col_part = nullptr;
  uint32_t* sort_keys = nullptr;
  // split-K workspace of the weight-gradient GEMMs (few output tiles, K = all tokens)
  float* splitk_ws = nullptr;
  int64_t splitk_elems = 0;

  // tile grids
  std::vector<TGrid> gx, gxmid, gh1, gqkvh, gP, gO, gh2, gu, gg, gstat1, gstat2, glse;
  TGrid gattn_d;
  TGrid gscores, gy, gstatf, gz, gdz, grow_loss, gloss, gtok;
  TGrid gdres, gdres_act, gdtmp, gdu, gdOh, gdqkv, gln_part, gcol_part, gkeys, gsplitk;
  std::vector<TGrid> gparam, ggrad;
  int64_t next_tile = 0;

  // fused backward + AdamW and host offload of AdamW moments
  bool offload = false;                 // some moments live in pinned host memory
  std::vector<Chunk> chunks;
  std::vector<std::vector<int>> chunks_of;  // parameter -> its chunks, in row order
  float *host_m = nullptr, *host_v = nullptr;          // pinned host pools (host addresses)
  float *host_m_dev = nullptr, *host_v_dev = nullptr;  // the same pools as device addresses
  int64_t n_host_mv = 0, n_dev_mv = 0, n_grad = 0;
  float* ring = nullptr;                 // gradient ring slots [n_ring][ring_elems]
  int n_ring = 0;
  int64_t ring_elems = 0;
  std::vector<TGrid> gpchunk;            // per parameter: one tile per chunk
  TGrid gring;
  uint64_t h2d_bytes = 0, d2h_bytes = 0;

  Program fwd, bwd, bwdf, opt;
  Program bwda;  // backward that adds into the gradients (minibatch accumulation)
  Executor ex;
  cudaEvent_t done_event = nullptr;
  int state = 0;  // 0: created, 1: forward done, 2: backward done
  int n_acc = 0;  // minibatch gradients summed in the gradient buffers since the last update
  int64_t step = 0;
  double last_fwd_ms = 0, last_bwd_ms = 0, last_opt_ms = 0;
};

namespace {

nnt_status fail(nnt_model* m, nnt_status s) {
  if (m) m->err = thread_error();
  t_model_err = thread_error();
  return s;
}

// cudaMemcpyAsync behind the copy fault hook; `what` names the copy in the error text.
nnt_status copy_async(void* dst, const void* src, size_t n, cudaMemcpyKind k, cudaStream_t st,
                      const char* what) {
  if (fault_hit(FAULT_COPY)) {
    set_thread_error("%s: async copy submission failed (injected)", what);
    return NNT_ERR_CUDA;
  }
  cudaError_t e = cudaMemcpyAsync(dst, src, n, k, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_thread_error("%s: %s", what, cudaGetErrorString(e));
    return NNT_ERR_CUDA;
  }
  return NNT_OK;
}

template <typename Ptr>
nnt_status dalloc(nnt_model* m, Ptr*& p, size_t bytes) {
  void* q = nullptr;
  if (bytes == 0) bytes = 16;
  if (m->dry) {
    m->device_bytes += bytes;
    p = nullptr;
    return NNT_OK;
  }
  if (fault_hit(FAULT_DEVICE_ALLOC)) {
    set_thread_error("cudaMalloc of %zu bytes failed (injected); %llu bytes already held", bytes,
                     (unsigned long long)m->device_bytes);
    return NNT_ERR_OOM;
  }
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_thread_error("cudaMalloc of %zu bytes failed (%s); %llu bytes already held", bytes,
                     cudaGetErrorString(e), (unsigned long long)m->device_bytes);
    return NNT_ERR_OOM;
  }
  m->dev_allocs.push_back(q);
  m->device_bytes += bytes;
  p = static_cast<Ptr*>(q);
  return NNT_OK;
}

TGrid new_grid(nnt_model* m, int a, int b = 1, int c = 1, int d = 1) {
  TGrid t;
  t.base = m->next_tile;
  t.g[0] = a;
  t.g[1] = b;
  t.g[2] = c;
  t.g[3] = d;
  m->next_tile += (int64_t)a * b * c * d;
  return t;
}

// Add the tiles of box [a0,a1) x [b0,b1) x [c0,c1) x [d0,d1) (-1 = whole axis).
void box(std::vector<TileUse>& u, const TGrid& t, int mode, int a0 = 0, int a1 = -1, int b0 = 0,
         int b1 = -1, int c0 = 0, int c1 = -1, int d0 = 0, int d1 = -1) {
  if (a1 < 0) a1 = t.g[0];
  if (b1 < 0) b1 = t.g[1];
  if (c1 < 0) c1 = t.g[2];
  if (d1 < 0) d1 = t.g[3];
  for (int a = a0; a < a1; ++a)
    for (int b = b0; b < b1; ++b)
      for (int c = c0; c < c1; ++c)
        for (int d = d0; d < d1; ++d)
          u.push_back({t.base + (((int64_t)a * t.g[1] + b) * t.g[2] + c) * t.g[3] + d, mode});
}

int tiles_of(int n, int t) { return (int)ceil_div(n, t); }
int tile_lo(int i, int t) { return i * t; }
int tile_hi(int i, int t, int n) { return std::min(n, (i + 1) * t); }

double causal_rows(int q0, int nq) {  // sum_{q=q0}^{q0+nq-1} (q+1)
  return (double)nq * q0 + (double)nq * (nq + 1) / 2.0;
}

// ------------------------------------------------------------ model build

nnt_status validate(const nnt_gpt2_config* c, const nnt_tiles* t) {
  NNT_CHECK_ARG(c, "NULL config");
  NNT_CHECK_ARG(c->n_layer >= 0 && c->d_model > 0 && c->n_head > 0 && c->d_ff > 0 && c->vocab > 0 &&
                    c->n_ctx > 0 && c->batch > 0,
                "config sizes must be positive");
  NNT_CHECK_ARG(c->dtype == NNT_F32 || c->dtype == NNT_BF16, "dtype must be NNT_F32 or NNT_BF16");
  NNT_CHECK_ARG(c->d_model % c->n_head == 0, "d_model %% n_head != 0");
  NNT_CHECK_ARG(c->d_model % 8 == 0 && c->d_ff % 8 == 0,
                "d_model and d_ff must be multiples of 8");
  const int hd = c->d_model / c->n_head;
  NNT_CHECK_ARG(hd % 8 == 0, "head size must be a multiple of 8");
  NNT_CHECK_ARG(c->dtype == NNT_F32 || hd % 16 == 0, "bf16 needs a head size multiple of 16");
  NNT_CHECK_ARG(c->vocab <= 65536, "vocab must be <= 65536 (uint16 token ids)");
  NNT_CHECK_ARG(c->n_ctx % 4 == 0, "n_ctx must be a multiple of 4");
  NNT_CHECK_ARG((int64_t)c->batch * c->n_ctx <= kMaxTokens, "batch*n_ctx must be <= %d", kMaxTokens);
  NNT_CHECK_ARG(c->d_model <= 32768, "d_model must be <= 32768");
  if (t) {
    NNT_CHECK_ARG(t->batch_tile >= 0 && t->seq_tile >= 0 && t->embd_tile >= 0 && t->inner_tile >= 0 &&
                      t->head_tile >= 0 && t->vocab_tile >= 0,
                  "tile sizes must be >= 0");
    const int tb = t->batch_tile ? t->batch_tile : c->batch;
    const int ts = t->seq_tile ? t->seq_tile : c->n_ctx;
    const int th = t->head_tile ? t->head_tile : c->n_head;
    NNT_CHECK_ARG(c->batch % tb == 0, "batch %% batch_tile != 0");
    NNT_CHECK_ARG(c->n_ctx % ts == 0, "n_ctx %% seq_tile != 0 (sequence length must be divisible by seq-tile)");
    NNT_CHECK_ARG(c->n_head % th == 0, "n_head %% head_tile != 0");
    NNT_CHECK_ARG(ts % 4 == 0 || ts == c->n_ctx, "seq_tile must be a multiple of 4");
    const int te = t->embd_tile ? t->embd_tile : c->d_model;
    const int ti = t->inner_tile ? t->inner_tile : c->d_ff;
    const int tv = t->vocab_tile ? t->vocab_tile : c->vocab;
    NNT_CHECK_ARG(te % 8 == 0 || te >= c->d_model, "embd_tile must be a multiple of 8");
    NNT_CHECK_ARG(ti % 8 == 0 || ti >= c->d_ff, "inner_tile must be a multiple of 8");
    NNT_CHECK_ARG(tv % 8 == 0 || tv >= c->vocab, "vocab_tile must be a multiple of 8");
  }
  return NNT_OK;
}

int axis_tile(const nnt_model* m, int64_t n) {
  if (n == m->d) return m->te;
  if (n == 3 * (int64_t)m->d) return m->te;
  if (n == m->f) return m->ti;
  if (n == m->V) return m->tv;
  if (n == m->S) return m->ts;
  return (int)n;
}

// Parameters whose gradients are streamed through the ring when offloading:
// the four weight matrices of every layer.
bool ring_param(const nnt_model* m, int i) { return i >= 2 && i < 2 + 12 * m->L && m->params[i].kind == 0; }

// AdamW chunks: vectors whole; matrices in runs of whole out-tiles of at most
// 2^27 elements (512 MiB of fp32), so a chunk is a contiguous row block.
void plan_chunks(nnt_model* m) {
  m->chunks.clear();
  m->chunks_of.assign(m->params.size(), {});
  for (int i = 0; i < (int)m->params.size(); ++i) {
    const ParamInfo& p = m->params[i];
    if (p.shape1 == 0) {
      Chunk c;
      c.param = i;
      c.r0 = 0;
      c.r1 = 1;
      c.e0 = 0;
      c.n = p.n;
      c.t0 = 0;
      c.t1 = tiles_of((int)p.shape0, axis_tile(m, p.shape0));
      m->chunks_of[i].push_back((int)m->chunks.size());
      m->chunks.push_back(c);
      continue;
    }
    const int64_t rows = p.shape0, cols = p.shape1;
    const int64_t tr = axis_tile(m, rows);
    const int64_t per = tr * std::max<int64_t>(1, (1ll << 27) / (tr * cols));
    for (int64_t r0 = 0; r0 < rows; r0 += per) {
      Chunk c;
      c.param = i;
      c.r0 = r0;
      c.r1 = std::min(rows, r0 + per);
      c.e0 = r0 * cols;
      c.n = (c.r1 - c.r0) * cols;
      c.t0 = (int)(r0 / tr);
      c.t1 = (int)ceil_div(c.r1, tr);
      m->chunks_of[i].push_back((int)m->chunks.size());
      m->chunks.push_back(c);
    }
  }
}

// Gradients, AdamW moments and (when offloading) the ring and staging slots.
// Everything fits in `budget` device bytes: flat gradient and moment buffers
// with the master layout. Otherwise, with host offload allowed: gradients of the
// layer matrices go through a ring of slots (the fused backward updates each
// chunk as soon as its gradient is final), the other gradients keep a device
// buffer, and the moments of as many chunks as fit stay on the device while the
// rest live in pinned, device-mapped host memory that the AdamW kernel reads
// and writes directly.
nnt_status alloc_param_state(nnt_model* m, uint64_t budget) {
  plan_chunks(m);
  const uint64_t flat_state = (uint64_t)m->n_flat * 12;
  if (m->device_bytes + flat_state <= budget || !m->opts.allow_host_offload) {
    m->offload = false;
    const size_t pf = (size_t)m->n_flat * 4;
    NNT_TRY(dalloc(m, m->grad, pf));
    NNT_TRY(dalloc(m, m->mom1, pf));
    NNT_TRY(dalloc(m, m->mom2, pf));
    if (!m->dry) {
      NNT_CUDA_TRY(cudaMemset(m->grad, 0, pf));
      NNT_CUDA_TRY(cudaMemset(m->mom1, 0, pf));
      NNT_CUDA_TRY(cudaMemset(m->mom2, 0, pf));
    }
    m->n_grad = m->n_dev_mv = m->n_flat;
    for (ParamInfo& p : m->params) p.goff = p.off;
    for (Chunk& c : m->chunks) {
      const int64_t off = m->params[c.param].off + c.e0;
      c.goff = off;
      c.mv_off = off;
    }
    return NNT_OK;
  }
  m->offload = true;
  int64_t max_ring = 0, n_grad = 0;
  for (int i = 0; i < (int)m->params.size(); ++i) {
    ParamInfo& p = m->params[i];
    if (ring_param(m, i)) {
      p.goff = -1;
      continue;
    }
    p.goff = n_grad;  // contiguous per parameter (the LM head and scatter see [V, d])
    n_grad += round_up(p.n, 64);
  }
  for (Chunk& c : m->chunks) {
    c.ring = ring_param(m, c.param);
    if (c.ring) max_ring = std::max(max_ring, c.n);
    else c.goff = m->params[c.param].goff + c.e0;
  }
  m->n_grad = n_grad;
  NNT_TRY(dalloc(m, m->grad, (size_t)std::max<int64_t>(n_grad, 64) * 4));
  if (!m->dry) NNT_CUDA_TRY(cudaMemset(m->grad, 0, (size_t)n_grad * 4));
  m->n_ring = max_ring ? 4 : 0;
  m->ring_elems = round_up(max_ring, 64);
  if (m->n_ring) NNT_TRY(dalloc(m, m->ring, (size_t)m->n_ring * m->ring_elems * 4));
  int r = 0;
  for (Chunk& c : m->chunks)
    if (c.ring) c.slot = r++ % m->n_ring;
  // moments: small chunks first on the device, then large ones while they fit
  std::vector<int> order(m->chunks.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return m->chunks[a].n < m->chunks[b].n; });
  const uint64_t used = m->device_bytes;
  uint64_t room = budget > used ? budget - used : 0;
  int64_t dev_mv = 0, host_mv = 0;
  for (int i : order) {
    Chunk& c = m->chunks[i];
    const uint64_t need = (uint64_t)round_up(c.n, 64) * 8;
    if (need <= room) {
      c.host = false;
      c.mv_off = dev_mv;
      dev_mv += round_up(c.n, 64);
      room -= need;
    } else {
      c.host = true;
      c.mv_off = host_mv;
      host_mv += round_up(c.n, 64);
    }
  }
  m->n_dev_mv = dev_mv;
  m->n_host_mv = host_mv;
  NNT_TRY(dalloc(m, m->mom1, (size_t)std::max<int64_t>(dev_mv, 64) * 4));
  NNT_TRY(dalloc(m, m->mom2, (size_t)std::max<int64_t>(dev_mv, 64) * 4));
  if (m->dry) {
    m->host_bytes += (uint64_t)host_mv * 8;
    return NNT_OK;
  }
  NNT_CUDA_TRY(cudaMemset(m->mom1, 0, (size_t)dev_mv * 4));
  NNT_CUDA_TRY(cudaMemset(m->mom2, 0, (size_t)dev_mv * 4));
  if (host_mv) {
    void* hm = nullptr;
    void* hv = nullptr;
    const unsigned fl = cudaHostAllocMapped | cudaHostAllocPortable;
    if (fault_hit(FAULT_HOST_ALLOC) || cudaHostAlloc(&hm, (size_t)host_mv * 4, fl) != cudaSuccess ||
        fault_hit(FAULT_HOST_ALLOC) || cudaHostAlloc(&hv, (size_t)host_mv * 4, fl) != cudaSuccess) {
      cudaGetLastError();
      if (hm) cudaFreeHost(hm);
      set_thread_error("pinned host allocation of 2 x %lld bytes for AdamW moments failed",
                       (long long)host_mv * 4);
      return NNT_ERR_OOM;
    }
    m->host_m = (float*)hm;
    m->host_v = (float*)hv;
    m->host_bytes += (uint64_t)host_mv * 8;
    memset(m->host_m, 0, (size_t)host_mv * 4);
    memset(m->host_v, 0, (size_t)host_mv * 4);
    void* dm = nullptr;
    void* dv = nullptr;
    NNT_CUDA_TRY(cudaHostGetDevicePointer(&dm, m->host_m, 0));
    NNT_CUDA_TRY(cudaHostGetDevicePointer(&dv, m->host_v, 0));
    m->host_m_dev = (float*)dm;
    m->host_v_dev = (float*)dv;
  }
  return NNT_OK;
}

nnt_status alloc_all(nnt_model* m) {
  const int L = m->L, d = m->d, f = m->f, T = m->T, H = m->H, S = m->S, B = m->B;
  const size_t as = m->act_size;
  // parameters: each tensor starts on a 64-element boundary
  auto add_param = [&](const std::string& name, int64_t s0, int64_t s1, int kind) {
    ParamInfo p;
    p.name = name;
    p.shape0 = s0;
    p.shape1 = s1;
    p.n = s0 * (s1 ? s1 : 1);
    p.off = m->n_flat;
    p.kind = kind;
    m->n_flat += round_up(p.n, 64);
    m->n_scalar += p.n;
    m->params.push_back(p);
  };
  add_param("wte", m->V, d, 0);
  add_param("wpe", S, d, 0);
  for (int l = 0; l < L; ++l) {
    std::string p = "h" + std::to_string(l) + ".";
    add_param(p + "ln1.g", d, 0, 2);
    add_param(p + "ln1.b", d, 0, 3);
    add_param(p + "qkv.w", 3 * d, d, 0);
    add_param(p + "qkv.b", 3 * d, 0, 1);
    add_param(p + "o.w", d, d, 0);
    add_param(p + "o.b", d, 0, 1);
    add_param(p + "ln2.g", d, 0, 2);
    add_param(p + "ln2.b", d, 0, 3);
    add_param(p + "fc.w", f, d, 0);
    add_param(p + "fc.b", f, 0, 1);
    add_param(p + "proj.w", d, f, 0);
    add_param(p + "proj.b", d, 0, 1);
  }
  add_param("ln_f.g", d, 0, 2);
  add_param("ln_f.b", d, 0, 3);
  size_t free_b = m->free_device, total_b = 0;
  if (!m->dry) NNT_CUDA_TRY(cudaMemGetInfo(&free_b, &total_b));
  const size_t pf = (size_t)m->n_flat * 4;
  NNT_TRY(dalloc(m, m->master, pf));
  NNT_TRY(dalloc(m, m->wbf, (size_t)m->n_flat * 2));
  NNT_TRY(dalloc(m, m->hyper_dev, sizeof(AdamHyperDev)));
  if (!m->dry) {
    NNT_CUDA_TRY(cudaMemset(m->master, 0, pf));
    NNT_CUDA_TRY(cudaMemset(m->wbf, 0, (size_t)m->n_flat * 2));
  }

  NNT_TRY(dalloc(m, m->tokens_dev, (size_t)B * (S + 1) * 2));
  m->x.resize(L + 1);
  m->xmid.resize(L);
  m->mu1.resize(L);
  m->r1.resize(L);
  m->mu2.resize(L);
  m->r2.resize(L);
  m->u.resize(L);
  m->h1.resize(L);
  m->qkvh.resize(L);
  m->P.resize(L);
  m->lse.resize(L);
  m->O.resize(L);
  m->h2.resize(L);
  m->g.resize(L);
  const size_t Td = (size_t)T * d;
  for (int l = 0; l <= L; ++l) NNT_TRY(dalloc(m, m->x[l], Td * 4));
  for (int l = 0; l < L; ++l) {
    NNT_TRY(dalloc(m, m->xmid[l], Td * 4));
    NNT_TRY(dalloc(m, m->mu1[l], (size_t)T * 4));
    NNT_TRY(dalloc(m, m->r1[l], (size_t)T * 4));
    NNT_TRY(dalloc(m, m->mu2[l], (size_t)T * 4));
    NNT_TRY(dalloc(m, m->r2[l], (size_t)T * 4));
    NNT_TRY(dalloc(m, m->h1[l], Td * as));
    NNT_TRY(dalloc(m, m->qkvh[l], 3 * Td * as));
    if (m->flash)
      NNT_TRY(dalloc(m, m->lse[l], (size_t)B * H * S * 4));
    else
      NNT_TRY(dalloc(m, m->P[l], (size_t)B * H * S * S * as));
    NNT_TRY(dalloc(m, m->O[l], Td * as));
    NNT_TRY(dalloc(m, m->h2[l], Td * as));
    NNT_TRY(dalloc(m, m->u[l], (size_t)T * f * as));
    NNT_TRY(dalloc(m, m->g[l], (size_t)T * f * as));
  }
  if (m->flash) {
    NNT_TRY(dalloc(m, m->attn_d, (size_t)B * H * S * 4));
    if (S % 8 == 0) NNT_TRY(dalloc(m, m->attn_ds, (size_t)B * H * S * S * 2));
  }
  else
    NNT_TRY(dalloc(m, m->scores, (size_t)B * H * S * S * 4));
  NNT_TRY(dalloc(m, m->y, Td * as));
  NNT_TRY(dalloc(m, m->muf, (size_t)T * 4));
  NNT_TRY(dalloc(m, m->rf, (size_t)T * 4));
  NNT_TRY(dalloc(m, m->z, (size_t)T * m->ldz * 4));
  NNT_TRY(dalloc(m, m->dz, (size_t)T * m->lddz * as));
  NNT_TRY(dalloc(m, m->row_loss, (size_t)T * 4));
  NNT_TRY(dalloc(m, m->loss_dev, 16));
  NNT_TRY(dalloc(m, m->dres, Td * 4));
  NNT_TRY(dalloc(m, m->dres_act, Td * as));
  NNT_TRY(dalloc(m, m->dtmp, Td * 4));
  NNT_TRY(dalloc(m, m->du, (size_t)T * f * as));
  NNT_TRY(dalloc(m, m->dOh, Td * as));
  NNT_TRY(dalloc(m, m->dqkv, 3 * Td * as));
  NNT_TRY(dalloc(m, m->ln_part_g,
                 (size_t)std::max<int64_t>(ln_colsum_chunks(T), (int64_t)m->n_tok * ln_bwd_fused_ctas(m->TT, m->d)) *
                     3 * d * 4));
  const int64_t maxcols = std::max<int64_t>(3 * d, f);
  NNT_TRY(dalloc(m, m->col_part, (size_t)colsum_nparts(T) * maxcols * 4));
  if (m->act == NNT_BF16 && m->backend == 0) {  // 32 MB: the split weight-gradient GEMMs of small models
    m->splitk_elems = 8ll << 20;
    NNT_TRY(dalloc(m, m->splitk_ws, (size_t)m->splitk_elems * 4));
  }
  NNT_TRY(dalloc(m, m->sort_keys, (size_t)T * 4));
  const uint64_t budget = m->opts.hbm_budget_bytes
                              ? m->opts.hbm_budget_bytes
                              : (free_b > (2ull << 30) ? free_b - (2ull << 30) : 0);
  if (m->dry) {
    m->host_bytes += 64;
    return alloc_param_state(m, budget);
  }
  // padding columns of the logits must stay finite: zero them once
  NNT_CUDA_TRY(cudaMemset(m->z, 0, (size_t)T * m->ldz * 4));
  NNT_CUDA_TRY(cudaMemset(m->dz, 0, (size_t)T * m->lddz * as));
  void* lh = nullptr;
  if (fault_hit(FAULT_HOST_ALLOC)) {
    set_thread_error("pinned host allocation of the loss word failed (injected)");
    return NNT_ERR_OOM;
  }
  NNT_CUDA_TRY(cudaMallocHost(&lh, 64));
  m->loss_host = (float*)lh;
  m->host_bytes += 64;
  // gradients and AdamW moments last, once everything else is placed
  return alloc_param_state(m, budget);
}

nnt_status init_params(nnt_model* m, cudaStream_t st) {
  const double std = m->opts.init_std > 0 ? (double)m->opts.init_std : 0.02;
  for (size_t i = 0; i < m->params.size(); ++i) {
    const ParamInfo& p = m->params[i];
    float* w = m->master + p.off;
    if (p.kind == 2) NNT_TRY(launch_fill(w, p.n, 1.f, st));
    else if (p.kind == 3 || (p.kind == 1 && m->opts.init_zero_bias)) NNT_TRY(launch_fill(w, p.n, 0.f, st));
    else NNT_TRY(launch_init_normal(w, p.n, m->opts.init_seed, (uint64_t)i, std, st));
  }
  NNT_TRY(launch_cast_bf16(m->master, m->wbf, m->n_flat, st));
  return NNT_OK;
}

const ParamInfo& P_(nnt_model* m, int l, int which) {  // which: index within a layer block
  return m->params[2 + 12 * l + which];
}
enum { LN1G = 0, LN1B, QKVW, QKVB, OW, OB, LN2G, LN2B, FCW, FCB, PROJW, PROJB };

// pointer helpers
float* pm(nnt_model* m, const ParamInfo& p) { return m->master + p.off; }
float* pg(nnt_model* m, const ParamInfo& p) { return m->grad + p.goff; }
const void* pw(nnt_model* m, const ParamInfo& p) {  // GEMM operand copy of a weight
  if (m->act == NNT_BF16) return m->wbf + p.off;
  return m->master + p.off;
}

struct Builder {
  nnt_model* m;
  int row0(int rt) const { return rt * m->TT; }
  int bt_of(int rt) const { return rt / m->n_st; }
  int st_of(int rt) const { return rt % m->n_st; }

  // GEMM task helper
  void gemm_task(Program& P, int type, const GemmArgs& g0, std::vector<TileUse> uses, double flops) {
    Task t;
    t.type = type;
    GemmArgs g = g0;
    const int be = m->backend;
    // GEMMs with too few output tiles for the SMs (the weight gradients of small
    // layers) split K through the shared workspace, one such task at a time
    if (m->splitk_ws && be == 0 && gemm_tc_supported(g) && gemm_split_k(g, m->splitk_elems) > 1) {
      g.ws = m->splitk_ws;
      g.ws_elems = m->splitk_elems;
      box(uses, m->gsplitk, ACC_RW);
      t.kernels = 2;
    }
    t.uses = std::move(uses);
    t.flops = flops;
    t.fn = [g, be](cudaStream_t s) { return gemm(g, be, s); };
    P.add(std::move(t));
  }
  GemmArgs base() const {
    GemmArgs g;
    g.op_dtype = m->act;
    g.tm = m->tm;
    return g;
  }
  // column tiles of the qkv axis: part-major, te-sized inside each part
  void qkv_cols(int ct, int& c0, int& c1) const {
    const int part = ct / m->nce, c = ct % m->nce;
    c0 = part * m->d + tile_lo(c, m->te);
    c1 = part * m->d + tile_hi(c, m->te, m->d);
  }
  // Consecutive column tiles [t0, t1) merged into one GEMM launch until the
  // launch is at least gemm_min_cols wide; tiles stay the dependency unit.
  template <class Lo, class Hi>
  std::vector<std::pair<int, int>> groups(int n, Lo lo, Hi hi) const {
    std::vector<std::pair<int, int>> out;
    int t0 = 0;
    while (t0 < n) {
      int t1 = t0 + 1;
      while (t1 < n && hi(t1 - 1) - lo(t0) < m->gemm_min_cols) ++t1;
      out.push_back({t0, t1});
      t0 = t1;
    }
    return out;
  }
  std::vector<std::pair<int, int>> col_groups(int n, int tile, int N) const {
    return groups(n, [=](int t) { return tile_lo(t, tile); }, [=](int t) { return tile_hi(t, tile, N); });
  }
  // head-tile range overlapped by columns [c0, c1) of one part (c relative to part)
  void head_tiles(int c0, int c1, int& h0, int& h1) const {
    const int hl = c0 / m->hd, hh = (c1 + m->hd - 1) / m->hd;
    h0 = hl / m->th;
    h1 = (hh - 1) / m->th + 1;
  }
};

// -------------------------------------------------------------- forward
// Fused-attention arguments for the (sequence, head) items of one (batch tile,
// head tile) of the step's buffers.
FlashArgs flash_args(const nnt_model* m, int bt, int ht) {
  FlashArgs a;
  a.S = m->S;
  a.hd = m->hd;
  a.nz = m->tb * m->th;
  a.zm = ZMap{bt * m->tb, ht * m->th, m->th, m->H};
  a.z_total = (int64_t)m->B * m->H;
  a.tm = m->tm;
  return a;
}

void build_forward(nnt_model* m) {
  Builder b{m};
  Program& P = m->fwd;
  const int d = m->d, f = m->f, T = m->T, S = m->S, H = m->H, hd = m->hd, V = m->V;
  const size_t as = m->act_size;
  const float eps = m->cfg.ln_eps > 0 ? m->cfg.ln_eps : 1e-5f;
  const int act = m->act;

  // embedding per token tile
  for (int rt = 0; rt < m->n_tok; ++rt) {
    Task t;
    t.type = TT_EMBED;
    box(t.uses, m->gtok, ACC_R);
    box(t.uses, m->gx[0], ACC_W, rt, rt + 1);
    const int b0 = b.bt_of(rt) * m->tb, s0 = b.st_of(rt) * m->ts;
    t.bytes = (double)m->TT * d * 12 + m->TT * 2.0;
    t.fn = [m, b0, s0](cudaStream_t s) {
      return launch_embedding_fwd(m->tokens_dev, m->S + 1, m->master + m->params[0].off,
                                  m->master + m->params[1].off, m->x[0], m->d, m->V, m->tm, b0,
                                  m->tb, s0, m->ts, s);
    };
    P.add(std::move(t));
  }

  auto ln_fwd_task = [&](int type, const float* const* xin, const TGrid& gxin, const ParamInfo* pgm,
                         const ParamInfo* pbt, void* const* yout, const TGrid& gyout, float* const* mu,
                         float* const* rs, const TGrid& gst, int rt) {
    Task t;
    t.type = type;
    box(t.uses, gxin, ACC_R, rt, rt + 1);
    box(t.uses, gyout, ACC_W, rt, rt + 1);
    box(t.uses, gst, ACC_W, rt, rt + 1);
    t.bytes = (double)m->TT * d * (4 + as) + 8.0 * m->TT;
    const int64_t r0 = (int64_t)rt * m->TT;
    t.fn = [=](cudaStream_t s) {
      return launch_layernorm_fwd(*xin + r0 * d, pm(m, *pgm), pm(m, *pbt),
                                  (char*)*yout + r0 * d * as, *mu + r0, *rs + r0, m->TT, d, eps,
                                  act, s);
    };
    P.add(std::move(t));
  };

  for (int l = 0; l < m->L; ++l) {
    // LN1
    for (int rt = 0; rt < m->n_tok; ++rt)
      ln_fwd_task(TT_LN_FWD, &m->x[l], m->gx[l], &P_(m, l, LN1G), &P_(m, l, LN1B), &m->h1[l],
                  m->gh1[l], &m->mu1[l], &m->r1[l], m->gstat1[l], rt);
    // QKV projection, epilogue writes head-major q/k/v
    auto qlo = [&](int ct) { int a, c; b.qkv_cols(ct, a, c); return a; };
    auto qhi = [&](int ct) { int a, c; b.qkv_cols(ct, a, c); return c; };
    for (int rt = 0; rt < m->n_tok; ++rt)
      for (auto [t0, t1] : b.groups(3 * m->nce, qlo, qhi)) {
        const int c0 = qlo(t0), c1 = qhi(t1 - 1);
        GemmArgs g = b.base();
        g.M = T; g.N = 3 * d; g.K = d;
        g.m0 = b.row0(rt); g.mt = m->TT; g.n0 = c0; g.nt = c1 - c0;
        g.A = m->h1[l]; g.lda = d; g.a_trans = 0;
        g.B = pw(m, P_(m, l, QKVW)); g.ldb = d; g.b_trans = 0;
        g.C = m->qkvh[l]; g.c_dtype = act; g.out_mode = OUT_HEADSPLIT;
        g.hs_B = m->B; g.hs_H = H; g.hs_S = S; g.hs_hd = hd; g.hs_B = m->B; g.hs_S = S; g.hs_H = H; g.hs_d = d;
        g.bias = pm(m, P_(m, l, QKVB));
        std::vector<TileUse> u;
        box(u, m->gh1[l], ACC_R, rt, rt + 1);
        for (int ct = t0; ct < t1; ++ct) {
          const int part = ct / m->nce;
          int h0, h1;
          b.head_tiles(qlo(ct) - part * d, qhi(ct) - part * d, h0, h1);
          box(u, m->gqkvh[l], ACC_W, part, part + 1, b.bt_of(rt), b.bt_of(rt) + 1, h0, h1,
              b.st_of(rt), b.st_of(rt) + 1);
        }
        b.gemm_task(P, TT_GEMM_QKV, g, std::move(u), 2.0 * m->TT * (c1 - c0) * d);
      }
    // attention per (batch tile, head tile, query tile)
    const size_t zq = (size_t)S * hd;  // elements of one head's q (or k, v)
    const char* qkv_base = (const char*)m->qkvh[l];
    const int64_t BH = (int64_t)m->B * H;
    if (m->flash) {
      // one fused task per (batch tile, head tile): O and the row log-sum-exp
      const bf16* qp = reinterpret_cast<const bf16*>(qkv_base);
      for (int bt = 0; bt < m->n_bt; ++bt)
        for (int ht = 0; ht < m->n_ht; ++ht) {
          FlashArgs fa = flash_args(m, bt, ht);
          fa.o = static_cast<bf16*>(m->O[l]);
          fa.ldo = d;
          fa.lse = m->lse[l];
          Task t;
          t.type = TT_FLASH_FWD;
          box(t.uses, m->gqkvh[l], ACC_R, 0, 3, bt, bt + 1, ht, ht + 1);
          box(t.uses, m->gO[l], ACC_W, bt * m->n_st, (bt + 1) * m->n_st);
          box(t.uses, m->glse[l], ACC_W, bt, bt + 1, ht, ht + 1);
          t.flops = 2 * 2.0 * hd * causal_rows(0, S) * fa.nz;  // Q K^T and P V, causal half
          t.fn = [=](cudaStream_t s) { return launch_flash_fwd(qp, qp + BH * zq, qp + 2 * BH * zq, fa, s); };
          P.add(std::move(t));
        }
    }
    for (int bt = 0; bt < (m->flash ? 0 : m->n_bt); ++bt)
      for (int ht = 0; ht < m->n_ht; ++ht)
        for (int st = 0; st < m->n_st; ++st) {
          const int nz = m->tb * m->th;
          ZMap zm{bt * m->tb, ht * m->th, m->th, H};
          const int q0 = st * m->ts, nq = m->ts;
          // scores = Q K^T / sqrt(hd), causal tiles only
          {
            GemmArgs g = b.base();
            g.M = S; g.N = S; g.K = hd; g.nbatch = nz; g.zm = zm;
            g.m0 = q0; g.mt = nq; g.n0 = 0; g.nt = std::min<int>(S, (int)round_up(q0 + nq, kCausalBlock));
            g.A = qkv_base; g.lda = hd; g.a_zs = zq; g.a_trans = 0;
            g.B = qkv_base + BH * zq * as; g.ldb = hd; g.b_zs = zq; g.b_trans = 0;
            g.C = m->scores; g.ldc = S; g.c_zs = (int64_t)S * S; g.c_dtype = NNT_F32;
            g.alpha = 1.0f / sqrtf((float)hd);
            g.causal = CAUSAL_TILES;
            std::vector<TileUse> u;
            box(u, m->gqkvh[l], ACC_R, 0, 2, bt, bt + 1, ht, ht + 1);
            box(u, m->gscores, ACC_W, bt, bt + 1, ht, ht + 1, st, st + 1);
            b.gemm_task(P, TT_GEMM_QK, g, std::move(u), 2.0 * hd * causal_rows(q0, nq) * nz);
          }
          {
            Task t;
            t.type = TT_SOFTMAX_FWD;
            box(t.uses, m->gscores, ACC_R, bt, bt + 1, ht, ht + 1, st, st + 1);
            box(t.uses, m->gP[l], ACC_W, bt, bt + 1, ht, ht + 1, st, st + 1);
            t.bytes = causal_rows(q0, nq) * nz * (4 + as);
            void* Pl = m->P[l];
            t.fn = [=](cudaStream_t s) {
              return launch_softmax_fwd(m->scores, Pl, S, zm, nz, q0, nq, act, s);
            };
            P.add(std::move(t));
          }
          // O = P V, merged back to token-major [T, d]
          {
            GemmArgs g = b.base();
            g.M = S; g.N = hd; g.K = S; g.nbatch = nz; g.zm = zm;
            g.m0 = q0; g.mt = nq; g.n0 = 0; g.nt = hd;
            g.A = m->P[l]; g.lda = S; g.a_zs = (int64_t)S * S; g.a_trans = 0;
            g.B = qkv_base + 2 * BH * zq * as; g.ldb = hd; g.b_zs = zq; g.b_trans = 1;
            g.C = m->O[l]; g.ldc = d; g.c_dtype = act; g.out_mode = OUT_HEADMERGE;
            g.hs_hd = hd; g.hs_B = m->B; g.hs_S = S; g.hs_H = H;
            g.causal = CAUSAL_K_UPPER;
            std::vector<TileUse> u;
            box(u, m->gP[l], ACC_R, bt, bt + 1, ht, ht + 1, st, st + 1);
            box(u, m->gqkvh[l], ACC_R, 2, 3, bt, bt + 1, ht, ht + 1);
            box(u, m->gO[l], ACC_W, bt * m->n_st + st, bt * m->n_st + st + 1);
            b.gemm_task(P, TT_GEMM_PV, g, std::move(u), 2.0 * hd * causal_rows(q0, nq) * nz);
          }
        }
    // attention output projection + residual: xmid = x + O Wo^T + bo
    for (int rt = 0; rt < m->n_tok; ++rt)
      for (auto [t0, t1] : b.col_groups(m->nce, m->te, d)) {
        const int c0 = tile_lo(t0, m->te), c1 = tile_hi(t1 - 1, m->te, d);
        GemmArgs g = b.base();
        g.M = T; g.N = d; g.K = d;
        g.m0 = b.row0(rt); g.mt = m->TT; g.n0 = c0; g.nt = c1 - c0;
        g.A = m->O[l]; g.lda = d;
        g.B = pw(m, P_(m, l, OW)); g.ldb = d;
        g.C = m->xmid[l]; g.ldc = d; g.c_dtype = NNT_F32;
        g.bias = pm(m, P_(m, l, OB));
        g.resid = m->x[l]; g.ld_resid = d;
        std::vector<TileUse> u;
        box(u, m->gO[l], ACC_R, rt, rt + 1);
        box(u, m->gx[l], ACC_R, rt, rt + 1, t0, t1);
        box(u, m->gxmid[l], ACC_W, rt, rt + 1, t0, t1);
        b.gemm_task(P, TT_GEMM_ATTN_O, g, std::move(u), 2.0 * m->TT * (c1 - c0) * d);
      }
    // LN2
    for (int rt = 0; rt < m->n_tok; ++rt)
      ln_fwd_task(TT_LN_FWD, &m->xmid[l], m->gxmid[l], &P_(m, l, LN2G), &P_(m, l, LN2B), &m->h2[l],
                  m->gh2[l], &m->mu2[l], &m->r2[l], m->gstat2[l], rt);
    // FC + GELU: u = h2 W1^T + b1 (kept, fp32), g = gelu(u)
    for (int rt = 0; rt < m->n_tok; ++rt)
      for (auto [t0, t1] : b.col_groups(m->ncf, m->ti, f)) {
        const int c0 = tile_lo(t0, m->ti), c1 = tile_hi(t1 - 1, m->ti, f);
        GemmArgs g = b.base();
        g.M = T; g.N = f; g.K = d;
        g.m0 = b.row0(rt); g.mt = m->TT; g.n0 = c0; g.nt = c1 - c0;
        g.A = m->h2[l]; g.lda = d;
        g.B = pw(m, P_(m, l, FCW)); g.ldb = d;
        g.C = m->g[l]; g.ldc = f; g.c_dtype = act;
        g.bias = pm(m, P_(m, l, FCB));
        g.epi = EPI_GELU; g.aux = m->u[l]; g.ld_aux = f; g.aux_dtype = act;
        std::vector<TileUse> u;
        box(u, m->gh2[l], ACC_R, rt, rt + 1);
        box(u, m->gu[l], ACC_W, rt, rt + 1, t0, t1);
        box(u, m->gg[l], ACC_W, rt, rt + 1, t0, t1);
        b.gemm_task(P, TT_GEMM_FC, g, std::move(u), 2.0 * m->TT * (c1 - c0) * d);
      }
    // MLP projection + residual: x[l+1] = xmid + g W2^T + b2
    for (int rt = 0; rt < m->n_tok; ++rt)
      for (auto [t0, t1] : b.col_groups(m->nce, m->te, d)) {
        const int c0 = tile_lo(t0, m->te), c1 = tile_hi(t1 - 1, m->te, d);
        GemmArgs g = b.base();
        g.M = T; g.N = d; g.K = f;
        g.m0 = b.row0(rt); g.mt = m->TT; g.n0 = c0; g.nt = c1 - c0;
        g.A = m->g[l]; g.lda = f;
        g.B = pw(m, P_(m, l, PROJW)); g.ldb = f;
        g.C = m->x[l + 1]; g.ldc = d; g.c_dtype = NNT_F32;
        g.bias = pm(m, P_(m, l, PROJB));
        g.resid = m->xmid[l]; g.ld_resid = d;
        std::vector<TileUse> u;
        box(u, m->gg[l], ACC_R, rt, rt + 1);
        box(u, m->gxmid[l], ACC_R, rt, rt + 1, t0, t1);
        box(u, m->gx[l + 1], ACC_W, rt, rt + 1, t0, t1);
        b.gemm_task(P, TT_GEMM_MLP_PROJ, g, std::move(u), 2.0 * m->TT * (c1 - c0) * f);
      }
  }
  // final LN
  const ParamInfo& lnfg = m->params[2 + 12 * m->L];
  const ParamInfo& lnfb = m->params[3 + 12 * m->L];
  for (int rt = 0; rt < m->n_tok; ++rt)
    ln_fwd_task(TT_LN_FWD, &m->x[m->L], m->gx[m->L], &lnfg, &lnfb, &m->y, m->gy, &m->muf, &m->rf,
                m->gstatf, rt);
  // tied LM head: z = y wte^T (fp32 logits)
  for (int rt = 0; rt < m->n_tok; ++rt)
    for (auto [t0, t1] : b.col_groups(m->ncv, m->tv, V)) {
      const int c0 = tile_lo(t0, m->tv), c1 = tile_hi(t1 - 1, m->tv, V);
      GemmArgs g = b.base();
      g.M = T; g.N = V; g.K = d;
      g.m0 = b.row0(rt); g.mt = m->TT; g.n0 = c0; g.nt = c1 - c0;
      g.A = m->y; g.lda = d;
      g.B = pw(m, m->params[0]); g.ldb = d;
      g.C = m->z; g.ldc = m->ldz; g.c_dtype = NNT_F32;
      std::vector<TileUse> u;
      box(u, m->gy, ACC_R, rt, rt + 1);
      box(u, m->gz, ACC_W, rt, rt + 1, t0, t1);
      b.gemm_task(P, TT_GEMM_LM_HEAD, g, std::move(u), 2.0 * m->TT * (c1 - c0) * d);
    }
  // cross-entropy + dlogits per token tile (over every vocab tile)
  const float inv_T = 1.0f / (float)T;
  for (int rt = 0; rt < m->n_tok; ++rt) {
    Task t;
    t.type = TT_XENT;
    box(t.uses, m->gz, ACC_R, rt, rt + 1);
    box(t.uses, m->gtok, ACC_R);
    box(t.uses, m->gdz, ACC_W, rt, rt + 1);
    box(t.uses, m->grow_loss, ACC_W, rt, rt + 1);
    t.bytes = (double)m->TT * V * (4 + as) + 2.0 * m->TT;
    const int64_t r0 = (int64_t)rt * m->TT;
    t.fn = [=](cudaStream_t s) {
      return launch_cross_entropy(m->z, m->ldz, r0, m->TT, V, m->tokens_dev, m->tm, nullptr, 0,
                                  m->dz, m->lddz, m->row_loss, inv_T, act, s);
    };
    P.add(std::move(t));
  }
  {
    Task t;
    t.type = TT_LOSS;
    box(t.uses, m->grow_loss, ACC_R);
    box(t.uses, m->gloss, ACC_W);
    t.bytes = 4.0 * T;
    t.fn = [m](cudaStream_t s) { return launch_mean_loss(m->row_loss, m->T, m->loss_dev, s); };
    P.add(std::move(t));
  }
}

// -------------------------------------------------------------- backward
// Backward program. fused: each parameter chunk gets its AdamW task as soon as
// its gradient is final and every task that reads the old weights has been
// issued (weight reads are declared, so the executor orders the update after
// them); moments in pinned host memory are updated in place over NVLink-C2C.
// acc (not with fused): every gradient write adds to the stored gradient
// instead of replacing it.
void build_backward(nnt_model* m, Program& P, bool fused, bool acc = false) {
  Builder b{m};
  // rows of at most 1024 features: LayerNorm backward with its column sums in one pass
  const bool fused_ln = m->d <= 1024;
  const int ln_g = ln_bwd_fused_ctas(m->TT, m->d);  // partial rows per token tile
  const int GW = acc ? ACC_RW : ACC_W;  // access of the tasks that write parameter gradients
  const int d = m->d, f = m->f, T = m->T, S = m->S, H = m->H, hd = m->hd, V = m->V;
  const size_t as = m->act_size;
  const int act = m->act;

  auto grad_ptr = [m](const Chunk& c) -> float* {
    if (c.ring) return m->ring + (int64_t)c.slot * m->ring_elems;
    return m->grad + c.goff;
  };
  auto adam_chunk = [&](int ci) {
    if (!fused) return;
    const Chunk c = m->chunks[ci];
    const ParamInfo& p = m->params[c.param];
    const int k = ci - m->chunks_of[c.param][0];
    float* gptr = grad_ptr(c);
    // host-resident moments are read and written in place over NVLink-C2C
    // (pinned, device-mapped memory); device-resident ones from the pool
    float* mptr = c.host ? m->host_m_dev + c.mv_off : m->mom1 + c.mv_off;
    float* vptr = c.host ? m->host_v_dev + c.mv_off : m->mom2 + c.mv_off;
    const int64_t n = c.n;
    Task t;
    t.type = TT_ADAMW;
    t.bytes = 30.0 * n;
    box(t.uses, m->gpchunk[c.param], ACC_RW, k, k + 1);
    box(t.uses, m->ggrad[c.param], ACC_R, c.t0, c.t1);
    if (c.ring) box(t.uses, m->gring, ACC_R, c.slot, c.slot + 1);
    float* w = m->master + p.off + c.e0;
    bf16* wb = m->wbf + p.off + c.e0;
    const float* hyper = reinterpret_cast<const float*>(m->hyper_dev);
    const bool host = c.host;
    t.fn = [=](cudaStream_t s) {
      return launch_adamw_dev(w, gptr, mptr, vptr, wb, n, hyper, s, host ? 152 : 0);
    };
    if (host) t.type = TT_ADAMW_HOST;
    // updates run on the last stream, next to the GEMM chain on the others
    t.stream_hint = m->opts.n_streams - 1;
    P.add(std::move(t));
  };
  auto adam_param = [&](int pi) {
    for (int ci : m->chunks_of[pi]) adam_chunk(ci);
  };
  auto param_index = [m](const ParamInfo& p) { return (int)(&p - m->params.data()); };

  // dX tasks: out[rows rt, cols ct] = dY[rt] * W  (W [out, in], K = out); the
  // caller lists the tiles read and written.
  auto dx_gemm = [&](int type, const void* dY, int64_t ldy, int K, const ParamInfo& W, int64_t ldw,
                     void* out, int out_dtype, int N, int tileN, int rt, int t0, int t1,
                     GemmArgs proto, std::vector<TileUse> uses) {
    const int c0 = tile_lo(t0, tileN), c1 = tile_hi(t1 - 1, tileN, N);
    GemmArgs g = proto;
    g.M = T; g.N = N; g.K = K;
    g.m0 = b.row0(rt); g.mt = m->TT; g.n0 = c0; g.nt = c1 - c0;
    g.A = dY; g.lda = ldy; g.a_trans = 0;
    g.B = pw(m, W); g.ldb = ldw; g.b_trans = 1;
    g.C = out; if (!g.ldc) g.ldc = N; g.c_dtype = out_dtype;
    box(uses, m->gpchunk[param_index(W)], ACC_R);  // reads the weight (before its update)
    b.gemm_task(P, type, g, std::move(uses), 2.0 * m->TT * (c1 - c0) * K);
  };
  // dW tasks: grad[out tile, in tile] = dY^T X over all tokens
  auto dw_gemm = [&](int type, const void* dY, const TGrid& gdY, int64_t ldy, int Nout, int tOut,
                     const void* X, const TGrid& gX, int64_t ldx, int Nin, int tIn, const ParamInfo& W,
                     int gidx) {
    if (fused) {  // one GEMM per AdamW chunk (whole rows), then its update
      for (int ci : m->chunks_of[gidx]) {
        const Chunk c = m->chunks[ci];
        GemmArgs g = b.base();
        g.M = Nout; g.N = Nin; g.K = T;
        g.m0 = (int)c.r0; g.mt = (int)(c.r1 - c.r0); g.n0 = 0; g.nt = Nin;
        g.A = dY; g.lda = ldy; g.a_trans = 1;
        g.B = X; g.ldb = ldx; g.b_trans = 1;
        g.C = grad_ptr(c); g.c_row0 = c.r0; g.ldc = Nin; g.c_dtype = NNT_F32;
        std::vector<TileUse> u;
        box(u, gdY, ACC_R);
        box(u, gX, ACC_R);
        box(u, m->ggrad[gidx], ACC_W, c.t0, c.t1);
        if (c.ring) box(u, m->gring, ACC_W, c.slot, c.slot + 1);
        b.gemm_task(P, TT_GEMM_DW, g, std::move(u), 2.0 * (c.r1 - c.r0) * Nin * T);
        adam_chunk(ci);
      }
      return;
    }
    for (auto [ot0, ot1] : b.col_groups(tiles_of(Nout, tOut), tOut, Nout))
      for (auto [it0, it1] : b.col_groups(tiles_of(Nin, tIn), tIn, Nin)) {
        const int o0 = tile_lo(ot0, tOut), o1 = tile_hi(ot1 - 1, tOut, Nout);
        const int i0 = tile_lo(it0, tIn), i1 = tile_hi(it1 - 1, tIn, Nin);
        GemmArgs g = b.base();
        g.M = Nout; g.N = Nin; g.K = T;
        g.m0 = o0; g.mt = o1 - o0; g.n0 = i0; g.nt = i1 - i0;
        g.A = dY; g.lda = ldy; g.a_trans = 1;
        g.B = X; g.ldb = ldx; g.b_trans = 1;
        g.C = pg(m, W); g.ldc = Nin; g.c_dtype = NNT_F32;
        g.beta = acc ? 1 : 0;
        std::vector<TileUse> u;
        box(u, gdY, ACC_R);
        box(u, gX, ACC_R);
        box(u, m->ggrad[gidx], GW, ot0, ot1, it0, it1);
        b.gemm_task(P, TT_GEMM_DW, g, std::move(u), 2.0 * (o1 - o0) * (i1 - i0) * T);
      }
  };
  auto colsum_task = [&](const void* a, int a_dtype, const TGrid& ga, int N, const ParamInfo& bp, int gidx) {
    Task t;
    t.type = TT_COLSUM;
    t.kernels = 2;
    box(t.uses, ga, ACC_R);
    box(t.uses, m->gcol_part, ACC_RW);
    box(t.uses, m->ggrad[gidx], GW);
    t.bytes = (double)T * N * (a_dtype == NNT_BF16 ? 2 : 4);
    float* out = pg(m, bp);
    const int accum = acc ? 1 : 0;
    t.fn = [=](cudaStream_t s) {
      return launch_colsum(a, a_dtype, T, N, N, m->col_part, out, accum, s);
    };
    P.add(std::move(t));
    adam_param(gidx);
  };
  // LN backward per token tile, then one column reduction over all tokens for
  // the gain/shift gradients and (bias_idx >= 0) the gradient of the bias whose
  // output gradient is the new residual gradient.
  auto ln_bwd = [&](const float* dy, const TGrid& gdy, const float* xin, const TGrid& gxin, const float* mu,
                    const float* rs, const TGrid& gst, const ParamInfo& gm, const ParamInfo& bt_,
                    int gidx_g, int gidx_b, bool has_resid, int bias_idx) {
    for (int rt = 0; rt < m->n_tok; ++rt) {
      Task t;
      t.type = TT_LN_BWD;
      box(t.uses, gdy, ACC_R, rt, rt + 1);
      box(t.uses, gxin, ACC_R, rt, rt + 1);
      box(t.uses, gst, ACC_R, rt, rt + 1);
      box(t.uses, m->gdres, has_resid ? ACC_RW : ACC_W, rt, rt + 1);
      box(t.uses, m->gdres_act, ACC_W, rt, rt + 1);
      box(t.uses, m->gpchunk[gidx_g], ACC_R);  // reads the gain (before its update)
      t.bytes = (double)m->TT * d * (4 * (has_resid ? 4 : 3) + as);
      const int64_t r0 = (int64_t)rt * m->TT;
      const float* gam = pm(m, gm);
      if (fused_ln) {
        // the column sums of this token tile go to its slice of the partials
        box(t.uses, m->gln_part, ACC_W, rt, rt + 1);
        float* part = m->ln_part_g + (int64_t)rt * ln_g * 3 * d;
        const int want_out = bias_idx >= 0;
        t.fn = [=](cudaStream_t s) {
          return launch_ln_bwd_fused(dy + r0 * d, xin + r0 * d, mu + r0, rs + r0, gam,
                                     has_resid ? m->dres + r0 * d : nullptr, m->dres + r0 * d,
                                     (char*)m->dres_act + r0 * d * as, m->TT, d, act, part, want_out, s);
        };
      } else {
        t.fn = [=](cudaStream_t s) {
          return launch_layernorm_bwd(dy + r0 * d, xin + r0 * d, mu + r0, rs + r0, gam,
                                      has_resid ? m->dres + r0 * d : nullptr, m->dres + r0 * d,
                                      (char*)m->dres_act + r0 * d * as, m->TT, d, act, s);
        };
      }
      P.add(std::move(t));
    }
    Task t;
    t.type = TT_LN_PARTS;
    t.kernels = fused_ln ? 1 : 2;
    if (!fused_ln) {
      box(t.uses, gdy, ACC_R);
      box(t.uses, gxin, ACC_R);
      box(t.uses, gst, ACC_R);
      box(t.uses, m->gdres, ACC_R);
    }
    box(t.uses, m->gln_part, fused_ln ? ACC_R : ACC_RW);
    box(t.uses, m->ggrad[gidx_g], GW);
    box(t.uses, m->ggrad[gidx_b], GW);
    if (bias_idx >= 0) box(t.uses, m->ggrad[bias_idx], GW);
    float* og = pg(m, gm);
    float* ob = pg(m, bt_);
    float* obias = bias_idx >= 0 ? pg(m, m->params[bias_idx]) : nullptr;
    const int accum = acc ? 1 : 0;
    if (fused_ln) {
      const int64_t np = (int64_t)m->n_tok * ln_g;
      t.bytes = (double)np * 3 * d * 4;
      t.fn = [=](cudaStream_t s) {
        return launch_sum_parts3(m->ln_part_g, np, d, og, ob, obias, accum, s);
      };
    } else {
      t.bytes = (double)T * d * 4 * (bias_idx >= 0 ? 3 : 2);
      t.fn = [=](cudaStream_t s) {
        return launch_ln_bwd_colsums(dy, xin, mu, rs, obias ? m->dres : nullptr, T, d, m->ln_part_g, og,
                                     ob, obias, accum, s);
      };
    }
    P.add(std::move(t));
    adam_param(gidx_g);
    adam_param(gidx_b);
    if (bias_idx >= 0) adam_param(bias_idx);
  };
  const int pidx_lnf = 2 + 12 * m->L;

  // LM head backward: dy_f = dz wte (fp32), dwte = dz^T y
  for (int rt = 0; rt < m->n_tok; ++rt)
    for (auto [t0, t1] : b.col_groups(m->nce, m->te, d)) {
      const int c0 = tile_lo(t0, m->te), c1 = tile_hi(t1 - 1, m->te, d);
      GemmArgs g = b.base();
      g.M = T; g.N = d; g.K = V;
      g.m0 = b.row0(rt); g.mt = m->TT; g.n0 = c0; g.nt = c1 - c0;
      g.A = m->dz; g.lda = m->lddz; g.a_trans = 0;
      g.B = pw(m, m->params[0]); g.ldb = d; g.b_trans = 1;
      g.C = m->dtmp; g.ldc = d; g.c_dtype = NNT_F32;
      std::vector<TileUse> u;
      box(u, m->gdz, ACC_R, rt, rt + 1);
      box(u, m->gdtmp, ACC_W, rt, rt + 1, t0, t1);
      box(u, m->gpchunk[0], ACC_R);  // reads wte (before its update)
      b.gemm_task(P, TT_GEMM_LM_DX, g, std::move(u), 2.0 * m->TT * (c1 - c0) * V);
    }
  for (int vt = 0; vt < m->ncv; ++vt)
    for (auto [t0, t1] : b.col_groups(m->nce, m->te, d)) {
      const int v0 = tile_lo(vt, m->tv), v1 = tile_hi(vt, m->tv, V);
      const int c0 = tile_lo(t0, m->te), c1 = tile_hi(t1 - 1, m->te, d);
      GemmArgs g = b.base();
      g.M = V; g.N = d; g.K = T;
      g.m0 = v0; g.mt = v1 - v0; g.n0 = c0; g.nt = c1 - c0;
      g.A = m->dz; g.lda = m->lddz; g.a_trans = 1;
      g.B = m->y; g.ldb = d; g.b_trans = 1;
      g.C = pg(m, m->params[0]); g.ldc = d; g.c_dtype = NNT_F32;
      g.beta = acc ? 1 : 0;
      std::vector<TileUse> u;
      box(u, m->gdz, ACC_R);
      box(u, m->gy, ACC_R);
      box(u, m->ggrad[0], GW, vt, vt + 1, t0, t1);
      b.gemm_task(P, TT_GEMM_LM_DW, g, std::move(u), 2.0 * (v1 - v0) * (c1 - c0) * T);
    }
  // final LN backward (no residual input: dres starts here)
  ln_bwd(m->dtmp, m->gdtmp, m->x[m->L], m->gx[m->L], m->muf, m->rf, m->gstatf, m->params[pidx_lnf],
         m->params[pidx_lnf + 1], pidx_lnf, pidx_lnf + 1, false,
         m->L > 0 ? 2 + 12 * (m->L - 1) + PROJB : -1);

  const size_t zq = (size_t)S * hd;
  const int64_t BH = (int64_t)m->B * H;
  for (int l = m->L - 1; l >= 0; --l) {
    const int pi = 2 + 12 * l;
    // MLP: du = (dres W2) * gelu'(u)
    for (int rt = 0; rt < m->n_tok; ++rt)
      for (auto [t0, t1] : b.col_groups(m->ncf, m->ti, f)) {
        GemmArgs proto = b.base();
        proto.epi = EPI_GELU_BWD;
        proto.aux = m->u[l];
        proto.aux_dtype = act;
        proto.ld_aux = f;
        std::vector<TileUse> u;
        box(u, m->gdres_act, ACC_R, rt, rt + 1);
        box(u, m->gu[l], ACC_R, rt, rt + 1, t0, t1);
        box(u, m->gdu, ACC_W, rt, rt + 1, t0, t1);
        dx_gemm(TT_GEMM_DX, m->dres_act, d, d, P_(m, l, PROJW), f, m->du, act, f, m->ti, rt, t0, t1,
                proto, std::move(u));
      }
    dw_gemm(TT_GEMM_DW, m->dres_act, m->gdres_act, d, d, m->te, m->g[l], m->gg[l], f, f, m->ti,
            P_(m, l, PROJW), pi + PROJW);
    // dX before dW for each weight, so a fused update follows every read of it
    for (int rt = 0; rt < m->n_tok; ++rt)
      for (auto [t0, t1] : b.col_groups(m->nce, m->te, d)) {
        std::vector<TileUse> u;
        box(u, m->gdu, ACC_R, rt, rt + 1);
        box(u, m->gdtmp, ACC_W, rt, rt + 1, t0, t1);
        dx_gemm(TT_GEMM_DX, m->du, f, f, P_(m, l, FCW), d, m->dtmp, NNT_F32, d, m->te, rt, t0, t1,
                b.base(), std::move(u));
      }
    dw_gemm(TT_GEMM_DW, m->du, m->gdu, f, f, m->ti, m->h2[l], m->gh2[l], d, d, m->te, P_(m, l, FCW),
            pi + FCW);
    colsum_task(m->du, act, m->gdu, f, P_(m, l, FCB), pi + FCB);
    ln_bwd(m->dtmp, m->gdtmp, m->xmid[l], m->gxmid[l], m->mu2[l], m->r2[l], m->gstat2[l],
           P_(m, l, LN2G), P_(m, l, LN2B), pi + LN2G, pi + LN2B, true, pi + OB);
    // attention output projection: dO (head-major), dWo, dbo
    for (int rt = 0; rt < m->n_tok; ++rt)
      for (auto [t0, t1] : b.col_groups(m->nce, m->te, d)) {
        GemmArgs proto = b.base();
        proto.out_mode = OUT_HEADSPLIT;
        proto.hs_B = m->B; proto.hs_H = H; proto.hs_S = S; proto.hs_hd = hd; proto.hs_d = d;
        proto.ldc = d;
        const int c0 = tile_lo(t0, m->te), c1 = tile_hi(t1 - 1, m->te, d);
        int h0, h1;
        b.head_tiles(c0, c1, h0, h1);
        std::vector<TileUse> u;
        box(u, m->gdres_act, ACC_R, rt, rt + 1);
        box(u, m->gdOh, ACC_W, 0, 1, b.bt_of(rt), b.bt_of(rt) + 1, h0, h1, b.st_of(rt), b.st_of(rt) + 1);
        dx_gemm(TT_GEMM_DX, m->dres_act, d, d, P_(m, l, OW), d, m->dOh, act, d, m->te, rt, t0, t1,
                proto, std::move(u));
      }
    dw_gemm(TT_GEMM_DW, m->dres_act, m->gdres_act, d, d, m->te, m->O[l], m->gO[l], d, d, m->te,
            P_(m, l, OW), pi + OW);
    // attention backward per (batch tile, head tile)
    const char* qkv_base = (const char*)m->qkvh[l];
    if (m->flash) {
      // fused: recomputes P from the saved log-sum-exp; dQ, dK, dV head-merged into dqkv
      const bf16* qp = reinterpret_cast<const bf16*>(qkv_base);
      for (int bt = 0; bt < m->n_bt; ++bt)
        for (int ht = 0; ht < m->n_ht; ++ht) {
          FlashArgs fa = flash_args(m, bt, ht);
          fa.o = static_cast<bf16*>(m->O[l]);
          fa.ldo = d;
          fa.lse = m->lse[l];
          fa.D = m->attn_d;
          fa.ds = m->attn_ds;
          fa.dq = fa.dk = fa.dv = static_cast<bf16*>(m->dqkv);
          fa.ldd = 3 * d;
          fa.dq_col = 0;
          fa.dk_col = d;
          fa.dv_col = 2 * d;
          Task t;
          t.type = TT_FLASH_BWD;
          t.kernels = 3;
          box(t.uses, m->gqkvh[l], ACC_R, 0, 3, bt, bt + 1, ht, ht + 1);
          box(t.uses, m->gO[l], ACC_R, bt * m->n_st, (bt + 1) * m->n_st);
          box(t.uses, m->glse[l], ACC_R, bt, bt + 1, ht, ht + 1);
          box(t.uses, m->gdOh, ACC_R, 0, 1, bt, bt + 1, ht, ht + 1);
          box(t.uses, m->gattn_d, ACC_RW, bt, bt + 1, ht, ht + 1);
          box(t.uses, m->gdqkv, ACC_W, 0, 3, bt * m->n_st, (bt + 1) * m->n_st, ht, ht + 1);
          t.flops = 4 * 2.0 * hd * causal_rows(0, S) * fa.nz;  // dV, dP, dQ, dK, causal half
          const bf16* dO = static_cast<const bf16*>(m->dOh);
          t.fn = [=](cudaStream_t s) {
            return launch_flash_bwd(qp, qp + BH * zq, qp + 2 * BH * zq, dO, fa, s);
          };
          P.add(std::move(t));
        }
    }
    for (int bt = 0; bt < (m->flash ? 0 : m->n_bt); ++bt)
      for (int ht = 0; ht < m->n_ht; ++ht) {
        const int nz = m->tb * m->th;
        ZMap zm{bt * m->tb, ht * m->th, m->th, H};
        // dV = P^T dO per key tile
        for (int kt = 0; kt < m->n_st; ++kt) {
          const int k0 = kt * m->ts, nk = m->ts;
          GemmArgs g = b.base();
          g.M = S; g.N = hd; g.K = S; g.nbatch = nz; g.zm = zm;
          g.m0 = k0; g.mt = nk; g.n0 = 0; g.nt = hd;
          g.A = m->P[l]; g.lda = S; g.a_zs = (int64_t)S * S; g.a_trans = 1;
          g.B = m->dOh; g.ldb = hd; g.b_zs = zq; g.b_trans = 1;
          g.C = m->dqkv; g.ldc = 3 * d; g.c_dtype = act; g.out_mode = OUT_HEADMERGE;
          g.c_col_off = 2 * d; g.hs_hd = hd; g.hs_B = m->B; g.hs_S = S; g.hs_H = H;
          g.causal = CAUSAL_K_LOWER;
          std::vector<TileUse> u;
          box(u, m->gP[l], ACC_R, bt, bt + 1, ht, ht + 1);
          box(u, m->gdOh, ACC_R, 0, 1, bt, bt + 1, ht, ht + 1);
          box(u, m->gdqkv, ACC_W, 2, 3, bt * m->n_st + kt, bt * m->n_st + kt + 1, ht, ht + 1);
          const double pairs = (double)nk * S - causal_rows(k0, nk) + nk;  // sum_k (S - k)
          b.gemm_task(P, TT_GEMM_ATTN_BWD, g, std::move(u), 2.0 * hd * pairs * nz);
        }
        // dP = dO V^T, dS = softmax_bwd(P, dP) (into P's buffer), dQ = dS K per query tile
        for (int st = 0; st < m->n_st; ++st) {
          const int q0 = st * m->ts, nq = m->ts;
          {
            GemmArgs g = b.base();
            g.M = S; g.N = S; g.K = hd; g.nbatch = nz; g.zm = zm;
            g.m0 = q0; g.mt = nq; g.n0 = 0; g.nt = std::min<int>(S, (int)round_up(q0 + nq, kCausalBlock));
            g.A = m->dOh; g.lda = hd; g.a_zs = zq; g.a_trans = 0;
            g.B = qkv_base + 2 * BH * zq * as; g.ldb = hd; g.b_zs = zq; g.b_trans = 0;
            g.C = m->scores; g.ldc = S; g.c_zs = (int64_t)S * S; g.c_dtype = NNT_F32;
            g.causal = CAUSAL_TILES;
            std::vector<TileUse> u;
            box(u, m->gdOh, ACC_R, 0, 1, bt, bt + 1, ht, ht + 1, st, st + 1);
            box(u, m->gqkvh[l], ACC_R, 2, 3, bt, bt + 1, ht, ht + 1);
            box(u, m->gscores, ACC_W, bt, bt + 1, ht, ht + 1, st, st + 1);
            b.gemm_task(P, TT_GEMM_ATTN_BWD, g, std::move(u), 2.0 * hd * causal_rows(q0, nq) * nz);
          }
          {
            Task t;
            t.type = TT_SOFTMAX_BWD;
            box(t.uses, m->gscores, ACC_R, bt, bt + 1, ht, ht + 1, st, st + 1);
            box(t.uses, m->gP[l], ACC_RW, bt, bt + 1, ht, ht + 1, st, st + 1);
            t.bytes = causal_rows(q0, nq) * nz * (4 + 2 * as);
            void* Pl = m->P[l];
            const float scale = 1.0f / sqrtf((float)hd);
            t.fn = [=](cudaStream_t s) {
              return launch_softmax_bwd(Pl, m->scores, Pl, S, zm, nz, q0, nq, scale, act, s);
            };
            P.add(std::move(t));
          }
          {
            GemmArgs g = b.base();
            g.M = S; g.N = hd; g.K = S; g.nbatch = nz; g.zm = zm;
            g.m0 = q0; g.mt = nq; g.n0 = 0; g.nt = hd;
            g.A = m->P[l]; g.lda = S; g.a_zs = (int64_t)S * S; g.a_trans = 0;
            g.B = qkv_base + BH * zq * as; g.ldb = hd; g.b_zs = zq; g.b_trans = 1;
            g.C = m->dqkv; g.ldc = 3 * d; g.c_dtype = act; g.out_mode = OUT_HEADMERGE;
            g.c_col_off = 0; g.hs_hd = hd; g.hs_B = m->B; g.hs_S = S; g.hs_H = H;
            g.causal = CAUSAL_K_UPPER;
            std::vector<TileUse> u;
            box(u, m->gP[l], ACC_R, bt, bt + 1, ht, ht + 1, st, st + 1);
            box(u, m->gqkvh[l], ACC_R, 1, 2, bt, bt + 1, ht, ht + 1);
            box(u, m->gdqkv, ACC_W, 0, 1, bt * m->n_st + st, bt * m->n_st + st + 1, ht, ht + 1);
            b.gemm_task(P, TT_GEMM_ATTN_BWD, g, std::move(u), 2.0 * hd * causal_rows(q0, nq) * nz);
          }
        }
        // dK = dS^T Q per key tile
        for (int kt = 0; kt < m->n_st; ++kt) {
          const int k0 = kt * m->ts, nk = m->ts;
          GemmArgs g = b.base();
          g.M = S; g.N = hd; g.K = S; g.nbatch = nz; g.zm = zm;
          g.m0 = k0; g.mt = nk; g.n0 = 0; g.nt = hd;
          g.A = m->P[l]; g.lda = S; g.a_zs = (int64_t)S * S; g.a_trans = 1;
          g.B = qkv_base; g.ldb = hd; g.b_zs = zq; g.b_trans = 1;
          g.C = m->dqkv; g.ldc = 3 * d; g.c_dtype = act; g.out_mode = OUT_HEADMERGE;
          g.c_col_off = d; g.hs_hd = hd; g.hs_B = m->B; g.hs_S = S; g.hs_H = H;
          g.causal = CAUSAL_K_LOWER;
          std::vector<TileUse> u;
          box(u, m->gP[l], ACC_R, bt, bt + 1, ht, ht + 1);
          box(u, m->gqkvh[l], ACC_R, 0, 1, bt, bt + 1, ht, ht + 1);
          box(u, m->gdqkv, ACC_W, 1, 2, bt * m->n_st + kt, bt * m->n_st + kt + 1, ht, ht + 1);
          const double pairs = (double)nk * S - causal_rows(k0, nk) + nk;
          b.gemm_task(P, TT_GEMM_ATTN_BWD, g, std::move(u), 2.0 * hd * pairs * nz);
        }
      }
    // QKV projection backward (dX first, then dW and its update)
    for (int rt = 0; rt < m->n_tok; ++rt)
      for (auto [t0, t1] : b.col_groups(m->nce, m->te, d)) {
        std::vector<TileUse> u;
        box(u, m->gdqkv, ACC_R, 0, 3, rt, rt + 1);
        box(u, m->gdtmp, ACC_W, rt, rt + 1, t0, t1);
        dx_gemm(TT_GEMM_DX, m->dqkv, 3 * d, 3 * d, P_(m, l, QKVW), d, m->dtmp, NNT_F32, d, m->te, rt,
                t0, t1, b.base(), std::move(u));
      }
    dw_gemm(TT_GEMM_DW, m->dqkv, m->gdqkv, 3 * d, 3 * d, m->te, m->h1[l], m->gh1[l], d, d, m->te,
            P_(m, l, QKVW), pi + QKVW);
    colsum_task(m->dqkv, act, m->gdqkv, 3 * d, P_(m, l, QKVB), pi + QKVB);
    ln_bwd(m->dtmp, m->gdtmp, m->x[l], m->gx[l], m->mu1[l], m->r1[l], m->gstat1[l], P_(m, l, LN1G),
           P_(m, l, LN1B), pi + LN1G, pi + LN1B, true, l > 0 ? pi - 12 + PROJB : -1);
  }
  // embedding backward: token sort, wte scatter-add (after the LM-head dW), wpe sums
  {
    Task t;
    t.type = TT_EMB_SORT;
    box(t.uses, m->gtok, ACC_R);
    box(t.uses, m->gkeys, ACC_W);
    t.bytes = 6.0 * T;
    t.fn = [m](cudaStream_t s) {
      return launch_token_sort(m->tokens_dev, m->S + 1, m->B, m->S, m->sort_keys, s);
    };
    P.add(std::move(t));
  }
  {
    Task t;
    t.type = TT_EMB_SCATTER;
    box(t.uses, m->gkeys, ACC_R);
    box(t.uses, m->gdres, ACC_R);
    box(t.uses, m->ggrad[0], ACC_RW);
    t.bytes = (double)T * d * 12;
    t.fn = [m](cudaStream_t s) {
      return launch_embedding_scatter(m->sort_keys, m->T, m->dres, m->tm, m->S,
                                      pg(m, m->params[0]), m->d, m->V, s);
    };
    P.add(std::move(t));
    adam_param(0);
  }
  for (int st = 0; st < m->n_st; ++st) {
    Task t;
    t.type = TT_WPE_GRAD;
    for (int bt = 0; bt < m->n_bt; ++bt) box(t.uses, m->gdres, ACC_R, bt * m->n_st + st, bt * m->n_st + st + 1);
    box(t.uses, m->ggrad[1], GW, st, st + 1);
    t.bytes = (double)T / m->n_st * d * 4 + (double)m->ts * d * 4;
    const int s0 = st * m->ts;
    const int accum = acc ? 1 : 0;
    t.fn = [m, s0, accum](cudaStream_t s) {
      return launch_wpe_grad(m->dres, m->tm, m->B, s0, m->ts, m->d, pg(m, m->params[1]), accum, s);
    };
    P.add(std::move(t));
  }
  adam_param(1);
}

void build_optimizer(nnt_model* m) {
  // one AdamW task per chunk of the flat parameter buffers (<= 256 Mi elements)
  if (m->offload) return;  // offloaded models update inside the fused backward only
  const int64_t chunk = 256ll << 20;
  for (int64_t o = 0; o < m->n_flat; o += chunk) {
    const int64_t n = std::min(chunk, m->n_flat - o);
    Task t;
    t.type = TT_ADAMW;
    t.bytes = 30.0 * n;
    t.fn = [m, o, n](cudaStream_t s) {
      return launch_adamw_dev(m->master + o, m->grad + o, m->mom1 + o, m->mom2 + o, m->wbf + o, n,
                              reinterpret_cast<const float*>(m->hyper_dev), s);
    };
    m->opt.add(std::move(t));
  }
}

void make_grids(nnt_model* m) {
  const int L = m->L;
  for (int l = 0; l <= L; ++l) m->gx.push_back(new_grid(m, m->n_tok, m->nce));
  for (int l = 0; l < L; ++l) {
    m->gxmid.push_back(new_grid(m, m->n_tok, m->nce));
    m->gh1.push_back(new_grid(m, m->n_tok, m->nce));
    m->gstat1.push_back(new_grid(m, m->n_tok));
    m->gqkvh.push_back(new_grid(m, 3, m->n_bt, m->n_ht, m->n_st));
    m->gP.push_back(new_grid(m, m->n_bt, m->n_ht, m->n_st));
    m->glse.push_back(new_grid(m, m->n_bt, m->n_ht));
    m->gO.push_back(new_grid(m, m->n_tok, m->nce));
    m->gh2.push_back(new_grid(m, m->n_tok, m->nce));
    m->gstat2.push_back(new_grid(m, m->n_tok));
    m->gu.push_back(new_grid(m, m->n_tok, m->ncf));
    m->gg.push_back(new_grid(m, m->n_tok, m->ncf));
  }
  m->gscores = new_grid(m, m->n_bt, m->n_ht, m->n_st);
  m->gattn_d = new_grid(m, m->n_bt, m->n_ht);
  m->gy = new_grid(m, m->n_tok, m->nce);
  m->gstatf = new_grid(m, m->n_tok);
  m->gz = new_grid(m, m->n_tok, m->ncv);
  m->gdz = new_grid(m, m->n_tok, m->ncv);
  m->grow_loss = new_grid(m, m->n_tok);
  m->gloss = new_grid(m, 1);
  m->gtok = new_grid(m, 1);
  m->gdres = new_grid(m, m->n_tok, m->nce);
  m->gdres_act = new_grid(m, m->n_tok, m->nce);
  m->gdtmp = new_grid(m, m->n_tok, m->nce);
  m->gdu = new_grid(m, m->n_tok, m->ncf);
  m->gdOh = new_grid(m, 1, m->n_bt, m->n_ht, m->n_st);
  m->gdqkv = new_grid(m, 3, m->n_tok, m->n_ht);
  m->gln_part = new_grid(m, m->n_tok);
  m->gcol_part = new_grid(m, 1);
  m->gkeys = new_grid(m, 1);
  m->gsplitk = new_grid(m, 1);
  // parameter gradients: weights tiled [out tile, in tile], vectors by their axis
  for (const ParamInfo& p : m->params) {
    int a = tiles_of((int)p.shape0, axis_tile(m, p.shape0));
    int bcount = p.shape1 ? tiles_of((int)p.shape1, axis_tile(m, p.shape1)) : 1;
    m->ggrad.push_back(new_grid(m, a, bcount));
  }
  for (size_t i = 0; i < m->params.size(); ++i)
    m->gpchunk.push_back(new_grid(m, (int)m->chunks_of[i].size()));
  m->gring = new_grid(m, std::max(1, m->n_ring));
}

nnt_status wait_event(nnt_model* m, cudaEvent_t ev) {
  const uint32_t tmo = m->opts.timeout_ms ? m->opts.timeout_ms : 600000u;
  if (fault_hit(FAULT_EVENT_WAIT)) {
    set_thread_error("wait for the device timed out after %u ms (injected)", tmo);
    return NNT_ERR_TIMEOUT;
  }
  auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return NNT_OK;
    if (e != cudaErrorNotReady) {
      set_thread_error("device work failed: %s", cudaGetErrorString(e));
      return NNT_ERR_CUDA;
    }
    auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0).count();
    if (ms > tmo) {
      set_thread_error("wait for the device timed out after %u ms", tmo);
      return NNT_ERR_TIMEOUT;
    }
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

nnt_status sync_model(nnt_model* m) {
  NNT_CUDA_TRY(cudaEventRecord(m->done_event, m->ex.main_));
  return wait_event(m, m->done_event);
}

nnt_status check_device_error(nnt_model* m) {
  uint32_t code = 0;
  NNT_TRY(read_and_clear_device_error(&code, m->ex.main_));
  if (code & DEVERR_TOKEN_RANGE) {
    set_thread_error("token id >= vocab (%d) in the batch", m->V);
    return NNT_ERR_INVALID_ARG;
  }
  if (code) {
    set_thread_error("device error word 0x%x", code);
    return NNT_ERR_INTERNAL;
  }
  return NNT_OK;
}

void free_model(nnt_model* m) {
  if (!m) return;
  cudaDeviceSynchronize();
  for (void* p : m->dev_allocs) cudaFree(p);
  m->dev_allocs.clear();
  if (m->loss_host) cudaFreeHost(m->loss_host);
  if (m->host_m) cudaFreeHost(m->host_m);
  if (m->host_v) cudaFreeHost(m->host_v);
  if (m->done_event) cudaEventDestroy(m->done_event);
  cudaStream_t own = m->ex.main_;
  bool owned = m->opts.stream == nullptr;
  m->ex.~Executor();
  new (&m->ex) Executor();
  if (owned && own) cudaStreamDestroy(own);
}

// Learning rate of AdamW iteration t (1-based) under the README's warm-up
// flags: --start-lr is the rate of the first iteration and --full-lr-iter the
// iteration from which the full --lr applies. The pages do not say how the
// rate moves in between; it is read as a straight line from start_lr at t = 1
// to lr at t = full_lr_iter. full_lr_iter <= 1 means the full rate throughout.
double scheduled_lr(const nnt_adamw* hp, int64_t t) {
  if (hp->full_lr_iter <= 1 || t >= hp->full_lr_iter) return hp->lr;
  const double frac = (double)(t - 1) / (double)(hp->full_lr_iter - 1);
  return (double)hp->start_lr + ((double)hp->lr - (double)hp->start_lr) * frac;
}

bool valid_adamw(const nnt_adamw* hp) {
  if (!(hp->lr >= 0) || !(hp->beta1 >= 0 && hp->beta1 < 1) || !(hp->beta2 >= 0 && hp->beta2 < 1) ||
      !(hp->eps > 0) || !(hp->weight_decay >= 0) || !(hp->start_lr >= 0) || hp->full_lr_iter < 0) {
    set_thread_error("invalid AdamW hyper-parameters");
    return false;
  }
  return true;
}

// Device copy of the hyper-parameters of iteration t: the captured AdamW
// graphs read them from there, so one graph serves every step.
nnt_status upload_hyper(nnt_model* m, const nnt_adamw* hp, int64_t t, float gscale) {
  AdamHyperDev& h = m->hyper_host;
  h.lr = (float)scheduled_lr(hp, t);
  h.b1 = hp->beta1; h.b2 = hp->beta2; h.eps = hp->eps; h.wd = hp->weight_decay;
  h.bc1 = (float)(1.0 - pow((double)hp->beta1, (double)t));
  h.bc2 = (float)(1.0 - pow((double)hp->beta2, (double)t));
  h.gscale = gscale;
  return copy_async(m->hyper_dev, &h, sizeof h, cudaMemcpyHostToDevice, m->ex.main_,
                    "hyper-parameter upload");
}

// nnt_backward (acc = false) and nnt_backward_accumulate (acc = true).
nnt_status run_backward(nnt_model* m, bool acc, const char* who) {
  if (!m) {
    set_thread_error("NULL model");
    return fail(m, NNT_ERR_INVALID_ARG);
  }
  if (m->state != 1) {
    set_thread_error("%s needs a preceding nnt_forward", who);
    return fail(m, NNT_ERR_STATE);
  }
  if (m->offload) {
    set_thread_error("this model offloads AdamW moments: gradients are not kept whole; use "
                     "nnt_backward_adamw");
    return fail(m, NNT_ERR_STATE);
  }
  // the first minibatch after an update writes the gradients, later ones add
  const bool add = acc && m->n_acc > 0;
  auto t0 = std::chrono::steady_clock::now();
  nnt_status s = add ? m->ex.run(m->bwda, m->opts.use_cuda_graph ? kSlotBwdAcc : -1)
                     : m->ex.run(m->bwd, m->opts.use_cuda_graph ? 1 : -1);
  if (s != NNT_OK) {
    m->n_acc = 0;  // the gradients are no longer a known sum
    return fail(m, s);
  }
  m->n_acc = add ? m->n_acc + 1 : 1;
  m->state = 2;
  if (m->opts.trace) {
    s = sync_model(m);
    if (s == NNT_OK) s = m->ex.collect_trace(add ? m->bwda : m->bwd);
    if (s != NNT_OK) return fail(m, s);
    m->last_bwd_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  }
  return NNT_OK;
}

// Model fields that follow from the config, tile sizes and options.
nnt_status setup_fields(nnt_model* m, const nnt_gpt2_config* cfg, const nnt_tiles* tiles,
                        const nnt_options* opts) {
  m->cfg = *cfg;
  nnt_tiles zt{};
  m->tiles = tiles ? *tiles : zt;
  nnt_options zo{};
  m->opts = opts ? *opts : zo;
  m->act = cfg->dtype;
  m->act_size = m->act == NNT_BF16 ? 2 : 4;
  m->L = cfg->n_layer; m->d = cfg->d_model; m->H = cfg->n_head; m->hd = m->d / m->H;
  m->f = cfg->d_ff; m->V = cfg->vocab; m->S = cfg->n_ctx; m->B = cfg->batch; m->T = m->B * m->S;
  m->tb = m->tiles.batch_tile ? m->tiles.batch_tile : m->B;
  m->ts = m->tiles.seq_tile ? m->tiles.seq_tile : m->S;
  m->te = m->tiles.embd_tile ? std::min(m->tiles.embd_tile, m->d) : m->d;
  m->ti = m->tiles.inner_tile ? std::min(m->tiles.inner_tile, m->f) : m->f;
  m->th = m->tiles.head_tile ? m->tiles.head_tile : m->H;
  m->tv = m->tiles.vocab_tile ? std::min(m->tiles.vocab_tile, m->V) : m->V;
  m->n_bt = m->B / m->tb; m->n_st = m->S / m->ts; m->n_ht = m->H / m->th;
  m->n_tok = m->n_bt * m->n_st; m->TT = m->tb * m->ts;
  m->nce = tiles_of(m->d, m->te); m->ncf = tiles_of(m->f, m->ti); m->ncv = tiles_of(m->V, m->tv);
  m->tm = TokMap{m->S, m->tb, m->ts, m->n_st};
  m->ldz = round_up(m->V, 4);
  m->lddz = round_up(m->V, 8);
  m->backend = m->opts.gemm_backend;
  m->gemm_min_cols = m->opts.gemm_min_task_cols == 0 ? 8192 : std::max(0, m->opts.gemm_min_task_cols);
  if (m->opts.n_streams <= 0) m->opts.n_streams = 2;
  m->opts.n_streams = std::min(m->opts.n_streams, 8);
  {
    const bool usable = m->act == NNT_BF16 && m->backend == 0 && flash_supported(m->hd);
    if (m->opts.flash_attention > 0 && !usable) {
      set_thread_error("flash attention needs bf16, tensor-core GEMMs and head size 64 or 128 "
                       "(head size %d)", m->hd);
      return NNT_ERR_INVALID_ARG;
    }
    m->flash = m->opts.flash_attention >= 0 && usable;
  }

  return NNT_OK;
}

uint64_t host_mem_available() {
  FILE* fh = fopen("/proc/meminfo", "r");
  if (!fh) return 0;
  char line[256];
  unsigned long long kb = 0;
  while (fgets(line, sizeof line, fh))
    if (sscanf(line, "MemAvailable: %llu kB", &kb) == 1) break;
  fclose(fh);
  return (uint64_t)kb * 1024;
}

// Device and pinned-host bytes of the model's allocations, from a dry run of
// the allocation plan; free_device is the free device memory the default
// device budget is taken from.
nnt_status plan_bytes(const nnt_gpt2_config* cfg, const nnt_tiles* tiles, const nnt_options* opts,
                      uint64_t free_device, uint64_t* dev, uint64_t* host) {
  nnt_model tmp;
  NNT_TRY(setup_fields(&tmp, cfg, tiles, opts));
  tmp.dry = true;
  tmp.free_device = free_device;
  NNT_TRY(alloc_all(&tmp));
  *dev = tmp.device_bytes;
  *host = tmp.host_bytes;
  return NNT_OK;
}

}  // namespace

extern "C" {


nnt_status nnt_create_model(const nnt_gpt2_config* cfg, const nnt_tiles* tiles,
                            const nnt_options* opts, nnt_model** out) {
  if (!out) {
    set_thread_error("out is NULL");
    t_model_err = thread_error();
    return NNT_ERR_INVALID_ARG;
  }
  *out = nullptr;
  nnt_status s = validate(cfg, tiles);
  if (s != NNT_OK) return fail(nullptr, s);
  nnt_model* m = new nnt_model();
  s = setup_fields(m, cfg, tiles, opts);
  if (s != NNT_OK) {
    delete m;
    return fail(nullptr, s);
  }
  {
    // the whole allocation plan must fit before anything is allocated
    size_t free_b = 0, total_b = 0;
    cudaError_t e = cudaMemGetInfo(&free_b, &total_b);
    if (e != cudaSuccess) {
      set_thread_error("cudaMemGetInfo: %s", cudaGetErrorString(e));
      delete m;
      return fail(nullptr, NNT_ERR_CUDA);
    }
    uint64_t dev = 0, host = 0;
    s = plan_bytes(cfg, tiles, opts, free_b, &dev, &host);
    if (s != NNT_OK) {
      delete m;
      return fail(nullptr, s);
    }
    const uint64_t avail = host_mem_available();
    const uint64_t host_budget = m->opts.host_budget_bytes
                                     ? m->opts.host_budget_bytes
                                     : (avail > (8ull << 30) ? avail - (8ull << 30) : avail);
    if (dev > free_b) {
      set_thread_error("the model needs %.2f GiB of device memory, %.2f GiB are free", dev / 1073741824.0,
                       free_b / 1073741824.0);
      delete m;
      return fail(nullptr, NNT_ERR_OOM);
    }
    if (host > 64 && host_budget && host > host_budget) {
      set_thread_error("the model needs %.2f GiB of pinned host memory, the budget is %.2f GiB",
                       host / 1073741824.0, host_budget / 1073741824.0);
      delete m;
      return fail(nullptr, NNT_ERR_OOM);
    }
  }

  cudaStream_t main = (cudaStream_t)m->opts.stream;
  if (!main) {
    cudaError_t e = cudaStreamCreate(&main);
    if (e != cudaSuccess) {
      set_thread_error("cudaStreamCreate: %s", cudaGetErrorString(e));
      delete m;
      return fail(nullptr, NNT_ERR_CUDA);
    }
  }
  s = m->ex.init(main, m->opts.n_streams, true, m->opts.trace != 0, TT_COUNT);
  if (s == NNT_OK && cudaEventCreateWithFlags(&m->done_event, cudaEventDisableTiming) != cudaSuccess)
    s = NNT_ERR_CUDA;
  if (s == NNT_OK) s = alloc_all(m);
  if (s == NNT_OK) s = init_params(m, main);
  if (s == NNT_OK) {
    make_grids(m);
    build_forward(m);
    if (!m->offload) {
      build_backward(m, m->bwd, false);
      build_backward(m, m->bwda, false, true);
    }
    build_backward(m, m->bwdf, true);
    build_optimizer(m);
    m->fwd.finalize(m->opts.n_streams);
    m->bwd.finalize(m->opts.n_streams);
    m->bwda.finalize(m->opts.n_streams);
    m->bwdf.finalize(m->opts.n_streams);
    m->opt.finalize(1);
    s = sync_model(m);
  }
  if (s != NNT_OK) {
    fail(nullptr, s);
    free_model(m);
    delete m;
    return s;
  }
  *out = m;
  return NNT_OK;
}

nnt_status nnt_plan_memory(const nnt_gpt2_config* cfg, const nnt_tiles* tiles, const nnt_options* opts,
                           uint64_t* device_bytes, uint64_t* host_pinned_bytes) {
  if (!device_bytes || !host_pinned_bytes) {
    set_thread_error("NULL output");
    return fail(nullptr, NNT_ERR_INVALID_ARG);
  }
  nnt_status s = validate(cfg, tiles);
  if (s != NNT_OK) return fail(nullptr, s);
  size_t free_b = 0, total_b = 0;
  if (!(opts && opts->hbm_budget_bytes)) {
    cudaError_t e = cudaMemGetInfo(&free_b, &total_b);
    if (e != cudaSuccess) {
      cudaGetLastError();
      set_thread_error("cudaMemGetInfo: %s (set hbm_budget_bytes to plan without a device)",
                       cudaGetErrorString(e));
      return fail(nullptr, NNT_ERR_CUDA);
    }
  }
  s = plan_bytes(cfg, tiles, opts, free_b, device_bytes, host_pinned_bytes);
  return s == NNT_OK ? s : fail(nullptr, s);
}

nnt_status nnt_forward(nnt_model* m, const uint16_t* tokens, int32_t tokens_on_device,
                       float* loss_out) {
  if (!m || !tokens) {
    set_thread_error("NULL model or tokens");
    return fail(m, NNT_ERR_INVALID_ARG);
  }
  auto t0 = std::chrono::steady_clock::now();
  const size_t tb = (size_t)m->B * (m->S + 1) * 2;
  cudaStream_t st = m->ex.main_;
  nnt_status s = NNT_OK;
  s = copy_async(m->tokens_dev, tokens, tb, tokens_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                 st, "token copy");
  if (s != NNT_OK) return fail(m, s);
  s = m->ex.run(m->fwd, m->opts.use_cuda_graph ? 0 : -1);
  if (s != NNT_OK) return fail(m, s);
  m->state = 1;
  if (loss_out || m->opts.trace) {
    s = copy_async(m->loss_host, m->loss_dev, 4, cudaMemcpyDeviceToHost, st, "loss read-back");
    if (s == NNT_OK) s = sync_model(m);  // bounded wait for the step and the copy
    if (s != NNT_OK) {
      m->state = 0;
      return fail(m, s);
    }
    s = check_device_error(m);
    if (s != NNT_OK) {
      m->state = 0;
      return fail(m, s);
    }
    if (loss_out) *loss_out = *m->loss_host;
    if (m->opts.trace) {
      s = m->ex.collect_trace(m->fwd);
      if (s != NNT_OK) return fail(m, s);
    }
    m->last_fwd_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  }
  return NNT_OK;
}

nnt_status nnt_backward(nnt_model* m) { return run_backward(m, false, "nnt_backward"); }

nnt_status nnt_backward_accumulate(nnt_model* m) {
  return run_backward(m, true, "nnt_backward_accumulate");
}

nnt_status nnt_adamw_step(nnt_model* m, const nnt_adamw* hp) {
  if (!m || !hp) {
    set_thread_error("NULL model or hyper-parameters");
    return fail(m, NNT_ERR_INVALID_ARG);
  }
  if (m->n_acc < 1) {
    set_thread_error("nnt_adamw_step needs a preceding nnt_backward or nnt_backward_accumulate");
    return fail(m, NNT_ERR_STATE);
  }
  if (m->offload) {
    set_thread_error("this model offloads AdamW moments; use nnt_backward_adamw");
    return fail(m, NNT_ERR_STATE);
  }
  if (!valid_adamw(hp)) return fail(m, NNT_ERR_INVALID_ARG);
  auto t0 = std::chrono::steady_clock::now();
  const int64_t t = m->step + 1;
  if (upload_hyper(m, hp, t, 1.0f / (float)m->n_acc) != NNT_OK) return fail(m, NNT_ERR_CUDA);
  nnt_status s = m->ex.run(m->opt, m->opts.use_cuda_graph ? 2 : -1);
  if (s != NNT_OK) return fail(m, s);
  m->step = t;
  m->state = 0;
  m->n_acc = 0;
  if (m->opts.trace) {
    s = sync_model(m);
    if (s == NNT_OK) s = m->ex.collect_trace(m->opt);
    if (s != NNT_OK) return fail(m, s);
    m->last_opt_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  }
  return NNT_OK;
}

nnt_status nnt_backward_adamw(nnt_model* m, const nnt_adamw* hp) {
  if (!m || !hp) {
    set_thread_error("NULL model or hyper-parameters");
    return fail(m, NNT_ERR_INVALID_ARG);
  }
  if (m->state != 1) {
    set_thread_error("nnt_backward_adamw needs a preceding nnt_forward");
    return fail(m, NNT_ERR_STATE);
  }
  if (m->n_acc > 0) {
    set_thread_error("nnt_backward_adamw cannot add to accumulated gradients: finish the "
                     "accumulation with nnt_backward_accumulate + nnt_adamw_step");
    return fail(m, NNT_ERR_STATE);
  }
  if (!valid_adamw(hp)) return fail(m, NNT_ERR_INVALID_ARG);
  auto t0 = std::chrono::steady_clock::now();
  const int64_t t = m->step + 1;
  if (upload_hyper(m, hp, t, 1.0f) != NNT_OK) return fail(m, NNT_ERR_CUDA);
  nnt_status s = m->ex.run(m->bwdf, m->opts.use_cuda_graph ? 3 : -1);
  if (s != NNT_OK) return fail(m, s);
  m->step = t;
  m->state = 0;
  for (const Chunk& c : m->chunks)
    if (c.host) {
      m->h2d_bytes += (uint64_t)c.n * 8;  // m and v read over C2C
      m->d2h_bytes += (uint64_t)c.n * 8;  // and written back
    }
  if (m->opts.trace) {
    s = sync_model(m);
    if (s == NNT_OK) s = m->ex.collect_trace(m->bwdf);
    if (s != NNT_OK) return fail(m, s);
    m->last_bwd_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  }
  return NNT_OK;
}

void nnt_destroy(nnt_model* m) {
  if (!m) return;
  free_model(m);
  delete m;
}

int32_t nnt_num_params(const nnt_model* m) { return m ? (int32_t)m->params.size() : -1; }

nnt_status nnt_param_info(const nnt_model* m, int32_t i, const char** name, int64_t shape[2]) {
  if (!m || i < 0 || i >= (int32_t)m->params.size()) {
    set_thread_error("bad parameter index");
    return NNT_ERR_INVALID_ARG;
  }
  if (name) *name = m->params[i].name.c_str();
  if (shape) {
    shape[0] = m->params[i].shape0;
    shape[1] = m->params[i].shape1;
  }
  return NNT_OK;
}

static nnt_status copy_param(nnt_model* m, int32_t i, float* base, float* host, bool to_dev) {
  if (!m || !host || i < 0 || i >= (int32_t)m->params.size()) {
    set_thread_error("bad model, buffer or parameter index");
    return fail(m, NNT_ERR_INVALID_ARG);
  }
  const ParamInfo& p = m->params[i];
  cudaStream_t st = m->ex.main_;
  if (to_dev) {
    nnt_status c = copy_async(base + p.off, host, p.n * 4, cudaMemcpyHostToDevice, st, "parameter upload");
    if (c != NNT_OK) return fail(m, c);
    if (base == m->master) {
      nnt_status s = launch_cast_bf16(m->master + p.off, m->wbf + p.off, p.n, st);
      if (s != NNT_OK) return fail(m, s);
    }
  } else {
    nnt_status c = copy_async(host, base + p.off, p.n * 4, cudaMemcpyDeviceToHost, st, "parameter read-back");
    if (c != NNT_OK) return fail(m, c);
  }
  nnt_status s = sync_model(m);
  return s == NNT_OK ? s : fail(m, s);
}

nnt_status nnt_get_param(nnt_model* m, int32_t i, float* host_buf) {
  return copy_param(m, i, m ? m->master : nullptr, host_buf, false);
}
nnt_status nnt_set_param(nnt_model* m, int32_t i, const float* host_buf) {
  return copy_param(m, i, m ? m->master : nullptr, const_cast<float*>(host_buf), true);
}
nnt_status nnt_get_grad(nnt_model* m, int32_t i, float* host_buf) {
  if (m && i >= 0 && i < (int32_t)m->params.size() && m->params[i].goff < 0) {
    set_thread_error("gradients of %s are streamed through the ring and not kept",
                     m->params[i].name.c_str());
    return fail(m, NNT_ERR_STATE);
  }
  if (m && i >= 0 && i < (int32_t)m->params.size() && host_buf) {
    const ParamInfo& p = m->params[i];
    nnt_status s = copy_async(host_buf, m->grad + p.goff, p.n * 4, cudaMemcpyDeviceToHost, m->ex.main_,
                              "gradient read-back");
    if (s != NNT_OK) return fail(m, s);
    s = sync_model(m);
    return s == NNT_OK ? s : fail(m, s);
  }
  set_thread_error("bad model, buffer or parameter index");
  return fail(m, NNT_ERR_INVALID_ARG);
}
nnt_status nnt_get_adam_state(nnt_model* m, int32_t i, int32_t which, float* host_buf) {
  if (which != 0 && which != 1) {
    set_thread_error("which must be 0 (m) or 1 (v)");
    return fail(m, NNT_ERR_INVALID_ARG);
  }
  if (!m || !host_buf || i < 0 || i >= (int32_t)m->params.size()) {
    set_thread_error("bad model, buffer or parameter index");
    return fail(m, NNT_ERR_INVALID_ARG);
  }
  nnt_status s = sync_model(m);
  if (s != NNT_OK) return fail(m, s);
  for (int ci : m->chunks_of[i]) {
    const Chunk& c = m->chunks[ci];
    float* dst = host_buf + c.e0;
    if (c.host) {
      memcpy(dst, (which ? m->host_v : m->host_m) + c.mv_off, (size_t)c.n * 4);
    } else {
      s = copy_async(dst, (which ? m->mom2 : m->mom1) + c.mv_off, (size_t)c.n * 4, cudaMemcpyDeviceToHost,
                     m->ex.main_, "AdamW state read-back");
      if (s != NNT_OK) return fail(m, s);
    }
  }
  s = sync_model(m);
  return s == NNT_OK ? s : fail(m, s);
}

nnt_status nnt_get_logits(nnt_model* m, float* host_buf) {
  if (!m || !host_buf) {
    set_thread_error("NULL model or buffer");
    return fail(m, NNT_ERR_INVALID_ARG);
  }
  // storage rows are tile-major; copy each run of seq_tile positions of one
  // sequence to its (b, s) place
  for (int bt = 0; bt < m->n_bt; ++bt)
    for (int st = 0; st < m->n_st; ++st)
      for (int bl = 0; bl < m->tb; ++bl) {
        const int b = bt * m->tb + bl, s0 = st * m->ts;
        const int64_t src_row = m->tm.row(b, s0);
        if (fault_hit(FAULT_COPY)) {
          set_thread_error("logits read-back: async copy submission failed (injected)");
          return fail(m, NNT_ERR_CUDA);
        }
        if (cudaMemcpy2DAsync(host_buf + ((int64_t)b * m->S + s0) * m->V, (size_t)m->V * 4,
                              m->z + src_row * m->ldz, (size_t)m->ldz * 4, (size_t)m->V * 4, m->ts,
                              cudaMemcpyDeviceToHost, m->ex.main_) != cudaSuccess)
          return fail(m, NNT_ERR_CUDA);
      }
  nnt_status s = sync_model(m);
  return s == NNT_OK ? s : fail(m, s);
}

nnt_status nnt_get_stats(const nnt_model* m, nnt_stats* out) {
  if (!m || !out) {
    set_thread_error("NULL model or stats");
    return NNT_ERR_INVALID_ARG;
  }
  memset(out, 0, sizeof *out);
  out->last_forward_ms = m->last_fwd_ms;
  out->last_backward_ms = m->last_bwd_ms;
  out->last_adamw_ms = m->last_opt_ms;
  out->device_bytes = m->device_bytes;
  out->host_pinned_bytes = m->host_bytes;
  out->n_tasks_forward = (int64_t)m->fwd.size();
  out->n_tasks_backward = (int64_t)m->bwd.size();
  out->n_tasks_adamw = (int64_t)m->opt.size();
  out->n_tiles = m->next_tile;
  out->n_params = m->n_scalar;
  out->n_streams = m->opts.n_streams;
  out->offload_active = m->offload ? 1 : 0;
  out->h2d_bytes = m->h2d_bytes;
  out->d2h_bytes = m->d2h_bytes;
  out->kernels_forward = m->fwd.kernels();
  out->kernels_backward = m->offload ? m->bwdf.kernels() : m->bwd.kernels();
  out->kernels_adamw = m->opt.kernels();
  out->flash_attention = m->flash ? 1 : 0;
  return NNT_OK;
}

int32_t nnt_get_task_times(const nnt_model* m, int32_t max_types, const char** names,
                           int64_t* launches, double* ms, double* flops, double* bytes) {
  if (!m) return -1;
  const int n = std::min<int>(max_types, TT_COUNT);
  for (int i = 0; i < n; ++i) {
    if (names) names[i] = kTaskNames[i];
    if (launches) launches[i] = m->ex.type_launches_.empty() ? 0 : m->ex.type_launches_[i];
    if (ms) ms[i] = m->ex.type_ms_.empty() ? 0 : m->ex.type_ms_[i];
    if (flops) flops[i] = m->ex.type_flops_.empty() ? 0 : m->ex.type_flops_[i];
    if (bytes) bytes[i] = m->ex.type_bytes_.empty() ? 0 : m->ex.type_bytes_[i];
  }
  return TT_COUNT;
}

nnt_status nnt_set_trace(nnt_model* m, int32_t on) {
  if (!m) {
    set_thread_error("NULL model");
    return NNT_ERR_INVALID_ARG;
  }
  nnt_status s = sync_model(m);
  if (s != NNT_OK) return fail(m, s);
  m->opts.trace = on ? 1 : 0;
  m->ex.set_trace(on != 0);
  m->ex.reset_trace();
  // traced runs are serialised on one stream, so each task's time is its own
  const int ns = on ? 1 : m->opts.n_streams;
  m->fwd.finalize(ns);
  m->bwd.finalize(ns);
  m->bwdf.finalize(ns);
  m->ex.drop_graphs();
  return NNT_OK;
}

const char* nnt_last_error(const nnt_model* m) {
  if (m) return m->err.c_str();
  return thread_error();  // the last error of any call on this thread
}

}  // extern "C"
