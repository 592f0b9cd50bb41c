/*
 * nnt.h -- C ABI of the GB300 tile-task GPT2 training step (libnnt.so).
 *
 * What the library computes: one GPT2 training step -- forward pass, backward
 * pass and a fused AdamW update -- with every tensor split into tiles along all
 * of its axes and every layer run as small tasks that read and write a few
 * tiles. This is the mechanism the NNTile review page (pith.science, "The
 * reading", section "What carries the argument") describes: embedding, linear,
 * layer norm, softmax, attention, cross-entropy and Adam written tile-wise, so
 * the training loop is one graph of tile tasks. The GPT2 example interface
 * (model config, tile sizes per axis, token ids, optimizer flags) follows the
 * NNTile README (skillagent.dev "NNTile"), section "Minimal working GPT
 * example".
 *
 * Conventions used by every function below:
 *   - Return value: NNT_OK or an error code; nnt_last_error() gives a message.
 *     After any error the model handle stays valid and destroyable.
 *   - Pointers named *_dev are CUDA device pointers (e.g. torch tensors'
 *     data_ptr()); pointers named *_host are host memory. The caller owns every
 *     buffer it passes; the library never frees caller memory and keeps no
 *     pointer to it after the call returns (device work on caller buffers is
 *     ordered on the model's stream).
 *   - Weight matrices are row-major [out, in]; activations are token-major
 *     [batch, seq, features].
 *   - Token windows are uint16 [batch, seq + 1] (the nanoGPT-style uint16 token
 *     stream of the README's "Minimal working GPT example"): inputs are
 *     columns 0..seq-1, next-token targets columns 1..seq.
 *   - A model issues its work on one CUDA stream (nnt_options.stream; when that
 *     is NULL, a blocking stream the model creates and destroys, which the
 *     legacy default stream orders against) plus library-owned side streams
 *     that are joined back into it before each call returns. The stand-alone
 *     tile tasks (nnt_op_*) run on the stream they are given.
 *   - Environment (for measurement; the defaults choose per shape):
 *     NNT_GEMM_BN=64|128|192|256 forces the width of the tensor-core GEMM's
 *     128 x BN output tiles; NNT_CE_KERNEL=pair|twopass forces the
 *     cross-entropy kernel (the two-CTA-cluster kernel holds rows of up to
 *     55296 logits in shared memory; the two-pass kernel takes any row).
 */
#ifndef NNT_H
#define NNT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NNT_OK = 0,
  NNT_ERR_INVALID_ARG = 1, /* bad size, tile size, pointer or token id */
  NNT_ERR_OOM = 2,         /* device or pinned-host allocation failed */
  NNT_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  NNT_ERR_TIMEOUT = 4,     /* a bounded wait ran out (host wait or device spin) */
  NNT_ERR_STATE = 5,       /* call out of order (e.g. backward before forward) */
  NNT_ERR_INTERNAL = 6
} nnt_status;

/* Compute dtype of activations and GEMM operands. Master weights, gradients and
 * AdamW moments are always fp32. NNT_F32 runs fp32 GEMMs on CUDA cores
 * (the NNTile experiments used TF32/fp32, review page "Circularity Check");
 * NNT_BF16 runs bf16 tensor-core GEMMs with fp32 accumulation. */
typedef enum { NNT_F32 = 0, NNT_BF16 = 1 } nnt_dtype;

/* GPT2 shape (README "Minimal working GPT example": --config-path JSON). The
 * sequence length is n_ctx; batch is the number of sequences per step
 * (--minibatch). ln_eps <= 0 selects 1e-5. */
typedef struct {
  int32_t n_layer, d_model, n_head, d_ff, vocab, n_ctx, batch;
  int32_t dtype; /* nnt_dtype */
  float ln_eps;
} nnt_gpt2_config;

/* Tile sizes per axis, 0 = whole axis (README flags --minibatch-tile,
 * --seq-tile, --embd-tile, --inner-tile, --head-tile). n_ctx must be divisible
 * by seq_tile, n_head by head_tile and batch by batch_tile; embd_tile,
 * inner_tile and vocab_tile need not divide their axes (ragged last tile), as
 * the same README section states for --embd-tile and --inner-tile. */
typedef struct {
  int32_t batch_tile, seq_tile, embd_tile, inner_tile, head_tile, vocab_tile;
} nnt_tiles;

/* Library options. Zero-initialised options are valid defaults. */
typedef struct {
  void* stream;                /* cudaStream_t the step runs on (NULL = a stream of the model's own) */
  uint64_t hbm_budget_bytes;   /* device bytes the model may use; 0 = free memory - 2 GiB */
  int32_t allow_host_offload;  /* 1: tiles that do not fit go to pinned host RAM */
  uint64_t init_seed;          /* weights drawn on the device from this seed ... */
  float init_std;              /* ... as N(0, init_std^2) (0 selects 0.02); LN g=1, b=0 */
  int32_t init_zero_bias;      /* 1: linear biases start at 0 instead of N(0, std^2) */
  int32_t n_streams;           /* streams the tile executor may use (0 = 2, max 8) */
  int32_t use_cuda_graph;      /* 1: capture each phase once and replay it */
  uint32_t timeout_ms;         /* bound on every host wait (0 = 600000) */
  int32_t gemm_backend;        /* 0 = tensor cores (bf16) / CUDA cores (fp32); 1 = CUDA-core GEMM always */
  int32_t trace;               /* 1: time every task with CUDA events (nnt_get_task_times) */
  int32_t gemm_min_task_cols;  /* consecutive output column tiles share one GEMM launch until it
                                  is this wide (0 = 8192; negative = one launch per tile) */
  int32_t flash_attention;     /* README --flashattention: fused attention tile tasks that keep
                                  the scores on chip (no [B,H,S,S] buffers). 0 = on when usable
                                  (bf16, tensor-core GEMMs, head size 64 or 128), 1 = required
                                  (INVALID_ARG when not usable), -1 = off (materialised scores,
                                  softmax and P V as separate tasks) */
  uint64_t host_budget_bytes;  /* pinned host bytes the model may take (offloaded AdamW moments);
                                  0 = the host's available memory - 8 GiB */
} nnt_options;

/* AdamW hyper-parameters (README: --optimizer=fusedadamw, --optimizer-eps=1e-8,
 * --weight-decay=0.1, --lr=3e-4; decoupled weight decay per the pages' reference
 * "Decoupled Weight Decay Regularization"). Betas are not on the pages: 0.9 and
 * 0.999 are used by the tests.
 * Warm-up (README: --start-lr, --full-lr-iter): AdamW iteration t (1-based,
 * counted by the model) uses start_lr at t = 1, lr from t = full_lr_iter on,
 * and the straight line between them in between (the pages give the two end
 * points only). full_lr_iter <= 1 (e.g. a zero-initialised struct) applies lr
 * from the first iteration. INVALID_ARG for a negative rate, weight decay or
 * full_lr_iter, eps <= 0, or a beta outside [0, 1). */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
  float start_lr;       /* rate of iteration 1 when full_lr_iter > 1 */
  int32_t full_lr_iter; /* first iteration at the full rate lr */
} nnt_adamw;

typedef struct nnt_model nnt_model;

typedef struct {
  double last_forward_ms, last_backward_ms, last_adamw_ms; /* host wall time of the last calls */
  uint64_t device_bytes;        /* bytes allocated on the device by this model */
  uint64_t host_pinned_bytes;   /* bytes in pinned host RAM (offloaded tiles) */
  uint64_t h2d_bytes, d2h_bytes;/* cumulative host<->device moment traffic of offloaded chunks */
  int64_t n_tasks_forward, n_tasks_backward, n_tasks_adamw;
  int64_t n_tiles;
  int64_t n_params;             /* scalar parameter count */
  int32_t n_streams;
  int32_t offload_active;
  int64_t kernels_forward, kernels_backward, kernels_adamw; /* kernel launches per call */
  int32_t flash_attention;      /* 1 when the fused attention tasks are in use */
} nnt_stats;

/* ---------------------------------------------------------------- model API */

/* Validate the shape and tiles, allocate every tile (device, or pinned host for
 * offloaded ones), draw the weights from opts->init_seed on the device, build
 * the static task graph of the step and its stream schedule.
 * Errors: INVALID_ARG if n_ctx % seq_tile, n_head % head_tile,
 * batch % batch_tile or d_model % n_head is non-zero, if d_model, d_ff or the
 * head size is not a multiple of 8 (bf16: head size a multiple of 16), if vocab
 * > 65536, or if batch*n_ctx > 1048576; OOM if the allocation plan (see
 * nnt_plan_memory) needs more device memory than is free, or more pinned host
 * memory than host_budget_bytes -- checked before anything is allocated.
 * *out is NULL on error. */
nnt_status nnt_create_model(const nnt_gpt2_config* cfg, const nnt_tiles* tiles,
                            const nnt_options* opts, nnt_model** out);

/* Device and pinned-host bytes nnt_create_model would allocate for this
 * configuration, from the same allocation plan (host offload of AdamW moments
 * included), without allocating anything. With opts->hbm_budget_bytes set no
 * CUDA call is made; with 0 the plan starts from the current device's free
 * memory (needs a device). Errors: as nnt_create_model's argument checks. */
nnt_status nnt_plan_memory(const nnt_gpt2_config* cfg, const nnt_tiles* tiles,
                           const nnt_options* opts, uint64_t* device_bytes,
                           uint64_t* host_pinned_bytes);

/* Forward pass and mean next-token cross-entropy (README --loss-reduction=mean).
 * tokens: uint16 [batch][n_ctx + 1], in host memory (tokens_on_device = 0,
 * copied in on the model's stream) or device memory (1). loss_out (host, may be
 * NULL) receives the loss; the call waits for it with the timeout bound.
 * Token ids >= vocab are reported as INVALID_ARG (checked on the device). */
nnt_status nnt_forward(nnt_model* m, const uint16_t* tokens, int32_t tokens_on_device,
                       float* loss_out);

/* Backward pass of the last forward: fp32 gradients of every parameter
 * (overwritten, not accumulated). STATE error if no forward preceded it, or if
 * the model offloads AdamW moments (use nnt_backward_adamw). */
nnt_status nnt_backward(nnt_model* m);

/* Gradient accumulation over minibatches (README: --batch sequences per
 * optimizer step, processed --minibatch at a time; the step happens once the
 * whole batch's gradients are collected). Backward pass of the last forward
 * whose gradients are ADDED to those stored since the last AdamW update; the
 * first call after an update (or after nnt_backward's overwrite) starts the
 * sum. nnt_adamw_step then uses the mean of the k summed minibatch gradients,
 * which for minibatches of equal token count is the gradient of the mean loss
 * over the whole batch. Call pattern for a batch of k minibatches:
 * k x (nnt_forward, nnt_backward_accumulate), then nnt_adamw_step. Same
 * STATE rules as nnt_backward; a failed call leaves the sum undefined, so the
 * next call starts a new one. */
nnt_status nnt_backward_accumulate(nnt_model* m);

/* One fused AdamW update of every parameter tile from the current gradients
 * (their mean over the minibatches accumulated since the last update); the
 * step counter starts at 1 and grows by one per call. STATE error if no
 * backward preceded it since the last update. */
nnt_status nnt_adamw_step(nnt_model* m, const nnt_adamw* hp);

/* Backward pass fused with AdamW: each parameter chunk is updated as soon as
 * its gradient is final and every task of this pass that reads its old value
 * has been issued, so AdamW overlaps the rest of the backward (the update is
 * the same as nnt_backward + nnt_adamw_step). Required for models whose AdamW
 * moments are offloaded to pinned host memory (nnt_options.allow_host_offload
 * when the state does not fit the device budget): there, gradients of the
 * layer matrices only pass through a small ring of device slots and cannot be
 * read back, and the AdamW kernel updates the moments of host-resident chunks
 * in place in pinned, device-mapped host memory (over NVLink-C2C on GB300).
 * Same STATE/INVALID_ARG rules as nnt_backward / nnt_adamw_step. */
nnt_status nnt_backward_adamw(nnt_model* m, const nnt_adamw* hp);
/* (nnt_backward_adamw does not add to accumulated gradients: STATE error while
 * minibatch gradients are pending an nnt_adamw_step.) */

/* Free everything the model owns. NULL-safe; always succeeds. */
void nnt_destroy(nnt_model* m);

/* ------------------------------------------------ parity / checkpoint surface */

/* Number of named parameter tensors, in the fixed order: wte, wpe, then per
 * layer ln1.g ln1.b qkv.w qkv.b o.w o.b ln2.g ln2.b fc.w fc.b proj.w proj.b,
 * then ln_f.g ln_f.b. Returns -1 for NULL. */
int32_t nnt_num_params(const nnt_model* m);

/* Name (static storage owned by the model) and shape (shape[1] = 0 for
 * vectors) of parameter i. */
nnt_status nnt_param_info(const nnt_model* m, int32_t i, const char** name, int64_t shape[2]);

/* Copy parameter i (fp32 master), its gradient, or an AdamW moment
 * (which = 0: m, 1: v) to/from a host fp32 buffer of shape[0]*max(shape[1],1)
 * elements. nnt_set_param also refreshes the bf16 copy. Synchronous. */
nnt_status nnt_get_param(nnt_model* m, int32_t i, float* host_buf);
nnt_status nnt_set_param(nnt_model* m, int32_t i, const float* host_buf);
nnt_status nnt_get_grad(nnt_model* m, int32_t i, float* host_buf);
nnt_status nnt_get_adam_state(nnt_model* m, int32_t i, int32_t which, float* host_buf);

/* Copy the logits of the last forward to host: fp32 [batch][n_ctx][vocab]. */
nnt_status nnt_get_logits(nnt_model* m, float* host_buf);

nnt_status nnt_get_stats(const nnt_model* m, nnt_stats* out);

/* Per-task-type timing of the last traced call (opts.trace = 1): for task type
 * k < n, name[k], launches[k] and total device milliseconds[k] (CUDA events on
 * the stream each task ran on), flops[k] and bytes[k] (algorithmic work).
 * Returns the number of task types, or -1. */
int32_t nnt_get_task_times(const nnt_model* m, int32_t max_types, const char** names,
                           int64_t* launches, double* ms, double* flops, double* bytes);

/* Switch per-task CUDA-event timing on (1) or off (0) for the following calls.
 * While tracing, the tasks run in program order on one stream (in a separate
 * captured graph when graphs are enabled), so each task's time is its own. */
nnt_status nnt_set_trace(nnt_model* m, int32_t on);

/* Last error message of this model (or of the calling thread when m is NULL). */
const char* nnt_last_error(const nnt_model* m);

/* ------------------------------------------------------ executor schedule
 *
 * The executor's plan for a task graph given only by its tile accesses, as the
 * model's own programs get it: tasks are submitted in program order, each
 * declaring the tiles it reads and writes, and the dependencies follow from
 * those accesses (review page "The reading" / "What carries the argument";
 * first page, abstract: a sequential task flow whose runtime infers the
 * dependencies). Host only: no device work and no CUDA call, so it runs without
 * a GPU; it exposes the scheduler for inspection and tests.
 *
 * Tasks are 0..n_tasks-1 in program order. Task i's accesses are entries
 * use_off[i] .. use_off[i+1]-1 (use_off has n_tasks + 1 entries, use_off[0] = 0,
 * non-decreasing) of use_tile (any int64 tile id) and use_mode (1 read,
 * 2 write, 3 read and write). copy_task (NULL = none) marks host<->device copy
 * tasks, which run on one extra copy stream; stream_hint (NULL = none) pins a
 * task to a compute stream (>= 0, clamped to n_streams - 1) or leaves it to the
 * scheduler (-1). n_streams >= 1 compute streams.
 *
 * Outputs (caller-owned, n_tasks entries unless stated): stream_out[i] in
 * 0..n_streams-1, or n_streams for the copy stream; task i's direct
 * dependencies are dep_task[dep_off[i] .. dep_off[i+1]-1] (the last writer of
 * each tile it uses, and for a tile it writes the readers since that writer;
 * ascending), and the tasks it waits for on other streams (one event wait
 * each; dependencies already implied by stream order or by earlier waits are
 * left out) are wait_task[wait_off[i] .. wait_off[i+1]-1]. dep_off and wait_off
 * have n_tasks + 1 entries. dep_cap and wait_cap are the capacities of dep_task
 * and wait_task: when one is too small the call fills both offset arrays,
 * writes nothing else and returns INVALID_ARG, so the caller can size the
 * arrays from dep_off[n_tasks] and wait_off[n_tasks] and call again. Also
 * INVALID_ARG on n_tasks < 0, n_streams < 1, a NULL required array, bad
 * offsets or a mode outside 1..3. */
nnt_status nnt_plan_schedule(int32_t n_tasks, const int64_t* use_off, const int64_t* use_tile,
                             const int32_t* use_mode, const int32_t* copy_task,
                             const int32_t* stream_hint, int32_t n_streams, int32_t* stream_out,
                             int64_t* dep_off, int32_t* dep_task, int64_t dep_cap,
                             int64_t* wait_off, int32_t* wait_task, int64_t wait_cap);

/* ------------------------------------------------------ single tile tasks
 *
 * The step's tile kernels as stand-alone calls on caller device buffers, used
 * by the kernel tests and the kernel sweep. All pointers are device pointers,
 * all matrices row-major with the given leading dimension (elements), `stream`
 * is a cudaStream_t (NULL = legacy default). dtype selects fp32 (NNT_F32) or
 * bf16 (NNT_BF16) for the arguments documented as "act". The calls only
 * enqueue work; they do not synchronise. INVALID_ARG on bad sizes or NULL
 * pointers; CUDA on a launch failure.
 */

/* Layer normalisation over each row (reference "Layer Normalization";
 * review page "What carries the argument" lists layer norm among the tile
 * tasks): y = g * (x - mean)/sqrt(var + eps) + b with biased variance.
 * x fp32 [rows, cols]; y act [rows, cols]; mean, rstd fp32 [rows]. */
nnt_status nnt_op_layernorm_fwd(const float* x_dev, const float* g_dev, const float* b_dev,
                                void* y_dev, float* mean_dev, float* rstd_dev,
                                int64_t rows, int64_t cols, float eps, int32_t dtype,
                                void* stream);

/* Layer-norm backward: dx = rstd*(gdy - mean(gdy) - xhat*mean(gdy*xhat)) with
 * gdy = g*dy, added to resid_dev when not NULL (dx_dev = resid + that); also
 * writes an act copy of dx to dx_act_dev when not NULL; dg = sum_rows dy*xhat
 * and db = sum_rows dy (fp32 [cols], overwritten). All row data fp32. */
nnt_status nnt_op_layernorm_bwd(const float* dy_dev, const float* x_dev, const float* mean_dev,
                                const float* rstd_dev, const float* g_dev, const float* resid_dev,
                                float* dx_dev, void* dx_act_dev, float* dg_dev, float* db_dev,
                                int64_t rows, int64_t cols, int32_t dtype, void* stream);

/* Causal softmax over the last axis of nmat square [seq, seq] fp32 score
 * matrices (entry (q, k) with k > q masked to probability 0): P act. Only
 * columns k < ceil((q+1)/128)*128 of row q are read or written; columns beyond
 * q among them are written as 0. */
nnt_status nnt_op_softmax_causal_fwd(const float* s_dev, void* p_dev, int64_t nmat, int64_t seq,
                                     int32_t dtype, void* stream);

/* Softmax backward: dS = scale * P * (dP - rowsum(dP * P)); P act, dP fp32,
 * dS act; same causal column range as the forward. */
nnt_status nnt_op_softmax_causal_bwd(const void* p_dev, const float* dp_dev, void* ds_dev,
                                     int64_t nmat, int64_t seq, float scale, int32_t dtype,
                                     void* stream);

/* Fused causal attention (the README's --flashattention option; the pages
 * list it as a memory-saving flag whose kernel NNTile does not have yet):
 * O = softmax_causal(Q K^T / sqrt(hd)) V without materialising the scores.
 * q, k, v, o: bf16 [Z][S][hd] device buffers (Z = sequences x heads, rows of
 * one (sequence, head) contiguous, 16-byte aligned); lse: fp32 [Z][S], the
 * base-2 log-sum-exp of each row's scaled scores, so that the probabilities
 * are 2^(s * log2(e) / sqrt(hd) - lse) (saved for the backward). hd must be 64
 * or 128 (INVALID_ARG otherwise); any S >= 1. Scores and P are bf16 MMA
 * operands with fp32 accumulation, P rounded to bf16 before P V. Runs on
 * `stream`; the library keeps no reference to the buffers. A bounded wait
 * that runs out is reported through nnt_op_read_error. */
nnt_status nnt_op_flash_attention_fwd(const void* q_dev, const void* k_dev, const void* v_dev,
                                      void* o_dev, float* lse_dev, int64_t Z, int64_t S,
                                      int64_t hd, void* stream);

/* Backward of nnt_op_flash_attention_fwd: dq, dk, dv (bf16 [Z][S][hd],
 * overwritten) from q, k, v, the forward's o and lse, and do = dL/dO (bf16
 * [Z][S][hd]). P is recomputed from lse; D = rowsum(do * o) goes to a
 * library-owned scratch buffer (grown with cudaMalloc when too small). Sums run
 * in a fixed order (no atomics): same inputs, same bits. */
nnt_status nnt_op_flash_attention_bwd(const void* q_dev, const void* k_dev, const void* v_dev,
                                      const void* o_dev, const void* do_dev, const float* lse_dev,
                                      void* dq_dev, void* dk_dev, void* dv_dev, int64_t Z,
                                      int64_t S, int64_t hd, void* stream);

/* tanh-form GELU over n elements: g = gelu(u) (u fp32, g act) and its
 * backward du = dg * gelu'(u) (dg act, du act). */
nnt_status nnt_op_gelu_fwd(const float* u_dev, void* g_dev, int64_t n, int32_t dtype, void* stream);
nnt_status nnt_op_gelu_bwd(const void* dg_dev, const float* u_dev, void* du_dev, int64_t n,
                           int32_t dtype, void* stream);

/* Mean cross-entropy over rows of logits z (fp32 [rows, ldz], first `cols`
 * columns valid; README --loss-reduction=mean) with uint16 targets
 * (tgt_dev[r * tgt_stride]) and its gradient dz = (softmax(z) - onehot)/rows
 * written as act [rows, lddz] (columns cols..lddz-1 written as 0). loss_dev: one
 * fp32 (the mean). row_loss_dev: fp32 [rows] scratch for per-row losses.
 * ldz and lddz are multiples of 4 and at least cols (INVALID_ARG otherwise);
 * a target >= cols sets the device error word (nnt_op_read_error). */
nnt_status nnt_op_cross_entropy(const float* z_dev, int64_t rows, int64_t cols, int64_t ldz,
                                const uint16_t* tgt_dev, int64_t tgt_stride, void* dz_dev,
                                int64_t lddz, float* row_loss_dev, float* loss_dev,
                                int32_t dtype, void* stream);

/* Fused AdamW over n fp32 elements (decoupled weight decay): updates w, m, v in
 * place from g, writes a bf16 copy of the new w to w_bf16_dev when not NULL.
 * bc1 = 1 - beta1^t and bc2 = 1 - beta2^t are the bias corrections. */
nnt_status nnt_op_adamw(float* w_dev, const float* g_dev, float* m_dev, float* v_dev,
                        void* w_bf16_dev, int64_t n, float lr, float beta1, float beta2,
                        float eps, float weight_decay, float bc1, float bc2, void* stream);

/* Embedding gather: x[b,s,:] = wte[ids[b*ids_stride + s], :] + wpe[s, :]
 * (fp32 [batch, seq, d]). */
nnt_status nnt_op_embedding_fwd(const uint16_t* ids_dev, int64_t ids_stride, const float* wte_dev,
                                const float* wpe_dev, float* x_dev, int64_t batch, int64_t seq,
                                int64_t d, int64_t vocab, void* stream);

/* Embedding scatter-add, deterministic: dwte[ids[t]] += dx[t] for token
 * t = b*seq + s in increasing t order, dwpe[s] += dx[b, s] in increasing b
 * order (fp32). Needs batch*seq <= 1048576; uses library scratch of
 * 4*batch*seq bytes (allocated once per device and grown on demand). */
nnt_status nnt_op_embedding_bwd(const uint16_t* ids_dev, int64_t ids_stride, const float* dx_dev,
                                float* dwte_dev, float* dwpe_dev, int64_t batch, int64_t seq,
                                int64_t d, int64_t vocab, void* stream);

/* Same as nnt_op_embedding_bwd (same results, bit for bit), but it allocates
 * nothing. It is meant for callers that cannot allocate device memory while
 * they run: hosts that own all device memory through their own allocator or a
 * fixed budget (a library allocation would bypass it, or fail), and loops that
 * cannot afford the implicit device synchronisation of an allocation. The
 * NNTile pages have no counterpart of this call; it only changes where the
 * scratch lives.
 * Scratch: one fixed array of 16384 uint32 sort keys (64 KiB) compiled into
 * the library, present on every device that loads it until the process exits;
 * so batch*seq must be <= 16384 (INVALID_ARG otherwise, before any work).
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Every call uses the same array: calls whose GPU
 * work overlaps (different streams, no ordering between them) race and give
 * wrong results. Calls never free or allocate anything. */
nnt_status nnt_op_embedding_bwd_noalloc(const uint16_t* ids_dev, int64_t ids_stride,
                                        const float* dx_dev, float* dwte_dev, float* dwpe_dev,
                                        int64_t batch, int64_t seq, int64_t d, int64_t vocab,
                                        void* stream);

/* Tile GEMM C = alpha * op(A) op(B) (+ beta * C): op(A) is [M, K], op(B) is
 * [K, N]. a_trans = 0: A stored [M][lda] (K contiguous); 1: A stored [K][lda]
 * (M contiguous). b_trans = 0: B stored [N][ldb] (K contiguous, i.e. a weight
 * [out, in] giving x W^T); 1: B stored [K][ldb] (N contiguous). A, B act
 * (dtype); C fp32 (c_dtype NNT_F32) or act; beta is 0 or 1 (fp32 C only).
 * backend 0 = tensor cores for bf16, 1 = CUDA cores. Requires lda, ldb
 * multiples of 8 and 16-byte aligned A, B for bf16 tensor cores. */
nnt_status nnt_op_gemm(const void* a_dev, int64_t lda, int32_t a_trans, const void* b_dev,
                       int64_t ldb, int32_t b_trans, void* c_dev, int64_t ldc, int32_t c_dtype,
                       int64_t M, int64_t N, int64_t K, float alpha, float beta, int32_t dtype,
                       int32_t backend, void* stream);

/* Device error word of the kernels (bad token ids, exhausted bounded waits):
 * read and clear. 0 = none. */
nnt_status nnt_op_read_error(uint32_t* code_out, void* stream);

/* ---- failure detection (tests) ----------------------------------------
 * Host-side fault injection, off by default: after
 * nnt_set_fault_injection(kind, n) the n-th call of that kind from now on
 * fails the way the real failure would, without any GPU work failing:
 *   NNT_FAULT_DEVICE_ALLOC  a device allocation of nnt_create_model -> NNT_ERR_OOM
 *   NNT_FAULT_HOST_ALLOC    a pinned host allocation (loss word, offloaded
 *                           AdamW moments) -> NNT_ERR_OOM
 *   NNT_FAULT_COPY          an async copy submission of the model API (token
 *                           upload, loss read-back, parameter/gradient/state
 *                           copies) -> NNT_ERR_CUDA, the copy not issued
 *   NNT_FAULT_EVENT_WAIT    a host wait for the model's stream -> NNT_ERR_TIMEOUT
 *                           (the device work itself still completes)
 * n = 0 disarms. Calls of other kinds are not counted. After an injected
 * failure the model (if created) stays valid and destroyable; nnt_create_model
 * frees everything it had allocated and sets *out to NULL.
 * Thread-safe; the counters are process-wide. */
typedef enum {
  NNT_FAULT_DEVICE_ALLOC = 0,
  NNT_FAULT_HOST_ALLOC = 1,
  NNT_FAULT_COPY = 2,
  NNT_FAULT_EVENT_WAIT = 3
} nnt_fault_kind;
nnt_status nnt_set_fault_injection(int32_t kind, int64_t nth);

/* Bounded device wait, self-test: one CTA waits on an mbarrier phase that
 * nothing completes (arrive = 0) or that its own thread completes first
 * (arrive = 1), giving up after limit_ns nanoseconds of %globaltimer (1 us ..
 * 1 s, INVALID_ARG otherwise). On giving up it ORs the wait-timeout bit (2)
 * into the device error word (nnt_op_read_error) and returns; the GPU context
 * stays usable. The same bounded wait guards every mbarrier wait of the
 * tensor-core kernels (their limit: 5 s). */
nnt_status nnt_op_wait_selftest(int64_t limit_ns, int32_t arrive, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NNT_H */
