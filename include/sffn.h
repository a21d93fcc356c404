/*
 * sffn.h -- C ABI of the predictor-gated, activation-sparse FFN decode library
 * (libsffn.so, CUDA kernels for sm_103a).
 *
 * What it computes.  For one decode token x (or a small batch of tokens), a
 * per-layer online predictor scores every FFN neuron, the neurons predicted
 * active are compacted into an ascending index list, and only their rows of
 * W_up (and W_gate for ReGLU) and of W_down^T are read and accumulated:
 *
 *   h      = V x                                   (predictor hidden layer)
 *   s_i    = U_i . h + pb_i ;  i active  <=>  s_i > tau   (strict)
 *   a_i    = max(0, W_up[i] . x + b_i)                       (ReLU)
 *          = max(0, W_gate[i] . x + b_i) * (W_up[i] . x)      (ReGLU)
 *   y      = sum over active i, of a_i * W_down^T[i, :]
 *
 * Sources (the pages on PowerInfer and activation sparsity):
 *   - predict-then-skip: "Predictores de espacialidad adaptativa" of the
 *     PowerInfer page (unite.ai) and the adaptive sparse predictor of the
 *     sparsity page (blogs.novita.ai, section 在線推理);
 *   - neuron table (index list -> matrix row): PowerInfer page, "Colocacion y
 *     gestion de neuronas";
 *   - row/column neuron-aware operators: PowerInfer page, "Operador consciente
 *     de neuronas"; skipped rows contribute zero: sparsity page, opening
 *     section on ReLU activation sparsity;
 *   - coalesced, fused kernels: sparsity page, section 工程影響.
 * The predictor's low-rank linear form and the row layouts below are this
 * library's reading; the pages give no formula.
 *
 * Conventions shared by every entry point.
 *   - Device pointers are borrowed, never freed, and must stay valid until the
 *     work queued on `stream` has finished.  The library allocates no device
 *     memory of its own: every call takes a caller-owned `workspace`.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  All device work is queued asynchronously on it; no entry point
 *     synchronises except sffn_read_device_status.
 *   - Layouts are row-major with one row per neuron:
 *       W_up, W_gate, W_down^T : [d_ff][d_model]   (dtype)
 *       U : [d_ff][rank] (dtype),  V : [rank][d_model] (dtype)
 *       b, pb : [d_ff] float32
 *       x : [batch][d_model] (dtype),  y : [batch][d_model] float32
 *     W_down^T is the down projection stored transposed, so the output row of
 *     neuron i is contiguous.  Every matrix row, x row and y row must start on
 *     a 16-byte boundary: base pointers 16-byte aligned and d_model * sizeof
 *     (dtype) and rank * sizeof(dtype) multiples of 16.
 *   - Index lists are in the stored (possibly hot-first permuted) neuron order.
 *   - Return values report argument validation and launch errors.  Conditions
 *     found on the device (a bounded wait that timed out, a capacity limit) are
 *     recorded in a status word inside the workspace and read with
 *     sffn_read_device_status.  Kernels never trap.
 *   - The workspace must be zero-filled once before its first use
 *     (sffn_workspace_init does it); every call leaves it reusable, except
 *     after a device status of SFFN_ERR_TIMEOUT, when it must be zero-filled
 *     again.  Two calls that share a workspace must be ordered (same stream,
 *     or synchronised): calls that overlap on the GPU race.
 */
#ifndef SFFN_H
#define SFFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SFFN_OK = 0,
  SFFN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, mismatch  */
  SFFN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. dtype)       */
  SFFN_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed         */
  SFFN_ERR_CAPACITY = 4,     /* device: a list outgrew its buffer            */
  SFFN_ERR_TIMEOUT = 5,      /* device: a bounded wait ran out               */
  SFFN_ERR_WORKSPACE = 6     /* workspace null, misaligned or too small      */
} sffn_status;

typedef enum { SFFN_F32 = 0, SFFN_F16 = 1, SFFN_BF16 = 2 } sffn_dtype;
typedef enum { SFFN_RELU = 0, SFFN_REGLU = 1 } sffn_act;

typedef struct sffn_layer* sffn_layer_t;

/* One FFN layer and its predictor.  All pointers are device pointers. */
typedef struct {
  int32_t d_model;      /* model width d                                    */
  int32_t d_ff;         /* FFN width (number of neurons)                    */
  int32_t rank;         /* predictor rank r (rows of V, columns of U)       */
  int32_t max_batch;    /* largest batch later calls may pass (1..32)       */
  int32_t dtype;        /* sffn_dtype of weights, U, V and x               */
  int32_t act;          /* sffn_act                                         */
  const void* w_up;     /* [d_ff][d_model]                                  */
  const void* w_gate;   /* [d_ff][d_model], ReGLU only, else NULL           */
  const void* w_downT;  /* [d_ff][d_model]                                  */
  const float* b;       /* [d_ff] bias of the gated pre-activation; NULL=0  */
  const void* pred_U;   /* [d_ff][rank]                                     */
  const void* pred_V;   /* [rank][d_model]                                  */
  const float* pred_b;  /* [d_ff] predictor bias                            */
  float tau;            /* threshold: neuron i is active iff s_i > tau      */
  int32_t flags;        /* SFFN_FLAG_* bits, 0 for the defaults            */
  int32_t hot_rows;     /* neurons [0, hot_rows) are "hot": under a hot-first
                           order (sffn_hot_first_perm) the neurons active for
                           nearly every token.  Their rows may be fetched
                           before the predictor has decided; results do not
                           depend on it (only the predicted set is used).
                           0 = no such prefetch.                            */
  float expected_active; /* expected number of predicted-active neurons per
                           token (e.g. from the profile counts), 0 = unknown;
                           a hint for how much work to start before the
                           active rows are balanced over the SMs.           */
  int32_t warm_rows;    /* neurons [0, warm_rows) are likely active (e.g. the
                           hot-first rows active for >= 20% of profile tokens):
                           the batch-1 kernel pulls their rows into L2 while
                           the predictor runs, when DRAM is otherwise idle.
                           Speculative: rows that turn out inactive cost DRAM
                           bandwidth only; results do not depend on it.
                           0 = none; must be in [0, d_ff].                  */
  int32_t dense_min_batch; /* dense fallback: calls of at least this many
                           tokens (2..32; 16-bit weights) read EVERY row once,
                           as two tensor-core GEMMs (cuBLASLt, fp32
                           accumulation) with each token's predicted mask and
                           the activation applied between them, instead of
                           gathering the union of the tokens' active rows.
                           Worth it once that union covers most of the layer
                           (the sparsity page, section 工程影響: the benefit of
                           sparsity decays with the batch; PowerInfer-2 page,
                           4.1.1: low-sparsity prefill runs every neuron as one
                           dense cluster).  Results are the masked FFN either
                           way.  The union is only known on the device after
                           the predictor, so the switch is by batch size; the
                           benchmark measures the crossover.  The workspace
                           grows by the GEMMs' buffers and a 16 MiB cuBLASLt
                           workspace.  0 = never.                            */
} sffn_layer_desc;

/* Batch-1 calls normally run the whole layer (predictor, threshold, gather,
 * activation, down projection) as one kernel launch; this flag selects the
 * multi-kernel path (separate predictor, score and gather kernels) that larger
 * batches use, with its deterministic cross-block reduction. */
#define SFFN_FLAG_MULTI_KERNEL 1
/* Batch-1 kernel: after the predictor, even out the token's active rows over
 * the SMs (each block publishes its count and list; every block computes the
 * same assignment, keeping its own rows up to its share and taking the surplus
 * of others).  Costs about four global round trips; pays off when the uneven
 * split of active rows costs more (wide rows, many rows per SM).  Needs d_ff
 * of at least 8 rows per block and a grid of at most 256 blocks (layers that
 * run two blocks per SM use 2 x the SM count), otherwise ignored. */
#define SFFN_FLAG_BALANCE 2
/* Batches of 3 to 32 tokens with fp16/bf16 weights (d_model a multiple of 128)
 * normally run on the tensor-core union path: the union of the tokens' active
 * rows is read once, both products are tcgen05 MMAs (the predictor's scores
 * too, when the rank is a multiple of 64), and y is accumulated with float atomics
 * (summation order varies from run to run).  With this flag such batches use
 * the CUDA-core predictor and row gather instead (passes of up to 4 tokens,
 * fixed-order reduction, bit-reproducible). */
#define SFFN_FLAG_ROW_GATHER 4
/* The layer's weights, biases and predictor matrices are static: no kernel
 * writes them while the layer exists (they were written, and the writes
 * synchronised, before the first call).  Batch-1 calls may start while the
 * previous kernel on the stream is still finishing (programmatic dependent
 * launch); with this flag they stage the weights they need first (V rows, U
 * rows, biases, hot rows) before waiting for that kernel, which saves about
 * 1 us per call on the OPT-6.7B layer.  Without it they only warm L2 with
 * them before the wait, so a kernel queued just before the call may still be
 * writing the weights (a reorder, a dequantisation). */
#define SFFN_FLAG_STATIC_WEIGHTS 8
/* Bundled rows: neuron i's rows of the FFN matrices are stored side by side
 * in one matrix, passed as w_up (w_gate and w_downT must be NULL):
 *   ReGLU: bundle[i] = [ W_gate[i] | W_up[i] | W_down^T[i] ]   ([d_ff][3*d_model])
 *   ReLU : bundle[i] = [ W_up[i] | W_down^T[i] ]               ([d_ff][2*d_model])
 * (sffn_bundle_rows builds it).  The rows a neuron needs are then one
 * contiguous stretch of memory, read as one stream: PowerInfer-2 page, 4.4
 * "Neuron-Cluster-Level Pipeline" (the i-th neurons of Gate, Up and Down
 * co-activate in up to 80% of cases, so they are stored together).  Results
 * are those of the unbundled layer. */
#define SFFN_FLAG_BUNDLED 16

/* Validates the descriptor and records it with launch settings chosen for the
 * current device.  Allocates only host memory.  Returns INVALID_ARG for bad
 * shapes or pointers, UNSUPPORTED for shapes outside the kernels' limits. */
sffn_status sffn_create_layer(const sffn_layer_desc* desc, sffn_layer_t* out);
sffn_status sffn_destroy_layer(sffn_layer_t layer);

/* Bytes of workspace a call with `batch` tokens needs (0 on bad arguments). */
size_t sffn_workspace_size(sffn_layer_t layer, int32_t batch);

/* How a layer's batch-1 calls run on its device, as chosen at creation (no
 * compute; for tuning and tests).  All fields are written; on error the
 * struct is untouched.  Errors: SFFN_ERR_INVALID_ARG for a NULL argument. */
typedef struct {
  int32_t fused;          /* 1: the single-launch layer kernel, 0: multi-kernel  */
  int32_t grid;           /* its blocks (0 when not fused)                       */
  int32_t blocks_per_sm;  /* 1 or 2                                              */
  int32_t cluster;        /* 2: pairs of blocks even out their rows, else 0      */
  int32_t ring_stages;    /* row stages per block                                */
  int32_t hot_stages;     /* of which filled before the predictor has decided    */
} sffn_layer_info;
sffn_status sffn_get_layer_info(sffn_layer_t layer, sffn_layer_info* info);

/* Zero-fills a workspace (cudaMemsetAsync on `stream`). */
sffn_status sffn_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Predictor + compaction (the online predictor and the neuron table).
 *   x        : [batch][d_model] dtype, device
 *   idx      : [batch][d_ff] int32, device; row t receives the ascending list
 *              of token t's active neurons in its first n_active[t] entries
 *   n_active : [batch] int32, device */
sffn_status sffn_predict(sffn_layer_t layer, const void* x, int32_t batch, int32_t* idx,
                         int32_t* n_active, void* workspace, size_t workspace_bytes,
                         void* stream);

/* No counterpart in the paper: a library convenience.
 *
 * The batch-1 sparse FFN (as sffn_forward with batch 1, no index outputs) for
 * callers that cannot allocate device memory: serving loops and embedded
 * runtimes that own all device memory up front in a fixed pool and forbid
 * cudaMalloc while running (it may synchronise the device, and it fragments a
 * pool sized to the byte), and programs whose device memory belongs to another
 * framework's allocator.  The caller passes x ([d_model], dtype, device) and
 * y ([d_model] float32, device); the kernel's scratch is a fixed 256 KiB array
 * inside the library, held on every device that loads the library until the
 * process exits.  Nothing here calls cudaMalloc or cudaFree.
 *   - Layers needing more scratch than that (a 256-byte header, 128 bytes per
 *     block of the single-launch kernel for its barrier words, and 128 bytes
 *     per predictor rank row for the tagged slots through which the blocks
 *     share the hidden layer h) are rejected with SFFN_ERR_UNSUPPORTED and a
 *     message giving both sizes; so are layers created with
 *     SFFN_FLAG_MULTI_KERNEL or outside the single-launch kernel's limits.
 *   - The layer's device must be current.  Every call looks up the array's
 *     device address there (cudaGetSymbolAddress); the first lookup on a
 *     device loads the library's kernels, so make the first call on each
 *     device before any stream capture.
 *   - Every call shares the one array and clears its counters first, so calls
 *     that overlap on the GPU (other streams, other threads) race; order them.
 *   - A device-side wait that ran out (SFFN_ERR_TIMEOUT: the kernel needs all
 *     its blocks resident at once, which kernels of other streams holding SMs
 *     can prevent; y is then incomplete) is recorded in the array's status
 *     word, which later calls keep; read and clear it with
 *     sffn_noalloc_read_status. */
sffn_status sffn_forward_noalloc(sffn_layer_t layer, const void* x, float* y, void* stream);

/* Status word of sffn_forward_noalloc's fixed array on the current device:
 * synchronises `stream`, copies the first device-side error since the last
 * read to *status (an sffn_status value, SFFN_OK if none) and clears it.
 * No counterpart in the paper; allocates nothing. */
sffn_status sffn_noalloc_read_status(int32_t* status, void* stream);

/* Predictor scores s = U (V x) + pb as float32 [batch][d_ff] (diagnostics:
 * the same kernels as sffn_predict, scores written out). */
sffn_status sffn_predict_scores(sffn_layer_t layer, const void* x, int32_t batch, float* scores,
                                void* workspace, size_t workspace_bytes, void* stream);

/* The sparse FFN for a batch of decode tokens: predict, compact, gather the
 * active rows, apply ReLU / ReGLU, accumulate the down projection.
 *
 * Batch-1 calls on the single-launch kernel (and sffn_forward_stack at batch
 * 1, and sffn_forward_noalloc) need every block of their grid resident at
 * once: each block waits (bounded) for values all other blocks publish.
 * Layer creation checks that the grid fits an otherwise idle GPU; if kernels
 * of other streams or processes hold SMs while such a call runs, the resident
 * blocks can wait out the limit (sffn_set_wait_limit_ns): the call then leaves
 * SFFN_ERR_TIMEOUT in the status word and an incomplete y.  Check the status
 * (sffn_read_device_status) when the GPU is shared with concurrent work.
 * The same holds for the row-gather kernel (one grid barrier before its
 * fixed-order reduction) and, within a block only, for the union kernel.
 *
 *   y            : [batch][d_model] float32, device (overwritten)
 *   idx_out      : NULL or [batch][d_ff] int32 (as sffn_predict)
 *   n_active_out : NULL or [batch] int32
 * Each token uses its own predicted set; a batch reads the union of the rows
 * once.  Results do not depend on which other tokens share the batch beyond
 * floating-point summation order. */
sffn_status sffn_forward(sffn_layer_t layer, const void* x, int32_t batch, float* y,
                         int32_t* idx_out, int32_t* n_active_out, void* workspace,
                         size_t workspace_bytes, void* stream);

/* The no-skip FFN (every neuron computed, no predictor), same layouts as
 * sffn_forward: the dense contrast of the sparse path. */
sffn_status sffn_dense_forward(sffn_layer_t layer, const void* x, int32_t batch, float* y,
                               void* workspace, size_t workspace_bytes, void* stream);

/* x_out = round_dtype(LayerNorm(x + y) * gamma + beta) per token, biased
 * variance, float32 arithmetic; gamma/beta NULL mean 1 and 0.
 *   x, x_out : [batch][d_model] dtype;  y : [batch][d_model] float32 */
sffn_status sffn_residual_layernorm(const void* x, const float* y, int32_t batch,
                                    int32_t d_model, int32_t dtype, const float* gamma,
                                    const float* beta, float eps, void* x_out, void* stream);

/* Greedy-shaped decode through a stack of layers (equal d_model and dtype):
 * every step runs each layer's sparse FFN followed by residual + LayerNorm,
 * x_{l+1} = round(LN(x_l + y_l)), and the next step starts from the last
 * layer's output.
 *   x0         : [batch][d_model] dtype, first step's input
 *   x_out      : [n_steps][batch][d_model] dtype, last layer's output per step
 *   x_trace    : NULL or [n_steps][n_layers][batch][d_model] dtype, the input
 *                of every layer at every step
 *   mask_trace : NULL or [n_steps][n_layers][batch][Wmax] uint32, the mask
 *                words each layer call used (bit i%32 of word i/32: neuron i
 *                predicted active), Wmax = ceil(largest d_ff / 32); words past
 *                a narrower layer's ceil(d_ff/32) are zero
 *   y_trace    : NULL or [n_steps][n_layers][batch][d_model] float32, each
 *                layer call's sparse-FFN output (the y that the residual +
 *                LayerNorm consumed)
 *   ln_gamma, ln_beta : NULL or [d_model] float32 shared by all layers
 * The traces record what this run computed (not a recomputation), for checks
 * of every layer of a long decode; they cost extra writes and are meant for
 * tests and diagnostics. */
sffn_status sffn_forward_stack(const sffn_layer_t* layers, int32_t n_layers, const void* x0,
                               int32_t batch, int32_t n_steps, void* x_out, void* x_trace,
                               uint32_t* mask_trace, float* y_trace, const float* ln_gamma,
                               const float* ln_beta, float ln_eps, int32_t options,
                               void* workspace, size_t workspace_bytes, void* stream);

/* options of sffn_forward_stack.
 *
 * SFFN_STACK_LOOKAHEAD: look-ahead masks, the asynchronous sparsity predictor
 * of the DejaVu design (sparsity page, section "如何充分利用結構化稀疏性進行
 * 加速": the next layer's MLP sparsity is predicted ahead of time, so that
 * prediction overlaps the current layer's work).  Layer calls are numbered
 * across steps; call k > 0 uses the neurons that its layer's own predictor
 * (U, V, pb, tau) scores above tau on the INPUT OF CALL k - 1, and call 0 the
 * ones it scores on x0.  Each call's kernel reads its rows at once and, while
 * they stream in, evaluates the next layer's predictor on its own input.
 * This changes results: a neuron whose score crosses tau between the two
 * inputs is decided differently than by the exact predictor (the benchmark
 * reports the recall and precision of these masks against the exact ones).
 * Requires batch 1 and layers of equal shape and launch configuration (see
 * sffn_get_layer_info) on the single-launch kernel without
 * SFFN_FLAG_BALANCE; otherwise SFFN_ERR_UNSUPPORTED.  mask_trace, when given,
 * records the look-ahead masks the calls used. */
#define SFFN_STACK_LOOKAHEAD 1
size_t sffn_stack_workspace_size(const sffn_layer_t* layers, int32_t n_layers, int32_t batch);

/* Offline profile pass (hot/cold classification by activation frequency):
 * counts[i] = number of the n_tokens rows of X (device, [n_tokens][d_model])
 * for which neuron i is predicted active.  counts: [d_ff] int32, device,
 * overwritten. */
sffn_status sffn_profile_counts(sffn_layer_t layer, const void* X, int32_t n_tokens,
                                int32_t* counts, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Host-side: perm[new] = old, neurons by descending count, ties by ascending
 * index.  counts and perm are host arrays of d_ff entries. */
sffn_status sffn_hot_first_perm(const int32_t* counts, int32_t d_ff, int32_t* perm);

/* dst row i = src row perm[i] (device pointers, 4-byte aligned, rows of
 * row_bytes bytes, a multiple of 4; perm is a device int32 array of `rows`
 * entries; src and dst must not overlap).  Used to apply the hot-first order
 * to W_up, W_gate, W_down^T, U and b together. */
sffn_status sffn_permute_rows(const void* src, void* dst, const int32_t* perm, int32_t rows,
                              int64_t row_bytes, void* stream);

/* Builds the bundled row layout of SFFN_FLAG_BUNDLED on `stream`:
 * bundle[i] = [W_gate[i] | W_up[i] | W_down^T[i]] when w_gate is given (ReGLU),
 * [W_up[i] | W_down^T[i]] when it is NULL (ReLU).  All pointers are device
 * pointers, 16-byte aligned, the matrices [d_ff][d_model] of `dtype`, the
 * bundle [d_ff][(2 or 3) * d_model], not overlapping them.  Byte copies only
 * (three strided cudaMemcpy2DAsync). */
sffn_status sffn_bundle_rows(const void* w_up, const void* w_gate, const void* w_downT, int32_t d_ff,
                             int32_t d_model, int32_t dtype, void* bundle, void* stream);

/* Synchronises `stream`, copies the workspace status word to *status (an
 * sffn_status value) and clears it. */
sffn_status sffn_read_device_status(void* workspace, int32_t* status, void* stream);

/* Test hook for the bounded waits: queues a one-block kernel that waits, with
 * the library's grid-barrier code and a limit of timeout_ns nanoseconds, for
 * an arrival that never comes; the status word then reads SFFN_ERR_TIMEOUT. */
sffn_status sffn_debug_wait_timeout(void* workspace, size_t workspace_bytes, int64_t timeout_ns,
                                    void* stream);

/* Test hook for the co-residency requirement of sffn_forward: queues
 * `blocks` one-warp blocks that each hold smem_bytes of dynamic shared memory
 * (0..the per-block opt-in maximum) on their SM for ns nanoseconds of wall
 * time (at most 2e9) and then exit; they touch no memory.  Launched on one
 * stream while a batch-1 call runs on another, they keep part of the call's
 * grid from being resident.  Errors: SFFN_ERR_INVALID_ARG outside the ranges. */
sffn_status sffn_debug_occupy(int64_t ns, int32_t blocks, int32_t smem_bytes, void* stream);

/* Profiling hook: the next n_pairs launches of a call's dominant kernel (the
 * single-launch layer kernel at batch 1, the tensor-core union kernel or the
 * row-gather kernel; of sffn_forward, sffn_dense_forward and
 * sffn_forward_stack), counted from this call, are each bracketed on their
 * stream by records of start_events[i] and stop_events[i] (cudaEvent_t passed
 * as void*), i = 0, 1, ...; later launches are not.  While the stream is being
 * captured the records become graph nodes, so a graph replay times every
 * bracketed launch inside the graph.  n_pairs = 0 switches it off.  The arrays
 * are copied; the events must outlive their use.  Process-wide, not
 * thread-safe: for timing.  SFFN_ERR_INVALID_ARG for NULL arrays or events. */
sffn_status sffn_set_profile_events(void* const* start_events, void* const* stop_events, int32_t n_pairs);

/* Limit of every device-side wait, in nanoseconds (default 1e9). */
sffn_status sffn_set_wait_limit_ns(int64_t ns);

const char* sffn_status_string(sffn_status status);
/* Message of the last failed call on this host thread ("" if none). */
const char* sffn_last_error(void);
int32_t sffn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SFFN_H */
