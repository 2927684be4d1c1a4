/*
 * onebit_adam.h -- C ABI of the GB300 (sm_103a) 1-bit Adam optimizer step.
 *
 * The method ("1-bit Adam: Communication Efficient Large-Scale Training with Adam's Convergence
 * Speed", Tang et al. 2021) has two stages:
 *   - warm-up: uncompressed Adam on the workers' averaged gradient (Sec. 4.3; AIMech page
 *     "1-bit Adam (Two-Stage Preconditioner-Frozen Error-Compensated Adam)", summary formulas
 *     m_t = b1 m_{t-1} + (1-b1) g_t, v_t = b2 v_{t-1} + (1-b2) g_t^2);
 *   - compression: the variance is frozen as V = diag(sqrt(v_Tw) + eps) (Sec. 3.3 and 5: momentum
 *     SGD with a coordinate-wise learning rate) and momentum is exchanged with error-compensated
 *     1-bit compression through a gather-then-broadcast exchange (Sec. 6 and Sec. 11; AIMech
 *     page's compressed-allreduce mechanism: worker error delta^(i), server error epsilon).
 *
 * Two forms.  In the single-GPU form (onebit_adam_init) all n data-parallel workers are simulated on
 * one GPU: worker i's gradient is one of the n gradient buffers passed to a step, and the exchange is
 * index arithmetic over the workers' packed messages in this GPU's memory.  In the multi-GPU form
 * (onebit_adam_init_rank, near the end of this file) every GPU holds a share of the workers and of the
 * server shards, and the caller's collectives carry the packed messages between the library's calls.
 * The library itself never communicates across GPUs.
 *
 * Per compression step, for every tensor k of the parameter list:
 *   worker i:   m_i = b1*m + (1-b1)*g_i;  c_i = m_i + delta_i;
 *               s_ik = ||c_i||_2 / sqrt(L_k) (scale that preserves the magnitude, Sec. 4.3 and the
 *               codewithpapers "1-bit Adam" page);  bits_i = [c_i >= 0];  delta_i = c_i - s_ik*sign(c_i)
 *   server j:   over shard j of tensor k:  a = (sum_{i=0..n-1} s_ik*sign_i) / n + eps_srv;
 *               S_kj = ||a||_2 / sqrt(len_kj);  bitsS = [a >= 0];  eps_srv = a - S_kj*sign(a)
 *   broadcast:  m = S_kj*sign(a) becomes the shared momentum;  x = x - lr*(m / (sqrt(v_Tw)+eps)).
 * The n-term server sum is taken in worker order 0..n-1 in fp32; all elementwise arithmetic is fp32
 * with no fused multiply-add; norms are accumulated in double and rounded once to fp32.
 *
 * Conventions used by every entry point:
 *   - Errors: every call returns a status and never aborts, and no C++ exception leaves it (a host
 *     allocation that fails is ONEBIT_ERR_NOMEM).  Argument and phase checks happen on the host
 *     before anything is enqueued; a failed check changes no state.  CUDA launch or copy
 *     failures return ONEBIT_ERR_CUDA (onebit_adam_last_error() gives the CUDA message).  When a
 *     step call fails that way after some of its kernels were enqueued, the step count does not
 *     advance and the parameters and optimizer state are unspecified: resume from a checkpoint
 *     (onebit_adam_set_step + onebit_adam_import).  A non-finite scale found on the device sets a
 *     sticky flag read by onebit_adam_get_status().
 *   - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Calls enqueue work and
 *     return without synchronising, except where stated.  All calls on one handle must be ordered
 *     on one stream (or synchronised by the caller): the handle's state is updated in stream order.
 *   - Memory: parameters and gradients are caller-owned device memory.  Gradients are only read
 *     and must stay valid until the enqueued work completes.  Parameters are updated in place.
 *     All optimizer state lives in the workspace (caller-provided or library-allocated).
 *   - Layout: a parameter list has T tensors of numel L_k (one flat buffer is T = 1).  State
 *     exported or imported per element is the concatenation of the tensors, without padding
 *     (D = sum L_k).  Packed sign words: tensor k owns ceil(L_k/32) uint32 words, concatenated;
 *     bit b of word w of tensor k is element 32w+b; a set bit means the value is >= 0 (+0 and -0
 *     give 1, NaN gives 0); bits past L_k are 0.  Server shards of tensor k: S_k = 32*ceil(L_k/(32n)),
 *     shard j = [j*S_k, min((j+1)*S_k, L_k)), possibly short or empty (an empty shard has scale 0).
 */
#ifndef ONEBIT_ADAM_H
#define ONEBIT_ADAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct onebit_adam onebit_adam_t; /* opaque, owned by the library */
typedef void* onebit_stream_t;            /* a cudaStream_t */

typedef enum {
  ONEBIT_OK = 0,
  ONEBIT_ERR_INVALID_ARG = 1, /* a NULL or out-of-range argument, or an inconsistent config */
  ONEBIT_ERR_PHASE = 2,       /* the call is not legal in the handle's current phase */
  ONEBIT_ERR_CUDA = 3,        /* a CUDA runtime call failed */
  ONEBIT_ERR_NOMEM = 4,       /* a library allocation failed */
  ONEBIT_ERR_WORKSPACE = 5,   /* the caller's workspace is too small or misaligned */
  ONEBIT_ERR_NONFINITE = 6,   /* a worker or server scale was NaN or infinite */
  ONEBIT_ERR_UNSUPPORTED = 7, /* a valid request the library does not support */
  ONEBIT_ERR_BOUNDS = 8       /* checked builds only: a kernel's bounds check found a unit of work whose
                               * accesses would leave its buffers, and skipped it */
} onebit_status_t;

typedef enum { ONEBIT_F32 = 0, ONEBIT_F16 = 1, ONEBIT_BF16 = 2 } onebit_dtype_t;

typedef enum { ONEBIT_PHASE_WARMUP = 0, ONEBIT_PHASE_COMPRESS = 1 } onebit_phase_t;

/* What export/import/state_size address. */
typedef enum {
  ONEBIT_STATE_M = 0,             /* shared momentum m: D fp32 */
  ONEBIT_STATE_V = 1,             /* warm-up: v; after the freeze: den = sqrt(v_Tw)+eps.  D fp32 */
  ONEBIT_STATE_WORKER_ERROR = 2,  /* delta_i of one worker: D fp32 */
  ONEBIT_STATE_SERVER_ERROR = 3,  /* eps_srv: D fp32 */
  ONEBIT_STATE_WORKER_BITS = 4,   /* last message of one worker: W uint32 (export only) */
  ONEBIT_STATE_SERVER_BITS = 5,   /* last broadcast: W uint32 (export only) */
  ONEBIT_STATE_WORKER_SCALES = 6, /* last worker scales: n*T fp32, [worker][tensor or block] (export only) */
  ONEBIT_STATE_SERVER_SCALES = 7  /* last server scales: T*n fp32, [tensor or block][shard] (export only) */
} onebit_state_t;

/* The kernels, for onebit_adam_kernel_times(). */
typedef enum {
  ONEBIT_K_WARMUP = 0,         /* fused worker-average + Adam */
  ONEBIT_K_FREEZE = 1,         /* den = sqrt(v)+eps */
  ONEBIT_K_WORKER = 2,         /* momentum + error + sign pack + norm partials, all workers */
  ONEBIT_K_WORKER_SCALE = 3,   /* worker scales from the partials (and the partials' exact-range repair) */
  ONEBIT_K_SERVER = 4,         /* unpack + ordered average + server error + sign pack + partials */
  ONEBIT_K_SERVER_SCALE = 5,   /* server shard scales from the partials */
  ONEBIT_K_UPDATE = 6,         /* unpack broadcast + preconditioned update */
  ONEBIT_K_EXPORT = 7,         /* state export / import */
  ONEBIT_K_EC_UPDATE = 8,      /* Adam on the broadcast gradient (gradient-compression baseline) */
  ONEBIT_K_EXCHANGE = 9,       /* multi-GPU form: packing and unpacking of the exchange buffers */
  ONEBIT_NUM_KERNELS = 10
} onebit_kernel_t;

typedef struct {
  float beta1;             /* b1, 0 <= b1 < 1 */
  float beta2;             /* b2, 0 <= b2 < 1 */
  float eps;               /* epsilon of V = diag(sqrt(v) + eps), >= 0 */
  float lr;                /* gamma */
  int64_t warmup_steps;    /* T_w >= 1: warm-up steps before the variance is frozen */
  int32_t n_workers;       /* n, 1 <= n <= 256 */
  int32_t n_tensors;       /* T >= 1 (1 = one flat buffer) */
  const int64_t* numel;    /* host array [T], L_k >= 0, 1 <= sum L_k <= 2^40 (more is
                            * ONEBIT_ERR_UNSUPPORTED: no device holds that much state) */
  int32_t grad_dtype;      /* onebit_dtype_t */
  int32_t bias_correction; /* 0: the pages' formulas (default); 1: Kingma-Ba bias correction */
  int64_t scale_block;     /* scale granularity.  0 (default): one worker scale per tensor and n
                            * server shards per tensor.  B > 0, a multiple of 32: the per-chunk
                            * parameter-server form of Tang et al. Sec. 11 -- every tensor is cut
                            * into blocks of B elements (the last may be shorter; an empty tensor
                            * keeps one empty block) and each block is compressed as a tensor of its
                            * own, with its own worker scales and its own n server shards.  The
                            * scale exports and onebit_adam_plan_chunks() then index blocks, tensor
                            * k's blocks in order after those of tensor k-1; gradients, parameters
                            * and every per-element state keep the caller's tensor layout.  Any other
                            * value is ONEBIT_ERR_INVALID_ARG. */
} onebit_adam_config_t;

/* Bytes of device workspace a config needs (256-byte aligned pieces included). */
onebit_status_t onebit_adam_workspace_size(const onebit_adam_config_t* cfg, size_t* bytes);

/* Create a handle.  params: host array [T] of device pointers to the fp32 parameters, kept for the
 * handle's lifetime.  workspace: device memory of at least onebit_adam_workspace_size() bytes,
 * 256-byte aligned, caller-owned; or NULL for a library cudaMalloc freed by onebit_adam_free().
 * The state is zeroed on `stream` (m = v = 0, t = 0, phase WARMUP). */
onebit_status_t onebit_adam_init(const onebit_adam_config_t* cfg, float* const* params, void* workspace,
                                 size_t workspace_bytes, onebit_stream_t stream, onebit_adam_t** out);

/* One warm-up Adam step (legal while phase == WARMUP and t < T_w): the mean of the n workers'
 * gradients, summed in worker order (the uncompressed allreduce of the warm-up stage, Tang et al.
 * Sec. 4.3 and 6), then m = b1 m + (1-b1) g, v = b2 v + (1-b2) g^2, x -= lr m/(sqrt(v)+eps) (the
 * AIMech page's summary formulas).  grads: host array [n*T] of device pointers, ordered
 * [worker][tensor], each L_k values of grad_dtype.  t += 1. */
onebit_status_t onebit_adam_warmup_step(onebit_adam_t* h, const void* const* grads, onebit_stream_t stream);

/* Freeze the variance: den = sqrt(v) + eps (v / (1 - b2^t) first with bias correction) -- the
 * preconditioner V = diag(sqrt(v_Tw) + eps) of the AIMech page, under which the compression stage is
 * momentum SGD with a coordinate-wise learning rate (Tang et al. Sec. 3.3 and 5).  Legal in phase
 * WARMUP after at least one warm-up step; the phase becomes COMPRESS, worker and server errors start
 * at 0 and the first compression step reads the fp32 warm-up momentum. */
onebit_status_t onebit_adam_freeze_variance(onebit_adam_t* h, onebit_stream_t stream);

/* One compression-stage step (legal in phase COMPRESS): the three steps of Tang et al. Sec. 11 --
 * every worker updates its momentum and compresses it with error compensation (Sec. 4.1, 4.3; the
 * codewithpapers page's scale), every server shard averages the workers' messages and compresses
 * again with its own error (the AIMech page's compressed-allreduce mechanism), and the broadcast
 * momentum updates the parameters -- as stated at the top of this file.  grads as for warmup_step.
 * t += 1. */
onebit_status_t onebit_adam_compress_step(onebit_adam_t* h, const void* const* grads, onebit_stream_t stream);

/* One step of the baseline the method is contrasted with ("1-bit Adam ...", Sec. 3.2 and 4.2):
 * error-compensated 1-bit compression of the GRADIENTS (c_i = g_i + delta_i, worker and server
 * compression and error feedback exactly as in the compression stage), then every worker runs plain
 * Adam on the broadcast g_hat = S*sign(a): m = b1 m + (1-b1) g_hat, v = b2 v + (1-b2) g_hat^2,
 * x -= lr * m/(sqrt(v)+eps) (bias-corrected if configured).  Legal in phase WARMUP (any t); it
 * shares m and v with warmup_step, keeps its own error memories (exported as WORKER_ERROR /
 * SERVER_ERROR) and a freeze resets them.  t += 1. */
onebit_status_t onebit_adam_ec_adam_step(onebit_adam_t* h, const void* const* grads, onebit_stream_t stream);

/* The same two steps with HOST gradient buffers ([n*T] host pointers, pinned or pageable): the
 * library copies them into one of two device staging buffers it owns (allocated on first use,
 * 2 x n*D*grad bytes, used alternately) on internal copy streams, and `stream` waits for those
 * copies before the step's kernels.  The copies wait only until their staging buffer is free again,
 * not for earlier work on `stream`, so that one step's copies overlap the previous step's kernels:
 * the host buffers must already hold this step's gradients when the call is made.  Pageable sources
 * are copied before the call returns; pinned sources must stay valid until `stream` has passed this
 * step. */
onebit_status_t onebit_adam_warmup_step_host(onebit_adam_t* h, const void* const* host_grads, onebit_stream_t stream);
onebit_status_t onebit_adam_compress_step_host(onebit_adam_t* h, const void* const* host_grads, onebit_stream_t stream);

/* Release the handle (synchronises its device; frees library allocations only). */
onebit_status_t onebit_adam_free(onebit_adam_t* h);

/* Synchronise `stream` and report the sticky device flags: ONEBIT_OK, ONEBIT_ERR_NONFINITE (a scale
 * was NaN or infinite), or ONEBIT_ERR_CUDA when a kernel gave up waiting (about one second) for its
 * own asynchronous copies and stopped early (onebit_adam_last_error() says so).  A checked build
 * (the library compiled with -DONEBIT_CHECKS) also reports ONEBIT_ERR_BOUNDS, first of all: some
 * kernel found a chunk, scale range or exchange range whose accesses would leave its buffers and
 * skipped it (onebit_adam_last_error() names the kernels); the state of that step is not
 * meaningful.  A normal build has no such checks. */
onebit_status_t onebit_adam_get_status(onebit_adam_t* h, onebit_stream_t stream);
/* Clear the sticky device flag (enqueued on `stream`). */
onebit_status_t onebit_adam_clear_status(onebit_adam_t* h, onebit_stream_t stream);

/* Current step count t and phase (host-side state, no synchronisation). */
onebit_status_t onebit_adam_get_step(const onebit_adam_t* h, int64_t* t, int32_t* phase);
/* Set t and the phase, for resuming from a checkpoint.  Moving to COMPRESS marks the errors zero
 * and the momentum as the fp32 buffer (import them afterwards); the V buffer must then hold den. */
onebit_status_t onebit_adam_set_step(onebit_adam_t* h, int64_t t, int32_t phase, onebit_stream_t stream);

/* Bytes of one export/import buffer for `what` (see onebit_state_t). */
onebit_status_t onebit_adam_state_size(const onebit_adam_t* h, int32_t what, size_t* bytes);

/* Copy state `what` (worker index for per-worker items, else ignored) into device memory `dst`
 * (onebit_adam_state_size() bytes) on `stream`.  Errors and the momentum are materialised in fp32.
 * `dst` holds the result once `stream` has passed the copy. */
onebit_status_t onebit_adam_export(onebit_adam_t* h, int32_t what, int32_t worker, void* dst, onebit_stream_t stream);

/* Load state `what` (M, V, WORKER_ERROR, SERVER_ERROR) from device memory `src` on `stream`.
 * An imported error is used exactly by the next step that reads errors: a compression step, or in
 * phase WARMUP a gradient-compression baseline step (a freeze still resets the errors to zero).
 * Importing M makes the next compression step read this fp32 momentum.  The copy is enqueued on
 * `stream`: `src` must stay valid and unchanged until `stream` has passed it. */
onebit_status_t onebit_adam_import(onebit_adam_t* h, int32_t what, int32_t worker, const void* src, onebit_stream_t stream);

/* Bytes one worker sends per compression step (sign words + one fp32 scale per tensor) and the
 * bytes the same vector takes in fp32: the 1/32 volume behind the codewithpapers page's 97% (96.9%)
 * reduction against fp32. */
onebit_status_t onebit_adam_comm_bytes(const onebit_adam_t* h, uint64_t* compressed, uint64_t* fp32_bytes);

/* Per-kernel timing with CUDA events recorded around every launch on the launch stream.
 * kernel_times synchronises the recorded events, writes the total milliseconds and launch counts
 * accumulated since the previous call (arrays of ONEBIT_NUM_KERNELS), and resets them. */
onebit_status_t onebit_adam_set_timing(onebit_adam_t* h, int32_t enable);
onebit_status_t onebit_adam_kernel_times(onebit_adam_t* h, double* ms, int64_t* launches);
/* Kernel launches enqueued by this handle since init. */
onebit_status_t onebit_adam_launch_count(const onebit_adam_t* h, int64_t* launches);

/* Variance-norm monitor ("1-bit Adam ...", Sec. 3.3: the variance's norm settles early in
 * training, which is why the variance can be frozen).  While enabled, every warm-up step also
 * computes ||v_t||_2 over the whole parameter list (exact squares, double accumulation) and copies
 * it to a pinned host slot (enabling allocates that slot).  variance_norm() waits for the last
 * monitored step's value and returns it with its step index t; ONEBIT_ERR_PHASE if no monitored
 * warm-up step has run. */
onebit_status_t onebit_adam_set_variance_monitor(onebit_adam_t* h, int32_t enable);
onebit_status_t onebit_adam_variance_norm(onebit_adam_t* h, double* norm, int64_t* step);

/* Automatic freeze.  The pages motivate freezing with the variance's norm, which stabilises early in
 * training (Tang et al. Sec. 3.3) and sets the warm-up length T_w (the AIMech page).  With tol > 0,
 * every following warm-up step also computes ||v_t||_2 (as the variance monitor does), waits for it
 * (the call then synchronises `stream`), and freezes the variance before returning -- exactly as
 * onebit_adam_freeze_variance() does -- at the first step whose norm changed by at most tol relative
 * to the previous step's (|n_t - n_{t-1}| <= tol * n_{t-1}), or at the step that reaches T_w.  The
 * caller reads the phase with onebit_adam_get_step().  tol = 0 turns it off; a negative or non-finite
 * tol is ONEBIT_ERR_INVALID_ARG.  Enabling it allocates the monitor's pinned host slot once
 * (ONEBIT_ERR_NOMEM if that fails). */
onebit_status_t onebit_adam_set_auto_freeze(onebit_adam_t* h, double tol);

/* Set the learning rate gamma used by the following steps (warm-up, compression and baseline).  The
 * pages keep gamma constant; this serves the schedules training uses (warm-up ramps, decay).  The
 * new value must be finite, else ONEBIT_ERR_INVALID_ARG.  A step captured in a CUDA graph keeps the
 * gamma it was captured with. */
onebit_status_t onebit_adam_set_lr(onebit_adam_t* h, float lr);

/* Caps the CTAs that every streaming kernel launch of this handle uses (0, the default: as many as
 * fill the GPU).  No counterpart on the method's pages: it lets a caller leave SMs to work running
 * concurrently on other streams.  Results do not depend on it, bit for bit: every partial sum is
 * per chunk and reduced in a fixed order, whatever the grid.  Negative values are
 * ONEBIT_ERR_INVALID_ARG. */
onebit_status_t onebit_adam_set_max_ctas(onebit_adam_t* h, int32_t max_ctas);

/* Failure-detection test hooks; nothing here makes the GPU fault.
 *   ONEBIT_FAULT_STALL_COPIES makes the next steps' shared-memory staged kernels wait for `value`
 *     bytes (1..2^20) that no copy delivers, so that their bounded waits run out (about one second):
 *     the kernel stops early, the sticky flag is set and onebit_adam_get_status() returns
 *     ONEBIT_ERR_CUDA, with the CUDA context still usable.  The state of that step is not meaningful.
 *   ONEBIT_FAULT_FAIL_ALLOC makes the handle's next `value` (1..1000) device or pinned allocations
 *     fail as if memory were exhausted (the host-gradient staging buffers, the variance monitor's
 *     slot): the call returns ONEBIT_ERR_NOMEM and, like every failed check, changes no state.
 *   ONEBIT_FAULT_TIGHTEN_BOUNDS (checked builds only; ONEBIT_ERR_UNSUPPORTED otherwise) makes the
 *     bounds checks withhold the last `value` padded elements (a multiple of 32, 32..the padded
 *     total) from every state row.  The units that reach into them are skipped as if their
 *     descriptors were out of bounds and get_status() returns ONEBIT_ERR_BOUNDS.  The checks only get
 *     stricter: no access leaves the buffers.
 *   ONEBIT_FAULT_NONE turns all of them off. */
typedef enum {
  ONEBIT_FAULT_NONE = 0,
  ONEBIT_FAULT_STALL_COPIES = 1,
  ONEBIT_FAULT_FAIL_ALLOC = 2,
  ONEBIT_FAULT_TIGHTEN_BOUNDS = 3
} onebit_fault_t;
onebit_status_t onebit_adam_set_fault_injection(onebit_adam_t* h, int32_t kind, int64_t value);

/* The work chunks the kernels use for a config (host only, no GPU needed): up to `cap` rows of
 * five int64 {tensor, shard, start element within the tensor, length, padded state offset}.
 * *count receives the total number of chunks.  These are the server-side chunks (server, update,
 * warm-up and export kernels): they never cross a tensor or a server shard. */
onebit_status_t onebit_adam_plan_chunks(const onebit_adam_config_t* cfg, int64_t* rows, int64_t cap, int64_t* count);

/* The worker kernel's chunks (host only): rows of six int64 {tensor, first shard, start element
 * within the tensor, length, padded state offset, shard length if the chunk holds several whole
 * shards else 0}.  They never cross a tensor.  Where a tensor's shards are at least a chunk long they
 * equal the server-side chunks; where shards are shorter, one worker chunk holds several whole shards,
 * so that the worker kernel keeps long units. */
onebit_status_t onebit_adam_plan_worker_chunks(const onebit_adam_config_t* cfg, int64_t* rows, int64_t cap,
                                               int64_t* count);

/* ---- Multi-GPU form: the n workers spread over `world` GPUs, one process (rank) per GPU ----
 *
 * The pages' system runs the exchange across machines: every worker compresses its momentum, an
 * all-to-all sends each server the workers' compressed chunks of its shard, every server averages,
 * compresses again and keeps its own error, and an allgather brings the result to every worker, which
 * updates its copy of the model (Tang et al. Sec. 6 and Sec. 11 steps 1-3; the AIMech page's
 * "gather-then-broadcast"; the NCCL backend of the 1-bit LAMB page's abstract).  In this form rank r
 * of `world` (n a multiple of world, nl = n/world) simulates workers r*nl .. r*nl+nl-1 and serves
 * shards r*nl .. r*nl+nl-1 of every tensor (or scale block); it keeps a full copy of x, m and den, the
 * c of its own workers and the server state of its own shards.  A compression step is split at the
 * exchange: the caller moves the buffers between the calls with its collectives (an all-to-all with
 * equal blocks, then an all-gather), and each rank's results are bit-identical to a single GPU
 * simulating all n workers (onebit_adam_init).  The warm-up step takes every worker's gradient (n*T
 * pointers, e.g. after an all-gather of the ranks' gradients) and computes the same ordered mean on
 * every rank; compress_step, compress_step_host and ec_adam_step return ONEBIT_ERR_UNSUPPORTED when
 * world > 1.  Exports: WORKER_ERROR only for this rank's workers (else ONEBIT_ERR_INVALID_ARG);
 * SERVER_ERROR on this rank's shards (other elements read 0); WORKER_BITS rows of other ranks' workers
 * hold only this rank's shards.  Imports: WORKER_ERROR for this rank's workers; SERVER_ERROR on this
 * rank's shards. */

/* Workspace bytes of rank `rank` of `world` (0 <= rank < world, n_workers a multiple of world). */
onebit_status_t onebit_adam_workspace_size_rank(const onebit_adam_config_t* cfg, int32_t rank, int32_t world,
                                                size_t* bytes);
/* Create rank `rank`'s handle; the other arguments as for onebit_adam_init.  world = 1 gives a handle
 * equal to onebit_adam_init's on which the split step is legal too (its exchange buffers may be NULL). */
onebit_status_t onebit_adam_init_rank(const onebit_adam_config_t* cfg, int32_t rank, int32_t world,
                                      float* const* params, void* workspace, size_t workspace_bytes,
                                      onebit_stream_t stream, onebit_adam_t** out);
/* Words (uint32) of one block of the all-to-all (send_block; the send and receive buffers hold `world`
 * blocks each, block q for / from rank q) and of one block of the all-gather (bcast_block; this rank's
 * contribution, the gathered buffer holds `world` blocks in rank order).  The same on every rank. */
onebit_status_t onebit_adam_exchange_words(const onebit_adam_t* h, int64_t* send_block, int64_t* bcast_block);
/* Step 1 (Sec. 11 step 1, workers): this rank's workers form their momentum with error compensation
 * and compress it; block q of `send` (device, world*send_block words) receives, for each of this
 * rank's workers, its scales and the sign words of rank q's shards.  grads: host array [nl*T] of
 * device pointers, [local worker][tensor].  Legal in phase COMPRESS outside a split step.  This
 * rank's own block of `send` is not written (its data never leaves). */
onebit_status_t onebit_adam_compress_begin(onebit_adam_t* h, const void* const* grads, uint32_t* send,
                                           onebit_stream_t stream);
/* Step 2 (Sec. 11 step 2, servers): `recv` (device, world*send_block words; block p from rank p, as
 * an all-to-all of the send buffers delivers it) brings every worker's message for this rank's
 * shards; the shards are averaged, compressed again with the server error, and `bcast` (device,
 * bcast_block words) receives this rank's server scales and sign words.  Legal after
 * compress_begin. */
onebit_status_t onebit_adam_compress_serve(onebit_adam_t* h, const uint32_t* recv, uint32_t* bcast,
                                           onebit_stream_t stream);
/* Step 3 (Sec. 11 step 3, broadcast and update): `gathered` (device, world*bcast_block words, the
 * all-gather of every rank's bcast block in rank order) completes the broadcast momentum, and the
 * parameters are updated.  Legal after compress_serve; t += 1.  `send`, `recv`, `bcast` and
 * `gathered` must stay valid until `stream` has passed the call that reads or writes them; with
 * world = 1 they are not touched and may be NULL.  Between compress_begin and compress_end the
 * handle is inside a split step: every other step call and every import returns ONEBIT_ERR_PHASE.
 * A split step that cannot be completed (a collective failed) is abandoned with
 * onebit_adam_set_step, after which the state is restored from a checkpoint (onebit_adam_import). */
onebit_status_t onebit_adam_compress_end(onebit_adam_t* h, const uint32_t* gathered, onebit_stream_t stream);
/* The exchange copies of rank `rank` of `world` (host only): up to `cap` rows of eight int64 {stage
 * (0 begin pack, 1 serve unpack, 2 serve pack, 3 end unpack), source region, source row, source
 * offset, destination region, destination row, destination offset, words}.  Regions: 0 worker sign
 * words (row = worker, offset = word in the concatenation of the tensors' words), 1 worker scales (row
 * = worker, offset = tensor), 2 server sign words (row 0), 3 server scales (row = tensor, offset =
 * shard), 4 the exchange buffer (row = block, offset = word in the block).  *count receives the number
 * of rows, *send_block and *bcast_block the block sizes in words. */
onebit_status_t onebit_adam_plan_exchange(const onebit_adam_config_t* cfg, int32_t rank, int32_t world, int64_t* rows,
                                          int64_t cap, int64_t* count, int64_t* send_block, int64_t* bcast_block);

/* Largest vector onebit_worker_compress_noalloc() accepts (elements). */
#define ONEBIT_NOALLOC_MAX_LEN 268435456

/* Worker compression of one vector, for callers that may not allocate device memory.
 *
 * No counterpart on the method's pages: it is a service of this library.  Code that runs under a
 * framework whose caching allocator owns every device byte, in a latency-critical loop where
 * cudaMalloc's implicit device-wide synchronisation is not acceptable, or in a plug-in that is handed
 * buffers but no right to allocate, cannot obtain scratch memory.  This call needs none from the
 * caller and allocates none itself (no cudaMalloc, cudaFree or allocating library routine): its
 * scratch (per-chunk sum-of-squares partials and the scale, 32 KB) is a file-scope __device__ array
 * that every GPU loading this library holds until the process exits.
 *
 * Computes, in the worker kernel's fp32 operation order:
 *   c = (beta1*m + (1-beta1)*g) + err_in;   scale = ||c||_2 / sqrt(len);
 *   bits = [c >= 0] packed (bit b of word w = element 32w+b, padding bits 0);
 *   err_out = c - scale*sign(c).
 * m: len fp32, device.  grad: len values of grad_dtype, device.  err_in: len fp32, device, or NULL
 * for a zero error.  bits_out: ceil(len/32) uint32, device.  scale_out: one fp32, device.  err_out:
 * len fp32, device.  Every output must be disjoint from every input and from the other outputs,
 * except that err_in may be exactly err_out (the error is then updated in place); any other overlap,
 * a NULL input or output other than err_in, or a len outside 1 <= len <= ONEBIT_NOALLOC_MAX_LEN is
 * ONEBIT_ERR_INVALID_ARG, and nothing is enqueued.  Pointers of any alignment are accepted (32-byte
 * aligned fp32 buffers and 16-byte aligned 16-bit gradients take the vector loads).
 * Non-finite inputs are not reported: the call returns before its kernels run, so a NaN or infinite
 * norm reaches scale_out (and err_out) as is -- a caller that needs the check tests *scale_out.
 *
 * The first call on a device looks up the scratch array's device address (once per device, with
 * that device current); make that first call before any stream capture.  Every call on a device
 * shares the one scratch array and leaves the last call's contents in it; nothing in it needs
 * clearing because each call writes every slot it reads.  Calls that overlap on the GPU (issued to
 * different streams without ordering between them) race on the array and give wrong results. */
onebit_status_t onebit_worker_compress_noalloc(const float* m, const void* grad, int32_t grad_dtype,
                                               const float* err_in, float beta1, int64_t len, uint32_t* bits_out,
                                               float* scale_out, float* err_out, onebit_stream_t stream);

/* Static description of a status code. */
const char* onebit_adam_error_string(onebit_status_t status);
/* Message of the last CUDA failure seen by this handle ("" if none).  With h = NULL: the message of
 * the last onebit_adam_init that failed on the calling thread ("" if none), since a failed init
 * returns no handle.  The string stays valid until the next call on the same handle (or, for
 * NULL, the next onebit_adam_init on this thread). */
const char* onebit_adam_last_error(const onebit_adam_t* h);

#ifdef __cplusplus
}
#endif
#endif /* ONEBIT_ADAM_H */
