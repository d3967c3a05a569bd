/*
 * muon.h -- C ABI of the B300 (sm_103a) Muon optimizer-step library (libmuon.so).
 *
 * The operation is the Muon step of the nanochat pretraining recipe as the page
 * "Cara Melatih ChatGPT Sendiri dengan Budget 50 Dolar" (apidog.com) describes
 * it in section "2. Pengoptimal Muon (nanochat/optim.py)" (and its dev.to
 * translation, section "2. ตัวปรับปรุง Muon"): every 2-D weight matrix gets a
 * momentum update, the update direction is normalised and driven toward its
 * orthogonal polar factor by quintic Newton-Schulz iterations (one (a, b, c)
 * row per iteration: A = X X^T, B = b A + c A A, X <- a X + B X), and the
 * weight moves along the result.  The pages print neither the momentum form
 * nor the normalisation nor the update scale; this library takes
 *
 *   m' = beta m + g                       (stored back into the momentum buffer)
 *   u  = nesterov ? g + beta m' : m'
 *   X0 = u / (||u||_F + eps), transposed first when rows > cols (long side = columns)
 *   K iterations with rows 0..K-1 of the coefficient table
 *   O  = X_K, transposed back;  p <- p - lr * sqrt(max(1, rows/cols)) * O
 *
 * (momentum_mode 1 uses m' = beta m + (1-beta) g, u = nesterov ? (1-beta) g + beta m' : m').
 *
 * Precision: p, g, m are float32 (fp32 state); the Newton-Schulz operands X, A,
 * B are stored as bfloat16 (round to nearest even) and every product
 * accumulates in fp32; the last iteration's result O is formed in fp32 and
 * applied to p without being stored: p' = p + fp32(-lr sqrt(max(1, rows/cols)) O),
 * the addition made in fp32 by the memory system (a TMA reduce-add).
 *
 * Conventions shared by every entry point:
 *  - All functions return a muon_status; none aborts, throws or prints.
 *  - Matrices are dense, contiguous, row-major float32 arrays in device memory
 *    of the device that was current at muon_init, owned by the caller.
 *  - Work is enqueued on the caller's CUDA stream and is asynchronous; argument
 *    errors are reported synchronously, device-side errors (a timed-out wait,
 *    an out-of-range tile) are latched in a device status word and returned by
 *    muon_get_status.
 *  - One process-global context; the functions are not thread-safe.
 *  - Steps of a context with the same list of shapes share one workspace (and
 *    the NorMuon buffers), and every step shares the device status word; a call
 *    orders its work only after earlier work on its own `stream`.  Steps issued
 *    on different streams must therefore be ordered by the caller (an event, or
 *    one stream for all of them); steps that overlap on the GPU race.
 *  - The library's kernels let the next kernel on the stream begin launching
 *    early (programmatic dependent launch).  Ordinary launches are unaffected;
 *    a caller's kernel launched with programmatic stream serialization must, as
 *    CUDA requires of any such kernel, execute griddepcontrol.wait before it
 *    reads what the step wrote.
 */
#ifndef MUON_H
#define MUON_H

#ifdef __cplusplus
extern "C" {
#endif

/* Every entry point below is exported with default visibility; the library
 * hides everything else. */
#if defined(__GNUC__)
#define MUON_API __attribute__((visibility("default")))
#else
#define MUON_API
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* muon_stream_t;

typedef enum muon_status {
    MUON_OK = 0,
    MUON_ERR_INVALID_ARG = 1,         /* NULL pointer, n_mats < 0, ns_steps out of range, bad config */
    MUON_ERR_UNSUPPORTED_SHAPE = 2,   /* rows or cols < 8 or not a multiple of 8 (16-byte bf16 rows) */
    MUON_ERR_MISALIGNED = 3,          /* a matrix pointer is not 16-byte aligned */
    MUON_ERR_NOT_INITIALIZED = 4,     /* muon_init has not succeeded */
    MUON_ERR_CUDA = 5,                /* a CUDA runtime/driver call failed */
    MUON_ERR_OUT_OF_MEMORY = 6,       /* workspace allocation failed */
    MUON_ERR_DEVICE_TIMEOUT = 7,      /* a kernel's bounded wait expired (device status) */
    MUON_ERR_DEVICE_BOUNDS = 8,       /* a kernel refused launch parameters whose tile list does not
                                         match its classes (device status; that launch ran no tile) */
    MUON_ERR_UNSUPPORTED_DEVICE = 9,  /* no device, or the current device is not sm_103 */
    MUON_ERR_SCRATCH_LIMIT = 10       /* the request needs more than the fixed scratch of
                                         muon_momentum_norm_noalloc holds */
} muon_status;

/* Stored (PyTorch (out_features, in_features)) shape of one parameter matrix. */
typedef struct muon_shape {
    int rows;
    int cols;
} muon_shape;

enum {
    MUON_MOMENTUM_SGD_NESTEROV = 0, /* m' = beta m + g (default) */
    MUON_MOMENTUM_EMA = 1           /* m' = beta m + (1 - beta) g */
};

enum {
    MUON_DEBUG_KEEP_O = 1,            /* also write O (fp32, stored layout) for muon_debug_copy_ns_output */
    MUON_DEBUG_POISON_WORKSPACE = 2,  /* fill the bf16 workspace with NaN before every step */
    MUON_DEBUG_TIME_KERNELS = 4,      /* record CUDA events around every launch (muon_kernel_times) */
    MUON_DEBUG_INJECT_LOST_LOAD = 8,  /* test hook: one operand load of the first Gram launch is never
                                         issued, so the consumer's bounded wait must expire and the step
                                         reports MUON_ERR_DEVICE_TIMEOUT; the result is then invalid */
    MUON_DEBUG_INJECT_BAD_TILES = 16  /* test hook: the first Gram launch is given one tile more than its
                                         classes hold; the kernel's parameter check must refuse it (no
                                         tile runs) and the step reports MUON_ERR_DEVICE_BOUNDS; the
                                         result is then invalid */
};

typedef struct muon_config {
    const double* coeffs;   /* (a, b, c) rows, one per Newton-Schulz iteration, row-major; NULL
                               selects the default: (3.4445, -4.7750, 2.0315) for every row */
    int n_coeff_rows;       /* rows in coeffs (1..16); ignored when coeffs is NULL (then 5) */
    double eps;             /* added to ||u||_F before dividing; <= 0 selects 1e-7 */
    int momentum_mode;      /* MUON_MOMENTUM_* */
    int debug_flags;        /* MUON_DEBUG_* bit set; 0 for production */
    double wait_timeout_s;  /* limit of every in-kernel wait; <= 0 selects 5 s */
} muon_config;

/*
 * Create the process-global context on the current CUDA device.
 * cfg may be NULL (all defaults).  The coefficient table is copied.
 * Errors: MUON_ERR_UNSUPPORTED_DEVICE (not sm_103), MUON_ERR_INVALID_ARG (bad
 * config), MUON_ERR_CUDA.  Calling it again replaces the context (the old one
 * is destroyed first).  Allocates only a few hundred bytes of device memory;
 * the workspace is sized by the first muon_step.
 */
MUON_API muon_status muon_init(const muon_config* cfg);

/*
 * One Muon step over n_mats independent matrices, enqueued on `stream`.
 *   params[i]        device float32 rows x cols, updated in place (p <- p - lr s O)
 *   grads[i]         device float32 rows x cols, read only
 *   momentum_bufs[i] device float32 rows x cols, updated in place (m <- m')
 *   shapes[i]        stored shape; rows, cols >= 8 and multiples of 8
 *   n_mats >= 0 (0 is a no-op); lr, beta as in the formulas above;
 *   nesterov 0/1; ns_steps 0..n_coeff_rows (0 gives O = X0).
 * The host arrays are read during the call only.  A matrix must not alias
 * another one of the same call.  Matrices of equal oriented shape are batched
 * into the same launches.  The context keeps one workspace per distinct list
 * of shapes, up to 8 (a caller that steps several groups of matrices, such as
 * the buckets of a sharded step, alternates between them without rebuilding);
 * a ninth list drops the least recently used workspace, which synchronises
 * the device.  When the weight pointers differ from the previous call with the
 * same shapes, their tensor maps are re-encoded, which also synchronises the
 * device (a step still running on another stream may use the old ones).  The
 * workspace of a new shape list is allocated by the call.  Otherwise the call
 * only enqueues kernels on `stream` and never blocks the host, so after one
 * uncaptured call with the same shapes and weight pointers a step can be
 * captured into a CUDA graph and replayed, with each step's gradients copied
 * into the captured gradient buffers.  Errors: MUON_ERR_NOT_INITIALIZED,
 * MUON_ERR_INVALID_ARG, MUON_ERR_UNSUPPORTED_SHAPE, MUON_ERR_MISALIGNED,
 * MUON_ERR_OUT_OF_MEMORY, MUON_ERR_CUDA.  On an argument error nothing is
 * enqueued.
 */
MUON_API muon_status muon_step(float* const params[], const float* const grads[],
                      float* const momentum_bufs[], const muon_shape shapes[], int n_mats,
                      float lr, float beta, int nesterov, int ns_steps, muon_stream_t stream);

/*
 * One Muon step with NorMuon variance scaling of the orthogonalised update.
 * The apidog.com page (section "2. Pengoptimal Muon", paragraph "Reduksi
 * Varians NorMuon") and the dev.to page ("NorMuon variance scaling") sketch a
 * per-neuron rescale after orthogonalisation; the sketch leaves the reduced
 * dimension, the second-moment state and the new-norm term open.  This library
 * takes: a neuron is a stored row (an output unit), and with O the update of
 * muon_step,
 *   v_mean_i = mean_j O_ij^2 ;  V_i <- beta2 V_i + (1 - beta2) v_mean_i ;
 *   step_i = 1 / sqrt(V_i + eps2) ;
 *   ratio = sqrt(sum_i v_mean_i) / max(sqrt(sum_i v_mean_i step_i^2), 1e-10)
 *   p_ij <- p_ij - lr sqrt(max(1, rows/cols)) step_i ratio O_ij
 * which keeps the Frobenius norm of the update.
 *   second_moments[i]  device float32 array of shapes[i].rows elements, 4-byte
 *                      aligned, caller-owned, updated in place (zero-initialise
 *                      it before the first step)
 *   beta2 in [0, 1), eps2 >= 0; ns_steps >= 1; other arguments as muon_step.
 * O is materialised in a bf16 workspace (one more allocation of half the size
 * of the weights, made by the first call on a shape list), and the row
 * statistics and the update read it from there; the per-row reduction is
 * deterministic.  With MUON_DEBUG_KEEP_O, muon_debug_copy_ns_output
 * returns the scaled update step_i ratio O.  Errors as muon_step.
 */
MUON_API muon_status muon_step_normuon(float* const params[], const float* const grads[],
                                       float* const momentum_bufs[], float* const second_moments[],
                                       const muon_shape shapes[], int n_mats, float lr, float beta, int nesterov,
                                       int ns_steps, float beta2, float eps2, muon_stream_t stream);

/*
 * Ownership of the matrices of a step across `world` data-parallel ranks, for
 * the ZeRO-2-style sharded step the pages describe (apidog.com section
 * "2. Pengoptimal Muon", paragraph "Pelatihan Terdistribusi": reduce-scatter the
 * gradients, each rank updates the matrices it owns, all-gather the weights).
 * Host only (needs no device and no muon_init).  Matrices are assigned largest
 * first, each to the rank with the least Newton-Schulz work so far (work per
 * matrix: 3 m^2 n + m^3 with m <= n its sides; ties go to the lower rank), so
 * the ranks' work differs by at most one matrix's.  owner_out[i] receives the
 * rank of matrix i.  Errors: MUON_ERR_INVALID_ARG (world < 1, n_mats < 0, NULL
 * arrays), MUON_ERR_UNSUPPORTED_SHAPE.
 */
MUON_API muon_status muon_partition(const muon_shape shapes[], int n_mats, int world, int owner_out[]);

/* Free the workspace and the context.  Synchronises the device first. */
MUON_API muon_status muon_destroy(void);

/*
 * Synchronise `stream`, then return and clear the device status word:
 * MUON_OK, MUON_ERR_DEVICE_TIMEOUT or MUON_ERR_DEVICE_BOUNDS (or MUON_ERR_CUDA
 * if the stream itself reports an error).
 */
MUON_API muon_status muon_get_status(muon_stream_t stream);

/* Static English text for a status code (never NULL). */
MUON_API const char* muon_status_string(muon_status s);

/*
 * Counters of the last muon_step: kernel launches it enqueued, workspace bytes,
 * shape classes, and the algorithmic Newton-Schulz flop count
 * (per matrix and iteration 3 m^2 n + m^3 with m <= n the oriented sides).
 */
typedef struct muon_step_info {
    int launches;
    int n_classes;
    long long workspace_bytes;
    double ns_alg_flops;
    double elementwise_alg_bytes;  /* 14 B/elem momentum+norm pass + 8 B/elem weight update */
} muon_step_info;
MUON_API muon_status muon_get_step_info(muon_step_info* out);

/*
 * Host-only planning query (needs no device and no muon_init): validates the
 * shapes exactly as muon_step does and describes the step it would run --
 * oriented shape classes (matrices with equal (min side, max side,
 * transposed) share launches), kernel launches per step, workspace bytes,
 * algorithmic Newton-Schulz flops (3 m^2 n + m^3 per matrix and iteration),
 * executed tensor-core flops of the CTA-pair tiles (axpy: 256 rows, or 128 for
 * the last row pair of a matrix with an odd number of 128-row blocks; Gram and
 * polynomial: 256 x 256 tiles, diagonal ones included, except that with an odd
 * block count each even diagonal block runs alone as a 128 x 128 tile; ragged
 * tiles counted whole), algorithmic elementwise bytes (22 per element),
 * momentum CTAs, and pair tiles per Gram/polynomial launch and per axpy launch.
 * ns_steps is checked against the current context's table (16 rows without one).
 */
typedef struct muon_plan_info {
    int n_classes;
    int launches;
    long long workspace_bytes;
    double ns_alg_flops;
    double ns_executed_flops;
    double elementwise_alg_bytes;
    int momentum_ctas;
    long long sym_tiles;
    long long axpy_tiles;
} muon_plan_info;
MUON_API muon_status muon_plan_query(const muon_shape shapes[], int n_mats, int ns_steps, muon_plan_info* out);

/*
 * Kernel timing (needs MUON_DEBUG_TIME_KERNELS): synchronises on the recorded
 * events and returns, per kernel kind, the summed device milliseconds and the
 * launch count since the previous call, then resets them.  Kinds:
 * 0 momentum+norm, 1 Gram, 2 polynomial, 3 axpy, 4 axpy with fused weight
 * update, 5 standalone weight update (ns_steps == 0), 6 last axpy writing O
 * (NorMuon step), 7 NorMuon row statistics and weight update.  n_kinds <= 8.
 */
MUON_API muon_status muon_kernel_times(double* ms_out, int* launches_out, int n_kinds);

/*
 * Test support.  muon_debug_copy_ns_output copies O of matrix `mat` of the last
 * step (float32, stored rows x cols layout) to the device buffer dst on
 * `stream`; needs MUON_DEBUG_KEEP_O.  muon_debug_copy_norms copies ||u||_F of
 * the first n matrices of the last step to host memory (synchronises).
 */
MUON_API muon_status muon_debug_copy_ns_output(int mat, float* dst_device, muon_stream_t stream);
MUON_API muon_status muon_debug_copy_norms(float* dst_host, int n);

/*
 * AdamW step for the parameters Muon does not take.  The optimizer split of
 * the method ("Train your own ChatGPT" on dev.to, section "2. ตัวปรับปรุง Muon",
 * optimizer table; the apidog.com page, same section) sends 2-D matrices to
 * Muon and embeddings, lm_head and scalar parameters to AdamW.  The pages name
 * AdamW without a formula; this library takes decoupled weight decay with
 * bias-corrected moments, step t >= 1:
 *
 *   p <- p (1 - lr weight_decay)
 *   m <- beta1 m + (1 - beta1) g            (exp_avg)
 *   v <- beta2 v + (1 - beta2) g^2          (exp_avg_sq)
 *   p <- p - (lr / (1 - beta1^t)) m / (sqrt(v / (1 - beta2^t)) + eps)
 *
 * in fp32 (the bias corrections in fp64 on the host).
 *   params[i], grads[i], exp_avg[i], exp_avg_sq[i]: device float32 arrays of
 *     numels[i] elements (any shape, contiguous), 16-byte aligned
 *     (MUON_ERR_MISALIGNED); params, exp_avg, exp_avg_sq are updated in place,
 *     grads are read only; all caller-owned.  numels[i] >= 0 (0 is skipped).
 *   beta1, beta2 in [0, 1); eps >= 0; lr, weight_decay finite; step >= 1.
 * All tensors of a call go into one launch (128 tensors per launch), enqueued
 * on `stream`.  Needs no muon_init; the current device must be sm_103
 * (MUON_ERR_UNSUPPORTED_DEVICE).  Errors: MUON_ERR_INVALID_ARG,
 * MUON_ERR_MISALIGNED, MUON_ERR_UNSUPPORTED_DEVICE, MUON_ERR_CUDA; on an
 * argument error nothing is enqueued.
 */
MUON_API muon_status muon_adamw_step(float* const params[], const float* const grads[], float* const exp_avg[],
                                     float* const exp_avg_sq[], const long long numels[], int n_tensors,
                                     float lr, float beta1, float beta2, float eps, float weight_decay, int step,
                                     muon_stream_t stream);

/*
 * Momentum + norm pass without any allocation.  (The pages have no counterpart:
 * this entry point exists for callers, not for the method.)
 *
 * For callers that cannot call cudaMalloc.  Examples: a process whose device
 * memory is already handed out by another runtime's caching pool, a service
 * that must not allocate (cudaMalloc and cudaFree may synchronise the device
 * and stall other streams) once it is serving, and code running where
 * allocation is forbidden.  It runs the first stage of muon_step on the
 * caller's buffers.  It allocates nothing, needs no muon_init, and keeps its
 * scratch (per-tile norm partials, per-matrix tickets and 1/(||u|| + eps)) in
 * one fixed array inside the library:
 *
 *   m' = beta m + g (stored back into momentum_bufs[i]); EMA form with
 *        momentum_mode MUON_MOMENTUM_EMA, as in muon_step
 *   u  = nesterov ? g + beta m' : m'
 *   x0_out[i]  = bf16(u), round to nearest even, unscaled, in the oriented
 *                layout: rows x cols row-major when rows <= cols, else the
 *                transpose (cols x rows row-major)
 *   norms_out[i] = ||u||_F (fp32, from a fixed-order fp64 sum of per-tile
 *                  fp32 partials, so it is bitwise reproducible)
 *
 * Arguments: grads[i] (read only) and momentum_bufs[i] are device float32
 * rows x cols; x0_out[i] is a device bf16 buffer of rows * cols elements;
 * norms_out is a device float array of n_mats; all are caller-owned, and the
 * matrix pointers must be 16-byte aligned (MUON_ERR_MISALIGNED).  Shapes follow
 * the muon_step rule (MUON_ERR_UNSUPPORTED_SHAPE).  eps <= 0 selects 1e-7; it
 * only enters an internal 1/(||u|| + eps) that this entry point does not return.
 *
 * Limits (MUON_ERR_SCRATCH_LIMIT beyond them, checked before anything is
 * enqueued): n_mats <= 1024, and every group of 192 consecutive matrices
 * covers at most 262144 tiles of 64 x 64 stored elements, i.e. at most about
 * 1.07e9 elements.  The scratch array is about 1.01 MiB of device memory.
 * Every device that loads the library holds it until the process exits.
 *
 * The first call on a device looks up the array's device address with that
 * device current.  Make that first call before any stream capture begins.
 * Later calls only enqueue work.  The address is cached per device together
 * with the ID of the context it was found in; a call made in another context
 * of that device (after cudaDeviceReset, say) looks it up again.  Concurrent
 * first calls from several host threads are safe.  Every call on a device shares the one array:
 * calls whose work overlaps on the GPU (other streams, other host threads)
 * race and give wrong results.  Serialise them, e.g. on one stream.  Each call
 * clears the tickets it uses before its kernel runs.
 * Errors: MUON_ERR_INVALID_ARG, MUON_ERR_UNSUPPORTED_SHAPE, MUON_ERR_MISALIGNED,
 * MUON_ERR_SCRATCH_LIMIT, MUON_ERR_UNSUPPORTED_DEVICE, MUON_ERR_CUDA.
 */
MUON_API muon_status muon_momentum_norm_noalloc(const float* const grads[], float* const momentum_bufs[],
                                                void* const x0_out[], float* norms_out,
                                                const muon_shape shapes[], int n_mats, float beta,
                                                int nesterov, int momentum_mode, double eps,
                                                muon_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MUON_H */
