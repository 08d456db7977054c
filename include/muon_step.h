/*
 * muon_step.h -- C ABI of the GB300 (sm_103a) Muon + AdamW optimizer step.
 *
 * Sources, cited by page title and section:
 *   [OPT] "LLM training series, part 2: optimizers (SGD -> Adam -> AdamW ->
 *         Muon)", mhpq.cn article.
 *   [K2]  "Kimi K2 ... what is worth noting", Zhihu answer by toothacher17.
 *
 * The library is stateless.  Every tensor is owned by the caller; every call
 * only enqueues work on the caller's CUDA stream and returns.  Pointers named
 * "device" must be CUDA device (or managed) memory of the current device;
 * pointers named "host" are ordinary host memory read before the call
 * returns.  Every call that launches kernels first asks the driver who owns
 * each device buffer it is given (one query per allocation) and refuses host
 * memory, another device's memory or an unknown address with
 * MUON_ERR_INVALID_ARG before anything is enqueued; that check is left out
 * while `stream` is being captured into a graph, where only launches are
 * recorded.  No exception crosses this boundary; errors are returned as a
 * muon_status_t and describe host-side validation or launch failures, not
 * asynchronous kernel faults.  `stream` is a cudaStream_t passed as void*
 * (NULL = the legacy default stream).
 *
 * Layout: every matrix is row-major, contiguous, rows x cols = (out, in).
 */
#ifndef MUON_STEP_H
#define MUON_STEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MUON_OK = 0,
    MUON_ERR_INVALID_ARG = 1,          /* null pointer, bad size, bad hparam,
                                          a buffer not on the current device  */
    MUON_ERR_UNSUPPORTED_DTYPE = 2,    /* g_dtype not a muon_dtype_t          */
    MUON_ERR_MISALIGNED = 3,           /* pointer below its element alignment */
    MUON_ERR_WORKSPACE_TOO_SMALL = 4,  /* a single matrix needs more          */
    MUON_ERR_CUDA = 5,                 /* a CUDA runtime call failed          */
    MUON_ERR_TIMEOUT = 6,              /* a kernel gave up on a bounded wait  */
    MUON_ERR_NO_DEVICE = 7,            /* no sm_103 device is current         */
    MUON_STEP_SKIPPED = 8              /* (device status) the non-finite guard
                                          skipped the step; nothing changed   */
} muon_status_t;

/* Gradient element types.  Every one widens to fp32 exactly before the
 * momentum update.  fp16 gradients are those of FP16 mixed-precision
 * training, whose overflow to inf the guard of [OPT] section 5.4 catches. */
typedef enum { MUON_F32 = 0, MUON_BF16 = 1, MUON_F16 = 2 } muon_dtype_t;

/* One hidden weight matrix under Muon.  All three buffers are device memory
 * of rows*cols elements; W and M are fp32 and updated in place, G is read
 * only.  W, M and fp32 G must be 4-byte aligned, bf16 or fp16 G 2-byte aligned;
 * 16-byte alignment enables the vectorised path.  Matrices of one call must
 * not overlap one another. */
typedef struct {
    float* W;          /* device, fp32 master weight                         */
    const void* G;     /* device, gradient, g_dtype                          */
    float* M;          /* device, fp32 momentum buffer                       */
    int64_t rows;      /* > 0                                                */
    int64_t cols;      /* > 0                                                */
    int32_t g_dtype;   /* muon_dtype_t                                       */
    int32_t reserved;  /* must be 0                                          */
} muon_matrix_t;

/* Hyper-parameters of one Muon step, all applied as fp32 values.
 * Defaults of the reference configuration: lr 0.02, weight_decay 0.1,
 * momentum 0.95, nesterov 1, ns_steps 5, (ns_a, ns_b, ns_c) =
 * (3.4445, -4.7750, 2.0315), norm_eps 1e-7, rms_scale 0.2, scale_mode 0,
 * skip_nonfinite 0, max_grad_norm 0, ns_coeffs NULL. */
typedef struct {
    float lr;
    float weight_decay;
    float momentum;    /* mu in [0, 1]                                       */
    int32_t nesterov;  /* 1: Nesterov look-ahead, 0: plain moving average   */
    int32_t ns_steps;  /* Newton-Schulz steps, 0..100                        */
    float ns_a, ns_b, ns_c;
    float norm_eps;    /* added to the Frobenius norm, >= 0                  */
    float rms_scale;   /* scale_mode 0: update = rms_scale sqrt(max(m,n)) O  */
    /* Update scale ([K2] section 3): 0 = rms_scale * sqrt(max(rows, cols)),
     * matching AdamW's update RMS (section 3.1); 1 = max(1, sqrt(rows/cols))
     * = max(1, sqrt(d_out/d_in)), the muP-style adjustment (section 3.2).  */
    int32_t scale_mode;
    /* [OPT] section 5.4, the "Inf guard": 1 = if any gradient element of
     * the call is NaN or +-inf, change nothing (every W and M keeps its old
     * value) and record MUON_STEP_SKIPPED in the workspace status.          */
    int32_t skip_nonfinite;
    /* [OPT] section 5.4, gradient clipping as a safety net: > 0 = scale all
     * gradients of the call by clip = min(1, max_grad_norm / (||G||_global
     * + 1e-6)) (fp64, rounded to fp32; ||G||_global over every element of
     * every matrix of the call) before the momentum update.  <= 0: off.     */
    float max_grad_norm;
    int32_t reserved0; /* must be 0                                          */
    /* NULL: (ns_a, ns_b, ns_c) at every NS step.  Otherwise host memory of
     * 3 * ns_steps floats, step s using (a, b, c) = ns_coeffs[3s..3s+2]
     * (e.g. the page's cubic (1.5, -0.5, 0), [OPT] section 4.2, or a
     * per-step schedule); read before the call returns.                    */
    const float* ns_coeffs;
} muon_hparams_t;

/* One row of the execution plan (see muon_plan). */
typedef struct {
    int32_t mat_idx;     /* index into the caller's matrix array           */
    int32_t transposed;  /* 1 when rows > cols                             */
    int32_t group_id;    /* index of the distinct (m', n') pair            */
    int32_t slot;        /* position within (chunk, group)                 */
    int32_t chunk_id;    /* workspace pass the matrix is processed in      */
    int32_t reserved;
    int64_t mp;          /* m' = min(rows, cols)                           */
    int64_t np;          /* n' = max(rows, cols)                           */
} muon_plan_entry_t;

/* AdamW hyper-parameters, fp32. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} adamw_hparams_t;

/* Workspace bytes one matrix occupies while its chunk is processed:
 *   2 * R(2 * m' * L(n')) + 2 * R(2 * m' * L(m')) + 8192
 * R(x) = x rounded up to 256, L(x) = x rounded up to 8 (two bf16 X buffers
 * of m' x n', the bf16 Gram buffers A = X X^T and B = bA + cA^2 of m' x m',
 * and an 8 KiB record of pointers and norm partial sums).  0 on bad dims. */
size_t muon_workspace_bytes_per_matrix(int64_t rows, int64_t cols);

/* Workspace size for a call: the sum over all matrices when that fits in
 * `budget_bytes` (one chunk), else the largest multiple-chunk requirement,
 * max(budget_bytes, largest single matrix).  *out_bytes receives it. */
muon_status_t muon_workspace_size(const muon_matrix_t* mats, int64_t count,
                                  size_t budget_bytes, size_t* out_bytes);

/* The execution plan for `count` matrices and a workspace of `ws_bytes`
 * (host call; only rows/cols are read).  `out` (host, count entries)
 * receives the matrices in execution order: sorted by (m', n') ascending,
 * ties by caller index; chunks cut greedily so each chunk's summed
 * muon_workspace_bytes_per_matrix <= ws_bytes.  Deterministic.
 * [K2] section 2.2: fine-grained experts make many small matrices, which
 * the grouped launches batch by shape. */
muon_status_t muon_plan(const muon_matrix_t* mats, int64_t count,
                        size_t ws_bytes, muon_plan_entry_t* out);

/* One Muon step on `count` matrices (host array `mats`), enqueued on
 * `stream`.  For every matrix, with m' = min(rows, cols), n' = max:
 *   M  = mu M + (1-mu) G                       ([OPT] section 2.1)
 *   u  = (1-mu) G + mu M    (nesterov = 1; u = M when 0)
 *   X0 = bf16(u), transposed to m' x n' when rows > cols;  s = 1/(||u||_F + eps)
 *   ns_steps times, starting from X = s X0 (s applied in fp32 inside the
 *   first step, never stored):  A = X X^T;  B = b A + c A A;  X = a X + B X
 *                    (bf16 storage, fp32 accumulation; [OPT] section 4.2)
 *   W  = W - lr (wd W + rms_scale sqrt(n') O),  O = final X in W's layout
 *        (decoupled decay on the old W, [OPT] section 3.1; RMS matched to
 *        AdamW's 0.2-0.4, [K2] section 3.1)
 * `workspace` is device memory of `ws_bytes` (>= the largest single
 * matrix's muon_workspace_bytes_per_matrix), 256-byte aligned; it must not
 * be used by other work until the step has finished on `stream`.
 * count == 0 is a no-op.  A kernel that gives up on a bounded wait records
 * MUON_ERR_TIMEOUT in the workspace; read it with muon_query_status.
 * The call enqueues kernels only (no memset, no host<->device copy, no
 * synchronisation; its first kernel clears the workspace status), so it may
 * run inside a CUDA stream capture once one call has run on the device
 * outside a capture (the first call sets kernel attributes);
 * muon_step_graph_create needs no such call.  Its kernels are chained by
 * programmatic dependent launch: each waits for the one ahead of it before
 * it touches memory, so work the caller enqueues before or after the call
 * on the same stream is ordered with it as usual. */
muon_status_t muon_step_batched(const muon_matrix_t* mats, int64_t count,
                                const muon_hparams_t* hp, void* workspace,
                                size_t ws_bytes, void* stream);

/* Per-matrix statistics of one step (no counterpart in the update itself;
 * the closing notes of [OPT], after section 5.4, advise logging numerical
 * statistics of the optimizer state to see trouble before the loss does;
 * these are the Muon step's own: the norm it divides by and the RMS it
 * matches).  fp64:
 *   u_norm      ||u||_F, the Frobenius norm of the look-ahead the step
 *               normalised: sqrt of the sum of the momentum pass's fp32
 *               tile sums of u^2, summed in fp64
 *   update_rms  sqrt(sum fl(scale * O)^2 / (rows * cols)), the RMS of the
 *               RMS-matched update before lr and decay ([K2] section 3.1:
 *               about 0.2, in AdamW's 0.2-0.4 band, with scale_mode 0);
 *               each square in fp32, tile sums in fp32, summed in fp64
 * Both are NaN for every matrix when the non-finite guard skipped the step. */
typedef struct {
    double u_norm;
    double update_rms;
} muon_matrix_stats_t;

/* muon_step_batched plus per-matrix statistics: `stats` is device memory of
 * `count` entries, 8-byte aligned, entry i for mats[i], written on `stream`
 * during the step.  Costs one extra read of each matrix's NS output (2 bytes
 * per element) and two launches per workspace chunk.  Same arguments,
 * checks and errors as muon_step_batched; a null `stats` is
 * MUON_ERR_INVALID_ARG, a misaligned one MUON_ERR_MISALIGNED. */
muon_status_t muon_step_batched_stats(const muon_matrix_t* mats, int64_t count,
                                      const muon_hparams_t* hp, void* workspace,
                                      size_t ws_bytes, muon_matrix_stats_t* stats,
                                      void* stream);

/* Size of the library-owned device scratch used by muon_step_batched_noalloc:
 * 64 MiB on every GPU where the library's device code is loaded, held until
 * the process exits. */
#define MUON_STATIC_SCRATCH_BYTES (64u << 20)

/* The same Muon step as muon_step_batched, for callers that cannot allocate
 * device memory (e.g. an optimizer plug-in inside a framework that owns all
 * device memory through its own pool, or a C caller with no device
 * allocator): the workspace is a static device array inside the library,
 * so this call allocates nothing -- no cudaMalloc, no cudaFree, no
 * allocating library routine.  The pages have no counterpart; it is an
 * interface variant of the step above.  The caller still passes every
 * W, G, M buffer.
 *   - every matrix must fit the scratch on its own:
 *     muon_workspace_bytes_per_matrix(rows, cols) <= MUON_STATIC_SCRATCH_BYTES
 *     (e.g. up to 2048 x 5632), else MUON_ERR_WORKSPACE_TOO_SMALL and
 *     nothing is enqueued; larger call lists run in several passes;
 *   - the first call on a device resolves the scratch's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it for
 *     the life of the process; make that first call before any stream
 *     capture, and do not call this entry point again in a process that
 *     has reset the device (cudaDeviceReset), whose kept address is stale;
 *   - all calls on a device share the one scratch, which keeps the previous
 *     call's contents (the step rewrites everything it reads, and clears its
 *     status word itself): calls that overlap on the GPU (other streams,
 *     other threads) race and must be serialised by the caller;
 *   - the status word of a timed-out wait lands in the scratch, which the
 *     caller cannot address: muon_query_status does not apply. */
muon_status_t muon_step_batched_noalloc(const muon_matrix_t* mats, int64_t count,
                                        const muon_hparams_t* hp, void* stream);

/* ---- The step as a CUDA graph (no counterpart on the pages) ------------- */

/* muon_step_batched enqueues only kernels (the per-matrix records travel as
 * kernel parameters), so a caller may capture it into a
 * CUDA graph of its own.  The calls below do that for the caller.
 *
 * A captured step replays the whole launch sequence of one
 * muon_step_batched call with everything the call read fixed at capture:
 * the W, G, M and workspace addresses, the shapes, the plan and the
 * hyper-parameters (lr, weight decay, momentum, NS coefficients, guard
 * settings).  Each replay reads the current contents of G and updates W and
 * M in place, like the eager call; to change a hyper-parameter, capture
 * again.  Replays on one workspace must not overlap on the GPU. */
typedef struct muon_graph_s* muon_graph_t;

/* Captures one muon_step_batched call with these arguments (same meaning,
 * same checks and errors) into a graph and instantiates it; *out receives
 * the handle, NULL on failure.  Nothing runs on the GPU.  Must be called
 * with the device that holds the buffers current.  Host memory the call
 * reads (mats, hp, hp->ns_coeffs) may be freed when it returns; the device
 * buffers must outlive the handle.  count == 0 gives a handle whose launch
 * is a no-op. */
muon_status_t muon_step_graph_create(const muon_matrix_t* mats, int64_t count,
                                     const muon_hparams_t* hp, void* workspace,
                                     size_t ws_bytes, muon_graph_t* out);

/* Enqueues one replay of the captured step on `stream` (a stream of the
 * device the graph was created on).  MUON_ERR_INVALID_ARG on a NULL
 * handle, MUON_ERR_CUDA if the launch fails. */
muon_status_t muon_step_graph_launch(muon_graph_t graph, void* stream);

/* Frees the graph (host and driver objects; no device buffer of the
 * caller's).  Replays already enqueued still run.  NULL is a no-op. */
muon_status_t muon_step_graph_destroy(muon_graph_t graph);

/* Newton-Schulz alone on a batch of `count` wide bf16 matrices (device,
 * [count][mp][np] row-major, bf16 bit patterns, mp <= np), writing the
 * result to X_out (same layout; may not alias X_in):
 *   for s < ns_steps: A = X X^T; B = b A + c A A; X = a X + B X
 * ([OPT] section 4.2) with (a, b, c) = coeffs[0..2] at every step when
 * ncoeff_sets == 1, or coeffs[3s..3s+2] when ncoeff_sets == ns_steps
 * (host memory, read before the call returns).
 * workspace: device, >= muon_workspace_bytes_per_matrix(mp, np) (larger
 * batches run in several passes), 256-byte aligned.  X_in and X_out must
 * be 2-byte aligned. */
muon_status_t muon_newton_schulz(const uint16_t* X_in, uint16_t* X_out,
                                 int64_t count, int64_t mp, int64_t np,
                                 int32_t ns_steps, const float* coeffs,
                                 int32_t ncoeff_sets, void* workspace,
                                 size_t ws_bytes, void* stream);

/* AdamW on flat fp32 device buffers of n elements, in place on p, m, v
 * ([OPT] sections 2.3 and 3.1), step >= 1:
 *   bc1 = 1 - beta1^step, bc2 = 1 - beta2^step   (fp64 on the host -> fp32)
 *   m = beta1 m + (1-beta1) g;  v = beta2 v + (1-beta2) g*g
 *   p = p - lr ( (m/bc1) / (sqrt(v/bc2) + eps) + wd p )
 * every operation a separately rounded fp32 op in that order (no fused
 * multiply-add).  Buffers must be 4-byte aligned and must not overlap;
 * 16-byte alignment enables the vectorised path.  n == 0 is a no-op. */
muon_status_t adamw_step(float* p, const float* g, float* m, float* v,
                         int64_t n, const adamw_hparams_t* hp, int64_t step,
                         void* stream);

/* One tensor of a multi-tensor AdamW step: n fp32 elements in each of four
 * device buffers (any shape, contiguous), p, m, v updated in place. */
typedef struct {
    float* p;
    const float* g;
    float* m;
    float* v;
    int64_t n;
} adamw_tensor_t;

/* AdamW on `count` tensors (host array) with one set of hyper-parameters
 * and one step count: every tensor is updated exactly as adamw_step would
 * update it, bit for bit, in one launch per 448 tensors.  The rest of the
 * parameters besides Muon's matrices -- embedding, LM head, norm gains and
 * biases ([OPT] section 4.3) -- are many tensors, most of them small.
 *   - each tensor follows adamw_step's rules (4-byte aligned buffers, its
 *     four buffers disjoint); 16-byte alignment of all four enables the
 *     vector path for that tensor;
 *   - no buffer of one tensor may overlap a buffer of another;
 *   - n == 0 tensors are skipped; count == 0 is a no-op.
 * Errors as adamw_step's; nothing is enqueued when one tensor fails a check.
 * A launch error (MUON_ERR_CUDA) after the first launch leaves the tensors
 * of the launches already enqueued (whole groups of 448, in array order)
 * updated and the rest untouched; the call does not say which.
 * Like adamw_step, it enqueues kernels only (the tensor table travels as
 * kernel parameters), so a caller may capture it in a CUDA graph. */
muon_status_t adamw_step_batched(const adamw_tensor_t* tensors, int64_t count,
                                 const adamw_hparams_t* hp, int64_t step, void* stream);

/* Failure-detection self-check (no counterpart on the pages).  Enqueues on
 * `stream` one thread that waits, through the same bounded mbarrier wait as
 * the Newton-Schulz kernels, on a barrier nothing ever arrives on.  After
 * `limit_us` microseconds (1 .. 10^7) the wait gives up: it records
 * MUON_ERR_TIMEOUT in the status word of `workspace` (device, >= 256 bytes,
 * 256-byte aligned; the word is cleared first) and the kernel returns, so
 * the context stays usable.  Read the result with muon_query_status.
 * Returns MUON_OK once the check is enqueued. */
muon_status_t muon_check_bounded_wait(void* workspace, int64_t limit_us, void* stream);

/* Synchronises `stream`, reads and clears the status word a step left in
 * `workspace`; returns MUON_OK or what was recorded (MUON_ERR_TIMEOUT,
 * MUON_STEP_SKIPPED). */
muon_status_t muon_query_status(void* workspace, void* stream);

/* ---- Instrumentation (no counterpart on the pages) --------------------- */

/* Kernel kinds the library launches. */
typedef enum {
    MUON_KERNEL_MOMENTUM_NORM = 0,  /* momentum, look-ahead, sum of squares */
    MUON_KERNEL_NORM_FINALIZE = 1,  /* per-matrix norm scale                */
    MUON_KERNEL_X0_RESCALE = 2,     /* X0 rescale for out-of-range norms    */
    MUON_KERNEL_NS_SYRK = 3,        /* A = X X^T                            */
    MUON_KERNEL_NS_POLY = 4,        /* B = b A + c A A                      */
    MUON_KERNEL_NS_UPDATE = 5,      /* X = a X + B X                        */
    MUON_KERNEL_FINAL_UPDATE = 6,   /* W -= lr (wd W + scale O)             */
    MUON_KERNEL_ADAMW = 7,          /* AdamW                                */
    MUON_KERNEL_GRAD_GUARD = 8,     /* global gradient norm / non-finite    */
    MUON_KERNEL_DESC_UPLOAD = 9,    /* per-matrix records into the workspace */
    MUON_KERNEL_STATS = 10,         /* per-matrix step statistics           */
    MUON_KERNEL_COUNT = 11
} muon_kernel_kind_t;

/* Process-wide count of kernels this library has launched (all kinds); a
 * graph replay adds the number of kernels its capture enqueued.  Launches
 * made while a graph is captured are not counted. */
int64_t muon_launch_count(void);

/* enable != 0: from now on every launch is bracketed by two CUDA events
 * recorded on its stream (library-owned events; the launches themselves are
 * unchanged); launches inside muon_step_graph_create's capture and graph
 * replays are not timed.  Enabling or disabling drops the records collected
 * so far. */
muon_status_t muon_set_timing(int32_t enable);

/* Waits for the recorded events, writes the summed milliseconds and the
 * number of launches per muon_kernel_kind_t into the host arrays (nkinds
 * entries, kinds beyond MUON_KERNEL_COUNT get 0) and drops the records. */
muon_status_t muon_timing_read(double* ms_per_kind, int64_t* launches_per_kind,
                               int32_t nkinds);

/* Static name of a kernel kind ("ns_update", ...). */
const char* muon_kernel_name(int32_t kind);

/* Static description of a status code. */
const char* muon_status_string(muon_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t muon_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MUON_STEP_H */
