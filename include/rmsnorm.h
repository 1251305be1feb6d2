/*
 * rmsnorm.h — C ABI of the GB300 (sm_103a) RMSNorm forward library
 * (librmsnorm_gb300.so).
 *
 * The operation. For a row-major activation x[M, N] and a weight w[N]:
 *
 *   rstd[i] = 1 / sqrt( (1/N) * sum_{j<N} x[i,j]^2 + eps )          (fp32)
 *   y[i,j]  = dtype( (x[i,j] * rstd[i]) * (offset + w[j]) )
 *
 * with offset 0 for Llama-style weights and 1 for Gemma-style weights.
 * Defined by the kernel listing of "Why cutile's rmsnorm required full
 * register" (TileGym issue #169): x is widened to fp32 before squaring, the
 * row sum of squares is divided by the true N, eps is added inside the rsqrt,
 * the fp32 rstd is stored "for backward", the normalised row is scaled by
 * (offset + w) in fp32 and cast once to x's dtype (the listing's cast to the
 * dtype of X, whatever that dtype is: bf16, fp16 or fp32). The same formula, with
 * offset 0, is the Overview and Verification formula of "RMSNorm Kernel
 * Optimization" (skillmd): out = x / sqrt(mean(x^2) + eps) * weight.
 * Arithmetic is fp32 throughout (sum of squares, mean, rsqrt, products); y is
 * rounded to nearest-even once (for fp32 y, the products are fp32 products).
 * Results are deterministic: the same inputs and
 * launch shape always give the same bits.
 *
 * Memory. Every pointer is a DEVICE pointer on the calling thread's current
 * CUDA device (cudaSetDevice), allocated by the caller, except the host
 * buffers of rmsnorm_fwd_host(). The library never allocates or frees caller
 * memory, copies it only in rmsnorm_fwd_host(), and never synchronises except
 * in rmsnorm_check_device_status().
 *   x     [M, N] bf16, fp16 or fp32, contiguous row-major (row i at x + i*N)
 *   w     [N]    same dtype as x
 *   y     [M, N] same dtype as x; may equal x exactly (in place), must not
 *                otherwise overlap x, w or rstd
 *   rstd  [M]    fp32; must not overlap x, w or y; may be NULL (inference:
 *                rstd is then not stored)
 * rmsnorm_fwd_strided() takes row strides instead (row i of x at x + i*ldx,
 * of y at y + i*ldy, in elements, each >= N), for rows that are slices of
 * wider tensors; the overlap rules then apply to the spans from the first to
 * the last element of each array.
 * x, w, y need only their element alignment (2 bytes; 4 for fp32) and rstd
 * 4 bytes. 16-byte-aligned x, w, y whose rows are whole 16-byte vectors (N a
 * multiple of 8; of 4 for fp32) take the vectorised kernels; anything else
 * takes the general kernel.
 *
 * Streams and errors. Work is enqueued on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and the call returns at once. Kernels are launched
 * with programmatic dependent launch allowed: a kernel may be scheduled while
 * the previous kernel on the stream finishes, but it touches no memory before
 * that kernel has completed, so stream order is kept. The return value
 * reports argument errors (checked on the host before any CUDA call) and launch
 * errors only. Kernels with bounded waits record a timeout in a per-device
 * status word instead of hanging; rmsnorm_check_device_status() reads it.
 * Calls are thread-safe. rmsnorm_last_error() gives a detail string for the
 * last failed call on the calling thread.
 */
#ifndef RMSNORM_GB300_H
#define RMSNORM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RMSNORM_GB300_VERSION 1

typedef enum rmsnorm_dtype {
    RMSNORM_DTYPE_BF16 = 0,
    RMSNORM_DTYPE_FP16 = 1,
    RMSNORM_DTYPE_FP32 = 2
} rmsnorm_dtype_t;

typedef enum rmsnorm_status {
    RMSNORM_OK = 0,
    RMSNORM_ERR_NULL = -1,           /* a required pointer is NULL */
    RMSNORM_ERR_SHAPE = -2,          /* M < 0, N <= 0, or x larger than 2^48 bytes */
    RMSNORM_ERR_DTYPE = -3,          /* dtype is not an rmsnorm_dtype_t value */
    RMSNORM_ERR_SCALAR = -4,         /* eps negative or not finite, or offset not finite */
    RMSNORM_ERR_EPS = -4,            /* the same code under the name of the eps check */
    RMSNORM_ERR_OVERLAP = -5,        /* buffers overlap other than y == x exactly */
    RMSNORM_ERR_CUDA = -6,           /* a CUDA runtime call or launch failed */
    RMSNORM_ERR_DEVICE_TIMEOUT = -7, /* a kernel's bounded wait ran out (see rmsnorm_check_device_status) */
    RMSNORM_ERR_UNSUPPORTED = -8,    /* the forced variant cannot take these arguments */
    RMSNORM_ERR_OPTIONS = -9,        /* malformed rmsnorm_options_t */
    RMSNORM_ERR_ALIGN = -10,         /* x, w or y not aligned to their element size, or rstd not
                                        4-byte aligned */
    RMSNORM_ERR_WORKSPACE = -11      /* the backward's workspace is smaller than it needs */
} rmsnorm_status_t;

/* Kernel variants. RMSNORM_VARIANT_AUTO lets the planner choose. */
typedef enum rmsnorm_variant {
    RMSNORM_VARIANT_AUTO = 0,
    /* A team of 1..32 lanes of one warp per row, row held in registers,
     * several rows per warp when N is small (warp-per-row and
     * multi-row-per-warp). Needs 16-byte alignment and rows of whole 16-byte
     * vectors, at most 2 KB per row (N <= 1024 bf16/fp16, 512 fp32). */
    RMSNORM_VARIANT_WARP = 1,
    /* One CTA per row, row held in registers across the CTA, cross-warp sum
     * through shared memory. Needs 16-byte alignment and rows of whole 16-byte
     * vectors, at most 64 KB per row (N <= 32768 bf16/fp16, 16384 fp32). */
    RMSNORM_VARIANT_CTA = 2,
    /* Rows staged in shared memory by TMA bulk copies (cp.async.bulk with an
     * mbarrier), multi-stage pipeline, bounded waits. Needs 16-byte alignment
     * and rows of whole 16-byte vectors; rows up to the shared-memory limit. */
    RMSNORM_VARIANT_TMA = 3,
    /* Any alignment and any N: one CTA per row, two passes over the row. */
    RMSNORM_VARIANT_GENERIC = 4,
    /* Rows longer than one CTA's shared memory: a row split over a thread-block
     * cluster of 2..16 CTAs, each staging its column slice by TMA bulk copy; the
     * slice sums meet through distributed shared memory. Needs 16-byte alignment
     * and rows of whole 16-byte vectors; rows up to 16 slices of about 70 KB. */
    RMSNORM_VARIANT_CLUSTER = 5
} rmsnorm_variant_t;

/* Optional knobs for rmsnorm_fwd_ex(). Zero-initialise, then set fields. */
/* rmsnorm_options_t.flags bits. */
#define RMSNORM_FLAG_NO_PDL 1       /* launch without programmatic dependent launch */
#define RMSNORM_FLAG_BLOCKED_ROWS 2 /* each CTA takes one contiguous block of rows
                                       (default: CTAs stride over rows in passes) */
/* The caller promises that no kernel still running earlier on the stream
 * writes x or w. The kernel may then start reading them while the previous
 * kernel finishes (overlapping launches); its writes of y and rstd still wait
 * for that kernel to complete. Without the promise every read and write waits
 * (the kernel may still ask for its first rows of x to be brought into L2
 * before it waits: a hint that returns no values, see prewait_prefetch).
 * Ignored with RMSNORM_FLAG_NO_PDL and by the general kernel. */
#define RMSNORM_FLAG_EARLY_LOADS 4
/* The caller promises only that no kernel still running earlier on the stream
 * writes w (a weight that is not being updated, as in inference); x may be
 * the previous kernel's output. The kernel then reads w before the previous
 * kernel finishes and waits only before reading x, taking the weight load off
 * the critical path of a chain of dependent kernels. Ignored with
 * RMSNORM_FLAG_NO_PDL and by the general kernel; implied by EARLY_LOADS. */
#define RMSNORM_FLAG_EARLY_WEIGHTS 16
/* TMA variant with packed rows: y is written into the shared-memory stage and
 * leaves with one bulk copy (cp.async.bulk shared -> global) per stage instead
 * of per-thread stores. Ignored by the other variants and for strided rows. */
#define RMSNORM_FLAG_BULK_STORE 32
/* rmsnorm_fwd_host only: no ring and no copies; the kernel reads x and writes
 * y and rstd in page-locked host memory through their device addresses (the
 * GPU's own loads and stores cross the host link). Needs every host buffer to
 * be page-locked (cudaHostAlloc / cudaHostRegister), else
 * RMSNORM_ERR_UNSUPPORTED; takes no workspace; only the plain-load kernels
 * (WARP, CTA, GENERIC) run. Ignored by the device-memory calls. */
#define RMSNORM_FLAG_HOST_DIRECT 8

typedef struct rmsnorm_options {
    int32_t struct_size;     /* sizeof(rmsnorm_options_t) */
    int32_t variant;         /* rmsnorm_variant_t; 0 = automatic */
    int32_t max_ctas;        /* >0 caps the persistent grid; 0 = SMs x resident CTAs */
    int32_t lanes_per_row;   /* WARP: lanes per row (1..32, power of two); CTA: threads per
                                row (= per CTA); TMA: threads per row (16..1024);
                                GENERIC: threads per CTA; 0 = planner's choice */
    int32_t stages;          /* WARP: rows each team keeps in flight (1, 2 or 4); TMA: pipeline
                                depth (1..8); CLUSTER: 1..4; 0 = planner's choice */
    int32_t rows_per_stage;  /* TMA: rows per stage; 0 = planner's choice */
    int32_t flags;           /* RMSNORM_FLAG_* bits */
    int32_t cluster_size;    /* CLUSTER: CTAs per row (2..16); 0 = planner's choice */
    int64_t wait_limit_ns;   /* TMA: bound on each mbarrier wait in ns; 0 = 1 second */
    int32_t l2_prefetch;     /* WARP and TMA: L2 prefetch distance (a hint: cp.async.bulk.
                                prefetch.L2, no effect on results). WARP: each team asks
                                for its rows this many passes past the ones held in
                                registers to be brought into L2; TMA: each CTA, for this
                                many chunks past its ring's stages (packed rows; not in
                                the 512-thread plans nor fp16 plans of 128-thread teams
                                and up, where it reads 0). Ignored by the other variants
                                and by rmsnorm_bwd. 1..15; 0 = planner's choice; -1 = none */
    int32_t prewait_prefetch; /* WARP and TMA: before it waits for the previous kernel on
                                the stream, the kernel asks for its first rows to be brought
                                into L2 (cp.async.bulk.prefetch.L2, a hint: x is still read
                                after the wait, so the stream order is kept) and the WARP
                                kernel lets the next kernel be scheduled at once. WARP: this
                                many passes of each team's rows; TMA: this many chunks of
                                each CTA's. Under RMSNORM_FLAG_EARLY_LOADS a positive count
                                (or the planner, for the shapes where it measured faster)
                                replaces the loads before the wait with it; -1 keeps them.
                                rmsnorm_bwd: the warp and CTA row kernels prefetch this many
                                of their first rows of x and dy (default 1). Ignored by the
                                other variants. With RMSNORM_FLAG_NO_PDL the planner never
                                picks it and the forward TMA kernel ignores a count.
                                1..15; 0 = planner's choice; -1 = none */
} rmsnorm_options_t;

/* What the planner picked (rmsnorm_plan_info). */
typedef struct rmsnorm_plan {
    int32_t variant;         /* rmsnorm_variant_t actually launched */
    int32_t threads;         /* threads per CTA */
    int32_t grid;            /* CTAs launched (persistent grid) */
    int32_t lanes_per_row;   /* threads cooperating on one row */
    int32_t vecs_per_lane;   /* 16-byte vectors each thread holds per row (0: general kernel) */
    int32_t rows_per_stage;  /* TMA variant: rows per shared-memory stage (else 0) */
    int32_t stages;          /* TMA variant: pipeline depth (else 0) */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t ctas_per_sm;     /* resident CTAs per SM (occupancy calculator) */
    int32_t sm_count;        /* SMs on the device */
    int32_t cluster_size;    /* CTAs per cluster (cluster variant; else 0) */
    int32_t l2_prefetch;     /* L2 prefetch distance in use (WARP, TMA; 0 = none) */
    int32_t prewait_prefetch; /* pre-wait L2 prefetch in use (WARP passes, TMA chunks; 0 =
                                none); when positive, x is read only after the wait */
} rmsnorm_plan_t;

/*
 * RMSNorm forward: y = x * rsqrt(mean(x^2) + eps) * (offset + w), rstd kept.
 *   x, w, y, rstd  device pointers as described above (x and y may be NULL
 *                  when M == 0, rstd may always be NULL; w must not be NULL)
 *   M              rows (>= 0; M == 0 launches nothing and returns RMSNORM_OK)
 *   N              columns (> 0)
 *   eps            >= 0 and finite; added to the mean of squares inside the root
 *   offset         finite; 0 = Llama, 1 = Gemma
 *   dtype          rmsnorm_dtype_t of x, w and y
 *   stream         cudaStream_t to enqueue on (NULL = legacy default stream)
 * Returns RMSNORM_OK or a negative rmsnorm_status_t; on error nothing is
 * launched and rmsnorm_last_error() says why.
 */
int rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N,
                float eps, float offset, int dtype, void* stream);

/* rmsnorm_fwd with explicit options (variant choice, grid cap, pipeline depth,
 * wait bound). `opts` may be NULL (same as rmsnorm_fwd). */
int rmsnorm_fwd_ex(const void* x, const void* w, void* y, float* rstd, int64_t M, int64_t N,
                   float eps, float offset, int dtype, const rmsnorm_options_t* opts,
                   void* stream);

/* rmsnorm_fwd_ex over strided rows: row i of x starts at element i*ldx, row i
 * of y at element i*ldy (ldx, ldy >= N; in place needs y == x and ldy == ldx).
 * The vectorised kernels additionally need ldx and ldy to be multiples of 8;
 * other strides take the general kernel. Same operation and errors as
 * rmsnorm_fwd; RMSNORM_ERR_SHAPE if a stride is below N. */
int rmsnorm_fwd_strided(const void* x, int64_t ldx, const void* w, void* y, int64_t ldy,
                        float* rstd, int64_t M, int64_t N, float eps, float offset, int dtype,
                        const rmsnorm_options_t* opts, void* stream);

/*
 * The forward over activations in HOST memory. The pages' kernels take device
 * tensors and have no counterpart for this; it is the library's data path for
 * activations that live in host memory (offloaded or served from host RAM).
 * Same operation and arguments as rmsnorm_fwd_ex, except:
 *   x_host, y_host  [M, N] contiguous, in host memory (pinned with
 *                   cudaHostAlloc/cudaHostRegister for the copies to run
 *                   asynchronously and overlap; pageable memory is correct but
 *                   slower); y_host may equal x_host exactly
 *   rstd_host       [M] fp32 in host memory, or NULL
 *   w               [N] DEVICE pointer (weights stay resident)
 *   chunk_rows      rows moved per chunk (> 0), or 0 for about 4 MiB of x
 *   workspace       DEVICE memory, 16-byte aligned, of workspace_bytes >=
 *                   rmsnorm_fwd_host_workspace_size(M, N, dtype, chunk_rows);
 *                   owned by the caller, used by this call until it completes
 *                   on `stream`, and not to be shared with work running at the
 *                   same time
 * Unless RMSNORM_FLAG_HOST_DIRECT is set (see there; then the workspace may be
 * NULL), rows move in chunks through a ring of up to four slots of the workspace:
 * host->device copies of x on a copy-in stream, the forward kernel in place on
 * each slot on `stream`, device->host copies of y and rstd on a copy-out
 * stream, chained by events. The two copy streams are the library's, one pair
 * per device (made on first use, with that device current, and kept for the
 * life of the process). Both directions of the host link thus run at once.
 * The copy-in stream first waits for the work already on `stream`, and before
 * returning `stream` is made to wait for the last copy-out, so work enqueued
 * on `stream` after this call sees y and rstd in host memory; the host must
 * not read them before that work (or a stream synchronisation) completes.
 * RMSNORM_FLAG_EARLY_LOADS is ignored.
 * Errors: as rmsnorm_fwd_ex, plus RMSNORM_ERR_NULL (workspace), _ALIGN
 * (workspace), _WORKSPACE (too small), _OVERLAP (workspace against x, y, rstd
 * or w), _CUDA. Argument errors are found before anything is enqueued.
 */
int rmsnorm_fwd_host(const void* x_host, const void* w, void* y_host, float* rstd_host, int64_t M,
                     int64_t N, float eps, float offset, int dtype, int64_t chunk_rows,
                     void* workspace, int64_t workspace_bytes, const rmsnorm_options_t* opts,
                     void* stream);

/* Device workspace bytes rmsnorm_fwd_host needs for these sizes and chunk rows
 * (written to *bytes; 0 when M == 0). No CUDA call. */
int rmsnorm_fwd_host_workspace_size(int64_t M, int64_t N, int dtype, int64_t chunk_rows,
                                    int64_t* bytes);

/* Fills *out with the launch rmsnorm_fwd_ex would make for these arguments on
 * the current device (no launch). x, w, y are used only for their alignment
 * and may be any values with the alignment the real call will have. */
int rmsnorm_plan_info(int64_t M, int64_t N, int dtype, const void* x, const void* w,
                      const void* y, const rmsnorm_options_t* opts, rmsnorm_plan_t* out);

/*
 * Backward, consuming the rstd the forward kept. The pages state only that
 * rstd is kept "for backward"; the formulas are the chain rule of the forward
 * above (s_j = offset + w_j):
 *   c_i   = sum_j dy[i,j] * s_j * x[i,j]
 *   dx    = rstd[i] * (dy[i,j] * s_j - x[i,j] * rstd[i]^2 * c_i / N)   (x's dtype)
 *   dw[j] = sum_i dy[i,j] * x[i,j] * rstd[i]                              (fp32)
 * fp32 arithmetic; dx rounded once to nearest even; dw summed per CTA over its
 * rows, then over CTAs in a fixed order (deterministic for a fixed device).
 * The sum over CTAs is a second launch.
 *   x, dy, dx  [M, N] x's dtype (bf16, fp16 or fp32), contiguous; dx may equal
 *              x or dy exactly
 *   w          [N]    x's dtype
 *   rstd       [M]    fp32, as written by rmsnorm_fwd
 *   dw         [N]    fp32 output (overwritten; zero when M == 0)
 *   workspace  device scratch of at least rmsnorm_bwd_workspace_size() bytes,
 *              16-byte aligned, owned by the caller; its contents are
 *              overwritten. Calls sharing one workspace must not overlap on
 *              the GPU (one stream, or ordered streams).
 * With N % 8 == 0 and 16-byte aligned buffers, rows of up to 1024 columns take
 * a warp-per-row kernel and rows of up to 16384 columns a CTA-per-row kernel
 * (variant TMA: rows of up to 16 KB staged into shared memory by bulk copies,
 * bounded waits as in the forward, reported by rmsnorm_check_device_status);
 * others the general kernel, which keeps a CTA's dw partial row in shared memory
 * up to about 56K columns and, past that, in its own row of the workspace (any
 * N; the grid is then capped so that the partial rows stay within 64 MB).
 * Options: variant AUTO, WARP, CTA or GENERIC, lanes_per_row (CTA: threads per
 * CTA), max_ctas, RMSNORM_FLAG_NO_PDL, and
 * RMSNORM_FLAG_EARLY_LOADS, which here is the caller's promise that no kernel
 * still running earlier on the stream writes x, w or rstd (dy may be that
 * kernel's output, as in a chain of backward kernels): the warp and CTA
 * kernels then read the weights and their first row's x and rstd before that
 * kernel completes, and dy and every store only after it.
 */
int rmsnorm_bwd(const void* x, const void* w, const float* rstd, const void* dy, void* dx,
                float* dw, int64_t M, int64_t N, float offset, int dtype, void* workspace,
                int64_t workspace_bytes, const rmsnorm_options_t* opts, void* stream);

/*
 * rmsnorm_bwd without a workspace; allocates nothing. (The pages have no
 * counterpart: this entry point exists for callers, not for the method.)
 * Some callers cannot allocate device memory at the point of the call: a
 * plugin inside a host framework that owns every device allocation, or a
 * real-time path whose memory plan is fixed at start-up. Here the dw partials
 * go to a fixed 8 MiB fp32 array built into the library, which every GPU that
 * loads the library holds until the process exits. The grid is capped so that
 * grid * N fits in it; N above 2^21 is rejected with RMSNORM_ERR_WORKSPACE.
 * The first call on a device looks up the array's device address (a CUDA
 * runtime call, with that device current); make that first call before any
 * stream capture. All calls on a device share the array, and each call
 * overwrites the part it uses before reading it, so nothing carries over
 * between calls; calls that overlap on the GPU (concurrent streams) race on it.
 * Same arguments as rmsnorm_bwd otherwise; callers who can allocate should
 * prefer rmsnorm_bwd.
 */
int rmsnorm_bwd_noalloc(const void* x, const void* w, const float* rstd, const void* dy, void* dx,
                        float* dw, int64_t M, int64_t N, float offset, int dtype,
                        const rmsnorm_options_t* opts, void* stream);

/* Fills *out with the launch of the row kernel rmsnorm_bwd would make for
 * these sizes and options on the current device with 16-byte aligned buffers
 * (no launch); variant is RMSNORM_VARIANT_WARP, _CTA, _TMA or _GENERIC. */
int rmsnorm_bwd_plan_info(int64_t M, int64_t N, int dtype, const rmsnorm_options_t* opts,
                          rmsnorm_plan_t* out);

/* Bytes of workspace rmsnorm_bwd needs for these sizes and options on the
 * current device, for any buffer alignment (written to *bytes). */
int rmsnorm_bwd_workspace_size(int64_t M, int64_t N, int dtype, const rmsnorm_options_t* opts,
                               int64_t* bytes);

/* Synchronises `stream`, then reads and clears the current device's status
 * word. Returns RMSNORM_OK, RMSNORM_ERR_DEVICE_TIMEOUT if any kernel since the
 * last check gave up a bounded wait, or RMSNORM_ERR_CUDA. */
int rmsnorm_check_device_status(void* stream);

/* Static text for a status code. */
const char* rmsnorm_strerror(int status);

/* Detail of the last failed call on this thread ("" if none). */
const char* rmsnorm_last_error(void);

/* RMSNORM_GB300_VERSION of the loaded library. */
int rmsnorm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_GB300_H */
