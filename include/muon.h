/*
 * muon.h -- C ABI of the GB300 (sm_103a) Muon / Periodic Row-wise Muon optimizer step.
 *
 * What the library computes (per 2-D weight matrix W of shape A x B, row-major):
 *
 *   momentum      M <- mu*M + G
 *                 ("Muon is Scalable for LLM Training" notes, section 2.1, Eq. (1));
 *   Newton-Schulz X0 = M/||M||_F, five times X <- a X + b (X X^T) X + c (X X^T)^2 X,
 *                 (a, b, c) = (3.4445, -4.7750, 2.0315), run on the short side of M
 *                 (same page, section 2.1, Eq. (2); section 2.2 for N = 5);
 *   RowNorm       each of the min(A, B) lines of M along its long dimension scaled
 *                 to unit L2 norm: rows when A <= B, columns when A > B
 *                 ("Scaling Muon for Diffusion Transformers", abstract and the
 *                 Periodic Row-wise / distributed-implementation paragraphs);
 *   apply         W <- W - eta*(s*U + lambda*W) with s = 0.2*sqrt(max(A, B)) on NS5
 *                 steps and gamma*0.2*sqrt(max(A, B)) on RowNorm steps
 *                 ("Muon is Scalable" notes, Eq. (3), (4), (7));
 *   schedule      NS5 refresh iff step % K == 0 (step counted from 0), RowNorm
 *                 otherwise ("Scaling Muon for Diffusion Transformers", Periodic
 *                 Row-wise paragraph; K = 1 is vanilla Muon).
 *
 * Conventions for every entry point:
 *  - Memory: all tensor pointers are DEVICE pointers owned by the caller (for
 *    example PyTorch allocations).  The library allocates no device memory and
 *    frees nothing.  Scratch space comes from the caller's workspace `ws`
 *    (device, 256-byte aligned, at least muon_workspace_size() bytes).  A
 *    workspace holds one call's scratch: two calls whose GPU work may overlap
 *    (different streams, no ordering between them) need two workspaces.  Arrays
 *    of muon_matrix and arrays of output pointers are HOST arrays, read during
 *    the call only.
 *  - Layout: W, G, M, O and R are row-major A x B with leading dimension B (dense).
 *    M is always fp32.  W and G are fp32 or bf16 (MUON_DTYPE_*); within one call
 *    every matrix uses the same (w_dtype, g_dtype) pair.
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Every
 *    call only enqueues work on it, never synchronises (except muon_check_status),
 *    and can be captured into a CUDA graph once the one-time set-up has run: the
 *    first call on a host thread and device creates a second stream and two
 *    events for that thread, and the first call on a device sets kernel attributes
 *    and queries occupancy.  Call muon_init() (or make one eager call) on each
 *    host thread and device before capturing the library's calls.
 *  - Errors: host-side validation happens before any launch; on error nothing is
 *    enqueued and a negative muon_status is returned.  Device-side failures
 *    (bounded waits that expired; non-finite norms when the finite check of
 *    muon_periodic_step_ex is on) are recorded in the workspace's status word and
 *    read by muon_check_status().
 *  - Non-finite values: NaN or Inf in G propagate through the arithmetic as IEEE
 *    defines it, deterministically.  A NaN or Inf in M makes ||M||_F (a refresh
 *    step) or that line's norm (a RowNorm step) non-finite; the direction is then
 *    M divided by that norm, so the whole matrix (refresh) or that line (RowNorm)
 *    of W becomes NaN, and an Inf norm turns the finite entries' direction into 0.
 *    Only an exactly zero norm is treated as a zero direction.
 *  - Matrices with A == 0 or B == 0 are accepted and skipped; n == 0 is a no-op.
 *  - Determinism: all reductions use a fixed order, so identical inputs give
 *    bit-identical outputs run to run.
 */
#ifndef MUON_GB300_MUON_H
#define MUON_GB300_MUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MUON_ABI_VERSION 2

typedef enum muon_status {
  MUON_OK = 0,
  MUON_ERR_INVALID = -1,     /* bad argument: null pointer, negative size, K < 1, step < 0 */
  MUON_ERR_UNSUPPORTED = -2, /* dtype not supported, mixed dtypes, size beyond limits */
  MUON_ERR_WORKSPACE = -3,   /* workspace null, misaligned or smaller than required */
  MUON_ERR_CUDA = -4,        /* a CUDA runtime or driver call failed */
  MUON_ERR_TIMEOUT = -5,     /* a device-side bounded wait expired (from muon_check_status) */
  MUON_ERR_NO_DEVICE = -6,   /* no usable sm_103 device is current */
  MUON_ERR_NONFINITE = -7    /* a momentum norm was NaN or Inf (from muon_check_status, when the
                                finite check of muon_periodic_step_ex was on) */
} muon_status;

enum { MUON_DTYPE_F32 = 0, MUON_DTYPE_BF16 = 1 };

/* Newton-Schulz arithmetic: bf16 operands with fp32 accumulation on the tensor
 * cores (tcgen05), or fp32 throughout on the CUDA cores. */
enum { MUON_NS5_BF16 = 0, MUON_NS5_F32 = 1 };

/* Branch reported by muon_periodic_step. */
enum { MUON_BRANCH_ROWNORM = 0, MUON_BRANCH_NS5 = 1 };

typedef struct muon_matrix {
  void* W;          /* device, A x B row-major, w_dtype; updated in place           */
  const void* G;    /* device, A x B row-major, g_dtype; the step's gradient         */
  float* M;         /* device, A x B row-major, fp32 momentum; updated in place      */
  int64_t rows;     /* A (0 <= A < 2^31)                                             */
  int64_t cols;     /* B (0 <= B < 2^31)                                             */
  int32_t w_dtype;  /* MUON_DTYPE_F32 or MUON_DTYPE_BF16                             */
  int32_t g_dtype;  /* MUON_DTYPE_F32 or MUON_DTYPE_BF16                             */
} muon_matrix;

typedef void* muon_stream_t; /* cudaStream_t */

/* Bytes of workspace any entry point needs for this matrix list and NS5 mode
 * (the maximum over all entry points; one workspace serves them all).
 * Returns 0 for n == 0, and (size_t)-1 for an invalid list. */
size_t muon_workspace_size(const muon_matrix* mats, int n, int ns5_mode);

/* Momentum, Eq. (1) of the "Muon is Scalable" notes (section 2.1):
 *   M_i <- mu*M_i + G_i for every matrix.
 * fro_sq_out: optional device array of n floats; when non-NULL it receives
 * ||M_i||_F^2 of the updated momentum (fixed-order fp32 reduction), and ws must
 * be a valid workspace.  W is not read.  ws may be NULL when fro_sq_out is NULL. */
int muon_momentum(const muon_matrix* mats, int n, float mu, float* fro_sq_out,
                  void* ws, size_t ws_bytes, muon_stream_t stream);

/* Frobenius norm of the current momentum, the normaliser of X0 = M/||M||_F
 * (section 2.1 of the "Muon is Scalable" notes): fro_out[i] = ||M_i||_F (device,
 * n floats).  M is read only; G and W are not read. */
int muon_fro_norm(const muon_matrix* mats, int n, float* fro_out,
                  void* ws, size_t ws_bytes, muon_stream_t stream);

/* Same result as muon_fro_norm, for callers that cannot allocate device memory
 * (for example a plugin inside a host framework that owns every device
 * allocation, or code that must not call cudaMalloc mid-step because it would
 * synchronise the device).  The pages have no counterpart: this is a deployment
 * variant of the norm above.
 *  - No workspace: the per-tile partial sums live in a fixed 4 MiB array inside
 *    the library, resident on every GPU that loads it until the process exits.
 *  - Limit: at most 2^20 tiles of 64 x 128 elements per call (about 8.6e9
 *    elements of M in total); larger lists return MUON_ERR_UNSUPPORTED.
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress, which allocates nothing); the first call on a device
 *    may load the library's module there, so make that first call before any
 *    stream capture.  A device reset is handled: the next call finds the array
 *    again.
 *  - Same argument checks and status codes as muon_fro_norm (dtypes included).
 *  - All calls share the array.  Calls that overlap on the GPU (different
 *    streams, or different host threads) race on it; serialise them.
 *  - Allocates nothing, reads M only, writes fro_out[i] = ||M_i||_F.  Does not
 *    update muon_launch_count. */
int muon_fro_norm_noalloc(const muon_matrix* mats, int n, float* fro_out, muon_stream_t stream);

/* Newton-Schulz-5 of the current momentum, Eq. (2) of the "Muon is Scalable"
 * notes: O_i = NS5(M_i), computed on the short side of M_i and returned in
 * M_i's A x B orientation.  O_out: host array of n device pointers, each an
 * A x B row-major buffer of o_dtype.  ns5_mode selects the arithmetic
 * (MUON_NS5_BF16: bf16 tensor-core GEMMs, fp32 accumulate, bf16 intermediates;
 * MUON_NS5_F32: fp32 throughout).  M, G and W are not modified.  A zero M gives
 * O = 0. */
int muon_ns5_batched(const muon_matrix* mats, int n, int ns5_mode, void* const* O_out,
                     int o_dtype, void* ws, size_t ws_bytes, muon_stream_t stream);

/* RowNorm of the current momentum (Periodic Row-wise branch): R_i = M_i with each
 * row (A <= B) or each column (A > B) scaled to unit L2 norm; a zero line stays
 * zero.  R_out: host array of n device pointers to fp32 A x B buffers.  M is
 * read only. */
int muon_rownorm(const muon_matrix* mats, int n, float* const* R_out,
                 void* ws, size_t ws_bytes, muon_stream_t stream);

/* Apply, Eq. (4)/(7) of the "Muon is Scalable" notes:
 *   W_i <- W_i - eta*(scale_mul*sqrt(max(A, B))*U_i + lambda*W_i)
 * computed in fp32 with one rounding to w_dtype.  U: host array of n device
 * pointers to A x B buffers of u_dtype.  scale_mul is 0.2 for an NS5 direction
 * and 0.2*gamma for a RowNorm direction. */
int muon_apply(const muon_matrix* mats, int n, const void* const* U, int u_dtype,
               float scale_mul, float eta, float lambda, muon_stream_t stream);

/* One Periodic Row-wise Muon step over every matrix (K = 1: vanilla Muon):
 *   refresh = (step % K == 0);
 *   M <- mu*M + G;
 *   U = NS5(M) (refresh) or RowNorm(M) (otherwise);
 *   W <- W - eta*(s*U + lambda*W), s = 0.2*sqrt(max(A, B)), times gamma when not refreshing.
 * On refresh steps the apply is fused into the last Newton-Schulz GEMM.  On
 * RowNorm steps, wide and square matrices take one pass over memory (momentum,
 * row norms and apply); tall matrices take two row-contiguous passes in one
 * launch, the second re-reading the new momentum from L2.  The wide-row kernels
 * of a RowNorm step run on a second stream owned by the library (one per host
 * thread and device), forked from and joined back to `stream` with events, so
 * the call stays ordered on `stream` and capturable.  branch_out (host,
 * optional) receives MUON_BRANCH_NS5 or MUON_BRANCH_ROWNORM. */
int muon_periodic_step(const muon_matrix* mats, int n, int64_t step, int K, float gamma,
                       float mu, float eta, float lambda, int ns5_mode, void* ws,
                       size_t ws_bytes, muon_stream_t stream, int* branch_out);

/* One-time set-up for the current device and the calling host thread: checks the
 * device (sm_103), creates the thread's second stream and its fork/join events, sets
 * the tensor-core kernels' shared-memory attributes and caches occupancy figures.
 * Every entry point does the same on its first use; calling muon_init first makes
 * the first step capturable into a CUDA graph.  Allocates no device memory;
 * repeated calls are cheap no-ops.  Returns MUON_ERR_NO_DEVICE without a usable
 * device, MUON_ERR_CUDA if a set-up call fails. */
int muon_init(void);

/* Clears the status header of a fresh workspace (the first 256 bytes) on
 * `stream`.  Call once after allocating a workspace whose contents are not
 * already zero; the rest of the workspace needs no initialisation. */
int muon_workspace_init(void* ws, size_t ws_bytes, muon_stream_t stream);

/* Update scale of muon_periodic_step_ex. */
enum {
  MUON_SCALE_ADJUSTED_LR = 0, /* s = 0.2*sqrt(max(A, B)) ("Muon is Scalable" notes, Eq. (4)/(7)) */
  MUON_SCALE_UPDATE_NORM = 1  /* s = 0.2/RMS(U), "Update Norm", same notes, section 3.1, Eq. (6);
                                 on RowNorm steps the RMS is over the lines that carry the update,
                                 so it equals the Eq. (7) scale unless a line of M is zero */
};

typedef struct muon_step_options {
  int scale_mode;      /* MUON_SCALE_* */
  float* update_rms;   /* optional device array of n floats: RMS of each matrix's direction U
                          (the Newton-Schulz output, or the RowNorm of M) over its A*B elements,
                          as monitored against Lemma 1 ("Muon is Scalable" notes, section 2.2) */
  int check_finite;    /* nonzero: the kernels that reduce the momentum's norms (||M||_F^2 on a
                          refresh step, every line's sum of squares on a RowNorm step) set a bit
                          in the workspace status word when one is NaN or Inf, which
                          muon_check_status returns as MUON_ERR_NONFINITE.  The check reads
                          values the step computes anyway: it adds no memory traffic.  The
                          step's results are the same with the check on or off. */
} muon_step_options;

/* muon_periodic_step with options (opts == NULL: Eq. (4)/(7) scale, no telemetry).
 * With MUON_SCALE_UPDATE_NORM, refresh steps write O to the workspace, reduce its
 * sum of squares in a fixed order, then apply W <- W - eta*(0.2*O/RMS(O) + lambda*W)
 * in a separate pass (a zero O gives pure weight decay). */
int muon_periodic_step_ex(const muon_matrix* mats, int n, int64_t step, int K, float gamma,
                          float mu, float eta, float lambda, int ns5_mode,
                          const muon_step_options* opts, void* ws, size_t ws_bytes,
                          muon_stream_t stream, int* branch_out);

/* A parameter that Muon does not update (bias, normalisation weight, out-of-block
 * parameter), with its AdamW state. */
typedef struct muon_adamw_param {
  void* P;          /* device, numel elements of p_dtype; updated in place            */
  const void* G;    /* device, numel elements of g_dtype                             */
  float* m;         /* device, numel fp32 first moment (starts at 0)                 */
  float* v;         /* device, numel fp32 second moment (starts at 0)                */
  int64_t numel;
  int32_t p_dtype;  /* MUON_DTYPE_F32 or MUON_DTYPE_BF16                             */
  int32_t g_dtype;  /* MUON_DTYPE_F32 or MUON_DTYPE_BF16                             */
} muon_adamw_param;

/* AdamW on the parameters beside the Muon matrices ("Scaling Muon for Diffusion
 * Transformers", summary page: bias, normalisation and out-of-block parameters
 * keep AdamW, an auxiliary group at LR 1e-4; "Muon is Scalable" notes, section
 * 2.2: the two optimizers share learning rate and weight decay):
 *   m <- b1*m + (1-b1)*g;  v <- b2*v + (1-b2)*g^2;
 *   p <- p - lr*( (m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps) + weight_decay*p ),
 * fp32 arithmetic, one rounding to p_dtype (beta1 and beta2 are double so that 1-beta
 * is exact enough: 0.999 in fp32 would put 1.3e-5 into 1-beta2).  t counts steps from 1.  One launch
 * covers the whole list (host array); every entry uses the same dtype pair. */
int muon_adamw_step(const muon_adamw_param* params, int n, int64_t t, float lr, double beta1,
                    double beta2, float eps, float weight_decay, muon_stream_t stream);

/* Synchronises `stream`, reads and clears the device status word in `ws`, and
 * returns MUON_OK or the recorded error: MUON_ERR_TIMEOUT when a bounded wait
 * expired (it takes precedence), else MUON_ERR_NONFINITE when the finite check saw
 * a NaN or Inf norm.  The word accumulates over calls until it is read. */
int muon_check_status(void* ws, size_t ws_bytes, muon_stream_t stream);

/* Profiling hook (process-wide): up to 5 cudaEvent_t handles that
 * muon_periodic_step records on its stream at phase boundaries:
 *   [0] refresh step start, [1] first Newton-Schulz GEMM launch,
 *   [2] after the last Newton-Schulz GEMM, [3] RowNorm step start,
 *   [4] RowNorm step end.
 * NULL entries are skipped; n == 0 turns the hook off.  Recording also works
 * under stream capture (the records become graph nodes). */
int muon_profile_events(void* const* events, int n);

/* Number of kernels that the most recent entry-point call made by this host
 * thread enqueued (0 after a validation error). */
int muon_launch_count(void);

/* Static description of a status code. */
const char* muon_status_str(int status);

/* MUON_ABI_VERSION of the loaded library. */
int muon_abi_version(void);

/* Test hooks (process-wide, not for production use).
 * timeout_ms: limit of every device-side wait (default 4000 ms; 0 restores it).
 * flags: MUON_DEBUG_STALL_PRODUCER makes the tensor-core GEMM's load warp issue
 * nothing, and the tall-matrix RowNorm kernel publish no column norms, so that
 * their consumers' bounded waits expire and report MUON_ERR_TIMEOUT through
 * muon_check_status (no fault, no hang).
 * Tall matrices of RowNorm steps normally take two row-contiguous passes whose
 * second pass re-reads the new momentum from L2.  MUON_DEBUG_NO_CLUSTER sends
 * them through the plain two-pass kernels instead, MUON_DEBUG_TALL_CLUSTER
 * through the single-pass thread-block-cluster kernel (to test every path).
 * MUON_DEBUG_NO_OVERLAP runs the wide-row and tall-column kernels of a RowNorm
 * step one after the other on the caller's stream instead of side by side.
 * MUON_DEBUG_NO_PAIR runs the tensor-core Newton-Schulz GEMMs with one CTA per
 * 128 x 256 tile instead of 2-CTA clusters (tcgen05 cta_group::2) on 256 x 256 tiles. */
enum {
  MUON_DEBUG_STALL_PRODUCER = 1,
  MUON_DEBUG_NO_CLUSTER = 2,
  MUON_DEBUG_NO_OVERLAP = 4,
  MUON_DEBUG_TALL_CLUSTER = 8,
  MUON_DEBUG_NO_PAIR = 16
};
int muon_debug_set(int flags, int timeout_ms);

#ifdef __cplusplus
}
#endif
#endif /* MUON_GB300_MUON_H */
