/*
 * gsi.h -- C ABI of the GB300 (sm_103a) Gated Subspace Inference linear map.
 *
 * The operation is the one defined on the page "Technical summary: Gated
 * Subspace Inference for transformer acceleration":
 *   section 2.1, eq. 1:  x = V_k V_k^T x + r      (r is the residual)
 *   section 2.1, eq. 2:  y = W x = (W V_k)(V_k^T x) + W r = M g + W r,
 *                        with g = V_k^T x and the cached image M = W V_k
 *   section 2.2:         rho = ||r|| / ||x|| per token;
 *                        rho <  eps -> fast path, y = M g
 *                        rho >= eps -> slow path, y = W x
 *
 * Conventions shared by every entry point
 *   - All tensors are dense, row-major, contiguous.
 *       W    d_out x d    bf16          (the linear's weight)
 *       V_k  d x k        bf16          (orthonormal rank-k basis)
 *       M    d_out x k    bf16          (cached image W V_k)
 *       x    T x d        bf16          (T tokens)
 *       y    T x d_out    fp32          (outputs)
 *       gate T            uint8         (1 = slow path taken, 0 = fast path)
 *       rho  T            fp32          (residual ratio per token)
 *   - Pointers are DEVICE pointers unless the name says _host, and must be
 *     16-byte aligned.  Shapes must satisfy d % 8 == 0, d_out % 8 == 0,
 *     k in {16, 32, 64, 128, 256, 512} and k <= d (else
 *     GSI_ERR_UNSUPPORTED_SHAPE).
 *   - eps is an fp32 threshold compared as "rho < eps"; a tie goes to the
 *     slow path; eps <= 0 makes every token slow, eps = +inf makes every
 *     token with finite rho fast; NaN eps is GSI_ERR_INVALID_ARG.
 *   - A token with ||x|| = 0 has rho = 0.  A token containing NaN or Inf
 *     has rho = NaN and takes the slow path.  rho is computed in fp32, so a
 *     token whose squared norm is outside the fp32 normal range
 *     (roughly ||x|| > 1e19 or ||x|| < 1e-18) is outside the supported range.
 *   - Errors in arguments are reported synchronously by the return value.
 *     Kernel-side problems (a bounded wait that ran out) set a device status
 *     word that gsi_device_status() reads.  Nothing here traps or asserts on
 *     the device.
 */
#ifndef GSI_H
#define GSI_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gsi_handle *gsi_handle_t;
typedef struct gsi_group *gsi_group_t;

typedef enum {
    GSI_OK = 0,
    GSI_ERR_INVALID_ARG = 1,       /* null pointer, misalignment, NaN eps, T < 0 */
    GSI_ERR_UNSUPPORTED_SHAPE = 2, /* d, k, d_out outside the rules above */
    GSI_ERR_NOMEM = 3,             /* a device or host allocation failed */
    GSI_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
    GSI_ERR_WORKSPACE = 5,         /* T larger than the reserved workspace */
    GSI_ERR_TIMEOUT = 6,           /* a device-side bounded wait ran out */
    GSI_ERR_LAUNCH = 7,            /* a kernel saw an inconsistent launch and did nothing */
    GSI_ERR_RANK = 8               /* calibration: a block column vanished or the factorisation broke down */
} gsi_status_t;

/* Create a handle for one gated linear (section 2.1: W, V_k and M).
 *   W, V_k, M : device pointers, BORROWED: they must stay valid and unchanged
 *               for the handle's lifetime (nothing is copied).
 *   eps       : the gate threshold of section 2.2.
 *   out       : receives the handle.
 * The handle owns a small workspace (gate reductions, token index lists,
 * gathered operands) sized for T <= 512 tokens per call; gsi_reserve()
 * grows it.  Computes the Gram matrix V_k^T V_k (k x k) once, in fp64, and
 * from it the correction E = V_k^T V_k - I that the one-token path uses to
 * form ||r|| without a second pass over V_k.  Synchronises
 * the device once.  Thread-safe with respect to other handles. */
gsi_status_t gsi_create(const void *W, const void *V_k, const void *M,
                        int64_t d_out, int64_t d, int64_t k, float eps,
                        gsi_handle_t *out);

/* The gated map of sections 2.1-2.2 on T tokens.
 *   x     : T x d bf16 (device), 16-byte aligned.
 *   y     : T x d_out fp32 (device), 16-byte aligned, written in token order.
 *   gate  : T uint8 (device) or NULL.
 *   rho   : T fp32 (device, 4-byte aligned) or NULL.
 * A null x or y, or a misaligned x, y or rho -> GSI_ERR_INVALID_ARG.
 *   stream: CUDA stream; the call is asynchronous, allocates nothing, never
 *           synchronises, and may be captured in a CUDA graph.
 * T == 0 is a no-op.  T > reserved workspace -> GSI_ERR_WORKSPACE.
 * Calls on one handle must be ordered on the GPU (one stream, or streams
 * joined by events): the handle's workspace is shared by its calls.
 * T == 1 runs the decode path (one fused kernel: projection, gate, and the
 * GEMV that reads M on the fast path or W on the slow path); T > 1 runs the
 * batched path (projection, gate, compaction of the token indices, and
 * tensor-core GEMMs M G_fast^T and W X_slow^T scattered back). */
gsi_status_t gsi_forward(gsi_handle_t h, const void *x, int64_t T, float *y,
                         uint8_t *gate, float *rho, cudaStream_t stream);

/* gsi_forward on HOST buffers.
 * One token (T == 1) whose buffers are all page-locked host memory that the
 * device addresses directly (cudaHostAlloc / cudaMallocHost / cudaHostRegister
 * under unified addressing): a one-CTA kernel copies x into the handle's
 * device staging and the map writes y, gate and rho in place over the host
 * link (NVLink-C2C on Grace systems) -- two kernel launches, no copy nodes,
 * and consecutive calls on one stream chain like device calls.
 * More tokens with y, gate and rho in such memory: x (T x d bf16) is
 * copied into the handle's device staging, and the kernels write y, gate and
 * rho in place over the host link while they run (no copy of y back).
 * Otherwise: copies x to device staging buffers owned by the handle, runs
 * the map, and copies y (T x d_out fp32), gate and rho (either may be NULL)
 * back to the host buffers.  When the three are consecutive in
 * one host allocation -- y, then rho at y_host + T * d_out, then gate at
 * rho_host + T -- one copy returns all of them (two copies per call in all,
 * instead of four).
 * All work is queued on `stream`; with page-locked host buffers the call
 * returns before the work finishes and the caller synchronises the stream
 * before reading y; with pageable buffers the CUDA runtime may block.
 * Alignment as gsi_forward.  Staging buffers grow with gsi_reserve(). */
gsi_status_t gsi_forward_host(gsi_handle_t h, const void *x_host, int64_t T,
                              float *y_host, uint8_t *gate_host,
                              float *rho_host, cudaStream_t stream);

/* The cached image of section 2.1 (eq. 2): M = bf16(W V_k), computed with
 * fp32 accumulation and one round-to-nearest-even per entry.  W (d_out x d),
 * V_k (d x k) inputs and M (d_out x k) output are device pointers owned by
 * the caller.  Asynchronous on `stream`; allocates nothing. */
gsi_status_t gsi_precompute_M(const void *W, const void *V_k, void *M,
                              int64_t d_out, int64_t d, int64_t k,
                              cudaStream_t stream);

/* Grow the handle's workspace (device and host-staging) to max_T tokens per
 * call.  Synchronises the device.  Never shrinks. */
gsi_status_t gsi_reserve(gsi_handle_t h, int64_t max_T);

/* Synchronise `stream`, then read and clear the handle's device status
 * word: GSI_OK; GSI_ERR_TIMEOUT if a bounded device-side wait ran out in a
 * kernel of this handle since the last check; GSI_ERR_LAUNCH if a kernel
 * found its launch configuration inconsistent and returned without work.
 * In both error cases the outputs are not valid. */
gsi_status_t gsi_device_status(gsi_handle_t h, cudaStream_t stream);

/* Name the handle of the call that follows each one-token call on h, so that
 * h's decode kernel prefetches next's V_k, M and correction tiles into L2
 * while h's call runs.  A one-token call is bound by the latency of its
 * exchange between CTAs rather than by HBM bandwidth, so a fixed call order
 * (the linears of a decoder layer, layer after layer) can stream the next
 * call's operands from HBM in that time, and the next call then stages them
 * from L2.  This schedules memory traffic only: results are identical with or
 * without it.  The page has no counterpart; it serves its T = 1 decode path.
 *   next: a handle on the same device, h itself, or NULL to remove the link.
 * Applies to handles with k <= 256 (the one-barrier decode kernel); operands
 * above 64 MiB are not prefetched.  A CUDA graph captured before a change
 * keeps the link it was captured with.  Destroying either handle removes the
 * link.  Not thread-safe against concurrent gsi_set_prefetch or gsi_destroy
 * on the same handles.  Synchronous, host only. */
gsi_status_t gsi_set_prefetch(gsi_handle_t h, gsi_handle_t next);

/* As gsi_set_prefetch, with the operands of every member of a group (below)
 * as the target: for a call followed by a grouped launch.  Replaces any
 * previous target of h; NULL removes it. */
gsi_status_t gsi_set_prefetch_group(gsi_handle_t h, gsi_group_t next);

/* A group of 1 to 4 handles whose one-token calls are independent of one
 * another, run as ONE kernel launch (gsi_group_forward).  The page has no
 * counterpart: this schedules calls.  It serves decoder layers whose linears
 * read different inputs that are ready together.  For example, in a
 * parallel-residual block (GPT-J) the attention output projection and the
 * MLP output projection do not depend on each other.  Each member keeps its
 * own grid exchange on its share of the SMs (shares in proportion to its
 * V_k + M bytes), so the launch costs one dependent-launch boundary instead
 * of one per call.
 *   handles: n distinct handles on one device, all with the same k in
 *            {64, 128, 256}.  BORROWED: they must outlive the group.  A handle
 *            may belong to several groups and still be used alone.  All calls
 *            that involve one handle must be ordered on the GPU.
 * Computes each member's launch plan and tensor maps once.  Returns
 * GSI_ERR_UNSUPPORTED_SHAPE if a member's slices do not fit the kernel's
 * shared memory at its share of the SMs. */
gsi_status_t gsi_group_create(int n, const gsi_handle_t *handles, gsi_group_t *out);

/* One token through every member: for member m the same result as
 * gsi_forward(handles[m], x[m], 1, y[m], gate ? gate[m] : NULL,
 * rho ? rho[m] : NULL, stream).  x, y: arrays of n device pointers (16-byte
 * aligned); gate, rho: arrays of n device pointers (entries may be NULL) or
 * NULL.  Asynchronous on `stream`, allocates nothing. */
gsi_status_t gsi_group_forward(gsi_group_t g, const void *const *x, float *const *y,
                               uint8_t *const *gate, float *const *rho,
                               cudaStream_t stream);

/* gsi_group_forward with host buffers: for member m the same result as
 * gsi_forward_host(handles[m], x[m], 1, y[m], gate[m], rho[m], stream).
 * x, y: arrays of n host pointers (x 16-byte aligned); gate, rho: arrays of n
 * host pointers (entries may be NULL) or NULL.  When every buffer is
 * page-locked and addressable by the device, one launch of n CTAs copies each
 * member's x over the host link into that handle's staging, and the grouped
 * kernel writes y, gate and rho in place: no copy nodes.  Otherwise each x is
 * copied in and each output copied back through the handles' staging.
 * Asynchronous on `stream`: the host buffers must stay valid until it has
 * run.  A member handle must not be used by another call on the GPU at the
 * same time (its staging is shared). */
gsi_status_t gsi_group_forward_host(gsi_group_t g, const void *const *x_host,
                                    float *const *y_host,
                                    uint8_t *const *gate_host,
                                    float *const *rho_host,
                                    cudaStream_t stream);

/* The group's launches prefetch next's operands into L2 (as gsi_set_prefetch;
 * NULL removes the link). */
gsi_status_t gsi_group_set_prefetch(gsi_group_t g, gsi_handle_t next);

/* Release the group (not its handles).  Synchronises the device.  Removes
 * the prefetch links that point to it.  NULL is ignored. */
void gsi_group_destroy(gsi_group_t g);

/* Release the handle and its workspace (not W, V_k or M).  Synchronises the
 * device.  NULL is ignored. */
void gsi_destroy(gsi_handle_t h);

/* Static description of a status code. */
const char *gsi_status_string(gsi_status_t s);

/* Kernel launches that gsi_forward(h, ..., T, ...) issues for this T (for
 * launch accounting); 0 for T <= 0. */
int gsi_forward_launch_count(gsi_handle_t h, int64_t T);

/* One token (T = 1) of the gated map without a handle and without allocating:
 * for callers that cannot call cudaMalloc -- code running inside a framework
 * or server whose allocator owns all device memory (a pooling or caching
 * allocator that must see every allocation), or a fixed-memory deployment
 * where the first call must not fail for lack of memory.  The pages have no
 * counterpart to this entry point; it is an interface convenience.
 *   W, V_k, M, x, y, gate, rho, d_out, d, k, eps: as in gsi_create and
 *   gsi_forward (device pointers, 16-byte aligned, rho 4-byte aligned; gate,
 *   rho may be NULL).  Shapes as gsi_create: k in {16, ..., 512}, anything
 *   else is GSI_ERR_UNSUPPORTED_SHAPE.
 * The kernel's scratch (about 4.4 KB: two reduction buffers of up to
 * k + 4 = 516 floats, an arrival counter, a launch epoch and a status word)
 * lives in a fixed array that every GPU loading this library holds until
 * the process exits.  No cudaMalloc, cudaFree or allocating library routine
 * is called.  The first call on a device looks up that array's device
 * address (once per device, with the device current); make that first call
 * before any stream capture.  The launch plan of each (device, shape) is
 * kept on the host after its first call, so later calls of that shape make
 * no attribute or occupancy queries.
 * Each call clears the scratch on `stream` (one memset node) before its
 * kernel; all calls share the one array, so calls that overlap on the GPU
 * (different streams, no ordering) race and give wrong results.  There is no
 * status word to read a device-side timeout from: a call whose bounded wait
 * ran out writes NaN into rho (with gate = 1) and into the rows of y its
 * stalled CTAs own, so the outputs show it.  Asynchronous on `stream`. */
gsi_status_t gsi_forward_noalloc(const void *W, const void *V_k, const void *M,
                                 int64_t d_out, int64_t d, int64_t k, float eps,
                                 const void *x, float *y, uint8_t *gate,
                                 float *rho, cudaStream_t stream);

/* ---- Calibration of V_k -------------------------------------------------
 *
 * Section 2.3 of the page computes the basis once from one forward pass over
 * a representative calibration sequence, and gives no algorithm.  Here V_k
 * spans the top-k eigenvectors of the uncentred second moment C = X^T X of
 * the calibration tokens X (n x d): the rank-k subspace with the least summed
 * squared residual ||x - V_k V_k^T x||^2 (section 2.1, eq. 1) over those
 * tokens.  It is approached by block power iteration from a start block Q0:
 *   Q <- orth(X^T (X Q)),  iters times,
 * each product a tcgen05 GEMM with fp32 accumulation on bf16 operands (Q and
 * X Q are rounded to bf16 between the products), orth() a two-pass Cholesky
 * QR in fp32.  Only span(V_k) is defined: the basis inside the span (its
 * rotation, the order of its columns) is whatever the orthonormalisation
 * gives, and every use of V_k in this library depends on the span alone.
 * The caller computes M = W V_k with gsi_precompute_M afterwards.
 *
 *   X          n x d bf16, the calibration tokens (device)
 *   Q0         d x k bf16, the start block (device), full column rank; a
 *              seeded Gaussian block is the usual choice.  Its span should
 *              not be orthogonal to any top-k eigenvector (a random block is
 *              not, with probability 1)
 *   iters      number of applications of C (>= 0; 0 orthonormalises Q0)
 *   V_k        d x k bf16 output (device), orthonormal columns up to bf16
 *              rounding
 *   workspace  device scratch of at least gsi_calibrate_workspace_size()
 *              bytes, 256-byte aligned, owned by the caller, not shared by
 *              calls that may overlap on the GPU
 * Shapes: k in {16, 32, 64, 128, 256}, k <= d, k <= n, d % 8 == 0,
 * n % 8 == 0 (else GSI_ERR_UNSUPPORTED_SHAPE).  A workspace smaller than
 * required is GSI_ERR_WORKSPACE.  Asynchronous on `stream`; allocates
 * nothing; the launch sequence does not depend on the data, so a call can be
 * captured in a CUDA graph.  Each call clears the workspace's status word
 * first; gsi_calibrate_status() then reports the call's device-side outcome:
 * GSI_ERR_RANK when a column of the iterated block vanished (zero or
 * non-finite norm: X Q has a zero column, e.g. X = 0 or a zero column in
 * Q0) or a pivot of the unshifted Cholesky pass fell below 2^-20 on the
 * unit-diagonal Gram matrix; V_k is then not valid.  GSI_ERR_TIMEOUT when a
 * bounded wait of a tensor-core kernel ran out.  Tokens of rank below k are
 * not an error: the top-k eigenspace is then not unique, and V_k is one of
 * them up to the rounding that fills the missing directions. */
gsi_status_t gsi_calibrate_workspace_size(int64_t n, int64_t d, int64_t k,
                                          size_t *bytes);
gsi_status_t gsi_calibrate(const void *X, int64_t n, int64_t d, int64_t k,
                           const void *Q0, int iters, void *V_k,
                           void *workspace, size_t workspace_bytes,
                           cudaStream_t stream);
/* The depth cascade of section 2.3: the basis of each layer starts from the
 * basis just computed for the layer before it.  Layer 0 is
 * gsi_calibrate(X[0], ..., Q0, iters_first, V[0]); layer l > 0 is
 * gsi_calibrate(X[l], ..., V[l - 1], iters_next, V[l]).
 *   X  array of `layers` device pointers, each n x d bf16 (that layer's
 *      calibration tokens)
 *   V  array of `layers` distinct device pointers, each d x k bf16 (output)
 * The host arrays X and V are read during the call only.  One workspace
 * serves all layers; the status word is cleared once, at the start, and
 * gsi_calibrate_status() afterwards reports any layer's device-side error.
 * Shapes and errors as gsi_calibrate; layers < 1, a null entry or a
 * repeated V entry is GSI_ERR_INVALID_ARG.  Asynchronous on `stream`. */
gsi_status_t gsi_calibrate_cascade(const void *const *X, int layers, int64_t n,
                                   int64_t d, int64_t k, const void *Q0,
                                   int iters_first, int iters_next,
                                   void *const *V, void *workspace,
                                   size_t workspace_bytes, cudaStream_t stream);
/* gsi_calibrate with a CUDA event pair recorded on `stream` around every
 * kernel launch, for measurement: synchronises the stream, then writes each
 * launch's duration (ms) and kind to launch_ms[i] / launch_kind[i] (host
 * arrays of max_launches entries, launch order) and the number written to
 * *n_launches.  Kinds: 0 transpose, 1 tensor-core GEMM, 2 split-K sum,
 * 3 Gram matrix, 4 Cholesky, 5 forward substitution.  The events keep
 * neighbouring launches from overlapping, so the durations add up to a bit
 * more than a gsi_calibrate call takes. */
gsi_status_t gsi_calibrate_timed(const void *X, int64_t n, int64_t d, int64_t k,
                                 const void *Q0, int iters, void *V_k,
                                 void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream, float *launch_ms,
                                 int *launch_kind, int max_launches,
                                 int *n_launches);
/* Synchronise `stream` and read the status of the last gsi_calibrate on
 * this workspace (see above). */
gsi_status_t gsi_calibrate_status(const void *workspace, cudaStream_t stream);
/* Kernel launches one gsi_calibrate(n, d, k, iters) issues on the current
 * device (0 for unsupported shapes). */
int gsi_calibrate_launch_count(int64_t n, int64_t d, int64_t k, int iters);

/* ---- The depth cascade in rank-1 form ----------------------------------
 *
 * Section 2.3 of the page starts layer l + 1's basis from layer l's and
 * refines it with a few rank-1 corrections (DGKS updates) instead of a full
 * decomposition per layer.  gsi_refine_rank1 applies `corrections` such
 * corrections to a start basis V_in for the tokens X (C = X^T X):
 *   V = the positive-diagonal QR factor of V_in (CholeskyQR2, fp32)
 *   each correction: j = the column with the largest residual
 *     ||(I - V V^T) C v_j|| (the first of equals); q = that residual
 *     re-orthogonalised against V by classical Gram-Schmidt, repeated once
 *     when the first projection kept less than 1/sqrt(2) of its norm (the
 *     DGKS test), normalised; v_j <- cos(t) v_j + sin(t) q with
 *     t = atan2(2 s, a - b) / 2, a = v_j^T C v_j, b = q^T C q,
 *     s = v_j^T C q: the unit vector of span(v_j, q) with the largest
 *     Rayleigh quotient.  The update changes one column (rank one), keeps the
 *     columns orthonormal and never lowers trace(V^T C V).
 * C V is formed once on the tensor cores (bf16 operands, fp32 accumulation);
 * each correction's C q is two fp32 products over X on the CUDA cores; the
 * basis, C V and V^T C V are kept in fp32.  Unlike gsi_calibrate, the result
 * depends on the basis of V_in inside its span, not on the span alone.
 *
 *   X            n x d bf16 tokens (device)
 *   V_in         d x k bf16 start basis (device), full column rank
 *   corrections  >= 0 (0 returns the QR factor of V_in rounded to bf16)
 *   V_out        d x k bf16 output (device); may be V_in
 *   order        device int32 array of `corrections` entries receiving the
 *                column corrected at each step, or NULL
 *   workspace    device scratch of gsi_refine_rank1_workspace_size() bytes,
 *                256-byte aligned, owned by the caller; it is also a valid
 *                gsi_calibrate workspace for the same shape
 * Shapes and the status word as gsi_calibrate (gsi_calibrate_status reads
 * it; a non-finite residual sets GSI_ERR_RANK); with corrections > 0, also
 * n <= 32768 and d <= 32768 (one of their vectors is staged whole in shared
 * memory), else GSI_ERR_UNSUPPORTED_SHAPE.  A correction whose residual
 * vanishes after re-orthogonalisation (span(V) invariant under C) leaves V as
 * it is.  Asynchronous on `stream`; allocates nothing; the launch sequence
 * does not depend on the data (graph-capturable). */
gsi_status_t gsi_refine_rank1_workspace_size(int64_t n, int64_t d, int64_t k,
                                             size_t *bytes);
gsi_status_t gsi_refine_rank1(const void *X, int64_t n, int64_t d, int64_t k,
                              const void *V_in, int corrections, void *V_out,
                              int32_t *order, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);
/* The cascade in that form: layer 0 is gsi_calibrate(X[0], ..., Q0,
 * iters_first, V[0]); layer l > 0 is gsi_refine_rank1(X[l], ..., V[l - 1],
 * corrections, V[l]).  X and V as in gsi_calibrate_cascade; `order`, if not
 * NULL, receives (layers - 1) x corrections column indices, layer by layer.
 * The workspace is gsi_refine_rank1_workspace_size() bytes; the status word
 * is cleared once, at the start.  Asynchronous on `stream`. */
gsi_status_t gsi_calibrate_cascade_rank1(const void *const *X, int layers,
                                         int64_t n, int64_t d, int64_t k,
                                         const void *Q0, int iters_first,
                                         int corrections, void *const *V,
                                         int32_t *order, void *workspace,
                                         size_t workspace_bytes,
                                         cudaStream_t stream);
/* Kernel launches one gsi_refine_rank1 issues (0 for unsupported shapes):
 * the start basis, C V, and one persistent launch that runs every correction
 * (its CTAs are all resident at once and meet at bounded grid barriers; a
 * barrier that runs out sets GSI_ERR_TIMEOUT and leaves V_out unwritten). */
int gsi_refine_rank1_launch_count(int64_t n, int64_t d, int64_t k,
                                  int corrections);

#ifdef __cplusplus
}
#endif

#endif /* GSI_H */
