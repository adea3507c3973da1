/*
 * vla.h - C ABI of the GB300 (sm_103a) Variational Linear Attention forward scan.
 *
 * What the scan computes, for every (batch b, head h) pair independently and
 * for t = 1..T in order (global step g = t0 + t):
 *
 *   for i = 1..r:                                   "Mathematical Primitives" §3
 *     z = A u_{t,i};  delta = 1 + u_{t,i} . z       §2, execution pipeline
 *     if |delta| < 1e-6:  A += 1e-6 I               §2, singularity guard
 *     else:               A -= z z^T / delta        §2, exact inverse update
 *   if P > 0 and g % P == 0:  A += eps_n I          §2, periodic spectrum stabilisation
 *   s = phi(k_t) / sqrt(d);  alpha = A s            §1 (s read as a vector), §4
 *   S += v_t alpha^T;  n += phi(k_t)                §5 (S is d_v x d); README "VLA v3" item 5
 *   if ||S||_F > tau:  S *= tau / ||S||_F           §5, dynamic renormalisation
 *   o_t = S phi(q_t) / (n . phi(q_t) + 1e-6)        README "VLA v3" item 5 (calibrated readout)
 *
 * with phi(x) = ELU(x) + 1 (README "VLA v3" item 1): x + 1 for x > 0, exp(x)
 * otherwise.  A tracks M_t^{-1} for M_t = M_{t-1} + u u^T (§2, "Theoretical
 * Derivation").  q, k are the raw projections; phi is applied inside the scan.
 * u is taken as given (the pages form it as normalize(W_u k_raw), README item 2);
 * the scan does not renormalise it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Device pointers are CUDA device (or managed) memory on the handle's device;
 *   the caller allocates and owns them.  The library owns only the handle and
 *   its small device status block.
 * - Layouts are dense row-major with the pair index p = b * H + h outermost:
 *     q, k : [B, H, T, d]          io dtype
 *     v    : [B, H, T, d_v]        io dtype
 *     u    : [B, H, T, r, d]       io dtype (the r directions of a step are contiguous)
 *     o    : [B, H, T, d_v]        io dtype, written
 *     A    : [B, H, d, d]          float32, read and written in place
 *     S    : [B, H, d_v, d]        float32, read and written in place
 *     n    : [B, H, d]             float32, read and written in place
 *   q, k, v and u must start on a 16-byte boundary (they are streamed with bulk
 *   asynchronous copies), and so must A and S (moved as 16-byte vectors).  o
 *   must not overlap any input.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Every call that launches work is asynchronous on that stream; it
 *   returns after the launch.  Errors of the kernel itself are reported through
 *   vla_status(), never by trapping.
 * - A handle is not thread-safe: one host thread uses it at a time.
 */
#ifndef VLA_H
#define VLA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct vla_handle_s* vla_handle_t;

typedef enum {
  VLA_OK = 0,
  VLA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned pointer, bad parameter */
  VLA_ERR_UNSUPPORTED = 2,   /* valid but not built: (d, d_v, r, dtype, mode) outside the list below */
  VLA_ERR_CUDA = 3,          /* a CUDA runtime call failed; see vla_last_error() */
  VLA_ERR_NOMEM = 4          /* host or device allocation failed */
} vla_err_t;

typedef enum { VLA_F32 = 0, VLA_BF16 = 1 } vla_dtype_t;        /* dtype of q, k, v, u, o */

typedef enum {
  VLA_SEQUENTIAL = 0,   /* the pages' recurrence in its step order, taken in rounds of a few
                           steps in exact Woodbury form (one set of reductions per round;
                           the same result up to rounding) */
  VLA_CHUNKED = 1,      /* `chunk` steps at a time in exact Woodbury / LDL^T form */
  VLA_DELTA = 2         /* the delta-rule variant (gist.science summary §2.3, "Recursive
                           Update Rule"): A tracked as above, then alpha_hat = A k_hat / |A k_hat|
                           with k_hat = phi(k) / |phi(k)|, S += (v - S k_hat) alpha_hat^T; n,
                           renormalisation and readout unchanged; computed in rounds of
                           several steps like VLA_SEQUENTIAL (CTAs per pair chosen as its
                           default; see t0 below for split calls) */
} vla_mode_t;

/* Status flags, ORed over all pairs since the last vla_status() call. */
#define VLA_STATUS_NONFINITE 1u  /* a NaN/Inf reached delta, the readout or ||S|| ("Mathematical Primitives" §1, finite state enforcement) */
#define VLA_STATUS_TIMEOUT   2u  /* a bounded wait on an input copy expired; that pair stopped early */

typedef struct {
  unsigned int flags;                 /* VLA_STATUS_* */
  unsigned int reserved;
  unsigned long long guard_count;     /* directions where the singularity guard replaced the update */
  unsigned long long renorm_count;    /* steps where S was renormalised */
  unsigned long long chunk_fallbacks; /* VLA_CHUNKED: chunks that were taken step by step */
} vla_status_t;

/* Create a handle bound to CUDA device `device`.  Allocates the handle and a
 * small device status block; does not change the caller's current device.
 * Errors: INVALID_ARG (h == NULL or no such device), CUDA, NOMEM. */
vla_err_t vla_create(vla_handle_t* h, int device);

/* Run the scan above over T steps for B * H pairs, continuing from the state in
 * A, S, n (updated in place) and writing o.
 *
 *   B, H      >= 0; B * H == 0 is a no-op (pointers may then be NULL).
 *   T         >= 0; T == 0 leaves the state untouched (q, k, v, u, o may be NULL).
 *   d, dv     head and value width.  Built: d == dv in {16, 64, 128}.
 *   r         directions per step.  Built: 1 and 4.
 *   P         nudge period (>= 0; 0 disables the nudge).
 *   eps_n     nudge size (finite).
 *   tau       renormalisation threshold on ||S||_F (> 0; +inf disables it).
 *   t0        steps already taken by earlier calls on this state (>= 0): the
 *             nudge fires at global steps t0 + t that are multiples of P, so
 *             splitting a sequence into several calls computes the same
 *             recurrence: the same bits when the calls split it at multiples of
 *             the kernel's input tile (sequential and delta modes: 32 steps at
 *             d <= 64 and r = 1, 16 at d = 64, r = 4 and at d = 128, r = 1, 8 at
 *             d = 128, r = 4; chunked mode: the chunk, 64 steps at r = 1 and 16 at
 *             r = 4; window boundaries of vla_scan_fwd_host count as splits) while no
 *             renormalisation has fired before the split (a call ends by folding
 *             its lazy scale into S); the same values up to rounding otherwise.
 *   io_dtype  VLA_F32 or VLA_BF16 for q, k, v, u and o; state is always float32.
 *   mode      VLA_SEQUENTIAL (every built shape) or VLA_CHUNKED (d == dv == 64,
 *             r 1 or 4, bfloat16 or float32 I/O; `chunk` = steps per chunk, see the
 *             built list in the library's error message; its products run on the
 *             tensor cores in tf32, split into three passes (3xTF32) where they
 *             carry A and, with float32 I/O, everywhere).  Both compute the same
 *             recurrence; they differ in rounding only.  VLA_DELTA computes the delta-rule variant (every
 *             built shape; `chunk` must be 0).
 *   chunk     VLA_CHUNKED: steps per chunk (0 = the built default).  The library
 *             runs each pair on a cluster of two CTAs (the A side and the S side
 *             of every chunk on two SMs) while 2 B H CTAs fit on the device's
 *             SMs, on one CTA otherwise; both forms give the same bits except in
 *             a chunk where the guard fires (the same values up to rounding).
 *             VLA_SEQUENTIAL: CTAs per (batch, head) pair: 1 = one CTA holds
 *             both halves of the step; 2 = a cluster of two CTAs on two SMs, one
 *             tracking A, the other S (the same arithmetic and the same results
 *             bit for bit, except at d == 128, r == 1, where the cluster takes 4
 *             steps per reduction round and one CTA 2: equal up to rounding);
 *             4 or 8 (d in {64, 128}, r == 1) = a cluster of that many CTAs, each
 *             holding d/4 or d/8 rows of A and the same columns of S, exchanging
 *             partial sums every step (the step-by-step recurrence; slower than
 *             1 or 2 on the built workloads, since every step waits for a
 *             cross-SM exchange; at most 8 clusters of 8 run at once);
 *             0 = two for d == 128 while 2 B H CTAs fit on the device's SMs, else
 *             one.
 *   stream    cudaStream_t as void*.
 *
 * Errors (returned before any launch, nothing is written): INVALID_ARG for a
 * NULL handle or pointer, negative size, misaligned q/k/v/u/A/S (and o in
 * VLA_CHUNKED mode, which writes it in 16-byte pieces), P < 0, t0 < 0,
 * tau <= 0 or NaN, non-finite eps_n; UNSUPPORTED for shapes that are not built;
 * CUDA if the launch fails.  There is no CPU fallback. */
vla_err_t vla_scan_fwd(vla_handle_t h,
                       const void* q, const void* k, const void* v, const void* u,
                       float* A, float* S, float* n, void* o,
                       int B, int H, long long T, int d, int dv, int r,
                       int P, float eps_n, float tau, long long t0,
                       vla_dtype_t io_dtype, vla_mode_t mode, int chunk,
                       void* stream);

/* The same scan as vla_scan_fwd with every buffer in HOST memory: q, k, v, u are
 * read from the host, o is written there, and A, S, n are read at the start and
 * written back at the end.  All arguments but `seg` mean what they mean for
 * vla_scan_fwd, with the same layouts; nothing needs any alignment.
 *
 * The sequence is cut into windows of `seg` steps (0 = the library's choice: the
 * whole sequence up to 2048 steps, else about 32 windows of a multiple of 64 steps
 * and at least 512, larger for the copy engines; see below).  Each window of
 * q, k, v, u is copied in on a copy stream of the handle, scanned on `stream`, and
 * its o copied out on a second copy stream, so that the copies of one window
 * overlap the scan of its neighbours.  The state stays
 * on the device between windows and `t0` advances window by window, so the result is
 * that of vla_scan_fwd called once per window.
 *
 * Copy-in.  When each of q, k, v, u lies inside one page-locked host allocation
 * that CUDA maps into the device's address space (cudaHostAlloc, or cudaHostRegister
 * with mapping, which unified addressing gives every page-locked buffer) and starts
 * on a 16-byte boundary, a small gather kernel on the copy stream reads each window
 * through that mapping, on the SMs the scan leaves idle.  Otherwise the copy engines
 * move each window (cudaMemcpy2DAsync), and the default window grows to rows of at
 * least 512 KB: the engines lose about half their rate on narrower rows of several
 * tensors.  Copies from or to pageable memory are correct but do not overlap the
 * scan.  o and the state always go through the copy engines.  The call is
 * asynchronous on `stream`: it returns once every copy and launch is enqueued;
 * o, A, S and n are final, and the host buffers may be reused, once `stream` has
 * reached that point (cudaStreamSynchronize).  Work the caller put on `stream`
 * before the call, and any earlier call of this entry point on the handle, finish
 * before the first copy starts.
 *
 * The handle keeps a device workspace of the state plus three windows of
 * q, k, v, u and o (reallocated, after the previous call has finished, when a larger
 * one is needed; freed by vla_destroy), two streams and a few events.
 *
 * Errors: as for vla_scan_fwd (except alignment), and INVALID_ARG for seg < 0;
 * NOMEM when the workspace cannot be allocated (a smaller `seg` needs less);
 * CUDA when a copy or launch cannot be enqueued.  After a CUDA error part of the
 * work may be enqueued: synchronise `stream` before touching the buffers. */
vla_err_t vla_scan_fwd_host(vla_handle_t h,
                            const void* q, const void* k, const void* v, const void* u,
                            float* A, float* S, float* n, void* o,
                            int B, int H, long long T, int d, int dv, int r,
                            int P, float eps_n, float tau, long long t0,
                            vla_dtype_t io_dtype, vla_mode_t mode, int chunk, long long seg,
                            void* stream);

/* How the last vla_scan_fwd_host call on the handle moved its inputs: *gathered = 1
 * for the SM gather, 0 for the copy engines, -1 before any such call; *seg = the
 * window it used (steps).  Errors: INVALID_ARG for a NULL argument. */
vla_err_t vla_host_path_info(vla_handle_t h, int* gathered, long long* seg);

/* The learned penalty directions before the scan: for every token t < n_tokens and
 * rank i < r,  u[t][i] = W_u[i] k_raw[t] / max(|W_u[i] k_raw[t]|_2, 1e-12)  (README
 * "VLA v3" item 2, "u_t = normalize(W_u k_t^raw)").  The products run on the tensor
 * cores: bfloat16 keys as bf16 operands with W carried as three bf16 terms (about 24
 * bits), float32 keys in tf32 with keys and W split into hi + lo parts (about 2^-21
 * relative; float32 arithmetic on CUDA cores for d = 128 with float32 keys); fp32
 * accumulation, norm and scaling.  A product that does not complete sets
 * VLA_STATUS_TIMEOUT in the handle's status.
 *
 *   k_raw     [n_tokens, d] in io_dtype: the keys before the feature map (for the scan's
 *             layout, n_tokens = B H T and k_raw is the [B, H, T, d] tensor).
 *   W_u       [r, d, d] float32 on the device, row-major: W_u[i][j][m] weighs input m
 *             in output j; one set of weights for every token.
 *   u         [n_tokens, r, d] in io_dtype, written: exactly the scan's u input.
 *   d         16, 64 or 128;  r  1..8.
 * k_raw, W_u and u start on 16-byte boundaries (rows move as 16-byte vectors).
 * Asynchronous on `stream`; the caller owns every buffer.  Errors (before any launch):
 * INVALID_ARG for a NULL handle or pointer, a misaligned pointer, n_tokens < 0, r
 * outside 1..8; UNSUPPORTED for other d; CUDA if the launch fails. */
vla_err_t vla_project_u(vla_handle_t h, const void* k_raw, const float* W_u, void* u, long long n_tokens,
                        int d, int r, vla_dtype_t io_dtype, void* stream);

/* Self-test of the kernels' bounded waits: launches one CTA whose thread waits, for
 * limit_ms milliseconds (1..5000), on an mbarrier that nothing completes, gives up and
 * sets VLA_STATUS_TIMEOUT in the handle's status, the path a scan kernel takes when an
 * input copy or a tensor-core product does not land within its limit (2 s).  It
 * shows that a wait that runs out returns control and reports through vla_status()
 * with the context still usable.  Asynchronous on `stream`.  Errors: INVALID_ARG for a
 * NULL handle or limit_ms outside 1..5000; CUDA if the launch fails. */
vla_err_t vla_selftest_wait(vla_handle_t h, unsigned int limit_ms, void* stream);

/* Measurement helper, not part of the scan (the pages have no counterpart): the FP32
 * CUDA-core throughput of the handle's device, against which the scan's roofline is
 * quoted.  Launches 4 CTAs of 256 threads per SM; each thread runs 8 independent chains
 * of packed fp32 FMAs for `iters` rounds (rounded up to a multiple of 8).  *flops
 * receives the launch's flop count (FMA = 2); the caller times the launch on `stream`
 * (for instance with events) and divides.  Asynchronous on `stream`.  Errors:
 * INVALID_ARG for a NULL argument or iters outside 8..2^30; CUDA if the launch fails. */
vla_err_t vla_ffma_probe(vla_handle_t h, long long iters, double* flops, void* stream);

/* Synchronise `stream`, copy the accumulated status into *out and reset it.
 * Errors: INVALID_ARG (NULL argument), CUDA. */
vla_err_t vla_status(vla_handle_t h, void* stream, vla_status_t* out);

/* Message of the last failed call on this handle ("" if none).  The string is
 * owned by the handle and stays valid until the next call on it.  With h ==
 * NULL it returns the message of the last failed vla_create or
 * vla_scan_fwd_noalloc on this thread. */
const char* vla_last_error(vla_handle_t h);

/* Free the handle, its status block and the workspace of vla_scan_fwd_host
 * (synchronises its device first).
 * h == NULL is a no-op that returns VLA_OK. */
vla_err_t vla_destroy(vla_handle_t h);

/* ------------------------------------------------------------------------
 * Scan without any allocation.  The pages have no counterpart to this entry
 * point: it exists for callers that may not allocate device memory.  Typical
 * ones run inside a framework or server whose allocator owns the device's
 * memory (a caching allocator, an arena sized at start-up) and must not call
 * cudaMalloc behind its back: cudaMalloc synchronises the device and takes
 * memory the owner neither tracks nor can reuse.  Others keep no state between
 * calls and so have no place to keep a handle, whose creation allocates.
 *
 * It runs the same sequential scan as vla_scan_fwd (same arguments, layouts and
 * results) on the caller's current device, with d == dv == 64 and r in {1, 4}.
 * Its scratch -- one status record per (b, h) pair -- is a static array inside
 * the library of VLA_NOALLOC_MAX_PAIRS records (256 KB), which every GPU that
 * loads the library holds until the process exits.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library routine is called.
 *
 *   pair_status  NULL, or a caller-owned array of B*H records (device memory or
 *                host memory).  Record b*H+h receives that pair's status for
 *                this call (flags as in VLA_STATUS_*, guard, renormalisation and
 *                replay counts).  It is written with cudaMemcpyAsync on `stream`
 *                and is valid once the stream has reached that point.
 *
 * - Each call clears the records it uses before the scan, so a record never
 *   carries counts from an earlier call.
 * - All calls share the one array: calls that overlap on the GPU (different
 *   streams, or different host threads, without ordering between them) race on
 *   it.  Order such calls, for example on one stream.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) and keeps it for later calls; make that first call
 *   before any stream capture on that device.
 * - That kept address does not survive cudaDeviceReset: the reset unloads the
 *   library's device code, and the array may come back elsewhere.  A process
 *   that resets a device must not call this entry point on it afterwards.
 *
 * Errors (returned before any launch): INVALID_ARG as for vla_scan_fwd, and when
 * B*H exceeds VLA_NOALLOC_MAX_PAIRS; UNSUPPORTED for shapes other than
 * d == dv == 64, r in {1, 4}; CUDA when a runtime call fails.  The message is
 * available from vla_last_error(NULL) on the calling thread. */
#define VLA_NOALLOC_MAX_PAIRS 16384

typedef struct {
  unsigned int flags;             /* VLA_STATUS_* */
  unsigned int guard_count;
  unsigned int renorm_count;
  unsigned int chunk_fallbacks;   /* chunks replayed one direction at a time */
} vla_pair_status_t;

vla_err_t vla_scan_fwd_noalloc(const void* q, const void* k, const void* v, const void* u,
                               float* A, float* S, float* n, void* o,
                               int B, int H, long long T, int d, int dv, int r,
                               int P, float eps_n, float tau, long long t0,
                               vla_dtype_t io_dtype, vla_pair_status_t* pair_status,
                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VLA_H */
