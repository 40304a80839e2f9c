/*
 * es.h -- C ABI of libes.so, a GB300-native (sm_103a) `element-scan` library.
 *
 * Operation: "Nonlinear element scans" (sx.041.io/docs/element-scan.md).
 *   intro        h[t] = f(h[t-1], seq_1[t], ..., seq_n[t]) at every position
 *                outside one sequence axis, from h[-1] = initial; every
 *                output position holds the state after its own trip.
 *   :reverse     trips run from the last position to the first,
 *                h[t] = f(h[t+1], ...) from h[T] = initial; the final state
 *                is at position 0 (reverse paragraph of the intro).
 *   :state-axis  each lane carries a vector of 1..16 values along the last
 *                axis; a sequence whose last width is 1 is a per-trip value
 *                broadcast over the whole state ("Arguments and body").
 *   precision    the recurrence computes in f32 ("Precision and gradients").
 * Layout: every array is dense, C-contiguous, row-major f32 ("lucid.tensor"
 * page, contiguity paragraph).
 *
 * All pointers passed to es_scan_f32 except `seqs`, `shape` and `seq_widths`
 * are DEVICE pointers owned by the caller; the library never frees or keeps
 * them.  Calls are asynchronous on the caller's stream.  No function here
 * throws; every failure is a status code plus a thread-local message.
 */
#ifndef ES_H
#define ES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same handle type as cudaStream_t; NULL means the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *es_stream_t;

/* Bodies (element-scan page): each takes the state and two sequences.
 *   ES_TANH_DECAY  seqs (x, a):  h = tanh(x + a*h)            intro example
 *   ES_NORMCAP     seqs (x, a):  y = a*h + x; h = y / max(1, ||y||_2)
 *                                over the whole state vector   :state-axis example
 *   ES_MAXPLUS     seqs (x, c):  h = maximum(h - c, x)         :reverse example
 * Each body operation is one f32 operation rounded to nearest, in the order
 * written (no fused multiply-add); tanh, sqrt and division are CUDA's
 * tanhf, correctly rounded sqrtf and correctly rounded division; `maximum`
 * is IEEE 754-2019 maximum (+0 above -0, NaN propagates). */
typedef enum es_body {
    ES_TANH_DECAY = 0,
    ES_NORMCAP = 1,
    ES_MAXPLUS = 2
} es_body;

/* Status codes.  The E-DIM codes follow the error table of the "Tensor
 * operations" page ("Errors"): E-DIM-001 shapes do not fit, E-DIM-002 dtypes
 * differ. */
typedef enum es_status {
    ES_OK = 0,
    ES_E_DIM_001 = 1,     /* shapes do not fit: axis, widths, T = 0, rank    */
    ES_E_DIM_002 = 2,     /* dtype (reserved: only f32 entry points exist)   */
    ES_E_ARG = 3,         /* null / misaligned / overlapping pointer, bad id */
    ES_E_UNSUPPORTED = 4, /* valid on the pages but not in this library      */
    ES_E_CUDA = 5,        /* a CUDA runtime or driver call failed            */
    ES_E_TIMEOUT = 6,     /* a kernel gave up a bounded device-side wait     */
    ES_E_BODY = 7         /* a body program the contract rejects            */
} es_status;

#define ES_MAX_RANK 8
#define ES_MAX_STATE 16
#define ES_MAX_SEQS 8

/* Kernel paths.  es_scan_f32 picks one per call (ES_PATH_AUTO) from the
 * canonical view [O, T, J, W] (O = product of dims before the axis, T the
 * axis length, J lanes after it, W the state width, 1 for a scalar state). */
typedef enum es_path {
    ES_PATH_AUTO = 0,
    ES_PATH_EMPTY = 1,     /* no lanes: nothing is launched                    */
    ES_PATH_GENERIC = 2,   /* one thread per lane, direct loads, any layout    */
    ES_PATH_LANE_TMA = 3,  /* lanes innermost: TMA/mbarrier time-tile pipeline */
    ES_PATH_TIME_TMA = 4,  /* time innermost: TMA tiles transposed in SMEM     */
    ES_PATH_VEC_TMA = 5,   /* vector state: TMA pipeline + xor shuffles        */
    ES_PATH_MAT_TMA = 6,   /* matrix-scan, dense operands: TMA pipeline        */
    ES_PATH_MAT_CHUNKED = 7, /* matrix-scan, few long lanes: chunked scan (3 kernels) */
    ES_PATH_MAT_CHUNKED_TMA = 8 /* the same chunked scan, its scan passes on the TMA pipeline */
} es_path;

/*
 * es_scan_f32 -- run one element scan.
 *
 *   body        ES_TANH_DECAY, ES_NORMCAP or ES_MAXPLUS.
 *   initial     device f32, the output shape with `axis` removed (its last
 *               dim is the state width W under a state axis).
 *   seqs        HOST array of n_seqs DEVICE pointers, in the body's argument
 *               order after the state: (x, a) or (x, c).
 *   n_seqs      must be 2.
 *   shape, rank HOST array: the output shape, rank 1..ES_MAX_RANK, dims >= 0.
 *               Without a state axis every sequence has exactly this shape.
 *   axis        the sequence axis, -rank <= axis < rank (negative counts from
 *               the end); shape[axis] >= 1.
 *   state_width 0 for a scalar state; otherwise W = shape[rank-1] in 1..16
 *               (`:state-axis -1`), and axis may not be the last axis.
 *               ES_NORMCAP requires W >= 1 (a scalar state cannot reduce);
 *               the pointwise bodies accept both.
 *   seq_widths  NULL (every sequence has `shape`), or a HOST array of n_seqs
 *               last widths, each 1 (broadcast over the state) or W.
 *   reverse     0 forward; nonzero runs the trips from the last position.
 *   out         device f32 of `shape`; must not overlap any input.
 *   stream      the CUDA stream to enqueue on.
 *
 * Returns ES_OK once the kernel is enqueued (nothing is launched when a
 * dimension other than the axis is 0).  Argument errors return before any
 * CUDA call.  Pointers must be 4-byte aligned; 16-byte alignment (and row
 * widths that are multiples of 4 floats) selects the TMA paths.  The call
 * allocates no device memory; it keeps one small per-device status word
 * that bounded device waits report through es_device_status().
 */
es_status es_scan_f32(es_body body, const float *initial, const float *const *seqs,
                      int n_seqs, const int64_t *shape, int rank, int axis,
                      int state_width, const int64_t *seq_widths, int reverse,
                      float *out, es_stream_t stream);

/* The plan of a call: canonical view and chosen kernel.  Pure host logic
 * (same validation as es_scan_f32, no CUDA call), so it can be used and
 * tested on machines without a GPU.  Pointers are only inspected for null,
 * alignment and overlap. */
typedef struct es_plan_info {
    int64_t O, T, J, W;        /* canonical [O, T, J, W]                      */
    int64_t seq_width[ES_MAX_SEQS]; /* each sequence's last width (1 or W); 0 past n_seqs */
    int64_t elements;          /* O*T*J*W output values                       */
    int path;                  /* es_path chosen                              */
    int reverse;
} es_plan_info;

es_status es_plan_f32(es_body body, const float *initial, const float *const *seqs,
                      int n_seqs, const int64_t *shape, int rank, int axis,
                      int state_width, const int64_t *seq_widths, int reverse,
                      const float *out, es_plan_info *info);

/*
 * es_scan_backward_f32 -- gradients of one element scan.
 *
 * "Nonlinear element scans", "Precision and gradients": gradients flow to
 * `initial` and to every sequence, and the gradient of a scan is another
 * element scan over the same lanes in the opposite trip order that applies
 * the body's vector-Jacobian product once a trip (a forward scan's gradient
 * runs from the last trip to the first, a reverse scan's from the first to
 * the last).  Per trip, with h the trip's output, p the state before it and
 * lam the state's cotangent:
 *   ES_TANH_DECAY  m = lam*(1 - h*h); dx = m; da = m*p; lam <- m*a
 *   ES_MAXPLUS     the larger of p - c and x takes lam (dx = lam, or
 *                  dc = -lam and lam passes on); a tie splits lam evenly
 *   ES_NORMCAP     y = a*p + x is recomputed; if ||y|| <= 1 mu = lam, else
 *                  mu = (lam - h (h . lam)) / ||y||; dx = mu; da = mu*p;
 *                  lam <- a*mu
 * A width-one sequence receives the sum of its gradients over the state.
 *
 *   body .. reverse  exactly the arguments of the forward call.
 *   states           device f32 of `shape`: the forward output (saved states).
 *   grad_out         device f32 of `shape`: dL/d(states).
 *   grad_initial     device f32, the shape of `initial` (written).
 *   grad_seqs        HOST array of n_seqs DEVICE pointers, each with the
 *                    shape of its sequence (written).
 * The written buffers may not overlap any input or each other (ES_E_ARG).
 * Asynchronous on `stream`; no allocation; statuses as for es_scan_f32.
 */
es_status es_scan_backward_f32(es_body body, const float *initial, const float *const *seqs,
                               int n_seqs, const int64_t *shape, int rank, int axis,
                               int state_width, const int64_t *seq_widths, int reverse,
                               const float *states, const float *grad_out, float *grad_initial,
                               float *const *grad_seqs, es_stream_t stream);

/*
 * es_scan_host_f32 -- es_scan_f32 end to end on HOST buffers: the inputs are
 * copied into the caller's device buffers, scanned, and the states copied
 * back to `out_h`.  Lanes are independent ("Storage and execution"), so when
 * the sequence axis is not the first dimension the call splits along the
 * first dimension into `chunks` row pieces (0: the library's default, 8; at
 * most 64; never more than the rows), each a complete smaller scan, and
 * pipelines them on three library-owned streams: one piece's host-to-device
 * copies, another's scan and a third's device-to-host copy run at once.  The
 * results are those of es_scan_f32 on the whole call, bit for bit.
 *
 *   body .. reverse   as for es_scan_f32.
 *   initial_h, seqs_h (a HOST array of host pointers), out_h
 *                     host buffers of the call's shapes; page-locked memory
 *                     lets the copies overlap.
 *   initial_d, seqs_d (a HOST array of device pointers), out_d
 *                     caller-owned device buffers of the same shapes.
 *   chunks            pieces (see above).
 *   stream            the call starts after earlier work on `stream`, and
 *                     work enqueued on `stream` after it waits for all of it
 *                     (events); read out_h after synchronising `stream`.
 * No allocation per call (the streams and events are created once per
 * device).  Statuses as for es_scan_f32, and ES_E_ARG for a null host
 * pointer or `chunks` outside 0..64 (checked before any CUDA call).
 */
es_status es_scan_host_f32(es_body body, const float *initial_h, const float *const *seqs_h,
                           int n_seqs, const int64_t *shape, int rank, int axis,
                           int state_width, const int64_t *seq_widths, int reverse,
                           float *out_h, float *initial_d, float *const *seqs_d, float *out_d,
                           int chunks, es_stream_t stream);

/* Plan of a backward call (validation and kernel path, no CUDA call). */
es_status es_plan_backward_f32(es_body body, const float *initial, const float *const *seqs,
                               int n_seqs, const int64_t *shape, int rank, int axis,
                               int state_width, const int64_t *seq_widths, int reverse,
                               const float *states, const float *grad_out,
                               const float *grad_initial, float *const *grad_seqs,
                               es_plan_info *info);

/*
 * Body programs: an element scan whose body is given as text, in the pages'
 * notation ("Nonlinear element scans", "Arguments and body"):
 *
 *     (lambda (h x a) (tanh (+ x (* a h))))
 *
 * The first argument is the incoming state, one argument follows per
 * sequence.  The body may use pointwise arithmetic (+ - * / pow sqrt exp log
 * neg abs rsqrt sin cos tanh acos asin atan2 maximum minimum), the six
 * comparisons (< <= > >= = !=), `and` / `or` / `not`, `where`, `let`,
 * numbers, `true` / `false`, (cast v :f32) and (cast v :bool), and identity
 * `reshape` / `broadcast-to`; with a state axis also (sum v) and (max v),
 * with :axes [-1] and :keepdims, over the state's values ("Tensor
 * operations": operation names, plain numbers fold in double precision until
 * they meet a tensor and become f32 constants).  Every tensor operation is
 * one f32 operation rounded to nearest in the order written (no fused
 * multiply-add); transcendental functions are CUDA's f32 functions; maximum
 * and minimum are IEEE 754-2019.  The body must return an f32 value as wide
 * as the state.  Bodies the contract rejects give ES_E_BODY with a message
 * naming the problem (E-SCAN-001 for a name that is no argument or binding).
 *
 * A program is compiled for each call signature (state width, sequence
 * widths, kernel path) with NVRTC on first use and cached by its generated
 * source; later calls launch the cached kernel.
 */
typedef struct es_body_program *es_body_t;

/* Read and check `text` (a NUL-terminated host string); on success *body
 * owns a new program (release it with es_body_destroy). */
es_status es_body_create(const char *text, es_body_t *body);

/* Release a program (NULL is ignored).  Kernels compiled for it stay cached. */
es_status es_body_destroy(es_body_t body);

/* The number of sequences the program takes (its arguments minus the state),
 * or -1 for NULL. */
int es_body_n_seqs(es_body_t body);

/*
 * es_scan_body_f32 -- es_scan_f32 with a body program.  The arguments are
 * those of es_scan_f32 except `body`; n_seqs (1..ES_MAX_SEQS) must match the
 * program.  A scalar state (state_width 0) cannot use `sum` or `max` over the
 * state.  The first call of a signature compiles its kernel (host work, no
 * device synchronisation); statuses as for es_scan_f32 plus ES_E_BODY.
 */
es_status es_scan_body_f32(es_body_t body, const float *initial, const float *const *seqs,
                           int n_seqs, const int64_t *shape, int rank, int axis,
                           int state_width, const int64_t *seq_widths, int reverse,
                           float *out, es_stream_t stream);

/* Plan of a body-program call (validation, body check and kernel path; no
 * CUDA call, nothing compiled). */
es_status es_plan_body_f32(es_body_t body, const float *initial, const float *const *seqs,
                           int n_seqs, const int64_t *shape, int rank, int axis,
                           int state_width, const int64_t *seq_widths, int reverse,
                           const float *out, es_plan_info *info);

/* The CUDA functor generated for a signature (state_width as in
 * es_scan_body_f32, seq_widths NULL or n_seqs widths).  Writes at most `cap`
 * bytes including the NUL into `buf` (may be NULL with cap 0) and the full
 * length without the NUL into *needed.  No CUDA call. */
es_status es_body_source(es_body_t body, int state_width, int n_seqs, const int64_t *seq_widths,
                         char *buf, size_t cap, size_t *needed);

/* Compile ahead of time every kernel a signature (state_width, n_seqs,
 * seq_widths as in es_body_source) may use on `path` (ES_PATH_AUTO: on every
 * path it may take), so that later calls only load them.  Host work only
 * (NVRTC); no device is needed.  A compile failure is ES_E_CUDA with the
 * compiler's log. */
es_status es_body_prepare(es_body_t body, int state_width, int n_seqs, const int64_t *seq_widths,
                          int path);

/* es_scan_host_f32 with a body program (arguments as for es_scan_host_f32,
 * with the program in place of the body id). */
es_status es_scan_body_host_f32(es_body_t body, const float *initial_h, const float *const *seqs_h,
                                int n_seqs, const int64_t *shape, int rank, int axis,
                                int state_width, const int64_t *seq_widths, int reverse,
                                float *out_h, float *initial_d, float *const *seqs_d, float *out_d,
                                int chunks, es_stream_t stream);

/* NVRTC compilations so far in this process (kernel cache misses). */
uint64_t es_body_compile_count(void);

/*
 * es_scan_body_backward_f32 -- gradients of a body-program scan
 * ("Nonlinear element scans", "Precision and gradients": gradients flow to
 * `initial` and to every sequence; the gradient of a scan is another element
 * scan over the same lanes in the opposite trip order that applies the
 * body's vector-Jacobian product once a trip; comparisons and casts carry no
 * derivative, `where` passes it to the selected branch, and ties of
 * maximum / minimum and of the reduction `max` split it evenly).
 *
 * The VJP is derived from the body at compile time by reverse-mode
 * differentiation of its operations.  Per trip, with p the state before it
 * and lam the state's cotangent (the carried one plus grad_out of the trip),
 * the body is evaluated again at p, then its operations are swept backwards:
 * each one's derivative is formed in f32 with every operation rounded, the
 * contributions to a value are added in the reverse order of the operations
 * (a node's operands in argument order), and a width-one sequence, or any
 * width-one value a wide operation used, receives the sum of its wide
 * contribution over w = 0..W-1.  The rules per operation:
 *   a+b (g, g); a-b (g, -g); a*b (g*b, g*a); a/b (g/b, -(g*(a/b))/b);
 *   -a -g; |a| g*sign(a), 0 at 0; sqrt (g*0.5)/out; exp g*out; log g/a;
 *   tanh g*(1-out*out); sin g*cos(a); cos -(g*sin(a));
 *   rsqrt g*((out*out*out)*-0.5); acos -(g/sqrt(1-a*a)); asin g/sqrt(1-a*a);
 *   atan2(y, x) ((g*x)/(x*x+y*y), -(g*y)/(x*x+y*y));
 *   pow(a, b) (g*(b*pow(a, b-1)), 0 if out == 0 else g*(out*log(a)));
 *   maximum / minimum: the winner takes g, a tie (or NaN) gives g*0.5 each;
 *   where: g to the selected branch; sum: g to every value; max: g/count to
 *   each of its count equal maxima.
 *
 *   body .. reverse  exactly the arguments of the forward call.
 *   states           device f32 of `shape`: the forward output.
 *   grad_out         device f32 of `shape`: dL/d(states).
 *   grad_initial     device f32, the shape of `initial` (written).
 *   grad_seqs        HOST array of n_seqs DEVICE pointers, each with its
 *                    sequence's shape (written).
 * The written buffers may not overlap any input or each other (ES_E_ARG).
 * The kernel is one thread per lane (ES_PATH_GENERIC), compiled with NVRTC
 * on first use of a signature.  Asynchronous on `stream`; no allocation;
 * statuses as for es_scan_body_f32.
 */
es_status es_scan_body_backward_f32(es_body_t body, const float *initial, const float *const *seqs,
                                    int n_seqs, const int64_t *shape, int rank, int axis,
                                    int state_width, const int64_t *seq_widths, int reverse,
                                    const float *states, const float *grad_out,
                                    float *grad_initial, float *const *grad_seqs,
                                    es_stream_t stream);

/* Plan of a body-program backward call (validation, body check and kernel
 * path; no CUDA call, nothing compiled). */
es_status es_plan_body_backward_f32(es_body_t body, const float *initial, const float *const *seqs,
                                    int n_seqs, const int64_t *shape, int rank, int axis,
                                    int state_width, const int64_t *seq_widths, int reverse,
                                    const float *states, const float *grad_out,
                                    const float *grad_initial, float *const *grad_seqs,
                                    es_plan_info *info);

/* The functor with its vector-Jacobian product `vjp` for a signature
 * (arguments and output as in es_body_source).  No CUDA call. */
es_status es_body_source_backward(es_body_t body, int state_width, int n_seqs,
                                  const int64_t *seq_widths, char *buf, size_t cap, size_t *needed);

/* Compile ahead of time the backward kernel of a signature (as in
 * es_body_source).  No device needed. */
es_status es_body_prepare_backward(es_body_t body, int state_width, int n_seqs,
                                   const int64_t *seq_widths);

/*
 * es_matrix_scan_f32 -- matrix-scan ("Tensor operations", the `matrix-scan`
 * row of the operations table and the section "matrix-scan"):
 *
 *     h[t] = a[t] @ h[t-1] + b[t]    along `axis`, from h = 0 (so h[0] = b[0])
 *
 * and with `reverse` from the last position (h[T] = 0).  Every column of h
 * is its own recurrence on the shared a.
 *   a, a_shape, a_rank  device f32, shape lead_a + [n, n], n in 1..16.
 *   b, b_shape, b_rank  device f32, shape lead_b + [n, m], m >= 1.
 *                       lead_a and lead_b broadcast NumPy-style (right
 *                       aligned, each dim equal or 1) to one leading shape
 *                       of rank 1..ES_MAX_RANK.
 *   axis                counts among the leading dims (negative from the
 *                       end: -1 is the one before the matrices); its length
 *                       is at least one.
 *   projective          nonzero: the running product P of a, from the
 *                       identity, is divided by its largest magnitude after
 *                       every step, and h by the same number (for products of
 *                       projective maps that would overflow f32); needs
 *                       n + m <= 32.
 *   out                 device f32, the broadcast leading shape + [n, m];
 *                       must not overlap a or b.
 * Arithmetic: f32; each product a[i][j] * h[j][k] and each sum rounded, the
 * terms added in the order j = 0..n-1, then b[i][k] added (no fused
 * multiply-add); the projective scaling is an IEEE maximum of |P| and IEEE
 * divisions.  Shape errors are ES_E_DIM_001.  Dense operands (no broadcast)
 * with n in {2, 4, 8, 16}, n*m a multiple of 4 and at most 256, and 16-byte
 * aligned pointers take the TMA kernel (ES_PATH_MAT_TMA); anything else the
 * generic one.  Asynchronous on `stream`; no allocation.
 */
es_status es_matrix_scan_f32(const float *a, const int64_t *a_shape, int a_rank,
                             const float *b, const int64_t *b_shape, int b_rank,
                             int axis, int reverse, int projective, float *out,
                             es_stream_t stream);

/* Plan of a matrix-scan call (validation and kernel path; no CUDA call).
 * info: O, T, J the leading dims before, along and after the axis; W = n*m;
 * seq_width = {n*n, n*m}. */
es_status es_plan_matrix_scan_f32(const float *a, const int64_t *a_shape, int a_rank,
                                  const float *b, const int64_t *b_shape, int b_rank,
                                  int axis, int reverse, int projective, const float *out,
                                  es_plan_info *info);

/*
 * Few long lanes.  A matrix-scan over few lanes (lanes * m < 8192) and many
 * trips (T >= 256) leaves most of the GPU idle when run lane by lane; since
 * the recurrence composes (over trips s..e, h[e] = (a[e]...a[s]) h[s-1] + the
 * chunk's scan from zero), it can instead run as a chunked scan in three
 * launches: each (lane, chunk) scans from zero and forms its transition
 * product, one pass per lane carries the chunks' boundary states, and each
 * chunk is scanned again from its carry.  The carries reassociate the
 * chain, so these results agree with the sequential order to rounding
 * (within 1e-5 * (1 + |h|) for non-expansive a), not bit for bit.  The chunks'
 * products and boundary states need a workspace, which the caller provides
 * (the library allocates nothing); projective scans always run sequentially.
 * Dense operands with n in {2, 4, 8, 16}, n*m a multiple of 4, n + m <= 32
 * and 16-byte aligned bases run the two scan passes on the TMA pipeline
 * (ES_PATH_MAT_CHUNKED_TMA); anything else on direct-load kernels
 * (ES_PATH_MAT_CHUNKED).  Both take the same chunks and the same arithmetic
 * step for step, so they agree bit for bit.
 *
 * es_matrix_scan_workspace_f32: the workspace bytes a call with these shapes
 * would use (0 when it runs sequentially and needs none).  Host logic only.
 * es_matrix_scan_ws_f32: es_matrix_scan_f32 with a device workspace of
 * `workspace_bytes` (16-byte aligned, not overlapping the operands): the
 * chunked scan when it applies and the workspace suffices, else exactly
 * es_matrix_scan_f32.  Forcing ES_PATH_MAT_CHUNKED or ES_PATH_MAT_CHUNKED_TMA
 * (es_set_path_override) on a call that cannot take it is ES_E_UNSUPPORTED.
 * es_plan_matrix_scan_ws_f32: the checks and the path of that call without a
 * GPU (info->path: ES_PATH_MAT_CHUNKED_TMA, ES_PATH_MAT_CHUNKED or the
 * sequential path); the pointers are only checked, never read.
 */
es_status es_matrix_scan_workspace_f32(const int64_t *a_shape, int a_rank, const int64_t *b_shape,
                                       int b_rank, int axis, int projective, size_t *bytes);

es_status es_plan_matrix_scan_ws_f32(const float *a, const int64_t *a_shape, int a_rank,
                                     const float *b, const int64_t *b_shape, int b_rank,
                                     int axis, int reverse, int projective, const float *out,
                                     const void *workspace, size_t workspace_bytes, es_plan_info *info);

es_status es_matrix_scan_ws_f32(const float *a, const int64_t *a_shape, int a_rank,
                                const float *b, const int64_t *b_shape, int b_rank,
                                int axis, int reverse, int projective, float *out,
                                void *workspace, size_t workspace_bytes, es_stream_t stream);

/*
 * es_matrix_scan_static_f32 -- es_matrix_scan_ws_f32 for callers that cannot
 * allocate device memory: code that runs where cudaMalloc is unavailable or
 * not allowed (an allocator-free real-time or embedded host, a plug-in whose
 * host application owns every allocation, a call made while a memory pool
 * may not grow).  The pages have no counterpart: this is an interface choice
 * of the library.  The chunked scan for few long lanes runs in a scratch array
 * the library owns: a static device array of ES_STATIC_SCRATCH_BYTES, part of
 * the library's module, so every GPU that has loaded it holds it until the
 * process exits.  The call allocates nothing; the caller still passes a,
 * b and out (device, as for es_matrix_scan_ws_f32).
 *   set-up     the first call on a device, with that device current, loads
 *              the module that holds the array (its device memory is taken
 *              then), fetches the array's address (cudaGetSymbolAddress) and
 *              creates one event; make that first call before any stream
 *              capture.
 *   limit      a scan whose chunked form needs more than
 *              ES_STATIC_SCRATCH_BYTES (es_matrix_scan_workspace_f32) is
 *              refused with ES_E_UNSUPPORTED and a message giving both sizes;
 *              such a caller passes its own workspace to es_matrix_scan_ws_f32.
 *              Scans that need no scratch (many lanes) run as
 *              es_matrix_scan_f32.
 *   sharing    every call uses the same array, which keeps the last call's
 *              values; the scan writes every scratch value before reading
 *              it, so nothing needs clearing.  Calls that overlapped on the
 *              GPU would race in the array, so the library orders them: each
 *              call's kernels wait on an event the previous call recorded,
 *              whatever stream either was issued on.
 */
#define ES_STATIC_SCRATCH_BYTES (32u << 20)
es_status es_matrix_scan_static_f32(const float *a, const int64_t *a_shape, int a_rank,
                                    const float *b, const int64_t *b_shape, int b_rank,
                                    int axis, int reverse, int projective, float *out,
                                    es_stream_t stream);

/*
 * es_linear_scan_f32 -- linear-scan, the matrix-scan over one-by-one matrices
 * ("matrix-scan" section): h[t] = a[t] * h[t-1] + b[t] from h = 0, with a and
 * b broadcast NumPy-style to one shape (rank 0 is a number), `axis` counting
 * among its dims.  Same arithmetic (one product and one sum, rounded, in that
 * order).  Operands of one shape run on the element-scan kernels (lanes or
 * time innermost); broadcast operands on the generic matrix-scan kernel.
 */
es_status es_linear_scan_f32(const float *a, const int64_t *a_shape, int a_rank,
                             const float *b, const int64_t *b_shape, int b_rank,
                             int axis, int reverse, float *out, es_stream_t stream);

es_status es_plan_linear_scan_f32(const float *a, const int64_t *a_shape, int a_rank,
                                  const float *b, const int64_t *b_shape, int b_rank,
                                  int axis, int reverse, const float *out, es_plan_info *info);

/*
 * es_matrix_scan_backward_f32 -- gradients of a matrix-scan ("matrix-scan"
 * section: its gradient is the same scan run backwards on a's transposes; a
 * projective scan has no gradient).  With g[t] = dL/dh[t] (`grad_out`), the
 * cotangent
 *
 *     lam[t] = a[t+1]^T @ lam[t+1] + g[t]    (reverse: a[t-1]^T @ lam[t-1])
 *
 * runs from zero in the opposite trip order, past the last trip with the
 * zero matrix as coefficient; grad_b = lam and grad_a[t] = lam[t] @ h^T of
 * the state before trip t (zero before the first).  Every product is the
 * plain definition in f32: a^T's rows in order then g added; grad_a[i][j]
 * sums lam[i][k] * h[j][k] over k = 0..m-1 in order.
 *
 *   a .. projective  the forward call's arguments; a and b must have one
 *                    leading shape (no broadcasting: ES_E_UNSUPPORTED), and
 *                    a projective scan is ES_E_ARG.
 *   states           device f32: the forward's output.
 *   grad_out         device f32 of the output's shape.
 *   grad_a, grad_b   device f32 of a's and b's shapes (written); they may
 *                    not overlap any input or each other (ES_E_ARG).
 * Two kernels: the cotangent scan, then grad_a.  On the TMA path with at
 * least 256 trips both run in up to eight windows of trips, the scan windows
 * on `stream` and each window's grad_a on a library-owned stream per device
 * (created on first use, ordered after its scan window by an event) so that
 * it overlaps the next scan window; later work on `stream` waits for all of
 * it.  The results are the same bits either way.  No device allocation.
 */
es_status es_matrix_scan_backward_f32(const float *a, const int64_t *a_shape, int a_rank,
                                      const float *b, const int64_t *b_shape, int b_rank,
                                      int axis, int reverse, int projective,
                                      const float *states, const float *grad_out,
                                      float *grad_a, float *grad_b, es_stream_t stream);

/* Plan of a matrix-scan backward call (validation and the cotangent scan's
 * kernel path; no CUDA call). */
es_status es_plan_matrix_scan_backward_f32(const float *a, const int64_t *a_shape, int a_rank,
                                           const float *b, const int64_t *b_shape, int b_rank,
                                           int axis, int reverse, int projective,
                                           const float *states, const float *grad_out,
                                           const float *grad_a, const float *grad_b,
                                           es_plan_info *info);

/*
 * es_matrix_scan_backward_ws_f32 -- es_matrix_scan_backward_f32 with a
 * device workspace, for few long lanes.  The cotangent recurrence composes
 * over chunks of trips exactly as the forward scan does, so it runs as the
 * same chunked scan (chunk pass, link pass, final pass on the TMA kernel,
 * section "Few long lanes" above) with the transposed, one-trip-shifted
 * coefficient, then grad_a as before: four kernels.  It applies when the
 * forward call would be chunked on the TMA passes (ES_PATH_MAT_CHUNKED_TMA)
 * and `workspace_bytes` covers es_matrix_scan_workspace_f32 of the same
 * shapes (the geometry is the forward's); otherwise the call is exactly
 * es_matrix_scan_backward_f32.  The chunks reassociate the cotangent chain,
 * so grad_b and grad_a agree with the sequential gradient to rounding
 * (within 1e-5 * (1 + |value|) for non-expansive a), not bit for bit.
 *   workspace  device, 16-byte aligned, not overlapping any operand (ES_E_ARG).
 * Forcing ES_PATH_MAT_CHUNKED_TMA on a call that cannot take it, or
 * ES_PATH_MAT_CHUNKED (the direct-load chunk kernels have no gradient), is
 * ES_E_UNSUPPORTED.  es_plan_matrix_scan_backward_ws_f32: the checks and
 * the path without a GPU.
 */
es_status es_matrix_scan_backward_ws_f32(const float *a, const int64_t *a_shape, int a_rank,
                                         const float *b, const int64_t *b_shape, int b_rank,
                                         int axis, int reverse, int projective,
                                         const float *states, const float *grad_out,
                                         float *grad_a, float *grad_b,
                                         void *workspace, size_t workspace_bytes, es_stream_t stream);

es_status es_plan_matrix_scan_backward_ws_f32(const float *a, const int64_t *a_shape, int a_rank,
                                              const float *b, const int64_t *b_shape, int b_rank,
                                              int axis, int reverse, int projective,
                                              const float *states, const float *grad_out,
                                              const float *grad_a, const float *grad_b,
                                              const void *workspace, size_t workspace_bytes,
                                              es_plan_info *info);

/*
 * es_linear_scan_backward_f32 -- gradients of a linear-scan whose a and b
 * have one shape (ES_E_UNSUPPORTED otherwise): lam[t] = a[t+1] * lam[t+1] +
 * g[t] in the opposite trip order, grad_b = lam, grad_a[t] = lam[t] * h[t-1]
 * (zero before the first trip), one product and one sum a trip, rounded.  It
 * runs as the element-scan backward of the body (+ (* a h) b) from zero, on
 * the element-scan backward kernels.  Arguments as for the matrix form.
 */
es_status es_linear_scan_backward_f32(const float *a, const int64_t *a_shape, int a_rank,
                                      const float *b, const int64_t *b_shape, int b_rank,
                                      int axis, int reverse, const float *states,
                                      const float *grad_out, float *grad_a, float *grad_b,
                                      es_stream_t stream);

/* Plan of a linear-scan backward call (no CUDA call). */
es_status es_plan_linear_scan_backward_f32(const float *a, const int64_t *a_shape, int a_rank,
                                           const float *b, const int64_t *b_shape, int b_rank,
                                           int axis, int reverse, const float *states,
                                           const float *grad_out, const float *grad_a,
                                           const float *grad_b, es_plan_info *info);

/*
 * es_table_scan_i32 -- table-scan ("Tensor operations", the `table-scan` row
 * of the operations table and the section "table-scan"): a deterministic
 * automaton run along `axis` of `symbols`,
 *
 *     h[t] = table[h[t-1], symbols[t]]     from h[-1] = start
 *
 * every state kept, in `symbols`' shape (no gradient).
 *   table             device i32 [n_states, n_syms], row-major; n_states and
 *                     n_syms >= 1 (else ES_E_DIM_001).
 *   symbols, shape, rank, axis  device i32 of `shape` (rank 1..ES_MAX_RANK;
 *                     the pages' default axis is -1, the last).
 *   start             a state, 0 <= start < n_states (else ES_E_DIM_001).
 *   out               device i32 of `shape`; must not overlap an input.
 * As on the pages' CUDA backend, a symbol outside [0, n_syms) and a table
 * entry outside [0, n_states) are clamped into range (as `gather` clamps an
 * index); the clamped entry is the state, so every state is a valid row.
 * One thread per sequence with the table in shared memory when it has at
 * most 8192 entries (else read through the read-only path); the symbols are
 * streamed by the TMA pipelines (ES_PATH_TIME_TMA when the axis is last,
 * ES_PATH_LANE_TMA for >= 32 sequences side by side), else ES_PATH_GENERIC.
 * An axis of length 0 launches nothing.  Asynchronous on `stream`.
 */
es_status es_table_scan_i32(const int32_t *table, int64_t n_states, int64_t n_syms,
                            const int32_t *symbols, const int64_t *shape, int rank, int axis,
                            int32_t start, int32_t *out, es_stream_t stream);

es_status es_plan_table_scan_i32(const int32_t *table, int64_t n_states, int64_t n_syms,
                                 const int32_t *symbols, const int64_t *shape, int rank, int axis,
                                 int32_t start, const int32_t *out, es_plan_info *info);

/* Synchronise `stream`, then read and clear this device's status word.
 * Returns ES_E_TIMEOUT if a kernel since the last check gave up a bounded
 * wait (its outputs are then incomplete), ES_E_CUDA if the synchronisation
 * failed, else ES_OK. */
es_status es_device_status(es_stream_t stream);

/* Message of the last failed call on this thread ("" if none). */
const char *es_last_error(void);

/* Static name of a status code. */
const char *es_status_string(es_status status);

/* Kernel launches issued by this process so far (all devices). */
uint64_t es_launch_count(void);

/* Testing hooks (process-wide).
 *   es_set_path_override: force a path for later calls (ES_PATH_AUTO undoes
 *     it); a call the forced path cannot serve returns ES_E_UNSUPPORTED.
 *   es_set_wait_limit_ns: limit of every bounded device wait (default 2 s).
 *   es_set_drop_tile: the TMA producers skip the load of pipeline tile k
 *     (-1: off), so the consumers' bounded wait runs out; used to test the
 *     timeout path without faulting or hanging the GPU. */
es_status es_set_path_override(int path);
es_status es_set_wait_limit_ns(uint64_t ns);
es_status es_set_drop_tile(int64_t k);

#ifdef __cplusplus
}
#endif

#endif /* ES_H */
