/*
 * lrscan.h -- C ABI of the GB300 (sm_103a) chunked linear-recurrence library.
 *
 * The library evaluates the elementwise (diagonal) first-order linear
 * recurrence
 *
 *     h_t = a_t (.) h_{t-1} + b_t ,   h_{-1} = h0 ,
 *
 * along the sequence axis as a parallel prefix scan over the associative
 * operator (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2) (earlier element on the
 * left, identity (1, 0)), and the computations built on that scan (SRU and
 * LSTM cells, forward and backward; DEER solve and its gradient).
 *
 * Sources (blog.hotdry.top, all dated 2025-09-21):
 *   [P1] "CUDA并行化RNN训练：从O(T)到O(log T)的工程实践与参数调优":
 *        SRU paragraph (forget gate without h_{t-1}, highway reset gate),
 *        parallel-scan paragraph (associative operation, divide and conquer
 *        in log T for forward and backward), checklist item 2 (fuse all
 *        sigmoid/tanh/multiply-add into one kernel).
 *   [P2] "RNN CUDA内核优化：实现序列长度无关的恒定推理延迟":
 *        LSTM paragraph (C_t = f_t*C_{t-1} + i_t*C~_t is a linear recurrence,
 *        tree reduction in log2 T stages), memory paragraph (shared-memory
 *        tiling, coalesced access, warp-level non-divergent boundaries).
 *   [P4] DEER page (.../cuda-parallel-rnn-training-logt-optimization),
 *        section "核心原理：DEER 框架与牛顿法的工程映射" (Newton form, the three
 *        steps, the linear inverse solved as a prefix scan) and section
 *        "工程实现：CUDA 内核与内存布局的关键参数" (stop at ||y^(i+1)-y^(i)|| < eps
 *        or K_max).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Sequence tensors are [T, B, D] row-major with D contiguous (channel
 *    c = b*D + d, element (t, c) at offset t*B*D + c).  Per-step state tensors
 *    (h0, dh0, c0, dc0) are [B, D].  Per-feature parameters (w and the
 *    biases bf, br, bi, bc, bo, and their gradients) are [D] and always fp32.
 *  - `dtype` is the storage type of every sequence and state tensor:
 *    LR_F32 (fp32) or LR_BF16 (bfloat16).  All arithmetic is fp32; bf16
 *    results are rounded to nearest-even when stored.
 *  - All pointers are DEVICE pointers owned by the caller; the library never
 *    frees or retains them.  Inputs are read-only.  No output may alias an
 *    input or another output.  Pointers must be aligned to the element size;
 *    16-byte alignment plus D a multiple of 4 selects the vector path (4
 *    channels per lane: 16-byte fp32 / 8-byte bf16 accesses), anything else
 *    the scalar path.  On the vector path, when a time row (B*D elements) is
 *    a multiple of 16 bytes and at least 128 channels wide, tiles are staged
 *    through shared memory by the Tensor Memory Accelerator.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous on it except the DEER solves, which enqueue their Newton
 *    iterations in batches -- the first as long as the previous solve of the
 *    same form and shape took, then four -- and synchronise the stream once
 *    per batch to read the residuals (an iteration enqueued after the
 *    stopping test was met does no work).
 *  - Sizes: B, T, D >= 0 with B*T*D < 2^62; an empty problem is a no-op
 *    (gradients of the initial state are zeroed).
 *  - The library keeps one internal workspace per device (carry packets of
 *    the chunk states and aggregates, a tile ticket, an error word, DEER's
 *    second iterate buffer, residual slots, per-sequence stop state, clamp
 *    counters and the last iteration count of each DEER form and shape,
 *    bias-gradient partials), grown on demand with cudaMalloc.  Calls on
 *    different streams are serialised through it with CUDA events; every
 *    call records its event on every return once it has begun enqueueing,
 *    errors included, so a later call on another stream still waits for
 *    whatever a failed call enqueued.
 *  - CUDA graphs: the carry packets are tagged with an epoch that the kernels
 *    take on the device from the workspace's ticket word (every launch takes
 *    a fresh one), so a call of lr_scan_fwd, lr_scan_bwd, sru_fwd, sru_bwd,
 *    lstm_cell_fwd, lstm_cell_bwd or deer_diag_bwd captured into a graph
 *    gives the right result on every replay, with whatever the captured
 *    buffers hold then.  Make one uncaptured call of the same shape first
 *    (it sizes the workspace and sets up the kernels; capture fails if the
 *    workspace would have to grow).  A graph keeps using the workspace
 *    buffers it captured: the carry packets and the bias partials that a
 *    later, larger call outgrows are kept, not freed, until the process
 *    exits (lr_workspace_bytes counts the current ones only).  A captured
 *    call is ordered, when the graph runs, by the stream the graph is
 *    launched on only: do not run it concurrently with other calls on the
 *    same device.  The DEER solves read residuals back on the host and
 *    cannot be captured.
 *  - Return value: LR_OK, or an lr_status describing an argument or launch
 *    error detected before or while enqueuing the work.  Errors detected on
 *    the device while the kernels run (a carry or copy wait that ran out) are
 *    recorded in a sticky device error word read by lr_last_error().
 *  - Results are bitwise reproducible from run to run: every floating-point
 *    association depends on the shape and on which kernel the alignment
 *    selects, never on timing.
 */
#ifndef LRSCAN_H
#define LRSCAN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { LR_F32 = 0, LR_BF16 = 1 } lr_dtype;

typedef enum {
    LR_OK = 0,
    LR_ERR_INVALID_ARG = 1,   /* NULL required pointer, negative size, bad dtype */
    LR_ERR_ALIGN = 2,         /* pointer not aligned to its element size */
    LR_ERR_CUDA = 3,          /* a CUDA runtime call failed (message: lr_cuda_error_string) */
    LR_ERR_TIMEOUT = 4,       /* device: a carry wait ran out; outputs are NaN */
    LR_ERR_NONFINITE = 5,     /* DEER: a residual was NaN or Inf */
    LR_ERR_NOT_CONVERGED = 6, /* DEER: kmax iterations without residual < eps */
    LR_ERR_TOO_LARGE = 7      /* sizes beyond the supported range */
} lr_status;

/*
 * Forward scan (row a1): h_t = a_t * h_{t-1} + b_t for t = 0..T-1 with
 * h_{-1} = h0.  [P1] parallel-scan paragraph; [P2] LSTM paragraph.
 * Chunks of time rows are scanned in parallel; the state entering each chunk
 * comes from the aggregates of the chunks before it (for T <= 2048, the CTAs
 * of one thread-block cluster pass them through distributed shared memory;
 * otherwise they are published to global memory: a look-back over all of them
 * for short problems, walkers -- whole CTAs, or one warp in each CTA of the
 * warp-specialised kernel -- for long ones, a CTA walking its channel strip
 * through time for wide ones).
 *   a, b : [T,B,D] in   coefficients and inputs
 *   h0   : [B,D]   in   initial state; NULL means zeros
 *   h    : [T,B,D] out  states (h0 is not repeated in h)
 */
int lr_scan_fwd(const void* a, const void* b, const void* h0, void* h,
                int64_t B, int64_t T, int64_t D, int dtype, void* stream);

/*
 * Backward scan (row a2): BPTT of the forward scan for the loss whose
 * gradient with respect to every h_t is dh_t.  With
 *   delta_{T-1} = dh_{T-1},  delta_t = dh_t + a_{t+1} delta_{t+1}:
 *   db_t = delta_t,  da_t = delta_t h_{t-1} (h_{-1} = h0),  dh0 = a_0 delta_0.
 * [P1] parallel-scan paragraph (the same log-depth scan serves backward).
 *   a, h, dh : [T,B,D] in   (h = output of lr_scan_fwd)
 *   h0       : [B,D]   in   NULL means zeros
 *   da, db   : [T,B,D] out
 *   dh0      : [B,D]   out  may be NULL (not computed)
 */
int lr_scan_bwd(const void* a, const void* h, const void* h0, const void* dh,
                void* da, void* db, void* dh0,
                int64_t B, int64_t T, int64_t D, int dtype, void* stream);

/*
 * SRU layer forward, linear form (row a3), fused into one scan launch.
 * [P1] SRU paragraph and checklist item 2:
 *   f_t = sigmoid(uf_t + bf),  r_t = sigmoid(ur_t + br)
 *   c_t = f_t c_{t-1} + (1 - f_t) xt_t   (c_{-1} = c0)
 *   h_t = r_t tanh(c_t) + (1 - r_t) x_t
 *   xt, uf, ur, x : [T,B,D] in   precomputed projections and highway input
 *   bf, br        : [D] fp32 in  forget / reset biases
 *   c0            : [B,D]   in   NULL means zeros
 *   h, c          : [T,B,D] out  (c is kept for sru_bwd)
 */
int sru_fwd(const void* xt, const void* uf, const void* ur, const void* x,
            const float* bf, const float* br, const void* c0, void* h, void* c,
            int64_t B, int64_t T, int64_t D, int dtype, void* stream);

/*
 * SRU layer backward (row a4), given the forward c and the upstream dh:
 *   dr = dh (tanh c - x), dur = dr r (1-r), dx = dh (1-r),
 *   dc_t = dh_t r_t (1 - tanh^2 c_t) + f_{t+1} dc_{t+1}   (reverse scan)
 *   dxt = dc (1-f), duf = dc (c_{t-1} - xt) f (1-f), dc0 = f_0 dc_0,
 *   dbf[d] = sum_{t,b} duf,  dbr[d] = sum_{t,b} dur  (deterministic order).
 *   dxt, duf, dur, dx : [T,B,D] out;  dbf, dbr : [D] fp32 out (overwritten);
 *   dc0 : [B,D] out, may be NULL.
 */
int sru_bwd(const void* xt, const void* uf, const void* ur, const void* x,
            const float* bf, const float* br, const void* c0, const void* c,
            const void* dh, void* dxt, void* duf, void* dur, void* dx,
            float* dbf, float* dbr, void* dc0,
            int64_t B, int64_t T, int64_t D, int dtype, void* stream);

/*
 * DEER solve of the diagonal tanh RNN h_t = tanh(w (.) h_{t-1} + u_t) (row a5).
 * [P4] "核心原理": Newton iteration from the all-zero guess; iteration k
 * builds, from the previous iterate shifted by one step (ytil_{-1} = h0),
 *   s_t = w ytil_{t-1} + u_t,  J_t = w (1 - tanh^2 s_t),
 *   rhs_t = tanh(s_t) - J_t ytil_{t-1},
 * and solves y_t = J_t y_{t-1} + rhs_t by the scan (one fused launch).
 * [P4] "工程实现": stop at the first k with max|y^(k) - y^(k-1)| < eps (max
 * over all B*T*D entries) or at k = kmax.
 *   w          : [D] fp32 in
 *   u          : [T,B,D] in;  h0 : [B,D] in (NULL = zeros)
 *   y          : [T,B,D] out  the last iterate
 *   iters_out  : host int out, iterations performed (>= 1 unless T*B*D = 0)
 *   resid_out  : host float out, residual of the last iteration (may be NULL)
 *   resid_hist : host float[kmax] out, residual of every iteration (may be NULL)
 * Returns LR_ERR_NOT_CONVERGED or LR_ERR_NONFINITE (with y, iters and
 * residuals still written) when the iteration did not reach eps.
 */
int deer_diag_solve(const float* w, const void* u, const void* h0, void* y,
                    int64_t B, int64_t T, int64_t D, float eps, int kmax,
                    int* iters_out, float* resid_out, float* resid_hist,
                    int dtype, void* stream);

/*
 * DEER solve with an initial guess and a choice of stopping test (the next
 * row on the same scan).  [P4] "核心原理": the Newton iteration needs few steps
 * when the initial guess is close to the solution (in training, the previous
 * step's); [P4] "工程实现": stop at ||y^(i+1) - y^(i)|| < eps or K_max.
 *   y_init       : [T,B,D] in, the initial guess y^(0) (NULL = zeros); iteration 1
 *                  builds J and rhs from it and its residual is max|y^(1) - y^(0)|.
 *                  It may be y itself (the guess is copied first); no other
 *                  overlap with y is allowed.
 *   per_sequence : 0 = one stopping test over the whole batch (deer_diag_solve);
 *                  1 = each batch sequence b stops at its own first K_b with
 *                  max over (t, d) |y^(K_b) - y^(K_b - 1)| < eps (or a non-finite
 *                  residual -- one NaN entry makes it NaN -- or kmax); y[:, b] is
 *                  its iterate K_b.  Iterations continue until every sequence
 *                  stopped; a stopped sequence is no longer written, so a
 *                  sequence that turned non-finite stops alone.
 *   iters_out    : host int out, the largest K_b (per_sequence) or K
 *   resid_out    : host float out (may be NULL): the largest final residual
 *   resid_hist   : host float[kmax] out (may be NULL): residual of every
 *                  iteration (per_sequence: the largest over the sequences that
 *                  ran it)
 *   seq_iters    : host int[B] out (may be NULL): K_b (K for every b when
 *                  per_sequence = 0)
 *   seq_resid    : host float[B] out (may be NULL): each sequence's residual at K_b
 *   launched_out : host int out (may be NULL): the kernels the solve enqueued --
 *                  the iterations, including those that returned at once after
 *                  the solve stopped, and for long, narrow problems the pass that
 *                  publishes iteration 1's segment aggregates before it and the
 *                  one-thread kernel that closes the solve (per_sequence: also
 *                  the stop-state update after every iteration and the final
 *                  gather)
 * Status as deer_diag_solve: LR_ERR_NONFINITE if any sequence's residual was not
 * finite, else LR_ERR_NOT_CONVERGED if any sequence reached kmax without eps.
 */
int deer_diag_solve_ex(const float* w, const void* u, const void* h0, const void* y_init,
                       void* y, int64_t B, int64_t T, int64_t D, float eps, int kmax,
                       int per_sequence, int* iters_out, float* resid_out, float* resid_hist,
                       int* seq_iters, float* seq_resid, int* launched_out, int dtype,
                       void* stream);

/*
 * DEER solve in the ODE form (the next row on the same scan).  [P4] "监控与调优":
 * the coefficients of the linear inverse operator are exp(-G_i dt_i), with the
 * elements of G_i clamped to [-10, 10] and the clamps counted.  The ODE is the
 * continuous-time diagonal tanh RNN dy/dt = -y + tanh(w (.) y + u) on steps
 * dt[t], the input held at u_t over step t, y_{-1} = h0.  Iteration k
 * linearises at the previous iterate ytil (ytil_{-1} = h0; zeros before the
 * first iteration):
 *   G_t = 1 - w (1 - tanh^2(w ytil_{t-1} + u_t)) clamped to [-10, 10],
 *   z_t = (tanh(w ytil_{t-1} + u_t) - ytil_{t-1}) + G_t ytil_{t-1},
 *   y_t = exp(-G_t dt_t) y_{t-1} + (1 - exp(-G_t dt_t)) / G_t z_t  (dt_t z_t if G_t = 0),
 * one scan per iteration; the fixed point is the exponential-Euler rollout.
 * Stopping rule, outputs and statuses as deer_diag_solve.
 *   dt          : [T] fp32 in, step lengths (device)
 *   clamps_out  : host int64 out (may be NULL): clamped G evaluations of the
 *                 last iteration
 */
int deer_ode_solve(const float* w, const void* u, const float* dt, const void* h0, void* y,
                   int64_t B, int64_t T, int64_t D, float eps, int kmax, int* iters_out,
                   float* resid_out, float* resid_hist, int64_t* clamps_out, int dtype,
                   void* stream);

/*
 * Gradient through the DEER solution (the next row on the same scan):
 * [P4] "核心原理": at the fixed point y is the rollout of
 * h_t = tanh(w (.) h_{t-1} + u_t), so the gradient of a loss L with upstream
 * g = dL/dy is back-propagation through it, one reverse scan with coefficient
 * J_{t+1} = w (1 - y_{t+1}^2):
 *   delta_t = g_t + J_{t+1} delta_{t+1}  (delta_{T-1} = g_{T-1}),
 *   du_t = delta_t (1 - y_t^2),  dw_d = sum over t and batch of du_t y_{t-1},
 *   dh0 = w (1 - y_0^2) delta_0  (y_{-1} = h0).
 *   w      : [D] fp32 in;   y : [T,B,D] in, the solution (deer_diag_solve)
 *   h0     : [B,D] in (NULL = zeros);  dy : [T,B,D] in, the upstream gradient
 *   du     : [T,B,D] out;  dw : [D] fp32 out;  dh0 : [B,D] out (NULL = skip)
 * Asynchronous on `stream`.  Uses the workspace's per-tile partial sums for dw
 * (a fixed-order reduction: bitwise reproducible).
 */
int deer_diag_bwd(const float* w, const void* y, const void* h0, const void* dy, void* du,
                  float* dw, void* dh0, int64_t B, int64_t T, int64_t D, int dtype,
                  void* stream);

/*
 * LSTM cell-state scan with a fused gate producer (the next row on the same
 * scan).  [P2] LSTM paragraph: the cell update C_t = f_t C_{t-1} + i_t C~_t is
 * a linear recurrence in C with time-varying coefficients; checklist item 1:
 * the GILR-style cell, whose gate pre-activations come from the input only
 * (precomputed projections, no h_{t-1} term), keeps it linear.  One launch:
 *   f = sigmoid(zf + bf),  i = sigmoid(zi + bi),  C~ = tanh(zc + bc),
 *   o = sigmoid(zo + bo),
 *   C_t = f_t C_{t-1} + i_t C~_t   (C_{-1} = c0),   h_t = o_t tanh(C_t).
 *   zf, zi, zc, zo : [T,B,D] in   gate pre-activations (forget, input,
 *                                 candidate, output)
 *   bf, bi, bc, bo : [D] fp32 in  their biases
 *   c0             : [B,D]   in   NULL means zeros
 *   h, c           : [T,B,D] out  (c is kept for lstm_cell_bwd)
 * The GILR cell is the case zi = -zf, bi = -bf (i = 1 - f).
 */
int lstm_cell_fwd(const void* zf, const void* zi, const void* zc, const void* zo,
                  const float* bf, const float* bi, const float* bc, const float* bo,
                  const void* c0, void* h, void* c,
                  int64_t B, int64_t T, int64_t D, int dtype, void* stream);

/*
 * LSTM cell backward, given the forward c and the upstream dh = dL/dh_t
 * (back-propagation through time; the cell gradient is the reverse scan):
 *   dC_t = dh_t o_t (1 - tanh^2 C_t) + f_{t+1} dC_{t+1},
 *   dzf = dC C_{t-1} f (1-f),  dzi = dC C~ i (1-i),  dzc = dC i (1 - C~^2),
 *   dzo = dh tanh(C) o (1-o),  dc0 = f_0 dC_0,
 *   db*[d] = sum over t and batch of dz* (deterministic order).
 *   dzf, dzi, dzc, dzo : [T,B,D] out;  dbf, dbi, dbc, dbo : [D] fp32 out
 *   (overwritten);  dc0 : [B,D] out, may be NULL.
 */
int lstm_cell_bwd(const void* zf, const void* zi, const void* zc, const void* zo,
                  const float* bf, const float* bi, const float* bc, const float* bo,
                  const void* c0, const void* c, const void* dh,
                  void* dzf, void* dzi, void* dzc, void* dzo,
                  float* dbf, float* dbi, float* dbc, float* dbo, void* dc0,
                  int64_t B, int64_t T, int64_t D, int dtype, void* stream);

/*
 * Forward scan that allocates nothing (no counterpart in the pages: this is a
 * deployment variant of lr_scan_fwd, same arguments and results).
 * For callers that may not allocate device memory: code running under an
 * engine or framework that owns every device byte (a hidden cudaMalloc can
 * fail at run time or fragment its pool) and latency-critical loops (the
 * cudaFree that grows lr_scan_fwd's cached workspace synchronises the device).
 * Its scratch (chunk-state or chunk-aggregate packets, tile ticket) is one
 * fixed 8 MiB __device__ array that every GPU loading this library holds
 * until the process exits.
 *   - Problems needing more scratch than that return LR_ERR_TOO_LARGE: the
 *     array holds ~1 M 8-byte packets, one per channel per chunk of 32 fp32
 *     or 64 bf16 time steps, two for short problems (look-back protocol),
 *     three per chunk of 64 steps for long ones (walker protocol), none for
 *     T <= 2048 (cluster kernel); e.g. B*D = 1024 channels up to T = 16 K
 *     fp32 steps.
 *   - All calls share the array: calls whose kernels overlap on the GPU race
 *     and give wrong results; order them on one stream or with events.
 *   - Every call clears the array's internal error word and tile counter
 *     (one 8-byte memset on `stream`) before its launch.
 *   - The first call on a device looks up the array's address; make it before
 *     any stream capture.
 *   - err_dev: optional device word (4-byte aligned) into which device-side
 *     errors are OR-ed (bit 0: a carry wait ran out; h is then NaN).  The
 *     library never clears it: set it to zero before a call whose errors you
 *     want to tell apart.  With err_dev == NULL the errors go to the array's
 *     internal word, which nothing can read (lr_last_error() reads the other
 *     workspace): pass err_dev whenever a timed-out wait must be detected.
 */
int lr_scan_fwd_noalloc(const void* a, const void* b, const void* h0, void* h,
                        int64_t B, int64_t T, int64_t D, int dtype,
                        uint32_t* err_dev, void* stream);

/*
 * Reads and clears the device error word of the current device (synchronises
 * the device).  Returns LR_OK or the first recorded device error
 * (LR_ERR_TIMEOUT).  After an error it also resets the tile ticket, which a
 * launch that gave up leaves mid-count: call it after LR_ERR_TIMEOUT before
 * any further call on that device.
 */
int lr_last_error(void);

/* Static text for a status code. */
const char* lr_status_str(int status);

/* Text of the last CUDA runtime error seen by this thread's calls. */
const char* lr_cuda_error_string(void);

/* Bytes of device workspace currently held on the current device. */
int64_t lr_workspace_bytes(void);

/* Operations and carry protocols, as lr_plan_info names them. */
typedef enum {
    LR_OP_SCAN_FWD = 0,
    LR_OP_SCAN_BWD = 1,
    LR_OP_SRU_FWD = 2,
    LR_OP_SRU_BWD = 3,
    LR_OP_DEER = 4,
    LR_OP_DEER_BWD = 5,
    LR_OP_LSTM_FWD = 6,
    LR_OP_LSTM_BWD = 7,
    LR_OP_DEER_ODE = 8
} lr_op;
typedef enum {
    LR_PROTO_CHAIN = 0,   /* a tile waits for the state after the chunk before it,
                             or a CTA walks its channel strip through time */
    LR_PROTO_WALK = 1,    /* walker warps fold the published chunk aggregates */
    LR_PROTO_LOOK = 2,    /* every tile folds all earlier chunks' published aggregates */
    LR_PROTO_CLUSTER = 3  /* one thread-block cluster per channel tile, aggregates
                             passed through distributed shared memory */
} lr_protocol;

/*
 * The carry protocol a call of operation `op` plans for a problem of T steps
 * and C = B*D channels, from the shape alone: no device is needed and nothing
 * is launched.  `vec` is 1 when the call takes the 16-byte path (D a multiple
 * of 4 and every array 16-byte aligned).  Outputs (each may be NULL):
 *   protocol  : one of lr_protocol
 *   tma       : 1 when the chain or walker protocol stages tiles by TMA
 *   tile_rows : time rows of a chunk
 *   n_chunks  : ceil(T / tile_rows)
 * Within a protocol the launcher still picks the kernel at launch (strip or
 * TMA chain; warp-specialised, register or segmented walker).  Returns LR_OK,
 * or LR_ERR_INVALID_ARG for an unknown op or dtype or T, C < 1 (an empty
 * problem launches nothing).
 */
int lr_plan_info(int op, int dtype, int vec, int64_t T, int64_t C, int* protocol, int* tma,
                 int64_t* tile_rows, int64_t* n_chunks);

/*
 * Test hook for the bounded carry waits: launches both chain-protocol
 * forward scan kernels (register and TMA-staged) and the look-back kernel on
 * private 2-chunk problems whose first chunk is never published, one CTA
 * each, the cluster kernel on a private 2-chunk problem whose CTAs each
 * expect one chunk aggregate more than they receive, and the walker-protocol
 * kernels (the register one on the fp32 scalar
 * path, the warp-specialised one on the fp32 vector path, the segmented one
 * for a bf16 backward scan, and its consume-only form for a fp32 DEER
 * iteration whose aggregates count as published) on a private long problem
 * with no walkers, so no entering state is ever published.  Every wait is
 * limited to `spin_limit` polls and runs out.  It leaves LR_ERR_TIMEOUT in
 * the device error word.  Nothing faults or hangs.
 */
int lr_test_lookback_timeout(uint32_t spin_limit, void* stream);

/*
 * Test hook for the ordering of calls after an error: enters a call on
 * `stream` as every entry point does, enqueues a kernel that sleeps about
 * `sleep_ns` nanoseconds (bounded by the GPU's global timer) and then sets
 * x[0..n) to `value` (x: n fp32 device values, caller-owned), and returns
 * LR_ERR_CUDA as a call whose later launch failed would.  A following call
 * on another stream must still be ordered after that kernel.  Returns
 * LR_ERR_INVALID_ARG for n < 0 or x == NULL with n > 0.
 */
int lr_test_fail_after_enqueue(float* x, int64_t n, float value, uint64_t sleep_ns,
                               void* stream);

/*
 * Test hook for the activations of the fused kernels: tanh_out[i] = tanh(x[i]),
 * sigmoid_out[i] = 1 / (1 + exp(-x[i])) and expm1_out[i] = exp(x[i]) - 1 as the
 * SRU, LSTM and DEER kernels evaluate them (tanh and sigmoid in exponential
 * forms on the hardware exponential; e^x - 1 by its Taylor series near 0 and
 * the hardware exponential elsewhere -- the pages name the functions, [P1]
 * SRU paragraph, [P4] "核心原理" and "监控与调优", not how to evaluate them).
 * x, tanh_out, sigmoid_out: n fp32 device values each, caller-owned;
 * expm1_out likewise or NULL (not computed).  Asynchronous on `stream`.
 * Returns LR_ERR_INVALID_ARG for n < 0 or a null required pointer with n > 0.
 */
int lr_test_activations(const float* x, float* tanh_out, float* sigmoid_out, float* expm1_out,
                        int64_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LRSCAN_H */
