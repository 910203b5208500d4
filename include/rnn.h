/*
 * rnn.h: C ABI of the GB300 head-wise recurrent scan library (librnn_gb300.so).
 *
 * The operation is the one the FlashRNN announcement (hottg.com/neural/9889,
 * "FlashRNN: optimising RNNs on modern hardware", usage example) exposes as
 *     states, last_states = flashrnn(Wx, R, b, states=states_initial, function=...)
 * with Wx[B,T,G,N,D], R[G,N,D,D], b[G,N,D], states_initial[S,B,1,N,D] and the
 * result states[S,B,T,N,D]: N independent heads of size D; per step t and head n
 *     rec_g = h_{t-1} . R[g,n] + b[g,n]      (row vector h, D x D block, g < G)
 *     a_g   = Wx[b,t,g,n,:] + rec_g           (GRU: a_n = Wx_n + r * rec_n)
 * then the pointwise update of the chosen cell. The LSTM cell (gates i,f,g,o;
 * c = f c + i g; h = o tanh c) and the row-vector orientation are those of
 * developnotes "deep learning operators", section 5.3 LSTM (MyLSTM.forward).
 * GRU (gates r,z,n; h' = (1-z) n + z h), Elman (h' = tanh a) and sLSTM (gates
 * i,f,z,o; states h,c,n,m; exponential gating with stabiliser m) follow the
 * readings documented in the repository's design notes.
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers to dense, contiguous, row-major
 *    arrays in the order given, 16-byte aligned, of element type `dtype`
 *    (RNN_BF16: bfloat16 storage with fp32 arithmetic and fp32 carried c,n,m;
 *    RNN_F32: float32 throughout). The caller owns and allocates all memory;
 *    the library allocates nothing and never synchronises the stream except
 *    in rnn_check_status. Every call is asynchronous on `stream`
 *    (a cudaStream_t; NULL = legacy default stream).
 *  - Return value: RNN_OK (0) or a status below. Host-side validation errors
 *    are returned before anything is enqueued. Device-side errors (a bounded
 *    wait that ran out) are recorded in the workspace and reported by
 *    rnn_check_status.
 *  - B = 0 is an error (RNN_EINVAL). T = 0 is not: the last states equal the
 *    initial states and the backward passes dlast through to dstates0.
 */
#ifndef RNN_GB300_H
#define RNN_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define RNN_OK 0
#define RNN_EINVAL 1      /* bad dimensions, NULL required pointer, misalignment */
#define RNN_EUNSUPPORTED 2 /* no feasible kernel plan for the requested path */
#define RNN_ENOSPC 3      /* workspace smaller than rnn_workspace_size() */
#define RNN_ETIMEOUT 4    /* a device-side wait gave up (reported by rnn_check_status) */
#define RNN_ECUDA 5       /* a CUDA runtime call or launch failed */

/* ---- enumerations ---------------------------------------------------------- */
typedef enum { RNN_LSTM = 0, RNN_GRU = 1, RNN_ELMAN = 2, RNN_SLSTM = 3, RNN_SLSTM_LOGSIG = 4 } rnn_function_t;
/* (G, S) = (4, 2) LSTM, (3, 1) GRU, (1, 1) Elman, (4, 4) sLSTM.
 * State order: LSTM h,c; GRU h; Elman h; sLSTM h,c,n,m.
 * RNN_SLSTM: exponential forget gate, log f = a_f. RNN_SLSTM_LOGSIG: sigmoid
 * forget gate, log f = log sigmoid(a_f); otherwise identical. */
typedef enum { RNN_F32 = 0, RNN_BF16 = 1 } rnn_dtype_t;
typedef enum {
  RNN_PATH_AUTO = 0,        /* the planner picks */
  RNN_PATH_FUSED = 1,       /* persistent thread-block-cluster kernel, R resident on chip */
  RNN_PATH_ALTERNATING = 2, /* a per-step matrix product and a pointwise kernel, replayed as a CUDA graph */
  RNN_PATH_SIMT = 3,        /* plain per-head kernel, any size; the fp32 path */
  RNN_PATH_GRID = 4         /* persistent cooperative grid kernel for R too large for one cluster:
                               h (forward) and dr (backward) exchanged through L2 with step counters */
} rnn_path_t;

typedef struct {
  int B, T, N, D;
  int function; /* rnn_function_t */
  int dtype;    /* rnn_dtype_t */
  int path;     /* rnn_path_t */
} rnn_dims_t;

/* Workspace kinds for rnn_workspace_size. */
#define RNN_WS_FWD 0          /* rnn_fwd */
#define RNN_WS_BWD 1          /* rnn_bwd given the forward's tape */
#define RNN_WS_BWD_RECOMPUTE 2 /* rnn_bwd with tape == NULL (re-runs the forward) */

int rnn_num_gates(int function);  /* G, or -1 for an unknown function */
int rnn_num_states(int function); /* S, or -1 */

/* Bytes of the forward tape (fp32 gate pre-activations and carried states of
 * every step, [T][B][N][K][D] floats) that rnn_bwd reads; 0 for invalid dims. */
size_t rnn_tape_size(const rnn_dims_t *dims);

/* Bytes of scratch the call of the given kind needs (a multiple of 256;
 * at least 256). 0 for invalid dims. The caller allocates it: the usage
 * example of the FlashRNN announcement passes every tensor in ("a functional
 * structure, none of the parameters are tied to the flashrnn function"), and
 * this library keeps that contract for its scratch too. The size depends on
 * the plan chosen for the current device. */
size_t rnn_workspace_size(const rnn_dims_t *dims, int kind);

/*
 * Forward scan (FlashRNN announcement, usage example: the flashrnn call).
 *   Wx      [B,T,G,N,D]  input pre-activations                         (in)
 *   R       [G,N,D,D]    recurrent blocks, R[g,n,i,j], i = input unit    (in)
 *   b       [G,N,D]      bias                                           (in)
 *   states0 [S,B,1,N,D]  initial states, or NULL = all zeros            (in)
 *   states  [S,B,T,N,D]  state after every step (initial state excluded)(out)
 *   last    [S,B,1,N,D]  state after the last step, or NULL             (out)
 *   tape    rnn_tape_size() bytes, or NULL; written for rnn_bwd         (out)
 *   workspace / ws_bytes: at least rnn_workspace_size(dims, RNN_WS_FWD)
 * Errors: RNN_EINVAL, RNN_EUNSUPPORTED, RNN_ENOSPC, RNN_ECUDA.
 */
int rnn_fwd(const rnn_dims_t *dims, const void *Wx, const void *R, const void *b,
            const void *states0, void *states, void *last, void *tape,
            void *workspace, size_t ws_bytes, void *stream);

/*
 * Backward through time of rnn_fwd (the gradient of sum(states*dstates) +
 * sum(last*dlast) with respect to every input). The FlashRNN announcement's
 * usage example creates Wx, R, b and the initial states with
 * requires_grad=True: these four gradients are what its flashrnn call
 * returns through autograd.
 *   Wx, R, b, states0  the forward's inputs (states0 may be NULL = zeros)
 *   states             the forward's output [S,B,T,N,D]
 *   tape               the tape rnn_fwd wrote for these inputs, or NULL to have
 *                      it rebuilt inside the workspace (one extra forward)
 *   dstates [S,B,T,N,D] upstream gradient, or NULL = zero
 *   dlast   [S,B,1,N,D] upstream gradient of `last`, or NULL = zero
 *   dWx [B,T,G,N,D], dR [G,N,D,D], db [G,N,D], dstates0 [S,B,1,N,D]: outputs,
 *                      each may be NULL when not wanted
 *   workspace / ws_bytes: at least rnn_workspace_size(dims, RNN_WS_BWD) with a
 *                      tape, RNN_WS_BWD_RECOMPUTE without
 * Errors: as rnn_fwd.
 */
int rnn_bwd(const rnn_dims_t *dims, const void *Wx, const void *R, const void *b,
            const void *states0, const void *states, const void *tape,
            const void *dstates, const void *dlast, void *dWx, void *dR, void *db,
            void *dstates0, void *workspace, size_t ws_bytes, void *stream);

/*
 * Backward through time without caller workspace (no counterpart on the
 * pages: this entry point exists for callers of this library that cannot
 * allocate device memory -- code embedded in a host framework that owns the
 * whole device-memory budget, or loops that must not call cudaMalloc because
 * it can synchronise the device and stall the pipeline).
 * Same arguments and results as rnn_bwd, minus the workspace; `tape` is
 * required (rebuilding it would need tape-sized scratch). The scratch lives in
 * a fixed __device__ array of RNN_BWD_NOALLOC_SCRATCH_BYTES inside the library,
 * held by every GPU that loads it until the process exits. It holds the status
 * word and, for GRU or when dWx is NULL, the recurrent-branch gradients
 * (B*T*G*N*D elements of the storage type): problems whose need exceeds the
 * array (256 bytes + those gradients) return RNN_ENOSPC before any work. The
 * rest of the array holds the weight gradient's split-K partial sums when they
 * fit; when they do not, dR is computed without splitting K, so dR and db may
 * differ from rnn_bwd's in the order of their fp32 sums (not beyond rounding).
 * Paths: only the cluster kernels and the plain kernel run here. An explicit
 * RNN_PATH_GRID or RNN_PATH_ALTERNATING returns RNN_EUNSUPPORTED (their
 * exchange buffers would need workspace); under RNN_PATH_AUTO a problem whose
 * plan is one of those runs on the plain kernel instead.
 * The first call on a device looks the array's device address up (once per
 * device); make that first call before any stream capture. Every call shares
 * the array and keeps the last call's contents: calls whose work overlaps on
 * the GPU (different streams or threads) race; calls on one stream are safe.
 * Device-side wait time-outs are recorded in the array's status word (cleared
 * at the start of every call) and read by rnn_bwd_noalloc_status.
 * Errors: RNN_EINVAL (as rnn_bwd), RNN_EUNSUPPORTED, RNN_ENOSPC, RNN_ECUDA.
 */
#define RNN_BWD_NOALLOC_SCRATCH_BYTES (16u << 20)
int rnn_bwd_noalloc(const rnn_dims_t *dims, const void *Wx, const void *R, const void *b,
                    const void *states0, const void *states, const void *tape,
                    const void *dstates, const void *dlast, void *dWx, void *dR, void *db,
                    void *dstates0, void *stream);

/* Status of the most recent rnn_bwd_noalloc call on the current device (no
 * counterpart on the pages): synchronises `stream`, reads and clears the
 * status word of the library's fixed scratch array. Returns RNN_OK,
 * RNN_ETIMEOUT (a device-side wait of that call ran out; its results are not
 * valid) or RNN_ECUDA. */
int rnn_bwd_noalloc_status(void *stream);

/* Synchronises `stream`, reads and clears the device status word that kernels
 * running on `workspace` recorded. Returns RNN_OK, RNN_ETIMEOUT or RNN_ECUDA.
 * (The pages have no device-side error path; the status-code convention --
 * validation errors returned before any work, the empty-batch error, T = 0 as
 * a copy of the initial state -- follows the precedent of ruDNN 0.2.1,
 * src/kda/prepared.rs, prepare_chunk_kda.) */
int rnn_check_status(void *workspace, void *stream);

/* Writes a one-line description of the plan chosen for dims (path, cluster
 * size, tiles) or the reason none fits into buf (NUL-terminated, truncated to
 * len). Returns RNN_OK, RNN_EINVAL or RNN_EUNSUPPORTED. The plan is the
 * solution of an integer constraint problem over the tile and cluster sizes
 * (divisibility, warp, register and shared-memory limits, cluster
 * co-residency on the current device), the role the FlashRNN announcement's
 * overview gives its ConstrINT tuner ("hardware limits written as equalities,
 * inequalities and divisibility constraints"). */
int rnn_plan_describe(const rnn_dims_t *dims, int for_backward, char *buf, size_t len);

/* Planning for a stated device (for the planner's tests and what-if sizing):
 * with sms > 0, every later plan uses these limits -- sms SMs (1 .. 4096),
 * smem_per_cta bytes of shared memory per CTA (1024 .. 1048576) and clusters
 * of at most max_cluster CTAs (1 .. 16) -- instead of the current device's,
 * and co-residency is judged from the SM count alone. sms <= 0 returns to the
 * current device. Process-global; launches on a device smaller than the stated
 * one fail. Returns RNN_OK or RNN_EINVAL. */
int rnn_plan_set_limits(int sms, int smem_per_cta, int max_cluster);

/* The GPU's two dies as the grid kernels see them (no counterpart in the
 * pages: a placement aid of this implementation). A GB300 is two dies, each
 * with its own L2; the cooperative grid kernels put each batch group's CTAs
 * on one die and the group's step counter in a 1 KB block of the workspace
 * whose L2 home is on that die, which keeps the per-step exchange's L2 round
 * trips on the die. The SM-to-die map is measured once per device with L2
 * flag round trips (about 15 ms, on an internal stream, at the first grid
 * launch or here), and the home die of the workspace's counter blocks once
 * per workspace address on the caller's stream (a host synchronisation; a
 * stream that is capturing skips it, and that launch groups CTAs by block
 * index). Writes the number of SMs on each die (die 0 holds the SM of the
 * measurement's first CTA) and returns RNN_OK, or RNN_EUNSUPPORTED when the
 * current device shows no two-die structure or cannot be measured (grid
 * kernels then group CTAs by block index). RNN_DIE_PLACEMENT=0 in the
 * environment turns the placement off for later launches. Either pointer may
 * be NULL. */
int rnn_die_layout(int *sms_die0, int *sms_die1);

/* The die placement for stated measurements instead of the current device's
 * (no GPU needed: for tests and what-if use, as rnn_plan_set_limits is for
 * the planner). sm_lat[0..nsm) are the L2 flag round trips from the
 * measuring CTA to every CTA of a one-CTA-per-SM launch, entry 0 being the
 * measuring CTA itself; blk_lat[0..nblocks) the round trips between two CTAs
 * of die 0 on each 1 KB block of the counter region (nblocks <= 16). Each set
 * splits at the midpoint of its fastest and slowest entry when the slowest
 * is at least 1.3 times the fastest (else the measurement is not trusted);
 * the fast side is die 0. `groups` batch groups of C CTAs are split over the
 * dies as evenly as fits, groups 0 .. g0-1 on die 0; each group's step
 * counter goes in the first unused block homed on its die. Writes the SMs
 * per die, g0 and each group's counter word offset (block index x 256), any
 * pointer of which may be NULL. Returns RNN_OK; RNN_EUNSUPPORTED when a
 * measurement is not trusted, no split fits or a die has too few blocks
 * homed on it; RNN_EINVAL for groups outside 1..16, C < 1, nsm outside
 * 2..4096, nblocks outside 1..16 or a NULL latency array. */
int rnn_die_plan_for(int groups, int C, const unsigned long long *sm_lat, int nsm,
                     const unsigned long long *blk_lat, int nblocks, int *sms_die0, int *sms_die1,
                     int *groups_die0, int *ctr_words);

const char *rnn_strerror(int status);

/* Number of CUDA kernels this library has enqueued since it was loaded
 * (all streams, all devices). A diagnostic counter for benchmarks. */
unsigned long long rnn_kernel_launches(void);

/* Benchmarking aid. Registers two CUDA events (cudaEvent_t, or NULL to clear)
 * that rnn_fwd (which = 0) or rnn_bwd (which = 1) record on the call's stream
 * immediately before and after launching its recurrent-scan kernel, so that
 * the scan kernel can be timed inside a longer step. Process-global and not
 * thread-safe. Returns RNN_OK or RNN_EINVAL. */
int rnn_profile_events(int which, void *before, void *after);

/* Diagnostic phase trace of the persistent kernels (cluster and grid paths)
 * and of the plain kernels.
 * Registers a device buffer of 16 * steps unsigned 64-bit words, or NULL to
 * stop. Kernels launched afterwards have CTA 0, thread 0 write clock64() at
 * up to sixteen phase points of the steps [t0, t0 + steps) of their processing order
 * (the backward processes t = T-1 first). Forward phases: 0 step start,
 * 1 h_{t-1} available, 2 partial products written, 3 after the CTA barrier,
 * 4 Wx[t] staged, 5 cell update done, 6 after the CTA barrier, 7 h_t sent,
 * 11 the step's tail done (the states and tape stores issued; thread 0 of the
 * grid kernel issues its own at the next step, after that step's pull)
 * (points 8-10 are not recorded: inside the cell's loop they cost up to a
 * tenth of the forward step).
 * Cluster backward phases: 0 step start, 1 tape staged and the gate
 * activations evaluated, 2 partial dh available, 3 cell derivative done, 4
 * after the CTA barrier, 5 partial products computed, 6 partials sent. Grid
 * backward phases: 0 step start, 1 step counter reached and the gather of dr
 * issued, 2 the first pair's tape and activations evaluated and dr gathered,
 * 3 dh reduced, 4 tape staged, 5 cell derivative done, 6 published. Plain forward: 0 step start, 1 products
 * written, 2 after the CTA barrier, 5 cell inputs loaded, 6 cell done, 3
 * outputs stored, 4 after the CTA barrier. Plain backward: 0 step start, 1
 * cell derivative done, 2 after the CTA barrier, 3 products written, 4 after
 * the CTA barrier. Process-global, not thread-safe; returns RNN_OK or
 * RNN_EINVAL. */
int rnn_trace(void *buf, int t0, int steps);

/* Fault injection for tests of the device-side time-out path. With step >= 0,
 * the forward persistent kernels (cluster and grid paths) launched afterwards
 * make CTA 0 wait, at that step, on an mbarrier that nothing signals, for at
 * most limit_ns (1 ns .. 10 s). The wait runs out, the kernel records the
 * time-out in the workspace status word and carries on; the step exchange
 * itself is untouched, so results stay correct and rnn_check_status reports
 * RNN_ETIMEOUT. step < 0 switches injection off. Process-global; returns
 * RNN_OK or RNN_EINVAL. */
int rnn_debug_inject_wait(int step, unsigned long long limit_ns);

/*
 * Input projection ahead of the scan (developnotes "deep learning operators",
 * section 5.3 LSTM, MyLSTM.forward, computes each gate's input branch as
 * x_t W_ih^T + b_ih; the FlashRNN announcement's flashrnn() takes that product
 * as its input Wx). For BT = B*T rows, on the tensor cores:
 *     Wx[m, c] = sum_i x[m, i] * W_x[c, i] + bias[c]
 *   x    [BT][I]   layer input (row m = b*T + t)                        (in)
 *   W_x  [C][I]    weights in the weight_ih layout: C = G*N*D rows in the
 *                  order of Wx's (g, n, d) axes                          (in)
 *   bias [C]       or NULL                                              (in)
 *   Wx   [BT][C]   = the scan's Wx [B,T,G,N,D]                           (out)
 * All bf16 device pointers, 16-byte aligned; I and C multiples of 8 and at
 * least 64; BT >= 1. workspace: rnn_input_proj_workspace_size() bytes (its
 * first 256 bytes hold the status word that rnn_check_status reads).
 * Errors: RNN_EINVAL, RNN_ENOSPC, RNN_ECUDA.
 */
size_t rnn_input_proj_workspace_size(int BT, int I, int C); /* 0 for invalid sizes */
int rnn_input_proj_fwd(int BT, int I, int C, const void *x, const void *W, const void *bias, void *Wx,
                       void *workspace, size_t ws_bytes, void *stream);
/* Backward of rnn_input_proj_fwd given dWx [BT][C]: dx [BT][I] = dWx W_x,
 * dW [C][I] = dWx^T x, dbias [C] = column sums of dWx; each output may be
 * NULL when not wanted. Same conventions and errors as the forward. */
int rnn_input_proj_bwd(int BT, int I, int C, const void *x, const void *W, const void *dWx, void *dx, void *dW,
                       void *dbias, void *workspace, size_t ws_bytes, void *stream);

/* Latency floor of the cluster exchange (a measurement aid). Runs a kernel
 * whose steps hold only the h exchange of the forward cluster kernel: every
 * CTA of one cluster of C CTAs (1 .. 16) stages a slice of slice_bytes
 * (16 .. 4096, a multiple of 16), sends it to every CTA of the cluster with
 * one bulk copy per peer (lane 0 of each of the 8 warps issuing every 8th
 * copy), and waits on an mbarrier transaction count (bounded, 2 s) for the C
 * slices of the step, for `steps` (2 .. 1e6) steps. Writes to out[0] the
 * clock64 cycles per step seen by CTA 0 and to out[1] the status (0 = ok,
 * 1 = a wait ran out); `out` is a device buffer of two unsigned 64-bit words
 * owned by the caller. Asynchronous on `stream`. Returns RNN_OK, RNN_EINVAL
 * or RNN_ECUDA. */
int rnn_exchange_floor(int C, int slice_bytes, int steps, void *out, void *stream);

/* Latency floor of the grid kernels' exchange through L2 (a measurement aid).
 * Runs `groups` groups of C CTAs (a cooperative launch, one CTA per SM) whose
 * steps hold only the forward grid kernel's h exchange: each CTA stores its
 * D / C units of h for `rows` batch rows (2-byte stores), one release increment
 * of the group's step counter after a CTA barrier, then the next step's
 * acquire wait on the counter (bounded, 2 s) and the pull of the group's rows
 * from L2 with one bulk copy per row, for `steps` (2 .. 1e6) steps. C >= 1,
 * groups >= 1, rows 1 .. 32, D 8 .. 4096 with D % 8 == 0 and D % C == 0.
 * The CTAs are placed as the grid kernels place theirs (each group on one die
 * with its counter homed there, see rnn_die_layout), or by block index.
 * scratch: device memory owned by the caller, 256-byte aligned, of at least
 * 2*groups*rows*D*2 bytes rounded up to 256, plus 17664 bytes (the exchange
 * buffers, then a 1 KB-aligned region of 16 KB of counter blocks and the die
 * tickets). Writes to out[0] the clock64 cycles per step seen by the first
 * CTA of group 0 and to out[1] the status (0 = ok, 1 = a wait ran out).
 * Asynchronous on `stream`. Returns RNN_OK, RNN_EINVAL, RNN_ENOSPC,
 * RNN_EUNSUPPORTED (the CTAs cannot all be resident) or RNN_ECUDA. */
int rnn_exchange_floor_grid(int C, int groups, int rows, int D, int steps, void *scratch, size_t scratch_bytes,
                            void *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* RNN_GB300_H */
