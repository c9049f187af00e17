/*
 * ss_scan.h -- C ABI of the B300 selective state space scan (Mamba S6).
 *
 * The operation (from "State Space Models and Mamba", multigrid.ai/learn/
 * mamba-ssm, section "Selective state", equations delta_t, A_t and h_t, and
 * the readout y_t = C h_t of section "It is a linear recurrence"; the
 * selection parameters as listed in "Mamba: Linear-Time Sequence Modeling
 * with Selective State Spaces", azimuth.plus, section on S6):
 *
 *   for every batch row b, channel d, step t and state n < N:
 *     dt      = softplus(delta[b,d,t] + delta_bias[d])   (or without softplus)
 *     Abar    = exp(dt * A[d,n])
 *     h[n]    = Abar * h[n] + dt * B[b,n,t] * u[b,d,t]
 *     y[b,d,t]= (sum_n C[b,n,t] * h[n] + D[d] * u[b,d,t]) * silu(z[b,d,t])
 *
 * D (the skip term of the four-matrix model, "State space models and Mamba:
 * reading long sequences without attention", ai-trend.me, "Core idea") and
 * the SiLU gate z (branch B of the Mamba block, "What a Mamba block actually
 * contains", multigrid.ai) are optional.  The state h starts at zero.
 *
 * Layouts (row-major, C order; every array dense and contiguous):
 *   u, delta, z, y : (batch, dim, seqlen)   -- time is the fastest index
 *   B, C           : (batch, dstate, seqlen) -- shared by all channels of a row
 *   A              : (dim, dstate)  fp32
 *   D, delta_bias  : (dim)          fp32
 *   last_state     : (batch, dim, dstate) fp32
 * u, delta, B, C and z share one element type (ss_dims.in_dtype): fp32 or
 * bf16.  A, D, delta_bias, y and every state are always fp32.
 *
 * Pointers are DEVICE pointers (cudaMalloc'd or otherwise device-accessible
 * memory of the current device).  The caller owns every buffer, including
 * the chunked workspace; the library allocates nothing, never synchronises,
 * and enqueues all work on the given stream (NULL = legacy default stream).
 *
 * Errors: each call returns an ss_status.  Argument errors are detected on
 * the host before anything is launched (nothing is written then).  A failed
 * launch returns SS_ECUDA; ss_last_cuda_error() gives the CUDA error code.
 * Nothing aborts and nothing throws.
 */
#ifndef SS_SCAN_H
#define SS_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (same underlying type); NULL selects the legacy default stream. */
typedef struct CUstream_st* ss_stream_t;

typedef enum { SS_F32 = 0, SS_BF16 = 1 } ss_dtype;

typedef enum {
    SS_OK = 0,
    SS_EINVAL = -1,      /* bad size, missing required pointer, unsupported dstate */
    SS_EALIGN = -2,      /* a pointer is not aligned to its element size */
    SS_EDTYPE = -3,      /* in_dtype is neither SS_F32 nor SS_BF16 */
    SS_EWORKSPACE = -4,  /* chunked workspace missing, too small or misaligned */
    SS_ECUDA = -5,       /* a CUDA launch or call failed (see ss_last_cuda_error) */
    SS_ETIMEOUT = -6,    /* a bounded device-side wait gave up (see ss_device_status) */
    SS_EBOUNDS = -7      /* a device-side index check failed (SS_DEBUG_BOUNDS build only) */
} ss_status;

/* Largest supported state size N. */
#define SS_MAX_DSTATE 64

/*
 * Discretisation flag (ss_dims.flags).  Without it the input enters as the
 * equations print it, dt * B * u ("Selective state", multigrid.ai).  With
 * SS_FLAG_ZOH it enters with the zero-order-hold weight (exp(dt A) - 1) / A
 * (dt in the limit A -> 0): the exact solution over a step with the input held
 * constant, under which Theorem 1 of "Mamba: Linear-Time Sequence Modeling with
 * Selective State Spaces" (azimuth.plus) holds exactly (N = 1, A = -1 gives the
 * gated RNN h = (1 - sigmoid(g)) h + sigmoid(g) x).  Abar = exp(dt A) either way.
 */
#define SS_FLAG_ZOH 1

/*
 * Schedule flags, accepted by ss_scan_fwd and ss_scan_fwd_h0 only (other entry
 * points reject them with SS_EINVAL).  Both schedules compute the same
 * recurrence; results differ only in rounding order.
 *   SS_FLAG_SCHED_THREAD  one thread per channel holds the channel's N states
 *                         and walks all L steps.
 *   SS_FLAG_SCHED_WARP    one warp per channel: each lane owns 16 consecutive
 *                         steps of a 512-step segment, and the lanes' (decay
 *                         product, state) pairs are combined by a warp-shuffle
 *                         scan under the associative operator of the recurrence
 *                         ("Parallel scan", azimuth.plus).  Needs
 *                         1 <= N <= 16, L a multiple of 8 and 16-byte aligned
 *                         u, delta, z, y, B and C (either input weight);
 *                         otherwise SS_EINVAL.
 * With neither flag the library picks: the warp schedule where it is available
 * and batch * dim < 9216 (< 20480 with SS_FLAG_ZOH): too few channels to fill
 * the GPU one thread each; else the thread schedule.  Both flags together:
 * SS_EINVAL.
 */
#define SS_FLAG_SCHED_THREAD 2
#define SS_FLAG_SCHED_WARP 4

typedef struct {
    int64_t batch;     /* >= 0; at most 65535 */
    int64_t dim;       /* channels D, >= 0 */
    int64_t dstate;    /* state size N, 0 .. SS_MAX_DSTATE */
    int64_t seqlen;    /* sequence length L, >= 0 (ignored by ss_state_update) */
    int32_t in_dtype;  /* ss_dtype of u, delta, B, C, z */
    int32_t flags;     /* SS_FLAG_ZOH, plus SS_FLAG_SCHED_* where accepted; other bits: SS_EINVAL */
} ss_dims;

/*
 * Full-sequence scan (the "parallel" training/prefill face of the layer;
 * "The same layer has two faces", multigrid.ai, section "Why a linear
 * recurrence can be trained in parallel").  One pass over L per channel with
 * the state kept on chip; the (batch, L, dim, N) expanded state is never
 * written to device memory (ai-trend.me, "How it works"; azimuth.plus,
 * "Kernel fusion").
 *   u, delta, B, C, A, y   required (unless the corresponding size is 0)
 *   D, z, delta_bias       optional (NULL = absent: D = 0, no gate, bias 0)
 *   softplus_flag          nonzero: dt = softplus(delta + bias); zero: dt = delta + bias
 *   last_state             optional output: h after the last step (zeros if L = 0)
 */
int ss_scan_fwd(const ss_dims* dims, const void* u, const void* delta, const float* A,
                const void* B, const void* C, const float* D, const void* z,
                const float* delta_bias, int softplus_flag, float* y, float* last_state,
                ss_stream_t stream);

/*
 * Bytes of caller-provided device workspace that ss_scan_chunked needs for
 * these dims and chunk length (0 on invalid arguments).
 */
size_t ss_scan_chunked_workspace_bytes(const ss_dims* dims, int64_t chunk_len);

/*
 * Chunked scan for long sequences: the same result as ss_scan_fwd, computed
 * as (1) a local zero-start scan of every chunk of chunk_len steps but the
 * last, giving the chunk's end state and its decay product, (2) an exclusive
 * scan across chunks of the (decay product, state) pairs under the associative
 * operator (a1,b1) o (a2,b2) = (a1*a2, a2*b1 + b2), which gives each chunk its
 * true starting state, and (3) a fix-up pass that runs every chunk from that
 * state, writes y, and writes last_state from the last chunk.  The recurrence
 * is associative ("Parallel scan", azimuth.plus), which is what makes chunks
 * independent.  The local scan only needs each chunk's end state: walking a
 * chunk backward from its end, a state's remaining terms are exact zeros once
 * its weight exp(A R) underflows in fp32, and (with the softplus on) they are
 * left out, with the channels grouped by decay speed so that whole warps
 * stop together; the results are those of the full walk.
 *   chunk_len        >= 1
 *   workspace        device memory of at least ss_scan_chunked_workspace_bytes,
 *                    256-byte aligned; its contents on entry are ignored
 * Other arguments as ss_scan_fwd.  Three to four kernels are launched on
 * `stream` (none for the local scan when there is a single chunk).
 */
int ss_scan_chunked(const ss_dims* dims, const void* u, const void* delta, const float* A,
                    const void* B, const void* C, const float* D, const void* z,
                    const float* delta_bias, int softplus_flag, float* y, float* last_state,
                    int64_t chunk_len, void* workspace, size_t workspace_bytes,
                    ss_stream_t stream);

/*
 * One phase of ss_scan_chunked, for callers that schedule the phases
 * themselves (for example to time them, or to run other work between them).
 * Calling phases SS_PHASE_LOCAL, SS_PHASE_CARRY and SS_PHASE_FIXUP in this
 * order on one stream, with the same arguments and workspace, is exactly
 * ss_scan_chunked.  The local phase launches up to two kernels (the channel
 * order, then the local scan), the others one each.  The fix-up phase writes
 * y and last_state (the carry phase writes last_state only when L = 0).
 */
typedef enum { SS_PHASE_LOCAL = 1, SS_PHASE_CARRY = 2, SS_PHASE_FIXUP = 3 } ss_phase;

int ss_scan_chunked_phase(int phase, const ss_dims* dims, const void* u, const void* delta, const float* A,
                          const void* B, const void* C, const float* D, const void* z,
                          const float* delta_bias, int softplus_flag, float* y, float* last_state,
                          int64_t chunk_len, void* workspace, size_t workspace_bytes,
                          ss_stream_t stream);

/*
 * The same scans started from a given state instead of zeros: h0 is a
 * (batch, dim, dstate) fp32 device array (NULL = zeros) read before the first
 * step.  Running L1 steps, then L2 more steps from the first call's
 * last_state, gives the same y and final state as one call over L1 + L2 steps
 * (up to rounding order): a prompt's state can be computed once and reused,
 * as the recurrence face of the layer allows ("What it costs", multigrid.ai:
 * a shared system prompt replayed into a state).  With L = 0, last_state = h0.
 * Other arguments, results and errors as ss_scan_fwd / ss_scan_chunked;
 * SS_EALIGN if h0 is not 4-byte aligned.
 */
int ss_scan_fwd_h0(const ss_dims* dims, const float* h0, const void* u, const void* delta, const float* A,
                   const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                   int softplus_flag, float* y, float* last_state, ss_stream_t stream);

int ss_scan_chunked_h0(const ss_dims* dims, const float* h0, const void* u, const void* delta, const float* A,
                       const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                       int softplus_flag, float* y, float* last_state, int64_t chunk_len, void* workspace,
                       size_t workspace_bytes, ss_stream_t stream);

/*
 * One decode step on a persistent state (the recurrence face: a token costs
 * one update of a state whose size does not grow with the sequence;
 * mernstackdev.com, FAQ, and multigrid.ai, "The state, in bytes", which sizes
 * that (batch, dim, N) state).  dims->seqlen is ignored.
 *   state   (batch, dim, dstate) fp32, read and updated in place
 *   u, delta, z, y : (batch, dim)      B, C : (batch, dstate)
 * Other arguments as ss_scan_fwd.  Running L steps from a zero state gives
 * the same y and final state as ss_scan_fwd over those L steps.  Consecutive
 * calls on the same state pointer walk the state in opposite orders (a step
 * first reads what the previous one wrote last, while it is still in L2); the
 * order never changes a result.  Thread-safe; the per-pointer alternation is
 * kept on the host, so steps captured into a CUDA graph alternate as captured.
 */
int ss_state_update(const ss_dims* dims, float* state, const void* u, const void* delta,
                    const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* delta_bias, int softplus_flag, float* y,
                    ss_stream_t stream);

/*
 * ss_scan_chunked without a caller-provided workspace, for callers that cannot
 * allocate device memory themselves: code running where cudaMalloc is not
 * allowed or not wanted (inside a custom allocator or memory pool, a plugin
 * host that owns all device allocations, or a deployment that forbids
 * allocation after start-up).  The pages have no counterpart of this entry
 * point; it only changes who owns the workspace.
 *
 * The workspace is a fixed array of SS_STATIC_WORKSPACE_BYTES bytes inside the
 * library: every GPU that loads the library holds it until the process exits.
 * The caller still passes every input and output, as for ss_scan_chunked.
 *   - Returns SS_EWORKSPACE, without touching the device, when
 *     ss_scan_chunked_workspace_bytes(dims, chunk_len) exceeds
 *     SS_STATIC_WORKSPACE_BYTES (16 MiB: for example batch 1, dim 5120, N 16,
 *     L 65536 with chunk 2048 needs 11.3 MB).
 *   - Every call made outside a stream capture looks up the array's device
 *     address with cudaGetSymbolAddress (under a lock, with that device
 *     current); a call made while its stream is being captured uses the address
 *     of the last lookup on that device.  So make one call on a device before
 *     capturing a stream there, and again after a cudaDeviceReset, which ends
 *     the context the address belonged to.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Every call, on every stream, uses the same array, which keeps the last
 *     call's contents (nothing in it needs clearing: each call writes every
 *     entry before reading it).  Calls that overlap on the GPU (on different
 *     streams, or from several host threads) race on it: serialise them.
 * Other arguments, results and errors as ss_scan_chunked.
 */
#define SS_STATIC_WORKSPACE_BYTES (16u << 20)

int ss_scan_chunked_static(const ss_dims* dims, const void* u, const void* delta, const float* A,
                           const void* B, const void* C, const float* D, const void* z,
                           const float* delta_bias, int softplus_flag, float* y, float* last_state,
                           int64_t chunk_len, ss_stream_t stream);

/*
 * Causal depthwise convolution of width 4, optionally followed by SiLU: the
 * short convolution in front of the selective SSM ("What a Mamba block
 * actually contains", multigrid.ai; the block description of "Mamba:
 * Linear-Time Sequence Modeling with Selective State Spaces", azimuth.plus:
 * linear projection -> 1D convolution of kernel size 4 -> SiLU -> SSM).
 *
 *   out[b,d,t] = silu(bias[d] + sum_{k=0..3} weight[d,k] * x[b,d,t-3+k])   (x = 0 before t = 0)
 *
 * weight[d,3] weighs the current step.  Its output is the scan's input u.
 *   dims         batch, dim, seqlen and in_dtype (dstate is ignored; flags must be 0)
 *   x, out       (batch, dim, seqlen) of in_dtype (bf16 output is rounded to nearest even)
 *   weight       (dim, 4) fp32, 16-byte aligned;  bias (dim) fp32 or NULL
 *   silu_flag    nonzero: apply SiLU;  zero: the plain convolution
 * out must not overlap x.  Errors as ss_scan_fwd.  One kernel on `stream`.
 */
int ss_causal_conv1d(const ss_dims* dims, const void* x, const float* weight, const float* bias, int silu_flag,
                     void* out, ss_stream_t stream);

/*
 * Backward pass: the gradients of
 *
 *     Loss = sum_{b,d,t} dy[b,d,t] y[b,d,t] + sum_{b,d,n} dlast_state[b,d,n] last_state[b,d,n]
 *
 * where (y, last_state) is the forward scan of ss_scan_fwd_h0 on the same
 * inputs, with the input weight dims->flags selects (Euler, or SS_FLAG_ZOH).  The forward pass keeps
 * no states: this call recomputes them ("Recomputation" in "Mamba: Linear-Time
 * Sequence Modeling with Selective State Spaces", azimuth.plus: recompute the
 * intermediate states in the backward pass instead of storing them; likewise
 * "Fixed state instead of a growing cache", deepnoodle.ai).
 *
 * Inputs are those of ss_scan_fwd_h0 (h0 nullable), plus
 *   dy           (batch, dim, seqlen) fp32, the gradient of y
 *   dlast_state  (batch, dim, dstate) fp32 or NULL (zero), the gradient of last_state
 * Outputs, all fp32, caller-owned:
 *   du, ddelta   (batch, dim, seqlen)              required
 *   dz           (batch, dim, seqlen) or NULL      only when z is given (SS_EINVAL otherwise)
 *   dA           (dim, dstate)                     required
 *   dB, dC       (batch, dstate, seqlen)           required
 *   dD, ddelta_bias  (dim) or NULL                 the gradient at the given D / delta_bias
 *                                                  (at 0 when those are NULL)
 *   dh0          (batch, dim, dstate) or NULL      the gradient at the given h0 (at 0 when NULL)
 * ddelta is the gradient of the raw delta (before the bias and the softplus).
 * dA, dB, dC, dD and ddelta_bias are sums over many channels and steps; the
 * call zeroes them (cudaMemsetAsync on `stream`) and accumulates with atomic
 * adds, so their last bits may differ from run to run.
 *
 * Workspace: ss_scan_bwd_workspace_bytes(dims) bytes, 256-byte aligned, owned by
 * the caller (for batch 1, dim 5120, N 16, L 65536: 692 MB).  Errors as
 * ss_scan_chunked; SS_EALIGN if an fp32 array is not 4-byte aligned.
 * Four kernels and up to five memsets on `stream`, asynchronous.
 */
size_t ss_scan_bwd_workspace_bytes(const ss_dims* dims);

int ss_scan_bwd(const ss_dims* dims, const float* h0, const void* u, const void* delta, const float* A,
                const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                int softplus_flag, const float* dy, const float* dlast_state, float* du, float* ddelta,
                float* dA, float* dB, float* dC, float* dD, float* dz, float* ddelta_bias, float* dh0,
                void* workspace, size_t workspace_bytes, ss_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* ss_status_string(int status);

/* The CUDA error code (cudaError_t value) behind the last SS_ECUDA returned on
 * this host thread, or 0. */
int ss_last_cuda_error(void);

/*
 * The status word of the current device.  Kernels that wait on their own
 * asynchronous bulk copies bound every wait; one that gives up records it in
 * this word, skips the rest of its work and returns (its outputs are then not
 * valid) instead of hanging the device.  In the debug build (below), a failed
 * index check is recorded there too.  Returns SS_OK when nothing has been
 * recorded since the word was last cleared, SS_EBOUNDS when an index check
 * failed, SS_ETIMEOUT when a wait gave up, SS_ECUDA if the device could not be
 * queried.  Synchronous: it first waits for all work on the current device
 * (cudaDeviceSynchronize).  clear != 0 resets the word.
 */
int ss_device_status(int clear);

/*
 * The debug build.  Compiled with SS_DEBUG_BOUNDS (python -m
 * selective_state_space_117_b300.build --debug-bounds, which writes
 * libssscan_debug.so beside libssscan.so), every kernel checks the index
 * ranges it derives (rows of the inputs and outputs, the batch row of B and C,
 * A rows, state rows, workspace entries, the channel order) against the sizes
 * in ss_dims before using them.  A range outside its array is recorded in the
 * device status word (ss_device_status then returns SS_EBOUNDS) and the
 * accesses it guards are skipped: the kernel never traps and never touches
 * memory outside the arrays the dims describe.  The checks cannot see the
 * caller's allocation sizes, only the dims.  In the normal build they compile
 * away.  ss_debug_bounds_build returns 1 in the debug build, 0 otherwise.
 *
 * ss_selftest_bounds launches one check of a span known to lie outside its
 * array (nothing is accessed): in the debug build it records SS_EBOUNDS, in
 * the normal build nothing.  Asynchronous on `stream`; SS_ECUDA if the launch
 * failed.
 */
int ss_debug_bounds_build(void);
int ss_selftest_bounds(ss_stream_t stream);

/*
 * Diagnostic of the failure path above: launches one thread that waits, with
 * the library's bounded mbarrier wait, on a barrier that nothing ever arrives
 * on.  After the wait's limit (one second on the global timer) it gives up, records
 * SS_ETIMEOUT in the device status word and returns; the device stays usable.
 * Asynchronous on `stream`; read the result with ss_device_status.  Returns
 * SS_ECUDA if the launch failed.  Nothing else is touched.
 */
int ss_selftest_wait_timeout(ss_stream_t stream);

/*
 * Measurement of the exponential throughput that bounds the scan: every decay
 * exp(dt * A) is one ex2.approx.ftz.f32 (MUFU.EX2) after A is scaled by log2(e),
 * so the roofline's exponential term divides by this instruction's rate.  The
 * pages state the method's exponential count, not the hardware's rate, so this
 * call has no counterpart there; it measures the denominator on the GPU that
 * runs the scan.
 *
 * Launches one kernel of `blocks` blocks on `stream`.  Each thread runs several
 * independent chains of `iters` links x <- ex2(x) * (-1/2) (one MUFU.EX2 and one
 * multiply per link), enough exponentials in flight that the MUFU pipe, not
 * latency, bounds the loop.  *ex2_count (host pointer) receives the number of
 * exponentials the launch computes; time the launch with events on `stream`
 * and divide.  `sink` is a device float array of `blocks` entries that the
 * kernel never actually writes (it keeps the chains live).  Use at least a few
 * blocks per SM (for example 8 x the SM count) so that every SM is busy.
 * Returns SS_EINVAL for blocks < 1, iters < 1 or a NULL pointer, SS_ECUDA if
 * the launch failed.  Asynchronous.
 */
int ss_measure_ex2(int64_t blocks, int iters, float* sink, uint64_t* ex2_count, ss_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SS_SCAN_H */
