/*
 * ss_selective_scan.h -- C ABI of the GB300 (sm_103a) selective-scan forward.
 *
 * The operation is the forward pass of the Mamba selective scan, the
 * input-dependent diagonal linear recurrence defined by
 *   - "ТЕХНИЧЕСКОЕ ЗАДАНИЕ: Реализовать selective scan (Mamba)", Этап 1,
 *     steps 3-4 (discretisation A_bar = exp(delta*A), B_bar = delta*B,
 *     delta = softplus(.), read-out C*state + D*u, silu(z) gate);
 *   - "Mamba CUDA 实现解析" (mamba-code-explained), eq (4)-(7): channels are
 *     independent, A is a length-N vector per channel, and every state
 *     element follows v_k = a_k v_{k-1} + b_k u_k;
 *   - the same page, eq (10)-(12): the recurrence is a prefix scan under the
 *     associative operator (a1, v1) (+) (a2, c2) = (a2 a1, a2 v1 + c2), which
 *     is how the library evaluates it in parallel over time.
 *
 * For every batch b, channel d, state n and step t (state zero at t = 0):
 *   dt = delta[b,d,t] + delta_bias[d];  if (delta_softplus) dt = log(1 + e^dt)
 *   h[n] = exp(dt * A[d,n]) * h[n] + dt * B[b,n,t] * u[b,d,t]
 *   y[b,d,t] = (sum_n C[b,n,t] * h[n] + D[d] * u[b,d,t]) * silu(z[b,d,t])
 *   last_state[b,d,n] = h[n] after the last step
 * where the silu factor is 1 when z is NULL, D NULL means D = 0 and
 * delta_bias NULL means a zero bias.
 *
 * Threading and lifetime: the library keeps no pointer after a call returns
 * and holds no global state besides a per-device error word (see
 * ss_selective_scan_check).  Calls on different streams may run concurrently.
 *
 * Devices: a process drives one GPU with this library.  The forward kernels
 * for 8 or 16 states and the backward's 96-row kernels use more than 48 KB of
 * dynamic shared memory, and the library raises their limit once per process,
 * on the device current at its first call; a call that takes one of them on
 * another device of the same process fails with SS_ERR_CUDA (nothing is
 * launched, nothing written).  Run one process per GPU (as torchrun does).
 * The Mamba-2 forward raises its limit per device.
 */
#ifndef SS_SELECTIVE_SCAN_H_
#define SS_SELECTIVE_SCAN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(SS_BUILDING_LIBRARY)
#define SS_API __attribute__((visibility("default")))
#else
#define SS_API
#endif

/* Element type of u, delta, B, C, z and y.  A, D, delta_bias, last_state and
 * the internal state are always float32. */
typedef enum {
  SS_F32 = 0,  /* IEEE float32 */
  SS_BF16 = 1  /* bfloat16; y is rounded to nearest even */
} ss_dtype_t;

typedef enum {
  SS_OK = 0,
  SS_ERR_INVALID_ARGUMENT = 1, /* null required pointer, size <= 0, overlap of
                                  an output with an input, misaligned pointer */
  SS_ERR_UNSUPPORTED = 2,      /* unknown dtype, dstate outside 1..256, or a
                                  size that overflows 64-bit indexing */
  SS_ERR_CUDA = 3,             /* a CUDA runtime call or a launch failed */
  SS_ERR_TIMEOUT = 4,          /* a device-side wait gave up (reported by
                                  ss_selective_scan_check only) */
  SS_ERR_SCRATCH_LIMIT = 5     /* ss_selective_scan_fwd_noalloc: the problem needs
                                  more scratch than its fixed buffer holds */
} ss_status_t;

/*
 * ss_selective_scan_fwd -- enqueue one selective-scan forward on `stream`.
 *
 * Arguments (all pointers are DEVICE pointers owned by the caller; all
 * arrays are dense, row-major, with the last index contiguous):
 *   u          [batch, dim, seqlen]      dtype      input sequence
 *   delta      [batch, dim, seqlen]      dtype      raw step size (before bias/softplus)
 *   A          [dim, dstate]             float32    diagonal state matrix (normally < 0)
 *   B          [batch, dstate, seqlen]   dtype      input projection, shared by all channels
 *   C          [batch, dstate, seqlen]   dtype      output projection, shared by all channels
 *   D          [dim]                     float32    skip weight, or NULL (D = 0)
 *   z          [batch, dim, seqlen]      dtype      gate input, or NULL (no gate)
 *   delta_bias [dim]                     float32    step-size bias, or NULL (0)
 *   delta_softplus                       nonzero: dt = softplus(delta + bias)
 *                                        zero:    dt = delta + bias
 *   y          [batch, dim, seqlen]      dtype      output (written, never read)
 *   last_state [batch, dim, dstate]      float32    final state, or NULL (not written)
 *   batch, dim, dstate, seqlen           sizes; each must be >= 1
 *   dtype                                SS_F32 or SS_BF16
 *   stream                               a cudaStream_t (NULL = legacy default stream)
 *
 * Alignment: every pointer must be aligned to its element size (4 bytes for
 * float32 arrays, 2 bytes for bf16 arrays).  Rows whose start is also
 * 16-byte aligned (seqlen a multiple of 4 for float32, of 8 for bf16, and
 * aligned buffers) take the vectorised path.  Other calls of at least 2^16
 * rows x steps are run on the vectorised path through padded copies of the
 * rows in stream-ordered scratch, whose extra steps leave the state unchanged
 * (dt = 0 there), when that padding is exact: with the softplus, or with
 * float32 I/O, or without a delta bias; the remaining calls take a scalar
 * path.
 *
 * Behaviour: arguments are validated on the host first; on any error the
 * function returns that status, launches nothing and writes nothing.  On
 * success the work is enqueued on `stream` and the call returns without
 * synchronising; y and last_state are complete when the stream reaches that
 * point.  Long sequences use stream-ordered scratch memory
 * (cudaMallocAsync/cudaFreeAsync on `stream`) for the carries between
 * sequence chunks.  A device-side wait that gives up sets a per-device error
 * word that ss_selective_scan_check reports; no call traps.
 *
 * Limits: dstate in 1..256 (tuned for 16); seqlen and batch*dim*seqlen are
 * limited only by 64-bit indexing.  y must not overlap any input.
 */
SS_API ss_status_t ss_selective_scan_fwd(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream);

/*
 * ss_selective_scan_fwd_h0 -- the forward of ss_selective_scan_fwd started
 * from a given state instead of zero: the recurrence of
 * "从顺序到并行用PyTorch实现Blelloch算法加速Mamba状态空间模型" section 1 (the
 * sequential form suited to inference) run over a new segment of a sequence
 * whose earlier part ended in state h0.  Chaining calls with h0 = the previous
 * call's last_state gives the same y and last_state as one call over the
 * concatenated sequence (within the tolerances of the fp32 arithmetic).
 *
 * Arguments: those of ss_selective_scan_fwd, plus
 *   h0         [batch, dim, dstate]      float32    state before step 0, or NULL (zero)
 *
 * last_state may be h0 itself (the state updated in place); any other
 * overlap of an output with an input is SS_ERR_INVALID_ARGUMENT.  Validation,
 * asynchrony, scratch, errors and limits are those of ss_selective_scan_fwd.
 */
SS_API ss_status_t ss_selective_scan_fwd_h0(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const float* h0, void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream);

/*
 * ss_selective_scan_fwd_host -- the forward of ss_selective_scan_fwd_h0 on
 * arrays in HOST memory: every array argument (u, delta, A, B, C, D, z,
 * delta_bias, h0, y, last_state) is a host pointer, with the layouts,
 * dtypes, NULL options and overlap rules of ss_selective_scan_fwd_h0.
 * Page-locked (pinned) host memory lets the copies overlap the scan; pageable
 * memory works, with staged copies.
 *
 * The work goes in pieces, two in flight: the inputs of piece k+1 are copied
 * in on a stream of the call's own while piece k is scanned on `stream` and
 * the outputs of piece k-1 are copied out on a third stream.  With batch > 1
 * a piece is a slice of the batch (up to 8 slices; contiguous copies; each
 * slice an independent scan, so the results are those of
 * ss_selective_scan_fwd_h0 on that slice); a single sequence goes in
 * segments of about 4096 steps (up to 8; strided 2-D copies), each scanned
 * from the state the previous one left, which equals one call over the whole
 * sequence within the fp32 arithmetic's tolerance (chaining through the
 * state, as ss_selective_scan_fwd_h0 documents).  Device buffers for two
 * pieces are allocated and freed on `stream` (stream-ordered).
 *
 * Behaviour: validated on the host (errors launch nothing and write
 * nothing).  The call is synchronous: it returns once y and last_state are
 * in host memory (SS_OK), or with the first error.
 */
SS_API ss_status_t ss_selective_scan_fwd_host(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const float* h0, void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream);

/*
 * ss_selective_state_update -- one decode step (one token) of the selective
 * scan for every (batch, channel), with the state updated in place: the
 * token-by-token recurrent form that "从顺序到并行用PyTorch实现Blelloch算法加速Mamba
 * 状态空间模型" section 1 names as the one for inference, with the step of
 * "Mamba CUDA 实现解析" eq (4)-(7):
 *   dt   = softplus(dt_raw + dt_bias)      (or dt_raw + dt_bias)
 *   h[n] = exp(dt * A[d,n]) * h[n] + dt * B[b,n] * x
 *   y    = (sum_n C[b,n] * h[n] + D[d] * x) * silu(z)
 * It equals ss_selective_scan_fwd_h0 with seqlen = 1, h0 = last_state = state.
 *
 * Arguments (DEVICE pointers owned by the caller, dense, row-major):
 *   state      [batch, dim, dstate]      float32    state, read and overwritten
 *   x          [batch, dim]              dtype      token input (u of the scan)
 *   dt         [batch, dim]              dtype      raw step size
 *   A          [dim, dstate]             float32
 *   B, C       [batch, dstate]           dtype      the token's projections
 *   D          [dim]                     float32    or NULL (0)
 *   z          [batch, dim]              dtype      gate input, or NULL (no gate)
 *   dt_bias    [dim]                     float32    or NULL (0)
 *   dt_softplus                          nonzero: softplus on dt_raw + dt_bias
 *   y          [batch, dim]              dtype      output (written, never read)
 *   batch, dim, dstate                   sizes >= 1; dstate <= 256
 *   dtype, stream                        as for ss_selective_scan_fwd
 *
 * Behaviour: validated on the host (errors launch nothing and write
 * nothing); one kernel is enqueued on `stream` and the call returns without
 * synchronising.  It allocates no memory and has no device-side wait.  state
 * and y must not overlap each other or any input.
 */
SS_API ss_status_t ss_selective_state_update(
    float* state, const void* x, const void* dt, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* dt_bias, int dt_softplus, void* y,
    int64_t batch, int64_t dim, int64_t dstate, ss_dtype_t dtype, void* stream);

/*
 * ss_selective_scan_bwd -- the backward pass of ss_selective_scan_fwd: the
 * gradients of every input for a loss whose gradient is dy on y (and
 * dlast_state on last_state), which "ТЕХНИЧЕСКОЕ ЗАДАНИЕ: Реализовать
 * selective scan (Mamba)" asks for and to verify with gradcheck (Этап 3
 * step 4; section 5).  It is the chain rule through the forward's definition
 * run backwards in time: g_t = C_t dy'_t + a_{t+1} g_{t+1} over the states,
 * with the forward states recomputed from checkpoints.
 *
 * Inputs: those of ss_selective_scan_fwd (zero initial state; see
 * ss_selective_scan_bwd_h0 for a given one), plus
 *   dy          [batch, dim, seqlen]     dtype      gradient of y
 *   dlast_state [batch, dim, dstate]     float32    gradient of last_state, or NULL (0)
 * Outputs (written, never read):
 *   du, ddelta  [batch, dim, seqlen]     dtype
 *   dA          [dim, dstate]            float32
 *   dB, dC      [batch, dstate, seqlen]  float32    summed over the channels
 *   dD          [dim]                    float32    or NULL (not computed; ignored if D is NULL)
 *   dz          [batch, dim, seqlen]     dtype      required when z is given, else ignored
 *   dbias       [dim]                    float32    or NULL (ignored if delta_bias is NULL)
 *
 * Limits: dstate in 1..256 (else SS_ERR_UNSUPPORTED), run in groups of 16
 * states, one main kernel per group.  Sums over channels, time, batch and
 * state groups are evaluated in a fixed order: results are bitwise
 * reproducible.
 * Behaviour: validated on the host (errors launch nothing and write nothing);
 * the group kernels and two reductions are enqueued on `stream` with
 * stream-ordered scratch (cudaMallocAsync/cudaFreeAsync, about 8 bytes per
 * (row, step) for the state checkpoints, 128 bytes per 64-channel tile, step
 * and state group, and with several groups 12 bytes per (row, step) for the
 * row sums carried between them); no synchronisation and no device-side wait.
 * No output may overlap an input or another output.
 */
SS_API ss_status_t ss_selective_scan_bwd(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const void* dy, const float* dlast_state, void* du, void* ddelta, float* dA, float* dB,
    float* dC, float* dD, void* dz, float* dbias,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, ss_dtype_t dtype, void* stream);

/*
 * ss_selective_scan_bwd_h0 -- the backward of ss_selective_scan_fwd_h0: the
 * same gradients as ss_selective_scan_bwd for the forward started from the
 * state h0, and the gradient of h0 itself (the chain rule carried one step
 * past t = 0: dh0[n] = exp(dt_0 A[d,n]) g_0[n]; h0 also enters dA through the
 * first step's decay).
 *
 * Arguments: those of ss_selective_scan_bwd, plus
 *   h0          [batch, dim, dstate]     float32    the state before step 0, or NULL (0)
 *   dh0         [batch, dim, dstate]     float32    its gradient (written), or NULL
 * dh0 is written only when h0 is given.  Errors, limits, scratch and
 * behaviour are those of ss_selective_scan_bwd; h0 counts as an input and
 * dh0 as an output for the overlap rules.
 */
SS_API ss_status_t ss_selective_scan_bwd_h0(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus, const float* h0,
    const void* dy, const float* dlast_state, void* du, void* ddelta, float* dA, float* dB,
    float* dC, float* dD, void* dz, float* dbias, float* dh0,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen, ss_dtype_t dtype, void* stream);

/*
 * ss_mamba2_fwd -- the Mamba-2 forward (one scalar decay per head), the
 * recurrence of the Mamba-2 cuTile news page ("Прорыв в оптимизации
 * SSM-моделей", section "Технические детали оптимизации"), evaluated in
 * chunks with the page's jump formula on the tensor cores (tcgen05) for its
 * common shape, and as a selective scan per head group otherwise:
 *   dt_t = softplus(dt[b,t,h] + dt_bias[h])   (or dt + dt_bias when dt_softplus == 0)
 *   h_t  = exp(A[h] dt_t) h_{t-1} + dt_t x_t B_t^T       state [headdim, dstate], zero at t = 0
 *   y_t  = h_t C_t + D[h] x_t
 * for every batch b and head h; B_t and C_t are the rows of the head's group
 * g = h / (nheads / ngroups).
 *
 * Arguments (device pointers, dense row-major):
 *   x           [batch, seqlen, nheads, headdim]   dtype
 *   dt          [batch, seqlen, nheads]            dtype
 *   A           [nheads]                           float32
 *   B, C        [batch, seqlen, ngroups, dstate]   dtype
 *   D, dt_bias  [nheads]                           float32, or NULL (0)
 *   y           [batch, seqlen, nheads, headdim]   dtype (written)
 *   final_state [batch, nheads, headdim, dstate]   float32 (written), or NULL
 * Limits: dstate <= 256 (else SS_ERR_UNSUPPORTED); nheads a multiple of
 * ngroups and every pointer aligned to its element (else
 * SS_ERR_INVALID_ARGUMENT).
 * Two paths.  bf16 with headdim 64, 128 states and 16-byte aligned x, B, C
 * and y runs on the tensor cores: one kernel, one CTA per (batch, head), no
 * scratch; the products run on bf16 operands with fp32 accumulation, and the
 * decayed C.B weights, the decayed inputs and the state carried into a chunk
 * are rounded to bf16 where they enter a product (the state itself stays
 * fp32); its waits on the tensor cores are bounded (SS_ERR_TIMEOUT from
 * ss_selective_scan_check).  Every other call (fp32 or bf16, any head dim, up
 * to 256 states) runs each head group as one selective scan over the group's
 * heads' channels: channel-major copies of x, dt, B and C in scratch
 * allocated and freed on `stream` (stream-ordered allocation), the scan of
 * ss_selective_scan_fwd with the arithmetic of that call (fp32, bf16 only
 * where y is stored), and y copied back; several kernels.
 * Behaviour: validated on the host (errors launch nothing and write
 * nothing); no synchronisation.  y and final_state must not overlap any input
 * or each other.  The state starts at zero (see ss_mamba2_fwd_h0).
 */
SS_API ss_status_t ss_mamba2_fwd(
    const void* x, const void* dt, const float* A, const void* B, const void* C,
    const float* D, const float* dt_bias, int dt_softplus, void* y, float* final_state,
    int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
    int64_t dstate, ss_dtype_t dtype, void* stream);

/*
 * ss_mamba2_fwd_h0 -- ss_mamba2_fwd started from a given state: the same
 * recurrence run over a segment of a sequence whose earlier part left the
 * state initial_state (h_{-1}), as for the sequential form of
 * "从顺序到并行用PyTorch实现Blelloch算法加速Mamba状态空间模型" section 1.  The
 * given state enters chunk 0 the way a chunk's incoming state enters every
 * later chunk (the page's jump formula): y_t gains C_t exp(cum_t) h_{-1}, the
 * state carries exp(cum_end) h_{-1} forward; its bf16 copy feeds the tensor
 * cores like every carried state.
 *
 * Arguments: those of ss_mamba2_fwd, plus
 *   initial_state [batch, nheads, headdim, dstate]  float32  or NULL (zero)
 * final_state may be initial_state itself (the state updated in place); any
 * other overlap of an output with an input is SS_ERR_INVALID_ARGUMENT.
 * Limits, validation and behaviour are those of ss_mamba2_fwd.
 */
SS_API ss_status_t ss_mamba2_fwd_h0(
    const void* x, const void* dt, const float* A, const void* B, const void* C,
    const float* D, const float* dt_bias, int dt_softplus, const float* initial_state, void* y,
    float* final_state, int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
    int64_t ngroups, int64_t dstate, ss_dtype_t dtype, void* stream);

/*
 * ss_selective_scan_fwd_pc -- the forward with B and C given per channel:
 * the layout of "ТЕХНИЧЕСКОЕ ЗАДАНИЕ: Реализовать selective scan (Mamba)",
 * Этап 2 step 3 (the base kernel signature indexes B and C by batch, channel
 * and step), taken to dstate states.
 *
 * Arguments: those of ss_selective_scan_fwd, except
 *   B, C       [batch, dim, dstate, seqlen]   dtype   one row per channel
 *
 * Limits: dstate <= 256 (else SS_ERR_UNSUPPORTED); zero initial state (see
 * ss_selective_scan_fwd_pc_h0).
 * Behaviour: validated on the host (errors launch nothing and write
 * nothing); one kernel is enqueued on `stream`; no scratch, no device-side
 * wait, no synchronisation.  y and last_state must not overlap any input or
 * each other.
 */
SS_API ss_status_t ss_selective_scan_fwd_pc(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream);

/*
 * ss_selective_scan_fwd_pc_h0 -- ss_selective_scan_fwd_pc started from a given
 * state: the per-channel layout run over a new segment of a sequence whose
 * earlier part ended in state h0 (the sequential form of
 * "从顺序到并行用PyTorch实现Blelloch算法加速Mamba状态空间模型" section 1).
 *
 * Arguments: those of ss_selective_scan_fwd_pc, plus
 *   h0         [batch, dim, dstate]      float32    state before step 0, or NULL (zero)
 *
 * last_state may be h0 itself (the state updated in place); any other overlap
 * of an output with an input is SS_ERR_INVALID_ARGUMENT.  Limits, validation
 * and behaviour are those of ss_selective_scan_fwd_pc.
 */
SS_API ss_status_t ss_selective_scan_fwd_pc_h0(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    const float* h0, void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
SS_API const char* ss_status_string(ss_status_t status);

/*
 * ss_selective_scan_check -- synchronise `stream`, then report and clear the
 * device-side error word of the current device.  Returns SS_OK when every
 * call enqueued so far completed normally, SS_ERR_TIMEOUT when a bounded
 * device-side wait gave up, and SS_ERR_CUDA when the stream reports a CUDA
 * error.
 */
SS_API ss_status_t ss_selective_scan_check(void* stream);

/*
 * ss_selective_scan_fwd_noalloc -- the same forward as ss_selective_scan_fwd
 * for callers that cannot allocate device memory during a call: code that
 * runs where cudaMalloc/cudaMallocAsync is not allowed or not wanted, for
 * example under a caching allocator it must not bypass, inside a real-time
 * path that forbids allocator calls, or in a host that owns all device memory
 * up front.  The pages have no counterpart to this entry point; it is a
 * library service.
 *
 * Arguments, layouts, ownership and the result are those of
 * ss_selective_scan_fwd.  Instead of stream-ordered scratch it uses one
 * fixed 16 MiB buffer in the library's own device memory (a file-scope
 * __device__ array, present on every GPU that loads the library until the
 * process exits).  It calls no allocating function: it zeroes the part of the
 * buffer that must start at zero with cudaMemsetAsync on `stream` and
 * launches the scheduled kernel.
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * buffer's device address with cudaGetSymbolAddress; make that first call
 * before any stream capture on that device.  The address belongs to the
 * device's CUDA context: after the context is destroyed and created anew
 * (cudaDeviceReset), the next call looks it up again, so that call too
 * should come before any capture.
 *
 * Limits: the vector path only (every u/delta/z/y/B/C pointer 16-byte aligned
 * and seqlen a multiple of 4 for float32, of 8 for bf16), else
 * SS_ERR_UNSUPPORTED.  The chunk count is ss_selective_scan_fwd's, lowered to
 * the largest count whose carries fit the buffer (each chunk of a row tile
 * of 64 channels keeps 12 bytes per channel and state); a problem that does
 * not fit even unsplit (dstate > 16 needs a float32 row of
 * batch * dim * seqlen partial read-outs) returns SS_ERR_SCRATCH_LIMIT.  Like
 * every entry point of the shipped library it reads no environment variable.
 *
 * Concurrency: every call shares the one buffer per device, so calls whose
 * execution overlaps on the GPU (different streams, or graphs replayed
 * concurrently) race on it and give wrong results; order such calls on one
 * stream or use ss_selective_scan_fwd.
 */
SS_API ss_status_t ss_selective_scan_fwd_noalloc(
    const void* u, const void* delta, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* delta_bias, int delta_softplus,
    void* y, float* last_state,
    int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
    ss_dtype_t dtype, void* stream);

/*
 * ss_selective_scan_plan -- describe, without any CUDA call, how
 * ss_selective_scan_fwd would run a problem of these sizes on a device with
 * `sm_count` SMs.  Long sequences are split into chunks that run in
 * parallel and are joined by the prefix formulation of "Mamba CUDA 实现解析"
 * eq (11)-(12); this reports that split so callers can size scratch and
 * count launches.  `aligned16` states whether every u/delta/z/y/B/C pointer
 * will be 16-byte aligned.  Returns SS_ERR_INVALID_ARGUMENT for sizes <= 0 or
 * a NULL `plan`, SS_ERR_UNSUPPORTED as ss_selective_scan_fwd would; fills
 * `plan` on SS_OK.  (The test build of the library, which the package's
 * tests load, also honours the SS_NCHUNKS and SS_CTAS_PER_SM plan
 * overrides; the shipped library reads no environment variable.)
 */
typedef struct {
  int64_t nchunks;         /* sequence chunks */
  int64_t chunk_len;       /* steps per chunk (the last one may be shorter) */
  int64_t state_groups;    /* groups of at most 16 states */
  int64_t ctas;            /* CTAs of the main kernel */
  int64_t kernel_launches; /* kernels one call enqueues */
  int64_t scratch_bytes;   /* stream-ordered scratch one call allocates */
  int64_t vector_path;     /* 1: 16-byte vector path; 0: scalar path */
} ss_plan_t;

SS_API ss_status_t ss_selective_scan_plan(int64_t batch, int64_t dim, int64_t dstate,
                                          int64_t seqlen, ss_dtype_t dtype, int aligned16,
                                          int sm_count, ss_plan_t* plan);

#ifdef __cplusplus
}
#endif

#endif /* SS_SELECTIVE_SCAN_H_ */
