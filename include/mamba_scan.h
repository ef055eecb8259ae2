/*
 * mamba_scan.h -- C ABI of the B300 (sm_103a) selective state-space scan library
 * (libmambascan.so).
 *
 * What is computed (per batch b, channel d, state n, time l):
 *
 *   dt        = delta[b,d,l] + delta_bias[d]            (bias optional, 0 if NULL)
 *   dt        = softplus(dt)     if flags & MAMBA_FLAG_SOFTPLUS  ("Mamba 论文精读", youngju.dev,
 *                                                          §3.1: Delta_t = softplus(Linear_Delta(x_t)))
 *   dA        = exp(dt * A[d,n])                          (same page §2.2, ZOH: A_bar = exp(Delta A))
 *   dBu       = dt * B[b,n,l] * u[b,d,l]                   (same page §3.3 simplified scan: B_bar = Delta B)
 *   dBu       = (exp(dt*A[d,n]) - 1) / A[d,n] * B[b,n,l] * u[b,d,l]
 *                                   if flags & MAMBA_FLAG_ZOH (same page §2.2, the exact zero-order
 *                                                          hold B_bar = (Delta A)^-1 (exp(Delta A) - I)
 *                                                          Delta B for a diagonal A; dt where dt*A = 0)
 *   h[n]      = dA * h[n] + dBu,  h = 0 before l = 0       (same page §2.2 recurrence; §3.3 starts h at zero)
 *   y[b,d,l]  = sum_n C[b,n,l] * h[n]  (+ D[d] * u[b,d,l]) (§2.2 y_t = C h_t; the D skip term is the
 *                                                          output term of "Mamba的基础知识", weblog-19d,
 *                                                          状态空间模型 section)
 *   y        *= silu(z[b,d,l])          if z != NULL      ("Mamba 论文精读" §3.4 block gate)
 *
 * "mamba->jamba" (blog.csdn.net) §2.3 states the fused-kernel requirement this
 * library meets: only delta, A, B, C (and u, z) are read from HBM, discretisation,
 * scan and the contraction with C happen on chip, and only y (batch, D, L) is
 * written; no (batch, L, D, N) intermediate ever reaches device memory.
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers owned by the caller. The library allocates
 *     nothing and keeps no state between calls (apart from one device error
 *     word, see mamba_check_device_error). Scratch memory, where an entry point
 *     uses any, is a caller workspace (the *_ws entry points and the backward)
 *     or, for mamba_scan_fwd_noalloc, a fixed array the library reserves.
 *   - All tensors are dense, row-major, contiguous:
 *       u, delta, z, y : (batch, dim, seqlen)
 *       B, C           : (batch, dstate, seqlen)   -- one group, shared by all channels
 *       A              : (dim, dstate)             fp32, expected < 0 (not checked)
 *       D, delta_bias  : (dim)                     fp32
 *       state          : (batch, dim, dstate)      fp32
 *     For the state update, u/delta/z/y are (batch, dim) and B/C are (batch, dstate).
 *   - u, delta, z, B, C and y share io_dtype (fp32 or bf16). A, D, delta_bias and
 *     the state are always fp32; the recurrence and all accumulation are fp32.
 *   - dstate must be 8, 16, 32 or 64 for the selective scan (forward,
 *     backward, state update); anything else is MAMBA_ERR_SHAPE.
 *   - `flags` is a bit set of mamba_flag values; 0 and 1 keep the meaning of a
 *     plain softplus switch. An unknown bit, or a bit an entry point does not
 *     support, is MAMBA_ERR_FLAGS.
 *   - Base pointers of u, delta, z, y, B, C, A and state/final_state must be
 *     16-byte aligned; D and delta_bias 4-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and launch on the current CUDA device.
 *   - Every argument check happens on the host before any launch; on an error
 *     nothing is launched and nothing is written.
 */
#ifndef MAMBA_SCAN_H
#define MAMBA_SCAN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MAMBA_F32 = 0,
    MAMBA_BF16 = 1
} mamba_dtype;

typedef enum {
    MAMBA_OK = 0,
    MAMBA_ERR_NULL = -1,            /* a required pointer is NULL */
    MAMBA_ERR_SHAPE = -2,           /* negative size, unsupported dstate, or a size too large */
    MAMBA_ERR_DTYPE = -3,           /* io_dtype is not a mamba_dtype */
    MAMBA_ERR_ALIGN = -4,           /* a base pointer violates the alignment above */
    MAMBA_ERR_CUDA = -5,            /* a CUDA runtime/driver call failed (launch or tensor map) */
    MAMBA_ERR_DEVICE_TIMEOUT = -6,  /* a kernel gave up waiting on its own copies (see below) */
    MAMBA_ERR_WORKSPACE = -7,       /* workspace_bytes < mamba_scan_workspace_size(...) */
    MAMBA_ERR_FLAGS = -8,           /* flags holds an unknown bit, or one this entry point lacks */
    MAMBA_ERR_DEVICE_BOUNDS = -9    /* checked-bounds build only: a kernel computed an index outside
                                       a tensor and skipped that access (see mamba_checked_bounds) */
} mamba_status;

typedef enum {
    MAMBA_FLAG_SOFTPLUS = 1,  /* dt = softplus(delta + bias) instead of delta + bias */
    MAMBA_FLAG_ZOH = 2        /* exact zero-order-hold input gain instead of dt * B (every selective-scan
                                 entry point; not the SSD form) */
} mamba_flag;

/*
 * Selective scan (prefill / training forward).
 *   u, delta, z : (batch, dim, seqlen) io_dtype; z may be NULL (no gate)
 *   A           : (dim, dstate) fp32
 *   B, C        : (batch, dstate, seqlen) io_dtype
 *   D           : (dim) fp32 or NULL (no skip term)
 *   delta_bias  : (dim) fp32 or NULL (zero bias)
 *   flags       : MAMBA_FLAG_SOFTPLUS -> dt = softplus(delta + bias), else dt = delta + bias;
 *                 MAMBA_FLAG_ZOH -> exact zero-order-hold input gain (see the top)
 *   y           : (batch, dim, seqlen) io_dtype, written (bf16 by round-to-nearest-even)
 *   final_state : (batch, dim, dstate) fp32 or NULL; receives h after the last step
 *                 (zeros when seqlen == 0)
 * Any of batch, dim, seqlen may be 0 (nothing to compute; final_state, if given,
 * is zero-filled). When seqlen == 0, u, delta, B, C, z and y may be NULL (an
 * empty tensor's data pointer). y must not alias an input.
 * Allocates nothing and launches one kernel, which reads B and C in their own
 * layout. (A long sequence over few channels runs faster through
 * mamba_scan_fwd_ws with a workspace: see mamba_scan_workspace_size.)
 * Returns MAMBA_OK or a negative mamba_status.
 */
int mamba_scan_fwd(const void* u, const void* delta, const float* A,
                   const void* B, const void* C,
                   const float* D, const void* z,
                   const float* delta_bias, int flags,
                   void* y, float* final_state,
                   int batch, int dim, int seqlen, int dstate,
                   int io_dtype, void* stream);

/*
 * Bytes of device workspace mamba_scan_fwd_ws (and mamba_conv_scan_fwd_ws)
 * can use for these sizes on the current device; 0 when it needs none (the
 * usual case), when there is nothing to compute, an argument is out of range
 * or no device is current.
 * The workspace holds the carries of a sequence split: when batch *
 * ceil(dim / channels per warp) (16 channels a warp for dstate 8 and 16, 8 for
 * 32, 4 for 64) is below four warps per streaming multiprocessor, i.e. a long
 * sequence over few channels, the 16-step chunks are cut into S segments of at
 * least 64 chunks (S about 12 warps per scheduler over the warps of one pass,
 * at most 32): one kernel finds every segment's end state from zero (from
 * initial_state for the first) and the sum of dt over it, and the scan kernel
 * starts each segment from the state these give. The size is
 * (S - 1) * batch * dim * (dstate + 1) * 4 bytes, each part rounded up to 256.
 * The results are the same as in one pass up to the rounding of the state at
 * the segment boundaries.
 */
size_t mamba_scan_workspace_size(int batch, int dim, int seqlen, int dstate, int io_dtype);

/*
 * mamba_scan_fwd with a caller-provided workspace and an optional initial
 * state: same arguments, semantics and checks, plus
 *   initial_state   : (batch, dim, dstate) fp32, 16-byte aligned, or NULL for
 *                     zero: the state before the first step, so that a long
 *                     sequence can be scanned in pieces, each piece starting
 *                     from the previous piece's final_state ("mamba->jamba"
 *                     §2.2: the recurrence carries h from token to token);
 *                     with seqlen == 0, final_state receives it unchanged
 *   chunk_states    : (batch, dim, ceil(seqlen / 16), dstate) fp32, 16-byte
 *                     aligned, or NULL: receives the state before every 16-step
 *                     chunk (the first is initial_state), which mamba_scan_bwd
 *                     can take instead of recomputing it (training)
 *   workspace       : device buffer, 256-byte aligned, owned by the caller, of
 *                     at least mamba_scan_workspace_size(...) bytes, or NULL;
 *                     with NULL (or a size of 0) the scan runs in one pass,
 *                     otherwise split as mamba_scan_workspace_size describes;
 *                     its contents are scratch, needed only until the call's
 *                     kernels on `stream` have finished
 *   workspace_bytes : its size
 * Allocates nothing. Returns MAMBA_ERR_WORKSPACE if a non-NULL buffer is too
 * small, MAMBA_ERR_ALIGN if it is misaligned.
 */
int mamba_scan_fwd_ws(const void* u, const void* delta, const float* A,
                      const void* B, const void* C,
                      const float* D, const void* z,
                      const float* delta_bias, int flags,
                      const float* initial_state,
                      void* y, float* final_state, float* chunk_states,
                      int batch, int dim, int seqlen, int dstate,
                      int io_dtype, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * The scan of u = silu(conv1d(x)): the Mamba block's causal depthwise
 * convolution and SiLU in front of the scan ("Mamba 论文精读" (youngju.dev)
 * §3.4), fused into the scan kernel so that u never reaches device memory:
 *   u[b,d,l] = silu( sum_{k=0}^{3} conv_weight[d,k] * x[b,d,l-3+k] + conv_bias[d] )
 * Arguments as mamba_scan_fwd_ws with u replaced by
 *   x            : (batch, dim, seqlen) io_dtype, the convolution's input
 *   conv_weight  : (dim, conv_width) fp32, 16-byte aligned
 *   conv_bias    : (dim) fp32 or NULL
 *   conv_state   : (batch, dim, conv_width - 1) io_dtype or NULL: x at steps
 *                  -3..-1 (oldest first), for a sequence scanned in pieces;
 *                  NULL means zeros (the padding of a fresh sequence)
 *   conv_width   : must be 4 (MAMBA_ERR_SHAPE otherwise)
 * u is computed and used in fp32 (it is not rounded to the I/O dtype). The
 * workspace is the same as mamba_scan_fwd_ws's (mamba_scan_workspace_size).
 */
int mamba_conv_scan_fwd_ws(const void* x, const float* conv_weight, const float* conv_bias,
                           const void* conv_state, int conv_width,
                           const void* delta, const float* A,
                           const void* B, const void* C,
                           const float* D, const void* z,
                           const float* delta_bias, int flags,
                           const float* initial_state,
                           void* y, float* final_state,
                           int batch, int dim, int seqlen, int dstate,
                           int io_dtype, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Bytes of device workspace mamba_scan_bwd needs for these sizes (0 when there
 * is nothing to compute or an argument is out of range): the packed fp32 B/C
 * rows (batch * roundup(seqlen, 16) * 8 * dstate bytes), one fp32 state per
 * row per 16 steps (batch * dim * roundup(seqlen, 16) / 16 * 4 * dstate bytes)
 * and fp32 sums of dB and dC (batch * roundup(seqlen, 16) * 8 * dstate bytes),
 * each rounded up to 256 bytes.
 */
size_t mamba_scan_bwd_workspace_size(int batch, int dim, int seqlen, int dstate, int io_dtype);

/*
 * Backward of the selective scan (training): the gradients of
 * L = sum(dy * y), y the output of mamba_scan_fwd_ws with the same inputs,
 * with respect to every input. The states are recomputed from the inputs, as
 * "mamba->jamba" (blog.csdn.net) §2.3 describes for the backward pass, keeping
 * one fp32 state per row every 16 steps in the workspace in between.
 * Takes the same dstate values and flags as the forward (with MAMBA_FLAG_ZOH
 * the exact gain is differentiated, d gain / d dt = exp(dt A) and
 * d gain / dA = (dt exp(dt A) - gain) / A, its series near dt A = 0).
 * Inputs: as mamba_scan_fwd_ws (u, delta, A, B, C, D, z, delta_bias, flags,
 * initial_state), plus
 *   chunk_states    : the forward's chunk_states output for these same inputs,
 *                     or NULL: the backward then recomputes them (one more
 *                     sweep over the sequence)
 *   dy              : (batch, dim, seqlen) io_dtype, the gradient reaching y
 * Outputs (device, caller-owned, overwritten; 16-byte aligned except dD and
 * ddelta_bias, 4-byte):
 *   du, ddelta      : (batch, dim, seqlen) io_dtype
 *   dz              : (batch, dim, seqlen) io_dtype; required iff z is given
 *   dA              : (dim, dstate) fp32, summed over the batch
 *   dB, dC          : (batch, dstate, seqlen) io_dtype, summed over the channels
 *   dD              : (dim) fp32 or NULL (NULL required when D is NULL)
 *   ddelta_bias     : (dim) fp32 or NULL (NULL required when delta_bias is NULL)
 *   dinitial_state  : (batch, dim, dstate) fp32 or NULL; the gradient reaching
 *                     the state before the first step (zeros when seqlen == 0)
 * workspace/workspace_bytes as for mamba_scan_fwd_ws, sized by
 * mamba_scan_bwd_workspace_size. dA, dB, dC, dD and ddelta_bias are sums of
 * fp32 atomic additions, so their last bits may vary from run to run.
 * Returns MAMBA_OK or a negative mamba_status.
 */
int mamba_scan_bwd(const void* u, const void* delta, const float* A,
                   const void* B, const void* C,
                   const float* D, const void* z,
                   const float* delta_bias, int flags,
                   const float* initial_state, const float* chunk_states,
                   const void* dy,
                   void* du, void* ddelta, float* dA, void* dB, void* dC,
                   float* dD, void* dz, float* ddelta_bias, float* dinitial_state,
                   int batch, int dim, int seqlen, int dstate, int io_dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * mamba_scan_fwd without any allocation and without a caller workspace.
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory at call time (serving loops that reserve all
 * memory at start-up, plugins inside a framework that owns every device
 * allocation, programs with no allocator to provide a workspace).
 *
 * Same arguments, semantics and checks as mamba_scan_fwd, but a long sequence
 * over few channels is split as by mamba_scan_fwd_ws with a workspace (see
 * mamba_scan_workspace_size). The split's carries live in a fixed 1 MiB array
 * in device memory that the library reserves on every GPU that loads it, until
 * the process exits.
 *   - When the carries of the split mamba_scan_fwd_ws would take exceed 1 MiB,
 *     this call cuts fewer segments, the most whose carries fit (on a 148-SM
 *     GPU: 4 segments of 1 x 5120 channels at dstate 16, against 22), or none;
 *     it never needs more memory, so no size is rejected for lack of it.
 *   - The first call on a device that splits looks up the array's device
 *     address (cudaGetSymbolAddress) with that device current and caches it:
 *     make that first call before any stream capture is under way.
 *   - `stream` must belong to the current device (MAMBA_ERR_CUDA otherwise):
 *     the array's address is per device.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, or other host threads) race on it and must be serialised by the
 *     caller. Nothing needs clearing between calls: the first kernel of a
 *     split writes every carry the second reads.
 * Returns MAMBA_OK or a negative mamba_status (MAMBA_ERR_CUDA if the address
 * lookup fails).
 */
int mamba_scan_fwd_noalloc(const void* u, const void* delta, const float* A,
                           const void* B, const void* C,
                           const float* D, const void* z,
                           const float* delta_bias, int flags,
                           void* y, float* final_state,
                           int batch, int dim, int seqlen, int dstate,
                           int io_dtype, void* stream);

/*
 * Single-token recurrent state update (decode): one step of the recurrence above
 * applied in place to `state` ("mamba->jamba" §2.2: constant-time recurrent
 * inference; "Mamba 论文精读" §6: O(1) work and a fixed-size state per token).
 *   state       : (batch, dim, dstate) fp32, read and overwritten
 *   u, delta, z : (batch, dim) io_dtype; z may be NULL
 *   A           : (dim, dstate) fp32
 *   B, C        : (batch, dstate) io_dtype
 *   D           : (dim) fp32 or NULL;  delta_bias : (dim) fp32 or NULL
 *   flags       : as for mamba_scan_fwd
 *   y           : (batch, dim) io_dtype, written
 * Returns MAMBA_OK or a negative mamba_status.
 */
int mamba_state_update(float* state, const void* u, const void* delta, const float* A,
                       const void* B, const void* C,
                       const float* D, const void* z,
                       const float* delta_bias, int flags,
                       void* y, int batch, int dim, int dstate,
                       int io_dtype, void* stream);

/*
 * State-space dual (SSD) layer, the Mamba-2 form ("Mamba 论文精读" (youngju.dev)
 * §4.1: the recurrence h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t is dual to
 * the masked product Y = (T o M) X with M semiseparable; §5.2: multi-head,
 * headdim 64, larger states). Per batch row b and head h the state S is a
 * (headdim x dstate) fp32 matrix and the decay one scalar per step:
 *
 *   dt   = delta[b,h,l] + delta_bias[h]; softplus(dt) if flags & MAMBA_FLAG_SOFTPLUS
 *   S    = exp(dt * A[h]) * S + dt * x[b,h*64+p,l] * B[b,:,l]      (row p of S)
 *   y[b,h*64+p,l] = S[p,:] . C[b,:,l] + D[h] * x[b,h*64+p,l]
 *
 * computed chunk by chunk (64 steps) with the contractions on the tensor cores.
 *   x, y          : (batch, nheads * headdim, seqlen) bf16, channel = h * 64 + p
 *   delta         : (batch, nheads, seqlen) bf16
 *   A             : (nheads) fp32;  D, delta_bias : (nheads) fp32 or NULL
 *   B, C          : (batch, dstate, seqlen) bf16, one group shared by the heads
 *   initial_state : (batch, nheads, headdim, dstate) fp32 or NULL (zero)
 *   final_state   : the same shape, or NULL; receives S after the last step
 *   workspace     : as for mamba_scan_fwd_ws, sized by mamba_ssd_workspace_size
 *                   (0 bytes unless seqlen is not a multiple of 8: then row
 *                   copies of x, B and C at a 16-byte pitch)
 * Supported: io_dtype MAMBA_BF16 (MAMBA_ERR_DTYPE otherwise), headdim 64 and
 * dstate 64, 128 or 256 (MAMBA_ERR_SHAPE otherwise), flags MAMBA_FLAG_SOFTPLUS only
 * (MAMBA_ERR_FLAGS otherwise). Alignment: x, y, B, C and the states 16 bytes,
 * delta 2, A, D, delta_bias 4. State and accumulation are fp32; y is rounded to
 * bf16 once. Returns MAMBA_OK or a negative mamba_status.
 */
size_t mamba_ssd_workspace_size(int batch, int nheads, int headdim, int seqlen, int dstate, int io_dtype);

int mamba_ssd_fwd(const void* x, const void* delta, const float* A,
                  const void* B, const void* C,
                  const float* D, const float* delta_bias, int flags,
                  const float* initial_state, void* y, float* final_state,
                  int batch, int nheads, int headdim, int seqlen, int dstate,
                  int io_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Single-token step of the SSD form (decode), in place on the state: for each
 * batch row b, head h and channel p of the head,
 *   dt = delta[b,h] + delta_bias[h];  softplus(dt) if flags & MAMBA_FLAG_SOFTPLUS
 *   S[b,h,p,:] = exp(dt * A[h]) * S[b,h,p,:] + dt * x[b,h*64+p] * B[b,:]
 *   y[b,h*64+p] = S[b,h,p,:] . C[b,:] + D[h] * x[b,h*64+p]
 * (one step of mamba_ssd_fwd, so a sequence can be continued token by token
 * from its final_state).
 *   state   : (batch, nheads, headdim, dstate) fp32, read and overwritten, 16-byte aligned
 *   x, y    : (batch, nheads * headdim) io_dtype;  delta : (batch, nheads) io_dtype
 *   B, C    : (batch, dstate) io_dtype, 16-byte aligned
 *   A       : (nheads) fp32;  D, delta_bias : (nheads) fp32 or NULL
 * Supported: io_dtype MAMBA_F32 or MAMBA_BF16, headdim 64, dstate 64, 128 or 256,
 * flags MAMBA_FLAG_SOFTPLUS only. Returns MAMBA_OK or a negative mamba_status.
 */
int mamba_ssd_update(float* state, const void* x, const void* delta, const float* A,
                     const void* B, const void* C, const float* D, const float* delta_bias,
                     int flags, void* y, int batch, int nheads, int headdim, int dstate,
                     int io_dtype, void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device error word.
 * Kernels that wait on their own asynchronous copies give up after a bounded
 * number of polls (far beyond any normal copy time), set this word and return
 * early instead of hanging. In the checked-bounds build a kernel that computes
 * an index outside a tensor skips that access and sets the word too. The first
 * error recorded since the last check wins. Returns MAMBA_OK,
 * MAMBA_ERR_DEVICE_TIMEOUT, MAMBA_ERR_DEVICE_BOUNDS, or MAMBA_ERR_CUDA if the
 * synchronisation itself failed.
 */
int mamba_check_device_error(void* stream);

/*
 * 1 if this build of the library is the checked-bounds one, else 0. That
 * build (compiled with -DMAMBA_DEBUG_BOUNDS; the Python package builds it as
 * libmambascan_checked.so) exports the same calls with the same results, but
 * every global load and store its kernels make with ordinary instructions is
 * first checked against the extent of the tensor it belongs to, computed from
 * the call's sizes. An access outside is skipped (a load yields zero) and
 * recorded as MAMBA_ERR_DEVICE_BOUNDS in the device error word; nothing traps.
 * TMA copies are bounded by their tensor maps, which are encoded from the same
 * sizes. It is a testing aid (slower), not for production.
 */
int mamba_checked_bounds(void);

/* Human-readable name of a mamba_status value (static string, never NULL). */
const char* mamba_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int mamba_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SCAN_H */
