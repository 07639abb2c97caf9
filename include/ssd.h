/*
 * ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 SSD chunked-scan forward pass.
 *
 * The method: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels
 * in NVIDIA CUDA Tile" (trishampatil.com), sections "The Mamba-2 Recurrence"
 * through "Kernel 3: compute_out"; the formulas are printed in full in the
 * zhiding.cn rendering of the same NVIDIA / Jane Street article, section
 * "Mamba-2架构".  Per head, with decay a_t = A*dt_t < 0:
 *
 *     h_t = exp(a_t) h_{t-1} + dt_t B_t x_t^T          y_t = C_t^T h_t + D x_t
 *
 * evaluated chunk by chunk: chunk_cumsum (in-chunk log-space decay sums G),
 * fwd_pass_state (the state at every chunk start, carried with the jump
 * h <- exp(G_last) h + (exp(G_last - G) o B)^T X) and compute_out
 * (Y = exp(G) o (C h) + ((exp(G_i - G_j) o C B^T) o M)(dt o X) + D X).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All tensor pointers are DEVICE pointers (the current CUDA device), to
 *    contiguous row-major arrays in the layouts given below, 16-byte aligned
 *    (except ssd_fwd_host, whose tensors are in host memory).
 *    The caller owns every buffer; the library allocates no device memory and
 *    keeps no per-call state.  Inputs are only read.
 *  - Letters: b = batch, L = seqlen, H = nheads, P = headdim, N = dstate,
 *    G = ngroups (H % G == 0; head h reads group h / (H/G) of B and C),
 *    Q = chunk_size, nc = ceil(L / Q), Lp = nc * Q.
 *  - Layouts:  x, y [b, L, H, P] (dims.dtype)      dt [b, L, H] (fp32)
 *              B, C [b, L, G, N] (dims.dtype)      A, D [H] (fp32)
 *              init_state, final_state [b, H, P, N] (fp32)
 *    Intermediates (chunk_cumsum / fwd_pass_state outputs):
 *              Gcs, dtT [b, H, Lp] (fp32; token-contiguous, padded to Lp;
 *                  Gcs is pre-scaled by log2(e); padded tokens carry dt = 0)
 *              hiddens [b, H, nc, N, P] (dims.dtype): the state before each
 *                  chunk's first token, stored transposed (row n holds the P
 *                  values S[:, n]), the layout in which both the producing and
 *                  the consuming kernel move whole contiguous rows.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream: no host synchronisation inside.
 *  - Errors: all arguments are validated on the host BEFORE anything is
 *    enqueued; on an error the call returns a status != SSD_OK and launches
 *    nothing.  A failure reported by the CUDA runtime while enqueuing returns
 *    SSD_ERR_CUDA.  Nothing throws across this ABI.
 *  - Timeouts: every wait inside the tensor-core kernels (on a pipeline
 *    barrier, or on the state that another CTA hands on) is bounded, about
 *    1 s of SM clock; a wait that gives up ends its kernel early, with
 *    undefined outputs, instead of hanging the GPU.  Calls are asynchronous,
 *    so such a failure cannot be returned by the call that enqueued it: the
 *    kernel raises a page-locked host word at its end, and the FIRST launching
 *    call on that device that starts after the failed kernel has finished
 *    returns SSD_ERR_TIMEOUT (after validating its arguments) and enqueues
 *    nothing.  Reporting it synchronises the device and clears the record, so
 *    the call after that runs normally.  ssd_take_device_errors() reads and
 *    clears the same record on demand.  The first launching call in a process
 *    page-locks that host word once (make it before any stream capture); if
 *    that fails, only ssd_take_device_errors() reports timeouts.
 *  - Supported sizes: dtype SSD_F32 or SSD_BF16 (x, B, C, y share it);
 *    Q in {64, 128, 256}; P in {16, 32, ..., 256} (multiple of 16);
 *    N in {16, 32, ..., 256} (multiple of 16); H % G == 0; batch >= 0 and
 *    seqlen >= 0 (an empty problem enqueues at most a copy of init_state to
 *    final_state).  The device must be compute capability 10.3.
 */
#ifndef SSD_GB300_SSD_H
#define SSD_GB300_SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_ABI_VERSION 5

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

typedef enum {
    SSD_OK = 0,
    SSD_ERR_NULL = 1,       /* a required pointer is NULL                         */
    SSD_ERR_SHAPE = 2,      /* unsupported or inconsistent sizes                  */
    SSD_ERR_DTYPE = 3,      /* unknown dtype code                                 */
    SSD_ERR_ALIGN = 4,      /* a pointer is not 16-byte aligned                   */
    SSD_ERR_WORKSPACE = 5,  /* workspace smaller than ssd_fwd_workspace_bytes()   */
    SSD_ERR_ARCH = 6,       /* the current device is not compute capability 10.3  */
    SSD_ERR_CUDA = 7,       /* the CUDA runtime reported an error                 */
    SSD_ERR_ALIAS = 8,      /* an output overlaps an input                        */
    SSD_ERR_TIMEOUT = 9     /* a bounded wait in an earlier launch gave up        */
} ssd_status;

/* Problem sizes.  `dtype` is an ssd_dtype: the element type of x, B, C, y and
 * of the hiddens intermediate.  `reserved` must be 0. */
typedef struct {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size;
    int32_t dtype;
    int32_t reserved;
} ssd_dims;

/* Version of this ABI (SSD_ABI_VERSION of the library that was built). */
int ssd_abi_version(void);

/* Static English text for a status code; never NULL. */
const char* ssd_status_string(ssd_status s);

/* Bytes of device workspace that ssd_fwd needs for `d` (the Gcs, dtT and
 * hiddens intermediates and fwd_pass_state's scratch, each 256-byte aligned);
 * 0 if `d` is invalid or empty. */
size_t ssd_fwd_workspace_bytes(const ssd_dims* d);

/* Byte sizes of the two intermediate kinds: Gcs (== dtT) and hiddens.  Returns
 * SSD_OK, or an error for invalid `d` (outputs then untouched). */
ssd_status ssd_intermediate_bytes(const ssd_dims* d, size_t* gcs_bytes, size_t* hiddens_bytes);

/*
 * ssd_fwd -- the whole forward pass: chunk_cumsum, fwd_pass_state and
 * compute_out, in that order, on `stream`.
 *   x, dt, A, B, C      inputs (required).
 *   D                   per-head skip weight [H], or NULL for D = 0.
 *   init_state          [b, H, P, N] fp32, or NULL for a zero initial state.
 *   y                   output [b, L, H, P] (required).
 *   final_state         output [b, H, P, N] fp32, or NULL to skip.  It may be
 *                       the same pointer as init_state (in-place update: each
 *                       state slice is read before it is written); any other
 *                       overlap with an input is SSD_ERR_ALIAS.
 *   workspace           device scratch of >= ssd_fwd_workspace_bytes(d) bytes,
 *                       owned by the caller; its contents on entry do not
 *                       matter and on exit hold Gcs, dtT and hiddens (in that
 *                       order, each 256-byte aligned) and fwd_pass_state's
 *                       scratch.
 */
ssd_status ssd_fwd(const ssd_dims* d, const void* x, const float* dt, const float* A,
                   const void* B, const void* C, const float* D, const float* init_state,
                   void* y, float* final_state, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * ssd_chunk_cumsum -- step 1 ("Kernel 1: chunk_cumsum").
 *   Gcs[b, h, t] = log2(e) * sum_{k = chunk start .. t} A[h] * dt[b, k, h]
 *   dtT[b, h, t] = dt[b, t, h]
 * for t < L; for L <= t < Lp both treat dt as 0 (so Gcs holds the value at the
 * last real token and dtT holds 0).  Gcs and dtT: [b, H, Lp] fp32.
 */
ssd_status ssd_chunk_cumsum(const ssd_dims* d, const float* dt, const float* A,
                            float* Gcs, float* dtT, void* stream);

/* Bytes of device scratch that ssd_fwd_pass_state needs for `d`: for bf16, a
 * two-slot fp32 state buffer per (batch, head, 128-row block of N), through
 * which the units of one head's chunk sequence hand the state on, and a small
 * control block; for long chunk sequences (>= 64 chunks, N <= 128, P <= 64,
 * an even number of heads per group) also 32 MiB of per-range aggregate
 * states, with which the ranges of a sequence run independently and a short
 * scan joins them; 0 for fp32, or if `d` is invalid or empty. */
size_t ssd_fwd_pass_state_scratch_bytes(const ssd_dims* d);

/*
 * ssd_fwd_pass_state -- step 2 ("Kernel 2: fwd_pass_state").
 * For every (b, h), walking the chunks in order from S = init_state (or 0):
 *   hiddens[b, h, c] = S^T                                (in dims.dtype)
 *   S <- 2^{g_last} S + X_c^T (B_c o (dt_c 2^{g_last - g_c}))
 * where g = Gcs of chunk c and g_last its value at the chunk's last real token.
 * final_state (fp32, may be NULL, may equal init_state) receives the last S.
 * scratch: device memory of >= ssd_fwd_pass_state_scratch_bytes(d) bytes
 * (NULL allowed when that is 0), owned by the caller, contents on entry
 * irrelevant (the call clears what it needs on `stream` first); it must not
 * overlap any other argument (SSD_ERR_ALIAS), and a smaller size is
 * SSD_ERR_WORKSPACE.  Two calls that overlap on the GPU must not share it.
 */
ssd_status ssd_fwd_pass_state(const ssd_dims* d, const void* x, const void* B,
                              const float* Gcs, const float* dtT, const float* init_state,
                              void* hiddens, float* final_state, void* scratch,
                              size_t scratch_bytes, void* stream);

/*
 * ssd_compute_out -- step 3 ("Kernel 3: compute_out").  For every (b, chunk, h):
 *   Y = 2^{g} o (C h^T) + ((2^{g_i - g_j} [i >= j]) o (C B^T)) (dt o X) + D X
 * with h = hiddens[b, h, c]; the Q x Q matrix never leaves the chip.  D may be
 * NULL (D = 0).  y [b, L, H, P] in dims.dtype.
 */
ssd_status ssd_compute_out(const ssd_dims* d, const void* x, const void* B, const void* C,
                           const float* Gcs, const float* dtT, const void* hiddens,
                           const float* D, void* y, void* stream);

/*
 * ssd_take_device_errors -- read and clear the device-side error words of the
 * tensor-core kernels (and the host record behind SSD_ERR_TIMEOUT).  Every
 * wait inside those kernels is bounded; a wait that gives up (it never should)
 * sets a bit and the kernel ends early with undefined output instead of
 * hanging.  Bit 0: fwd_pass_state (bf16), bit 1: compute_out (bf16), bit 2:
 * the TF32 kernels of fp32 inputs.  Synchronises the current device; returns
 * 0xFFFFFFFF if the words cannot be read.
 */
unsigned int ssd_take_device_errors(void);

/*
 * ssd_debug_withhold_handoffs -- test hook for failure detection.  With `on`
 * nonzero, later bf16 fwd_pass_state launches on the current device skip
 * publishing the state at the end of each CTA's work range, so that the CTA
 * that continues the chain waits in vain.  That wait is bounded (about 1 s of
 * SM clock): it gives up, sets bit 0 of the error word and the launch ends
 * early with undefined hiddens / final_state (and y).  The device context stays
 * usable; ssd_take_device_errors() reports and clears the bit.  Pass 0 to
 * restore normal operation.  Not for production use.  Returns SSD_ERR_CUDA if
 * the flag cannot be written.
 */
ssd_status ssd_debug_withhold_handoffs(int on);

/*
 * ssd_step -- the token-by-token recurrence, for decoding and other short
 * inputs ("The Mamba-2 Recurrence"; the linear-time streaming mode in which
 * one call's final state is the next call's initial state).  For each
 * (b, h), starting from S = state[b, h] and for t = 0 .. seqlen-1 in order:
 *   S <- exp(A[h] dt[b,t,h]) S + dt[b,t,h] x[b,t,h,:] B[b,t,g,:]^T
 *   y[b,t,h,:] = S C[b,t,g,:] + D[h] x[b,t,h,:]        (g = h / (H/G))
 * and finally state[b, h] = S.  This is ssd_fwd's result computed without
 * chunking: one pass over the state (read once, written once), so it suits
 * a few tokens per call; long inputs belong to ssd_fwd.
 *   d          shapes and dtype as for ssd_fwd; chunk_size is not used.
 *   x, dt, A, B, C, D   as for ssd_fwd (D may be NULL).
 *   state      [b, H, P, N] fp32, read and updated in place (required).
 *   y          output [b, L, H, P] in the x dtype (required).
 * Pointers are device pointers, 16-byte aligned; state and y must not
 * overlap each other or an input (SSD_ERR_ALIAS).  Asynchronous on `stream`.
 */
ssd_status ssd_step(const ssd_dims* d, const void* x, const float* dt, const float* A,
                    const void* B, const void* C, const float* D, float* state, void* y,
                    void* stream);

/* Sizes of a depthwise causal conv1d: x and out are [batch, dim, seqlen] in
 * `dtype`; the filter has `width` taps per channel. */
typedef struct {
    int64_t batch, dim, seqlen, width;
    int32_t dtype;      /* ssd_dtype of x and out */
    int32_t reserved;   /* must be 0 */
} ssd_conv_dims;

/*
 * ssd_causal_conv1d -- the depthwise causal 1-D convolution that precedes the
 * SSD in a Mamba-2 block (Helion hackathon gallery, "Causal Conv1d"):
 *   out[b, d, t] = bias[d] + sum_{k=0}^{W-1} weight[d, k] x[b, d, t - W + 1 + k]
 * with x read as 0 at negative t (causal left padding, done in the kernel).
 *   d        batch >= 0, 1 <= dim <= 65535, seqlen >= 0, 1 <= width <= 8,
 *            batch <= 65535; else SSD_ERR_SHAPE (SSD_ERR_DTYPE for dtype).
 *   x        [batch, dim, seqlen] in d->dtype (required).
 *   weight   [dim, width] fp32 (required); bias [dim] fp32 or NULL (0).
 *   out      [batch, dim, seqlen] in d->dtype (required); it must not
 *            overlap x, weight or bias (SSD_ERR_ALIAS).
 * Device pointers, 16-byte aligned (SSD_ERR_ALIGN).  fp32 arithmetic.
 * Asynchronous on `stream`.
 */
ssd_status ssd_causal_conv1d(const ssd_conv_dims* d, const void* x, const float* weight,
                             const float* bias, void* out, void* stream);

/* Sizes of the Gated DeltaNet chunk kernels: q, k, w [batch, seqlen, nheads,
 * kdim]; u, v_new, o [batch, seqlen, nheads, vdim]; g [batch, seqlen, nheads];
 * h [batch, nheads, nchunks, kdim, vdim] with nchunks = ceil(seqlen / chunk);
 * h0, final_state [batch, nheads, kdim, vdim].  All fp32. */
typedef struct {
    int64_t batch, seqlen, nheads, kdim, vdim, chunk;
    int32_t dtype;      /* SSD_F32 only */
    int32_t reserved;   /* must be 0 */
} ssd_gdn_dims;

/*
 * ssd_gdn_chunk_fwd_h -- Gated DeltaNet state recurrence over chunks (Helion
 * hackathon gallery, "GDN chunk_fwd_h").  g is the in-chunk inclusive
 * cumulative log gate and g_last its value at the chunk's last token; per
 * (b, head), for each chunk in order:
 *   h[b, head, c] = S;  v_new = u - w S;  v_gated[t] = v_new[t] exp(g_last - g_t);
 *   S <- exp(g_last) S + k^T v_gated.
 * S starts at h0 (or 0 if NULL); final_state (may be NULL) receives the last S.
 *   d        4 <= kdim <= 128 with kdim % 4 == 0; 1 <= vdim <= 128;
 *            chunk in {16, 32, 64}; nheads >= 1;
 *            batch >= 0; seqlen >= 0 (else SSD_ERR_SHAPE; SSD_ERR_DTYPE unless fp32).
 *   k, w, u, g   inputs (required).   h, v_new   outputs (required).
 * Device pointers, 16-byte aligned; outputs must not overlap inputs or each
 * other (SSD_ERR_ALIAS).  Asynchronous on `stream`.
 */
ssd_status ssd_gdn_chunk_fwd_h(const ssd_gdn_dims* d, const float* k, const float* w,
                               const float* u, const float* g, const float* h0, float* h,
                               float* v_new, float* final_state, void* stream);

/*
 * ssd_gdn_chunk_fwd_o -- Gated DeltaNet chunk outputs ("GDN chunk_fwd_o"),
 * every chunk independent:
 *   o[t] = exp(g_t) q_t h[b, head, c] + sum_{j <= t in the chunk} (q_t . k_j) exp(g_t - g_j) v_new[j].
 * Inputs q, k, v_new, h (from ssd_gdn_chunk_fwd_h), g; output o.  Same rules
 * as ssd_gdn_chunk_fwd_h.
 */
ssd_status ssd_gdn_chunk_fwd_o(const ssd_gdn_dims* d, const float* q, const float* k,
                               const float* v_new, const float* h, const float* g, float* o,
                               void* stream);

/* Size of the fixed device scratch buffer used by ssd_fwd_noalloc: 32 MiB. */
#define SSD_NOALLOC_WORKSPACE_BYTES ((size_t)32 << 20)

/*
 * ssd_fwd_noalloc -- ssd_fwd for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point.  It exists for callers
 * that cannot call cudaMalloc or any other allocator on their path: a host
 * framework that owns all device memory and hands out only its own fixed
 * buffers, a latency-critical loop that must not call cudaMalloc/cudaFree
 * (those calls can synchronise the device and take driver-wide locks), or a
 * process whose device memory is already fully reserved by a pool.  Such a
 * caller still passes every input and
 * output; the scratch that ssd_fwd takes as `workspace` (the Gcs, dtT and
 * hiddens intermediates) lives instead in one statically sized device array of
 * SSD_NOALLOC_WORKSPACE_BYTES inside this library.  Every GPU that loads the
 * library holds that array until the process exits.
 *
 * Arguments, layouts, ownership and results are those of ssd_fwd, minus the
 * workspace.  Problems whose ssd_fwd_workspace_bytes() exceeds
 * SSD_NOALLOC_WORKSPACE_BYTES are rejected with SSD_ERR_WORKSPACE before
 * anything is enqueued; use ssd_fwd with a caller-owned workspace for those.
 * The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *
 * Set-up: the first call on each device (made with that device current) looks
 * up the device address of the static array once and caches it; make that
 * first call before any stream capture.
 *
 * Sharing: every call on a device uses the same array, and it keeps the last
 * call's contents.  The kernels overwrite every intermediate they read, so
 * nothing has to start at zero.  Calls that overlap on the GPU (on different
 * streams, or from different host threads without ordering) race on the array
 * and give wrong results: serialise them.
 */
ssd_status ssd_fwd_noalloc(const ssd_dims* d, const void* x, const float* dt, const float* A,
                           const void* B, const void* C, const float* D,
                           const float* init_state, void* y, float* final_state, void* stream);

/* Device bytes ssd_fwd_host needs as `staging` for `d` cut into `nslices`
 * batch slices (1 <= nslices <= min(batch, 64)); 0 if `d` or nslices is
 * invalid or the batch is empty. */
size_t ssd_fwd_host_staging_bytes(const ssd_dims* d, int nslices);

/*
 * ssd_fwd_host -- ssd_fwd on host buffers, with the host-device copies of one
 * part of the batch overlapping the computation of another.
 *
 * The batch is cut into nslices contiguous slices of ceil(batch / nslices)
 * elements (the last may be shorter).  For each slice in turn: its inputs are
 * copied to the device on streams[1], ssd_fwd runs on it on streams[0], and
 * its y and final_state are copied back on streams[2].  Two staging slots
 * alternate, so slice k + 1's inputs travel while slice k is computed and
 * slice k - 1's outputs travel back.  Every (batch, head) is an independent
 * recurrence, so each slice is an ssd_fwd problem of its own; its arithmetic
 * per (batch, head) is that of ssd_fwd on the slice.
 *
 *   d, A, D, and the meaning and layout of every tensor: as ssd_fwd, but x,
 *     dt, A, B, C, D, init_state, y and final_state are HOST pointers.  They
 *     should be page-locked (cudaHostAlloc, or pinned by the caller's
 *     framework): pageable memory makes each copy synchronous and removes the
 *     overlap.  final_state may be init_state itself (updated in place); other
 *     overlaps of an output with an input give SSD_ERR_ALIAS.
 *   staging     device buffer, 256-byte aligned, of at least
 *               ssd_fwd_host_staging_bytes(d, nslices) bytes: two slots, each
 *               with the device copies of one slice's tensors and its ssd_fwd
 *               workspace, and A and D.  Caller-owned.
 *   nslices     1 <= nslices <= min(batch, 64) (else SSD_ERR_SHAPE).
 *   streams     three cudaStream_t values: compute (the caller's stream),
 *               copy-in and copy-out.  They may coincide (the work then runs
 *               in order without overlap).
 * Ordering: the copies start after the work enqueued on streams[0] before the
 * call; the call makes streams[0] wait for its last copy, so work enqueued on
 * streams[0] after the call (or a synchronisation of it) sees y and
 * final_state complete in host memory.  The call returns once everything is
 * enqueued.  It creates and releases CUDA events; it allocates no memory.
 * Errors: the validation of ssd_fwd, plus SSD_ERR_WORKSPACE (staging too
 * small), SSD_ERR_ALIGN (staging), SSD_ERR_NULL, SSD_ERR_CUDA (a copy or an
 * event failed; the work already enqueued still completes before streams[0]
 * moves on).
 */
ssd_status ssd_fwd_host(const ssd_dims* d, const void* x, const float* dt, const float* A,
                        const void* B, const void* C, const float* D, const float* init_state,
                        void* y, float* final_state, void* staging, size_t staging_bytes,
                        int nslices, void* const* streams);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_SSD_H */
