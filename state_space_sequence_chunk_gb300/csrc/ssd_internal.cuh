// ssd_internal.cuh -- shared declarations of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

// log2(e): G is stored pre-multiplied by it so that every later exponential is
// a base-2 one ("Kernel 1: chunk_cumsum": e^v = 2^(v log2 e)).
constexpr float kLog2e = 1.4426950408889634f;

// Problem sizes after validation, with the derived quantities.
struct Problem {
    int64_t b, L, H, P, N, G, Q;
    int64_t nc;   // number of chunks, ceil(L / Q)
    int64_t Lp;   // padded token count nc * Q (row length of Gcs / dtT)
    int64_t hpg;  // heads per group, H / G
    int dtype;    // ssd_dtype
    int esize;    // bytes per element of x, B, C, y, hiddens
    // Set by ssd_fwd: the three launches form one chain on one stream, so the
    // tensor-core kernels are launched with programmatic dependent launch (each
    // may start its set-up while its predecessor drains; its first read of the
    // predecessor's output waits for that grid with griddepcontrol.wait).
    bool chained = false;
};

inline size_t round_up256(size_t v) { return (v + 255) / 256 * 256; }

// Scratch of the tensor-core fwd_pass_state (bf16 only; 0 bytes otherwise): a
// two-slot fp32 state ring per chain, then a control block of 32-bit words --
// word 0 the work-ticket counter, words kCtrlFlagOffset + chain the chains'
// hand-off flags.  The control block must be zero when the kernel starts.
constexpr int kCtrlFlagOffset = 32;
size_t fwd_pass_state_scratch_bytes(const Problem& p);
size_t fwd_pass_state_ctrl_offset(const Problem& p);
size_t fwd_pass_state_ctrl_bytes(const Problem& p);

// Launchers (defined next to their kernels).  All enqueue on `stream` and
// return cudaGetLastError().  chunk_cumsum also zeroes `zero_words` 32-bit
// words at `zero_ptr` (may be NULL), so that a following fwd_pass_state finds
// its control block cleared without a separate launch.
cudaError_t launch_chunk_cumsum(const Problem& p, const float* dt, const float* A, float* Gcs,
                                float* dtT, unsigned int* zero_ptr, int zero_words,
                                cudaStream_t stream);
// `scratch` holds fwd_pass_state_scratch_bytes(p) bytes; unless `ctrl_zeroed`,
// its control block is cleared with a memset first.
cudaError_t launch_fwd_pass_state(const Problem& p, const void* x, const void* B,
                                  const float* Gcs, const float* dtT, const float* init,
                                  void* hiddens, float* final_state, void* scratch,
                                  bool ctrl_zeroed, cudaStream_t stream);
cudaError_t launch_compute_out(const Problem& p, const void* x, const void* B, const void* C,
                               const float* Gcs, const float* dtT, const void* hiddens,
                               const float* D, void* y, cudaStream_t stream);

// Depthwise causal conv1d sizes after validation (ssd_causal_conv1d).
struct ConvProblem {
    int64_t b, dim, L, W;
    int dtype;   // ssd_dtype of x and out
    int esize;
};
cudaError_t launch_causal_conv1d(const ConvProblem& p, const void* x, const float* weight,
                                 const float* bias, void* out, cudaStream_t stream);

// Gated DeltaNet chunk kernels (ssd_gdn_chunk_fwd_h / _o), sizes after validation.
struct GdnProblem {
    int64_t B, T, H, K, V, C, NT;
};
cudaError_t launch_gdn_fwd_h(const GdnProblem& p, const float* k, const float* w, const float* u,
                             const float* g, const float* h0, float* h, float* v_new,
                             float* final_state, cudaStream_t stream);
cudaError_t launch_gdn_fwd_o(const GdnProblem& p, const float* q, const float* k,
                             const float* v_new, const float* h, const float* g, float* o,
                             cudaStream_t stream);

// The token-by-token recurrence over p.L tokens from `state` (in place).
cudaError_t launch_ssd_step(const Problem& p, const void* x, const float* dt, const float* A,
                            const void* B, const void* C, const float* D, float* state, void* y,
                            cudaStream_t stream);

// Tensor-core (tcgen05) variants for bf16 inputs.
cudaError_t launch_fwd_pass_state_tc(const Problem& p, const void* x, const void* B,
                                     const float* Gcs, const float* dtT, const float* init,
                                     void* hiddens, float* final_state, void* scratch,
                                     cudaStream_t stream);
bool compute_out_tc_supports(const Problem& p);
cudaError_t launch_compute_out_tc(const Problem& p, const void* x, const void* B, const void* C,
                                  const float* Gcs, const float* dtT, const void* hiddens,
                                  const float* D, void* y, cudaStream_t stream);
// Device-usable address of the current device's page-locked host word through
// which a tensor-core kernel reports, at its end, that one of its bounded waits
// gave up (see report_timeout_to_host); NULL if it could not be set up.  The
// first call page-locks the word (once per process).
unsigned int* host_timeout_word();
// SSD_ERR_TIMEOUT if a tensor-core kernel on the current device has raised
// its host word since the last report (the report synchronises the device and
// clears the device and host records), else SSD_OK (SSD_ERR_CUDA if the device
// cannot be queried).
ssd_status timeout_pending();
// TF32 tensor-core kernels for fp32 inputs (N <= 128, P <= 128): the chunk
// products of fwd_pass_state (written into the hiddens slots; the state scan
// follows) and compute_out.
bool tf32_path_supports(const Problem& p);
cudaError_t launch_fps_products_tf32(const Problem& p, const void* x, const void* B,
                                     const float* Gcs, const float* dtT, void* hiddens,
                                     cudaStream_t stream);
cudaError_t launch_compute_out_tf32(const Problem& p, const void* x, const void* B, const void* C,
                                    const float* Gcs, const float* dtT, const void* hiddens,
                                    const float* D, void* y, cudaStream_t stream);
unsigned int take_tf32_error();
// Gated DeltaNet on the TF32 tensor cores (K, V multiples of 16, at most 128).
bool gdn_tf32_supports(const GdnProblem& p);
cudaError_t launch_gdn_fwd_o_tf32(const GdnProblem& p, const float* q, const float* k,
                                  const float* v_new, const float* h, const float* g, float* o,
                                  cudaStream_t stream);
cudaError_t launch_gdn_fwd_h_tf32(const GdnProblem& p, const float* k, const float* w,
                                  const float* u, const float* g, const float* h0, float* h,
                                  float* v_new, float* final_state, cudaStream_t stream);
// Read and clear the device-side error word of a kernel module (bit 0: a
// bounded wait gave up).  Synchronous.
unsigned int take_fwd_pass_state_error();
// Test hook: nonzero makes fwd_pass_state withhold its range hand-offs.
cudaError_t set_fwd_pass_state_withhold(unsigned int on);
unsigned int take_compute_out_error();

// Launch kern on stream, with programmatic dependent launch when pdl is set
// (the kernel then waits on the previous grid with griddepcontrol.wait before
// it reads that grid's output).
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Element loads/stores shared by the kernels.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

}  // namespace ssd
