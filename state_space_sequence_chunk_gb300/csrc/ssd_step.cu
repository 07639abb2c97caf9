// ssd_step.cu -- the token-by-token recurrence for short inputs (decode).
//
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "The Mamba-2 Recurrence" (formulas in the zhiding.cn
// rendering, section "Mamba-2架构"): per (batch, head) and token t,
//     S <- exp(A dt_t) S + dt_t x_t B_t^T,      y_t = S C_t + D x_t,
// where S is the P x N state.  The pages name the linear-time streaming use --
// the final state of one call is the initial state of the next -- as the
// method's inference mode; this kernel takes a running state and advances it
// over a few tokens, where the chunked pass would be all set-up.
//
// The step is bound by the state's HBM traffic (read once, written once per
// call, 8 P N bytes per head), so the kernel is plain CUDA-core code shaped
// for coalescing: one CTA per (batch, head), each warp holding four state
// rows at a time, each lane float4 groups of a row (lanes cover 512
// consecutive bytes).  The rows stay in registers across the call's tokens;
// y_t[p] is a warp reduction of S C_t.  fp32 arithmetic throughout; x, B, C
// and y are bf16 or fp32.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kStepThreads = 256;
constexpr int kRows = 4;               // state rows per warp in flight

__device__ __forceinline__ float4 load4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
}

// kMaxGroupsPerLane float4 groups of a row per lane: 1 for N <= 128, 2 for N <= 256
template <typename T, int kMaxGroupsPerLane>
__global__ void __launch_bounds__(kStepThreads, kMaxGroupsPerLane == 1 ? 4 : 2)
ssd_step_kernel(const T* __restrict__ x, const float* __restrict__ dt,
                const float* __restrict__ A, const T* __restrict__ B, const T* __restrict__ C,
                const float* __restrict__ D, float* __restrict__ state, T* __restrict__ y,
                int L, int H, int P, int N, int G) {
    const int bh = blockIdx.x, b = bh / H, h = bh - b * H, g = h / (H / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int nwarps = kStepThreads / 32;
    const int n4 = N >> 2;
    const float a = A[h] * kLog2e;             // exp(A dt) = 2^(log2(e) A dt)
    const float dh = D != nullptr ? D[h] : 0.f;
    float* srow0 = state + (int64_t)bh * P * N;
    // kRows rows per warp at a time (rows p0, p0 + 8, ...): their loads are in
    // flight together, and B_t, C_t are loaded once for all of them
    for (int p0 = warp; p0 < P; p0 += nwarps * kRows) {
        float4 s[kRows][kMaxGroupsPerLane];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int p = p0 + r * nwarps;
#pragma unroll
            for (int k = 0; k < kMaxGroupsPerLane; ++k) {
                const int j = lane + 32 * k;
                s[r][k] = (p < P && j < n4) ? *reinterpret_cast<const float4*>(srow0 + (int64_t)p * N + 4 * j)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        for (int t = 0; t < L; ++t) {
            const int64_t bt = (int64_t)b * L + t;
            const float dtv = dt[bt * H + h];
            const float decay = exp2f(a * dtv);
            const T* Bt = B + (bt * G + g) * N;
            const T* Ct = C + (bt * G + g) * N;
            const T* xt = x + (bt * H + h) * P;
            float4 bv[kMaxGroupsPerLane], cv[kMaxGroupsPerLane];
#pragma unroll
            for (int k = 0; k < kMaxGroupsPerLane; ++k) {
                const int j = lane + 32 * k;
                if (j < n4) {
                    bv[k] = load4(Bt + 4 * j);
                    cv[k] = load4(Ct + 4 * j);
                }
            }
            float xv[kRows], part[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const int p = p0 + r * nwarps;
                xv[r] = p < P ? to_f32(xt[p]) : 0.f;
                const float coef = dtv * xv[r];
                part[r] = 0.f;
#pragma unroll
                for (int k = 0; k < kMaxGroupsPerLane; ++k) {
                    const int j = lane + 32 * k;
                    if (j < n4) {
                        s[r][k].x = fmaf(decay, s[r][k].x, coef * bv[k].x);
                        s[r][k].y = fmaf(decay, s[r][k].y, coef * bv[k].y);
                        s[r][k].z = fmaf(decay, s[r][k].z, coef * bv[k].z);
                        s[r][k].w = fmaf(decay, s[r][k].w, coef * bv[k].w);
                        part[r] = fmaf(s[r][k].x, cv[k].x, part[r]);
                        part[r] = fmaf(s[r][k].y, cv[k].y, part[r]);
                        part[r] = fmaf(s[r][k].z, cv[k].z, part[r]);
                        part[r] = fmaf(s[r][k].w, cv[k].w, part[r]);
                    }
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int r = 0; r < kRows; ++r) part[r] += __shfl_xor_sync(0xffffffffu, part[r], off);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    const int p = p0 + r * nwarps;
                    if (p < P) y[(bt * H + h) * P + p] = from_f32<T>(part[r] + dh * xv[r]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int p = p0 + r * nwarps;
#pragma unroll
            for (int k = 0; k < kMaxGroupsPerLane; ++k) {
                const int j = lane + 32 * k;
                if (p < P && j < n4) *reinterpret_cast<float4*>(srow0 + (int64_t)p * N + 4 * j) = s[r][k];
            }
        }
    }
}

}  // namespace

cudaError_t launch_ssd_step(const Problem& p, const void* x, const float* dt, const float* A,
                            const void* B, const void* C, const float* D, float* state, void* y,
                            cudaStream_t stream) {
    const dim3 grid((unsigned)(p.b * p.H));
    const bool wide = p.N > 128;
    if (p.dtype == SSD_BF16) {
        auto k = wide ? ssd_step_kernel<__nv_bfloat16, 2> : ssd_step_kernel<__nv_bfloat16, 1>;
        k<<<grid, kStepThreads, 0, stream>>>(
            (const __nv_bfloat16*)x, dt, A, (const __nv_bfloat16*)B, (const __nv_bfloat16*)C, D,
            state, (__nv_bfloat16*)y, (int)p.L, (int)p.H, (int)p.P, (int)p.N, (int)p.G);
    } else {
        auto k = wide ? ssd_step_kernel<float, 2> : ssd_step_kernel<float, 1>;
        k<<<grid, kStepThreads, 0, stream>>>(
            (const float*)x, dt, A, (const float*)B, (const float*)C, D, state, (float*)y,
            (int)p.L, (int)p.H, (int)p.P, (int)p.N, (int)p.G);
    }
    return cudaGetLastError();
}

}  // namespace ssd
