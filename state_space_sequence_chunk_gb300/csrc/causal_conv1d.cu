// causal_conv1d.cu -- depthwise causal 1-D convolution, the Mamba-2 block's
// neighbour of the SSD.
//
// Helion hackathon gallery (cerebralvalley.ai), "Causal Conv1d
// (causal_conv1d)": every channel is convolved with its own short filter of W
// taps, with causal (left) zero padding,
//     out[b, d, t] = bias[d] + sum_{k=0}^{W-1} weight[d, k] x[b, d, t - W + 1 + k].
// The entry notes that the filter fits in registers and that the kernel is
// bound by memory bandwidth; the padding is done in the kernel (no padded
// copy of x), as several of the gallery's entries recommend.
//
// GB300 design: plain CUDA-core code shaped for coalescing.  A thread owns two
// 16-byte vectors of one row (8 bf16 or 4 fp32 outputs each), loads both with
// vector loads, takes the W - 1 samples before each from the neighbouring lane
// by shuffles (lane 0 reads its own from global memory; they are in L1), and
// writes vector stores.  Rows whose length is not a multiple of the vector
// width take a one-output-per-thread kernel.  fp32 arithmetic; x and out are
// bf16 or fp32, weight and bias fp32.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kConvThreads = 256;

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
    static constexpr int kN = 8;
    __device__ static void load(const __nv_bfloat16* p, float* v) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ static void store(__nv_bfloat16* p, const float* v) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 t = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&t);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec<float> {
    static constexpr int kN = 4;
    __device__ static void load(const float* p, float* v) {
        const float4 u = *reinterpret_cast<const float4*>(p);
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
    __device__ static void store(float* p, const float* v) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

// Vector path: L % Vec<T>::kN == 0.  A CTA covers kSpan = kVecPerThread *
// threads * V consecutive samples of one row; thread i owns vectors i and
// i + threads, so both loads are in flight together and every warp access
// stays 512 contiguous bytes.  grid (ceil(L / kSpan), dim, batch).
constexpr int kVecPerThread = 2;
template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads)
conv1d_vec_kernel(const T* __restrict__ x, const float* __restrict__ weight,
                  const float* __restrict__ bias, T* __restrict__ out, int dim, int L) {
    constexpr int V = Vec<T>::kN;
    static_assert(W >= 1 && W - 1 <= V, "the halo must come from one neighbouring lane");
    const int d = blockIdx.y, b = blockIdx.z, lane = threadIdx.x & 31;
    const int64_t row = ((int64_t)b * dim + d) * L;
    float wk[W];
#pragma unroll
    for (int k = 0; k < W; ++k) wk[k] = __ldg(weight + (int64_t)d * W + k);
    const float bs = bias != nullptr ? __ldg(bias + d) : 0.f;
    float v[kVecPerThread][V];
    int t0[kVecPerThread];
#pragma unroll
    for (int r = 0; r < kVecPerThread; ++r) {
        t0[r] = ((blockIdx.x * kVecPerThread + r) * kConvThreads + threadIdx.x) * V;
        if (t0[r] < L) Vec<T>::load(x + row + t0[r], v[r]);
        else
#pragma unroll
            for (int i = 0; i < V; ++i) v[r][i] = 0.f;
    }
#pragma unroll
    for (int r = 0; r < kVecPerThread; ++r) {
        const bool live = t0[r] < L;
        // xx = the W - 1 samples before t0, then this vector's V samples
        float xx[W - 1 + V];
#pragma unroll
        for (int i = 0; i < V; ++i) xx[W - 1 + i] = v[r][i];
#pragma unroll
        for (int k = 0; k < W - 1; ++k) {
            float h = __shfl_up_sync(0xffffffffu, v[r][V - (W - 1) + k], 1);
            if (lane == 0) {
                const int ts = t0[r] - (W - 1) + k;
                h = (live && ts >= 0) ? to_f32(x[row + ts]) : 0.f;
            }
            xx[k] = h;
        }
        if (live) {
            float o[V];
#pragma unroll
            for (int i = 0; i < V; ++i) {
                float acc = bs;
#pragma unroll
                for (int k = 0; k < W; ++k) acc = fmaf(wk[k], xx[i + k], acc);
                o[i] = acc;
            }
            Vec<T>::store(out + row + t0[r], o);
        }
    }
}

// Any L: one output per thread.  grid (ceil(L / threads), dim, batch).
template <typename T>
__global__ void __launch_bounds__(kConvThreads)
conv1d_scalar_kernel(const T* __restrict__ x, const float* __restrict__ weight,
                     const float* __restrict__ bias, T* __restrict__ out, int dim, int L, int W) {
    const int d = blockIdx.y, b = blockIdx.z;
    const int t = blockIdx.x * kConvThreads + threadIdx.x;
    if (t >= L) return;
    const int64_t row = ((int64_t)b * dim + d) * L;
    float acc = bias != nullptr ? __ldg(bias + d) : 0.f;
    for (int k = 0; k < W; ++k) {
        const int ts = t - W + 1 + k;
        if (ts >= 0) acc = fmaf(__ldg(weight + (int64_t)d * W + k), to_f32(x[row + ts]), acc);
    }
    out[row + t] = from_f32<T>(acc);
}

template <typename T>
cudaError_t launch_t(const ConvProblem& p, const void* x, const float* weight, const float* bias,
                     void* out, cudaStream_t stream) {
    constexpr int V = Vec<T>::kN;
    const T* xt = (const T*)x;
    T* ot = (T*)out;
    const int dim = (int)p.dim, L = (int)p.L;
    // the vector path takes its W - 1 earlier samples from the left lane alone
    if (L % V == 0 && p.W - 1 <= V) {
        const int span = kVecPerThread * kConvThreads * V;
        const dim3 grid((unsigned)((L + span - 1) / span), (unsigned)dim, (unsigned)p.b);
        switch (p.W) {
            case 1: conv1d_vec_kernel<T, 1><<<grid, kConvThreads, 0, stream>>>(xt, weight, bias, ot, dim, L); break;
            case 2: conv1d_vec_kernel<T, 2><<<grid, kConvThreads, 0, stream>>>(xt, weight, bias, ot, dim, L); break;
            case 3: conv1d_vec_kernel<T, 3><<<grid, kConvThreads, 0, stream>>>(xt, weight, bias, ot, dim, L); break;
            case 4: conv1d_vec_kernel<T, 4><<<grid, kConvThreads, 0, stream>>>(xt, weight, bias, ot, dim, L); break;
            case 5: conv1d_vec_kernel<T, 5><<<grid, kConvThreads, 0, stream>>>(xt, weight, bias, ot, dim, L); break;
            default:
                if constexpr (V >= 7) {
                    if (p.W == 6) conv1d_vec_kernel<T, 6><<<grid, kConvThreads, 0, stream>>>(xt, weight, bias, ot, dim, L);
                    else if (p.W == 7) conv1d_vec_kernel<T, 7><<<grid, kConvThreads, 0, stream>>>(xt, weight, bias, ot, dim, L);
                    else if (p.W == 8) conv1d_vec_kernel<T, 8><<<grid, kConvThreads, 0, stream>>>(xt, weight, bias, ot, dim, L);
                    else return cudaErrorInvalidValue;
                } else {
                    return cudaErrorInvalidValue;
                }
        }
    } else {
        const dim3 grid((unsigned)((L + kConvThreads - 1) / kConvThreads), (unsigned)dim,
                        (unsigned)p.b);
        conv1d_scalar_kernel<T><<<grid, kConvThreads, 0, stream>>>(xt, weight, bias, ot, dim, L,
                                                                   (int)p.W);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_causal_conv1d(const ConvProblem& p, const void* x, const float* weight,
                                 const float* bias, void* out, cudaStream_t stream) {
    return p.dtype == SSD_BF16 ? launch_t<__nv_bfloat16>(p, x, weight, bias, out, stream)
                               : launch_t<float>(p, x, weight, bias, out, stream);
}

}  // namespace ssd
