// chunk_cumsum.cu -- step 1 of the SSD forward pass.
//
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Kernel 1: chunk_cumsum": for head h and token t of
// chunk c, Gcs = log2(e) * inclusive in-chunk cumulative sum of A[h] * dt.
// The zhiding.cn rendering, section "Mamba-2性能优化" (global memory layout),
// recommends storing the result token-contiguous, [batch, head, token], so
// that the two later kernels read it with contiguous (TMA-able) loads; dt is
// transposed into the same layout in the same pass.
//
// One CTA owns (batch, chunk, 8 heads) -- a grid of nc * H/8 * batch CTAs, so
// that enough loads are in flight.  The dt tile is read as 32-byte runs of 8
// consecutive heads per token and transposed through shared memory into one
// row per head.  Each of the 8 warps then scans one head: lane l owns the
// E = Q/32 consecutive tokens [l E, l E + E), sums them in registers, and one
// 5-step shuffle scan of the lanes' totals gives every lane its offset; each
// lane writes its E outputs as 16-byte (or 8-byte) stores.  Tokens past
// seqlen read as dt = 0, and the padded tail of the last chunk takes exactly
// the value at the last real token.
#include "sm100_ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr int kThreads = 256;
constexpr int kPitch = 256 + 4;   // floats per head row: the transposing stores hit 32 banks

template <int E>
__device__ __forceinline__ void load_run(const float* p, float (&v)[E]) {
    if constexpr (E == 2) {
        const float2 a = *reinterpret_cast<const float2*>(p);
        v[0] = a.x; v[1] = a.y;
    } else {
#pragma unroll
        for (int k = 0; k < E; k += 4) {
            const float4 a = *reinterpret_cast<const float4*>(p + k);
            v[k] = a.x; v[k + 1] = a.y; v[k + 2] = a.z; v[k + 3] = a.w;
        }
    }
}
template <int E>
__device__ __forceinline__ void store_run(float* p, const float (&v)[E]) {
    if constexpr (E == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    } else {
#pragma unroll
        for (int k = 0; k < E; k += 4)
            *reinterpret_cast<float4*>(p + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
    }
}

template <int Q>
__global__ void __launch_bounds__(kThreads)
chunk_cumsum_kernel(const float* __restrict__ dt, const float* __restrict__ A,
                    float* __restrict__ Gcs, float* __restrict__ dtT,
                    int L, int H, int Lp, unsigned int* zero_ptr, int zero_words) {
    constexpr int E = Q / 32;   // tokens per lane
    __shared__ __align__(16) float tile[kHeadsPerCta][kPitch];
    grid_launch_dependents();   // fwd_pass_state may start its set-up meanwhile
    // the first CTA also clears the next kernel's control block
    if (zero_ptr != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int i = threadIdx.x; i < zero_words; i += kThreads) zero_ptr[i] = 0u;
    static_assert(kThreads / 32 == kHeadsPerCta, "one warp per head");
    const int c = blockIdx.x, h0 = blockIdx.y * kHeadsPerCta, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = c * Q;

    // load of the [Q, 8] dt tile (zero outside [0, L) x [0, H)): thread i reads
    // head i % 8 of token i / 8, so a warp covers 4 tokens x 8 heads per load
#pragma unroll
    for (int i = threadIdx.x; i < Q * kHeadsPerCta; i += kThreads) {
        const int t = i / kHeadsPerCta, hh = i % kHeadsPerCta;
        const int tg = t0 + t, h = h0 + hh;
        float v = 0.f;
        if (tg < L && h < H) v = dt[((int64_t)b * L + tg) * H + h];
        tile[hh][t] = v;
    }
    __syncthreads();

    const int h = h0 + warp;
    if (h >= H) return;   // no barrier follows
    const float a = A[h];
    float d[E], g[E];
    load_run<E>(&tile[warp][lane * E], d);
    float run = 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) {
        run += a * d[k];
        g[k] = run;
    }
    // inclusive scan of the lanes' totals; lane l adds the total of lanes < l
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    const float base = incl - run;
#pragma unroll
    for (int k = 0; k < E; ++k) g[k] = (base + g[k]) * kLog2e;
    // ragged last chunk: the padded slots take exactly the value at the last
    // real token, so that g_last (read at the chunk's last slot) is
    // bit-identical to it
    const int tl = L - 1 - t0;  // local index of the chunk's last real token
    if (tl < Q - 1) {           // CTA-uniform
        float mine = 0.f;
#pragma unroll
        for (int k = 0; k < E; ++k)
            if (k == tl % E) mine = g[k];
        const float last = __shfl_sync(0xffffffffu, mine, tl / E);
#pragma unroll
        for (int k = 0; k < E; ++k)
            if (lane * E + k > tl) g[k] = last;
    }
    const int64_t row = ((int64_t)b * H + h) * Lp + t0 + lane * E;
    store_run<E>(Gcs + row, g);
    store_run<E>(dtT + row, d);
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Problem& p, const float* dt, const float* A, float* Gcs,
                                float* dtT, unsigned int* zero_ptr, int zero_words,
                                cudaStream_t stream) {
    dim3 grid((unsigned)p.nc, (unsigned)((p.H + kHeadsPerCta - 1) / kHeadsPerCta),
              (unsigned)p.b);
    auto kern = p.Q == 64 ? chunk_cumsum_kernel<64>
                          : (p.Q == 128 ? chunk_cumsum_kernel<128> : chunk_cumsum_kernel<256>);
    kern<<<grid, kThreads, 0, stream>>>(dt, A, Gcs, dtT, (int)p.L, (int)p.H, (int)p.Lp, zero_ptr,
                                        zero_words);
    return cudaGetLastError();
}

}  // namespace ssd
