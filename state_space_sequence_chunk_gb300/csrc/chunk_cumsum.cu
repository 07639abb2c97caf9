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
// One CTA owns (batch, chunk, 32 heads).  The dt tile is read row by row
// (32 consecutive heads per warp load, coalesced), transposed through shared
// memory, then each warp scans whole head columns: every lane sums a run of
// Q/32 consecutive tokens serially and a warp-shuffle scan adds the lane
// offsets.  Tokens past seqlen read as dt = 0, so the padded tail of the last
// chunk repeats the value at the last real token.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kHeadsPerCta = 32;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
chunk_cumsum_kernel(const float* __restrict__ dt, const float* __restrict__ A,
                    float* __restrict__ Gcs, float* __restrict__ dtT,
                    int L, int H, int Q, int Lp) {
    __shared__ float tile[256][kHeadsPerCta + 1];
    const int c = blockIdx.x, h0 = blockIdx.y * kHeadsPerCta, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = c * Q;

    // coalesced load of the [Q, 32] dt tile (zero outside [0, L) x [0, H))
    for (int t = warp; t < Q; t += kThreads / 32) {
        const int tg = t0 + t, h = h0 + lane;
        float v = 0.f;
        if (tg < L && h < H) v = dt[((int64_t)b * L + tg) * H + h];
        tile[t][lane] = v;
    }
    __syncthreads();

    const int per_lane = Q >> 5;  // Q in {64, 128, 256} -> 2, 4 or 8 tokens per lane
    for (int j = warp; j < kHeadsPerCta; j += kThreads / 32) {
        const int h = h0 + j;
        if (h >= H) break;
        const float a = A[h];
        float run = 0.f;
        float vals[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < per_lane) {
                const float v = tile[lane * per_lane + k][j];
                run += a * v;
                vals[k] = run;
            }
        }
        // inclusive warp scan of the lane totals -> exclusive offset per lane
        float incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const float excl = incl - run;
        float out[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) out[k] = (vals[k] + excl) * kLog2e;
        if (t0 + Q > L) {
            // ragged last chunk: the padded slots take exactly the value at the
            // last real token, so that g_last (read at the chunk's last slot) is
            // bit-identical to it
            const int last = L - 1 - t0, src_lane = last / per_lane, src_k = last % per_lane;
            float v = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k == src_k) v = out[k];
            v = __shfl_sync(0xffffffffu, v, src_lane);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (t0 + lane * per_lane + k > L - 1) out[k] = v;
        }
        float* grow = Gcs + ((int64_t)b * H + h) * Lp + t0 + lane * per_lane;
        float* drow = dtT + ((int64_t)b * H + h) * Lp + t0 + lane * per_lane;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < per_lane) {
                grow[k] = out[k];
                drow[k] = tile[lane * per_lane + k][j];
            }
        }
    }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Problem& p, const float* dt, const float* A, float* Gcs,
                                float* dtT, cudaStream_t stream) {
    dim3 grid((unsigned)p.nc, (unsigned)((p.H + kHeadsPerCta - 1) / kHeadsPerCta),
              (unsigned)p.b);
    chunk_cumsum_kernel<<<grid, kThreads, 0, stream>>>(dt, A, Gcs, dtT, (int)p.L, (int)p.H,
                                                        (int)p.Q, (int)p.Lp);
    return cudaGetLastError();
}

}  // namespace ssd
