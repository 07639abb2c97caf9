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
// consecutive heads per token, transposed through shared memory, then each of
// the 8 warps scans one head column in 32-token blocks with warp shuffles,
// carrying the running total between blocks.  Tokens past
// seqlen read as dt = 0, and the padded tail of the last chunk takes exactly
// the value at the last real token.
#include "sm100_ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
chunk_cumsum_kernel(const float* __restrict__ dt, const float* __restrict__ A,
                    float* __restrict__ Gcs, float* __restrict__ dtT,
                    int L, int H, int Q, int Lp, unsigned int* zero_ptr, int zero_words) {
    __shared__ float tile[256][kHeadsPerCta + 1];
    grid_launch_dependents();   // fwd_pass_state may start its set-up meanwhile
    // the first CTA also clears the next kernel's control block
    if (zero_ptr != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int i = threadIdx.x; i < zero_words; i += kThreads) zero_ptr[i] = 0u;
    static_assert(kThreads / 32 == kHeadsPerCta, "one warp per head column");
    const int c = blockIdx.x, h0 = blockIdx.y * kHeadsPerCta, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = c * Q;

    // load of the [Q, 8] dt tile (zero outside [0, L) x [0, H)): thread i reads
    // head i % 8 of token i / 8, so a warp covers 4 tokens x 8 heads per load
#pragma unroll 8
    for (int i = threadIdx.x; i < Q * kHeadsPerCta; i += kThreads) {
        const int t = i / kHeadsPerCta, hh = i % kHeadsPerCta;
        const int tg = t0 + t, h = h0 + hh;
        float v = 0.f;
        if (tg < L && h < H) v = dt[((int64_t)b * L + tg) * H + h];
        tile[t][hh] = v;
    }
    __syncthreads();

    // Each warp scans whole head columns.  Lane l takes tokens l, l + 32, ...:
    // the column reads are conflict-free and every store is a coalesced
    // 128-byte row.  A 32-token block is scanned with warp shuffles and the
    // running total of the earlier blocks is carried in a register.
    const int tl = L - 1 - t0;  // local index of the chunk's last real token
    for (int j = warp; j < kHeadsPerCta; j += kThreads / 32) {
        const int h = h0 + j;
        if (h >= H) break;
        const float a = A[h];
        float* grow = Gcs + ((int64_t)b * H + h) * Lp + t0;
        float* drow = dtT + ((int64_t)b * H + h) * Lp + t0;
        float carry = 0.f, last = 0.f;
        for (int k = 0; k < Q; k += 32) {
            const int t = k + lane;
            const float d = tile[t][j];
            float v = a * d;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += o;
            }
            float out = (carry + v) * kLog2e;
            carry += __shfl_sync(0xffffffffu, v, 31);
            // ragged last chunk: the padded slots take exactly the value at the
            // last real token, so that g_last (read at the chunk's last slot) is
            // bit-identical to it
            if (tl >= k && tl < k + 32) last = __shfl_sync(0xffffffffu, out, tl - k);
            if (t > tl) out = last;
            grow[t] = out;
            drow[t] = d;
        }
    }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Problem& p, const float* dt, const float* A, float* Gcs,
                                float* dtT, unsigned int* zero_ptr, int zero_words,
                                cudaStream_t stream) {
    dim3 grid((unsigned)p.nc, (unsigned)((p.H + kHeadsPerCta - 1) / kHeadsPerCta),
              (unsigned)p.b);
    chunk_cumsum_kernel<<<grid, kThreads, 0, stream>>>(dt, A, Gcs, dtT, (int)p.L, (int)p.H,
                                                        (int)p.Q, (int)p.Lp, zero_ptr,
                                                        zero_words);
    return cudaGetLastError();
}

}  // namespace ssd
