// fwd_pass_state_tc.cu -- step 2 of the SSD forward pass on the tcgen05
// tensor cores (bf16 inputs, fp32 state).
//
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Kernel 2: fwd_pass_state" (with "Step 1" and "Step 3"):
// per (batch, head) the chunks are walked in order; the state at each chunk
// start is stored, then the jump
//     S <- 2^{g_last} S + X_c^T (B_c o dt_c 2^{g_last - g_c})
// carries it across the chunk.
//
// GB300 design (what differs from the pages' cuTile kernel):
//  * The product is issued swapped, S^T (N x P) += B_c^T (s o X_c), so the
//    state dimension N is the MMA's M (128 TMEM lanes).  The zhiding.cn
//    rendering, "Mamba-2性能优化" (swapping the A/B operands), describes the same
//    B^T A^T = (A B)^T swap for Blackwell.
//  * Every chunk's product D_c = B_c^T (s o X_c) goes into a FRESH TMEM
//    accumulator (two, used alternately), and the epilogue warps fold it into
//    the running state held in registers, S <- 2^{g_last} S + D_c.  The
//    tensor core never waits for the previous chunk's state: only the cheap
//    register update is serial.
//  * x and B stream in 64-token sub-chunks through a multi-stage TMA ring
//    (128-byte swizzle, token-major rows, read as MN-major operands).  The
//    per-token scale s_q = dt_q 2^{g_last - g_q} is applied to the x rows in
//    shared memory by one warp (a row is contiguous in the swizzled tile).
//
// Warp roles (224 threads): 0 TMA producer, 1 MMA issuer (and TMEM owner),
// 2 row scaler, 3..6 epilogue (TMEM lane quarter = warp % 4).
//
// CTA = (128-row block of N, batch * head).  N and P are padded to the
// 64-element swizzle atom by the TMA's zero fill; padded rows/columns are
// computed and never stored.
#include <cuda.h>

#include "sm100_ptx.cuh"
#include "ssd_internal.cuh"
#include "tma_host.cuh"

namespace ssd {
namespace {

__device__ unsigned int g_fps_error;  // bit 0: a bounded wait gave up

constexpr int kSub = 64;            // tokens per pipeline stage
constexpr int kRowBytes = 128;      // one swizzle row (64 bf16)
constexpr int kThreads = 224;

template <int PP>
struct FpsCfg {
    static constexpr int kStages = PP == 64 ? 4 : 3;
    static constexpr int kXBytes = kSub * PP * 2;         // x sub-tile
    static constexpr int kBBytes = kSub * 128 * 2;        // B sub-tile (128 state rows)
    static constexpr int kVecOff = kXBytes + kBBytes;     // g[64], dt[64], last 4 g of the chunk
    static constexpr int kVecBytes = 2 * kSub * 4 + 16;
    static constexpr int kStageBytes = (kVecOff + kVecBytes + 1023) / 1024 * 1024;
    static constexpr int kTmemCols = 2 * PP;              // two accumulators
    static constexpr int kBarBytes = 256;
    static constexpr int kSmem = kStages * kStageBytes + kBarBytes + 1024;
    static constexpr uint32_t kIdesc = make_idesc(1, 128, PP, 1, 1);
};

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}

template <int PP>
__global__ void __launch_bounds__(kThreads, PP == 64 ? 2 : 1)
fwd_pass_state_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                  const float* __restrict__ Gcs, const float* __restrict__ dtT, const float* init,
                  __nv_bfloat16* __restrict__ hiddens, float* final_state, int H, int P, int N,
                  int Q, int nc, int Lp, int hpg) {
    using Cfg = FpsCfg<PP>;
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
    // barrier indices
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto scaled = [&](int s) { return smem_u32(bars + S + s); };
    auto empty = [&](int s) { return smem_u32(bars + 2 * S + s); };
    auto acc_full = [&](int j) { return smem_u32(bars + 3 * S + j); };
    auto acc_empty = [&](int j) { return smem_u32(bars + 3 * S + 2 + j); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * S + 4);

    const int mb = blockIdx.x, bh = blockIdx.y;
    const int b = bh / H, h = bh % H, grp = h / hpg;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsub = Q / kSub;
    const int total = nc * nsub;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(scaled(s), 32);
            mbar_init(empty(s), 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(acc_full(j), 1);
            mbar_init(acc_empty(j), 128);
        }
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), Cfg::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t stage0 = smem_u32(smem);

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            for (int i = 0; i < total; ++i) {
                const int s = i % S, k = i / S;
                mbar_wait(empty(s), (k & 1) ^ 1, &g_fps_error, 1u);
                const uint32_t xs = stage0 + s * Cfg::kStageBytes, bs = xs + Cfg::kXBytes;
                const int c = i / nsub, sub = i % nsub;
                const int t = c * Q + sub * kSub;
                mbar_arrive_expect_tx(full(s), Cfg::kXBytes + Cfg::kBBytes + Cfg::kVecBytes);
#pragma unroll
                for (int j = 0; j < PP / 64; ++j)
                    tma_load_4d(xs + j * kSub * kRowBytes, &tm_x, full(s), j * 64, h, t, b);
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    tma_load_4d(bs + j * kSub * kRowBytes, &tm_b, full(s), mb * 128 + j * 64, grp,
                                t, b);
                const int64_t ro = (int64_t)bh * Lp;
                const uint32_t vs = xs + Cfg::kVecOff;
                bulk_load(vs, Gcs + ro + t, kSub * 4, full(s));
                bulk_load(vs + kSub * 4, dtT + ro + t, kSub * 4, full(s));
                bulk_load(vs + 2 * kSub * 4, Gcs + ro + (int64_t)c * Q + Q - 4, 16, full(s));
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            for (int i = 0; i < total; ++i) {
                const int s = i % S, k = i / S;
                const int c = i / nsub, sub = i % nsub;
                const int acc = c & 1, use = c >> 1;
                if (sub == 0) mbar_wait(acc_empty(acc), (use & 1) ^ 1, &g_fps_error, 1u);
                mbar_wait(scaled(s), k & 1, &g_fps_error, 1u);
                tc_fence_after();
                const uint32_t xs = stage0 + s * Cfg::kStageBytes, bs = xs + Cfg::kXBytes;
#pragma unroll
                for (int kk = 0; kk < kSub / 16; ++kk) {
                    // A = B_c^T: M = 128 state rows (two 64-row swizzle atoms,
                    // kSub*128 bytes apart), K = 16 tokens, MN-major.
                    const uint64_t adesc = smem_desc_sw128(bs + kk * 16 * kRowBytes,
                                                           kSub * kRowBytes, 8 * kRowBytes);
                    // B = s o X_c: N = PP columns of P, K = 16 tokens, MN-major.
                    const uint64_t bdesc = smem_desc_sw128(xs + kk * 16 * kRowBytes,
                                                           kSub * kRowBytes, 8 * kRowBytes);
                    mma_f16_ss(tmem + acc * PP, adesc, bdesc, Cfg::kIdesc,
                               (sub > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(empty(s));
                if (sub == nsub - 1) mma_commit(acc_full(acc));
            }
        }
    } else if (warp == 2) {
        // ---------------- row scaler: x_q <- x_q * dt_q 2^{g_last - g_q} ----------------
        for (int i = 0; i < total; ++i) {
            const int s = i % S, k = i / S;
            mbar_wait(full(s), k & 1, &g_fps_error, 1u);
            uint8_t* xs = smem + s * Cfg::kStageBytes;
            const float* gv = reinterpret_cast<const float*>(xs + Cfg::kVecOff);
            const float* dv = gv + kSub;
            const float glast = gv[2 * kSub + 3];
            const float s0 = dv[lane] * exp2f(glast - gv[lane]);
            const float s1 = dv[lane + 32] * exp2f(glast - gv[lane + 32]);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int r = lane + 32 * half;
                const float sc = half ? s1 : s0;
#pragma unroll
                for (int j = 0; j < PP / 64; ++j) {
                    uint4* row = reinterpret_cast<uint4*>(xs + j * kSub * kRowBytes + r * kRowBytes);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        uint4 v = row[q];
                        v.x = pack_bf16(bf16lo(v.x) * sc, bf16hi(v.x) * sc);
                        v.y = pack_bf16(bf16lo(v.y) * sc, bf16hi(v.y) * sc);
                        v.z = pack_bf16(bf16lo(v.z) * sc, bf16hi(v.z) * sc);
                        v.w = pack_bf16(bf16lo(v.w) * sc, bf16hi(v.w) * sc);
                        row[q] = v;
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(scaled(s));
        }
    } else {
        // ---------------- epilogue: the serial state update ----------------
        const int quarter = warp & 3;
        const int n = mb * 128 + quarter * 32 + lane;
        const bool nok = n < N;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        float Sr[PP];
        const int64_t sbase = (int64_t)bh * P * N;
#pragma unroll
        for (int p = 0; p < PP; ++p)
            Sr[p] = (init != nullptr && nok && p < P) ? init[sbase + (int64_t)p * N + n] : 0.f;
        const float* grow = Gcs + (int64_t)bh * Lp;
        float gl_next = grow[Q - 1];  // g_last of the next chunk, loaded one chunk ahead
        for (int c = 0; c < nc; ++c) {
            const float gl = gl_next;
            if (c + 1 < nc) gl_next = grow[(int64_t)(c + 1) * Q + Q - 1];
            if (nok) {
                __nv_bfloat16* hp = hiddens + ((int64_t)bh * nc + c) * P * N + n;
#pragma unroll
                for (int p = 0; p < PP; ++p)
                    if (p < P) hp[(int64_t)p * N] = __float2bfloat16_rn(Sr[p]);
            }
            const float e = exp2f(gl);
            const int acc = c & 1, use = c >> 1;
            mbar_wait(acc_full(acc), use & 1, &g_fps_error, 1u);
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < PP / 16; ++j) {
                uint32_t r[16];
                tmem_ld_x16(lane_addr + acc * PP + 16 * j, r);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 16; ++q) Sr[16 * j + q] = fmaf(e, Sr[16 * j + q], __uint_as_float(r[q]));
            }
            tc_fence_before();
            mbar_arrive(acc_empty(acc));
        }
        if (final_state != nullptr && nok) {
#pragma unroll
            for (int p = 0; p < PP; ++p)
                if (p < P) final_state[sbase + (int64_t)p * N + n] = Sr[p];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

template <int PP>
cudaError_t launch_pp(const Problem& p, const void* x, const void* B, const float* Gcs,
                      const float* dtT, const float* init, void* hid, float* fin,
                      cudaStream_t stream) {
    using Cfg = FpsCfg<PP>;
    CUtensorMap tx, tb;
    const uint64_t xd[4] = {(uint64_t)p.P, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.b};
    const uint64_t xs[3] = {(uint64_t)p.P * 2, (uint64_t)p.H * p.P * 2,
                            (uint64_t)p.L * p.H * p.P * 2};
    const uint64_t bd[4] = {(uint64_t)p.N, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.b};
    const uint64_t bs[3] = {(uint64_t)p.N * 2, (uint64_t)p.G * p.N * 2,
                            (uint64_t)p.L * p.G * p.N * 2};
    const uint32_t box[4] = {64, 1, (uint32_t)kSub, 1};
    if (!encode_tmap_4d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, xd, xs, box,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_4d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, bd, bs, box,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    auto kern = fwd_pass_state_tc<PP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((p.N + 127) / 128), (unsigned)(p.b * p.H));
    kern<<<grid, kThreads, Cfg::kSmem, stream>>>(tx, tb, Gcs, dtT, init, (__nv_bfloat16*)hid, fin,
                                                 (int)p.H, (int)p.P, (int)p.N, (int)p.Q,
                                                 (int)p.nc, (int)p.Lp, (int)p.hpg);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_pass_state_tc(const Problem& p, const void* x, const void* B,
                                     const float* Gcs, const float* dtT, const float* init,
                                     void* hiddens, float* final_state, cudaStream_t stream) {
    if (p.P <= 64) return launch_pp<64>(p, x, B, Gcs, dtT, init, hiddens, final_state, stream);
    return launch_pp<128>(p, x, B, Gcs, dtT, init, hiddens, final_state, stream);
}

unsigned int take_fwd_pass_state_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_fps_error, sizeof(v)) != cudaSuccess) return ~0u;
    cudaMemcpyToSymbol(g_fps_error, &zero, sizeof(zero));
    return v;
}

}  // namespace ssd
