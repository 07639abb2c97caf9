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
//    accumulator, and the epilogue warps fold it into the running state kept
//    in a second TMEM region, S <- 2^{g_last} S + D_c.  The tensor core never
//    waits for the previous chunk's state, only for the epilogue to have read
//    the accumulator; keeping S in TMEM keeps registers low enough for four
//    CTAs per SM, so that a full batch*head grid is resident at once.
//  * x and B stream in 32-token sub-chunks through a multi-stage TMA ring
//    (128-byte swizzle, token-major rows, read as MN-major operands).  The
//    per-token scale s_q = dt_q 2^{g_last - g_q} is applied to the x rows in
//    shared memory (a row is contiguous in the swizzled tile).
//
// Warp roles (320 threads): 0 TMA producer, 1 MMA issuer (and TMEM owner),
// 2..5 row scalers, 6..9 state warps (the state update at each chunk
// boundary; TMEM lane quarter = warp % 4).  TMEM: columns
// [0, PP) accumulator, [PP, 2 PP) state S^T (lane = state row n, column = p).
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

constexpr int kSub = 32;            // tokens per pipeline stage
constexpr int kRowBytes = 128;      // one swizzle row (64 bf16)
constexpr int kScalerWarps = 4;
constexpr int kThreads = 32 * (2 + kScalerWarps + 4);

template <int PP>
struct FpsCfg {
    static constexpr int kStages = 5;
    static constexpr int kMinBlocks = PP == 64 ? 3 : 2;   // CTAs per SM (TMEM: 2*PP each)
    static constexpr int kXBytes = kSub * PP * 2;         // x sub-tile
    static constexpr int kBBytes = kSub * 128 * 2;        // B sub-tile (128 state rows)
    static constexpr int kVecOff = kXBytes + kBBytes;     // g[kSub], dt[kSub], last 4 g of the chunk
    static constexpr int kVecBytes = 2 * kSub * 4 + 16;
    static constexpr int kStageBytes = (kVecOff + kVecBytes + 1023) / 1024 * 1024;
    static constexpr int kTmemCols = 2 * PP;              // accumulator + state
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
__global__ void __launch_bounds__(kThreads, FpsCfg<PP>::kMinBlocks)
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
    const uint32_t acc_full = smem_u32(bars + 3 * S);
    const uint32_t acc_empty = smem_u32(bars + 3 * S + 1);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * S + 2);

    const int mb = blockIdx.x, bh = blockIdx.y;
    const int b = bh / H, h = bh % H, grp = h / hpg;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsub = Q / kSub;
    const int total = nc * nsub;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(scaled(s), 32 * kScalerWarps);
            mbar_init(empty(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 128);
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
                // the epilogue has read the previous chunk's product
                if (sub == 0) mbar_wait(acc_empty, (c & 1) ^ 1, &g_fps_error, 1u);
                mbar_wait(scaled(s), k & 1, &g_fps_error, 1u);
                tc_fence_after();
                const uint32_t xs = stage0 + s * Cfg::kStageBytes, bs = xs + Cfg::kXBytes;
                // A = B_c^T: M = 128 state rows (two 64-row swizzle atoms, kSub*128
                // bytes apart), K = 16 tokens, MN-major.  B = s o X_c: N = PP columns
                // of P, K = 16 tokens, MN-major.  Descriptors are built once; a K
                // step adds a compile-time offset to the start-address field.
                const uint64_t ad0 = smem_desc_sw128(bs, kSub * kRowBytes, 8 * kRowBytes);
                const uint64_t bd0 = smem_desc_sw128(xs, kSub * kRowBytes, 8 * kRowBytes);
#pragma unroll
                for (int kk = 0; kk < kSub / 16; ++kk)
                    mma_f16_ss(tmem, ad0 + (uint64_t)((kk * 16 * kRowBytes) >> 4),
                               bd0 + (uint64_t)((kk * 16 * kRowBytes) >> 4), Cfg::kIdesc,
                               (sub > 0 || kk > 0) ? 1u : 0u);
                mma_commit(empty(s));
                if (sub == nsub - 1) mma_commit(acc_full);
            }
        }
    } else if (warp < 2 + kScalerWarps) {
        // ---------------- scaler warps: x_q <- x_q * dt_q 2^{g_last - g_q} ----------------
        const int tid = threadIdx.x - 64;
        for (int i = 0; i < total; ++i) {
            const int s = i % S, k = i / S;
            mbar_wait(full(s), k & 1, &g_fps_error, 1u);
            uint8_t* xs = smem + s * Cfg::kStageBytes;
            const float* gv = reinterpret_cast<const float*>(xs + Cfg::kVecOff);
            const float* dv = gv + kSub;
            const float glast = gv[2 * kSub + 3];
            constexpr int kVecs = kSub * (PP / 64) * 8;   // 16-byte vectors in the x sub-tile
#pragma unroll
            for (int v = tid; v < kVecs; v += 32 * kScalerWarps) {
                const int box = v / (kSub * 8), r = (v / 8) % kSub, q = v % 8;
                // fp32 products, one rounding to bf16 (as the pages' cast of the
                // scaled operand)
                const float sc = dv[r] * exp2f(glast - gv[r]);
                uint4* ptr = reinterpret_cast<uint4*>(xs + box * kSub * kRowBytes + r * kRowBytes) + q;
                uint4 w = *ptr;
                w.x = pack_bf16(bf16lo(w.x) * sc, bf16hi(w.x) * sc);
                w.y = pack_bf16(bf16lo(w.y) * sc, bf16hi(w.y) * sc);
                w.z = pack_bf16(bf16lo(w.z) * sc, bf16hi(w.z) * sc);
                w.w = pack_bf16(bf16lo(w.w) * sc, bf16hi(w.w) * sc);
                *ptr = w;
            }
            fence_proxy_async_smem();
            mbar_arrive(scaled(s));
        }
    } else {
        // ---------------- state warps (the last four): the state update ----------------
        // Each thread owns TMEM lane (state row n) 32*(warp%4) + lane and, at each
        // chunk boundary, folds the finished chunk product into S.
        const int quarter = warp & 3;
        const int n = mb * 128 + quarter * 32 + lane;
        const bool nok = n < N;
        const uint32_t acc_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t st_addr = acc_addr + PP;
        const int64_t sbase = (int64_t)bh * P * N;
        // S^T row n <- init_state[b, h, :, n] (or 0)
#pragma unroll
        for (int j = 0; j < PP / 16; ++j) {
            __syncwarp();
            uint32_t r[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int p = 16 * j + q;
                r[q] = __float_as_uint((init != nullptr && nok && p < P)
                                           ? init[sbase + (int64_t)p * N + n] : 0.f);
            }
            tmem_st_x16(st_addr + 16 * j, r);
        }
        tmem_wait_st();
        // S <- 2^{g_last(c)} S + D_c, storing the chunk-start S^T to hiddens[c]
        auto chunk_update = [&](int c, float gl) {
            const float e = exp2f(gl);
            // hiddens[b, h, c] is stored transposed: row n holds S[:, n] (P values)
            __nv_bfloat16* hp = hiddens + (((int64_t)bh * nc + c) * N + n) * P;
            mbar_wait(acc_full, c & 1, &g_fps_error, 1u);
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < PP / 16; ++j) {
                // tcgen05.ld/st are warp-collective: every lane runs them, and the
                // warp is reconverged after the per-lane stores below
                __syncwarp();
                uint32_t d[16], sv[16];
                tmem_ld_x16(acc_addr + 16 * j, d);
                tmem_ld_x16(st_addr + 16 * j, sv);
                tmem_wait_ld();
                uint32_t nw[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    nw[q] = __float_as_uint(fmaf(e, __uint_as_float(sv[q]), __uint_as_float(d[q])));
                tmem_st_x16(st_addr + 16 * j, nw);
                // chunk-start state (before this chunk's update) -> hiddens[c]:
                // 16 contiguous bf16 of row n per slice (P is a multiple of 16)
                if (nok && 16 * j < P) {
                    uint4 w0, w1;
                    w0.x = pack_bf16(__uint_as_float(sv[0]), __uint_as_float(sv[1]));
                    w0.y = pack_bf16(__uint_as_float(sv[2]), __uint_as_float(sv[3]));
                    w0.z = pack_bf16(__uint_as_float(sv[4]), __uint_as_float(sv[5]));
                    w0.w = pack_bf16(__uint_as_float(sv[6]), __uint_as_float(sv[7]));
                    w1.x = pack_bf16(__uint_as_float(sv[8]), __uint_as_float(sv[9]));
                    w1.y = pack_bf16(__uint_as_float(sv[10]), __uint_as_float(sv[11]));
                    w1.z = pack_bf16(__uint_as_float(sv[12]), __uint_as_float(sv[13]));
                    w1.w = pack_bf16(__uint_as_float(sv[14]), __uint_as_float(sv[15]));
                    uint4* dst = reinterpret_cast<uint4*>(hp + 16 * j);
                    dst[0] = w0;
                    dst[1] = w1;
                }
            }
            __syncwarp();
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(acc_empty);
        };
        const float* gl_src = Gcs + (int64_t)bh * Lp + Q - 1;   // g_last of each chunk
        float gl_next = gl_src[0];
        for (int c = 0; c < nc; ++c) {
            const float gl = gl_next;
            if (c + 1 < nc) gl_next = gl_src[(int64_t)(c + 1) * Q];
            chunk_update(c, gl);
        }
        if (final_state != nullptr) {  // uniform: all lanes load, valid lanes store
#pragma unroll
            for (int j = 0; j < PP / 16; ++j) {
                __syncwarp();
                uint32_t sv[16];
                tmem_ld_x16(st_addr + 16 * j, sv);
                tmem_wait_ld();
                if (nok) {
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (16 * j + q < P)
                            final_state[sbase + (int64_t)(16 * j + q) * N + n] = __uint_as_float(sv[q]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();  // lane 0 ran the MMA loop alone: reconverge before the collective
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
