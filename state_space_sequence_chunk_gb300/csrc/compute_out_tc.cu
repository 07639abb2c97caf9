// compute_out_tc.cu -- step 3 of the SSD forward pass on the tcgen05 tensor
// cores (bf16 inputs, fp32 accumulation).
//
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", section "Kernel 3: compute_out" (with "Step 2" and "Step 3"):
// per (batch, chunk, head)
//     Y = 2^{g} o (C h^T) + ((2^{g_i - g_j} [i >= j]) o (C B^T)) (dt o X) + D X
// with the Q x Q matrix kept on chip and the causal mask applied as a select,
// so the overflowing above-diagonal exponentials never reach the output.
//
// GB300 design (what differs from the pages' cuTile kernel):
//  * Persistent CTAs, one per SM.  Work units (batch, chunk, head) are ordered
//    so that the heads sharing one B/C group are adjacent; each CTA takes a
//    contiguous, balanced range of units.  C B^T depends only on (batch,
//    chunk, group), so it is computed once per group on the tensor core and
//    kept in tensor memory as packed bf16, instead of once per head.
//  * Queries are processed in 128-row blocks (the MMA's M).  For block I:
//        acc  = C_I h^T                       (A = C from smem, B = h from smem)
//        acc *= 2^{g_i}                       (row scale, in TMEM, by the SIMT warps)
//        A_I  = (C B^T)_I o 2^{g_i - g_j} o dt_j, j <= i   (built by the SIMT warps
//               directly into TMEM, bf16)
//        acc += A_I X_{0..}                   (A from TMEM, B = X from smem)
//        y    = acc + D x                     (epilogue, stored from registers)
//    Two TMEM slots (block 0 / block 1 of a 256-token chunk, or alternate heads
//    for shorter chunks) let one block's MMAs overlap the other's SIMT work.
//  * x, h, C, B and the per-token g, dt vectors arrive by TMA / bulk copies
//    into a stage ring; B only passes through the ring once per group.
//
// Warp roles (576 threads): 0-7 two builder warpgroups (C B^T conversion,
// decay-weighted operands), 8-15 two epilogue warpgroups (slot 0 / slot 1: row
// scale and y), 16 TMA producer, 17 MMA issuer (and TMEM owner).  A SIMT thread
// owns TMEM lane (query row) 32*(warp%4) + lane; the SIMT warpgroups come first
// so that they start on warpgroup boundaries with no idle warps, which leaves
// 112 registers per thread.
//
// Supported here: bf16, P <= 64, and N <= 128 with Q in {64, 128, 256} or
// N <= 256 with Q in {64, 128} (the state padded to 128 or 256 by the TMA's
// zero fill).
#include <cuda.h>

#include "sm100_ptx.cuh"
#include "ssd_internal.cuh"
#include "tma_host.cuh"

namespace ssd {
namespace {

__device__ unsigned int g_co_error;  // bit 0: a bounded wait gave up

constexpr int kThreads = 576;
constexpr int kRowBytes = 128;
constexpr int kSimtWarp0 = 0;
constexpr int kSimtThreads = 512;   // 16 SIMT warps
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;


// NS = N padded to 128 or 256 (the state dimension, the K of C B^T and C h^T).
// NS = 256 serves Q <= 128 only (one 64 KB C buffer and three stages); its B
// tile (four 64-column atoms) spans two stage slots, atoms 0-1 in the first.
template <int Q, int NS = 128>
struct CoCfg {
    static_assert(NS == 128 || (NS == 256 && Q <= 128), "N = 256 is served for Q <= 128");
    static constexpr int kBlocks = Q > 128 ? 2 : 1;        // 128-row query blocks per chunk
    static constexpr int kBRows = Q < 128 ? Q : 128;        // rows of a key block
    static constexpr int kCRows = Q < 128 ? 128 : Q;        // rows reserved per C atom
    static constexpr int kNAtoms = NS / 64;                 // N in 64-wide swizzle atoms
    static constexpr int kKSteps = NS / 16;                 // K = 16 steps over the state
    static constexpr int kCAtomBytes = kCRows * kRowBytes;
    static constexpr int kCBytes = kNAtoms * kCAtomBytes;
    static constexpr int kCBufs = (Q > 128 || NS > 128) ? 1 : 2;
    static constexpr int kXBytes = Q * kRowBytes;           // x tile, P padded to 64
    static constexpr int kHBytes = NS * kRowBytes;          // h^T: NS rows of N x 64 of P
    static constexpr int kVecBytes = Q * 4;
    static constexpr int kStageBytes = ((kXBytes + kHBytes + 2 * kVecBytes) + 1023) / 1024 * 1024;
    static constexpr int kStages = (Q > 128 || NS > 128) ? 3 : 4;
    static constexpr int kBAtomBytes = kBRows * kRowBytes;
    // B atoms per stage slot: all of them, or two when N = 256 (Q <= 128)
    static constexpr bool kBSplit = NS > 128 && Q <= 128 && kNAtoms * kBAtomBytes > kStageBytes;
    static constexpr int kBSlots = (Q > 128 || kBSplit) ? 2 : 1;   // stage slots a B tile occupies
    static_assert(!kBSplit || 2 * kBAtomBytes <= kStageBytes, "two B atoms per stage slot");
    static constexpr int kBarBytes = 4096;  // barriers, TMEM holder, v_j tables
    static constexpr int kSmem = kCBufs * kCBytes + kStages * kStageBytes + kBarBytes + 1024;
    // TMEM columns (512 allocated)
    // layout, Q = 256: [0,192) CB blocks (0,0) (1,0) (1,1); [192,256) A slot 0;
    //   [256,384) A slot 1; [384,448) acc slot 0; [448,512) acc slot 1;
    //   fp32 scratch for C B^T: [256,384) and [384,512) (only while drained).
    // layout, Q <= 128: [0,64) CB buffer 0; [64,128) CB buffer 1; [128,192) A slot 0;
    //   [192,256) A slot 1; [256,320) acc slot 0; [320,384) acc slot 1; scratch [384,512).
    static constexpr uint32_t kCbBase = 0;
    static constexpr uint32_t kA0 = Q > 128 ? 192 : 128;
    static constexpr uint32_t kA1 = Q > 128 ? 256 : 192;
    static constexpr uint32_t kAcc0 = Q > 128 ? 384 : 256;
    static constexpr uint32_t kAcc1 = Q > 128 ? 448 : 320;
    static constexpr uint32_t kScratch = Q > 128 ? 256 : 384;
};

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t v) {
    return *reinterpret_cast<__nv_bfloat162*>(&v);
}
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) {
    return *reinterpret_cast<uint32_t*>(&v);
}
// One 32-byte store (eight 32-bit words); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
// Barrier among `n` threads (a multiple of 32) on hardware barrier `id` (1..15).
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// The units of a CTA: [u0, u1) of the list ordered (batch, chunk, head).
struct UnitInfo {
    int b, c, h, grp;
};
__device__ __forceinline__ UnitInfo unit_info(int u, int nc, int H, int hpg) {
    UnitInfo r;
    r.h = u % H;
    const int bc = u / H;
    r.c = bc % nc;
    r.b = bc / nc;
    r.grp = r.h / hpg;
    return r;
}
__device__ __forceinline__ bool new_group(int u, int u0, int H, int hpg) {
    return u == u0 || (u % H) % hpg == 0;
}

template <int Q, int NS>
__global__ void __launch_bounds__(kThreads, 1)
compute_out_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_c,
               const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_h,
               const float* __restrict__ Gcs, const float* __restrict__ dtT,
               const float* __restrict__ D, __nv_bfloat16* __restrict__ y, int L, int H, int P,
               int nc, int Lp, int hpg, int units, unsigned int* host_err) {
    using Cfg = CoCfg<Q, NS>;
    constexpr int NST = Cfg::kStages;
    constexpr int NCB = Cfg::kCBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* cbuf_ptr = smem;
    uint8_t* stage_ptr = smem + NCB * Cfg::kCBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage_ptr + NST * Cfg::kStageBytes);
    // barrier map
    uint64_t* b_full = bars;                 // [NST]  stage loaded (tx)
    uint64_t* b_empty = b_full + NST;        // [NST]  stage released (256 SIMT arrivals)
    uint64_t* b_grp = b_empty + NST;         // [NCB]  C + B of a group loaded (tx)
    uint64_t* b_cfree = b_grp + NCB;         // [NCB]  last C h^T of a group done (commit)
    uint64_t* b_cbfull = b_cfree + NCB;      // [2]    C B^T round done (commit)
    uint64_t* b_cbconv = b_cbfull + 2;       // [2]    C B^T round converted (256 arrivals)
    uint64_t* b_sdone = b_cbconv + 2;        // [2]    slot: C h^T done (commit)
    uint64_t* b_ddone = b_sdone + 2;         // [2]    slot: A X done (commit)
    uint64_t* b_aready = b_ddone + 2;        // [2]    slot: A built (128 arrivals)
    uint64_t* b_scaled = b_aready + 2;       // [2]    slot: acc row-scaled (128 arrivals)
    uint64_t* b_accfree = b_scaled + 2;      // [2]    slot: acc read by the epilogue (128)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(b_accfree + 2);
    // per-warpgroup, per-head-parity tables of the column factors v_j (bf16)
    __nv_bfloat16* vtab = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(bars) + 512);
    float* vtabf = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 1536);  // fp32 copy

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u0 = (int)((int64_t)blockIdx.x * units / gridDim.x);
    const int u1 = (int)((int64_t)(blockIdx.x + 1) * units / gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(b_full + s), 1);
            mbar_init(smem_u32(b_empty + s), kSimtThreads);
        }
        for (int s = 0; s < NCB; ++s) {
            mbar_init(smem_u32(b_grp + s), 1);
            mbar_init(smem_u32(b_cfree + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(b_cbfull + s), 1);
            mbar_init(smem_u32(b_cbconv + s), 256);
            mbar_init(smem_u32(b_sdone + s), 1);
            mbar_init(smem_u32(b_ddone + s), 1);
            mbar_init(smem_u32(b_aready + s), (Q > 128 && s == 0) ? 128 : 256);
            mbar_init(smem_u32(b_scaled + s), 128);
            mbar_init(smem_u32(b_accfree + s), 128);
        }
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_holder), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    unsigned int* err = &g_co_error;

    if (warp == kProducerWarp) {
        // ===================== TMA producer =====================
        if (lane == 0) {
            // each chunk-start state is read once: its lines go first in L2
            const uint64_t h_pol = l2_policy_evict_first();
            int sc = 0;   // stage ring counter
            int gi = -1;  // group counter
            for (int u = u0; u < u1; ++u) {
                const UnitInfo ui = unit_info(u, nc, H, hpg);
                if (new_group(u, u0, H, hpg)) {
                    ++gi;
                    const int cb = gi % NCB;
                    // C buffer reuse: the previous group in it has finished its C h^T
                    mbar_wait(smem_u32(b_cfree + cb), ((gi / NCB) & 1) ^ 1, err, 1u);
                    // B passes through kBSlots stage slots
                    int bslot[2];
                    for (int j = 0; j < Cfg::kBSlots; ++j) {
                        const int s = (sc + j) % NST, k = (sc + j) / NST;
                        mbar_wait(smem_u32(b_empty + s), (k & 1) ^ 1, err, 1u);
                        bslot[j] = s;
                    }
                    const uint32_t gbar = smem_u32(b_grp + cb);
                    mbar_arrive_expect_tx(gbar, Cfg::kNAtoms * (Q * kRowBytes) +
                                                    (Cfg::kBSplit ? 1 : Cfg::kBSlots) *
                                                        Cfg::kNAtoms * Cfg::kBAtomBytes);
                    const uint32_t cdst = smem_u32(cbuf_ptr + cb * Cfg::kCBytes);
                    for (int a = 0; a < Cfg::kNAtoms; ++a)
                        tma_load_4d(cdst + a * Cfg::kCAtomBytes, &tm_c, gbar, a * 64, ui.grp,
                                    ui.c * Q, ui.b);
                    for (int j = 0; j < Cfg::kBSlots; ++j) {
                        const uint32_t bdst = smem_u32(stage_ptr + bslot[j] * Cfg::kStageBytes);
                        if (Cfg::kBSplit) {   // atoms 2j, 2j + 1 of the chunk's keys
                            for (int a2 = 0; a2 < 2; ++a2)
                                tma_load_4d(bdst + a2 * Cfg::kBAtomBytes, &tm_b, gbar,
                                            (2 * j + a2) * 64, ui.grp, ui.c * Q, ui.b);
                        } else {              // all atoms of key block j
                            for (int a = 0; a < Cfg::kNAtoms; ++a)
                                tma_load_4d(bdst + a * Cfg::kBAtomBytes, &tm_b, gbar, a * 64, ui.grp,
                                            ui.c * Q + j * 128, ui.b);
                        }
                    }
                    // keep the slots' "full" phases in step with the ring (the B
                    // bytes themselves complete on the group barrier)
                    for (int j = 0; j < Cfg::kBSlots; ++j) mbar_arrive(smem_u32(b_full + bslot[j]));
                    sc += Cfg::kBSlots;
                }
                // head stage: x, h, g, dt.  h, g and dt come from the earlier
                // steps: the first head stage waits for them (the group's C and B,
                // inputs, were requested before)
                if (u == u0) grid_dependency_wait();
                const int s = sc % NST, k = sc / NST;
                mbar_wait(smem_u32(b_empty + s), (k & 1) ^ 1, err, 1u);
                const uint32_t fb = smem_u32(b_full + s);
                uint8_t* st = stage_ptr + s * Cfg::kStageBytes;
                mbar_arrive_expect_tx(fb, Cfg::kXBytes + Cfg::kHBytes + 2 * Cfg::kVecBytes);
                tma_load_4d(smem_u32(st), &tm_x, fb, 0, ui.h, ui.c * Q, ui.b);
                const int bh = ui.b * H + ui.h;
                tma_load_4d_hint(smem_u32(st + Cfg::kXBytes), &tm_h, fb, 0, 0, bh * nc + ui.c, 0,
                                 h_pol);
                const int64_t vo = (int64_t)bh * Lp + (int64_t)ui.c * Q;
                bulk_load(smem_u32(st + Cfg::kXBytes + Cfg::kHBytes), Gcs + vo, Cfg::kVecBytes, fb);
                bulk_load(smem_u32(st + Cfg::kXBytes + Cfg::kHBytes + Cfg::kVecBytes), dtT + vo,
                          Cfg::kVecBytes, fb);
                ++sc;
            }
        }
    } else if (warp == kMmaWarp) {
        // ===================== MMA issuer =====================
        if (lane == 0) {
            constexpr uint32_t kIdescCB = make_idesc(1, 128, Cfg::kBRows, 0, 0);
            constexpr uint32_t kIdescS = make_idesc(1, 128, 64, 0, 1);  // B = h, MN-major
            constexpr uint32_t kIdescD = make_idesc(1, 128, 64, 0, 1);
            int sc = 0, gi = -1, js = 0;  // stage, group, slot-job counters
            int cbq = 0;                  // C buffer of the current group
            for (int u = u0; u < u1; ++u) {
                const bool ng = new_group(u, u0, H, hpg);
                if (ng) {
                    ++gi;
                    cbq = gi % NCB;
                    mbar_wait(smem_u32(b_grp + cbq), (gi / NCB) & 1, err, 1u);
                    if (Q > 128) {
                        // the C B^T scratch overlaps slot memory: drain both slots
                        for (int s2 = 0; s2 < 2; ++s2) {
                            const int uses = (js + 1 - s2) / 2;  // completed uses of slot s2
                            if (uses > 0)
                                mbar_wait(smem_u32(b_accfree + s2), (uses - 1) & 1, err, 1u);
                        }
                    } else {
                        // scratch reuse: the previous group's conversion has read it
                        mbar_wait(smem_u32(b_cbconv), (gi & 1) ^ 1, err, 1u);
                    }
                    tc_fence_after();
                    const uint32_t cbase = smem_u32(cbuf_ptr + cbq * Cfg::kCBytes);
                    // rounds of C B^T blocks (I, J): Q=256: {(0,0),(1,0)} then {(1,1)}
                    const int rounds = Q > 128 ? 2 : 1;
                    for (int r = 0; r < rounds; ++r) {
                        if (r == 1) {
                            mbar_wait(smem_u32(b_cbconv), gi & 1, err, 1u);
                            tc_fence_after();
                        }
                        const int nblk = (Q > 128 && r == 0) ? 2 : 1;
                        for (int q = 0; q < nblk; ++q) {
                            const int I = (Q > 128) ? (r == 0 ? q : 1) : 0;
                            const int J = (Q > 128) ? (r == 0 ? 0 : 1) : 0;
                            const uint32_t bbase =
                                smem_u32(stage_ptr + ((sc + J) % NST) * Cfg::kStageBytes);
                            // with split B, atoms 2 and 3 sit in the next stage slot
                            const uint32_t bbase1 =
                                smem_u32(stage_ptr + ((sc + 1) % NST) * Cfg::kStageBytes);
                            const uint32_t dcol = tmem + Cfg::kScratch + q * 128;
                            const uint64_t ad0 = smem_desc_sw128(cbase + I * 128 * kRowBytes, 16, 8 * kRowBytes);
#pragma unroll
                            for (int kk = 0; kk < Cfg::kKSteps; ++kk) {  // K = the state columns
                                const int atom = kk / 4;
                                const uint32_t batom =
                                    Cfg::kBSplit ? (atom < 2 ? bbase + atom * Cfg::kBAtomBytes
                                                             : bbase1 + (atom - 2) * Cfg::kBAtomBytes)
                                                 : bbase + atom * Cfg::kBAtomBytes;
                                mma_f16_ss(dcol,
                                           ad0 + (uint64_t)((atom * Cfg::kCAtomBytes + (kk % 4) * 32) >> 4),
                                           smem_desc_sw128(batom + (kk % 4) * 32, 16, 8 * kRowBytes),
                                           kIdescCB, kk > 0 ? 1u : 0u);
                            }
                        }
                        mma_commit(smem_u32(b_cbfull + r));
                    }
                    sc += Cfg::kBSlots;
                }
                const int s = sc % NST, k = sc / NST;
                mbar_wait(smem_u32(b_full + s), k & 1, err, 1u);
                tc_fence_after();
                const uint32_t st = smem_u32(stage_ptr + s * Cfg::kStageBytes);
                const uint32_t cbase = smem_u32(cbuf_ptr + cbq * Cfg::kCBytes);
                // acc = C_I h^T for each block of this head
                for (int I = 0; I < Cfg::kBlocks; ++I) {
                    const int slot = (js + I) & 1, use = (js + I) >> 1;
                    mbar_wait(smem_u32(b_accfree + slot), (use & 1) ^ 1, err, 1u);
                    tc_fence_after();
                    const uint32_t acc = tmem + (slot ? Cfg::kAcc1 : Cfg::kAcc0);
                    // descriptors built once; the K steps add compile-time offsets to
                    // the start-address field (addr >> 4, no carry below 256 KB)
                    const uint64_t ad0 = smem_desc_sw128(cbase + I * 128 * kRowBytes, 16, 8 * kRowBytes);
                    // B = h^T tile [n][p]: MN-major (p contiguous), K = 16 state rows
                    const uint64_t bd0 = smem_desc_sw128(st + Cfg::kXBytes, 8 * kRowBytes, 8 * kRowBytes);
#pragma unroll
                    for (int kk = 0; kk < Cfg::kKSteps; ++kk)
                        mma_f16_ss(acc, ad0 + (uint64_t)(((kk / 4) * Cfg::kCAtomBytes + (kk % 4) * 32) >> 4),
                                   bd0 + (uint64_t)((kk * 16 * kRowBytes) >> 4), kIdescS, kk > 0 ? 1u : 0u);
                    mma_commit(smem_u32(b_sdone + slot));
                }
                // the C buffer is free once the group's last C h^T is done
                if (u + 1 == u1 || new_group(u + 1, u0, H, hpg)) mma_commit(smem_u32(b_cfree + cbq));
                // acc += A_I X
                for (int I = 0; I < Cfg::kBlocks; ++I) {
                    const int slot = (js + I) & 1, use = (js + I) >> 1;
                    mbar_wait(smem_u32(b_aready + slot), use & 1, err, 1u);
                    mbar_wait(smem_u32(b_scaled + slot), use & 1, err, 1u);
                    tc_fence_after();
                    const uint32_t acc = tmem + (slot ? Cfg::kAcc1 : Cfg::kAcc0);
                    const uint32_t abase = tmem + (slot ? Cfg::kA1 : Cfg::kA0);
                    const int ksteps = (Q > 128 ? (I + 1) * 128 : Q) / 16;
                    const uint64_t bd0 = smem_desc_sw128(st, 8 * kRowBytes, 8 * kRowBytes);
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)
                        if (kk < ksteps)
                            mma_f16_ts(acc, abase + kk * 8, bd0 + (uint64_t)((kk * 16 * kRowBytes) >> 4),
                                       kIdescD, 1u);
                    mma_commit(smem_u32(b_ddone + slot));
                }
                js += Cfg::kBlocks;
                ++sc;
            }
        }
    } else {
        // ===================== SIMT warpgroups =====================
        // Warpgroups 0 and 1 are builders: they convert C B^T once per group and
        // build the decay-weighted operands A of every head.  Warpgroups 2 and 3
        // serve TMEM slots 0 and 1: the 2^{g_i} row scale of the accumulator and
        // the y epilogue.  The builders of head h+1 thus run while the epilogue
        // of head h drains; only the MMA that reads an operand region orders them.
        const int w = (warp - kSimtWarp0) >> 2;          // 0..3
        const bool builder = w < 2;
        const int sel = w & 1;
        const int row = (warp & 3) * 32 + lane;          // TMEM lane / query row in block
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        int sc = 0, gi = -1, js = 0;
        for (int u = u0; u < u1; ++u) {
            __syncwarp();  // the previous unit's per-row stores may have diverged
            const UnitInfo ui = unit_info(u, nc, H, hpg);
            if (new_group(u, u0, H, hpg)) {
                ++gi;
                const int rounds = Q > 128 ? 2 : 1;
                if (builder) {
                    // convert C B^T (fp32 scratch) to packed bf16
                    const uint32_t cbdst = Q > 128 ? Cfg::kCbBase : Cfg::kCbBase + (gi & 1) * 64;
                    for (int r = 0; r < rounds; ++r) {
                        mbar_wait(smem_u32(b_cbfull + r), gi & 1, err, 1u);
                        tc_fence_after();
                        // round 0 of Q=256: builder 0 converts block (0,0), builder 1
                        // block (1,0); otherwise each takes half of the block's columns
                        int q, c0, ncol, dcol;
                        if (Q > 128 && r == 0) {
                            q = sel; c0 = 0; ncol = 128; dcol = sel * 64;
                        } else {
                            q = 0; ncol = Cfg::kBRows / 2; c0 = sel * ncol;
                            dcol = (Q > 128 ? 128 : 0) + c0 / 2;
                        }
                        for (int cc = 0; cc < ncol; cc += 32) {
                            __syncwarp();
                            uint32_t v[32], o[16];
                            tmem_ld_x32(tmem + lane_off + Cfg::kScratch + q * 128 + c0 + cc, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                o[e] = pack_bf16(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                            tmem_st_x16(tmem + lane_off + cbdst + dcol + cc / 2, o);
                        }
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(smem_u32(b_cbconv + r));
                    }
                    // both builders read the whole packed C B^T
                    mbar_wait(smem_u32(b_cbconv + (rounds - 1)), gi & 1, err, 1u);
                    tc_fence_after();
                }
                // release the stage slots that carried B
                for (int j = 0; j < Cfg::kBSlots; ++j) mbar_arrive(smem_u32(b_empty + (sc + j) % NST));
                sc += Cfg::kBSlots;
            }
            const int s = sc % NST, k = sc / NST;
            const float dh = (!builder && D) ? __ldg(D + ui.h) : 0.f;  // issued early
            mbar_wait(smem_u32(b_full + s), k & 1, err, 1u);
            const uint8_t* st = stage_ptr + s * Cfg::kStageBytes;
            const float* gv = reinterpret_cast<const float*>(st + Cfg::kXBytes + Cfg::kHBytes);
            const float* dv = gv + Q;
            const int use = js >> 1;   // use count of the slot(s) this head occupies
            if (builder) {
                const uint32_t cbsrc = Q > 128 ? Cfg::kCbBase : Cfg::kCbBase + (gi & 1) * 64;
                // ---- column factors v_j = 2^{g_e - g_j} dt_j (e = end of j's 32-key
                //      chunk) for every key of the chunk, shared by both builders ----
                // double-buffered by head parity: a builder may still read the
                // previous head's table while the other writes this one
                __nv_bfloat16* vb = vtab + ((js / Cfg::kBlocks) & 1) * 256;
                float* vf = vtabf + ((js / Cfg::kBlocks) & 1) * 256;
                {
                    const int j = sel * 128 + row;
                    if (j < Q) {
                        const float vj = exp2f(gv[j | 31] - gv[j]) * dv[j];
                        vb[j] = __float2bfloat16_rn(vj);
                        vf[j] = vj;
                    }
                }
                named_bar_sync(1, 256);
                const uint32_t* vb32 = reinterpret_cast<const uint32_t*>(vb);
                // ---- build A for query block I, keys [kb, ke), 32 keys at a time ----
                auto build = [&](int I, int kb, int ke, int slot) {
                    const int i = I * 128 + row;               // query row in the chunk
                    const float gi_ = (i < Q) ? gv[i] : 0.f;
                    const int dch = i >> 5;   // key chunk holding the diagonal (warp-uniform)
                    const uint32_t abase = tmem + lane_off + (slot ? Cfg::kA1 : Cfg::kA0);
                    for (int j0 = kb; j0 < ke; j0 += 32) {
                        __syncwarp();  // warp-collective TMEM access below
                        const int kc = j0 >> 5;
                        uint32_t o[16];
                        if (kc > dch) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) o[e] = 0u;
                        } else {
                            const int J = j0 >> 7, jl0 = j0 & 127;
                            const uint32_t blk = Q > 128 ? (I == 0 ? 0u : (J == 0 ? 64u : 128u)) : 0u;
                            uint32_t cbv[16];
                            tmem_ld_x16(tmem + lane_off + cbsrc + blk + jl0 / 2, cbv);
                            tmem_wait_ld();
                            // Factorised decay 2^{g_i - g_j} = 2^{g_i - g_e} 2^{g_e - g_j} with
                            // e the chunk's last key: below the diagonal chunk both factors
                            // are <= 1.  On the diagonal chunk the row factor may exceed 1
                            // (by at most the chunk's decay span), so the factorised form is
                            // used there only when that span is small enough to stay far from
                            // overflow; the entries above the diagonal are dropped by a
                            // select.  Otherwise the exact per-element exponent is used.
                            const float span = gv[j0] - gv[j0 + 31];   // >= 0, warp-uniform
                            const float uu = exp2f(gi_ - gv[j0 + 31]);
                            if (kc < dch) {
                                const __nv_bfloat162 u2 = __floats2bfloat162_rn(uu, uu);
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    const __nv_bfloat162 c2 = as_bf162(cbv[e]);
                                    const __nv_bfloat162 v2 = as_bf162(vb32[j0 / 2 + e]);
                                    o[e] = as_u32(__hmul2(__hmul2(c2, v2), u2));
                                }
                            } else if (span < 64.f) {
                                // diagonal chunk, moderate decay span: the same factors in
                                // fp32 (one rounding, as for the exact form), masked by a select
                                const float4* vq = reinterpret_cast<const float4*>(vf + j0);
#pragma unroll
                                for (int e4 = 0; e4 < 8; ++e4) {
                                    const float4 vv = vq[e4];
                                    const int ja = j0 + 4 * e4;
                                    const uint32_t c01 = cbv[2 * e4], c23 = cbv[2 * e4 + 1];
                                    const float a0 = (ja <= i) ? bf16lo(c01) * (vv.x * uu) : 0.f;
                                    const float a1 = (ja + 1 <= i) ? bf16hi(c01) * (vv.y * uu) : 0.f;
                                    const float a2 = (ja + 2 <= i) ? bf16lo(c23) * (vv.z * uu) : 0.f;
                                    const float a3 = (ja + 3 <= i) ? bf16hi(c23) * (vv.w * uu) : 0.f;
                                    o[2 * e4] = pack_bf16(a0, a1);
                                    o[2 * e4 + 1] = pack_bf16(a2, a3);
                                }
                            } else {
                                // diagonal chunk with a large decay span: exact exponent,
                                // masked by a select
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    const int ja = j0 + 2 * e, jc = ja + 1;
                                    const float wa = exp2f(gi_ - gv[ja]) * dv[ja];
                                    const float wc = exp2f(gi_ - gv[jc]) * dv[jc];
                                    const float va = (ja <= i) ? bf16lo(cbv[e]) * wa : 0.f;
                                    const float vc = (jc <= i) ? bf16hi(cbv[e]) * wc : 0.f;
                                    o[e] = pack_bf16(va, vc);
                                }
                            }
                        }
                        tmem_st_x16(abase + j0 / 2, o);
                    }
                    __syncwarp();
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(smem_u32(b_aready + slot));
                };
                // the previous A X product on a slot must be done before its A is rewritten
                auto a_free = [&](int slot) {
                    if (use > 0) mbar_wait(smem_u32(b_ddone + slot), (use - 1) & 1, err, 1u);
                    tc_fence_after();
                };
                if (Q > 128) {
                    // block 0: keys [0,128); block 1: keys [0,256); split for balance
                    if (sel == 0) {
                        a_free(0);
                        build(0, 0, 128, 0);
                        a_free(1);
                        build(1, 0, 64, 1);
                    } else {
                        a_free(1);
                        build(1, 64, 256, 1);
                    }
                } else {
                    const int slot = js & 1;
                    a_free(slot);
                    build(0, sel * (Q / 2), (sel + 1) * (Q / 2), slot);
                }
            } else {
                const int es = sel;    // this warpgroup's TMEM slot
                const int I = Q > 128 ? es : (((js & 1) == es) ? 0 : -1);
                if (I >= 0) {
                    const int i = I * 128 + row;
                    const uint32_t acc = tmem + lane_off + (es ? Cfg::kAcc1 : Cfg::kAcc0);
                    // ---- acc *= 2^{g_i} ----
                    mbar_wait(smem_u32(b_sdone + es), use & 1, err, 1u);
                    tc_fence_after();
                    {
                        const float sg = exp2f((i < Q) ? gv[i] : 0.f);
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            uint32_t v[32];
                            __syncwarp();
                            tmem_ld_x32(acc + h2 * 32, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * sg);
                            tmem_st_x32(acc + h2 * 32, v);
                        }
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    mbar_arrive(smem_u32(b_scaled + es));
                    // ---- epilogue: y = acc + D x ----
                    mbar_wait(smem_u32(b_ddone + es), use & 1, err, 1u);
                    tc_fence_after();
                    // the A X products are done: this row of x (for D x) is the
                    // last thing this warpgroup reads from the stage, which then
                    // goes back to the producer before y is computed and stored
                    uint4 xrow[8];
                    {
                        const uint8_t* xr = st + (i < Q ? i : 0) * kRowBytes;
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch)
                            xrow[ch] = *reinterpret_cast<const uint4*>(xr + ((ch ^ (i & 7)) << 4));
                    }
                    // The row's values are first used after the release, and the
                    // stage is refilled by the TMA (the async proxy): without this
                    // fence the loads could still be outstanding when the next unit's
                    // x lands in the stage (seen as the next unit's x in D x for the
                    // last head of a group, Q = 256, a few calls in a hundred)
                    fence_proxy_async_smem();
                    mbar_arrive(smem_u32(b_empty + s));
                    // y = acc + D x, 32 columns at a time, stored straight from
                    // registers: each thread writes its own row (128 contiguous
                    // bytes); 32-byte stores where the row is 32-byte aligned
                    const int t = ui.c * Q + i;   // token
                    const bool store = i < Q && t < L;
                    __nv_bfloat16* yr = y + (((int64_t)ui.b * L + (store ? t : 0)) * H + ui.h) * P;
                    const bool a32 = (reinterpret_cast<uintptr_t>(yr) & 31) == 0;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[32];
                        __syncwarp();
                        tmem_ld_x32(acc + half * 32, v);
                        tmem_wait_ld();
                        if (half == 1) {
                            tc_fence_before();
                            mbar_arrive(smem_u32(b_accfree + es));
                        }
#pragma unroll
                        for (int c2 = 2 * half; c2 < 2 * half + 2; ++c2) {
                            if (store && c2 * 16 < P) {   // P is a multiple of 16
                                uint32_t ow[8];
#pragma unroll
                                for (int hh = 0; hh < 2; ++hh) {
                                    const int ch = 2 * c2 + hh;
                                    const uint4 xv = xrow[ch];
                                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int p0 = (ch * 8 + 2 * e) & 31;
                                        ow[4 * hh + e] =
                                            pack_bf16(__uint_as_float(v[p0]) + dh * bf16lo(xw[e]),
                                                      __uint_as_float(v[p0 + 1]) + dh * bf16hi(xw[e]));
                                    }
                                }
                                __nv_bfloat16* dst = yr + c2 * 16;
                                if (a32) {
                                    st_global_v8(dst, ow);
                                } else {
                                    reinterpret_cast<uint4*>(dst)[0] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                                    reinterpret_cast<uint4*>(dst)[1] = make_uint4(ow[4], ow[5], ow[6], ow[7]);
                                }
                            }
                        }
                    }
                } else {
                    mbar_arrive(smem_u32(b_empty + s));   // no block of this head here
                }
            }
            if (builder) mbar_arrive(smem_u32(b_empty + s));
            js += Cfg::kBlocks;
            ++sc;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) report_timeout_to_host(err, host_err);
    if (warp == kMmaWarp) {
        __syncwarp();  // lane 0 ran the MMA loop alone: reconverge before the collective
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int Q, int NS>
cudaError_t launch_q(const Problem& p, const void* x, const void* B, const void* C,
                     const float* Gcs, const float* dtT, const void* hid, const float* D, void* y,
                     cudaStream_t stream) {
    using Cfg = CoCfg<Q, NS>;
    CUtensorMap tx, tc, tb, th;
    const uint64_t xd[4] = {(uint64_t)p.P, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.b};
    const uint64_t xs[3] = {(uint64_t)p.P * 2, (uint64_t)p.H * p.P * 2,
                            (uint64_t)p.L * p.H * p.P * 2};
    const uint64_t bd[4] = {(uint64_t)p.N, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.b};
    const uint64_t bs[3] = {(uint64_t)p.N * 2, (uint64_t)p.G * p.N * 2,
                            (uint64_t)p.L * p.G * p.N * 2};
    const uint64_t hd[4] = {(uint64_t)p.P, (uint64_t)p.N, (uint64_t)(p.b * p.H * p.nc), 1};
    const uint64_t hs[3] = {(uint64_t)p.P * 2, (uint64_t)p.N * p.P * 2,
                            (uint64_t)(p.b * p.H * p.nc) * p.N * p.P * 2};
    const uint32_t box_x[4] = {64, 1, (uint32_t)Q, 1};
    const uint32_t box_b[4] = {64, 1, (uint32_t)Cfg::kBRows, 1};
    const uint32_t box_h[4] = {64, (uint32_t)NS, 1, 1};
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (!encode_tmap_4d(&tx, bf, x, xd, xs, box_x, sw) ||
        !encode_tmap_4d(&tc, bf, C, bd, bs, box_x, sw) ||
        !encode_tmap_4d(&tb, bf, B, bd, bs, box_b, sw) ||
        !encode_tmap_4d(&th, bf, hid, hd, hs, box_h, sw))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    auto kern = compute_out_tc<Q, NS>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t units = p.b * p.nc * p.H;
    const int grid = (int)(units < sms ? units : sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)Cfg::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.chained ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, tx, tc, tb, th, Gcs, dtT, D, (__nv_bfloat16*)y, (int)p.L,
                           (int)p.H, (int)p.P, (int)p.nc, (int)p.Lp, (int)p.hpg, (int)units,
                           host_timeout_word());
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool compute_out_tc_supports(const Problem& p) {
    return p.dtype == SSD_BF16 && p.P <= 64 && (p.N <= 128 || (p.N <= 256 && p.Q <= 128)) &&
           p.b * p.nc * p.H < (1LL << 31);
}

cudaError_t launch_compute_out_tc(const Problem& p, const void* x, const void* B, const void* C,
                                  const float* Gcs, const float* dtT, const void* hiddens,
                                  const float* D, void* y, cudaStream_t stream) {
    if (p.N > 128) {   // Q <= 128 (compute_out_tc_supports)
        return p.Q == 64 ? launch_q<64, 256>(p, x, B, C, Gcs, dtT, hiddens, D, y, stream)
                         : launch_q<128, 256>(p, x, B, C, Gcs, dtT, hiddens, D, y, stream);
    }
    switch (p.Q) {
        case 64: return launch_q<64, 128>(p, x, B, C, Gcs, dtT, hiddens, D, y, stream);
        case 128: return launch_q<128, 128>(p, x, B, C, Gcs, dtT, hiddens, D, y, stream);
        default: return launch_q<256, 128>(p, x, B, C, Gcs, dtT, hiddens, D, y, stream);
    }
}

unsigned int take_compute_out_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_co_error, sizeof(v)) != cudaSuccess) return ~0u;
    cudaMemcpyToSymbol(g_co_error, &zero, sizeof(zero));
    return v;
}

}  // namespace ssd
