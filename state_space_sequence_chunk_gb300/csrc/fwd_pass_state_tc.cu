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
//  * A chain is the state block that one CTA carries: (batch, head, 128-row
//    block of N, 64-column block of P).  Its chunks are walked in order.  So
//    that every SM gets the same work whatever the number of chains (batch *
//    head rarely divides evenly over 152 SMs), the chains x chunks work units,
//    laid out chain after chain, are cut into one equal contiguous range per
//    resident CTA.  A range holds the tail of one chain, whole chains and the
//    head of another.  A CTA walks its head piece first and publishes the
//    state at its end (fp32, in a two-slot buffer per chain kept in L2), then
//    its whole chains, then its tail piece, which starts from the state that
//    the previous range's CTA published.  Ranges are longer than chains
//    whenever there is more work than CTAs per chain, so that state is ready
//    long before it is needed; every wait is bounded anyway, and ranges are
//    handed out in dispatch order, so a waited-for CTA is always running.
//  * The chunk products D_c = B_c^T (s o X_c) need no state, so the tensor core
//    runs ahead through three TMEM accumulators while the fold warps apply
//    hiddens[c] = S, S <- 2^{g_last} S + D_c, with S in a fourth TMEM slot.
//  * x and B stream in 64-token sub-chunks through a 4-stage TMA ring
//    (128-byte swizzle, token-major rows, read as MN-major operands); g and dt
//    of a chunk arrive once per chunk in a separate two-slot ring.  Few, large
//    copies matter: the TMA issue cost per copy, not the bytes, bounded the
//    rate of smaller stages.  The per-token scale s_q = dt_q 2^{g_last - g_q}
//    is applied to the x rows in shared memory (a row is contiguous in the
//    swizzled tile).
//
// Warp roles (384 threads, two CTAs per SM): 0 TMA producer, 1 MMA issuer (and
// TMEM owner), 2..7 row scalers, 8..11 fold warps (TMEM lane quarter =
// warp % 4).  TMEM: three accumulator slots and the state, 64 columns each.
//
// N and P are padded to the 64-element swizzle atom by the TMA's zero fill;
// padded rows/columns are computed and never stored.
#include <cuda.h>

#include <string.h>

#include <algorithm>

#include "sm100_ptx.cuh"
#include "ssd_internal.cuh"
#include "tma_host.cuh"

namespace ssd {
namespace {

__device__ unsigned int g_fps_error;  // bit 0: a bounded wait gave up
// Test hook (ssd_debug_withhold_handoffs): nonzero makes every range skip
// publishing its end state, so that the receiving ranges' bounded waits run out.
__device__ unsigned int g_fps_withhold;

constexpr int kSub = 64;            // tokens per pipeline stage
constexpr int kRowBytes = 128;      // one swizzle row (64 bf16)
constexpr int kCols = 64;           // state columns (of P) per chain
constexpr int kScalerWarps = 6;
constexpr int kFoldWarps = 4;
constexpr int kThreads = 32 * (2 + kScalerWarps + kFoldWarps);
// TMEM (256 columns): chunk-product accumulators and running-state slots of
// 64 columns each -- three accumulators and one state, or, with an init
// state, two and two (the next chain's initial state waits in the spare slot).
constexpr int kMaxAccSlots = 3;
template <bool kHasInit> __host__ __device__ constexpr int acc_slots() { return kHasInit ? 2 : 3; }
// TMA ring depth: four stages, or three when a 32 KB init-state tile shares
// the shared memory.
// kTmaH (P a multiple of 64, no init tile): the chunk-start states leave
// through a 16 KB shared tile and TMA tensor stores, which takes one stage.
template <bool kHasInit, bool kTmaH = false> __host__ __device__ constexpr int stages() {
    return (kHasInit || kTmaH) ? 3 : 4;
}
constexpr int kVecSlots = 2;        // per-chunk g / dt buffers
constexpr int kMinBlocks = 2;       // CTAs per SM
// Register cap: two 384-thread CTAs per SM stay below the register file's
// limit (per SM sub-partition, three warps of each CTA).
constexpr int kMaxRegs = 80;
constexpr int kXBytes = kSub * kCols * 2;          // x sub-tile
constexpr int kBBytes = kSub * 128 * 2;            // B sub-tile (128 state rows)
constexpr int kStageBytes = kXBytes + kBBytes;     // multiple of 1024
constexpr int kMaxQ = 256;
constexpr int kVecSlotBytes = 2 * kMaxQ * 4;       // g[Q], dt[Q] of one chunk
constexpr int kTmemCols = 256;
constexpr int kBarBytes = 512;
// state tile in shared memory (init in, final out): fp32 [64 p][128 n]
constexpr int kInitBytes = kCols * 128 * 4;
constexpr int kHTileBytes = 128 * kRowBytes;      // chunk-start state tile: 128 rows of 64 p
template <bool kHasInit, bool kTmaH = false>
__host__ __device__ constexpr int smem_bytes() {
    return stages<kHasInit, kTmaH>() * kStageBytes + (kHasInit ? kInitBytes : 0) +
           (kTmaH ? kHTileBytes : 0) + kVecSlots * kVecSlotBytes + kBarBytes + 1024;
}
constexpr uint32_t kIdesc = make_idesc(1, 128, kCols, 1, 1);
constexpr int kSlotFloats = 128 * kCols;           // one state slot of the hand-off buffer
static_assert(kStageBytes % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");

struct FpsParams {
    int H, P, N, Q, nc, Lp, hpg;
    int nmb, npb, nchains;   // row blocks of N, column blocks of P, chains
    int W;                   // work units: nchains * nc (< 2^31, checked on the host)
    int G;                   // CTAs (ranges)
    unsigned int* host_err;  // page-locked host word raised when a wait gave up (may be NULL)
};

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}

// The work range of range index k and the order of its pieces.  Units are
// numbered chain * nc + chunk; range k is [k W / G, (k+1) W / G).
struct Range {
    int lo, hi;
    int ch_first, ch_last;
    bool first_is_tail;   // the first chain's piece starts mid-chain (waits for a state)
    bool last_is_head;    // the last chain's piece ends mid-chain (publishes a state)
    __device__ int pieces() const { return ch_last - ch_first + 1; }
    // chain of the i-th piece in processing order: head piece, whole chains, tail piece
    __device__ int chain_at(int i) const {
        if (ch_first == ch_last) return ch_first;
        if (last_is_head) {
            if (i == 0) return ch_last;
            --i;
        }
        const int mid_lo = ch_first + (first_is_tail ? 1 : 0);
        const int mid_hi = ch_last - (last_is_head ? 1 : 0);
        return i <= mid_hi - mid_lo ? mid_lo + i : ch_first;
    }
};
__device__ __forceinline__ Range range_of(int k, const FpsParams& q) {
    Range r;
    r.lo = (int)((long long)k * q.W / q.G);
    r.hi = (int)((long long)(k + 1) * q.W / q.G);
    r.ch_first = r.lo / q.nc;
    r.ch_last = (r.hi - 1) / q.nc;
    r.first_is_tail = r.lo > r.ch_first * q.nc;
    r.last_is_head = r.hi < (r.ch_last + 1) * q.nc;
    return r;
}
// One piece: chunks [c0, c1) of chain ch = (bh*nmb + mb)*npb + pb.
struct Piece {
    int ch, bh, mb, pb, c0, c1;
};
__device__ __forceinline__ Piece piece_of(const Range& r, int i, const FpsParams& q) {
    Piece u;
    u.ch = r.chain_at(i);
    const int base = u.ch * q.nc;
    u.c0 = max(r.lo - base, 0);
    u.c1 = min(r.hi - base, q.nc);
    const int rb = u.ch / q.npb;
    u.pb = u.ch - rb * q.npb;
    u.bh = rb / q.nmb;
    u.mb = rb - u.bh * q.nmb;
    return u;
}

// Long chains (many ranges per chain) run in two passes instead of handing
// the state from range to range in order (a serial walk over every chunk of
// the chain):
//   kModeLocal  every piece starts from a zero state and keeps no hiddens; it
//               writes its end state A and its log2 decay sum to the aggregate
//               buffer (slot 2 k + [second chain of range k], per head of a
//               pair in the paired kernel);
//   scan        a CUDA-core kernel walks each chain's pieces in chunk order:
//               start = S, S <- 2^{sum} S + A, replacing A by the piece's
//               start state, and writes final_state;
//   kModeApply  every piece starts from its start state and writes hiddens.
// Ranges are then independent, and a chain's serial part is one fma per
// element and piece.  A range spans at most two chains in these modes (range
// length <= nc), so slot indices 2 k and 2 k + 1 cover every piece.
constexpr int kModeHandoff = 0;
constexpr int kModeLocal = 1;
constexpr int kModeApply = 2;

template <bool kHasInit, int kMode, bool kTmaH>
__global__ void __maxnreg__(kMaxRegs)
fwd_pass_state_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                  const __grid_constant__ CUtensorMap tm_h, const float* init, const float* __restrict__ Gcs,
                  const float* __restrict__ dtT, __nv_bfloat16* __restrict__ hiddens,
                  float* final_state, float* ring, unsigned int* ctrl, float* agg,
                  float* agg_lsum, const FpsParams q) {
    static_assert(kMode == kModeHandoff || !kHasInit, "the two passes take the initial state in the scan");
    static_assert(!kTmaH || (!kHasInit && kMode != kModeLocal), "the TMA-stored states need the shared tile");
    constexpr int S = stages<kHasInit, kTmaH>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* init_tile = reinterpret_cast<float*>(smem + S * kStageBytes);   // [64 p][128 n]
    uint8_t* htile = smem + S * kStageBytes + (kHasInit ? kInitBytes : 0);  // kTmaH: [128 n][64 p], swizzled
    uint8_t* vecs = htile + (kTmaH ? kHTileBytes : 0);                       // kVecSlots x (g[Q], dt[Q])
    uint64_t* bars = reinterpret_cast<uint64_t*>(vecs + kVecSlots * kVecSlotBytes);
    // barrier indices
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto scaled = [&](int s) { return smem_u32(bars + S + s); };
    auto empty = [&](int s) { return smem_u32(bars + 2 * S + s); };
    auto acc_full = [&](int k) { return smem_u32(bars + 3 * S + k); };
    constexpr int A = acc_slots<kHasInit>();
    constexpr int kB = 3 * S + 2 * kMaxAccSlots;   // first barrier after the ring / accumulator ones
    auto acc_empty = [&](int k) { return smem_u32(bars + 3 * S + kMaxAccSlots + k); };
    auto vec_full = [&](int v) { return smem_u32(bars + kB + v); };
    auto vec_empty = [&](int v) { return smem_u32(bars + kB + kVecSlots + v); };
    const uint32_t fold_done = smem_u32(bars + kB + 2 * kVecSlots);
    const uint32_t init_full = smem_u32(bars + kB + 2 * kVecSlots + 1);
    const uint32_t tile_free = smem_u32(bars + kB + 2 * kVecSlots + 2);
    const uint32_t mma_drain = smem_u32(bars + kB + 2 * kVecSlots + 3);
    // kTmaH: the state tile written (one arrival per fold warp) / read by its store
    const uint32_t h_full = smem_u32(bars + kB + 2 * kVecSlots + 4);
    const uint32_t h_free = smem_u32(bars + kB + 2 * kVecSlots + 5);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kB + 2 * kVecSlots + 6);
    int* range_id = reinterpret_cast<int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsub = q.Q / kSub;
    unsigned int* flags = ctrl + kCtrlFlagOffset;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(scaled(s), 32 * kScalerWarps);
            mbar_init(empty(s), 1);
        }
        for (int k = 0; k < A; ++k) {
            mbar_init(acc_full(k), 1);
            mbar_init(acc_empty(k), 32 * kFoldWarps);
        }
        for (int v = 0; v < kVecSlots; ++v) {
            mbar_init(vec_full(v), 1);
            mbar_init(vec_empty(v), 32 * kScalerWarps);
        }
        mbar_init(fold_done, kFoldWarps);
        mbar_init(init_full, 32 * kFoldWarps);
        mbar_init(tile_free, 32 * kFoldWarps);
        mbar_init(mma_drain, 1);
        mbar_init(h_full, kFoldWarps);
        mbar_init(h_free, 1);
        fence_mbar_init();
        // chunk_cumsum (G, dt, the cleared control block) must be complete
        grid_dependency_wait();
        // hand-offs need ranges in dispatch order (the range before this one
        // belongs to a CTA that is already running); the two passes have none
        *range_id = kMode == kModeHandoff ? (int)atomicAdd(ctrl, 1u) : (int)blockIdx.x;
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t stage0 = smem_u32(smem);
    const int rk = *range_id;
    const Range rg = range_of(rk, q);
    const int nchunks = rg.hi - rg.lo;
    grid_launch_dependents();   // compute_out may take each SM as this kernel leaves it

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            // a chain reads its x block once when the state is one block of N
            // rows: its lines are then loaded evict-first, leaving the L2 to what
            // is read again (with two blocks the other chain reads the same x)
            const bool x_once = q.nmb == 1;
            const uint64_t x_pol = x_once ? l2_policy_evict_first() : 0;
            int i = 0;   // stage counter
            int cv = 0;  // chunk counter (g / dt ring position)
            bool ok = true;
            for (int pi = 0; pi < rg.pieces() && ok; ++pi) {
                const Piece u = piece_of(rg, pi, q);
                const int b = u.bh / q.H, h = u.bh - b * q.H, grp = h / q.hpg;
                const int64_t ro = (int64_t)u.bh * q.Lp;
                for (int c = u.c0; c < u.c1 && ok; ++c, ++cv) {
                    // g and dt of the chunk, once per chunk
                    const int vslot = cv % kVecSlots;
                    if (!mbar_wait(vec_empty(vslot), ((cv / kVecSlots) & 1) ^ 1, &g_fps_error, 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t vs = smem_u32(vecs + vslot * kVecSlotBytes);
                    mbar_arrive_expect_tx(vec_full(vslot), 2 * q.Q * 4);
                    bulk_load(vs, Gcs + ro + (int64_t)c * q.Q, q.Q * 4, vec_full(vslot));
                    bulk_load(vs + kMaxQ * 4, dtT + ro + (int64_t)c * q.Q, q.Q * 4, vec_full(vslot));
                    for (int sub = 0; sub < nsub; ++sub, ++i) {
                        const int s = i % S, k = i / S;
                        if (!mbar_wait(empty(s), (k & 1) ^ 1, &g_fps_error, 1u)) {
                            ok = false;
                            break;
                        }
                        const uint32_t xs = stage0 + s * kStageBytes, bs = xs + kXBytes;
                        const int tok = c * q.Q + sub * kSub;
                        mbar_arrive_expect_tx(full(s), kXBytes + kBBytes);
                        if (x_once)
                            tma_load_4d_hint(xs, &tm_x, full(s), u.pb * kCols, h, tok, b, x_pol);
                        else
                            tma_load_4d(xs, &tm_x, full(s), u.pb * kCols, h, tok, b);
#pragma unroll
                        for (int jb = 0; jb < 2; ++jb)
                            tma_load_4d(bs + jb * kSub * kRowBytes, &tm_b, full(s),
                                        u.mb * 128 + jb * 64, grp, tok, b);
                    }
                }
            }
            // No copy may land in shared memory after the CTA has left: wait for the
            // last stages and g/dt slots issued (already complete unless a bounded
            // wait elsewhere gave up and the consumers stopped early).
            for (int j = i - min(i, S); j < i; ++j)
                (void)mbar_wait(full(j % S), (j / S) & 1, &g_fps_error, 1u);
            for (int j = cv - min(cv, kVecSlots); j < cv; ++j)
                (void)mbar_wait(vec_full(j % kVecSlots), (j / kVecSlots) & 1, &g_fps_error, 1u);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: one chunk product per accumulator slot ----------------
        if (lane == 0) {
            int i = 0;
            for (int qc = 0; qc < nchunks; ++qc) {
                const int slot = qc % A;
                bool ok = true;
                for (int sub = 0; sub < nsub; ++sub, ++i) {
                    const int s = i % S, k = i / S;
                    if (!mbar_wait(scaled(s), k & 1, &g_fps_error, 1u)) { ok = false; break; }
                    // the fold warps have read this slot's previous product
                    if (sub == 0 &&
                        !mbar_wait(acc_empty(slot), ((qc / A) & 1) ^ 1, &g_fps_error, 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xs = stage0 + s * kStageBytes, bs = xs + kXBytes;
                    // A = B_c^T: M = 128 state rows (two 64-row swizzle atoms, kSub*128
                    // bytes apart), K = 16 tokens, MN-major.  B = s o X_c: N = 64 columns
                    // of P, K = 16 tokens, MN-major.  A K step adds a compile-time offset
                    // to the start-address field.
                    const uint64_t ad0 = smem_desc_sw128(bs, kSub * kRowBytes, 8 * kRowBytes);
                    const uint64_t bd0 = smem_desc_sw128(xs, kSub * kRowBytes, 8 * kRowBytes);
#pragma unroll
                    for (int kk = 0; kk < kSub / 16; ++kk)
                        mma_f16_ss(tmem + slot * kCols, ad0 + (uint64_t)((kk * 16 * kRowBytes) >> 4),
                                   bd0 + (uint64_t)((kk * 16 * kRowBytes) >> 4), kIdesc,
                                   (sub > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(empty(s));
                    if (sub == nsub - 1) mma_commit(acc_full(slot));
                }
                if (!ok) break;
            }
            // every MMA issued has finished before TMEM is released
            mma_commit(mma_drain);
            (void)mbar_wait(mma_drain, 0, &g_fps_error, 1u);
        }
    } else if (warp < 2 + kScalerWarps) {
        // ---------------- scaler warps: x_q <- x_q * dt_q 2^{g_last - g_q} ----------------
        // 16-byte vectors of the stage's x tile (kSub rows x 8) dealt round-robin.
        const int tid = threadIdx.x - 64;
        constexpr int kVecs = kSub * 8;
        constexpr int kPer = (kVecs + 32 * kScalerWarps - 1) / (32 * kScalerWarps);
        const int nstages = nchunks * nsub;
        for (int i = 0; i < nstages; ++i) {
            const int s = i % S, k = i / S;
            const int cv = i / nsub, sub = i - cv * nsub, vslot = cv % kVecSlots;
            if (!mbar_wait(full(s), k & 1, &g_fps_error, 1u)) break;
            if (sub == 0 && !mbar_wait(vec_full(vslot), (cv / kVecSlots) & 1, &g_fps_error, 1u)) break;
            const float* gchunk = reinterpret_cast<const float*>(vecs + vslot * kVecSlotBytes);
            const float* gv = gchunk + sub * kSub;
            const float* dv = gv + kMaxQ;
            const float glast = gchunk[q.Q - 1];
            uint8_t* xs = smem + s * kStageBytes;
#pragma unroll
            for (int kq = 0; kq < kPer; ++kq) {
                const int v = tid + kq * 32 * kScalerWarps;
                if (v < kVecs) {
                    const int r = v >> 3;
                    // fp32 scale, one rounding to bf16 per product (as the pages'
                    // cast of the scaled operand)
                    const float sc = dv[r] * exp2f(glast - gv[r]);
                    uint4* ptr = reinterpret_cast<uint4*>(xs + r * kRowBytes) + (v & 7);
                    uint4 w = *ptr;
                    w.x = pack_bf16(bf16lo(w.x) * sc, bf16hi(w.x) * sc);
                    w.y = pack_bf16(bf16lo(w.y) * sc, bf16hi(w.y) * sc);
                    w.z = pack_bf16(bf16lo(w.z) * sc, bf16hi(w.z) * sc);
                    w.w = pack_bf16(bf16lo(w.w) * sc, bf16hi(w.w) * sc);
                    *ptr = w;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(scaled(s));
            if (sub == nsub - 1) mbar_arrive(vec_empty(vslot));
        }
    } else {
        // ---------------- fold warps: hiddens[c] = S, S <- 2^{g_last} S + D_c ----------------
        // Thread = TMEM lane = state row n of the chain's 128-row block.  The
        // running state S^T of a piece lives in a TMEM state slot (piece parity
        // picks the slot when there are two).  A hand-off slot in global memory
        // holds S^T as [16][128 rows][4] fp32, so that a warp's float4 accesses
        // cover 512 contiguous bytes.  Every exit from this loop is warp-uniform:
        // the warp-collective TMEM accesses and __syncwarp calls never wait for a
        // lane that has left.
        constexpr int kStates = kHasInit ? 2 : 1;
        const int quarter = warp & 3;
        const int rl = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t st_base = lane_base + A * kCols;
        // The state tile in shared memory: fp32 [64 p][128 n]; thread n only
        // reads / writes column n in the fold (conflict-free), and the copies to
        // and from global memory move whole 512-byte rows.  These copies use the
        // LSU path (cp.async in, vector stores out), not the TMA, so that they
        // never queue behind the x / B stream.
        float* tcol = init_tile + rl;
        auto tile_at = [&](int pp) -> float& { return tcol[pp * 128]; };
        int qc = 0;       // chunk counter (accumulator ring position)
        int ntile = 0;    // init tiles consumed (init_full phases)
        int nfree = 0;    // tile_free phases
        int ld_next = 0;  // next piece to consider for an init-tile load
        // Init tiles (rows p of [b, H, P, N], 128 columns of N, zero-filled past P
        // and N) are fetched by all fold threads, one piece ahead of their use.
        auto issue_next_init = [&]() {
            while (ld_next < rg.pieces() && piece_of(rg, ld_next, q).c0 != 0) ++ld_next;
            if (ld_next < rg.pieces()) {
                const Piece un = piece_of(rg, ld_next, q);
                const int rows = min(q.P - un.pb * kCols, kCols), ncols = min(q.N - un.mb * 128, 128);
                const float* g0 = init + ((int64_t)un.bh * q.P + un.pb * kCols) * q.N + un.mb * 128;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int idx = i * 128 + rl, pp = idx >> 5, c4 = idx & 31;
                    const bool v = pp < rows && 4 * c4 < ncols;
                    cp_async_16(smem_u32(init_tile + pp * 128 + 4 * c4),
                                v ? g0 + (int64_t)pp * q.N + 4 * c4 : g0, v ? 16u : 0u);
                }
                cp_async_mbar_arrive_noinc(init_full);
                ++ld_next;
            }
        };
        // the next init tile -> a TMEM state slot
        auto take_tile = [&](uint32_t slot_addr) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(init_full, ntile & 1, &g_fps_error, 1u))) return false;
            ++ntile;
#pragma unroll
            for (int jj = 0; jj < kCols / 16; ++jj) {
                uint32_t v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(tile_at(16 * jj + k));
                __syncwarp();
                tmem_st_x16(slot_addr + 16 * jj, v);
            }
            tmem_wait_st();
            return true;
        };
        // barrier of the fold threads over the tile buffer: every thread waits
        // until all of them have finished their accesses (warp-uniform result)
        auto tile_sync = [&]() -> bool {
            __syncwarp();
            mbar_arrive(tile_free);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(tile_free, nfree & 1, &g_fps_error, 1u));
            ++nfree;
            return ok;
        };
        if (kHasInit) issue_next_init();
        const float* gfirst = Gcs + q.Q - 1;   // g_last of chunk c of head bh: gfirst[bh*Lp + c*Q]
        float gl_first = 0.f;                  // g_last of the next piece's first chunk
        {
            const Piece u0 = piece_of(rg, 0, q);
            gl_first = gfirst[(int64_t)u0.bh * q.Lp + (int64_t)u0.c0 * q.Q];
        }
        for (int pi = 0; pi < rg.pieces(); ++pi) {
            const Piece u = piece_of(rg, pi, q);
            const int n = u.mb * 128 + rl;
            const bool nok = n < q.N;
            const int p0 = u.pb * kCols;
            const int64_t sbase = (int64_t)u.bh * q.P * q.N;
            const uint32_t sa = st_base + (pi % kStates) * kCols;
            const float* grow = gfirst + (int64_t)u.bh * q.Lp;
            float gl_next = gl_first;
            if (pi + 1 < rg.pieces()) {  // prefetch for the next piece
                const Piece un = piece_of(rg, pi + 1, q);
                gl_first = gfirst[(int64_t)un.bh * q.Lp + (int64_t)un.c0 * q.Q];
            }
            // kModeLocal / kModeApply: the piece's aggregate slot
            const int64_t aslot = 2 * (int64_t)rk + (u.ch == rg.ch_first ? 0 : 1);
            float lsum = 0.f;   // kModeLocal: log2 of the piece's decay product
            // the piece's initial state -> TMEM slot sa
            if (kMode == kModeApply) {
                // its start state, from the scan
                const float* src = agg + aslot * kSlotFloats;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    uint32_t v[16];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float4 f = __ldcg(reinterpret_cast<const float4*>(src + ((4 * jj + q4) * 128 + rl) * 4));
                        v[4 * q4] = __float_as_uint(f.x); v[4 * q4 + 1] = __float_as_uint(f.y);
                        v[4 * q4 + 2] = __float_as_uint(f.z); v[4 * q4 + 3] = __float_as_uint(f.w);
                    }
                    __syncwarp();
                    tmem_st_x16(sa + 16 * jj, v);
                }
            } else if (kMode == kModeLocal || u.c0 == 0) {
                if (kHasInit) {
                    if (pi == 0) {  // later pieces found theirs in sa already
                        if (!take_tile(sa)) break;
                        if (!tile_sync()) break;
                        issue_next_init();
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < kCols / 16; ++jj) {
                        uint32_t v[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) v[k] = 0u;
                        __syncwarp();
                        tmem_st_x16(sa + 16 * jj, v);
                    }
                }
            } else {
                // the state published by the CTA of the previous range
                bool ok = true;
                if (lane == 0) ok = flag_wait_geq(flags + u.ch, (unsigned)u.c0, &g_fps_error, 1u);
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                (void)ld_acquire_gpu(flags + u.ch);  // this lane's own acquire of the hand-off
                const float* src = ring + ((int64_t)u.ch * 2 + ((rk - 1) & 1)) * kSlotFloats;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    uint32_t v[16];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float4 f = __ldcg(reinterpret_cast<const float4*>(src + ((4 * jj + q4) * 128 + rl) * 4));
                        v[4 * q4] = __float_as_uint(f.x); v[4 * q4 + 1] = __float_as_uint(f.y);
                        v[4 * q4 + 2] = __float_as_uint(f.z); v[4 * q4 + 3] = __float_as_uint(f.w);
                    }
                    __syncwarp();
                    tmem_st_x16(sa + 16 * jj, v);
                }
            }
            tmem_wait_st();
            bool ok = true;
            for (int c = u.c0; c < u.c1; ++c, ++qc) {
                const float e = exp2f(gl_next);
                lsum += gl_next;
                if (c + 1 < u.c1) gl_next = grow[(int64_t)(c + 1) * q.Q];
                const int slot = qc % A;
                if (!__all_sync(0xffffffffu, mbar_wait(acc_full(slot), (qc / A) & 1, &g_fps_error, 1u))) {
                    ok = false;
                    break;
                }
                if (kTmaH && qc > 0) {
                    // the previous chunk's store has read the state tile
                    if (rl == 0) {
                        bulk_wait_group_read0();
                        mbar_arrive(h_free);
                    }
                    if (!__all_sync(0xffffffffu, mbar_wait(h_free, (qc - 1) & 1, &g_fps_error, 1u))) {
                        ok = false;
                        break;
                    }
                }
                tc_fence_after();
                const uint32_t acc = lane_base + slot * kCols;
                __nv_bfloat16* hp = hiddens + (((int64_t)u.bh * q.nc + c) * q.N + n) * q.P + p0;
                // kTmaH: row rl of the 128-byte-swizzled tile, 16-byte chunk j at (j ^ (rl % 8)) * 16
                uint8_t* trow = htile + rl * kRowBytes;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    __syncwarp();
                    uint32_t sv[16], d[16];
                    tmem_ld_x16(sa + 16 * jj, sv);
                    tmem_ld_x16(acc + 16 * jj, d);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        d[k] = __float_as_uint(fmaf(e, __uint_as_float(sv[k]), __uint_as_float(d[k])));
                    tmem_st_x16(sa + 16 * jj, d);
                    // chunk-start state S -> hiddens[c] (row n holds S[:, n]): 16
                    // contiguous bf16 per slice (P is a multiple of 16)
                    if (kMode != kModeLocal && nok && (kTmaH || p0 + 16 * jj < q.P)) {
                        uint4 w0, w1;
                        w0.x = pack_bf16(__uint_as_float(sv[0]), __uint_as_float(sv[1]));
                        w0.y = pack_bf16(__uint_as_float(sv[2]), __uint_as_float(sv[3]));
                        w0.z = pack_bf16(__uint_as_float(sv[4]), __uint_as_float(sv[5]));
                        w0.w = pack_bf16(__uint_as_float(sv[6]), __uint_as_float(sv[7]));
                        w1.x = pack_bf16(__uint_as_float(sv[8]), __uint_as_float(sv[9]));
                        w1.y = pack_bf16(__uint_as_float(sv[10]), __uint_as_float(sv[11]));
                        w1.z = pack_bf16(__uint_as_float(sv[12]), __uint_as_float(sv[13]));
                        w1.w = pack_bf16(__uint_as_float(sv[14]), __uint_as_float(sv[15]));
                        if (kTmaH) {
                            *reinterpret_cast<uint4*>(trow + (((2 * jj) ^ (rl & 7)) << 4)) = w0;
                            *reinterpret_cast<uint4*>(trow + (((2 * jj + 1) ^ (rl & 7)) << 4)) = w1;
                        } else {
                            uint4* hdst = reinterpret_cast<uint4*>(hp + 16 * jj);
                            hdst[0] = w0;
                            hdst[1] = w1;
                        }
                    }
                }
                if (kTmaH) {
                    fence_proxy_async_smem();   // tile writes -> the TMA store
                    __syncwarp();
                    if (lane == 0) mbar_arrive(h_full);
                }
                __syncwarp();
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(acc_empty(slot));
                if (kTmaH) {
                    // one thread stores the chunk's [128 n][64 p] block of hiddens
                    bool okh = true;
                    if (rl == 0) {
                        okh = mbar_wait(h_full, qc & 1, &g_fps_error, 1u);
                        if (okh) {
                            tma_store_3d(&tm_h, smem_u32(htile), p0, u.mb * 128, u.bh * q.nc + c);
                            bulk_commit_group();
                        }
                    }
                    if (!__all_sync(0xffffffffu, okh)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!__all_sync(0xffffffffu, ok)) break;
            if (kMode == kModeLocal) {
                // the piece's end state and log2 decay, for the scan
                float* dst = agg + aslot * kSlotFloats;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    __syncwarp();
                    uint32_t sv[16];
                    tmem_ld_x16(sa + 16 * jj, sv);
                    tmem_wait_ld();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        __stcg(reinterpret_cast<float4*>(dst + ((4 * jj + q4) * 128 + rl) * 4),
                               make_float4(__uint_as_float(sv[4 * q4]), __uint_as_float(sv[4 * q4 + 1]),
                                           __uint_as_float(sv[4 * q4 + 2]), __uint_as_float(sv[4 * q4 + 3])));
                }
                if (rl == 0) agg_lsum[aslot] = lsum;
                continue;
            }
            if (kMode == kModeApply) continue;   // final_state comes from the scan
            // the next piece's initial state into the spare slot, so that it can
            // start at once, before the tile buffer is reused below
            const bool next_tile = kHasInit && pi + 1 < rg.pieces() && piece_of(rg, pi + 1, q).c0 == 0;
            if (next_tile && !take_tile(st_base + ((pi + 1) % kStates) * kCols)) break;
            // the piece's final state: to final_state, or published for the next range
            const bool last = u.c1 == q.nc;
            if (last && final_state != nullptr && kHasInit) {
                // through the tile buffer: columns in, rows out as 16-byte stores
                if (next_tile && !tile_sync()) break;   // everyone has read the tile
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    __syncwarp();
                    uint32_t sv[16];
                    tmem_ld_x16(sa + 16 * jj, sv);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) tile_at(16 * jj + k) = __uint_as_float(sv[k]);
                }
                if (!tile_sync()) break;
                {
                    const int rows = min(q.P - p0, kCols), ncols = min(q.N - u.mb * 128, 128);
                    float* g0 = final_state + ((int64_t)u.bh * q.P + p0) * q.N + u.mb * 128;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int idx = i * 128 + rl, pp = idx >> 5, c4 = idx & 31;
                        if (pp < rows && 4 * c4 < ncols)
                            *reinterpret_cast<float4*>(g0 + (int64_t)pp * q.N + 4 * c4) =
                                *reinterpret_cast<const float4*>(init_tile + pp * 128 + 4 * c4);
                    }
                }
                if (!tile_sync()) break;   // the tile has been read before it is refilled
                issue_next_init();
            } else {
                if (next_tile) {
                    if (!tile_sync()) break;
                    issue_next_init();
                }
                if (last) {
                    if (final_state != nullptr) {
                        const int pl = nok ? q.P - p0 : 0;
#pragma unroll
                        for (int jj = 0; jj < kCols / 16; ++jj) {
                            __syncwarp();
                            uint32_t sv[16];
                            tmem_ld_x16(sa + 16 * jj, sv);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                if (16 * jj + k < pl)
                                    final_state[sbase + (int64_t)(p0 + 16 * jj + k) * q.N + n] =
                                        __uint_as_float(sv[k]);
                        }
                    }
                } else {
                    float* dst = ring + ((int64_t)u.ch * 2 + (rk & 1)) * kSlotFloats;
#pragma unroll
                    for (int jj = 0; jj < kCols / 16; ++jj) {
                        __syncwarp();
                        uint32_t sv[16];
                        tmem_ld_x16(sa + 16 * jj, sv);
                        tmem_wait_ld();
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            __stcg(reinterpret_cast<float4*>(dst + ((4 * jj + q4) * 128 + rl) * 4),
                                   make_float4(__uint_as_float(sv[4 * q4]), __uint_as_float(sv[4 * q4 + 1]),
                                               __uint_as_float(sv[4 * q4 + 2]), __uint_as_float(sv[4 * q4 + 3])));
                    }
                    // publish: every fold warp's stores, then one release of the
                    // chain's flag (a range publishes at most once)
                    __syncwarp();
                    if (lane == 0) mbar_arrive(fold_done);
                    bool okp = true;
                    if (rl == 0) {
                        okp = mbar_wait(fold_done, 0, &g_fps_error, 1u);
                        if (okp && *reinterpret_cast<volatile unsigned int*>(&g_fps_withhold) == 0u) {
                            __threadfence();
                            st_release_gpu(flags + u.ch, (unsigned)u.c1);
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, okp, 0)) break;
                }
            }
        }
        if (kHasInit) cp_async_wait_all();  // no copy into shared memory outlives the CTA
        if (kTmaH && rl == 0) bulk_wait_group0();   // the state stores have completed
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) report_timeout_to_host(&g_fps_error, q.host_err);
    if (warp == 1) {
        __syncwarp();  // lane 0 ran the MMA loop alone: reconverge before the collective
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ===========================================================================
// Paired variant (N <= 128, P <= 64, an even number of heads per group): one
// CTA per SM walks two adjacent heads of the same group in
// lockstep.  Both heads' chunk products take the same B tile as the MMA's A
// operand, so every B tile is loaded once for two heads, and the 512 TMEM
// columns of a whole SM hold both running states and six chunk products (three
// per head in flight).  A work unit is one chunk of a pair-chain (batch, head
// pair); ranges, pieces and hand-offs are those of the kernel above, with a
// hand-off flag and a two-slot buffer per head.  A chain's initial state is
// read from init_state at its first chunk (lane n of each warp takes column n,
// so every row of the read is one coalesced 128-byte line).
//
// The two x tiles of a stage sit side by side, so one N = 128 MMA per K step
// computes both heads' products (columns [0, 64) head 0, [64, 128) head 1 of a
// product-slot pair).  With P = 64 (kTmaH) the chunk-start states leave through
// a 128-byte-swizzled shared-memory tile per head and one TMA tensor store per
// chunk (full 128-byte lines), instead of 16-byte stores from every thread,
// one row per lane, that touch 32 lines per warp instruction.
// ===========================================================================
constexpr int kPProdSlots = 6;                    // chunk products in flight (3 per head)
constexpr int kPScalerWarps = 8;
constexpr int kPThreads = 32 * (2 + kPScalerWarps + 8);   // 576: + two fold warpgroups
constexpr int kPStageBytes = 2 * kXBytes + kBBytes;       // x0 | x1 | B, 32 KB
constexpr int kPVecSlots = 3;
constexpr int kPVecSlotBytes = 4 * kMaxQ * 4;     // g, dt of both heads
constexpr int kPBarBytes = 1024;
constexpr int kPHBytes = 128 * kRowBytes;         // hiddens tile of one head: <= 128 rows of 64 p
// TMA ring depth: five stages when two hiddens tiles share the shared memory
template <bool kTmaH> __host__ __device__ constexpr int pair_stages() { return kTmaH ? 5 : 6; }
template <bool kTmaH>
__host__ __device__ constexpr int pair_smem() {
    return pair_stages<kTmaH>() * kPStageBytes + (kTmaH ? 2 * kPHBytes : 0) +
           kPVecSlots * kPVecSlotBytes + kPBarBytes + 1024;
}
constexpr uint32_t kIdescPair = make_idesc(1, 128, 2 * kCols, 1, 1);

static_assert(kPStageBytes % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");

template <bool kTmaH, int kMode>
__global__ void __launch_bounds__(kPThreads, 1)
fwd_pass_state_pair_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                       const __grid_constant__ CUtensorMap tm_h, const float* init,
                       const float* __restrict__ Gcs, const float* __restrict__ dtT,
                       __nv_bfloat16* __restrict__ hiddens, float* final_state, float* ring,
                       unsigned int* ctrl, float* agg, float* agg_lsum, const FpsParams q) {
    static_assert(kMode != kModeLocal || !kTmaH, "the local pass stores no hiddens");
    constexpr int S = pair_stages<kTmaH>();
    constexpr int PS = kPProdSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* htile = smem + S * kPStageBytes;  // kTmaH: hiddens tiles of head 0 / 1
    uint8_t* vecs = htile + (kTmaH ? 2 * kPHBytes : 0);   // kPVecSlots x (g0, dt0, g1, dt1)
    uint64_t* bars = reinterpret_cast<uint64_t*>(vecs + kPVecSlots * kPVecSlotBytes);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto scaled = [&](int s) { return smem_u32(bars + S + s); };
    auto empty = [&](int s) { return smem_u32(bars + 2 * S + s); };
    auto prod_full = [&](int k) { return smem_u32(bars + 3 * S + k); };
    auto prod_empty = [&](int k) { return smem_u32(bars + 3 * S + PS + k); };
    auto vec_full = [&](int v) { return smem_u32(bars + 3 * S + 2 * PS + v); };
    auto vec_empty = [&](int v) { return smem_u32(bars + 3 * S + 2 * PS + kPVecSlots + v); };
    auto fold_done = [&](int hd) { return smem_u32(bars + 3 * S + 2 * PS + 2 * kPVecSlots + hd); };
    const uint32_t mma_drain = smem_u32(bars + 3 * S + 2 * PS + 2 * kPVecSlots + 2);
    // kTmaH: hiddens tile written (one arrival per fold warp) / read by its store
    auto h_full = [&](int hd) { return smem_u32(bars + 3 * S + 2 * PS + 2 * kPVecSlots + 3 + hd); };
    auto h_free = [&](int hd) { return smem_u32(bars + 3 * S + 2 * PS + 2 * kPVecSlots + 5 + hd); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * S + 2 * PS + 2 * kPVecSlots + 7);
    int* range_id = reinterpret_cast<int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsub = q.Q / kSub;
    unsigned int* flags = ctrl + kCtrlFlagOffset;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(scaled(s), 32 * kPScalerWarps);
            mbar_init(empty(s), 1);
        }
        for (int k = 0; k < PS; ++k) {
            mbar_init(prod_full(k), 1);
            mbar_init(prod_empty(k), 128);
        }
        for (int v = 0; v < kPVecSlots; ++v) {
            mbar_init(vec_full(v), 1);
            mbar_init(vec_empty(v), 32 * kPScalerWarps);
        }
        mbar_init(fold_done(0), 4);
        mbar_init(fold_done(1), 4);
        mbar_init(mma_drain, 1);
        for (int hd = 0; hd < 2; ++hd) {
            mbar_init(h_full(hd), 4);
            mbar_init(h_free(hd), 1);
        }
        fence_mbar_init();
        grid_dependency_wait();   // chunk_cumsum (G, dt, the cleared control block)
        // hand-offs need ranges in dispatch order; the two passes have none
        *range_id = kMode == kModeHandoff ? (int)atomicAdd(ctrl, 1u) : (int)blockIdx.x;
    }
    __syncwarp();
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t stage0 = smem_u32(smem);
    const int rk = *range_id;
    const Range rg = range_of(rk, q);
    const int nchunks = rg.hi - rg.lo;
    grid_launch_dependents();

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            // x is read once here: its lines are loaded evict-first, leaving the
            // L2 to what is read again (the group's B tiles, the states written here)
            const uint64_t x_pol = l2_policy_evict_first();
            int i = 0, cv = 0;
            bool ok = true;
            for (int pi = 0; pi < rg.pieces() && ok; ++pi) {
                const Piece u = piece_of(rg, pi, q);
                const int bh0 = 2 * u.bh;                  // the pair's first head
                const int b = bh0 / q.H, h0 = bh0 - b * q.H, grp = h0 / q.hpg;
                const int64_t ro = (int64_t)bh0 * q.Lp;
                for (int c = u.c0; c < u.c1 && ok; ++c, ++cv) {
                    const int vslot = cv % kPVecSlots;
                    if (!mbar_wait(vec_empty(vslot), ((cv / kPVecSlots) & 1) ^ 1, &g_fps_error, 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t vs = smem_u32(vecs + vslot * kPVecSlotBytes);
                    const int64_t co = (int64_t)c * q.Q;
                    mbar_arrive_expect_tx(vec_full(vslot), 4 * q.Q * 4);
                    bulk_load(vs, Gcs + ro + co, q.Q * 4, vec_full(vslot));
                    bulk_load(vs + kMaxQ * 4, dtT + ro + co, q.Q * 4, vec_full(vslot));
                    bulk_load(vs + 2 * kMaxQ * 4, Gcs + ro + q.Lp + co, q.Q * 4, vec_full(vslot));
                    bulk_load(vs + 3 * kMaxQ * 4, dtT + ro + q.Lp + co, q.Q * 4, vec_full(vslot));
                    for (int sub = 0; sub < nsub; ++sub, ++i) {
                        const int s = i % S, k = i / S;
                        if (!mbar_wait(empty(s), (k & 1) ^ 1, &g_fps_error, 1u)) {
                            ok = false;
                            break;
                        }
                        const uint32_t xs = stage0 + s * kPStageBytes, bs = xs + 2 * kXBytes;
                        const int tok = c * q.Q + sub * kSub;
                        mbar_arrive_expect_tx(full(s), kPStageBytes);
                        tma_load_4d_hint(xs, &tm_x, full(s), 0, h0, tok, b, x_pol);
                        tma_load_4d_hint(xs + kXBytes, &tm_x, full(s), 0, h0 + 1, tok, b, x_pol);
#pragma unroll
                        for (int jb = 0; jb < 2; ++jb)
                            tma_load_4d(bs + jb * kSub * kRowBytes, &tm_b, full(s), jb * 64, grp, tok, b);
                    }
                }
            }
            for (int j = i - min(i, S); j < i; ++j)
                (void)mbar_wait(full(j % S), (j / S) & 1, &g_fps_error, 1u);
            for (int j = cv - min(cv, kPVecSlots); j < cv; ++j)
                (void)mbar_wait(vec_full(j % kPVecSlots), (j / kPVecSlots) & 1, &g_fps_error, 1u);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: both heads' products share the B operand ----------------
        if (lane == 0) {
            int i = 0;
            for (int qc = 0; qc < nchunks; ++qc) {
                const int p0 = 2 * qc, p1 = 2 * qc + 1;   // product numbers of head 0 / 1
                const int sl0 = p0 % PS, sl1 = p1 % PS;
                bool ok = true;
                for (int sub = 0; sub < nsub; ++sub, ++i) {
                    const int s = i % S, k = i / S;
                    if (!mbar_wait(scaled(s), k & 1, &g_fps_error, 1u)) { ok = false; break; }
                    if (sub == 0 &&
                        (!mbar_wait(prod_empty(sl0), ((p0 / PS) & 1) ^ 1, &g_fps_error, 1u) ||
                         !mbar_wait(prod_empty(sl1), ((p1 / PS) & 1) ^ 1, &g_fps_error, 1u))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xs = stage0 + s * kPStageBytes, bs = xs + 2 * kXBytes;
                    const uint64_t ad0 = smem_desc_sw128(bs, kSub * kRowBytes, 8 * kRowBytes);
                    // B operand: x0 | x1, two 64-column swizzle atoms kXBytes apart;
                    // the products of slot pair (sl0, sl1 = sl0 + 1) are adjacent in TMEM
                    const uint64_t bd0 = smem_desc_sw128(xs, kXBytes, 8 * kRowBytes);
#pragma unroll
                    for (int kk = 0; kk < kSub / 16; ++kk) {
                        const uint64_t ko = (uint64_t)((kk * 16 * kRowBytes) >> 4);
                        const uint32_t acc = (sub > 0 || kk > 0) ? 1u : 0u;
                        mma_f16_ss(tmem + 128 + sl0 * kCols, ad0 + ko, bd0 + ko, kIdescPair, acc);
                    }
                    mma_commit(empty(s));
                    if (sub == nsub - 1) {
                        mma_commit(prod_full(sl0));
                        mma_commit(prod_full(sl1));
                    }
                }
                if (!ok) break;
            }
            mma_commit(mma_drain);
            (void)mbar_wait(mma_drain, 0, &g_fps_error, 1u);
        }
    } else if (warp < 2 + kPScalerWarps) {
        // ---------------- scaler warps: both heads' x rows ----------------
        const int tid = threadIdx.x - 64;
        constexpr int kVecs = 2 * kSub * 8;   // 16-byte vectors of the two x tiles
        constexpr int kPer = kVecs / (32 * kPScalerWarps);
        const int nstages = nchunks * nsub;
        for (int i = 0; i < nstages; ++i) {
            const int s = i % S, k = i / S;
            const int cv = i / nsub, sub = i - cv * nsub, vslot = cv % kPVecSlots;
            if (!mbar_wait(full(s), k & 1, &g_fps_error, 1u)) break;
            if (sub == 0 && !mbar_wait(vec_full(vslot), (cv / kPVecSlots) & 1, &g_fps_error, 1u)) break;
            const float* vbase = reinterpret_cast<const float*>(vecs + vslot * kPVecSlotBytes);
            uint8_t* xs = smem + s * kPStageBytes;
#pragma unroll
            for (int kq = 0; kq < kPer; ++kq) {
                const int v = tid + kq * 32 * kPScalerWarps;
                const int hd = v >> 9, r = (v >> 3) & (kSub - 1);
                const float* gch = vbase + hd * 2 * kMaxQ;    // g of this head's chunk
                const float* gv = gch + sub * kSub;
                const float* dv = gv + kMaxQ;
                const float sc = dv[r] * exp2f(gch[q.Q - 1] - gv[r]);
                uint4* ptr = reinterpret_cast<uint4*>(xs + hd * kXBytes + r * kRowBytes) + (v & 7);
                uint4 w = *ptr;
                w.x = pack_bf16(bf16lo(w.x) * sc, bf16hi(w.x) * sc);
                w.y = pack_bf16(bf16lo(w.y) * sc, bf16hi(w.y) * sc);
                w.z = pack_bf16(bf16lo(w.z) * sc, bf16hi(w.z) * sc);
                w.w = pack_bf16(bf16lo(w.w) * sc, bf16hi(w.w) * sc);
                *ptr = w;
            }
            fence_proxy_async_smem();
            mbar_arrive(scaled(s));
            if (sub == nsub - 1) mbar_arrive(vec_empty(vslot));
        }
    } else {
        // ---------------- fold warpgroups: one per head of the pair ----------------
        // Warps 10..13 fold head 0's products, 14..17 head 1's; thread = TMEM lane
        // = state row n; the running state of head hd sits in TMEM columns
        // [64 hd, 64 hd + 64).  Exits from this loop are warp-uniform.
        const int hd = (warp - 2 - kPScalerWarps) >> 2;
        const int quarter = warp & 3;
        const int rl = quarter * 32 + lane;
        const bool nok = rl < q.N;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t sa = lane_base + hd * kCols;
        int qc = 0;
        for (int pi = 0; pi < rg.pieces(); ++pi) {
            const Piece u = piece_of(rg, pi, q);
            const int bh = 2 * u.bh + hd;                  // this head
            const int ch = 2 * u.ch + hd;                  // its hand-off chain
            const int64_t sbase = (int64_t)bh * q.P * q.N;
            const float* grow = Gcs + (int64_t)bh * q.Lp + q.Q - 1;
            float gl_next = grow[(int64_t)u.c0 * q.Q];
            float lsum = 0.f;   // kModeLocal: log2 of the piece's decay product
            // kModeLocal / kModeApply: the piece's aggregate slot
            const int64_t aslot = (int64_t)(2 * rk + (u.ch == rg.ch_first ? 0 : 1)) * 2 + hd;
            if (kMode == kModeApply) {
                const float* src = agg + aslot * kSlotFloats;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    uint32_t v[16];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float4 f = __ldcg(reinterpret_cast<const float4*>(src + ((4 * jj + q4) * 128 + rl) * 4));
                        v[4 * q4] = __float_as_uint(f.x); v[4 * q4 + 1] = __float_as_uint(f.y);
                        v[4 * q4 + 2] = __float_as_uint(f.z); v[4 * q4 + 3] = __float_as_uint(f.w);
                    }
                    __syncwarp();
                    tmem_st_x16(sa + 16 * jj, v);
                }
            } else if (kMode == kModeLocal || u.c0 == 0) {
                // zero, or (hand-off mode) the chain's initial state [P][N]:
                // lane rl takes column n = rl, coalesced across the warp
                const float* ib = (kMode == kModeHandoff && init != nullptr && nok) ? init + sbase + rl : nullptr;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    uint32_t v[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        v[k] = (ib != nullptr && 16 * jj + k < q.P) ? __float_as_uint(__ldg(ib + (int64_t)(16 * jj + k) * q.N)) : 0u;
                    __syncwarp();
                    tmem_st_x16(sa + 16 * jj, v);
                }
            } else {
                bool ok = true;
                if (lane == 0) ok = flag_wait_geq(flags + ch, (unsigned)u.c0, &g_fps_error, 1u);
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                (void)ld_acquire_gpu(flags + ch);
                const float* src = ring + ((int64_t)ch * 2 + ((rk - 1) & 1)) * kSlotFloats;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    uint32_t v[16];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float4 f = __ldcg(reinterpret_cast<const float4*>(src + ((4 * jj + q4) * 128 + rl) * 4));
                        v[4 * q4] = __float_as_uint(f.x); v[4 * q4 + 1] = __float_as_uint(f.y);
                        v[4 * q4 + 2] = __float_as_uint(f.z); v[4 * q4 + 3] = __float_as_uint(f.w);
                    }
                    __syncwarp();
                    tmem_st_x16(sa + 16 * jj, v);
                }
            }
            tmem_wait_st();
            bool ok = true;
            for (int c = u.c0; c < u.c1; ++c, ++qc) {
                const float e = exp2f(gl_next);
                lsum += gl_next;
                if (c + 1 < u.c1) gl_next = grow[(int64_t)(c + 1) * q.Q];
                const int pn = 2 * qc + hd, slot = pn % PS;
                if (!__all_sync(0xffffffffu, mbar_wait(prod_full(slot), (pn / PS) & 1, &g_fps_error, 1u))) {
                    ok = false;
                    break;
                }
                if (kTmaH && qc > 0) {
                    // the previous chunk's store has read this head's tile
                    if (rl == 0) {
                        bulk_wait_group_read0();
                        mbar_arrive(h_free(hd));
                    }
                    if (!__all_sync(0xffffffffu, mbar_wait(h_free(hd), (qc - 1) & 1, &g_fps_error, 1u))) {
                        ok = false;
                        break;
                    }
                }
                tc_fence_after();
                const uint32_t acc = lane_base + 128 + slot * kCols;
                __nv_bfloat16* hp = hiddens + (((int64_t)bh * q.nc + c) * q.N + rl) * q.P;
                // row rl of the 128-byte-swizzled tile: 16-byte chunk j at (j ^ (rl % 8)) * 16
                uint8_t* trow = htile + hd * kPHBytes + rl * kRowBytes;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    __syncwarp();
                    uint32_t sv[16], d[16];
                    tmem_ld_x16(sa + 16 * jj, sv);
                    tmem_ld_x16(acc + 16 * jj, d);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        d[k] = __float_as_uint(fmaf(e, __uint_as_float(sv[k]), __uint_as_float(d[k])));
                    tmem_st_x16(sa + 16 * jj, d);
                    if (kMode == kModeLocal) {
                        // no hiddens in the local pass
                    } else if (kTmaH) {
                        if (nok) {
                            uint4 w0, w1;
                            w0.x = pack_bf16(__uint_as_float(sv[0]), __uint_as_float(sv[1]));
                            w0.y = pack_bf16(__uint_as_float(sv[2]), __uint_as_float(sv[3]));
                            w0.z = pack_bf16(__uint_as_float(sv[4]), __uint_as_float(sv[5]));
                            w0.w = pack_bf16(__uint_as_float(sv[6]), __uint_as_float(sv[7]));
                            w1.x = pack_bf16(__uint_as_float(sv[8]), __uint_as_float(sv[9]));
                            w1.y = pack_bf16(__uint_as_float(sv[10]), __uint_as_float(sv[11]));
                            w1.z = pack_bf16(__uint_as_float(sv[12]), __uint_as_float(sv[13]));
                            w1.w = pack_bf16(__uint_as_float(sv[14]), __uint_as_float(sv[15]));
                            *reinterpret_cast<uint4*>(trow + (((2 * jj) ^ (rl & 7)) << 4)) = w0;
                            *reinterpret_cast<uint4*>(trow + (((2 * jj + 1) ^ (rl & 7)) << 4)) = w1;
                        }
                    } else if (nok && 16 * jj < q.P) {
                        uint4 w0, w1;
                        w0.x = pack_bf16(__uint_as_float(sv[0]), __uint_as_float(sv[1]));
                        w0.y = pack_bf16(__uint_as_float(sv[2]), __uint_as_float(sv[3]));
                        w0.z = pack_bf16(__uint_as_float(sv[4]), __uint_as_float(sv[5]));
                        w0.w = pack_bf16(__uint_as_float(sv[6]), __uint_as_float(sv[7]));
                        w1.x = pack_bf16(__uint_as_float(sv[8]), __uint_as_float(sv[9]));
                        w1.y = pack_bf16(__uint_as_float(sv[10]), __uint_as_float(sv[11]));
                        w1.z = pack_bf16(__uint_as_float(sv[12]), __uint_as_float(sv[13]));
                        w1.w = pack_bf16(__uint_as_float(sv[14]), __uint_as_float(sv[15]));
                        uint4* hdst = reinterpret_cast<uint4*>(hp + 16 * jj);
                        hdst[0] = w0;
                        hdst[1] = w1;
                    }
                }
                if (kTmaH) {
                    fence_proxy_async_smem();   // tile writes -> the TMA store
                    __syncwarp();
                    if (lane == 0) mbar_arrive(h_full(hd));
                }
                __syncwarp();
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(prod_empty(slot));
                if (kTmaH) {
                    bool okh = true;
                    if (rl == 0) {
                        okh = mbar_wait(h_full(hd), qc & 1, &g_fps_error, 1u);
                        if (okh) {
                            tma_store_3d(&tm_h, smem_u32(htile + hd * kPHBytes), 0, 0, bh * q.nc + c);
                            bulk_commit_group();
                        }
                    }
                    if (!__all_sync(0xffffffffu, okh)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!__all_sync(0xffffffffu, ok)) break;
            const bool last = u.c1 == q.nc;
            if (kMode == kModeLocal) {
                // the piece's end state and log2 decay, for the scan
                float* dst = agg + aslot * kSlotFloats;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    __syncwarp();
                    uint32_t sv[16];
                    tmem_ld_x16(sa + 16 * jj, sv);
                    tmem_wait_ld();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        __stcg(reinterpret_cast<float4*>(dst + ((4 * jj + q4) * 128 + rl) * 4),
                               make_float4(__uint_as_float(sv[4 * q4]), __uint_as_float(sv[4 * q4 + 1]),
                                           __uint_as_float(sv[4 * q4 + 2]), __uint_as_float(sv[4 * q4 + 3])));
                }
                if (rl == 0) agg_lsum[aslot] = lsum;
            } else if (kMode == kModeApply) {
                // final_state comes from the scan
            } else if (last) {
                if (final_state != nullptr) {
                    const int pl = nok ? q.P : 0;
#pragma unroll
                    for (int jj = 0; jj < kCols / 16; ++jj) {
                        __syncwarp();
                        uint32_t sv[16];
                        tmem_ld_x16(sa + 16 * jj, sv);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (16 * jj + k < pl)
                                final_state[sbase + (int64_t)(16 * jj + k) * q.N + rl] = __uint_as_float(sv[k]);
                    }
                }
            } else {
                float* dst = ring + ((int64_t)ch * 2 + (rk & 1)) * kSlotFloats;
#pragma unroll
                for (int jj = 0; jj < kCols / 16; ++jj) {
                    __syncwarp();
                    uint32_t sv[16];
                    tmem_ld_x16(sa + 16 * jj, sv);
                    tmem_wait_ld();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        __stcg(reinterpret_cast<float4*>(dst + ((4 * jj + q4) * 128 + rl) * 4),
                               make_float4(__uint_as_float(sv[4 * q4]), __uint_as_float(sv[4 * q4 + 1]),
                                           __uint_as_float(sv[4 * q4 + 2]), __uint_as_float(sv[4 * q4 + 3])));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(fold_done(hd));
                bool okp = true;
                if (rl == 0) {
                    okp = mbar_wait(fold_done(hd), 0, &g_fps_error, 1u);
                    if (okp && *reinterpret_cast<volatile unsigned int*>(&g_fps_withhold) == 0u) {
                        __threadfence();
                        st_release_gpu(flags + ch, (unsigned)u.c1);
                    }
                }
                if (!__shfl_sync(0xffffffffu, okp, 0)) break;
            }
        }
        if (kTmaH && rl == 0) bulk_wait_group0();   // the hiddens stores have completed
    }
    __syncwarp();   // lanes that skipped a role loop wait for its lane 0
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) report_timeout_to_host(&g_fps_error, q.host_err);
    if (warp == 1) {
        __syncwarp();  // lane 0 ran the MMA loop alone: reconverge before the collective
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// The scan between the two passes (CUDA cores).  Thread = one element of a
// chain's state in the aggregate-slot layout (float4 column group, TMEM lane,
// component); blockIdx.y = the chain: batch * H + head for the paired kernel
// (its chains are head pairs, its slots per head), the chain itself for the
// one-head kernel (a 128-row block of N by a 64-column block of P of one
// head).  It walks the chain's pieces in chunk order (ranges k = the one
// holding the chain's first unit, k + 1, ...): start = S, S <- 2^{sum} S + A,
// with the piece's start state written over A.  S begins at init_state (or
// zero) and ends as final_state.  The pieces' slots and decays are staged in
// shared memory, kScanBatch at a time, and each thread loads the batch's A
// values before its serial fma chain, so that the loads overlap instead of
// queueing behind one another.
constexpr int kScanBatch = 32;
template <bool kPair>
__global__ void __launch_bounds__(256)
fwd_pass_state_scan(const float* init, float* agg, const float* __restrict__ agg_lsum,
                    float* final_state, const FpsParams q) {
    __shared__ int s_slot[kScanBatch];
    __shared__ float s_decay[kScanBatch];
    grid_launch_dependents();   // chained launch: the apply pass may set up meanwhile
    grid_dependency_wait();     // the local pass's aggregates
    const int f = blockIdx.x * blockDim.x + threadIdx.x;
    int pc, hd, bh, n, p;
    if (kPair) {
        bh = blockIdx.y; pc = bh >> 1; hd = bh & 1;
        n = (f >> 2) & 127;
        p = (f >> 9) * 4 + (f & 3);
    } else {
        pc = blockIdx.y; hd = 0;
        const int rb = pc / q.npb, pb = pc - rb * q.npb;
        bh = rb / q.nmb;
        const int mb = rb - bh * q.nmb;
        n = mb * 128 + ((f >> 2) & 127);
        p = pb * kCols + (f >> 9) * 4 + (f & 3);
    }
    const bool live = f < kSlotFloats;
    const bool valid = live && p < q.P && n < q.N;
    const int64_t sidx = ((int64_t)bh * q.P + p) * q.N + n;
    float S = (init != nullptr && valid) ? init[sidx] : 0.f;
    const int u0 = pc * q.nc, u1 = u0 + q.nc;   // the chain's units
    auto range_lo = [&](int k) { return (int)((long long)k * q.W / q.G); };
    int k0 = (int)((long long)u0 * q.G / q.W);
    while (k0 + 1 < q.G && range_lo(k0 + 1) <= u0) ++k0;
    while (k0 > 0 && range_lo(k0) > u0) --k0;
    int k1 = k0;                                 // one past the chain's last range
    while (k1 < q.G && range_lo(k1) < u1) ++k1;
    for (int kb = k0; kb < k1; kb += kScanBatch) {
        const int nb = min(kScanBatch, k1 - kb);
        __syncthreads();   // the previous batch's table has been read
        if ((int)threadIdx.x < nb) {
            const int k = kb + (int)threadIdx.x;
            const int piece = 2 * k + (range_lo(k) / q.nc == pc ? 0 : 1);
            const int slot = kPair ? piece * 2 + hd : piece;
            s_slot[threadIdx.x] = slot;
            s_decay[threadIdx.x] = exp2f(__ldcg(agg_lsum + slot));
        }
        __syncthreads();
        if (!live) continue;
        for (int i0 = 0; i0 < nb; i0 += 8) {
            float Av[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                Av[i] = i0 + i < nb ? __ldcg(agg + (int64_t)s_slot[i0 + i] * kSlotFloats + f) : 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i0 + i < nb) {
                    __stcg(agg + (int64_t)s_slot[i0 + i] * kSlotFloats + f, S);
                    S = fmaf(s_decay[i0 + i], S, Av[i]);
                }
            }
        }
    }
    if (final_state != nullptr && valid) final_state[sidx] = S;
}

int64_t chains(const Problem& p) { return p.b * p.H * ((p.N + 127) / 128) * ((p.P + 63) / 64); }
size_t ring_bytes(const Problem& p) {
    return round_up256((size_t)chains(p) * 2 * kSlotFloats * sizeof(float));
}
size_t ctrl_bytes(const Problem& p) {
    return round_up256((size_t)(kCtrlFlagOffset + chains(p)) * sizeof(unsigned int));
}

// Resident CTA slots of the current device, from the SM count and this
// kernel's per-CTA needs (shared memory, registers, TMEM), cached per device.
// (The occupancy calculator reports one CTA per SM for this kernel, while two
// run side by side.)
cudaError_t resident_ctas(int* out) {
    static int cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) {
        *out = cached[dev];
        return cudaSuccess;
    }
    int sms = 0, smem_sm = 0, regs_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) !=
            cudaSuccess)
        return e;
    int per_sm = std::min(smem_sm / (smem_bytes<true>() + 1024), 512 / kTmemCols);
    per_sm = std::min(per_sm, regs_sm / (kThreads * kMaxRegs));
    per_sm = std::max(1, std::min(per_sm, kMinBlocks));
    *out = sms * per_sm;
    if (dev >= 0 && dev < 64) cached[dev] = *out;
    return cudaSuccess;
}

// The paired kernel serves inputs whose state block fits one chain (N <= 128,
// P <= 64) and whose groups hold an even number of heads, so that heads 2k
// and 2k+1 read the same B.
bool pair_geometry(const Problem& p) {
    return p.N <= 128 && p.P <= 64 && p.H % 2 == 0 && p.hpg % 2 == 0;
}
bool paired(const Problem& p) { return pair_geometry(p); }

// Two passes for long chains (the local and apply modes with the scan between
// them), with an initial state or without, for either kernel.  The workspace
// holds kAggSlots aggregate slots whenever a problem could take this path:
// enough for 256 ranges of the paired kernel (four slots each: two pieces by
// two heads) or 512 of the one-head kernel (two each).  Whether a problem takes
// it depends on the device's SM count (a range must not span more than two
// chains).
constexpr int kTwoPassMinChunks = 64;
constexpr int kAggSlots = 1024;
bool two_pass_candidate(const Problem& p) {
    return p.dtype == SSD_BF16 && p.nc >= kTwoPassMinChunks;
}
size_t agg_state_bytes() { return round_up256((size_t)kAggSlots * kSlotFloats * 4); }
size_t agg_bytes(const Problem& p) {
    return two_pass_candidate(p) ? agg_state_bytes() + round_up256((size_t)kAggSlots * 4) : 0;
}
// Ranges of at most half a chain (so that every chain spans two or more
// ranges and no range spans more than two chains), within the slot capacity.
bool two_pass_fits(int64_t W, int64_t G, int64_t nc, int slots_per_range) {
    return G > 0 && (W + G - 1) / G <= nc / 2 && G * slots_per_range <= kAggSlots;
}

}  // namespace

size_t fwd_pass_state_scratch_bytes(const Problem& p) {
    if (p.dtype != SSD_BF16 || p.b == 0 || p.L == 0) return 0;
    return ring_bytes(p) + ctrl_bytes(p) + agg_bytes(p);
}
size_t fwd_pass_state_ctrl_offset(const Problem& p) { return ring_bytes(p); }
size_t fwd_pass_state_ctrl_bytes(const Problem& p) { return ctrl_bytes(p); }

cudaError_t launch_fwd_pass_state_tc(const Problem& p, const void* x, const void* B,
                                     const float* Gcs, const float* dtT, const float* init,
                                     void* hiddens, float* final_state, void* scratch,
                                     cudaStream_t stream) {
    float* ring = (float*)scratch;
    unsigned int* ctrl = (unsigned int*)((char*)scratch + ring_bytes(p));
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
    FpsParams q;
    q.H = (int)p.H; q.P = (int)p.P; q.N = (int)p.N; q.Q = (int)p.Q; q.nc = (int)p.nc;
    q.Lp = (int)p.Lp; q.hpg = (int)p.hpg;
    q.nmb = (int)((p.N + 127) / 128);
    q.npb = (int)((p.P + 63) / 64);
    q.nchains = (int)chains(p);
    q.host_err = host_timeout_word();
    if ((int64_t)q.nchains * p.nc >= (int64_t)1 << 31) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.chained ? 1 : 0;
    cudaError_t e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    float* agg = two_pass_candidate(p) ? (float*)((char*)scratch + ring_bytes(p) + ctrl_bytes(p)) : nullptr;
    float* lsum = agg != nullptr ? (float*)((char*)agg + agg_state_bytes()) : nullptr;
    if (paired(p)) {
        const int64_t W2 = (int64_t)(q.nchains / 2) * p.nc;
        const int64_t G2 = std::min<int64_t>(std::min<int64_t>(W2, sms), kAggSlots / 4);
        const bool two_pass = two_pass_candidate(p) && two_pass_fits(W2, G2, p.nc, 4) &&
                              p.b * p.H <= 65535;   // the scan's grid rows
        // one CTA per SM; a chain is a pair of heads (its flags and hand-off
        // slots stay per head: chains() counts heads)
        // P = 64: hiddens leave through TMA stores of [N rows][64 p] tiles
        const bool tma_h = p.P == 64;
        CUtensorMap th;
        memset(&th, 0, sizeof(th));
        if (tma_h) {
            const uint64_t hd[3] = {(uint64_t)p.P, (uint64_t)p.N, (uint64_t)(p.b * p.H * p.nc)};
            const uint64_t hs[2] = {(uint64_t)p.P * 2, (uint64_t)p.N * p.P * 2};
            const uint32_t hbox[3] = {64, (uint32_t)p.N, 1};
            if (!encode_tmap(&th, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, hiddens, hd, hs, hbox,
                             CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
        }
        q.nchains /= 2;
        q.W = q.nchains * q.nc;
        q.G = two_pass ? (int)G2 : std::min(q.W, sms);
        cfg.gridDim = dim3((unsigned)q.G);
        cfg.blockDim = dim3(kPThreads);
        using PairKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, const float*, const float*,
                                    const float*, __nv_bfloat16*, float*, float*, unsigned int*, float*,
                                    float*, FpsParams);
        auto launch_pair = [&](PairKernel pk, int psmem, float* agg, float* lsum) -> cudaError_t {
            cudaError_t le;
            if ((le = cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem)) !=
                    cudaSuccess ||
                (le = cudaFuncSetAttribute(pk, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
                return le;
            cfg.dynamicSmemBytes = (size_t)psmem;
            le = cudaLaunchKernelEx(&cfg, pk, tx, tb, th, two_pass ? nullptr : init, Gcs, dtT,
                                    (__nv_bfloat16*)hiddens, final_state, ring, ctrl, agg, lsum, q);
            return le != cudaSuccess ? le : cudaGetLastError();
        };
        if (!two_pass)
            return tma_h ? launch_pair(fwd_pass_state_pair_tc<true, kModeHandoff>, pair_smem<true>(),
                                       nullptr, nullptr)
                         : launch_pair(fwd_pass_state_pair_tc<false, kModeHandoff>, pair_smem<false>(),
                                       nullptr, nullptr);
        if ((e = launch_pair(fwd_pass_state_pair_tc<false, kModeLocal>, pair_smem<false>(), agg,
                             lsum)) != cudaSuccess)
            return e;
        if ((e = launch_chained(fwd_pass_state_scan<true>, dim3((kSlotFloats + 255) / 256, (unsigned)(p.b * p.H)),
                                dim3(256), 0, stream, p.chained, init, agg, (const float*)lsum, final_state,
                                q)) != cudaSuccess)
            return e;
        cfg.numAttrs = p.chained ? 1 : 0;   // the apply pass may set up while the scan runs
        return tma_h ? launch_pair(fwd_pass_state_pair_tc<true, kModeApply>, pair_smem<true>(), agg, lsum)
                     : launch_pair(fwd_pass_state_pair_tc<false, kModeApply>, pair_smem<false>(), agg,
                                   lsum);
    }
    // one-head kernel: two CTAs per SM
    int resident = 0;
    if ((e = resident_ctas(&resident)) != cudaSuccess) return e;
    q.W = q.nchains * q.nc;
    const int64_t G1 = std::min<int64_t>(std::min<int64_t>(q.W, resident), kAggSlots / 2);
    const bool two_pass = two_pass_candidate(p) && two_pass_fits(q.W, G1, p.nc, 2) &&
                          q.nchains <= 65535;   // the scan's grid rows
    q.G = two_pass ? (int)G1 : std::min(q.W, resident);
    cfg.gridDim = dim3((unsigned)q.G);
    cfg.blockDim = dim3(kThreads);
    // P a multiple of 64: the chunk-start states leave as TMA stores of
    // [min(N, 128) rows][64 p] blocks (rows past N are clipped by the TMA)
    const bool tma_h = p.P % 64 == 0;
    CUtensorMap th;
    memset(&th, 0, sizeof(th));
    if (tma_h) {
        const uint64_t hd[3] = {(uint64_t)p.P, (uint64_t)p.N, (uint64_t)(p.b * p.H * p.nc)};
        const uint64_t hs[2] = {(uint64_t)p.P * 2, (uint64_t)p.N * p.P * 2};
        const uint32_t hbox[3] = {64, (uint32_t)std::min<int64_t>(p.N, 128), 1};
        if (!encode_tmap(&th, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, hiddens, hd, hs, hbox,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    using OneKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, const float*, const float*,
                               const float*, __nv_bfloat16*, float*, float*, unsigned int*, float*,
                               float*, FpsParams);
    auto launch_one = [&](OneKernel k1, int smem, const float* init_in, float* fin, float* ag,
                          float* ls) -> cudaError_t {
        cudaError_t le;
        if ((le = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
                cudaSuccess ||   // all of the unified L1/shared storage as shared memory
            (le = cudaFuncSetAttribute(k1, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return le;
        cfg.dynamicSmemBytes = (size_t)smem;
        le = cudaLaunchKernelEx(&cfg, k1, tx, tb, th, init_in, Gcs, dtT, (__nv_bfloat16*)hiddens, fin,
                                ring, ctrl, ag, ls, q);
        return le != cudaSuccess ? le : cudaGetLastError();
    };
    if (!two_pass) {
        if (init != nullptr)
            return launch_one(fwd_pass_state_tc<true, kModeHandoff, false>, smem_bytes<true>(), init,
                              final_state, nullptr, nullptr);
        return tma_h ? launch_one(fwd_pass_state_tc<false, kModeHandoff, true>, smem_bytes<false, true>(),
                                  nullptr, final_state, nullptr, nullptr)
                     : launch_one(fwd_pass_state_tc<false, kModeHandoff, false>, smem_bytes<false>(),
                                  nullptr, final_state, nullptr, nullptr);
    }
    if ((e = launch_one(fwd_pass_state_tc<false, kModeLocal, false>, smem_bytes<false>(), nullptr, nullptr,
                        agg, lsum)) != cudaSuccess)
        return e;
    if ((e = launch_chained(fwd_pass_state_scan<false>, dim3((kSlotFloats + 255) / 256, (unsigned)q.nchains),
                            dim3(256), 0, stream, p.chained, init, agg, (const float*)lsum, final_state,
                            q)) != cudaSuccess)
        return e;
    return tma_h ? launch_one(fwd_pass_state_tc<false, kModeApply, true>, smem_bytes<false, true>(), nullptr,
                              nullptr, agg, lsum)
                 : launch_one(fwd_pass_state_tc<false, kModeApply, false>, smem_bytes<false>(), nullptr,
                              nullptr, agg, lsum);
}

cudaError_t set_fwd_pass_state_withhold(unsigned int on) {
    return cudaMemcpyToSymbol(g_fps_withhold, &on, sizeof(on));
}

unsigned int take_fwd_pass_state_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_fps_error, sizeof(v)) != cudaSuccess) return ~0u;
    cudaMemcpyToSymbol(g_fps_error, &zero, sizeof(zero));
    return v;
}

}  // namespace ssd
