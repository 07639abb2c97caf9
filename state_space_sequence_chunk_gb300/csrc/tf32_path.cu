// tf32_path.cu -- steps 2 and 3 of the SSD forward pass for fp32 inputs on the
// tcgen05 tensor cores (kind::tf32, fp32 accumulation in tensor memory).
//
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", sections "Kernel 2: fwd_pass_state" and "Kernel 3: compute_out"
// (the zhiding.cn rendering, section "compute_out", runs the last product as
// a TF32 dot).  Here every product of both steps is a TF32 tensor-core MMA:
//
//   chunk products  D_c^T (N x P) = (B_c o s)^T X_c,  s_q = dt_q 2^{g_last - g_q},
//                   written into chunk c's hiddens slot; the CUDA-core state
//                   scan then turns the slots into the chunk-start states
//                   (hiddens[c] <- S, S <- 2^{g_last} S + D_c), the only
//                   serial step of "Kernel 2";
//   compute_out     per 128-row query block I of a chunk:
//                     acc = C_I h^T
//                     for each key block J <= I:  S = C_I B_J^T,
//                       A = S o 2^{g_i - g_j} [j <= i]  (in tensor memory),
//                       acc = 2^{g_i} acc (before the first block),
//                       acc += A (dt o X_J)
//                     y = acc + D x.
//
// Operands.  tcgen05 reads TF32 operands K-major (the contraction index
// contiguous), so the CUDA-core threads write every tile into a 128-byte-
// swizzled K-major shared-memory layout, transposing where the tensor is
// stored the other way (h, X, and B for the chunk products) and rounding each
// value to TF32 on the way (cvt.rna: to nearest).  Rounding matters: the
// tensor core ignores the low 13 mantissa bits of an fp32 operand, and that
// truncation's bias, summed over a chunk, exceeds the 1e-3 bound on the small
// fp32 workload in an emulation of this arithmetic (1.3e-3 truncated against
// 4.2e-4 rounded).
//
// Work: one CTA of 128 threads per unit -- (batch*head, chunk) for the chunk
// products, (batch, chunk, head, query block) for compute_out; thread r owns
// tensor-memory lane r.  A unit's MMAs form a short chain, each issued by
// thread 0 and completed on an mbarrier that every thread waits on (bounded:
// a wait that gives up sets bit 0 of g_tf32_error and the CTA skips to its
// end).  Several CTAs share an SM, which overlaps one unit's operand writes
// with another's MMAs.
//
// Supported: fp32, N <= 128 (the state rows are the MMA's M = 128), P <= 128,
// any chunk size of the ABI; compute_out takes keys in blocks of min(Q, 128).
#include <algorithm>

#include "sm100_ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

__device__ unsigned int g_tf32_error;  // bit 0: a bounded wait gave up

constexpr int kThreads = 128;
// Registers are held to 65536 / (4 x 128) = 128 per thread, so that the
// register file is not what limits the CTAs per SM to fewer than four (the
// number that the tensor memory and the shared memory allow on the small
// shapes: a grid of 512 CTAs then runs in one wave on 152 SMs)
constexpr int kCtasPerSm = 4;
constexpr int kRowBytes = 128;   // one swizzle row: 32 fp32 values of K

__device__ __forceinline__ uint32_t to_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return r;
}

// Byte offset of element (r, k) in a K-major, 128-byte-swizzled tile of
// `rows` rows (a multiple of 8) of 4-byte values: K runs in atoms of 32 values
// (one 128-byte row each), rows in groups of 8 (1024 bytes); within a row the
// 16-byte chunk index is XORed with the row's index in its group.
__device__ __forceinline__ uint32_t swz(int r, int k, int rows) {
    return (uint32_t)((k >> 5) * rows * kRowBytes + (r >> 3) * 1024 + (r & 7) * kRowBytes +
                      ((((k & 31) >> 2) ^ (r & 7)) << 4) + (k & 3) * 4);
}

// Descriptor of K-step kk (8 values of K = 32 bytes) of such a tile.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk, int rows) {
    return smem_desc_sw128(tile + (uint32_t)((kk >> 2) * rows * kRowBytes + (kk & 3) * 32), 16,
                           8 * kRowBytes);
}

// Bytes of a tile of `rows` rows and K values (K rounded up to a 32-value atom).
__host__ __device__ constexpr int tile_bytes(int rows, int K) { return ((K + 31) / 32) * rows * kRowBytes; }
__host__ __device__ constexpr int up1024(int v) { return (v + 1023) / 1024 * 1024; }

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ float4 ldg4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }

// Column groups of a transposed tile that one warp covers: warp w takes the
// 4-column groups w, w + 4, w + 8, ... of `cols` (<= 128) columns.
constexpr int kMaxGroups = 8;

// Load this lane's row `src` (K index = the lane's k) for the warp's column
// groups into registers; nothing is stored yet, so every load is in flight
// at once.
__device__ __forceinline__ void load_groups(float4 (&v)[kMaxGroups], const float* src, bool valid,
                                            int cols, int warp) {
#pragma unroll
    for (int u = 0; u < kMaxGroups; ++u) {
        const int c4 = warp + 4 * u;
        v[u] = (valid && 4 * c4 < cols) ? ldg4(src + 4 * c4) : zero4();
    }
}
// Store them transposed: tile[4 c4 + e][k] = tf32(v.e * scale).
__device__ __forceinline__ void store_groups(const float4 (&v)[kMaxGroups], uint32_t tile, int rows,
                                             int k, float scale, int cols, int warp) {
#pragma unroll
    for (int u = 0; u < kMaxGroups; ++u) {
        const int c4 = warp + 4 * u;
        if (4 * c4 < cols) {
            st_shared_u32(tile + swz(4 * c4 + 0, k, rows), to_tf32(v[u].x * scale));
            st_shared_u32(tile + swz(4 * c4 + 1, k, rows), to_tf32(v[u].y * scale));
            st_shared_u32(tile + swz(4 * c4 + 2, k, rows), to_tf32(v[u].z * scale));
            st_shared_u32(tile + swz(4 * c4 + 3, k, rows), to_tf32(v[u].w * scale));
        }
    }
}

// Wait for the next phase of `bar`; `ok` turns false (for good) once a wait
// has given up, after which the remaining waits return at once.
__device__ __forceinline__ void chain_wait(uint32_t bar, uint32_t& phase, bool& ok) {
    if (ok) ok = mbar_wait(bar, phase, &g_tf32_error, 1u);
    phase ^= 1u;
}

// Power-of-two TMEM allocation (>= 32 columns) holding `cols` columns.
__host__ __device__ constexpr uint32_t tmem_cols_for(int cols) {
    uint32_t a = 32;
    while ((int)a < cols) a <<= 1;
    return a;
}

// ===========================================================================
// Chunk products: one CTA per (chunk, batch*head).
//   D_c^T[n][p] = sum_q tf32(B_q[n] s_q) tf32(x_q[p])
// K (the chunk's tokens) runs in 32-token sub-blocks through two buffers:
// the tiles of sub-block k + 1 are written while the MMAs of sub-block k run.
// ===========================================================================
struct FpsTf32 {
    int L, H, P, N, G, Q, nc, Lp, hpg;
    uint32_t tmem_cols;
    int a_bytes, x_bytes;   // one buffer's A tile (128 rows x 32) and X^T tile (P rows x 32)
};

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
fps_products_tf32(const float* __restrict__ x, const float* __restrict__ B,
                  const float* __restrict__ Gcs, const float* __restrict__ dtT,
                  float* __restrict__ hiddens, const FpsTf32 q, unsigned int* host_err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t s0 = smem_u32(smem);
    const uint32_t buf_bytes = (uint32_t)(q.a_bytes + q.x_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * buf_bytes);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, bh = blockIdx.y, b = bh / q.H, h = bh % q.H, grp = h / q.hpg;

    if (tid == 0) {
        mbar_init(smem_u32(bars), 1);
        mbar_init(smem_u32(bars + 1), 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_holder), q.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // chained launch: the next grid may start (every CTA of this one holds its
    // TMEM already); G and dt come from chunk_cumsum
    grid_launch_dependents();
    grid_dependency_wait();

    const float* grow = Gcs + (int64_t)bh * q.Lp + (int64_t)c * q.Q;
    const float* drow = dtT + (int64_t)bh * q.Lp + (int64_t)c * q.Q;
    const float glast = grow[q.Q - 1];   // padded slots repeat the last real token's value
    const int nsub = q.Q / 32;
    const uint32_t idesc = make_idesc(2, 128, (uint32_t)q.P, 0, 0);
    uint32_t ph0 = 0u, ph1 = 0u;   // next phase to wait for, per buffer
    bool ok = true;
    for (int sb = 0; sb < nsub; ++sb) {
        const int buf = sb & 1;
        // lane <-> token of the sub-block (the K index), warps <-> groups of 4
        // columns; the loads are issued before waiting for a free buffer
        const int t = c * q.Q + sb * 32 + lane;
        const bool valid = t < q.L;
        float4 vb[kMaxGroups], vx[kMaxGroups];
        load_groups(vb, B + (((int64_t)b * q.L + (valid ? t : 0)) * q.G + grp) * q.N, valid, q.N, warp);
        load_groups(vx, x + (((int64_t)b * q.L + (valid ? t : 0)) * q.H + h) * q.P, valid, q.P, warp);
        const float sc = valid ? drow[sb * 32 + lane] * exp2f(glast - grow[sb * 32 + lane]) : 0.f;
        if (sb >= 2) {   // sub-block sb-2's MMAs have consumed this buffer
            if (buf) chain_wait(smem_u32(bars + 1), ph1, ok);
            else chain_wait(smem_u32(bars), ph0, ok);
        }
        const uint32_t at = s0 + buf * buf_bytes, xt = at + q.a_bytes;
        if (ok) {
            store_groups(vb, at, 128, lane, sc, q.N, warp);   // A[n][q] = B_q[n] s_q
            store_groups(vx, xt, q.P, lane, 1.f, q.P, warp);  // X^T[p][q] = x_q[p]
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && ok) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32_ss(tmem, kmajor_desc(at, kk, 128), kmajor_desc(xt, kk, q.P), idesc,
                            (sb > 0 || kk > 0) ? 1u : 0u);
            mma_commit(smem_u32(bars + buf));
        }
    }
    // the last commit covers every MMA issued before it
    if ((nsub - 1) & 1) chain_wait(smem_u32(bars + 1), ph1, ok);
    else chain_wait(smem_u32(bars), ph0, ok);
    tc_fence_after();
    // D_c^T row n -> hiddens slot [n][p] of chunk c (rows n >= N are padding)
    __syncwarp();
    float* hrow = hiddens + ((int64_t)bh * q.nc + c) * (int64_t)q.N * q.P + (int64_t)tid * q.P;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    for (int p0 = 0; p0 < q.P; p0 += 16) {
        uint32_t v[16];
        tmem_ld_x16(tmem + lane_off + p0, v);
        tmem_wait_ld();
        if (ok && tid < q.N) {
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4*>(hrow + p0 + e) =
                    make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) report_timeout_to_host(&g_tf32_error, host_err);
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, q.tmem_cols);
    }
}

// ===========================================================================
// compute_out: one CTA per (query block I, chunk, batch*head).
// ===========================================================================
struct CoTf32 {
    int L, H, P, N, G, Q, nc, Lp, hpg;
    int KB;                      // keys per block: min(Q, 128)
    int nblk;                    // query blocks per chunk: Q / 128 (1 for Q <= 128)
    int pt, npt;                 // columns of P per CTA (<= 64 when P > 64), column tiles
    int crows;                   // rows of the C_I tile: min(Q, 128)
    uint32_t tmem_cols;
    uint32_t scol;               // first TMEM column of S / A (acc holds columns [0, pt))
    int c_bytes, b_bytes, h_bytes, x_bytes;   // C_I, B_J, h^T, (dt o X_J)^T tiles
    int x_sep;                   // 1: (dt o X)^T has a tile of its own (written up front);
                                 // 0: it reuses h^T's, once C h^T is done
    int kh, nks;                 // state columns per pass of the C h^T / C B^T products, passes
};

// A K-major tile whose rows are consecutive tokens of a [token][group][N]
// tensor (C or B: already K-major in memory).  Rows past `nvalid` are zero.
// Each thread issues a batch of 8 loads before its stores.
__device__ __forceinline__ void put_rows(uint32_t tile, int rows, const float* base, int64_t row_stride,
                                         int nvalid, int N, int tid) {
    const int n4s = N / 4, total = rows * n4s;
    for (int e0 = tid; e0 < total; e0 += kThreads * 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * kThreads, r = e / n4s, n4 = e - r * n4s;
            v[u] = (e < total && r < nvalid) ? ldg4(base + r * row_stride + 4 * n4) : zero4();
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + u * kThreads, r = e / n4s, n4 = e - r * n4s;
            if (e < total)
                st_shared_v4(tile + swz(r, 4 * n4, rows), to_tf32(v[u].x), to_tf32(v[u].y),
                             to_tf32(v[u].z), to_tf32(v[u].w));
        }
    }
}

// put_rows' tile copied by cp.async instead (16-byte pieces of raw fp32, rows
// past `nvalid` zeroed), so that the loads of the other tiles need not wait
// for it; round_rows then rounds it to TF32 in place once the copies have
// landed, each thread the pieces it copied itself.
__device__ __forceinline__ void async_rows(uint32_t tile, int rows, const float* base, int64_t row_stride,
                                           int nvalid, int N, int tid) {
    const int n4s = N / 4, total = rows * n4s;
    for (int e = tid; e < total; e += kThreads) {
        const int r = e / n4s, n4 = e - r * n4s;
        const uint32_t dst = tile + swz(r, 4 * n4, rows);
        if (r < nvalid) cp_async_16(dst, base + r * row_stride + 4 * n4, 16u);
        else st_shared_v4(dst, 0u, 0u, 0u, 0u);
    }
}
__device__ __forceinline__ void round_rows(uint32_t tile, int rows, int N, int tid) {
    const int n4s = N / 4, total = rows * n4s;
    for (int e = tid; e < total; e += kThreads) {
        const int r = e / n4s, n4 = e - r * n4s;
        const uint32_t a = tile + swz(r, 4 * n4, rows);
        uint32_t v0, v1, v2, v3;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                     : "r"(a)
                     : "memory");
        st_shared_v4(a, to_tf32(__uint_as_float(v0)), to_tf32(__uint_as_float(v1)),
                     to_tf32(__uint_as_float(v2)), to_tf32(__uint_as_float(v3)));
    }
}

// A transposed K-major tile: tile[p][k] = tf32(scale(k) * src(k)[p]) for
// k < Kdim and p < cols (a multiple of 4); src(k) is NULL for a zero row.
// The warps take blocks of 32 values of k by 16 columns in turn: lane l reads
// the four source rows k = 4 (l % 8) + i at columns 4 (l / 8) + e (16 bytes
// each), transposes the 4 x 4 values in registers and writes each column's
// four values of k as one 16-byte store; the eight lanes of a store phase then
// fill eight different 16-byte chunks of one tile row.  Up to four blocks (16
// loads per lane) are in flight before their stores.
template <typename Src, typename Scale>
__device__ __forceinline__ void put_transposed(uint32_t tile, int rows, int Kdim, int cols, Src src,
                                               Scale scale, int lane, int warp) {
    constexpr int kWarps = kThreads / 32;
    const int ncb = (cols + 15) / 16, nblk = (Kdim + 31) / 32 * ncb;
    const int kl = 4 * (lane & 7), cl = 4 * (lane >> 3);
    for (int b0 = warp; b0 < nblk; b0 += 4 * kWarps) {
        float4 v[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int blk = b0 + m * kWarps, kb = blk / ncb;
            const int k = 32 * kb + kl, c = 16 * (blk - kb * ncb) + cl;
            const bool live = blk < nblk && c < cols;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float* sp = (live && k + i < Kdim) ? src(k + i) : nullptr;
                v[m][i] = sp ? ldg4(sp + c) : zero4();
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int blk = b0 + m * kWarps, kb = blk / ncb;
            const int k = 32 * kb + kl, c = 16 * (blk - kb * ncb) + cl;
            if (blk < nblk && c < cols && k < Kdim) {
                float sc[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) sc[i] = k + i < Kdim ? scale(k + i) : 0.f;
                st_shared_v4(tile + swz(c, k, rows), to_tf32(v[m][0].x * sc[0]), to_tf32(v[m][1].x * sc[1]),
                             to_tf32(v[m][2].x * sc[2]), to_tf32(v[m][3].x * sc[3]));
                st_shared_v4(tile + swz(c + 1, k, rows), to_tf32(v[m][0].y * sc[0]), to_tf32(v[m][1].y * sc[1]),
                             to_tf32(v[m][2].y * sc[2]), to_tf32(v[m][3].y * sc[3]));
                st_shared_v4(tile + swz(c + 2, k, rows), to_tf32(v[m][0].z * sc[0]), to_tf32(v[m][1].z * sc[1]),
                             to_tf32(v[m][2].z * sc[2]), to_tf32(v[m][3].z * sc[3]));
                st_shared_v4(tile + swz(c + 3, k, rows), to_tf32(v[m][0].w * sc[0]), to_tf32(v[m][1].w * sc[1]),
                             to_tf32(v[m][2].w * sc[2]), to_tf32(v[m][3].w * sc[3]));
            }
        }
    }
}

// kGdn: the same kernel serves the Gated DeltaNet output chunk_fwd_o (Helion
// hackathon gallery, "GDN chunk_fwd_o"): o = e^{g} (q h) + causal((q k^T) o
// e^{g_i - g_j}) v_new -- C -> q, B -> k, x -> v_new, hiddens -> h, y -> o,
// one "group" per head, no dt (1) and no D; Gcs then points at the natural-log
// gate g [batch, T, H], scaled by log2(e) on load.
template <bool kGdn, bool kSplit>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
compute_out_tf32(const float* __restrict__ x, const float* __restrict__ B,
                 const float* __restrict__ C, const float* __restrict__ Gcs,
                 const float* __restrict__ dtT, const float* __restrict__ hiddens,
                 const float* __restrict__ D, float* __restrict__ y, const CoTf32 q,
                 unsigned int* host_err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t ct = smem_u32(smem);
    const uint32_t bt = ct + q.c_bytes;
    const uint32_t ht = bt + q.b_bytes;
    const uint32_t xt = q.x_sep ? ht + q.h_bytes : ht;
    float* gv = reinterpret_cast<float*>(smem + q.c_bytes + q.b_bytes + q.h_bytes +
                                         (q.x_sep ? q.x_bytes : 0));   // g[Q]
    float* dv = gv + q.Q;                                              // dt[Q]
    uint64_t* bar = reinterpret_cast<uint64_t*>(dv + q.Q);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int I = blockIdx.x / q.npt, c = blockIdx.y, bh = blockIdx.z;
    const int p0 = (blockIdx.x - I * q.npt) * q.pt;          // this CTA's columns of P
    const int pc = min(q.pt, q.P - p0);
    const int b = bh / q.H, h = bh % q.H, grp = h / q.hpg;
    const int t0 = c * q.Q;              // first token of the chunk
    const int i0 = I * 128;              // first query row of the block (in the chunk)
    const int64_t bc_stride = (int64_t)q.G * q.N;            // token stride of B and C
    const float* Cb = C + ((int64_t)b * q.L * q.G + grp) * q.N;
    const float* Bb = B + ((int64_t)b * q.L * q.G + grp) * q.N;
    const float* xb = x + ((int64_t)b * q.L * q.H + h) * q.P + p0;  // token t at xb + t H P
    const int64_t x_stride = (int64_t)q.H * q.P;

    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_holder), q.tmem_cols);
    grid_dependency_wait();   // chained launch: the state scan's output
    // C_I (rows = query rows) and B_0 (rows = keys) by cp.async, in flight while
    // the other operands are loaded.  With Q < 128 the C_I tile has Q rows;
    // the M = 128 products read 128 rows from it regardless, and the rows past
    // Q (whatever shared memory follows the tile) only reach accumulator lanes
    // that are never used.
    const int c_valid = min(min(q.Q - i0, 128), q.L - (t0 + i0));
    const int b_valid = min(q.KB, q.L - t0);
    // kSplit: the C h^T and C B^T products run in q.nks passes of q.kh state
    // columns, so that the tiles (and with them more CTAs) fit an SM; Q <= 128
    const int kh = kSplit ? q.kh : q.N;
    async_rows(ct, q.crows, Cb + (int64_t)(t0 + i0) * bc_stride, bc_stride, c_valid, kh, tid);
    async_rows(bt, q.KB, Bb + (int64_t)t0 * bc_stride, bc_stride, b_valid, kh, tid);
    cp_async_commit();
    for (int i = tid; i < q.Q; i += kThreads) {
        if (kGdn) {
            const int t = t0 + i;
            gv[i] = t < q.L ? Gcs[((int64_t)b * q.L + t) * q.H + h] * kLog2e : 0.f;
            dv[i] = 1.f;
        } else {
            gv[i] = Gcs[(int64_t)bh * q.Lp + t0 + i];
            dv[i] = dtT[(int64_t)bh * q.Lp + t0 + i];
        }
    }
    // h^T: rows = p, K = state n (hiddens holds [n][p])
    const float* hb = hiddens + ((int64_t)bh * q.nc + c) * (int64_t)q.N * q.P + p0;
    put_transposed(ht, pc, kh, pc, [&](int n) { return hb + (int64_t)n * q.P; },
                   [](int) { return 1.f; }, lane, warp);
    // (dt o X_J)^T: rows = p, K = keys of block J (zero past the sequence end)
    // (reads dv: the first call follows a barrier after dv is written; no
    // barrier inside, since later calls sit under the per-thread `ok`)
    auto put_x = [&](int J) {
        put_transposed(
            xt, pc, q.KB, pc,
            [&](int k) {
                const int t = t0 + J * q.KB + k;
                return t < q.L ? xb + (int64_t)t * x_stride : nullptr;
            },
            [&](int k) { return t0 + J * q.KB + k < q.L ? dv[J * q.KB + k] : 0.f; }, lane, warp);
    };
    if (q.x_sep) {
        __syncthreads();   // dv complete
        put_x(0);
    }
    cp_async_wait_all();
    round_rows(ct, q.crows, kh, tid);
    round_rows(bt, q.KB, kh, tid);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t acc = tmem, sreg = tmem + q.scol;
    const uint32_t idesc_p = make_idesc(2, 128, (uint32_t)pc, 0, 0);
    const uint32_t idesc_k = make_idesc(2, 128, (uint32_t)q.KB, 0, 0);
    const int nk_state = kh / 8;
    if (tid == 0) {
        for (int kk = 0; kk < nk_state; ++kk)
            mma_tf32_ss(acc, kmajor_desc(ct, kk, q.crows), kmajor_desc(ht, kk, pc), idesc_p,
                        kk > 0 ? 1u : 0u);
        for (int kk = 0; kk < nk_state; ++kk)
            mma_tf32_ss(sreg, kmajor_desc(ct, kk, q.crows), kmajor_desc(bt, kk, q.KB), idesc_k,
                        kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(bar));
    }
    uint32_t phase = 0;
    bool ok = true;
    if constexpr (kSplit) {
        // the remaining passes: each reloads the three tiles once the products
        // of the pass before have read them
        for (int ks = 1; ks < q.nks; ++ks) {
            const int n0 = ks * kh;
            chain_wait(smem_u32(bar), phase, ok);
            async_rows(ct, q.crows, Cb + (int64_t)(t0 + i0) * bc_stride + n0, bc_stride, c_valid, kh, tid);
            async_rows(bt, q.KB, Bb + (int64_t)t0 * bc_stride + n0, bc_stride, b_valid, kh, tid);
            cp_async_commit();
            put_transposed(ht, pc, kh, pc, [&](int n) { return hb + (int64_t)(n0 + n) * q.P; },
                           [](int) { return 1.f; }, lane, warp);
            cp_async_wait_all();
            round_rows(ct, q.crows, kh, tid);
            round_rows(bt, q.KB, kh, tid);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (tid == 0 && ok) {
                for (int kk = 0; kk < nk_state; ++kk)
                    mma_tf32_ss(acc, kmajor_desc(ct, kk, q.crows), kmajor_desc(ht, kk, pc), idesc_p, 1u);
                for (int kk = 0; kk < nk_state; ++kk)
                    mma_tf32_ss(sreg, kmajor_desc(ct, kk, q.crows), kmajor_desc(bt, kk, q.KB), idesc_k, 1u);
                mma_commit(smem_u32(bar));
            }
        }
    }

    const int r = tid;                     // query row in the block <-> TMEM lane
    const int i = i0 + r;                  // query row in the chunk
    const bool row_ok = i < q.Q;
    const float gi = row_ok ? gv[i] : 0.f;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int nJ = q.Q > 128 ? I + 1 : 1;
    for (int J = 0; J < nJ; ++J) {
        chain_wait(smem_u32(bar), phase, ok);   // S = C_I B_J^T (and, for J = 0, acc = C_I h^T)
        tc_fence_after();
        __syncwarp();
        if (J == 0) {
            // acc *= 2^{g_i}
            const float sg = exp2f(gi);
            for (int c0 = 0; c0 < pc; c0 += 16) {
                uint32_t v[16];
                tmem_ld_x16(acc + lane_off + c0, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * sg);
                tmem_st_x16(acc + lane_off + c0, v);
            }
        }
        // A = S o 2^{g_i - g_j}, j <= i, in place; the mask is a select (above
        // the diagonal the exponent is positive and may overflow)
        for (int c0 = 0; c0 < q.KB; c0 += 16) {
            uint32_t v[16];
            tmem_ld_x16(sreg + lane_off + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = J * q.KB + c0 + e;
                const float a = (row_ok && j <= i) ? __uint_as_float(v[e]) * exp2f(gi - gv[j]) : 0.f;
                v[e] = to_tf32(a);
            }
            tmem_st_x16(sreg + lane_off + c0, v);
        }
        // the X tile of block J, unless it was written up front: it replaces
        // h^T (J = 0: C h^T is done) or X_{J-1} (its MMA is done)
        if (ok && (!q.x_sep || J > 0)) put_x(J);
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && ok) {
            tc_fence_after();
            for (int kk = 0; kk < q.KB / 8; ++kk)
                mma_tf32_ts(acc, sreg + kk * 8, kmajor_desc(xt, kk, pc), idesc_p, 1u);
            mma_commit(smem_u32(bar));
        }
        if (J + 1 < nJ) {
            // B_{J+1} may be written now (the MMA that read B_J is done); S and
            // the X tile are free once acc += A X_J completes
            if (ok)
                put_rows(bt, q.KB, Bb + (int64_t)(t0 + (J + 1) * q.KB) * bc_stride, bc_stride,
                         min(q.KB, q.L - (t0 + (J + 1) * q.KB)), q.N, tid);
            fence_proxy_async_smem();
            chain_wait(smem_u32(bar), phase, ok);
            tc_fence_before();
            __syncthreads();
            if (tid == 0 && ok) {
                tc_fence_after();
                for (int kk = 0; kk < nk_state; ++kk)
                    mma_tf32_ss(sreg, kmajor_desc(ct, kk, q.crows), kmajor_desc(bt, kk, q.KB), idesc_k,
                                kk > 0 ? 1u : 0u);
                mma_commit(smem_u32(bar));
            }
        }
    }
    // y = acc + D x, one row per thread; the row of x is fetched before the
    // last product completes (its first 64 columns; the rest on the way)
    const int t = t0 + i;
    const bool store = row_ok && t < q.L;
    const float dh = D ? D[h] : 0.f;
    const float* xr = xb + (int64_t)(store ? t : 0) * x_stride;
    float* yr = y + ((int64_t)b * q.L * q.H + h) * q.P + p0 + (int64_t)(store ? t : 0) * x_stride;
    float4 xv[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) xv[u] = (store && 4 * u < pc) ? ldg4(xr + 4 * u) : zero4();
    chain_wait(smem_u32(bar), phase, ok);   // the last acc += A X
    tc_fence_after();
    __syncwarp();
#pragma unroll
    for (int c0 = 0; c0 < 128; c0 += 16) {
        if (c0 >= pc) break;
        uint32_t v[16];
        tmem_ld_x16(acc + lane_off + c0, v);
        tmem_wait_ld();
        if (store && ok) {
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 xe = c0 < 64 ? xv[(c0 + e) / 4] : ldg4(xr + c0 + e);
                *reinterpret_cast<float4*>(yr + c0 + e) =
                    make_float4(__uint_as_float(v[e]) + dh * xe.x, __uint_as_float(v[e + 1]) + dh * xe.y,
                                __uint_as_float(v[e + 2]) + dh * xe.z,
                                __uint_as_float(v[e + 3]) + dh * xe.w);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) report_timeout_to_host(&g_tf32_error, host_err);
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, q.tmem_cols);
    }
}

// ===========================================================================
// Gated DeltaNet chunk_fwd_h (Helion hackathon gallery, "GDN chunk_fwd_h"):
// one CTA per (64-column tile of V, batch*head), walking the chunks in order.
// The state is held transposed, S^T [v][k], as an fp32 tensor-memory
// accumulator (lane v of the tile, column k).  Per chunk c:
//   (a) CUDA cores: h[c] = S (into a shared staging tile), R = tf32(S^T) into
//       a second region (the A operand of the next product), then
//       S^T <- e^{g_last} S^T in place;
//   (b) D1^T = R w^T           M = v, N = the chunk's tokens, K = k
//                              (B operand: the w rows [t][k], K-major);
//   (c) CUDA cores: v_new[t][v] = u[t][v] - D1^T[v][t] (in place over the
//       staged u tile) and A2[v][t] = tf32(v_new e^{g_last - g_t}) over D1^T;
//   (d) S^T += A2 k            M = v, N = k, K = the chunk's tokens
//                              (B operand: k^T [k][t], written transposed).
// Only two warps own the tile's tensor-memory lanes, so the CUDA cores keep
// global memory off the chain: at the start of chunk c the other two warps
// request (cp.async) the rows of w (straight into its swizzled operand tile),
// k and g of chunk c + 1 and the u tile of chunk c; while (b) runs, the staged rows become the next
// chunk's TF32 tiles and all four warps write h[c] out as 16-byte stores, and
// while (d) runs they write v_new the same way.  Tokens past the sequence end
// read as zero rows, so their v_new and gated terms vanish.
// ===========================================================================
constexpr int kGdnVt = 64;   // V columns per CTA (TMEM lanes 0..63)
// Eight warps: warps 0, 1, 4, 5 reach TMEM lanes 0..63 (the tile's columns of
// V) and split the per-chunk state work by columns; warps 2, 3, 6, 7 issue the
// copies; every warp shares the conversions and the stores.
constexpr int kGdnThreads = 256;
constexpr int kGdnWarps = kGdnThreads / 32;

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

struct GdnH {
    int T, H, K, V, C, NT;
    int w_bytes, k_bytes;    // one buffer's w tile (C rows x K) and k^T tile (K rows x C)
    int raw_bytes;           // staging of one chunk's raw k rows: C x (K + 4) fp32
    uint32_t tmem_cols;
};

__global__ void __launch_bounds__(kGdnThreads)
gdn_fwd_h_tf32(const float* __restrict__ kmat, const float* __restrict__ w,
               const float* __restrict__ u, const float* __restrict__ g,
               const float* __restrict__ h0, float* __restrict__ hout, float* __restrict__ v_new,
               float* __restrict__ final_state, const GdnH q, unsigned int* host_err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t s0 = smem_u32(smem);
    const uint32_t buf_bytes = (uint32_t)(q.w_bytes + q.k_bytes);
    // raw k rows [C][K + 4]: the pad puts consecutive rows 4 banks apart, so the
    // transposing reads (lanes take rows) are conflict-free
    float* kraw = reinterpret_cast<float*>(smem + 2 * buf_bytes);
    const int kpitch = q.K + 4;
    float* hst = kraw + q.raw_bytes / 4;                                   // [K][64] h staging
    float* ubuf = hst + 128 * kGdnVt;                                      // [C][64] u, then v_new
    float* gstage = ubuf + 64 * kGdnVt;                                    // [64] raw g of a chunk
    float* gbuf = gstage + 64;                                             // [2][64] gates
    float* glast_s = gbuf + 2 * 64;                                        // [2] g_last
    uint64_t* bar = reinterpret_cast<uint64_t*>(glast_s + 2);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * kGdnVt, bh = blockIdx.y, b = bh / q.H, h = bh % q.H;
    const int vl = (warp & 3) * 32 + lane;            // this thread's TMEM lane
    const bool state_warp = (warp & 3) < kGdnVt / 32; // warps whose TMEM lanes hold the tile
    const int half = warp >> 2;                       // state warps: which share of the columns
    const int v = v0 + vl;                            // state warps: this thread's column of V
    const bool lane_ok = state_warp && v < q.V;
    const int nsi = half * 64 + (tid & 63);           // copy warps: index among the 128
    const int vt = min(kGdnVt, q.V - v0);             // columns of this tile (a multiple of 16)
    const int v4s = vt / 4;
    const int64_t tok_stride_k = (int64_t)q.H * q.K, tok_stride_v = (int64_t)q.H * q.V;
    const float* kb = kmat + (int64_t)b * q.T * tok_stride_k + (int64_t)h * q.K;
    const float* wb = w + (int64_t)b * q.T * tok_stride_k + (int64_t)h * q.K;
    const float* ub = u + (int64_t)b * q.T * tok_stride_v + (int64_t)h * q.V + v0;
    float* vnb = v_new + (int64_t)b * q.T * tok_stride_v + (int64_t)h * q.V + v0;
    const float* gb = g + (int64_t)b * q.T * q.H + h;

    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_holder), q.tmem_cols);
    // asynchronous copies of chunk c: w rows into their swizzled operand tile
    // (buffer c & 1), raw k rows and g (zero past the end)
    auto stage_wkg = [&](int c, int i, int ni) {   // issued by thread i of ni
        const int t0 = c * q.C, nv = min(q.C, q.T - t0), k4s = q.K / 4;
        const uint32_t wt = s0 + (c & 1) * buf_bytes;
        for (int e = i; e < q.C * k4s; e += ni) {
            const int t = e / k4s, k4 = e - t * k4s;
            const bool in = t < nv;
            const int64_t off = (int64_t)(t0 + (in ? t : 0)) * tok_stride_k + 4 * k4;
            cp_async_16(wt + swz(t, 4 * k4, q.C), wb + off, in ? 16u : 0u);
            cp_async_16(smem_u32(kraw + t * kpitch + 4 * k4), kb + off, in ? 16u : 0u);
        }
        for (int t = i; t < q.C; t += ni)
            cp_async_4(smem_u32(gstage + t), gb + (int64_t)(t0 + min(t, nv - 1)) * q.H, 4u);
    };
    // the u tile of chunk c: [C][vt]
    auto stage_u = [&](int c, int i, int ni) {   // issued by thread i of ni
        const int t0 = c * q.C, nv = min(q.C, q.T - t0);
        for (int e = i; e < q.C * v4s; e += ni) {
            const int t = e / v4s, v4 = e - t * v4s;
            const bool in = t < nv;
            cp_async_16(smem_u32(ubuf + t * kGdnVt + 4 * v4),
                        ub + (int64_t)(t0 + (in ? t : 0)) * tok_stride_v + 4 * v4, in ? 16u : 0u);
        }
    };
    // staged rows of chunk c -> its TF32 operand tiles (buffer c & 1): w rounded
    // in place, k transposed; gates gl = g_last, gate[t] = e^{g_last - g_t}
    // (0 past the end).  Each thread loads 8 vectors before storing any.
    auto convert = [&](int c) {
        const uint32_t wt = s0 + (c & 1) * buf_bytes, kt = wt + q.w_bytes;
        const int k4s = q.K / 4, total = q.C * k4s;
        for (int e0 = tid; e0 < total; e0 += kGdnThreads * 8) {
            uint4 x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = e0 + j * kGdnThreads, t = e / k4s, k4 = e - t * k4s;
                if (e < total)
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(x[j].x), "=r"(x[j].y), "=r"(x[j].z), "=r"(x[j].w)
                                 : "r"(wt + swz(t, 4 * k4, q.C)));
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = e0 + j * kGdnThreads, t = e / k4s, k4 = e - t * k4s;
                if (e < total)
                    st_shared_v4(wt + swz(t, 4 * k4, q.C), to_tf32(__uint_as_float(x[j].x)),
                                 to_tf32(__uint_as_float(x[j].y)), to_tf32(__uint_as_float(x[j].z)),
                                 to_tf32(__uint_as_float(x[j].w)));
            }
        }
        for (int t0 = 0; t0 < q.C; t0 += 32) {               // k^T: rows k, lanes take tokens t
            const int t = t0 + lane;
            for (int k40 = warp; k40 < k4s; k40 += kGdnWarps * 8) {
                float4 x[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int k4 = k40 + kGdnWarps * j;
                    x[j] = (t < q.C && k4 < k4s) ? *reinterpret_cast<const float4*>(kraw + t * kpitch + 4 * k4)
                                                 : zero4();
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int k4 = k40 + kGdnWarps * j;
                    if (t < q.C && k4 < k4s) {
                        st_shared_u32(kt + swz(4 * k4 + 0, t, q.K), to_tf32(x[j].x));
                        st_shared_u32(kt + swz(4 * k4 + 1, t, q.K), to_tf32(x[j].y));
                        st_shared_u32(kt + swz(4 * k4 + 2, t, q.K), to_tf32(x[j].z));
                        st_shared_u32(kt + swz(4 * k4 + 3, t, q.K), to_tf32(x[j].w));
                    }
                }
            }
        }
        const int nv = min(q.C, q.T - c * q.C);
        float* gc = gbuf + (c & 1) * 64;
        const float gl = gstage[nv - 1];
        for (int t = tid; t < q.C; t += kGdnThreads) gc[t] = t < nv ? expf(gl - gstage[t]) : 0.f;
        if (tid == 0) glast_s[c & 1] = gl;
    };
    if (q.NT > 0) {
        stage_wkg(0, tid, kGdnThreads);
        cp_async_wait_all();
        __syncthreads();
        convert(0);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // chunk 1's rows, a chunk ahead of their conversion (one cp.async group per
    // request: the copy warps keep the next chunk's rows and the current u tile
    // in flight at once)
    if (!state_warp && q.NT > 1) {
        stage_wkg(1, nsi, 128);
        cp_async_commit();
    }
    const uint32_t tmem = *tmem_holder;
    const uint32_t st_col = 0, r_col = 128, d_col = 256;   // S^T, R, D1^T / A2
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // S^T = h0^T (or 0), in the 32-column blocks that (a) of chunk 0 reads
    // back from the same warp (no barrier lies between them)
    if (state_warp) {
        const float* hb0 = h0 ? h0 + (int64_t)bh * q.K * q.V + v : nullptr;
        for (int kb = 32 * half; kb < q.K; kb += 64)
            for (int k0 = kb; k0 < min(kb + 32, q.K); k0 += 16) {
                uint32_t r[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    r[e] = __float_as_uint((hb0 && lane_ok) ? hb0[(int64_t)(k0 + e) * q.V] : 0.f);
                tmem_st_x16(tmem + lane_off + st_col + k0, r);
            }
        tmem_wait_st();
    }
    const uint32_t idesc1 = make_idesc(2, 128, (uint32_t)q.C, 0, 0);
    const uint32_t idesc2 = make_idesc(2, 128, (uint32_t)q.K, 0, 0);
    uint32_t phase = 0;
    bool ok = true;
    for (int c = 0; c < q.NT; ++c) {
        const int t0 = c * q.C, nv = min(q.C, q.T - t0);
        const float* gc = gbuf + (c & 1) * 64;
        const uint32_t wt = s0 + (c & 1) * buf_bytes, kt = wt + q.w_bytes;
        // the u tile of chunk c, issued by the copy warps while the state warps run (a)
        if (!state_warp) {
            stage_u(c, nsi, 128);
            cp_async_commit();
        }
        const float dec = expf(glast_s[c & 1]);
        // (a) h[c] = S (staged); R = tf32(S^T); S^T <- e^{g_last} S^T, 32
        // columns at a time (16 for the last block when K % 32 == 16)
        if (state_warp) {
            __syncwarp();
            for (int k0 = 32 * half; k0 < q.K; k0 += 64) {
                const int n = min(32, q.K - k0);   // 16 or 32: K is a multiple of 16
                uint32_t r[32];
                if (n == 32) {
                    tmem_ld_x32(tmem + lane_off + st_col + k0, r);
                } else {
                    uint32_t r16[16];
                    tmem_ld_x16(tmem + lane_off + st_col + k0, r16);
                    tmem_wait_ld();   // before the destination registers are read
#pragma unroll
                    for (int e = 0; e < 16; ++e) { r[e] = r16[e]; r[16 + e] = 0u; }
                }
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e)   // hst[k][v]: lanes write consecutive words
                    if (e < n) hst[(k0 + e) * kGdnVt + vl] = __uint_as_float(r[e]);
                uint32_t rt[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float sv = __uint_as_float(r[e]);
                    rt[e] = to_tf32(sv);
                    r[e] = __float_as_uint(sv * dec);
                }
                if (n == 32) {
                    tmem_st_x32(tmem + lane_off + r_col + k0, rt);
                    tmem_st_x32(tmem + lane_off + st_col + k0, r);
                } else {
                    uint32_t a16[16], b16[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) { a16[e] = rt[e]; b16[e] = r[e]; }
                    tmem_st_x16(tmem + lane_off + r_col + k0, a16);
                    tmem_st_x16(tmem + lane_off + st_col + k0, b16);
                }
            }
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        // (b) D1^T = R w^T
        if (tid == 0 && ok) {
            tc_fence_after();
            for (int kk = 0; kk < q.K / 8; ++kk)
                mma_tf32_ts(tmem + d_col, tmem + r_col + kk * 8, kmajor_desc(wt, kk, q.C), idesc1,
                            kk > 0 ? 1u : 0u);
            mma_commit(smem_u32(bar));
        }
        // meanwhile: h[c] out as 16-byte stores by all four warps
        if (ok) {
            float* hc = hout + ((int64_t)bh * q.NT + c) * q.K * q.V + v0;
            for (int e = tid; e < q.K * v4s; e += kGdnThreads) {
                const int k = e / v4s, v4 = e - k * v4s;
                *reinterpret_cast<float4*>(hc + (int64_t)k * q.V + 4 * v4) =
                    *reinterpret_cast<const float4*>(hst + k * kGdnVt + 4 * v4);
            }
        }
        // ... and the staged rows of chunk c + 1 (requested a chunk ago) become its
        // operand tiles in the other buffer (its last reader, (d) of chunk c - 1,
        // is complete)
        cp_async_wait_group<1>();   // all but the u tile of chunk c
        __syncthreads();
        if (c + 1 < q.NT && ok) convert(c + 1);
        fence_proxy_async_smem();
        cp_async_wait_group<0>();   // the u tile
        __syncthreads();
        chain_wait(smem_u32(bar), phase, ok);
        tc_fence_after();
        // the rows of chunk c + 2: its w tile goes where (b) of chunk c just read,
        // its raw k and g where convert(c + 1) just read
        if (!state_warp && c + 2 < q.NT) {
            stage_wkg(c + 2, nsi, 128);
            cp_async_commit();
        }
        // (c) v_new = u - D1 (over the staged u); A2 = tf32(v_new e^{g_last - g_t}) over D1^T
        if (state_warp) {
            __syncwarp();
            for (int c0 = 32 * half; c0 < q.C; c0 += 64) {
                const int n = min(32, q.C - c0);   // 16 or 32 (C is 16, 32 or 64)
                uint32_t r[32];
                if (n == 32) {
                    tmem_ld_x32(tmem + lane_off + d_col + c0, r);
                } else {
                    uint32_t r16[16];
                    tmem_ld_x16(tmem + lane_off + d_col + c0, r16);
                    tmem_wait_ld();   // before the destination registers are read
#pragma unroll
                    for (int e = 0; e < 16; ++e) { r[e] = r16[e]; r[16 + e] = 0u; }
                }
                // u and the gates into registers first, so that the loads are not
                // held behind the in-place stores
                float uv[32], gt[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    uv[e] = e < n ? ubuf[(c0 + e) * kGdnVt + vl] : 0.f;
                    gt[e] = e < n ? gc[c0 + e] : 0.f;
                }
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float vn = uv[e] - __uint_as_float(r[e]);
                    if (e < n) ubuf[(c0 + e) * kGdnVt + vl] = vn;
                    r[e] = to_tf32(vn * gt[e]);   // gate 0 past the end and beyond n
                }
                if (n == 32) {
                    tmem_st_x32(tmem + lane_off + d_col + c0, r);
                } else {
                    uint32_t r16[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) r16[e] = r[e];
                    tmem_st_x16(tmem + lane_off + d_col + c0, r16);
                }
            }
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        // (d) S^T += A2 k
        if (tid == 0 && ok) {
            tc_fence_after();
            for (int kk = 0; kk < q.C / 8; ++kk)
                mma_tf32_ts(tmem + st_col, tmem + d_col + kk * 8, kmajor_desc(kt, kk, q.K), idesc2,
                            1u);
            mma_commit(smem_u32(bar));
        }
        // meanwhile: v_new of the chunk's real tokens out as 16-byte stores
        if (ok) {
            for (int e = tid; e < nv * v4s; e += kGdnThreads) {
                const int t = e / v4s, v4 = e - t * v4s;
                *reinterpret_cast<float4*>(vnb + (int64_t)(t0 + t) * tok_stride_v + 4 * v4) =
                    *reinterpret_cast<const float4*>(ubuf + t * kGdnVt + 4 * v4);
            }
        }
        chain_wait(smem_u32(bar), phase, ok);
        tc_fence_after();
        __syncthreads();   // ubuf and hst are read above before the next chunk refills them
    }
    cp_async_wait_all();   // no copy into shared memory outlives the CTA
    // final_state = S
    if (state_warp && final_state != nullptr) {
        __syncwarp();
        float* fs = final_state + (int64_t)bh * q.K * q.V + v;
        for (int k0 = 16 * half; k0 < q.K; k0 += 32) {
            uint32_t r[16];
            tmem_ld_x16(tmem + lane_off + st_col + k0, r);
            tmem_wait_ld();
            if (lane_ok && ok) {
#pragma unroll
                for (int e = 0; e < 16; ++e) fs[(int64_t)(k0 + e) * q.V] = __uint_as_float(r[e]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) report_timeout_to_host(&g_tf32_error, host_err);
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, q.tmem_cols);
    }
}

}  // namespace

bool tf32_path_supports(const Problem& p) {
    return p.dtype == SSD_F32 && p.N <= 128 && p.P <= 128 && p.nc <= 65535 && p.b * p.H <= 65535;
}

cudaError_t launch_fps_products_tf32(const Problem& p, const void* x, const void* B,
                                     const float* Gcs, const float* dtT, void* hiddens,
                                     cudaStream_t stream) {
    FpsTf32 q;
    q.L = (int)p.L; q.H = (int)p.H; q.P = (int)p.P; q.N = (int)p.N; q.G = (int)p.G;
    q.Q = (int)p.Q; q.nc = (int)p.nc; q.Lp = (int)p.Lp; q.hpg = (int)p.hpg;
    q.tmem_cols = tmem_cols_for(q.P);
    q.a_bytes = tile_bytes(128, 32);
    q.x_bytes = up1024(tile_bytes(q.P, 32));
    const int smem = 2 * (q.a_bytes + q.x_bytes) + 64 + 1024;
    // no more CTAs per SM than the tensor memory holds
    const int by_tmem = 512 / (int)q.tmem_cols;
    const int smem_cta = std::max(smem, (228 * 1024) / by_tmem - 1024);
    cudaError_t e = cudaFuncSetAttribute(fps_products_tf32,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem_cta);
    if (e != cudaSuccess) return e;
    return launch_chained(fps_products_tf32, dim3((unsigned)p.nc, (unsigned)(p.b * p.H)), dim3(kThreads),
                          (size_t)smem_cta, stream, p.chained, (const float*)x, (const float*)B, Gcs,
                          dtT, (float*)hiddens, q, host_timeout_word());
}

namespace {
// Tile sizes, TMEM columns and shared memory of compute_out_tf32 for the
// sizes already in q (L .. hpg); returns the dynamic shared memory per CTA,
// or -1 if it does not fit.
int co_tf32_layout(CoTf32& q) {
    q.KB = q.Q < 128 ? q.Q : 128;
    q.nblk = q.Q > 128 ? q.Q / 128 : 1;
    // P > 64 is split into 64-column tiles (one CTA each): half the h^T and X
    // tiles per CTA, so that two CTAs share an SM
    q.pt = q.P > 64 ? 64 : q.P;
    q.npt = (q.P + q.pt - 1) / q.pt;
    q.crows = q.Q < 128 ? q.Q : 128;
    q.scol = (uint32_t)((q.pt + 31) / 32 * 32);
    q.tmem_cols = tmem_cols_for((int)q.scol + q.KB);
    const int per_sm = 228 * 1024;
    const int by_tmem = 512 / (int)q.tmem_cols;
    const int extras = 2 * q.Q * 4 + 64 + 1024;
    // The tiles for products over kh state columns per pass; returns the
    // dynamic shared memory per CTA, or -1 if it does not fit.
    auto fit = [&](CoTf32& o, int kh, bool allow_sep) {
        o = q;
        o.kh = kh;
        o.nks = q.N / kh;
        o.c_bytes = up1024(tile_bytes(o.crows, kh));
        o.b_bytes = up1024(tile_bytes(o.KB, kh));
        const int h_own = up1024(tile_bytes(o.pt, kh));
        o.x_bytes = up1024(tile_bytes(o.pt, o.KB));
        const int sep = o.c_bytes + o.b_bytes + h_own + o.x_bytes + extras;
        const int shared = o.c_bytes + o.b_bytes + std::max(h_own, o.x_bytes) + extras;
        // a tile of its own for X unless sharing h^T's lets more CTAs onto an SM
        o.x_sep = allow_sep && sep <= 200 * 1024 && per_sm / (sep + 1024) >= per_sm / (shared + 1024);
        o.h_bytes = o.x_sep ? h_own : std::max(h_own, o.x_bytes);
        int smem = o.x_sep ? sep : shared;
        // the M = 128 products read 128 rows of the C_I tile from each K atom's
        // start: with fewer rows that runs past the tile, which must stay
        // inside the allocation
        const int c_read = ((kh + 31) / 32 - 1) * o.crows * kRowBytes + 16 * 1024;
        smem = std::max(smem, c_read + extras);
        const int smem_cta = std::max(smem, per_sm / by_tmem - 1024);
        return smem_cta > 227 * 1024 ? -1 : smem_cta;
    };
    auto ctas = [&](int smem_cta) {
        return smem_cta < 0 ? 0 : std::min(std::min(by_tmem, kCtasPerSm), per_sm / (smem_cta + 1024));
    };
    CoTf32 whole, split;
    int smem_cta = fit(whole, q.N, true);
    q = whole;
    // two passes over a state of 128 (64 columns each, X sharing h^T's tile)
    // when that lets more CTAs share an SM; the query blocks of a 256-token
    // chunk reuse the whole C_I tile, so only for Q <= 128
    if (q.N > 64 && q.N % 64 == 0 && q.nblk == 1) {
        const int s2 = fit(split, 64, false);
        if (ctas(s2) > ctas(smem_cta)) {
            q = split;
            smem_cta = s2;
        }
    }
    return smem_cta;
}
}  // namespace

cudaError_t launch_compute_out_tf32(const Problem& p, const void* x, const void* B, const void* C,
                                    const float* Gcs, const float* dtT, const void* hiddens,
                                    const float* D, void* y, cudaStream_t stream) {
    CoTf32 q;
    q.L = (int)p.L; q.H = (int)p.H; q.P = (int)p.P; q.N = (int)p.N; q.G = (int)p.G;
    q.Q = (int)p.Q; q.nc = (int)p.nc; q.Lp = (int)p.Lp; q.hpg = (int)p.hpg;
    const int smem_cta = co_tf32_layout(q);
    if (smem_cta < 0) return cudaErrorInvalidValue;
    auto kern = q.nks > 1 ? compute_out_tf32<false, true> : compute_out_tf32<false, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_cta);
    if (e != cudaSuccess) return e;
    return launch_chained(kern,
                          dim3((unsigned)(q.nblk * q.npt), (unsigned)p.nc, (unsigned)(p.b * p.H)),
                          dim3(kThreads), (size_t)smem_cta, stream, p.chained, (const float*)x,
                          (const float*)B, (const float*)C, Gcs, dtT, (const float*)hiddens, D,
                          (float*)y, q, host_timeout_word());
}

bool gdn_tf32_supports(const GdnProblem& p) {
    return p.K % 16 == 0 && p.V % 16 == 0 && p.K <= 128 && p.V <= 128 && p.NT <= 65535 &&
           p.B * p.H <= 65535;
}

cudaError_t launch_gdn_fwd_o_tf32(const GdnProblem& p, const float* qm, const float* k,
                                  const float* v_new, const float* h, const float* g, float* o,
                                  cudaStream_t stream) {
    CoTf32 q;
    q.L = (int)p.T; q.H = (int)p.H; q.P = (int)p.V; q.N = (int)p.K; q.G = (int)p.H;
    q.Q = (int)p.C; q.nc = (int)p.NT; q.Lp = 0; q.hpg = 1;
    const int smem_cta = co_tf32_layout(q);
    if (smem_cta < 0) return cudaErrorInvalidValue;
    auto kern = q.nks > 1 ? compute_out_tf32<true, true> : compute_out_tf32<true, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_cta);
    if (e != cudaSuccess) return e;
    // operand roles: C <- q, B <- k, x <- v_new, hiddens <- h, y <- o, Gcs <- g
    kern<<<dim3((unsigned)(q.nblk * q.npt), (unsigned)p.NT, (unsigned)(p.B * p.H)), kThreads,
           (size_t)smem_cta, stream>>>(
        v_new, k, qm, g, nullptr, h, nullptr, o, q, host_timeout_word());
    return cudaGetLastError();
}

cudaError_t launch_gdn_fwd_h_tf32(const GdnProblem& p, const float* k, const float* w,
                                  const float* u, const float* g, const float* h0, float* h,
                                  float* v_new, float* final_state, cudaStream_t stream) {
    GdnH q;
    q.T = (int)p.T; q.H = (int)p.H; q.K = (int)p.K; q.V = (int)p.V; q.C = (int)p.C;
    q.NT = (int)p.NT;
    q.w_bytes = up1024(tile_bytes(q.C, q.K));
    q.k_bytes = up1024(tile_bytes(q.K, q.C));
    q.raw_bytes = q.C * (q.K + 4) * 4;
    q.tmem_cols = 512;   // S^T, R (128 columns each) and D1^T / A2: one CTA per SM
    const int smem = 2 * (q.w_bytes + q.k_bytes) + q.raw_bytes + 128 * kGdnVt * 4 +
                     64 * kGdnVt * 4 + 64 * 4 + 2 * 64 * 4 + 8 + 64 + 1024;
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gdn_fwd_h_tf32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem);
    if (e != cudaSuccess) return e;
    gdn_fwd_h_tf32<<<dim3((unsigned)((p.V + kGdnVt - 1) / kGdnVt), (unsigned)(p.B * p.H)), kGdnThreads,
                     (size_t)smem, stream>>>(k, w, u, g, h0, h, v_new, final_state, q,
                                             host_timeout_word());
    return cudaGetLastError();
}

unsigned int take_tf32_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tf32_error, sizeof(v)) != cudaSuccess) return ~0u;
    cudaMemcpyToSymbol(g_tf32_error, &zero, sizeof(zero));
    return v;
}

}  // namespace ssd
