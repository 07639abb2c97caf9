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

__global__ void __launch_bounds__(kThreads)
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
    uint32_t tmem_cols;
    uint32_t scol;               // first TMEM column of S / A (acc holds columns [0, P))
    int c_bytes, b_bytes, h_bytes, x_bytes;   // C_I, B_J, h^T, (dt o X_J)^T tiles
    int x_sep;                   // 1: (dt o X)^T has a tile of its own (written up front);
                                 // 0: it reuses h^T's, once C h^T is done
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

// A transposed K-major tile: tile[p][k] = tf32(scale(k) * src(k)[p]) for
// k < Kdim (lanes take k), p < cols (warps take groups of 4 columns); src(k)
// is NULL for a zero row.  Up to 16 loads per thread are issued before their
// stores.
template <typename Src, typename Scale>
__device__ __forceinline__ void put_transposed(uint32_t tile, int rows, int Kdim, int cols, Src src,
                                               Scale scale, int lane, int warp) {
    const int nkb = (Kdim + 31) / 32;
    for (int it0 = 0; it0 < nkb * kMaxGroups; it0 += 16) {
        float4 v[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int it = it0 + m, kb = it / kMaxGroups, c4 = warp + 4 * (it % kMaxGroups);
            const int k = kb * 32 + lane;
            const float* sp = (kb < nkb && k < Kdim && 4 * c4 < cols) ? src(k) : nullptr;
            v[m] = sp ? ldg4(sp + 4 * c4) : zero4();
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int it = it0 + m, kb = it / kMaxGroups, c4 = warp + 4 * (it % kMaxGroups);
            const int k = kb * 32 + lane;
            if (kb < nkb && k < Kdim && 4 * c4 < cols) {
                const float sc = scale(k);
                st_shared_u32(tile + swz(4 * c4 + 0, k, rows), to_tf32(v[m].x * sc));
                st_shared_u32(tile + swz(4 * c4 + 1, k, rows), to_tf32(v[m].y * sc));
                st_shared_u32(tile + swz(4 * c4 + 2, k, rows), to_tf32(v[m].z * sc));
                st_shared_u32(tile + swz(4 * c4 + 3, k, rows), to_tf32(v[m].w * sc));
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads)
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
    const int I = blockIdx.x, c = blockIdx.y, bh = blockIdx.z;
    const int b = bh / q.H, h = bh % q.H, grp = h / q.hpg;
    const int t0 = c * q.Q;              // first token of the chunk
    const int i0 = I * 128;              // first query row of the block (in the chunk)
    const int64_t bc_stride = (int64_t)q.G * q.N;            // token stride of B and C
    const float* Cb = C + ((int64_t)b * q.L * q.G + grp) * q.N;
    const float* Bb = B + ((int64_t)b * q.L * q.G + grp) * q.N;
    const float* xb = x + ((int64_t)b * q.L * q.H + h) * q.P;  // token t at xb + t H P
    const int64_t x_stride = (int64_t)q.H * q.P;

    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_holder), q.tmem_cols);
    for (int i = tid; i < q.Q; i += kThreads) {
        gv[i] = Gcs[(int64_t)bh * q.Lp + t0 + i];
        dv[i] = dtT[(int64_t)bh * q.Lp + t0 + i];
    }
    // C_I (rows = query rows) and B_0 (rows = keys)
    put_rows(ct, 128, Cb + (int64_t)(t0 + i0) * bc_stride, bc_stride,
             min(min(q.Q - i0, 128), q.L - (t0 + i0)), q.N, tid);
    put_rows(bt, q.KB, Bb + (int64_t)t0 * bc_stride, bc_stride, min(q.KB, q.L - t0), q.N, tid);
    // h^T: rows = p, K = state n (hiddens holds [n][p])
    const float* hb = hiddens + ((int64_t)bh * q.nc + c) * (int64_t)q.N * q.P;
    put_transposed(ht, q.P, q.N, q.P, [&](int n) { return hb + (int64_t)n * q.P; },
                   [](int) { return 1.f; }, lane, warp);
    // (dt o X_J)^T: rows = p, K = keys of block J (zero past the sequence end)
    // (reads dv: the first call follows a barrier after dv is written; no
    // barrier inside, since later calls sit under the per-thread `ok`)
    auto put_x = [&](int J) {
        put_transposed(
            xt, q.P, q.KB, q.P,
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
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t acc = tmem, sreg = tmem + q.scol;
    const uint32_t idesc_p = make_idesc(2, 128, (uint32_t)q.P, 0, 0);
    const uint32_t idesc_k = make_idesc(2, 128, (uint32_t)q.KB, 0, 0);
    const int nk_state = q.N / 8;
    if (tid == 0) {
        for (int kk = 0; kk < nk_state; ++kk)
            mma_tf32_ss(acc, kmajor_desc(ct, kk, 128), kmajor_desc(ht, kk, q.P), idesc_p,
                        kk > 0 ? 1u : 0u);
        for (int kk = 0; kk < nk_state; ++kk)
            mma_tf32_ss(sreg, kmajor_desc(ct, kk, 128), kmajor_desc(bt, kk, q.KB), idesc_k,
                        kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(bar));
    }

    const int r = tid;                     // query row in the block <-> TMEM lane
    const int i = i0 + r;                  // query row in the chunk
    const bool row_ok = i < q.Q;
    const float gi = row_ok ? gv[i] : 0.f;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int nJ = q.Q > 128 ? I + 1 : 1;
    uint32_t phase = 0;
    bool ok = true;
    for (int J = 0; J < nJ; ++J) {
        chain_wait(smem_u32(bar), phase, ok);   // S = C_I B_J^T (and, for J = 0, acc = C_I h^T)
        tc_fence_after();
        __syncwarp();
        if (J == 0) {
            // acc *= 2^{g_i}
            const float sg = exp2f(gi);
            for (int c0 = 0; c0 < q.P; c0 += 16) {
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
                mma_tf32_ts(acc, sreg + kk * 8, kmajor_desc(xt, kk, q.P), idesc_p, 1u);
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
                    mma_tf32_ss(sreg, kmajor_desc(ct, kk, 128), kmajor_desc(bt, kk, q.KB), idesc_k,
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
    float* yr = y + ((int64_t)b * q.L * q.H + h) * q.P + (int64_t)(store ? t : 0) * x_stride;
    float4 xv[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) xv[u] = (store && 4 * u < q.P) ? ldg4(xr + 4 * u) : zero4();
    chain_wait(smem_u32(bar), phase, ok);   // the last acc += A X
    tc_fence_after();
    __syncwarp();
#pragma unroll
    for (int c0 = 0; c0 < 128; c0 += 16) {
        if (c0 >= q.P) break;
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
    fps_products_tf32<<<dim3((unsigned)p.nc, (unsigned)(p.b * p.H)), kThreads, (size_t)smem_cta,
                        stream>>>((const float*)x, (const float*)B, Gcs, dtT, (float*)hiddens, q,
                                  host_timeout_word());
    return cudaGetLastError();
}

cudaError_t launch_compute_out_tf32(const Problem& p, const void* x, const void* B, const void* C,
                                    const float* Gcs, const float* dtT, const void* hiddens,
                                    const float* D, void* y, cudaStream_t stream) {
    CoTf32 q;
    q.L = (int)p.L; q.H = (int)p.H; q.P = (int)p.P; q.N = (int)p.N; q.G = (int)p.G;
    q.Q = (int)p.Q; q.nc = (int)p.nc; q.Lp = (int)p.Lp; q.hpg = (int)p.hpg;
    q.KB = q.Q < 128 ? q.Q : 128;
    q.nblk = q.Q > 128 ? q.Q / 128 : 1;
    q.scol = (uint32_t)((q.P + 31) / 32 * 32);
    q.tmem_cols = tmem_cols_for((int)q.scol + q.KB);
    q.c_bytes = up1024(tile_bytes(128, q.N));
    q.b_bytes = up1024(tile_bytes(q.KB, q.N));
    q.h_bytes = up1024(tile_bytes(q.P, q.N));
    q.x_bytes = up1024(tile_bytes(q.P, q.KB));
    const int extras = 2 * q.Q * 4 + 64 + 1024;
    q.x_sep = q.c_bytes + q.b_bytes + q.h_bytes + q.x_bytes + extras <= 200 * 1024;
    if (!q.x_sep) q.h_bytes = std::max(q.h_bytes, q.x_bytes);   // one tile for both
    const int smem = q.c_bytes + q.b_bytes + q.h_bytes + (q.x_sep ? q.x_bytes : 0) + extras;
    const int by_tmem = 512 / (int)q.tmem_cols;
    const int smem_cta = std::max(smem, (228 * 1024) / by_tmem - 1024);
    if (smem_cta > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(compute_out_tf32,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem_cta);
    if (e != cudaSuccess) return e;
    compute_out_tf32<<<dim3((unsigned)q.nblk, (unsigned)p.nc, (unsigned)(p.b * p.H)), kThreads,
                       (size_t)smem_cta, stream>>>(
        (const float*)x, (const float*)B, (const float*)C, Gcs, dtT, (const float*)hiddens, D,
        (float*)y, q, host_timeout_word());
    return cudaGetLastError();
}

unsigned int take_tf32_error() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tf32_error, sizeof(v)) != cudaSuccess) return ~0u;
    cudaMemcpyToSymbol(g_tf32_error, &zero, sizeof(zero));
    return v;
}

}  // namespace ssd
