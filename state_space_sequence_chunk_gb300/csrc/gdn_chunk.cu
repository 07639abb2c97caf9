// gdn_chunk.cu -- the Gated DeltaNet chunk kernels: a second chunked
// recurrence with the shape of fwd_pass_state and compute_out.
//
// Helion hackathon gallery (cerebralvalley.ai), "GDN chunk_fwd_h" and "GDN
// chunk_fwd_o" entries, chunk size C.  With g the in-chunk inclusive
// cumulative log gate and g_last its value at the chunk's last token:
//   chunk_fwd_h, per (batch, head) and chunk in order:
//     (1) store h;  (2) v_new = u - w h;  (3) v_gated[t] = v_new[t] exp(g_last - g_t);
//     (4) h <- exp(g_last) h;  (5) h <- h + k^T v_gated.
//   chunk_fwd_o, per chunk (independent):
//     o = (q h) o exp(g)  +  causal((q k^T) o exp(g_i - g_j)) v_new   (j <= i kept).
// Layouts: q, k, w [B, T, H, K]; u, v_new, o [B, T, H, V]; g [B, T, H];
// h [B, H, NT, K, V]; h0, final [B, H, K, V]; all fp32 (the pages run these
// products in fp32 / TF32).
//
// Shapes with K and V multiples of 16 (up to 128) run on the TF32 tensor cores
// (tf32_path.cu: the state held in tensor memory for chunk_fwd_h, and the
// compute_out kernel for chunk_fwd_o).  The kernels below serve the others,
// on the CUDA cores in fp32.  A CTA owns a tile of V
// columns (32 for chunk_fwd_h, 64 for chunk_fwd_o), stages the chunk's rows of
// k and w (or q and k) in shared memory -- transposed where an operand is read
// as four consecutive rows -- and keeps its state tile there.  Each thread
// computes a 4 x 4 or 4 x 2 register tile, so that every 16-byte shared-memory
// read feeds several FMAs.  chunk_fwd_h walks its chunks in order (one CTA per
// (batch, head, V tile)); chunk_fwd_o is one CTA per (batch, head, chunk, V
// tile).
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kGdnThreads = 256;   // 8 warps

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
constexpr int kVT = 32;            // V columns per CTA (one per lane)
constexpr int kWarps = kGdnThreads / 32;

// Transposed staging of a chunk's rows [t][K] into xT[kk][t] (pitch C + 4: the
// 4-row reads below are 16-byte aligned, and the transposing stores -- t
// fastest across a warp -- hit 32 distinct banks).
// A thread's share of a [C][K] tile is at most C * K / 4 / threads <= 8 vectors
// (K <= 128, C <= 64): all its loads are issued before the first store.
constexpr int kMaxVecPerThread = 8;
template <int C>
__device__ __forceinline__ void stage_transposed(const float* __restrict__ src, float* xT, int b,
                                                 int T, int t0, int nt, int H, int hh, int K) {
    const int K4 = K >> 2;
    float4 v[kMaxVecPerThread];
#pragma unroll
    for (int r = 0; r < kMaxVecPerThread; ++r) {
        const int i = threadIdx.x + r * kGdnThreads, t = i % C, k4 = i / C;
        v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < C * K4 && t < nt)
            v[r] = __ldg(reinterpret_cast<const float4*>(src + ((int64_t)(b * T + t0 + t) * H + hh) * K) + k4);
    }
#pragma unroll
    for (int r = 0; r < kMaxVecPerThread; ++r) {
        const int i = threadIdx.x + r * kGdnThreads, t = i % C, k4 = i / C;
        if (i < C * K4) {
            xT[(4 * k4 + 0) * (C + 4) + t] = v[r].x;
            xT[(4 * k4 + 1) * (C + 4) + t] = v[r].y;
            xT[(4 * k4 + 2) * (C + 4) + t] = v[r].z;
            xT[(4 * k4 + 3) * (C + 4) + t] = v[r].w;
        }
    }
}

// chunk_fwd_h: the chunk walk is software-pipelined.  A chunk's rows of k and
// w, its g values and this thread's u values are loaded into registers while
// the previous chunk's state update (4)-(5) runs, and stored into shared
// memory once that update no longer reads k; the L2 prefetch one chunk further
// ahead turns those loads into L2 hits.
template <int C>
__global__ void __launch_bounds__(kGdnThreads)
gdn_fwd_h_kernel(const float* __restrict__ k, const float* __restrict__ w,
                 const float* __restrict__ u, const float* __restrict__ g,
                 const float* __restrict__ h0, float* __restrict__ h, float* __restrict__ v_new,
                 float* __restrict__ final_state, int T, int H, int K, int V, int NT) {
    extern __shared__ __align__(16) float sm[];
    constexpr int CP = C + 4;
    float* ks = sm;                 // [C][K]   k rows (row-major)
    float* wT = ks + C * K;         // [K][C+4] w, transposed
    float* S = wT + K * CP;         // [K][32]  the state tile
    float* vg = S + K * kVT;        // [C][32]  gated v_new
    float* gs = vg + C * kVT;       // [C]
    const int bh = blockIdx.x, b = bh / H, hh = bh - b * H;
    const int v0 = blockIdx.y * kVT, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K4 = K >> 2;
    // thread maps: (2) 4 tokens x 2 columns; (4)(5) 4 state rows x 4 columns
    const int tt = threadIdx.x >> 4, tv2 = threadIdx.x & 15;
    const int tk = threadIdx.x >> 3, tv4 = threadIdx.x & 7;

    // registers of the chunk being loaded
    float4 kv[kMaxVecPerThread], wv[kMaxVecPerThread];
    float uv[4][2], gv = 0.f;
    auto issue = [&](int c) {   // loads of chunk c
        const int t0 = c * C, nt = min(C, T - t0);
#pragma unroll
        for (int r = 0; r < kMaxVecPerThread; ++r) {
            const int i = threadIdx.x + r * kGdnThreads;
            const int tk_ = i / K4, k4 = i - tk_ * K4;      // k: row-major
            kv[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < C * K4 && tk_ < nt)
                kv[r] = __ldg(reinterpret_cast<const float4*>(k + ((int64_t)(b * T + t0 + tk_) * H + hh) * K) + k4);
            const int tw = i % C, kw4 = i / C;              // w: transposed below
            wv[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < C * K4 && tw < nt)
                wv[r] = __ldg(reinterpret_cast<const float4*>(w + ((int64_t)(b * T + t0 + tw) * H + hh) * K) + kw4);
        }
        gv = ((int)threadIdx.x < nt) ? __ldg(g + (int64_t)(b * T + t0 + threadIdx.x) * H + hh) : 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = 4 * tt + r;
            const int64_t row = (int64_t)(b * T + t0 + t) * H + hh;
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                const int v = v0 + 2 * tv2 + q2;
                uv[r][q2] = (4 * tt < C && t < nt && v < V) ? __ldg(u + row * V + v) : 0.f;
            }
        }
        // chunk c + 1 into L2
        if (c + 1 < NT) {
            const int tn0 = t0 + C, ntn = min(C, T - tn0);
            const int kl = (K + 31) / 32;           // 128-byte lines of a k or w row
            const int per = 2 * kl + 2;
            for (int i = threadIdx.x; i < ntn * per; i += kGdnThreads) {
                const int t = i / per, j = i - t * per;
                const int64_t row = (int64_t)(b * T + tn0 + t) * H + hh;
                const float* ptr = j < kl ? k + row * K + 32 * j
                                 : j < 2 * kl ? w + row * K + 32 * (j - kl)
                                 : j == 2 * kl ? u + row * V + v0 : g + row;
                prefetch_l2(ptr);
            }
        }
    };
    auto commit = [&]() {       // the loaded chunk into shared memory
#pragma unroll
        for (int r = 0; r < kMaxVecPerThread; ++r) {
            const int i = threadIdx.x + r * kGdnThreads;
            if (i < C * K4) {
                reinterpret_cast<float4*>(ks)[i] = kv[r];
                const int tw = i % C, kw4 = i / C;
                wT[(4 * kw4 + 0) * CP + tw] = wv[r].x;
                wT[(4 * kw4 + 1) * CP + tw] = wv[r].y;
                wT[(4 * kw4 + 2) * CP + tw] = wv[r].z;
                wT[(4 * kw4 + 3) * CP + tw] = wv[r].w;
            }
        }
        if ((int)threadIdx.x < C) gs[threadIdx.x] = gv;
    };

    if (NT > 0) issue(0);
    for (int kk = warp; kk < K; kk += kWarps)
        S[kk * kVT + lane] = (h0 != nullptr && v0 + lane < V) ? h0[((int64_t)bh * K + kk) * V + v0 + lane] : 0.f;
    if (NT > 0) commit();
    for (int c = 0; c < NT; ++c) {
        const int t0 = c * C, nt = min(C, T - t0);
        __syncthreads();   // chunk c is in shared memory; S is up to date
        // (1) the chunk-start state
        float* hc = h + (((int64_t)bh * NT + c) * K) * V;
        if (v0 + lane < V)
            for (int kk = warp; kk < K; kk += kWarps) hc[(int64_t)kk * V + v0 + lane] = S[kk * kVT + lane];
        const float g_last = gs[nt - 1];
        // (2) v_new = u - w S for tokens 4 tt .. 4 tt + 3, columns 2 tv2, 2 tv2 + 1; (3) gate
        if (4 * tt < C) {
            float a[4][2] = {};
            #pragma unroll 4
            for (int kk = 0; kk < K; ++kk) {
                const float4 wq = *reinterpret_cast<const float4*>(wT + kk * CP + 4 * tt);
                const float2 sv = *reinterpret_cast<const float2*>(S + kk * kVT + 2 * tv2);
                const float wr[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    a[r][0] = fmaf(wr[r], sv.x, a[r][0]);
                    a[r][1] = fmaf(wr[r], sv.y, a[r][1]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * tt + r;
                if (t < nt) {
                    const int64_t row = (int64_t)(b * T + t0 + t) * H + hh;
                    const float gate = expf(g_last - gs[t]);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int v = v0 + 2 * tv2 + q;
                        const float vn = v < V ? uv[r][q] - a[r][q] : 0.f;
                        if (v < V) v_new[row * V + v] = vn;
                        vg[t * kVT + 2 * tv2 + q] = vn * gate;
                    }
                } else {
                    vg[t * kVT + 2 * tv2] = 0.f;
                    vg[t * kVT + 2 * tv2 + 1] = 0.f;
                }
            }
        }
        __syncthreads();   // vg is complete; S and wT are no longer read
        if (c + 1 < NT) issue(c + 1);   // in flight during (4)-(5)
        // (4) decay and (5) S += k^T v_gated for state rows 4 tk .. 4 tk + 3, columns 4 tv4 ..
        if (4 * tk < K) {
            const float decay = expf(g_last);
            float a[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float4 sv = *reinterpret_cast<const float4*>(S + (4 * tk + r) * kVT + 4 * tv4);
                a[r][0] = sv.x * decay; a[r][1] = sv.y * decay; a[r][2] = sv.z * decay; a[r][3] = sv.w * decay;
            }
            #pragma unroll 4
            for (int t = 0; t < nt; ++t) {
                const float4 kq = *reinterpret_cast<const float4*>(ks + t * K + 4 * tk);
                const float4 xv = *reinterpret_cast<const float4*>(vg + t * kVT + 4 * tv4);
                const float kr[4] = {kq.x, kq.y, kq.z, kq.w}, xr[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int q = 0; q < 4; ++q) a[r][q] = fmaf(kr[r], xr[q], a[r][q]);
            }
            // every thread owns distinct S entries and all reads of S are done (barrier above)
#pragma unroll
            for (int r = 0; r < 4; ++r)
                *reinterpret_cast<float4*>(S + (4 * tk + r) * kVT + 4 * tv4) = make_float4(a[r][0], a[r][1], a[r][2], a[r][3]);
        }
        if (c + 1 < NT) {
            __syncthreads();   // every read of ks, gs and vg for chunk c is done
            commit();
        }
    }
    __syncthreads();
    if (final_state != nullptr && v0 + lane < V)
        for (int kk = warp; kk < K; kk += kWarps)
            final_state[((int64_t)bh * K + kk) * V + v0 + lane] = S[kk * kVT + lane];
}

// chunk_fwd_o: one CTA per (batch, head, chunk, 64-column half of V).  The
// chunk's masked q k^T is computed once per CTA (twice per chunk for V = 128,
// against four times with 32-column tiles) and the o tile is a 4 x 4 register
// tile per thread.  The h half-tile [K][64] is loaded into registers while
// q k^T is computed, and is stored into the space of the transposed k once
// q k^T no longer needs it.
constexpr int kVO = 64;                 // V columns per chunk_fwd_o CTA
constexpr int kHPerThread = 128 * kVO / kGdnThreads;   // 32: h values a thread carries (K <= 128)
template <int C>
__global__ void __launch_bounds__(kGdnThreads)
gdn_fwd_o_kernel(const float* __restrict__ q, const float* __restrict__ k,
                 const float* __restrict__ v_new, const float* __restrict__ h,
                 const float* __restrict__ g, float* __restrict__ o, int T, int H, int K, int V,
                 int NT) {
    extern __shared__ __align__(16) float sm[];
    constexpr int CP = C + 4;
    const int KH = K * (CP > kVO ? CP : kVO);
    float* qT = sm;                     // [K][C+4] q, transposed
    float* kT = qT + K * CP;            // [K][C+4] k, transposed (A phase) ...
    float* hs = kT;                     // ... then [K][64] h (o phase)
    float* vs = kT + KH;                // [C][64]
    float* AT = vs + C * kVO;           // [C][C+4] A, transposed: AT[j][i]
    float* gs = AT + C * CP;            // [C]
    const int bh = blockIdx.x, b = bh / H, hh = bh - b * H, c = blockIdx.y;
    const int v0 = blockIdx.z * kVO;
    const int t0 = c * C, nt = min(C, T - t0);
    // this thread's column of the h and v_new tiles, and its first row
    const int col = threadIdx.x & (kVO - 1), row0 = threadIdx.x / kVO;
    constexpr int kRowStep = kGdnThreads / kVO;   // 4
    const bool cok = v0 + col < V;
    const float* hc = h + (((int64_t)bh * NT + c) * K) * V + v0 + col;
    float hv[kHPerThread];
#pragma unroll
    for (int r = 0; r < kHPerThread; ++r) {
        const int kk = row0 + kRowStep * r;
        hv[r] = (kk < K && cok) ? __ldg(hc + (int64_t)kk * V) : 0.f;
    }
    stage_transposed<C>(q, qT, b, T, t0, nt, H, hh, K);
    stage_transposed<C>(k, kT, b, T, t0, nt, H, hh, K);
    {
        constexpr int kVRows = C / kRowStep;
        float xv[kVRows];
#pragma unroll
        for (int r = 0; r < kVRows; ++r) {
            const int t = row0 + kRowStep * r;
            xv[r] = (t < nt && cok) ? __ldg(v_new + ((int64_t)(b * T + t0 + t) * H + hh) * V + v0 + col) : 0.f;
        }
#pragma unroll
        for (int r = 0; r < kVRows; ++r) vs[(row0 + kRowStep * r) * kVO + col] = xv[r];
    }
    if ((int)threadIdx.x < C) gs[threadIdx.x] = (int)threadIdx.x < nt ? g[(int64_t)(b * T + t0 + threadIdx.x) * H + hh] : 0.f;
    __syncthreads();
    // A = (q k^T) o exp(g_i - g_j), j <= i: 4 x 4 tiles (rows 4 ti, columns 4 tj)
    {
        const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
        if (4 * ti < C && 4 * tj < C) {
            float a[4][4] = {};
            if (4 * tj <= 4 * ti + 3) {   // tiles wholly above the diagonal stay zero
                #pragma unroll 4
                for (int kk = 0; kk < K; ++kk) {
                    const float4 qv = *reinterpret_cast<const float4*>(qT + kk * CP + 4 * ti);
                    const float4 kv = *reinterpret_cast<const float4*>(kT + kk * CP + 4 * tj);
                    const float qr[4] = {qv.x, qv.y, qv.z, qv.w}, kr[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int s2 = 0; s2 < 4; ++s2) a[r][s2] = fmaf(qr[r], kr[s2], a[r][s2]);
                }
            }
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                const int j = 4 * tj + s2;
                float cl[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = 4 * ti + r;
                    cl[r] = (j <= i && i < nt) ? a[r][s2] * expf(gs[i] - gs[j]) : 0.f;
                }
                *reinterpret_cast<float4*>(AT + j * CP + 4 * ti) = make_float4(cl[0], cl[1], cl[2], cl[3]);
            }
        }
    }
    __syncthreads();   // every read of kT is done: h takes its place
#pragma unroll
    for (int r = 0; r < kHPerThread; ++r) {
        const int kk = row0 + kRowStep * r;
        if (kk < K) hs[kk * kVO + col] = hv[r];
    }
    __syncthreads();
    // o[i] = exp(g_i) q_i h + sum_{j <= i} A[i][j] v_new[j]: rows 4 ti, columns 4 tv
    {
        const int ti = threadIdx.x >> 4, tv = threadIdx.x & 15;
        if (4 * ti < C) {
            float in[4][4] = {}, ia[4][4] = {};
            #pragma unroll 4
            for (int kk = 0; kk < K; ++kk) {
                const float4 qv = *reinterpret_cast<const float4*>(qT + kk * CP + 4 * ti);
                const float4 hv4 = *reinterpret_cast<const float4*>(hs + kk * kVO + 4 * tv);
                const float qr[4] = {qv.x, qv.y, qv.z, qv.w}, hr[4] = {hv4.x, hv4.y, hv4.z, hv4.w};
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) in[r][s2] = fmaf(qr[r], hr[s2], in[r][s2]);
            }
            const int jmax = min(nt, 4 * ti + 4);
            #pragma unroll 4
            for (int j = 0; j < jmax; ++j) {
                const float4 av = *reinterpret_cast<const float4*>(AT + j * CP + 4 * ti);
                const float4 xv = *reinterpret_cast<const float4*>(vs + j * kVO + 4 * tv);
                const float ar[4] = {av.x, av.y, av.z, av.w}, xr[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) ia[r][s2] = fmaf(ar[r], xr[s2], ia[r][s2]);
            }
            const int vc = v0 + 4 * tv;   // this thread's first column
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = 4 * ti + r;
                if (i < nt) {
                    const float eg = expf(gs[i]);
                    float* orow = o + ((int64_t)(b * T + t0 + i) * H + hh) * V;
                    float ov[4];
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) ov[s2] = in[r][s2] * eg + ia[r][s2];
                    if ((V & 3) == 0 && vc + 3 < V) {
                        *reinterpret_cast<float4*>(orow + vc) = make_float4(ov[0], ov[1], ov[2], ov[3]);
                    } else {
#pragma unroll
                        for (int s2 = 0; s2 < 4; ++s2)
                            if (vc + s2 < V) orow[vc + s2] = ov[s2];
                    }
                }
            }
        }
    }
}

template <int C>
cudaError_t launch_c(const GdnProblem& p, bool fwd_h, const float* q, const float* k,
                     const float* w, const float* u, const float* g, const float* h0, float* h,
                     float* v_new, float* final_state, float* o, cudaStream_t stream) {
    const int K = (int)p.K, V = (int)p.V, NT = (int)p.NT, T = (int)p.T, H = (int)p.H;
    const unsigned vtiles = (unsigned)((V + kVT - 1) / kVT);
    cudaError_t e;
    if (fwd_h) {
        const size_t smem = (size_t)(C * K + K * (C + 4) + K * kVT + C * kVT + C) * sizeof(float);
        auto kern = gdn_fwd_h_kernel<C>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
            return e;
        kern<<<dim3((unsigned)(p.B * p.H), vtiles), kGdnThreads, smem, stream>>>(
            k, w, u, g, h0, h, v_new, final_state, T, H, K, V, NT);
    } else {
        const int kh = K * ((C + 4) > kVO ? (C + 4) : kVO);
        const size_t smem =
            (size_t)(K * (C + 4) + kh + C * kVO + C * (C + 4) + C) * sizeof(float);
        auto kern = gdn_fwd_o_kernel<C>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
            return e;
        const unsigned vhalves = (unsigned)((V + kVO - 1) / kVO);
        kern<<<dim3((unsigned)(p.B * p.H), (unsigned)NT, vhalves), kGdnThreads, smem, stream>>>(
            q, k, v_new, h, g, o, T, H, K, V, NT);
    }
    return cudaGetLastError();
}

cudaError_t launch_any(const GdnProblem& p, bool fwd_h, const float* q, const float* k,
                       const float* w, const float* u, const float* g, const float* h0, float* h,
                       float* v_new, float* final_state, float* o, cudaStream_t stream) {
    switch (p.C) {
        case 16: return launch_c<16>(p, fwd_h, q, k, w, u, g, h0, h, v_new, final_state, o, stream);
        case 32: return launch_c<32>(p, fwd_h, q, k, w, u, g, h0, h, v_new, final_state, o, stream);
        default: return launch_c<64>(p, fwd_h, q, k, w, u, g, h0, h, v_new, final_state, o, stream);
    }
}

}  // namespace

cudaError_t launch_gdn_fwd_h(const GdnProblem& p, const float* k, const float* w, const float* u,
                             const float* g, const float* h0, float* h, float* v_new,
                             float* final_state, cudaStream_t stream) {
    if (gdn_tf32_supports(p) && p.T > 0)   // tensor cores (tf32_path.cu)
        return launch_gdn_fwd_h_tf32(p, k, w, u, g, h0, h, v_new, final_state, stream);
    return launch_any(p, true, nullptr, k, w, u, g, h0, h, v_new, final_state, nullptr, stream);
}

cudaError_t launch_gdn_fwd_o(const GdnProblem& p, const float* q, const float* k,
                             const float* v_new, const float* h, const float* g, float* o,
                             cudaStream_t stream) {
    if (gdn_tf32_supports(p))   // tensor cores (tf32_path.cu)
        return launch_gdn_fwd_o_tf32(p, q, k, v_new, h, g, o, stream);
    return launch_any(p, false, q, k, nullptr, nullptr, g, nullptr, const_cast<float*>(h),
                      const_cast<float*>(v_new), nullptr, o, stream);
}

}  // namespace ssd
