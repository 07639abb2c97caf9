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
// This first GB300 version runs on the CUDA cores in fp32.  A CTA owns a
// 32-column tile of V (lane = column), stages the chunk's K-wide rows of k, w
// (or q, k) in shared memory, and keeps its state tile in shared memory;
// every inner product reads one operand as a warp-wide broadcast and the
// other conflict-free.  chunk_fwd_h walks its chunks in order (one CTA per
// (batch, head, V tile)); chunk_fwd_o is one CTA per (batch, head, chunk,
// V tile).
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kGdnThreads = 256;   // 8 warps
constexpr int kVT = 32;            // V columns per CTA (one per lane)
constexpr int kWarps = kGdnThreads / 32;

template <int C>
__global__ void __launch_bounds__(kGdnThreads)
gdn_fwd_h_kernel(const float* __restrict__ k, const float* __restrict__ w,
                 const float* __restrict__ u, const float* __restrict__ g,
                 const float* __restrict__ h0, float* __restrict__ h, float* __restrict__ v_new,
                 float* __restrict__ final_state, int T, int H, int K, int V, int NT) {
    extern __shared__ float sm[];
    float* ks = sm;                 // [C][K]
    float* ws = ks + C * K;         // [C][K]
    float* S = ws + C * K;          // [K][32]
    float* vg = S + K * kVT;        // [C][32]
    float* gs = vg + C * kVT;       // [C]
    const int bh = blockIdx.x, b = bh / H, hh = bh - b * H;
    const int v0 = blockIdx.y * kVT, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v = v0 + lane;
    const bool vok = v < V;
    for (int kk = warp; kk < K; kk += kWarps)
        S[kk * kVT + lane] = (h0 != nullptr && vok) ? h0[((int64_t)bh * K + kk) * V + v] : 0.f;
    for (int c = 0; c < NT; ++c) {
        const int t0 = c * C, nt = min(C, T - t0);
        __syncthreads();   // the previous chunk's readers of ks / ws are done
        // rows of K floats, 16-byte vectors, several loads in flight per thread
        const int K4 = K >> 2;
#pragma unroll 4
        for (int i = threadIdx.x; i < nt * K4; i += kGdnThreads) {
            const int t = i / K4, k4 = i - t * K4;
            const int64_t src = ((int64_t)(b * T + t0 + t) * H + hh) * K + 4 * k4;
            reinterpret_cast<float4*>(ks)[i] = __ldg(reinterpret_cast<const float4*>(k + src));
            reinterpret_cast<float4*>(ws)[i] = __ldg(reinterpret_cast<const float4*>(w + src));
        }
        if ((int)threadIdx.x < nt) gs[threadIdx.x] = g[(int64_t)(b * T + t0 + threadIdx.x) * H + hh];
        __syncthreads();
        // (1) the chunk-start state
        float* hc = h + (((int64_t)bh * NT + c) * K) * V;
        if (vok)
            for (int kk = warp; kk < K; kk += kWarps) hc[(int64_t)kk * V + v] = S[kk * kVT + lane];
        const float g_last = gs[nt - 1];
        // (2) v_new = u - w h, (3) gate; tokens warp, warp + 8, ...
        float acc[C / kWarps];
#pragma unroll
        for (int i = 0; i < C / kWarps; ++i) acc[i] = 0.f;
        for (int kk = 0; kk < K; ++kk) {
            const float s = S[kk * kVT + lane];
#pragma unroll
            for (int i = 0; i < C / kWarps; ++i) acc[i] = fmaf(ws[(warp + kWarps * i) * K + kk], s, acc[i]);
        }
#pragma unroll
        for (int i = 0; i < C / kWarps; ++i) {
            const int t = warp + kWarps * i;
            if (t < nt) {
                const int64_t row = (int64_t)(b * T + t0 + t) * H + hh;
                const float vn = vok ? u[row * V + v] - acc[i] : 0.f;
                if (vok) v_new[row * V + v] = vn;
                vg[t * kVT + lane] = vn * expf(g_last - gs[t]);
            }
        }
        __syncthreads();
        // (4) decay and (5) h += k^T v_gated; state rows warp, warp + 8, ...
        const float decay = expf(g_last);
        for (int kb = warp; kb < K; kb += kWarps * 4) {
            float a4[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int kk = kb + kWarps * r;
                a4[r] = kk < K ? S[kk * kVT + lane] * decay : 0.f;
            }
            for (int t = 0; t < nt; ++t) {
                const float x = vg[t * kVT + lane];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int kk = kb + kWarps * r;
                    if (kk < K) a4[r] = fmaf(ks[t * K + kk], x, a4[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int kk = kb + kWarps * r;
                if (kk < K) S[kk * kVT + lane] = a4[r];
            }
        }
    }
    __syncthreads();
    if (final_state != nullptr && vok)
        for (int kk = warp; kk < K; kk += kWarps)
            final_state[((int64_t)bh * K + kk) * V + v] = S[kk * kVT + lane];
}

template <int C>
__global__ void __launch_bounds__(kGdnThreads)
gdn_fwd_o_kernel(const float* __restrict__ q, const float* __restrict__ k,
                 const float* __restrict__ v_new, const float* __restrict__ h,
                 const float* __restrict__ g, float* __restrict__ o, int T, int H, int K, int V,
                 int NT) {
    extern __shared__ float sm[];
    const int KP = K + 1;               // padded k rows: lanes read different rows
    float* qs = sm;                     // [C][K]
    float* ks = qs + C * K;             // [C][K + 1]
    float* hs = ks + C * KP;            // [K][32]
    float* vs = hs + K * kVT;           // [C][32]
    float* As = vs + C * kVT;           // [C][C + 1]
    float* gs = As + C * (C + 1);       // [C]
    const int bh = blockIdx.x, b = bh / H, hh = bh - b * H, c = blockIdx.y;
    const int v0 = blockIdx.z * kVT, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v = v0 + lane;
    const bool vok = v < V;
    const int t0 = c * C, nt = min(C, T - t0);
    const int K4 = K >> 2;
#pragma unroll 4
    for (int i = threadIdx.x; i < nt * K4; i += kGdnThreads) {
        const int t = i / K4, k4 = i - t * K4;
        const int64_t src = ((int64_t)(b * T + t0 + t) * H + hh) * K + 4 * k4;
        reinterpret_cast<float4*>(qs)[i] = __ldg(reinterpret_cast<const float4*>(q + src));
        const float4 kv = __ldg(reinterpret_cast<const float4*>(k + src));
        float* kd = ks + t * KP + 4 * k4;
        kd[0] = kv.x; kd[1] = kv.y; kd[2] = kv.z; kd[3] = kv.w;
    }
    const float* hc = h + (((int64_t)bh * NT + c) * K) * V;
#pragma unroll 4
    for (int kk = warp; kk < K; kk += kWarps) hs[kk * kVT + lane] = vok ? __ldg(hc + (int64_t)kk * V + v) : 0.f;
#pragma unroll 4
    for (int t = warp; t < nt; t += kWarps)
        vs[t * kVT + lane] = vok ? __ldg(v_new + ((int64_t)(b * T + t0 + t) * H + hh) * V + v) : 0.f;
    if ((int)threadIdx.x < nt) gs[threadIdx.x] = g[(int64_t)(b * T + t0 + threadIdx.x) * H + hh];
    __syncthreads();
    // A[i][j] = (q_i . k_j) exp(g_i - g_j) for j <= i, else 0; rows warp + 8a, columns lane + 32b
    for (int i = warp; i < nt; i += kWarps) {
        for (int j0 = 0; j0 < nt; j0 += 32) {
            const int j = j0 + lane;
            float a = 0.f;
            if (j <= i) {
                for (int kk = 0; kk < K; ++kk) a = fmaf(qs[i * K + kk], ks[j * KP + kk], a);
                a *= expf(gs[i] - gs[j]);
            }
            if (j < C) As[i * (C + 1) + j] = a;
        }
    }
    __syncthreads();
    // o[i] = exp(g_i) q_i h + sum_{j <= i} A[i][j] v_new[j]
    for (int i = warp; i < nt; i += kWarps) {
        float inter = 0.f;
        for (int kk = 0; kk < K; ++kk) inter = fmaf(qs[i * K + kk], hs[kk * kVT + lane], inter);
        float intra = 0.f;
        for (int j = 0; j <= i; ++j) intra = fmaf(As[i * (C + 1) + j], vs[j * kVT + lane], intra);
        if (vok) o[((int64_t)(b * T + t0 + i) * H + hh) * V + v] = inter * expf(gs[i]) + intra;
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
        const size_t smem = (size_t)(2 * C * K + K * kVT + C * kVT + C) * sizeof(float);
        auto kern = gdn_fwd_h_kernel<C>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
            return e;
        kern<<<dim3((unsigned)(p.B * p.H), vtiles), kGdnThreads, smem, stream>>>(
            k, w, u, g, h0, h, v_new, final_state, T, H, K, V, NT);
    } else {
        const size_t smem =
            (size_t)(C * K + C * (K + 1) + K * kVT + C * kVT + C * (C + 1) + C) * sizeof(float);
        auto kern = gdn_fwd_o_kernel<C>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
            return e;
        kern<<<dim3((unsigned)(p.B * p.H), (unsigned)NT, vtiles), kGdnThreads, smem, stream>>>(
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
    return launch_any(p, true, nullptr, k, w, u, g, h0, h, v_new, final_state, nullptr, stream);
}

cudaError_t launch_gdn_fwd_o(const GdnProblem& p, const float* q, const float* k,
                             const float* v_new, const float* h, const float* g, float* o,
                             cudaStream_t stream) {
    return launch_any(p, false, q, k, nullptr, nullptr, g, nullptr, const_cast<float*>(h),
                      const_cast<float*>(v_new), nullptr, o, stream);
}

}  // namespace ssd
