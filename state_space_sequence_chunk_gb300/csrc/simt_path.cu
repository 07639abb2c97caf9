// simt_path.cu -- fwd_pass_state and compute_out on the CUDA cores (fp32 FMA),
// and the dispatch of both steps between these kernels and the tensor-core
// ones (tcgen05: bf16 in fwd_pass_state_tc.cu / compute_out_tc.cu, TF32 in
// tf32_path.cu).
//
// These are the straightforward tiled forms of steps 2 and 3 of "Accelerating
// Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA CUDA Tile"
// (sections "Kernel 2: fwd_pass_state" and "Kernel 3: compute_out"), with all
// arithmetic in fp32; they serve the shapes the tensor-core kernels do not
// (fp32 with N or P above 128, bf16 compute_out with P > 64 or N > 128).
#include "sm100_ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// fwd_pass_state on the CUDA cores (fp32 inputs, whose hiddens are fp32), in
// two kernels so that the chunks run in parallel:
//   fps_chunk_products: per (16 rows of P, chunk, batch*head), the chunk's
//     product D_c[p][n] = sum_q x[q][p] (dt_q 2^{g_last - g_q}) B[q][n], written
//     into that chunk's slot of hiddens (same size: [n][p], fp32);
//   fps_state_scan: per (state element, batch*head), over the chunks in order,
//     hiddens[c] <- S (replacing D_c), S <- 2^{g_last} S + D_c, from S = init.
// This is "Kernel 2: fwd_pass_state" with its loop over chunks split at the
// only serial step (the state update is linear in S); thread t of the
// products kernel owns row p = t / 16 and state columns n = t % 16 + 16 k.
// ---------------------------------------------------------------------------
constexpr int kPT = 16;    // rows of P per CTA
constexpr int kSub = 32;   // tokens per staged sub-chunk
constexpr int kMaxN = 256;

__global__ void __launch_bounds__(kThreads)
fps_chunk_products(const float* __restrict__ x, const float* __restrict__ B,
                   const float* __restrict__ Gcs, const float* __restrict__ dtT,
                   float* __restrict__ hiddens, int L, int H, int P, int N, int G, int Q, int nc,
                   int Lp, int hpg) {
    extern __shared__ float sm[];
    float* xs = sm;                    // [kSub][kPT]
    float* bs = xs + kSub * kPT;       // [kSub][N]
    float* sc = bs + kSub * N;         // [kSub] per-token scale
    const int p0 = blockIdx.x * kPT, c = blockIdx.y;
    const int bh = blockIdx.z, bidx = bh / H, h = bh % H, grp = h / hpg;
    const int tid = threadIdx.x, pl = tid / 16, nl = tid % 16;
    const int nper = N / 16;
    const float* grow = Gcs + (int64_t)bh * Lp;
    const float* drow = dtT + (int64_t)bh * Lp;
    const int t0 = c * Q;
    const float glast = grow[t0 + Q - 1];  // padded tokens repeat the last real value
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    for (int s0 = 0; s0 < Q; s0 += kSub) {
        __syncthreads();
        // loads: x 2 per thread, B up to kSub * kMaxN / threads = 32 per thread, all in flight
        {
            constexpr int kXPer = kSub * kPT / kThreads, kBPer = kSub * kMaxN / kThreads;
            float xv[kXPer], bv[kBPer];
#pragma unroll
            for (int r = 0; r < kXPer; ++r) {
                const int i = tid + r * kThreads, q = i / kPT, pp = i % kPT, tg = t0 + s0 + q;
                xv[r] = tg < L ? x[(((int64_t)bidx * L + tg) * H + h) * P + p0 + pp] : 0.f;
            }
#pragma unroll
            for (int r = 0; r < kBPer; ++r) {
                const int i = tid + r * kThreads, q = i / N, n = i % N, tg = t0 + s0 + q;
                bv[r] = (i < kSub * N && tg < L) ? B[(((int64_t)bidx * L + tg) * G + grp) * N + n] : 0.f;
            }
#pragma unroll
            for (int r = 0; r < kXPer; ++r) xs[tid + r * kThreads] = xv[r];
#pragma unroll
            for (int r = 0; r < kBPer; ++r)
                if (tid + r * kThreads < kSub * N) bs[tid + r * kThreads] = bv[r];
            if (tid < kSub) {
                const int tq = t0 + s0 + tid;
                sc[tid] = drow[tq] * exp2f(glast - grow[tq]);
            }
        }
        __syncthreads();
        for (int q = 0; q < kSub; ++q) {
            const float xv = xs[q * kPT + pl] * sc[q];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                if (k < nper) acc[k] = fmaf(xv, bs[q * N + nl + 16 * k], acc[k]);
        }
    }
    // D_c into the chunk's hiddens slot, [n][p]
    float* hrow = hiddens + (((int64_t)bidx * H + h) * nc + c) * (int64_t)N * P + p0 + pl;
#pragma unroll
    for (int k = 0; k < 16; ++k)
        if (k < nper) hrow[(int64_t)(nl + 16 * k) * P] = acc[k];
}

// One thread per state element (n, p) of one (batch, head): f = n P + p, so
// the hiddens slots are read and written coalesced.  Eight chunks' products
// are loaded before their serial fma chain.
constexpr int kScanBatch = 8;
__global__ void __launch_bounds__(kThreads)
fps_state_scan(const float* __restrict__ Gcs, const float* init, float* __restrict__ hiddens,
               float* final_state, int H, int P, int N, int Q, int nc, int Lp) {
    grid_launch_dependents();   // chained launch: compute_out may set up meanwhile
    grid_dependency_wait();     // the chunk products
    const int f = blockIdx.x * kThreads + threadIdx.x, bh = blockIdx.y;
    if (f >= P * N) return;
    const int n = f / P, p = f - n * P;
    const int64_t sidx = ((int64_t)bh * P + p) * N + n;
    float S = init != nullptr ? init[sidx] : 0.f;
    float* hb = hiddens + (int64_t)bh * nc * N * P + f;
    const float* grow = Gcs + (int64_t)bh * Lp + Q - 1;
    for (int c0 = 0; c0 < nc; c0 += kScanBatch) {
        float Dv[kScanBatch], gl[kScanBatch];
#pragma unroll
        for (int i = 0; i < kScanBatch; ++i) {
            const int c = c0 + i;
            Dv[i] = c < nc ? hb[(int64_t)c * N * P] : 0.f;
            gl[i] = c < nc ? grow[(int64_t)c * Q] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kScanBatch; ++i) {
            const int c = c0 + i;
            if (c < nc) {
                hb[(int64_t)c * N * P] = S;
                S = fmaf(exp2f(gl[i]), S, Dv[i]);
            }
        }
    }
    if (final_state != nullptr) final_state[sidx] = S;
}

// ---------------------------------------------------------------------------
// compute_out: one CTA per (32 query rows, chunk, batch*head).  Thread t owns
// row i = t / 8 and columns p = t % 8 + 8 k, k < KP (KP = 16 covers P <= 128,
// KP = 32 covers P <= 256).
//   acc = 2^{g_i} (C_i . h^T)
//   for each 32-token key block j <= i:
//       cb[i][j] = C_i . B_j, masked to j <= i and scaled by 2^{g_i - g_j} dt_j
//       acc += cb . X_j
//   y = acc + D x_i
// The mask is a select, so the unsafe above-diagonal exponentials never reach
// the output ("Kernel 3: compute_out").
// ---------------------------------------------------------------------------
constexpr int kRows = 32;

template <typename T, int KP>
__global__ void __launch_bounds__(kThreads)
compute_out_simt(const T* __restrict__ x, const T* __restrict__ B, const T* __restrict__ C,
                 const float* __restrict__ Gcs, const float* __restrict__ dtT,
                 const T* __restrict__ hiddens, const float* __restrict__ D, T* __restrict__ y,
                 int L, int H, int P, int N, int G, int Q, int nc, int Lp, int hpg) {
    extern __shared__ float sm[];
    const int NS = N + 1;              // padded row stride
    float* cs = sm;                    // [kRows][NS]   query rows of C
    float* bs = cs + kRows * NS;       // [kRows][NS]   key rows of B
    float* hs = bs + kRows * NS;       // [P][33]       32-column slice of h
    float* xs = hs + P * 33;           // [kRows][P]    key rows of X
    float* cb = xs + kRows * P;        // [kRows][33]
    float* gq = cb + kRows * 33;       // [Q]
    float* dq = gq + Q;                // [Q]

    const int i0 = blockIdx.x * kRows, c = blockIdx.y, bh = blockIdx.z;
    const int bidx = bh / H, h = bh % H, grp = h / hpg;
    const int tid = threadIdx.x, il = tid / 8, pl = tid % 8;
    const int pper = P / 8;
    const int t0 = c * Q;

    for (int i = tid; i < Q; i += kThreads) {
        gq[i] = Gcs[(int64_t)bh * Lp + t0 + i];
        dq[i] = dtT[(int64_t)bh * Lp + t0 + i];
    }
    for (int i = tid; i < kRows * N; i += kThreads) {
        const int r = i / N, n = i % N, tg = t0 + i0 + r;
        cs[r * NS + n] = tg < L ? to_f32(C[(((int64_t)bidx * L + tg) * G + grp) * N + n]) : 0.f;
    }

    float acc[KP];
#pragma unroll
    for (int k = 0; k < KP; ++k) acc[k] = 0.f;

    // state term C_i . h^T, h staged 32 state columns at a time
    const T* hbase = hiddens + (((int64_t)bidx * H + h) * nc + c) * (int64_t)P * N;
    for (int n0 = 0; n0 < N; n0 += 32) {
        __syncthreads();
        // consecutive threads read consecutive p of one state column (coalesced);
        // the odd row stride keeps the transposed smem writes conflict-free
#pragma unroll 4
        for (int i = tid; i < P * 32; i += kThreads) {
            const int nn = i / P, pp = i % P;
            hs[pp * 33 + nn] = (n0 + nn < N) ? to_f32(hbase[(int64_t)(n0 + nn) * P + pp]) : 0.f;
        }
        __syncthreads();
        const int nlim = min(32, N - n0);
        for (int nn = 0; nn < nlim; ++nn) {
            const float cv = cs[il * NS + n0 + nn];
#pragma unroll
            for (int k = 0; k < KP; ++k)
                if (k < pper) acc[k] = fmaf(cv, hs[(pl + 8 * k) * 33 + nn], acc[k]);
        }
    }
    const int irow = i0 + il;
    {
        const float sgi = exp2f(gq[irow]);
#pragma unroll
        for (int k = 0; k < KP; ++k) acc[k] *= sgi;
    }

    // intra-chunk term, key blocks j0 <= i0
    for (int j0 = 0; j0 <= i0; j0 += kRows) {
        __syncthreads();
#pragma unroll 4
        for (int i = tid; i < kRows * N; i += kThreads) {
            const int r = i / N, n = i % N, tg = t0 + j0 + r;
            bs[r * NS + n] = tg < L ? to_f32(B[(((int64_t)bidx * L + tg) * G + grp) * N + n]) : 0.f;
        }
#pragma unroll 4
        for (int i = tid; i < kRows * P; i += kThreads) {
            const int r = i / P, pp = i % P, tg = t0 + j0 + r;
            xs[i] = tg < L ? to_f32(x[(((int64_t)bidx * L + tg) * H + h) * P + pp]) : 0.f;
        }
        __syncthreads();
        // 32 x 32 block of C B^T: thread -> row il, columns pl + 8 k (k < 4)
        for (int k = 0; k < 4; ++k) {
            const int jl = pl + 8 * k;
            float s = 0.f;
            for (int n = 0; n < N; ++n) s = fmaf(cs[il * NS + n], bs[jl * NS + n], s);
            const int ig = i0 + il, jg = j0 + jl;
            // select, never multiply: 2^{g_i - g_j} may overflow above the diagonal
            const float w = (jg <= ig) ? s * exp2f(gq[ig] - gq[jg]) * dq[jg] : 0.f;
            cb[il * 33 + jl] = w;
        }
        __syncthreads();
        for (int jl = 0; jl < kRows; ++jl) {
            const float w = cb[il * 33 + jl];
#pragma unroll
            for (int k = 0; k < KP; ++k)
                if (k < pper) acc[k] = fmaf(w, xs[jl * P + pl + 8 * k], acc[k]);
        }
    }

    const int tg = t0 + irow;
    if (tg < L) {
        const float dv = D ? D[h] : 0.f;
        const int64_t base = (((int64_t)bidx * L + tg) * H + h) * P;
#pragma unroll
        for (int k = 0; k < KP; ++k) {
            if (k < pper) {
                const int pp = pl + 8 * k;
                y[base + pp] = from_f32<T>(acc[k] + dv * to_f32(x[base + pp]));
            }
        }
    }
}

cudaError_t launch_fps(const Problem& p, const void* x, const void* B, const float* Gcs,
                      const float* dtT, const float* init, void* hid, float* fin,
                      cudaStream_t stream) {
    const size_t smem = (size_t)(kSub * kPT + kSub * p.N + kSub) * sizeof(float);
    cudaError_t e;
    if (tf32_path_supports(p)) {
        // the chunk products on the tensor cores (TF32)
        if ((e = launch_fps_products_tf32(p, x, B, Gcs, dtT, hid, stream)) != cudaSuccess) return e;
    } else {
        e = cudaFuncSetAttribute(fps_chunk_products, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        fps_chunk_products<<<dim3((unsigned)(p.P / kPT), (unsigned)p.nc, (unsigned)(p.b * p.H)),
                             kThreads, smem, stream>>>((const float*)x, (const float*)B, Gcs, dtT,
                                                       (float*)hid, (int)p.L, (int)p.H, (int)p.P,
                                                       (int)p.N, (int)p.G, (int)p.Q, (int)p.nc,
                                                       (int)p.Lp, (int)p.hpg);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return launch_chained(fps_state_scan,
                          dim3((unsigned)((p.P * p.N + kThreads - 1) / kThreads), (unsigned)(p.b * p.H)),
                          dim3(kThreads), 0, stream, p.chained, Gcs, init, (float*)hid, fin, (int)p.H,
                          (int)p.P, (int)p.N, (int)p.Q, (int)p.nc, (int)p.Lp);
}

template <typename T>
cudaError_t launch_co(const Problem& p, const void* x, const void* B, const void* C,
                      const float* Gcs, const float* dtT, const void* hid, const float* D,
                      void* y, cudaStream_t stream) {
    const int NS = (int)p.N + 1;
    const size_t smem = (size_t)(2 * kRows * NS + p.P * 33 + kRows * p.P + kRows * 33 + 2 * p.Q) *
                        sizeof(float);
    auto kern = p.P > 128 ? compute_out_simt<T, 32> : compute_out_simt<T, 16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.Q / kRows), (unsigned)p.nc, (unsigned)(p.b * p.H));
    kern<<<grid, kThreads, smem, stream>>>((const T*)x, (const T*)B, (const T*)C, Gcs, dtT,
                                           (const T*)hid, D, (T*)y, (int)p.L, (int)p.H,
                                           (int)p.P, (int)p.N, (int)p.G, (int)p.Q, (int)p.nc,
                                           (int)p.Lp, (int)p.hpg);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_pass_state(const Problem& p, const void* x, const void* B,
                                  const float* Gcs, const float* dtT, const float* init,
                                  void* hiddens, float* final_state, void* scratch,
                                  bool ctrl_zeroed, cudaStream_t stream) {
    if (p.dtype == SSD_BF16) {
        if (!ctrl_zeroed) {
            const cudaError_t e = cudaMemsetAsync((char*)scratch + fwd_pass_state_ctrl_offset(p), 0,
                                                  fwd_pass_state_ctrl_bytes(p), stream);
            if (e != cudaSuccess) return e;
        }
        return launch_fwd_pass_state_tc(p, x, B, Gcs, dtT, init, hiddens, final_state, scratch,
                                        stream);
    }
    return launch_fps(p, x, B, Gcs, dtT, init, hiddens, final_state, stream);
}

cudaError_t launch_compute_out(const Problem& p, const void* x, const void* B, const void* C,
                               const float* Gcs, const float* dtT, const void* hiddens,
                               const float* D, void* y, cudaStream_t stream) {
    if (compute_out_tc_supports(p))
        return launch_compute_out_tc(p, x, B, C, Gcs, dtT, hiddens, D, y, stream);
    if (tf32_path_supports(p))
        return launch_compute_out_tf32(p, x, B, C, Gcs, dtT, hiddens, D, y, stream);
    if (p.dtype == SSD_BF16)
        return launch_co<__nv_bfloat16>(p, x, B, C, Gcs, dtT, hiddens, D, y, stream);
    return launch_co<float>(p, x, B, C, Gcs, dtT, hiddens, D, y, stream);
}

}  // namespace ssd
