/*
 * ssd_oracle.c -- the CPU oracle for the Mamba-2 SSD forward pass (and the
 * causal depthwise conv1d that precedes it in a Mamba-2 block).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or constant with the CUDA
 * library; the two meet only through the seeded input generator.
 *
 * Everything is plain, single-threaded fp64 C with no blocking, fusion or
 * reordering beyond what the cited definition states, so that it can be read
 * against the source by eye.
 *
 * Sources (cited by page title and section):
 *   [P1] "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
 *        NVIDIA CUDA Tile" (trishampatil.com), sections "The Mamba-2
 *        Recurrence", "Step 1: Jump the State Across a Chunk with One Matmul",
 *        "Step 2: Compute a Chunk of Outputs from One State", "Step 3: Add Back
 *        the Decay, Safely, in Log-Space", "Kernel 1: chunk_cumsum".
 *   [P2] The zhiding.cn Chinese rendering of the NVIDIA / Jane Street cuTile
 *        Mamba-2 article, section "Mamba-2架构" (the recurrence and the chunked
 *        closed forms, given there as LaTeX).
 *   [P3] The Helion hackathon gallery (cerebralvalley.ai), its "Causal Conv1d
 *        (causal_conv1d)" entries (the convolution's definition).
 *
 * Layouts (row-major, contiguous; b = batch, t = token, h = head, g = group):
 *   x    [batch, seqlen, nheads, headdim]      dt   [batch, seqlen, nheads]
 *   B, C [batch, seqlen, ngroups, dstate]      A, D [nheads]
 *   init, final [batch, nheads, headdim, dstate]   y [batch, seqlen, nheads, headdim]
 * The state of one head is held as S[p][n] (headdim x dstate); the pages write
 * the same matrix as (dstate x headdim), which changes nothing in the math.
 * Head h reads group h / (nheads / ngroups) of B and C ([P1] "Kernel 2:
 * fwd_pass_state", the group index used by the kernel body).
 *
 * Parity status of each function is recorded in its comment; every function
 * here is pinned by the CPU tests (tests/test_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARGS 1
#define ORACLE_NO_MEMORY 2

static int dims_ok(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                   int64_t dstate, int64_t ngroups) {
    if (batch < 0 || seqlen < 0 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1)
        return 0;
    if (nheads % ngroups != 0) return 0;
    return 1;
}

/*
 * ssd_oracle_recurrence -- the plain sequential recurrence, token by token.
 *
 * [P2] "Mamba-2架构": h_t = exp(A*dt_t) h_{t-1} + dt_t B_t x_t^T and
 * y_t = c_t^T h_t + D x_t.  [P1] "The Mamba-2 Recurrence" states the same
 * (dt_t > 0, A < 0, so exp(A*dt_t) lies in (0, 1]).  The output reads the
 * state AFTER the token-t update (h_t, not h_{t-1}): the causal mask of the
 * chunk form keeps the diagonal, which needs h_t.
 *
 * Arguments: D may be NULL (treated as 0); init may be NULL (zero state);
 * final_state may be NULL (not written).  If ckpt is not NULL and
 * ckpt_every > 0, the state held BEFORE token c*ckpt_every is written to
 * ckpt[b, h, c] for c = 0 .. ceil(seqlen/ckpt_every)-1 (layout
 * [batch, nheads, nchunks, headdim, dstate]); these are the chunk-start
 * states that the chunked method carries between chunks.
 * Returns 0 on success, nonzero on bad arguments or allocation failure.
 */
int ssd_oracle_recurrence(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                          int64_t dstate, int64_t ngroups,
                          const double* x, const double* dt, const double* A,
                          const double* B, const double* C, const double* D,
                          const double* init, double* y, double* final_state,
                          int64_t ckpt_every, double* ckpt) {
    if (!dims_ok(batch, seqlen, nheads, headdim, dstate, ngroups)) return ORACLE_BAD_ARGS;
    if (!x || !dt || !A || !B || !C || !y) return ORACLE_BAD_ARGS;
    const int64_t P = headdim, N = dstate, H = nheads, G = ngroups, L = seqlen;
    const int64_t heads_per_group = H / G;
    const int64_t nchunks = (ckpt && ckpt_every > 0) ? (L + ckpt_every - 1) / ckpt_every : 0;
    double* S = (double*)malloc((size_t)(P * N) * sizeof(double));
    if (!S) return ORACLE_NO_MEMORY;

    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            const int64_t g = h / heads_per_group;
            if (init) memcpy(S, init + ((b * H + h) * P) * N, (size_t)(P * N) * sizeof(double));
            else memset(S, 0, (size_t)(P * N) * sizeof(double));

            for (int64_t t = 0; t < L; ++t) {
                if (nchunks > 0 && t % ckpt_every == 0) {
                    double* dst = ckpt + (((b * H + h) * nchunks + t / ckpt_every) * P) * N;
                    memcpy(dst, S, (size_t)(P * N) * sizeof(double));
                }
                const double dtv = dt[(b * L + t) * H + h];
                const double decay = exp(A[h] * dtv);
                const double* xt = x + ((b * L + t) * H + h) * P;
                const double* Bt = B + ((b * L + t) * G + g) * N;
                const double* Ct = C + ((b * L + t) * G + g) * N;
                /* h_t = exp(a_t) h_{t-1} + b_t x_t^T with b_t = dt_t B_t */
                for (int64_t p = 0; p < P; ++p)
                    for (int64_t n = 0; n < N; ++n)
                        S[p * N + n] = decay * S[p * N + n] + dtv * Bt[n] * xt[p];
                /* y_t = c_t^T h_t + D x_t */
                double* yt = y + ((b * L + t) * H + h) * P;
                const double Dh = D ? D[h] : 0.0;
                for (int64_t p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) acc += Ct[n] * S[p * N + n];
                    yt[p] = acc + Dh * xt[p];
                }
            }
            if (final_state)
                memcpy(final_state + ((b * H + h) * P) * N, S, (size_t)(P * N) * sizeof(double));
        }
    }
    free(S);
    return ORACLE_OK;
}

/*
 * ssd_oracle_chunk_cumsum -- the per-chunk cumulative decay sums.
 *
 * [P1] "Kernel 1: chunk_cumsum": for head h and token t in chunk c,
 * G[b, h, t] = log2(e) * sum_{k = c*Q .. t} A[h] * dt[b, k, h]: an inclusive
 * sum that restarts at every chunk start, scaled by log2(e) so that the later
 * exponentials can be taken base 2 (e^v = 2^(v log2 e)).  The output here is
 * laid out [batch, nheads, seqlen] (the token-contiguous layout that [P2]
 * "Mamba-2性能优化" recommends); the pages' kernel stores [batch, seqlen, nheads].
 * Returns 0 on success.
 */
int ssd_oracle_chunk_cumsum(int64_t batch, int64_t seqlen, int64_t nheads, int64_t chunk,
                            const double* dt, const double* A, double* G) {
    if (batch < 0 || seqlen < 0 || nheads < 1 || chunk < 1 || !dt || !A || !G)
        return ORACLE_BAD_ARGS;
    const double log2e = 1.0 / log(2.0);
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t h = 0; h < nheads; ++h) {
            double run = 0.0;
            for (int64_t t = 0; t < seqlen; ++t) {
                if (t % chunk == 0) run = 0.0;
                run += A[h] * dt[(b * seqlen + t) * nheads + h];
                G[(b * nheads + h) * seqlen + t] = log2e * run;
            }
        }
    return ORACLE_OK;
}

/*
 * ssd_oracle_chunked -- the chunked closed form, used ONLY to pin the
 * recurrence above (it is an independent evaluation of the same function).
 *
 * [P2] "Mamba-2架构" and [P1] "Step 3: Add Back the Decay, Safely, in
 * Log-Space": inside a chunk of T tokens with start state h, let g hold the
 * inclusive cumulative sum of a_t = A*dt_t (natural log space here, no base-2
 * scaling) and g_last its value at the chunk's last token.  Then
 *   h_next = exp(g_last) h + (exp(g_last - g) * B)^T X            (jump)
 *   Y = exp(g) * (C h) + ((exp(g_i - g_j) * (C B^T)) o M) X + D X  (outputs)
 * with b_j = dt_j B_j (so the dt factor rides on B), M the causal mask that
 * keeps j <= i.  A ragged last chunk simply has fewer tokens; g_last is the
 * value at its last real token.  Arguments as ssd_oracle_recurrence, plus the
 * chunk length Q >= 1.
 */
int ssd_oracle_chunked(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                       int64_t dstate, int64_t ngroups, int64_t Q,
                       const double* x, const double* dt, const double* A,
                       const double* B, const double* C, const double* D,
                       const double* init, double* y, double* final_state) {
    if (!dims_ok(batch, seqlen, nheads, headdim, dstate, ngroups) || Q < 1) return ORACLE_BAD_ARGS;
    if (!x || !dt || !A || !B || !C || !y) return ORACLE_BAD_ARGS;
    const int64_t P = headdim, N = dstate, H = nheads, G = ngroups, L = seqlen;
    const int64_t heads_per_group = H / G;
    double* S = (double*)malloc((size_t)(P * N) * sizeof(double));
    double* Snew = (double*)malloc((size_t)(P * N) * sizeof(double));
    double* g = (double*)malloc((size_t)Q * sizeof(double));
    if (!S || !Snew || !g) { free(S); free(Snew); free(g); return ORACLE_NO_MEMORY; }

    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            const int64_t grp = h / heads_per_group;
            if (init) memcpy(S, init + ((b * H + h) * P) * N, (size_t)(P * N) * sizeof(double));
            else memset(S, 0, (size_t)(P * N) * sizeof(double));
            const double Dh = D ? D[h] : 0.0;

            for (int64_t c0 = 0; c0 < L; c0 += Q) {
                const int64_t T = (L - c0 < Q) ? (L - c0) : Q;
                double run = 0.0;
                for (int64_t i = 0; i < T; ++i) {
                    run += A[h] * dt[(b * L + c0 + i) * H + h];
                    g[i] = run;
                }
                const double glast = g[T - 1];

                /* outputs of the chunk from the chunk-start state S */
                for (int64_t i = 0; i < T; ++i) {
                    const int64_t ti = c0 + i;
                    const double* Ci = C + ((b * L + ti) * G + grp) * N;
                    const double* xi = x + ((b * L + ti) * H + h) * P;
                    double* yi = y + ((b * L + ti) * H + h) * P;
                    for (int64_t p = 0; p < P; ++p) {
                        /* exp(g_i) * (C h)_i */
                        double inter = 0.0;
                        for (int64_t n = 0; n < N; ++n) inter += Ci[n] * S[p * N + n];
                        /* sum_{j<=i} exp(g_i - g_j) (C_i . B_j) dt_j x_j */
                        double intra = 0.0;
                        for (int64_t j = 0; j <= i; ++j) {
                            const int64_t tj = c0 + j;
                            const double* Bj = B + ((b * L + tj) * G + grp) * N;
                            double cb = 0.0;
                            for (int64_t n = 0; n < N; ++n) cb += Ci[n] * Bj[n];
                            intra += exp(g[i] - g[j]) * cb * dt[(b * L + tj) * H + h] *
                                     x[((b * L + tj) * H + h) * P + p];
                        }
                        yi[p] = exp(g[i]) * inter + intra + Dh * xi[p];
                    }
                }

                /* jump the state across the chunk */
                for (int64_t p = 0; p < P; ++p)
                    for (int64_t n = 0; n < N; ++n) {
                        double acc = 0.0;
                        for (int64_t j = 0; j < T; ++j) {
                            const int64_t tj = c0 + j;
                            acc += exp(glast - g[j]) * dt[(b * L + tj) * H + h] *
                                   B[((b * L + tj) * G + grp) * N + n] *
                                   x[((b * L + tj) * H + h) * P + p];
                        }
                        Snew[p * N + n] = exp(glast) * S[p * N + n] + acc;
                    }
                memcpy(S, Snew, (size_t)(P * N) * sizeof(double));
            }
            if (final_state)
                memcpy(final_state + ((b * H + h) * P) * N, S, (size_t)(P * N) * sizeof(double));
        }
    }
    free(S); free(Snew); free(g);
    return ORACLE_OK;
}

/*
 * ssd_oracle_causal_conv1d -- depthwise causal 1-D convolution, the Mamba /
 * Mamba-2 block's neighbour of the SSD (parity pinned: tests/oracle_pins.py).
 *
 * [P3] Helion hackathon gallery, the "Causal Conv1d (causal_conv1d)" entry:
 * each channel is convolved independently with a short filter of W taps,
 * with causal (left) zero padding:
 *   out[b, d, t] = bias[d] + sum_{k=0}^{W-1} weight[d, k] * x[b, d, t - W + 1 + k],
 * where x at a negative time index reads as 0.
 * Layouts: x, out [batch, dim, seqlen]; weight [dim, width]; bias [dim] or
 * NULL (treated as 0).  Returns 0 on success.
 */
int ssd_oracle_causal_conv1d(int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                             const double* x, const double* weight, const double* bias,
                             double* out) {
    if (batch < 0 || dim < 1 || seqlen < 0 || width < 1 || !x || !weight || !out)
        return ORACLE_BAD_ARGS;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const double* xr = x + (b * dim + d) * seqlen;
            double* orow = out + (b * dim + d) * seqlen;
            for (int64_t t = 0; t < seqlen; ++t) {
                double acc = bias ? bias[d] : 0.0;
                for (int64_t k = 0; k < width; ++k) {
                    const int64_t ts = t - width + 1 + k;
                    if (ts >= 0) acc += weight[d * width + k] * xr[ts];
                }
                orow[t] = acc;
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Gated DeltaNet chunk kernels -- a second chunked recurrence with the shape
 * of fwd_pass_state / compute_out.
 *
 * [P3] Helion hackathon gallery, the "GDN chunk_fwd_h" and "GDN chunk_fwd_o"
 * entries, chunk size C.  Layouts: k, w, q [B, T, H, K]; u, v_new, o
 * [B, T, H, V]; g [B, T, H] = the in-chunk inclusive cumulative log gate
 * (natural log, <= 0); h [B, H, NT, K, V] the state at each chunk start;
 * h0, final_state [B, H, K, V] (h0 may be NULL: zero state).  g_last is g at
 * the chunk's last valid token (a ragged last chunk ends at T).
 *
 * ssd_oracle_gdn_fwd_h, per chunk in order, the page's five steps:
 *   (1) store h; (2) v_new = u - w @ h; (3) gate: v_gated[t] = v_new[t] *
 *   exp(g_last - g_t); (4) decay: h *= exp(g_last); (5) h += k^T @ v_gated.
 * Returns 0 on success.
 */
int ssd_oracle_gdn_fwd_h(int64_t batch, int64_t seqlen, int64_t nheads, int64_t kdim, int64_t vdim,
                         int64_t chunk, const double* k, const double* w, const double* u,
                         const double* g, const double* h0, double* h, double* v_new,
                         double* final_state) {
    if (batch < 0 || seqlen < 0 || nheads < 1 || kdim < 1 || vdim < 1 || chunk < 1) return ORACLE_BAD_ARGS;
    if (!k || !w || !u || !g || !h || !v_new) return ORACLE_BAD_ARGS;
    const int64_t H = nheads, K = kdim, V = vdim, T = seqlen, NT = (T + chunk - 1) / chunk;
    double* S = (double*)malloc((size_t)(K * V) * sizeof(double));
    double* vg = (double*)malloc((size_t)(chunk * V) * sizeof(double));
    if (!S || !vg) { free(S); free(vg); return ORACLE_NO_MEMORY; }
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t hh = 0; hh < H; ++hh) {
            if (h0) memcpy(S, h0 + (b * H + hh) * K * V, (size_t)(K * V) * sizeof(double));
            else memset(S, 0, (size_t)(K * V) * sizeof(double));
            for (int64_t c = 0; c < NT; ++c) {
                const int64_t t0 = c * chunk, t1 = (t0 + chunk < T) ? t0 + chunk : T;
                /* (1) store the chunk-start state */
                memcpy(h + ((b * H + hh) * NT + c) * K * V, S, (size_t)(K * V) * sizeof(double));
                const double g_last = g[(b * T + t1 - 1) * H + hh];
                for (int64_t t = t0; t < t1; ++t) {
                    const double* wt = w + ((b * T + t) * H + hh) * K;
                    const double* ut = u + ((b * T + t) * H + hh) * V;
                    double* vt = v_new + ((b * T + t) * H + hh) * V;
                    const double gate = exp(g_last - g[(b * T + t) * H + hh]);
                    for (int64_t v = 0; v < V; ++v) {
                        /* (2) v_new = u - w @ h */
                        double acc = 0.0;
                        for (int64_t kk = 0; kk < K; ++kk) acc += wt[kk] * S[kk * V + v];
                        vt[v] = ut[v] - acc;
                        /* (3) gate */
                        vg[(t - t0) * V + v] = vt[v] * gate;
                    }
                }
                /* (4) decay, then (5) h += k^T @ v_gated */
                const double decay = exp(g_last);
                for (int64_t kk = 0; kk < K; ++kk)
                    for (int64_t v = 0; v < V; ++v) {
                        double acc = S[kk * V + v] * decay;
                        for (int64_t t = t0; t < t1; ++t)
                            acc += k[((b * T + t) * H + hh) * K + kk] * vg[(t - t0) * V + v];
                        S[kk * V + v] = acc;
                    }
            }
            if (final_state)
                memcpy(final_state + (b * H + hh) * K * V, S, (size_t)(K * V) * sizeof(double));
        }
    }
    free(S);
    free(vg);
    return ORACLE_OK;
}

/*
 * ssd_oracle_gdn_fwd_o, per chunk, the page's three products:
 *   inter[t] = (q_t @ h) * exp(g_t);
 *   intra[i] = sum_{j <= i} (q_i . k_j) exp(g_i - g_j) v_new[j]   (the causal mask keeps j = i);
 *   o = inter + intra.
 * h is the chunk-start state from ssd_oracle_gdn_fwd_h.  Returns 0 on success.
 */
int ssd_oracle_gdn_fwd_o(int64_t batch, int64_t seqlen, int64_t nheads, int64_t kdim, int64_t vdim,
                         int64_t chunk, const double* q, const double* k, const double* v_new,
                         const double* h, const double* g, double* o) {
    if (batch < 0 || seqlen < 0 || nheads < 1 || kdim < 1 || vdim < 1 || chunk < 1) return ORACLE_BAD_ARGS;
    if (!q || !k || !v_new || !h || !g || !o) return ORACLE_BAD_ARGS;
    const int64_t H = nheads, K = kdim, V = vdim, T = seqlen, NT = (T + chunk - 1) / chunk;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t hh = 0; hh < H; ++hh) {
            for (int64_t c = 0; c < NT; ++c) {
                const int64_t t0 = c * chunk, t1 = (t0 + chunk < T) ? t0 + chunk : T;
                const double* S = h + ((b * H + hh) * NT + c) * K * V;
                for (int64_t i = t0; i < t1; ++i) {
                    const double* qi = q + ((b * T + i) * H + hh) * K;
                    const double gi = g[(b * T + i) * H + hh];
                    double* oi = o + ((b * T + i) * H + hh) * V;
                    for (int64_t v = 0; v < V; ++v) {
                        double inter = 0.0;
                        for (int64_t kk = 0; kk < K; ++kk) inter += qi[kk] * S[kk * V + v];
                        oi[v] = inter * exp(gi);
                    }
                    for (int64_t j = t0; j <= i; ++j) {
                        const double* kj = k + ((b * T + j) * H + hh) * K;
                        double qk = 0.0;
                        for (int64_t kk = 0; kk < K; ++kk) qk += qi[kk] * kj[kk];
                        const double a = qk * exp(gi - g[(b * T + j) * H + hh]);
                        const double* vj = v_new + ((b * T + j) * H + hh) * V;
                        for (int64_t v = 0; v < V; ++v) oi[v] += a * vj[v];
                    }
                }
            }
        }
    }
    return ORACLE_OK;
}
