/*
 * neattn_ref.cpp -- fp64 CPU oracle for causal grouped-query self-attention with
 * rotary position embeddings (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes, and where the pages say so:
 *   - Causal self-attention: each position attends to itself and the positions
 *     before it ("Tiny hackable CUDA language model implementation", Core
 *     Mechanics, causal self-attention bullet).  Self is included (j <= i): with a
 *     strict mask row 0 would have no keys at all.
 *   - Grouped-query attention: a smaller set of key/value heads, each shared by
 *     several query heads ("NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의
 *     LLM", 기술 사양, GQA bullet; model-config table: Q/KV heads 4/2 and 12/4).
 *     Query head h uses key/value head h / G with G = Hq / Hkv (contiguous groups;
 *     the pages do not fix the mapping).
 *   - RoPE applied to queries and keys (same page, 기술 사양, RoPE bullet; "Tiny
 *     hackable ...", RoPE bullet: rotation matrices on queries and keys encode
 *     relative position).  Adjacent pairs (2i, 2i+1) are rotated by the angle
 *     t * theta^(-2i/D) at position t = 0..T-1.
 *   - The result is the one FlashAttention reaches without storing the T x T
 *     matrix (same page, 커널 구현).  This oracle DOES store it: it is the plain
 *     definition, softmax(s * Q' K'^T + causal mask) V with s = 1/sqrt(D).
 *   - Backward by hand, checked in double precision against central finite
 *     differences (same page, 검증 및 안정성; "NanoEuler – 순수 C/CUDA로 ...",
 *     Core Mechanics, second bullet).  Here the backward is the vector-Jacobian
 *     product of L = <dO, O> written out from the chain rule through softmax.
 *
 * Layout: Q, O, dO, dQ are [B, T, Hq, D]; K, V, dK, dV are [B, T, Hkv, D];
 * LSE and Delta are [B, Hq, T]; P is [B, Hq, T, T].  Everything is fp64, row-major.
 * LSE is the natural log of the row sum of exp of the scaled logits.
 */
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

inline int64_t idx4(int b, int t, int h, int d, int T, int H, int D) {
    return (((int64_t)b * T + t) * H + h) * D + d;
}

/* Angle of pair i at position t: t * theta^(-2i/D), formed directly in fp64. */
inline double rope_angle(int t, int i, int D, double theta) {
    return (double)t * std::pow(theta, -2.0 * (double)i / (double)D);
}

/* x' = R_t x on adjacent pairs: (x0, x1) -> (x0 c - x1 s, x0 s + x1 c). */
void rotate_row(const double* x, double* out, int t, int D, double theta) {
    for (int i = 0; i < D / 2; ++i) {
        double a = rope_angle(t, i, D, theta);
        double c = std::cos(a), s = std::sin(a);
        double x0 = x[2 * i], x1 = x[2 * i + 1];
        out[2 * i] = x0 * c - x1 * s;
        out[2 * i + 1] = x0 * s + x1 * c;
    }
}

/* y = R_t^T g: the transpose (inverse) rotation, used to pull gradients back. */
void rotate_row_transpose(const double* g, double* out, int t, int D, double theta) {
    for (int i = 0; i < D / 2; ++i) {
        double a = rope_angle(t, i, D, theta);
        double c = std::cos(a), s = std::sin(a);
        double g0 = g[2 * i], g1 = g[2 * i + 1];
        out[2 * i] = g0 * c + g1 * s;
        out[2 * i + 1] = -g0 * s + g1 * c;
    }
}

bool bad_shape(int B, int T, int Hq, int Hkv, int D) {
    return B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || (D % 2) != 0 ||
           (Hq % Hkv) != 0;
}

/* Rotated copy of one head's rows: out[t][d] = (R_t x_t)[d] for t < T. */
void rotated_head(const double* x, int b, int h, int T, int H, int D, double theta,
                  std::vector<double>& out) {
    out.assign((size_t)T * D, 0.0);
    for (int t = 0; t < T; ++t)
        rotate_row(&x[idx4(b, t, h, 0, T, H, D)], &out[(size_t)t * D], t, D, theta);
}

/* Materialised causal softmax for one (b, h): P[i][j] for j <= i, 0 above the
 * diagonal; lse[i] = ln sum_j exp(S_ij). */
void probs_one_head(const std::vector<double>& qr, const std::vector<double>& kr, int T,
                    int D, std::vector<double>& P, std::vector<double>& lse) {
    const double s = 1.0 / std::sqrt((double)D);
    P.assign((size_t)T * T, 0.0);
    lse.assign((size_t)T, 0.0);
    std::vector<double> S((size_t)T);
    for (int i = 0; i < T; ++i) {
        double m = -INFINITY;
        for (int j = 0; j <= i; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qr[(size_t)i * D + d] * kr[(size_t)j * D + d];
            S[j] = s * dot;
            if (S[j] > m) m = S[j];
        }
        double sum = 0.0;
        for (int j = 0; j <= i; ++j) sum += std::exp(S[j] - m);
        for (int j = 0; j <= i; ++j) P[(size_t)i * T + j] = std::exp(S[j] - m) / sum;
        lse[i] = m + std::log(sum);
    }
}

}  // namespace

extern "C" {

/* cos/sin of t * theta^(-2i/D) for t < T, i < D/2, each [T, D/2]. */
int ne_ref_rope_table(double* cos_out, double* sin_out, int T, int D, double theta) {
    if (T < 0 || D <= 0 || (D % 2) != 0) return 1;
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < D / 2; ++i) {
            double a = rope_angle(t, i, D, theta);
            cos_out[(size_t)t * (D / 2) + i] = std::cos(a);
            sin_out[(size_t)t * (D / 2) + i] = std::sin(a);
        }
    return 0;
}

/* Apply R_t to every row of x [B, T, H, D] (used by the tests to pin RoPE). */
int ne_ref_rope_apply(const double* x, double* out, int B, int T, int H, int D, double theta) {
    if (B < 0 || T < 0 || H <= 0 || D <= 0 || (D % 2) != 0) return 1;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t)
            for (int h = 0; h < H; ++h)
                rotate_row(&x[idx4(b, t, h, 0, T, H, D)], &out[idx4(b, t, h, 0, T, H, D)], t, D,
                           theta);
    return 0;
}

/* Forward: O = softmax(s Q'K'^T + mask) V, LSE.  P (optional, may be NULL) gets the
 * full [B, Hq, T, T] probability matrix. */
int ne_ref_attn_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                    double* P_out, int B, int T, int Hq, int Hkv, int D, double theta) {
    if (bad_shape(B, T, Hq, Hkv, D)) return 1;
    const int G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h) {
            const int g = h / G;
            std::vector<double> qr, kr, P, l;
            rotated_head(q, b, h, T, Hq, D, theta, qr);
            rotated_head(k, b, g, T, Hkv, D, theta, kr);
            probs_one_head(qr, kr, T, D, P, l);
            for (int i = 0; i < T; ++i) {
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int j = 0; j <= i; ++j)
                        acc += P[(size_t)i * T + j] * v[idx4(b, j, g, d, T, Hkv, D)];
                    o[idx4(b, i, h, d, T, Hq, D)] = acc;
                }
                lse[((int64_t)b * Hq + h) * T + i] = l[i];
            }
            if (P_out) {
                double* dst = P_out + ((int64_t)b * Hq + h) * (int64_t)T * T;
                std::memcpy(dst, P.data(), sizeof(double) * (size_t)T * T);
            }
        }
    return 0;
}

/* Backward: the VJP of L = <dO, O>.  Per (b, q head h) with kv head g = h / G:
 *   dP = dO V^T,  Delta_i = sum_j P_ij dP_ij,  dS = P o (dP - Delta),
 *   dQ' = s dS K',  dK' += s dS^T Q',  dV += P^T dO  (sums over the G heads of g),
 *   dQ = R^T dQ',   dK = R^T dK'.
 * delta_out (optional, may be NULL) gets Delta as [B, Hq, T]. */
int ne_ref_attn_bwd(const double* q, const double* k, const double* v, const double* dO,
                    double* dq, double* dk, double* dv, double* delta_out, int B, int T, int Hq,
                    int Hkv, int D, double theta) {
    if (bad_shape(B, T, Hq, Hkv, D)) return 1;
    const int G = Hq / Hkv;
    const double s = 1.0 / std::sqrt((double)D);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int g = 0; g < Hkv; ++g) {
            std::vector<double> kr, qr, P, l;
            rotated_head(k, b, g, T, Hkv, D, theta, kr);
            std::vector<double> dkr((size_t)T * D, 0.0), dvg((size_t)T * D, 0.0);
            std::vector<double> dP((size_t)T * T), dS((size_t)T * T), dqr((size_t)T * D);
            for (int h = g * G; h < (g + 1) * G; ++h) {
                rotated_head(q, b, h, T, Hq, D, theta, qr);
                probs_one_head(qr, kr, T, D, P, l);
                for (int i = 0; i < T; ++i) {
                    double delta = 0.0;
                    for (int j = 0; j <= i; ++j) {
                        double acc = 0.0;
                        for (int d = 0; d < D; ++d)
                            acc += dO[idx4(b, i, h, d, T, Hq, D)] * v[idx4(b, j, g, d, T, Hkv, D)];
                        dP[(size_t)i * T + j] = acc;
                        delta += P[(size_t)i * T + j] * acc;
                    }
                    for (int j = 0; j <= i; ++j)
                        dS[(size_t)i * T + j] = P[(size_t)i * T + j] * (dP[(size_t)i * T + j] - delta);
                    if (delta_out) delta_out[((int64_t)b * Hq + h) * T + i] = delta;
                }
                for (int i = 0; i < T; ++i)
                    for (int d = 0; d < D; ++d) {
                        double acc = 0.0;
                        for (int j = 0; j <= i; ++j) acc += dS[(size_t)i * T + j] * kr[(size_t)j * D + d];
                        dqr[(size_t)i * D + d] = s * acc;
                    }
                for (int j = 0; j < T; ++j)
                    for (int d = 0; d < D; ++d) {
                        double acck = 0.0, accv = 0.0;
                        for (int i = j; i < T; ++i) {
                            acck += dS[(size_t)i * T + j] * qr[(size_t)i * D + d];
                            accv += P[(size_t)i * T + j] * dO[idx4(b, i, h, d, T, Hq, D)];
                        }
                        dkr[(size_t)j * D + d] += s * acck;
                        dvg[(size_t)j * D + d] += accv;
                    }
                for (int t = 0; t < T; ++t)
                    rotate_row_transpose(&dqr[(size_t)t * D], &dq[idx4(b, t, h, 0, T, Hq, D)], t, D,
                                         theta);
            }
            for (int t = 0; t < T; ++t) {
                rotate_row_transpose(&dkr[(size_t)t * D], &dk[idx4(b, t, g, 0, T, Hkv, D)], t, D,
                                     theta);
                for (int d = 0; d < D; ++d) dv[idx4(b, t, g, d, T, Hkv, D)] = dvg[(size_t)t * D + d];
            }
        }
    return 0;
}

/* Selected query rows of one (b, q head h), for checks at sizes where the full matrices
 * do not fit: for each row i in rows[0..n) the same definitions as above restricted to
 * that row -- S_ij = s q'_i . k'_j (j <= i), P_ij = exp(S_ij - LSE_i), O_i = sum_j P_ij v_j,
 * and, when dO is given, dP_ij = dO_i . v_j, Delta_i = sum_j P_ij dP_ij,
 * dq_i = R_i^T s sum_j P_ij (dP_ij - Delta_i) k'_j.  Outputs are [n, D] (o, dq) and [n]
 * (lse, delta); dO, dq and delta may be NULL. */
int ne_ref_attn_qrows(const double* q, const double* k, const double* v, const double* dO, int b, int h,
                      const int* rows, int n, double* o, double* lse, double* dq, double* delta, int B,
                      int T, int Hq, int Hkv, int D, double theta) {
    if (bad_shape(B, T, Hq, Hkv, D) || b < 0 || b >= B || h < 0 || h >= Hq) return 1;
    for (int r = 0; r < n; ++r)
        if (rows[r] < 0 || rows[r] >= T) return 1;
    const int g = h / (Hq / Hkv);
    const double s = 1.0 / std::sqrt((double)D);
    std::vector<double> kr;
    rotated_head(k, b, g, T, Hkv, D, theta, kr);
#pragma omp parallel for schedule(dynamic)
    for (int r = 0; r < n; ++r) {
        const int i = rows[r];
        std::vector<double> qi((size_t)D), S((size_t)i + 1), P((size_t)i + 1), dP((size_t)i + 1);
        rotate_row(&q[idx4(b, i, h, 0, T, Hq, D)], qi.data(), i, D, theta);
        double m = -INFINITY;
        for (int j = 0; j <= i; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qi[d] * kr[(size_t)j * D + d];
            S[j] = s * dot;
            if (S[j] > m) m = S[j];
        }
        double sum = 0.0;
        for (int j = 0; j <= i; ++j) sum += std::exp(S[j] - m);
        const double l = m + std::log(sum);
        for (int j = 0; j <= i; ++j) P[j] = std::exp(S[j] - l);
        lse[r] = l;
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int j = 0; j <= i; ++j) acc += P[j] * v[idx4(b, j, g, d, T, Hkv, D)];
            o[(size_t)r * D + d] = acc;
        }
        if (!dO) continue;
        double dl = 0.0;
        for (int j = 0; j <= i; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += dO[idx4(b, i, h, d, T, Hq, D)] * v[idx4(b, j, g, d, T, Hkv, D)];
            dP[j] = acc;
            dl += P[j] * acc;
        }
        if (delta) delta[r] = dl;
        if (dq) {
            std::vector<double> dqr((size_t)D, 0.0);
            for (int j = 0; j <= i; ++j) {
                const double ds = P[j] * (dP[j] - dl);
                for (int d = 0; d < D; ++d) dqr[d] += s * ds * kr[(size_t)j * D + d];
            }
            rotate_row_transpose(dqr.data(), &dq[(size_t)r * D], i, D, theta);
        }
    }
    return 0;
}

/* Selected key rows of one (b, kv head g): dV_j = sum_h sum_{i >= j} P_ij dO_i and
 * dk_j = R_j^T s sum_h sum_{i >= j} dS_ij q'_i over the G query heads h of g, with P and
 * dS as above.  Every query row i >= min(rows) is needed, each for its LSE_i and Delta_i,
 * so rows near the end of the sequence are cheap.  Outputs dk, dv are [n, D]. */
int ne_ref_attn_krows(const double* q, const double* k, const double* v, const double* dO, int b, int g,
                      const int* rows, int n, double* dk, double* dv, int B, int T, int Hq, int Hkv,
                      int D, double theta) {
    if (bad_shape(B, T, Hq, Hkv, D) || b < 0 || b >= B || g < 0 || g >= Hkv) return 1;
    int jmin = T;
    for (int r = 0; r < n; ++r) {
        if (rows[r] < 0 || rows[r] >= T) return 1;
        if (rows[r] < jmin) jmin = rows[r];
    }
    if (n == 0) return 0;
    const int G = Hq / Hkv;
    const double s = 1.0 / std::sqrt((double)D);
    std::vector<double> kr;
    rotated_head(k, b, g, T, Hkv, D, theta, kr);
    std::vector<double> acck((size_t)n * D, 0.0), accv((size_t)n * D, 0.0);
    for (int h = g * G; h < (g + 1) * G; ++h) {
        // LSE_i and Delta_i of every query row that can see one of the requested keys.
        const int nq = T - jmin;
        std::vector<double> L((size_t)nq), Dl((size_t)nq), qr((size_t)nq * D);
#pragma omp parallel for schedule(dynamic)
        for (int ii = 0; ii < nq; ++ii) {
            const int i = jmin + ii;
            double* qi = &qr[(size_t)ii * D];
            rotate_row(&q[idx4(b, i, h, 0, T, Hq, D)], qi, i, D, theta);
            std::vector<double> S((size_t)i + 1);
            double m = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qi[d] * kr[(size_t)j * D + d];
                S[j] = s * dot;
                if (S[j] > m) m = S[j];
            }
            double sum = 0.0;
            for (int j = 0; j <= i; ++j) sum += std::exp(S[j] - m);
            const double l = m + std::log(sum);
            double dl = 0.0;
            for (int j = 0; j <= i; ++j) {
                double dp = 0.0;
                for (int d = 0; d < D; ++d) dp += dO[idx4(b, i, h, d, T, Hq, D)] * v[idx4(b, j, g, d, T, Hkv, D)];
                dl += std::exp(S[j] - l) * dp;
            }
            L[ii] = l;
            Dl[ii] = dl;
        }
#pragma omp parallel for schedule(dynamic)
        for (int r = 0; r < n; ++r) {
            const int j = rows[r];
            for (int i = j; i < T; ++i) {
                const int ii = i - jmin;
                const double* qi = &qr[(size_t)ii * D];
                double dot = 0.0, dp = 0.0;
                for (int d = 0; d < D; ++d) {
                    dot += qi[d] * kr[(size_t)j * D + d];
                    dp += dO[idx4(b, i, h, d, T, Hq, D)] * v[idx4(b, j, g, d, T, Hkv, D)];
                }
                const double p = std::exp(s * dot - L[ii]);
                const double ds = p * (dp - Dl[ii]);
                for (int d = 0; d < D; ++d) {
                    acck[(size_t)r * D + d] += s * ds * qi[d];
                    accv[(size_t)r * D + d] += p * dO[idx4(b, i, h, d, T, Hq, D)];
                }
            }
        }
    }
    for (int r = 0; r < n; ++r) {
        rotate_row_transpose(&acck[(size_t)r * D], &dk[(size_t)r * D], rows[r], D, theta);
        for (int d = 0; d < D; ++d) dv[(size_t)r * D + d] = accv[(size_t)r * D + d];
    }
    return 0;
}

/* The steps before attention in every layer ("NanoEuler: C와 CUDA로 밑바닥부터 구축한
 * GPT-2 규모의 LLM", 기술 사양: RMSNorm as pre-normalization without bias, RoPE on queries
 * and keys; the model uses no biases at all).  For token row m of x [B*T, dim]:
 *   r_m  = sqrt(mean_c x_mc^2 + eps)                     (RMSNorm, gain gamma [dim])
 *   xh_m = x_m / r_m * gamma
 *   y_m  = W xh_m,  W [(Hq + 2 Hkv) D, dim]              (one bias-free projection)
 * and y_m splits into q (rows 0 .. Hq D - 1 of W), k (next Hkv D) and v (last Hkv D),
 * each head D wide.  With rotate, q and k are rotated by R_t, t = m mod T (the RoPE of
 * the attention above); v never is.  Outputs q [B, T, Hq, D], k and v [B, T, Hkv, D]. */
int ne_ref_qkv_prologue(const double* x, const double* gamma, const double* w, double* q, double* k, double* v,
                        int B, int T, int dim, int Hq, int Hkv, int D, double eps, double theta, int rotate) {
    if (bad_shape(B, T, Hq, Hkv, D) || dim <= 0 || !(eps >= 0.0)) return 1;
    const int N = (Hq + 2 * Hkv) * D;
    const int64_t M = (int64_t)B * T;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const double* xm = x + m * dim;
        double ss = 0.0;
        for (int c = 0; c < dim; ++c) ss += xm[c] * xm[c];
        const double r = std::sqrt(ss / (double)dim + eps);
        std::vector<double> xh((size_t)dim), y((size_t)N), yr((size_t)D);
        for (int c = 0; c < dim; ++c) xh[c] = xm[c] / r * gamma[c];
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int c = 0; c < dim; ++c) acc += w[(int64_t)n * dim + c] * xh[c];
            y[n] = acc;
        }
        const int t = (int)(m % T);
        for (int h = 0; h < Hq + 2 * Hkv; ++h) {
            const double* yh = &y[(size_t)h * D];
            const bool rot = rotate && h < Hq + Hkv;
            if (rot) rotate_row(yh, yr.data(), t, D, theta);
            const double* src = rot ? yr.data() : yh;
            double* dst = h < Hq ? q + (m * Hq + h) * D
                                 : (h < Hq + Hkv ? k + (m * Hkv + (h - Hq)) * D : v + (m * Hkv + (h - Hq - Hkv)) * D);
            for (int d = 0; d < D; ++d) dst[d] = src[d];
        }
    }
    return 0;
}

int ne_ref_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

}  /* extern "C" */
