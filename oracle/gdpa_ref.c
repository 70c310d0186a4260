/*
 * GDPA float64 reference loops.  TEST INFRASTRUCTURE ONLY: the parity tests,
 * the smoke check and the CPU-baseline leg of the benchmark call this; the
 * library never does.
 *
 * Generalized Dot-Product Attention, as described on "범용 내적 어텐션(GDPA):
 * 실제 추천 시스템 학습 부하를 위한 커널 최적화" (aitrends.kr), section
 * "핵심 요약" and the first paragraph of "섹션별 상세": attention whose softmax
 * is replaced by an element-wise activation (GELU, SiLU, ...).  Per sample b
 * of a jagged batch and per head h:
 *
 *     O_b = act(alpha * Q_b K_b^T) V_b
 *
 * with no row normalisation (the page's design notes drop the softmax
 * correction step entirely), summing only over valid (query, key) pairs.
 * The Taylor activation is the 6th-order polynomial printed under the SFU
 * paragraph of the same page.
 *
 * Readings where the page is silent:
 *   - alpha multiplies the score inside the activation: act(alpha * q.k).
 *   - A masked pair contributes exactly zero (it is skipped), rather than
 *     act(-inf) (the Taylor polynomial is +inf there).
 *   - Causal window W: key j is valid for query i iff i - W < j <= i
 *     (positions counted from the start of each sample).
 *   - Rows with no valid key give zero output and zero dQ.
 *
 * The softmax variant (kind 5) is the other attention kernel the GEM page
 * ("GEM 트레이닝: Meta가 LLM 규모의 광고 파운데이션 모델 효율성을 두 배로
 * 높인 방법", techlist.io; section "GPU 연산 효율을 높인 맞춤형 커널과
 * 정밀도", the kernel list) names next to GDPA:
 * Jagged Flash Attention, softmax attention over the same jagged batches.
 * Per query row, over its valid keys only: O_i = sum_j w_j V_j with
 * w_j = exp(s_j - m) / sum_l exp(s_l - m), s_j = alpha q_i.k_j, m = max_j s_j
 * (the standard softmax, evaluated with the max subtracted); a row with no
 * valid key gives zero.  Its row statistic lse_i = log sum_j exp(s_j) (-inf
 * without a valid key) and its gradients, with P_ij the softmax weights,
 * dP_ij = dO_i.V_j and D_i = sum_j P_ij dP_ij = dO_i.O_i:
 *     dV_j += P_ij dO_i,  dS_ij = P_ij (dP_ij - D_i),
 *     dQ_i += alpha dS_ij K_j,  dK_j += alpha dS_ij Q_i.
 *
 * Layout: token-major with heads interleaved, X[t][h][c], t a global token
 * index, q_off / kv_off exclusive prefix sums of the per-sample lengths.
 * Everything is double; inputs are the (possibly bf16-rounded) values upcast.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { REF_GELU_ERF = 0, REF_GELU_TANH = 1, REF_SILU = 2, REF_TAYLOR6 = 3, REF_IDENTITY = 4,
       REF_SOFTMAX = 5 };
enum { REF_MASK_NONE = 0, REF_MASK_CAUSAL_WINDOW = 1 };

static const double REF_PI = 3.14159265358979323846;

/* act(x); the GELU forms are x * Phi(x) (erf) and the usual tanh fit of it */
static double ref_act(int kind, double x) {
    switch (kind) {
    case REF_GELU_ERF:
        return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
    case REF_GELU_TANH: {
        double u = sqrt(2.0 / REF_PI) * (x + 0.044715 * x * x * x);
        return 0.5 * x * (1.0 + tanh(u));
    }
    case REF_SILU:
        return x / (1.0 + exp(-x));
    case REF_TAYLOR6: {
        /* 1/2 x + x^2/sqrt(2 pi) - x^4/(6 sqrt(2 pi)) + x^6/(40 sqrt(2 pi)) */
        double c2 = 1.0 / sqrt(2.0 * REF_PI);
        double x2 = x * x;
        return 0.5 * x + c2 * x2 - (c2 / 6.0) * x2 * x2 + (c2 / 40.0) * x2 * x2 * x2;
    }
    default:
        return x;
    }
}

/* d act / dx */
static double ref_dact(int kind, double x) {
    switch (kind) {
    case REF_GELU_ERF: {
        double cdf = 0.5 * (1.0 + erf(x / sqrt(2.0)));
        double pdf = exp(-0.5 * x * x) / sqrt(2.0 * REF_PI);
        return cdf + x * pdf;
    }
    case REF_GELU_TANH: {
        double k = sqrt(2.0 / REF_PI);
        double u = k * (x + 0.044715 * x * x * x);
        double t = tanh(u);
        double du = k * (1.0 + 3.0 * 0.044715 * x * x);
        return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * du;
    }
    case REF_SILU: {
        double s = 1.0 / (1.0 + exp(-x));
        return s * (1.0 + x * (1.0 - s));
    }
    case REF_TAYLOR6: {
        double c2 = 1.0 / sqrt(2.0 * REF_PI);
        double x2 = x * x;
        return 0.5 + 2.0 * c2 * x - 4.0 * (c2 / 6.0) * x2 * x + 6.0 * (c2 / 40.0) * x2 * x2 * x;
    }
    default:
        return 1.0;
    }
}

static int ref_valid(int i, int j, int mask, int window) {
    if (mask == REF_MASK_CAUSAL_WINDOW)
        return j <= i && j > i - window;
    return 1;
}

double gdpa_ref_act(int kind, double x) { return ref_act(kind, x); }
double gdpa_ref_dact(int kind, double x) { return ref_dact(kind, x); }

int gdpa_ref_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Number of valid (query, key) pairs summed over samples (per head). */
int64_t gdpa_ref_pairs(int B, const int32_t* q_off, const int32_t* kv_off, int mask, int window) {
    int64_t n = 0;
    for (int b = 0; b < B; ++b) {
        int lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
        for (int i = 0; i < lq; ++i)
            for (int j = 0; j < lkv; ++j)
                n += ref_valid(i, j, mask, window);
    }
    return n;
}

/* Softmax row (kind 5): O_i over the valid keys of row i of sample b, head h */
static void ref_softmax_row(const double* q, const double* K, const double* V, double* o, int i,
                            int lkv, int64_t row, int d, double alpha, int mask, int window) {
    double m = -INFINITY;
    for (int j = 0; j < lkv; ++j) {
        if (!ref_valid(i, j, mask, window)) continue;
        const double* k = K + (int64_t)j * row;
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += q[c] * k[c];
        if (alpha * s > m) m = alpha * s;
    }
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (m == -INFINITY) return;   /* no valid key */
    double z = 0.0;
    for (int j = 0; j < lkv; ++j) {
        if (!ref_valid(i, j, mask, window)) continue;
        const double* k = K + (int64_t)j * row;
        const double* v = V + (int64_t)j * row;
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += q[c] * k[c];
        const double w = exp(alpha * s - m);
        z += w;
        for (int c = 0; c < d; ++c) o[c] += w * v[c];
    }
    for (int c = 0; c < d; ++c) o[c] /= z;
}

/* lse[t][h] of the softmax variant */
void gdpa_ref_lse(int B, int H, int d, const int32_t* q_off, const int32_t* kv_off,
                  const double* Q, const double* K, double* lse, double alpha, int mask,
                  int window) {
    const int64_t row = (int64_t)H * d;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            int lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
            for (int i = 0; i < lq; ++i) {
                const double* q = Q + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                double m = -INFINITY, z = 0.0;
                for (int pass = 0; pass < 2; ++pass) {
                    for (int j = 0; j < lkv; ++j) {
                        if (!ref_valid(i, j, mask, window)) continue;
                        const double* k = K + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                        double s = 0.0;
                        for (int c = 0; c < d; ++c) s += q[c] * k[c];
                        if (pass == 0) {
                            if (alpha * s > m) m = alpha * s;
                        } else {
                            z += exp(alpha * s - m);
                        }
                    }
                    if (m == -INFINITY) break;
                }
                lse[(int64_t)(q_off[b] + i) * H + h] = m == -INFINITY ? -INFINITY : m + log(z);
            }
        }
    }
}

/* Gradients of the softmax variant (see the header comment) */
void gdpa_ref_softmax_bwd(int B, int H, int d, const int32_t* q_off, const int32_t* kv_off,
                          const double* Q, const double* K, const double* V, const double* dO,
                          double* dQ, double* dK, double* dV, double alpha, int mask, int window) {
    const int64_t row = (int64_t)H * d;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            int lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
            for (int i = 0; i < lq; ++i) {
                double* dq = dQ + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                for (int c = 0; c < d; ++c) dq[c] = 0.0;
            }
            for (int j = 0; j < lkv; ++j) {
                double* dk = dK + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                double* dv = dV + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                for (int c = 0; c < d; ++c) { dk[c] = 0.0; dv[c] = 0.0; }
            }
            for (int i = 0; i < lq; ++i) {
                const double* q = Q + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                const double* go = dO + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                double* dq = dQ + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                /* the row's weights P_ij and dP_ij, then D_i */
                double m = -INFINITY, z = 0.0, dsum = 0.0;
                for (int j = 0; j < lkv; ++j) {
                    if (!ref_valid(i, j, mask, window)) continue;
                    const double* k = K + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double s = 0.0;
                    for (int c = 0; c < d; ++c) s += q[c] * k[c];
                    if (alpha * s > m) m = alpha * s;
                }
                if (m == -INFINITY) continue;   /* no valid key: no gradient */
                for (int j = 0; j < lkv; ++j) {
                    if (!ref_valid(i, j, mask, window)) continue;
                    const double* k = K + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double s = 0.0;
                    for (int c = 0; c < d; ++c) s += q[c] * k[c];
                    z += exp(alpha * s - m);
                }
                for (int j = 0; j < lkv; ++j) {
                    if (!ref_valid(i, j, mask, window)) continue;
                    const double* k = K + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    const double* v = V + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double s = 0.0, dp = 0.0;
                    for (int c = 0; c < d; ++c) { s += q[c] * k[c]; dp += go[c] * v[c]; }
                    dsum += exp(alpha * s - m) / z * dp;
                }
                for (int j = 0; j < lkv; ++j) {
                    if (!ref_valid(i, j, mask, window)) continue;
                    const double* k = K + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    const double* v = V + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double* dk = dK + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double* dv = dV + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double s = 0.0, dp = 0.0;
                    for (int c = 0; c < d; ++c) { s += q[c] * k[c]; dp += go[c] * v[c]; }
                    const double p = exp(alpha * s - m) / z;
                    const double g = p * (dp - dsum);
                    for (int c = 0; c < d; ++c) {
                        dv[c] += p * go[c];
                        dq[c] += alpha * g * k[c];
                        dk[c] += alpha * g * q[c];
                    }
                }
            }
        }
    }
}

/* O[t][h][:] = sum over valid j of act(alpha * Q_t . K_j) V_j (kind 5: the
 * softmax-weighted sum instead) */
void gdpa_ref_fwd(int B, int H, int d, const int32_t* q_off, const int32_t* kv_off,
                  const double* Q, const double* K, const double* V, double* O,
                  double alpha, int act, int mask, int window) {
    const int64_t row = (int64_t)H * d;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            int lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
            for (int i = 0; i < lq; ++i) {
                const double* q = Q + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                double* o = O + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                if (act == REF_SOFTMAX) {
                    ref_softmax_row(q, K + (int64_t)kv_off[b] * row + (int64_t)h * d,
                                    V + (int64_t)kv_off[b] * row + (int64_t)h * d, o, i, lkv, row,
                                    d, alpha, mask, window);
                    continue;
                }
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                for (int j = 0; j < lkv; ++j) {
                    if (!ref_valid(i, j, mask, window)) continue;
                    const double* k = K + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    const double* v = V + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double s = 0.0;
                    for (int c = 0; c < d; ++c) s += q[c] * k[c];
                    double p = ref_act(act, alpha * s);
                    for (int c = 0; c < d; ++c) o[c] += p * v[c];
                }
            }
        }
    }
}

/*
 * Gradients of O with respect to Q, K, V given dO.  With x = alpha * q_i.k_j:
 *   dV_j += act(x) dO_i
 *   g     = (dO_i . V_j) act'(x)
 *   dQ_i += alpha g K_j,   dK_j += alpha g Q_i
 * Each (b, h) touches only its own rows, so the outer loop is race-free.
 */
void gdpa_ref_bwd(int B, int H, int d, const int32_t* q_off, const int32_t* kv_off,
                  const double* Q, const double* K, const double* V, const double* dO,
                  double* dQ, double* dK, double* dV,
                  double alpha, int act, int mask, int window) {
    const int64_t row = (int64_t)H * d;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            int lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
            for (int i = 0; i < lq; ++i) {
                double* dq = dQ + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                for (int c = 0; c < d; ++c) dq[c] = 0.0;
            }
            for (int j = 0; j < lkv; ++j) {
                double* dk = dK + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                double* dv = dV + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                for (int c = 0; c < d; ++c) { dk[c] = 0.0; dv[c] = 0.0; }
            }
            for (int i = 0; i < lq; ++i) {
                const double* q = Q + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                const double* go = dO + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                double* dq = dQ + (int64_t)(q_off[b] + i) * row + (int64_t)h * d;
                for (int j = 0; j < lkv; ++j) {
                    if (!ref_valid(i, j, mask, window)) continue;
                    const double* k = K + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    const double* v = V + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double* dk = dK + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double* dv = dV + (int64_t)(kv_off[b] + j) * row + (int64_t)h * d;
                    double s = 0.0, dp = 0.0;
                    for (int c = 0; c < d; ++c) { s += q[c] * k[c]; dp += go[c] * v[c]; }
                    double x = alpha * s;
                    double p = ref_act(act, x);
                    double g = dp * ref_dact(act, x);
                    for (int c = 0; c < d; ++c) {
                        dv[c] += p * go[c];
                        dq[c] += alpha * g * k[c];
                        dk[c] += alpha * g * q[c];
                    }
                }
            }
        }
    }
}
