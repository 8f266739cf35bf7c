/*
 * CPU FP64 oracle for exact scaled-dot-product attention forward, its chunk-pair partials and the
 * exact LSE merge of partials. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the library's product path never does. It shares no code
 * with the CUDA path.
 *
 * What it computes (the plain definition; the pages never print the formula, so this follows
 * their statement of the problem):
 *   - "stream-cqsa 2.2.0 -> 2.2.2" diff, stream_cqsa/api.py, `attention` docstring: the call is a
 *     drop-in for torch's F.scaled_dot_product_attention (SDPA), "exact";
 *   - "stream-cqsa 2.2.2 -> 2.2.3" diff, stream_cqsa/oom_fallback.py, `stream_cqsa_auto`: each
 *     call yields a per-row log-sum-exp ("lse") besides the output;
 *   - "stream-cqsa 2.2.0 -> 2.2.2" diff, README profile-sweep section: outputs of subproblems are
 *     merged into an accumulator.
 *
 * For query row i of head (b, h), with absolute positions q_off + i and kv_off + j:
 *   A_i   = { j : 0 <= j < Nkv and (not causal or kv_off + j <= q_off + i) }
 *   s_ij  = scale * sum_c q_ic k_jc                (double; fp16/bf16 inputs widened exactly)
 *   M_i   = max_{j in A_i} s_ij
 *   p_ij  = exp(s_ij - M_i),   l_i = sum_j p_ij   (Neumaier-compensated sums)
 *   O_ic  = (sum_j p_ij v_jc) / l_i
 *   LSE_i = M_i + log(l_i)                         (natural log, scale included)
 * A row with A_i empty (a chunk pair entirely above the causal diagonal, or Nkv = 0) has O = 0 and
 * LSE = -inf. The whole score row is materialised. `scale` arrives as the fp32 value the GPU uses,
 * widened to double, so both sides compute with the identical scale.
 *
 * Merge of n partials of the same rows over disjoint key sets (exact in exact arithmetic):
 *   M = max_k LSE_k,  lse = M + log(sum_k exp(LSE_k - M)),  O = sum_k exp(LSE_k - lse) O_k;
 * all-empty rows (M = -inf) give O = 0, lse = -inf.
 *
 * A second routine, written separately, evaluates tiny problems in long double without the max
 * subtraction (p_ij = exp(s_ij) directly), as a brute-force cross-check of the first.
 *
 * The backward (gradients of q, k, v from an upstream dO) is defined at `oracle_attn_bwd` below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* ---- exact widening of the storage types -------------------------------------------------- */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int fr = h & 0x3ff;
    double v;
    if (ex == 0) {
        v = ldexp((double)fr, -24);                 /* subnormal: fr * 2^-24 */
    } else if (ex == 31) {
        v = fr ? NAN : INFINITY;
    } else {
        v = ldexp((double)(fr | 0x400), ex - 25);   /* (1024 + fr) * 2^(ex - 15 - 10) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE 754 binary32. */
static double bfloat_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 7) & 0xff;
    int fr = h & 0x7f;
    double v;
    if (ex == 0) {
        v = ldexp((double)fr, -133);                /* subnormal: fr * 2^(-126 - 7) */
    } else if (ex == 255) {
        v = fr ? NAN : INFINITY;
    } else {
        v = ldexp((double)(fr | 0x80), ex - 134);   /* (128 + fr) * 2^(ex - 127 - 7) */
    }
    return sign ? -v : v;
}

static double widen(const uint16_t* base, int64_t idx, int dtype) {
    return dtype == 0 ? half_bits_to_double(base[idx]) : bfloat_bits_to_double(base[idx]);
}

/* element (b, h, n, c) of a tensor with `rows` tokens; layout 0 = [B,H,rows,d], 1 = [B,rows,H,d] */
static int64_t at(int layout, int64_t H, int64_t rows, int64_t d, int64_t b, int64_t h, int64_t n, int64_t c) {
    return layout == 0 ? ((b * H + h) * rows + n) * d + c : ((b * rows + n) * H + h) * d + c;
}

/* Neumaier's improvement of Kahan summation (A. Neumaier, ZAMM 54, 1974). */
typedef struct { double s, c; } nsum;
static void nsum_add(nsum* a, double x) {
    double t = a->s + x;
    if (fabs(a->s) >= fabs(x)) a->c += (a->s - t) + x;
    else a->c += (x - t) + a->s;
    a->s = t;
}
static double nsum_get(const nsum* a) { return a->s + a->c; }

/*
 * Attention rows of one chunk pair (the whole problem when q_off = kv_off = 0, Nq = Nkv = N).
 * q: [B,H,Nq,d] (or [B,Nq,H,d]), k, v: [B,H,Nkv,d] (or [B,Nkv,H,d]) storage bits of `dtype`
 * (0 fp16, 1 bf16). rows: nrows triples (b, h, i) with 0 <= i < Nq. out: nrows x d, lse: nrows.
 * Rows are evaluated head by head: the K and V of one (b, h) are widened to double once (an exact
 * conversion), then each row of that head is computed from its definition. Each product q_ic k_jc
 * of two 16-bit values is exact in double; the d-term dot product is summed plainly (error ~1e-14
 * relative to the sum of |terms|), the long sums over keys with compensation.
 * Returns 0, or -1 on a bad argument or allocation failure.
 */
int oracle_attn_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, int layout, int dtype,
                     int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t d, int64_t q_off,
                     int64_t kv_off, int causal, double scale, const int64_t* rows, int64_t nrows,
                     double* out, double* lse) {
    if (B < 1 || H < 1 || Nq < 0 || Nkv < 0 || d < 1 || (dtype != 0 && dtype != 1)) return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t* t = rows + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= H || t[2] < 0 || t[2] >= Nq) return -1;
    }
    int bad = 0;
    size_t kv_elems = (size_t)(Nkv > 0 ? Nkv : 1) * (size_t)d;
    double* kd = (double*)malloc(sizeof(double) * kv_elems);
    double* vd = (double*)malloc(sizeof(double) * kv_elems);
    if (!kd || !vd) {
        free(kd);
        free(vd);
        return -1;
    }
    for (int64_t b = 0; b < B && !bad; ++b) {
        for (int64_t h = 0; h < H && !bad; ++h) {
            int64_t cnt = 0;
            for (int64_t r = 0; r < nrows; ++r) cnt += (rows[3 * r] == b && rows[3 * r + 1] == h);
            if (cnt == 0) continue;
            /* exact widening of this head's keys and values */
#pragma omp parallel for schedule(static)
            for (int64_t j = 0; j < Nkv; ++j) {
                for (int64_t c = 0; c < d; ++c) {
                    kd[j * d + c] = widen(k, at(layout, H, Nkv, d, b, h, j, c), dtype);
                    vd[j * d + c] = widen(v, at(layout, H, Nkv, d, b, h, j, c), dtype);
                }
            }
#pragma omp parallel
            {
                double* s = (double*)malloc(sizeof(double) * (size_t)(Nkv > 0 ? Nkv : 1));
                double* qi = (double*)malloc(sizeof(double) * (size_t)d);
                nsum* acc = (nsum*)malloc(sizeof(nsum) * (size_t)d);
                if (!s || !qi || !acc) {
#pragma omp atomic write
                    bad = 1;
                }
#pragma omp for schedule(dynamic, 1)
                for (int64_t r = 0; r < nrows; ++r) {
                    if (bad || rows[3 * r] != b || rows[3 * r + 1] != h) continue;
                    int64_t i = rows[3 * r + 2];
                    double* o = out + r * d;
                    for (int64_t c = 0; c < d; ++c) qi[c] = widen(q, at(layout, H, Nq, d, b, h, i, c), dtype);
                    /* allowed keys are j < jend (causal: kv_off + j <= q_off + i) */
                    int64_t jend = Nkv;
                    if (causal) {
                        int64_t lim = q_off + i - kv_off + 1;
                        if (lim < jend) jend = lim;
                        if (jend < 0) jend = 0;
                    }
                    if (jend == 0) {
                        for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
                        lse[r] = -INFINITY;
                        continue;
                    }
                    double m = -INFINITY;
                    for (int64_t j = 0; j < jend; ++j) {
                        const double* kj = kd + j * d;
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += qi[c] * kj[c];
                        s[j] = scale * dot;
                        if (s[j] > m) m = s[j];
                    }
                    nsum l = {0.0, 0.0};
                    for (int64_t c = 0; c < d; ++c) acc[c] = (nsum){0.0, 0.0};
                    for (int64_t j = 0; j < jend; ++j) {
                        double p = exp(s[j] - m);
                        const double* vj = vd + j * d;
                        nsum_add(&l, p);
                        for (int64_t c = 0; c < d; ++c) nsum_add(&acc[c], p * vj[c]);
                    }
                    double lv = nsum_get(&l);
                    for (int64_t c = 0; c < d; ++c) o[c] = nsum_get(&acc[c]) / lv;
                    lse[r] = m + log(lv);
                }
                free(s);
                free(qi);
                free(acc);
            }
        }
    }
    free(kd);
    free(vd);
    return bad ? -1 : 0;
}

/*
 * Exact merge of n partials. O_parts[k]: rows x d, LSE_parts[k]: rows (double). out: rows x d,
 * lse: rows. Partials are combined in the order k = 0 .. n-1.
 */
int oracle_merge(const double* const* O_parts, const double* const* LSE_parts, int n, int64_t rows,
                 int64_t d, double* out, double* lse) {
    if (n < 1 || rows < 0 || d < 1) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int k = 0; k < n; ++k) if (LSE_parts[k][r] > m) m = LSE_parts[k][r];
        double* o = out + r * d;
        if (m == -INFINITY) {
            for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        nsum z = {0.0, 0.0};
        for (int k = 0; k < n; ++k) nsum_add(&z, exp(LSE_parts[k][r] - m));
        double L = m + log(nsum_get(&z));
        for (int64_t c = 0; c < d; ++c) {
            nsum a = {0.0, 0.0};
            for (int k = 0; k < n; ++k) {
                if (LSE_parts[k][r] == -INFINITY) continue;   /* an empty part has weight 0 */
                nsum_add(&a, exp(LSE_parts[k][r] - L) * O_parts[k][r * d + c]);
            }
            o[c] = nsum_get(&a);
        }
        lse[r] = L;
    }
    return 0;
}

/*
 * Brute force for tiny problems (scores must stay small: no max subtraction), in long double,
 * [B,H,N,d] layout, whole problem (no offsets). out: B*H*N*d, lse: B*H*N.
 */
int oracle_attn_bruteforce_ld(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                              int64_t B, int64_t H, int64_t N, int64_t d, int causal, double scale,
                              double* out, double* lse) {
    if (B < 1 || H < 1 || N < 1 || d < 1 || N > 4096) return -1;
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const int64_t base = bh * N * d;
        for (int64_t i = 0; i < N; ++i) {
            long double den = 0.0L;
            long double num[512];
            if (d > 512) return -1;
            for (int64_t c = 0; c < d; ++c) num[c] = 0.0L;
            for (int64_t j = 0; j < N; ++j) {
                if (causal && j > i) break;
                long double sc = 0.0L;
                for (int64_t c = 0; c < d; ++c)
                    sc += (long double)widen(q, base + i * d + c, dtype) * (long double)widen(k, base + j * d + c, dtype);
                long double e = expl((long double)scale * sc);
                den += e;
                for (int64_t c = 0; c < d; ++c) num[c] += e * (long double)widen(v, base + j * d + c, dtype);
            }
            for (int64_t c = 0; c < d; ++c) out[(bh * N + i) * d + c] = (double)(num[c] / den);
            lse[bh * N + i] = (double)logl(den);
        }
    }
    return 0;
}

/* exact widening exposed for the tests (storage bits -> double) */
void oracle_widen(const uint16_t* bits, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = widen(bits, i, dtype);
}

/*
 * Backward of the same attention: the gradients of a scalar loss with respect to q, k and v, given
 * its gradient dO with respect to the output. The pages name the call (`stream_cqsa_backward`,
 * "stream-cqsa 2.2.0 -> 2.2.2" diff, README list of explicit entry points) and say it consumes the
 * forward's per-row log-sum-exp ("2.2.2 -> 2.2.3" diff, stream_cqsa/oom_fallback.py,
 * `stream_cqsa_auto` docstring), but print no formula; this is the chain rule through
 * O_i = sum_j P_ij v_j and the row softmax P_i = softmax(s_i), s_ij = scale q_i . k_j:
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   dS_ij = P_ij (dP_ij - sum_m P_im dP_im)        (softmax Jacobian applied to dP_i)
 *   dQ_i  = scale sum_j dS_ij k_j,     dK_j = scale sum_i dS_ij q_i
 * with P_ij = 0 outside A_i (causal: j <= i). Inputs and outputs are doubles in [B,H,N,d] (the
 * Python wrapper widens 16-bit storage exactly); the forward's O and LSE come back as well. Per
 * head the whole P and dS matrices are materialised (N*N doubles each): rows in parallel, then the
 * key-side sums column by column. Returns 0, or -1 on a bad argument or allocation failure.
 */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout, int64_t B,
                    int64_t H, int64_t N, int64_t d, int causal, double scale, double* out, double* lse,
                    double* dq, double* dk, double* dv) {
    if (B < 1 || H < 1 || N < 1 || d < 1 || N > 8192) return -1;
    double* P = (double*)malloc(sizeof(double) * (size_t)N * (size_t)N);
    double* dS = (double*)malloc(sizeof(double) * (size_t)N * (size_t)N);
    if (!P || !dS) {
        free(P);
        free(dS);
        return -1;
    }
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const double* qh = q + bh * N * d;
        const double* kh = k + bh * N * d;
        const double* vh = v + bh * N * d;
        const double* gh = dout + bh * N * d;
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t i = 0; i < N; ++i) {
            const int64_t jend = causal ? i + 1 : N;
            double* Pi = P + i * N;
            double* dSi = dS + i * N;
            double m = -INFINITY;
            for (int64_t j = 0; j < jend; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += qh[i * d + c] * kh[j * d + c];
                Pi[j] = scale * dot;
                if (Pi[j] > m) m = Pi[j];
            }
            nsum l = {0.0, 0.0};
            for (int64_t j = 0; j < jend; ++j) {
                Pi[j] = exp(Pi[j] - m);
                nsum_add(&l, Pi[j]);
            }
            const double lv = nsum_get(&l);
            for (int64_t j = 0; j < jend; ++j) Pi[j] /= lv;
            for (int64_t j = jend; j < N; ++j) Pi[j] = 0.0;
            lse[bh * N + i] = m + log(lv);
            for (int64_t c = 0; c < d; ++c) {
                nsum a = {0.0, 0.0};
                for (int64_t j = 0; j < jend; ++j) nsum_add(&a, Pi[j] * vh[j * d + c]);
                out[(bh * N + i) * d + c] = nsum_get(&a);
            }
            /* dP_ij, then its P-weighted row mean, then dS_ij */
            nsum D = {0.0, 0.0};
            for (int64_t j = 0; j < jend; ++j) {
                double dp = 0.0;
                for (int64_t c = 0; c < d; ++c) dp += gh[i * d + c] * vh[j * d + c];
                dSi[j] = dp;
                nsum_add(&D, Pi[j] * dp);
            }
            const double Dv = nsum_get(&D);
            for (int64_t j = 0; j < jend; ++j) dSi[j] = Pi[j] * (dSi[j] - Dv);
            for (int64_t j = jend; j < N; ++j) dSi[j] = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                nsum a = {0.0, 0.0};
                for (int64_t j = 0; j < jend; ++j) nsum_add(&a, dSi[j] * kh[j * d + c]);
                dq[(bh * N + i) * d + c] = scale * nsum_get(&a);
            }
        }
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t j = 0; j < N; ++j) {
            const int64_t i0 = causal ? j : 0;
            for (int64_t c = 0; c < d; ++c) {
                nsum a = {0.0, 0.0}, g = {0.0, 0.0};
                for (int64_t i = i0; i < N; ++i) {
                    nsum_add(&a, P[i * N + j] * gh[i * d + c]);
                    nsum_add(&g, dS[i * N + j] * qh[i * d + c]);
                }
                dv[(bh * N + j) * d + c] = nsum_get(&a);
                dk[(bh * N + j) * d + c] = scale * nsum_get(&g);
            }
        }
    }
    free(P);
    free(dS);
    return 0;
}

/*
 * The same gradients, evaluated only at listed rows or columns, for problems too large for
 * oracle_attn_bwd (which holds a head's N x N matrices). Inputs are 16-bit storage bits in
 * [B,H,N,d] (0 fp16, 1 bf16), widened exactly; `scale` as in oracle_attn_rows. The definitions are
 * those above:
 *   dQ_i  = scale sum_{j in A_i} dS_ij k_j,  dS_ij = P_ij (dP_ij - D_i),  D_i = sum_j P_ij dP_ij
 *   dV_j  = sum_{i : j in A_i} P_ij dO_i,    dK_j = scale sum_{i : j in A_i} dS_ij q_i
 * with P_ij = exp(s_ij - LSE_i), LSE_i = log sum_{j in A_i} exp(s_ij) and dP_ij = dO_i . v_j.
 *
 * oracle_attn_bwd_rows: dq (nrows x d) of the listed (b, h, i); each row needs only its own scores.
 * oracle_attn_bwd_cols: dk, dv (ncols x d) of the listed (b, h, j); for every head holding a listed
 * column it first evaluates LSE_i and D_i of every row of that head from their definitions, then the
 * column sums over the rows that see the column.
 * Both return 0, or -1 on a bad argument or allocation failure.
 */

/* this head's k, v (and q, dout when wanted) widened exactly to double, [N, d] each */
static void widen_head(const uint16_t* src, int dtype, int64_t bh, int64_t N, int64_t d, double* dst) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t c = 0; c < d; ++c) dst[j * d + c] = widen(src, (bh * N + j) * d + c, dtype);
}

/* scores s_ij = scale q_i . k_j for j < jend, their max, and LSE_i = m + log sum exp(s_ij - m) */
static double row_scores(const double* qi, const double* kd, int64_t jend, int64_t d, double scale, double* s) {
    double m = -INFINITY;
    for (int64_t j = 0; j < jend; ++j) {
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += qi[c] * kd[j * d + c];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    nsum l = {0.0, 0.0};
    for (int64_t j = 0; j < jend; ++j) nsum_add(&l, exp(s[j] - m));
    return m + log(nsum_get(&l));
}

int oracle_attn_bwd_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout, int dtype,
                         int64_t B, int64_t H, int64_t N, int64_t d, int causal, double scale,
                         const int64_t* rows, int64_t nrows, double* dq) {
    if (B < 1 || H < 1 || N < 1 || d < 1 || (dtype != 0 && dtype != 1)) return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t* t = rows + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= H || t[2] < 0 || t[2] >= N) return -1;
    }
    double* kd = (double*)malloc(sizeof(double) * (size_t)N * (size_t)d);
    double* vd = (double*)malloc(sizeof(double) * (size_t)N * (size_t)d);
    int bad = (!kd || !vd);
    for (int64_t bh = 0; bh < B * H && !bad; ++bh) {
        int64_t cnt = 0;
        for (int64_t r = 0; r < nrows; ++r) cnt += (rows[3 * r] * H + rows[3 * r + 1] == bh);
        if (cnt == 0) continue;
        widen_head(k, dtype, bh, N, d, kd);
        widen_head(v, dtype, bh, N, d, vd);
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)N);
            double* dp = (double*)malloc(sizeof(double) * (size_t)N);
            double* qi = (double*)malloc(sizeof(double) * (size_t)d);
            double* gi = (double*)malloc(sizeof(double) * (size_t)d);
            if (!s || !dp || !qi || !gi) {
#pragma omp atomic write
                bad = 1;
            }
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < nrows; ++r) {
                if (bad || rows[3 * r] * H + rows[3 * r + 1] != bh) continue;
                const int64_t i = rows[3 * r + 2];
                const int64_t jend = causal ? i + 1 : N;
                for (int64_t c = 0; c < d; ++c) {
                    qi[c] = widen(q, (bh * N + i) * d + c, dtype);
                    gi[c] = widen(dout, (bh * N + i) * d + c, dtype);
                }
                const double lse = row_scores(qi, kd, jend, d, scale, s);
                nsum D = {0.0, 0.0};
                for (int64_t j = 0; j < jend; ++j) {
                    s[j] = exp(s[j] - lse); /* P_ij */
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += gi[c] * vd[j * d + c];
                    dp[j] = dot;
                    nsum_add(&D, s[j] * dot);
                }
                const double Dv = nsum_get(&D);
                for (int64_t c = 0; c < d; ++c) {
                    nsum a = {0.0, 0.0};
                    for (int64_t j = 0; j < jend; ++j) nsum_add(&a, s[j] * (dp[j] - Dv) * kd[j * d + c]);
                    dq[r * d + c] = scale * nsum_get(&a);
                }
            }
            free(s);
            free(dp);
            free(qi);
            free(gi);
        }
    }
    free(kd);
    free(vd);
    return bad ? -1 : 0;
}

int oracle_attn_bwd_cols(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout, int dtype,
                         int64_t B, int64_t H, int64_t N, int64_t d, int causal, double scale,
                         const int64_t* cols, int64_t ncols, double* dk, double* dv) {
    if (B < 1 || H < 1 || N < 1 || d < 1 || (dtype != 0 && dtype != 1)) return -1;
    for (int64_t r = 0; r < ncols; ++r) {
        const int64_t* t = cols + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= H || t[2] < 0 || t[2] >= N) return -1;
    }
    const size_t nd = (size_t)N * (size_t)d;
    double* qd = (double*)malloc(sizeof(double) * nd);
    double* kd = (double*)malloc(sizeof(double) * nd);
    double* vd = (double*)malloc(sizeof(double) * nd);
    double* gd = (double*)malloc(sizeof(double) * nd);
    double* lse = (double*)malloc(sizeof(double) * (size_t)N);
    double* Dr = (double*)malloc(sizeof(double) * (size_t)N);
    int bad = (!qd || !kd || !vd || !gd || !lse || !Dr);
    for (int64_t bh = 0; bh < B * H && !bad; ++bh) {
        int64_t cnt = 0, jmin = N;
        for (int64_t r = 0; r < ncols; ++r)
            if (cols[3 * r] * H + cols[3 * r + 1] == bh) {
                ++cnt;
                if (cols[3 * r + 2] < jmin) jmin = cols[3 * r + 2];
            }
        if (cnt == 0) continue;
        widen_head(q, dtype, bh, N, d, qd);
        widen_head(k, dtype, bh, N, d, kd);
        widen_head(v, dtype, bh, N, d, vd);
        widen_head(dout, dtype, bh, N, d, gd);
        /* LSE_i and D_i of every row that sees a listed column (causal: i >= the smallest listed j) */
        const int64_t i0 = causal ? jmin : 0;
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)N);
            if (!s) {
#pragma omp atomic write
                bad = 1;
            }
#pragma omp for schedule(dynamic, 16)
            for (int64_t i = i0; i < N; ++i) {
                if (bad) continue;
                const int64_t jend = causal ? i + 1 : N;
                const double* qi = qd + i * d;
                const double* gi = gd + i * d;
                lse[i] = row_scores(qi, kd, jend, d, scale, s);
                nsum D = {0.0, 0.0};
                for (int64_t j = 0; j < jend; ++j) {
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += gi[c] * vd[j * d + c];
                    nsum_add(&D, exp(s[j] - lse[i]) * dot);
                }
                Dr[i] = nsum_get(&D);
            }
            free(s);
        }
        if (bad) break;
        /* the listed columns: sums over the rows i that see key j */
#pragma omp parallel
        {
            nsum* av = (nsum*)malloc(sizeof(nsum) * (size_t)d);
            nsum* ak = (nsum*)malloc(sizeof(nsum) * (size_t)d);
            if (!av || !ak) {
#pragma omp atomic write
                bad = 1;
            }
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < ncols; ++r) {
                if (bad || cols[3 * r] * H + cols[3 * r + 1] != bh) continue;
                const int64_t j = cols[3 * r + 2];
                const double* kj = kd + j * d;
                const double* vj = vd + j * d;
                for (int64_t c = 0; c < d; ++c) {
                    av[c] = (nsum){0.0, 0.0};
                    ak[c] = (nsum){0.0, 0.0};
                }
                for (int64_t i = causal ? j : 0; i < N; ++i) {
                    const double* qi = qd + i * d;
                    const double* gi = gd + i * d;
                    double sd = 0.0, dp = 0.0;
                    for (int64_t c = 0; c < d; ++c) {
                        sd += qi[c] * kj[c];
                        dp += gi[c] * vj[c];
                    }
                    const double P = exp(scale * sd - lse[i]);
                    const double dS = P * (dp - Dr[i]);
                    for (int64_t c = 0; c < d; ++c) {
                        nsum_add(&av[c], P * gi[c]);
                        nsum_add(&ak[c], dS * qi[c]);
                    }
                }
                for (int64_t c = 0; c < d; ++c) {
                    dv[r * d + c] = nsum_get(&av[c]);
                    dk[r * d + c] = scale * nsum_get(&ak[c]);
                }
            }
            free(av);
            free(ak);
        }
    }
    free(qd);
    free(kd);
    free(vd);
    free(gd);
    free(lse);
    free(Dr);
    return bad ? -1 : 0;
}
