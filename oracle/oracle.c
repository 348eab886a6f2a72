/*
 * fp64 CPU oracle for exact attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or
 * calls this file: only tests/, the smoke check and the CPU-baseline leg of
 * the benchmark do. It shares no code with the CUDA library.
 *
 * What it computes is the plain definition of attention, not the tiled
 * algorithm: the method is exact, so its result is that of standard
 * attention ("FlashAttention" blog post, section "Standard Attention":
 * S = Q K^T, P = softmax(S) row-wise, O = P V; "FlashAttention: Fast and
 * Memory-Efficient Exact Attention with IO-Awareness", section "Masalah dan
 * Motivasi"). Each query row i is handled on its own: its score row S_i, its
 * probability row P_i and, for the backward, its dP_i row are materialised
 * in full (N entries, fp64), which is the definition restated one row at a
 * time so that N = 16K fits in memory. Matrix products that sum over rows
 * (dK, dV) are accumulated as the sum over i of the outer products, which is
 * the definition of that product.
 *
 * Readings of points the pages leave open (each also listed in the design
 * notes of the repository):
 *  - S is scaled: S = scale * Q K^T (the pages write Q K^T).
 *  - Masks set S_ij = -inf: causal (j > i), key padding (j >= kv_len[b]),
 *    block mask (M[i/block][j/block] == 0); they combine by AND.
 *  - Softmax is the safe softmax with m = row max ("FlashAttention" blog
 *    post, section "Tiling"); LSE_i = m_i + ln(sum_j exp(S_ij - m_i)).
 *  - Dropout (inverted): P^_ij = P_ij * Z_ij / (1 - p); LSE excludes it.
 *    Z_ij = 1 iff u >= T, T = min(floor(p * 2^32), 2^32 - 1), where u is word
 *    (j mod 4) of Philox4x32-10 with key (lo32(seed), hi32(seed)) and
 *    counter (floor(j/4), i, h, b).
 *  - A row with every key masked has O_i = 0, LSE_i = -inf and contributes
 *    no gradient.
 *  - Backward is closed form through the softmax Jacobian:
 *    dV = P^T dO, dP = (dO V^T) o Z/(1-p),
 *    dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik), dQ = scale dS K,
 *    dK = scale dS^T Q.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* Philox4x32-10, from Salmon, Moraes, Dror and Shaw, "Parallel Random     */
/* Numbers: As Easy as 1, 2, 3" (SC'11): a 4-word counter, a 2-word key,   */
/* ten rounds of two 32x32->64 multiplications, key bumped by the Weyl     */
/* constants between rounds.                                               */
/* ---------------------------------------------------------------------- */
#define PHILOX_MUL0 0xD2511F53u
#define PHILOX_MUL1 0xCD9E8D57u
#define PHILOX_WEYL0 0x9E3779B9u
#define PHILOX_WEYL1 0xBB67AE85u

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_WEYL0;
            k1 += PHILOX_WEYL1;
        }
        uint64_t prod0 = (uint64_t)PHILOX_MUL0 * (uint64_t)x0;
        uint64_t prod1 = (uint64_t)PHILOX_MUL1 * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Keep threshold for drop probability p: T = min(floor(p * 2^32), 2^32-1). */
static uint64_t keep_threshold(double p) {
    double t = floor(p * 4294967296.0);
    if (t < 0.0) t = 0.0;
    if (t > 4294967295.0) t = 4294967295.0;
    return (uint64_t)t;
}

uint64_t oracle_keep_threshold(double p) { return keep_threshold(p); }

/* Z_ij for one (b, h, i, j). */
static int keep_bit(uint64_t seed, uint64_t thr, int b, int h, int i, int j) {
    uint32_t ctr[4] = {(uint32_t)(j / 4), (uint32_t)i, (uint32_t)h, (uint32_t)b};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t r[4];
    oracle_philox4x32_10(ctr, key, r);
    return (uint64_t)r[j % 4] >= thr;
}

/* Full keep mask Z, uint8 [B,H,N,N]. */
void oracle_dropout_keep(uint8_t* keep, int B, int H, int N, double p, uint64_t seed) {
    uint64_t thr = keep_threshold(p);
    long total = (long)B * H * N;
#pragma omp parallel for schedule(static)
    for (long row = 0; row < total; ++row) {
        int i = (int)(row % N);
        int h = (int)((row / N) % H);
        int b = (int)(row / ((long)N * H));
        uint8_t* z = keep + row * (long)N;
        for (int j = 0; j < N; ++j) z[j] = (uint8_t)keep_bit(seed, thr, b, h, i, j);
    }
}

/* ---------------------------------------------------------------------- */
/* Problem description shared by the entry points below.                  */
/* ---------------------------------------------------------------------- */
typedef struct {
    int B, H, N, d;
    double scale;
    int causal;
    const uint8_t* block_mask; /* nb x nb or NULL */
    int block;                 /* block edge of block_mask */
    const int32_t* kv_len;     /* [B] or NULL */
    double dropout_p;
    uint64_t seed;
} problem;

static int masked(const problem* pr, int b, int i, int j) {
    if (pr->causal && j > i) return 1;
    if (pr->kv_len && j >= pr->kv_len[b]) return 1;
    if (pr->block_mask) {
        int nb = (pr->N + pr->block - 1) / pr->block;
        if (!pr->block_mask[(long)(i / pr->block) * nb + (j / pr->block)]) return 1;
    }
    return 0;
}

/*
 * One query row of one head: fills s (scores, -inf where masked), p (softmax
 * probabilities, 0 where masked) and returns LSE_i (or -inf for a fully
 * masked row).
 */
static double softmax_row(const problem* pr, const double* Q, const double* K, int b, int i,
                          double* s, double* p) {
    const int N = pr->N, d = pr->d;
    const double* qi = Q + (long)i * d;
    double m = -INFINITY;
    for (int j = 0; j < N; ++j) {
        if (masked(pr, b, i, j)) { s[j] = -INFINITY; continue; }
        const double* kj = K + (long)j * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += qi[c] * kj[c];
        s[j] = pr->scale * acc;
        if (s[j] > m) m = s[j];
    }
    if (m == -INFINITY) {
        for (int j = 0; j < N; ++j) p[j] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (int j = 0; j < N; ++j) {
        p[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
        l += p[j];
    }
    for (int j = 0; j < N; ++j) p[j] /= l;
    return m + log(l);
}

/* Dropout multiplier Z_ij / (1 - p) for the row, written into zs. */
static void dropout_row(const problem* pr, uint64_t thr, int b, int h, int i, double* zs) {
    const int N = pr->N;
    if (pr->dropout_p <= 0.0) {
        for (int j = 0; j < N; ++j) zs[j] = 1.0;
        return;
    }
    const double inv = 1.0 / (1.0 - pr->dropout_p);
    for (int j = 0; j < N; ++j) zs[j] = keep_bit(pr->seed, thr, b, h, i, j) ? inv : 0.0;
}

static int nthreads_or_default(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

static int head_of(const int32_t* heads, int idx) { return heads ? heads[idx] : idx; }

/*
 * Forward: O [B,H,N,d], LSE [B,H,N]. If heads != NULL only the listed flat
 * head indices (b*H + h) are computed; other outputs are left untouched.
 */
int oracle_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
               int B, int H, int N, int d, double scale, int causal,
               const uint8_t* block_mask, int block, const int32_t* kv_len,
               double dropout_p, uint64_t seed, const int32_t* heads, int nheads, int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d <= 0) return -1;
    problem pr = {B, H, N, d, scale, causal, block_mask, block > 0 ? block : 128, kv_len, dropout_p, seed};
    const uint64_t thr = keep_threshold(dropout_p);
    const int nh = heads ? nheads : B * H;
    const long rows = (long)nh * N;
    const int nt = nthreads_or_default(nthreads);
#pragma omp parallel num_threads(nt)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * 3);
        double* p = s + N;
        double* zs = p + N;
#pragma omp for schedule(dynamic, 8)
        for (long r = 0; r < rows; ++r) {
            const int hh = head_of(heads, (int)(r / N));
            const int i = (int)(r % N);
            const int b = hh / H, h = hh % H;
            const long base = (long)hh * N * d;
            const double* Q = q + base;
            const double* K = k + base;
            const double* V = v + base;
            double* oi = o + base + (long)i * d;
            lse[(long)hh * N + i] = softmax_row(&pr, Q, K, b, i, s, p);
            dropout_row(&pr, thr, b, h, i, zs);
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            for (int j = 0; j < N; ++j) {
                if (p[j] == 0.0) continue;
                const double w = p[j] * zs[j];
                const double* vj = V + (long)j * d;
                for (int c = 0; c < d; ++c) oi[c] += w * vj[c];
            }
        }
        free(s);
    }
    return 0;
}

/*
 * Backward: dQ, dK, dV [B,H,N,d] from Q, K, V and dO, in closed form.
 * Recomputes P from its definition; does not use the forward's outputs.
 */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
               double* dq, double* dk, double* dv,
               int B, int H, int N, int d, double scale, int causal,
               const uint8_t* block_mask, int block, const int32_t* kv_len,
               double dropout_p, uint64_t seed, const int32_t* heads, int nheads, int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d <= 0) return -1;
    problem pr = {B, H, N, d, scale, causal, block_mask, block > 0 ? block : 128, kv_len, dropout_p, seed};
    const uint64_t thr = keep_threshold(dropout_p);
    const int nh = heads ? nheads : B * H;
    const int nt = nthreads_or_default(nthreads);
    const long nd = (long)N * d;
    double* priv = (double*)calloc((size_t)nt * 2 * (size_t)(nd > 0 ? nd : 1), sizeof(double));
    if (!priv) return -2;
    for (int hi = 0; hi < nh; ++hi) {
        const int hh = head_of(heads, hi);
        const int b = hh / H, h = hh % H;
        const long base = (long)hh * nd;
        const double* Q = q + base;
        const double* K = k + base;
        const double* V = v + base;
        const double* dO = dout + base;
        memset(priv, 0, sizeof(double) * (size_t)nt * 2 * (size_t)nd);
#pragma omp parallel num_threads(nt)
        {
            int tid = 0;
#ifdef _OPENMP
            tid = omp_get_thread_num();
#endif
            double* dK_t = priv + (long)tid * 2 * nd;
            double* dV_t = dK_t + nd;
            double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * 4);
            double* p = s + N;
            double* zs = p + N;
            double* dp = zs + N;
#pragma omp for schedule(dynamic, 4)
            for (int i = 0; i < N; ++i) {
                const double* qi = Q + (long)i * d;
                const double* doi = dO + (long)i * d;
                double* dqi = dq + base + (long)i * d;
                for (int c = 0; c < d; ++c) dqi[c] = 0.0;
                double lse_i = softmax_row(&pr, Q, K, b, i, s, p);
                if (lse_i == -INFINITY) continue;
                dropout_row(&pr, thr, b, h, i, zs);
                /* dP_i = (dO_i V^T) o Z/(1-p); D_i = sum_j P_ij dP_ij */
                double Di = 0.0;
                for (int j = 0; j < N; ++j) {
                    if (p[j] == 0.0) { dp[j] = 0.0; continue; }
                    const double* vj = V + (long)j * d;
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += doi[c] * vj[c];
                    dp[j] = acc * zs[j];
                    Di += p[j] * dp[j];
                }
                for (int j = 0; j < N; ++j) {
                    if (p[j] == 0.0) continue;
                    const double ds = p[j] * (dp[j] - Di);
                    const double w = p[j] * zs[j];
                    const double* kj = K + (long)j * d;
                    double* dkj = dK_t + (long)j * d;
                    double* dvj = dV_t + (long)j * d;
                    for (int c = 0; c < d; ++c) {
                        dqi[c] += scale * ds * kj[c];
                        dkj[c] += scale * ds * qi[c];
                        dvj[c] += w * doi[c];
                    }
                }
            }
            free(s);
        }
        double* dK = dk + base;
        double* dV = dv + base;
        for (long e = 0; e < nd; ++e) { dK[e] = 0.0; dV[e] = 0.0; }
        for (int t = 0; t < nt; ++t) {
            const double* dK_t = priv + (long)t * 2 * nd;
            const double* dV_t = dK_t + nd;
            for (long e = 0; e < nd; ++e) { dK[e] += dK_t[e]; dV[e] += dV_t[e]; }
        }
    }
    free(priv);
    return 0;
}

/* Probabilities P (pre-dropout, [N,N]) and scores S of one head, for tests. */
int oracle_probs(const double* q, const double* k, double* s_out, double* p_out,
                 int B, int H, int N, int d, double scale, int causal,
                 const uint8_t* block_mask, int block, const int32_t* kv_len, int head) {
    problem pr = {B, H, N, d, scale, causal, block_mask, block > 0 ? block : 128, kv_len, 0.0, 0};
    const int b = head / H;
    const long base = (long)head * N * d;
    for (int i = 0; i < N; ++i)
        softmax_row(&pr, q + base, k + base, b, i, s_out + (long)i * N, p_out + (long)i * N);
    return 0;
}

int oracle_max_threads(void) { return nthreads_or_default(0); }

/* ---------------------------------------------------------------------- */
/* 8-bit floating point inputs (the FP8 forward of the "Flash Attention"  */
/* guide, section "Flash Attention 3 / Presisi FP8 native"). The format is */
/* E4M3 of the OCP 8-bit floating point specification: 1 sign bit, 4       */
/* exponent bits with bias 7, 3 mantissa bits; exponent 0 holds the        */
/* subnormals m/8 * 2^-6; there are no infinities and S.1111.111 is NaN,   */
/* so the largest finite magnitude is 1.75 * 2^8 = 448. Each code decodes  */
/* exactly to a double, times the caller's per-head dequantisation factor. */
/* ---------------------------------------------------------------------- */
static double e4m3_decode(uint8_t x) {
    const int sign = x >> 7, e = (x >> 3) & 15, m = x & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);          /* (m / 8) * 2^(1 - 7) */
    else
        v = ldexp(8.0 + (double)m, e - 10); /* (1 + m / 8) * 2^(e - 7) */
    return sign ? -v : v;
}

/* out[r * row_len + c] = decode(in[...]) * descale[r / rows_per_scale]:
 * a [n_scales * rows_per_scale, row_len] array with one factor per block of
 * rows (per head for [B,H,N,d]). */
void oracle_e4m3_dequantize(const uint8_t* in, double* out, long n_scales, long rows_per_scale, long row_len,
                            const double* descale) {
    for (long s = 0; s < n_scales; ++s) {
        const long base = s * rows_per_scale * row_len;
        for (long e = 0; e < rows_per_scale * row_len; ++e)
            out[base + e] = e4m3_decode(in[base + e]) * descale[s];
    }
}
