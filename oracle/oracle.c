/*
 * oracle.c -- plain, slow CPU oracle of DSpark's serial Markov draft walk.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code with the CUDA library.
 *
 * What it computes (sources, by page title and section):
 *
 *  - The walk recurrence: "Keeping the Draft Walk on Chip: One Launch for
 *    DSpark's Markov Head", section "The serial part of a parallel drafter":
 *    prev = anchor; for each step k, u = W1[prev] (rank 256),
 *    logit_k = bf16(base_k + W2 @ u), tok_k = argmax (or a sample of
 *    softmax(logit_k / T)), prev = tok_k.
 *  - The rounding points: same page, same section (the default walk also
 *    rounds W2 @ u to bf16 before the add) and section "B200: the bf16 table
 *    fits on chip" (fp32 accumulation, bias rounded to bf16, then the sum
 *    rounded to bf16).  Here the projection is accumulated in fp64, which is
 *    the exact value up to fp64 rounding, and rounded to bf16 once.
 *  - Ties go to the smallest token id: same page, section "The idea: make
 *    the walk resident" (the inverted row index in the 64-bit key).
 *  - Sampling: per-row Gumbel-max with Philox noise keyed by seed, request,
 *    step and token (same section), computed in fp32 as the plain fp32
 *    Gumbel noise named by vLLM pull request #64442, section "Details".
 *    Tokens then follow softmax(logit / T).
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *  - bf16 rounding is IEEE round-to-nearest-even, from the exact value.
 *  - The base + bias sum is formed exactly (fp64) and rounded once.
 *  - Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) with key
 *    (lo32(seed), hi32(seed)) and counter (v >> 2, k, b, 0); token v uses
 *    output word v & 3.
 *  - The uniform is U = (2 * (x >> 9) + 1) * 2^-24, the midpoint of one of
 *    2^23 equal bins of (0,1); it is exact in fp32.
 *  - The Gumbel score is s = fp32(logit / T) + fp32(-log(fp32(-log U))),
 *    every operation rounded to fp32 (each fp64 result below is rounded to
 *    fp32 at the same points).  T == 0 selects greedy argmax of the bf16
 *    logits with no noise drawn; T < 0 or a non-finite T is an error.
 *
 * A second sampler (orc_walk2, sampler = 1) follows the large-batch scheme of
 * the same blog post, section "The idea: make the walk resident" (an inverse
 * CDF inside 8-row groups, Gumbel-max across the groups) with the in-group
 * step of vLLM pull request #64442, section "Details" (a uniform times the
 * group's mass, the first token whose running sum of fp32 weights passes it).
 * Readings: groups are the 8 consecutive tokens 8j .. 8j + 7 (the last group
 * stops at V); z_v = logit_v / T; m_j = the group's largest z; weights
 * w_v = exp(z_v - m_j) and mass S_j = their sum; group score
 * s_j = m_j + log(S_j) - log(-log U1_j); the group with the largest score
 * wins (ties: the smallest j) and its token is the first v whose running sum
 * of weights exceeds U2_j * S_j; the two uniforms of group j are the Philox
 * words 2 (j & 1) and 2 (j & 1) + 1 of counter (j >> 1, k, b, 1).  All of it
 * in fp64.  Tokens then follow softmax(logit / T) as well.
 *
 * Recurrent heads (orc_walk3, cell = 1 or 2) follow "Keeping the Draft Walk on
 * Chip", section "Beyond DSpark: other serial heads": the head keeps a small
 * state, updates it each step, and projects the new state through the same
 * W2 (the Markov head projects W1[prev]).  The pages name DSpark's gated and
 * RNN heads and where their 256 x 256 recurrent matrix M lives, but print no
 * cell equations.  Readings:
 *   h_{-1} = 0; x_k = W1[prev_k] (prev_0 = anchor); p_k = M @ h_{k-1} (fp64);
 *   gated: z = 1 / (1 + exp(-p_k)), h_k = bf16((1 - z) * h_{k-1} + z * x_k);
 *   RNN:   h_k = bf16(tanh(p_k + x_k));
 *   GRU (cell = 3; the page's GRU heads): three token tables X_r, X_z, X_n
 *   [V, r] stand for the input projections folded into per-token rows, and
 *   M stacks three recurrent matrices [3r, r]; with p_g = M_g @ h_{k-1},
 *   r = sig(X_r[prev] + p_r), z = sig(X_z[prev] + p_z),
 *   n = tanh(X_n[prev] + r * p_n), h_k = bf16((1 - z) * n + z * h_{k-1});
 *   the projected vector is u_k = h_k; each element's value is formed in fp64
 *   and rounded to bf16 once.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_EANCHOR (-5)
#define ORC_ETEMP (-7)

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 bits -> the exact value it denotes (bf16 is the top half of fp32). */
double orc_bf16_to_f64(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bf16, ties to even.  bf16 has 8 significant
 * bits and fp32's exponent range: normal numbers are n * 2^(e-8) with
 * 128 <= n < 256, subnormals are multiples of 2^-133.  The quantum q of x is
 * therefore 2^(e-8) where 2^(e-1) <= |x| < 2^e, but never below 2^-133.
 */
uint16_t orc_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);                 /* a = m * 2^e, 0.5 <= m < 1 */
    int qexp = e - 8;
    if (qexp < -133)
        qexp = -133;
    double scaled = ldexp(a, -qexp);    /* exact: a power-of-two scaling */
    double n = floor(scaled);
    double frac = scaled - n;           /* exact */
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0))
        n += 1.0;
    double r = ldexp(n, qexp);          /* n <= 256: at most 9 bits, exact */
    if (r >= 0x1p128)                   /* beyond the largest finite bf16 */
        return sign | 0x7F80;
    float f = (float)r;                 /* exact: 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return sign | (uint16_t)(bits >> 16);
}

/* -------------------------------------------------------------- Philox --- */

/*
 * Philox4x32 with 10 rounds.  One round: the products M0*c0 and M1*c2 are
 * split into high and low words; the new counter is
 * (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)).
 * Between rounds the key is bumped by the Weyl constants (W0, W1).
 */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += W0;
            k1 += W1;
        }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32 random bits that token v of request b at step k draws. */
uint32_t orc_noise_bits(uint64_t seed, int b, int k, int64_t v)
{
    uint32_t ctr[4] = {(uint32_t)(v >> 2), (uint32_t)k, (uint32_t)b, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return out[v & 3];
}

/* Bits -> uniform in (0,1): the midpoint of bin (x >> 9) of 2^23 bins. */
float orc_uniform(uint32_t x)
{
    return (float)ldexp(2.0 * (double)(x >> 9) + 1.0, -24);
}

/* Gumbel noise g = -log(-log U), each log's result rounded to fp32. */
float orc_gumbel(float U)
{
    float e = (float)(-log((double)U));
    return (float)(-log((double)e));
}

/* Selection score of one logit at temperature T > 0, in fp32 steps. */
float orc_sample_score(uint16_t logit, float T, float g)
{
    float q = (float)(orc_bf16_to_f64(logit) / (double)T); /* fp32 quotient */
    return (float)((double)q + (double)g);                 /* fp32 sum */
}


/* ------------------------------------------------------ group sampler --- */

/* The two uniforms of group j of request b at step k (see the header). */
void orc_group_uniforms(uint64_t seed, int b, int k, int64_t j, float *U1, float *U2)
{
    uint32_t ctr[4] = {(uint32_t)(j >> 1), (uint32_t)k, (uint32_t)b, 1u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    *U1 = orc_uniform(out[2 * (j & 1)]);
    *U2 = orc_uniform(out[2 * (j & 1) + 1]);
}

/*
 * Group inverse-CDF sampling of one row of bf16 logits at temperature T > 0.
 * Returns the token; per group j (ng = ceil(V / 8) groups) it stores the
 * group score, the in-group pick and the pick's margin: the distance of
 * U2_j * S_j to the nearest running-sum boundary, relative to S_j.
 */
int64_t orc_group_sample(const uint16_t *logit, int64_t V, float T, uint64_t seed, int b,
                         int k, float *gscore, int32_t *gpick, float *gmargin)
{
    const int64_t ng = (V + 7) / 8;
    int64_t best_j = 0;
    double best_s = -INFINITY;
    for (int64_t j = 0; j < ng; ++j) {
        const int64_t v0 = 8 * j;
        const int n = (int)(V - v0 < 8 ? V - v0 : 8);
        double z[8], w[8];
        double m = -INFINITY;
        for (int i = 0; i < n; ++i) {
            z[i] = orc_bf16_to_f64(logit[v0 + i]) / (double)T;
            if (z[i] > m)
                m = z[i];
        }
        double S = 0.0;
        for (int i = 0; i < n; ++i) {
            w[i] = exp(z[i] - m);
            S += w[i];
        }
        float U1, U2;
        orc_group_uniforms(seed, b, k, j, &U1, &U2);
        const double s = m + log(S) - log(-log((double)U1));
        const double target = (double)U2 * S;
        double run = 0.0, margin = INFINITY;
        int pick = n - 1;
        for (int i = 0; i < n; ++i) {
            run += w[i];
            const double d = fabs(run - target) / S;
            if (d < margin)
                margin = d;
            if (run > target) {
                pick = i;
                break;
            }
        }
        if (gscore)
            gscore[j] = (float)s;
        if (gpick)
            gpick[j] = (int32_t)(v0 + pick);
        if (gmargin)
            gmargin[j] = (float)margin;
        if (s > best_s) {
            best_s = s;
            best_j = j;
        }
    }
    /* the winner's pick, recomputed so that the return does not depend on gpick */
    const int64_t v0 = 8 * best_j;
    const int n = (int)(V - v0 < 8 ? V - v0 : 8);
    double z[8], w[8], m = -INFINITY, S = 0.0;
    for (int i = 0; i < n; ++i) {
        z[i] = orc_bf16_to_f64(logit[v0 + i]) / (double)T;
        if (z[i] > m)
            m = z[i];
    }
    for (int i = 0; i < n; ++i) {
        w[i] = exp(z[i] - m);
        S += w[i];
    }
    float U1, U2;
    orc_group_uniforms(seed, b, k, best_j, &U1, &U2);
    const double target = (double)U2 * S;
    double run = 0.0;
    for (int i = 0; i < n; ++i) {
        run += w[i];
        if (run > target)
            return v0 + i;
    }
    return v0 + n - 1;
}

/* ------------------------------------------------------ recurrent cells --- */

#define ORC_CELL_MARKOV 0
#define ORC_CELL_GATED 1
#define ORC_CELL_RNN 2
#define ORC_CELL_GRU 3

static double orc_sigmoid(double t) { return 1.0 / (1.0 + exp(-t)); }

/* fp64 dot product sum_j a[j * stride] b[j] of bf16 values, in j order */
static double orc_row_dot(const uint16_t *a, int64_t stride, const uint16_t *b, int r)
{
    double s = 0.0;
    for (int j = 0; j < r; ++j)
        s += orc_bf16_to_f64(a[j * stride]) * orc_bf16_to_f64(b[j]);
    return s;
}

/*
 * One state update of a recurrent head (see the header): from the previous
 * state hprev (bf16 bits, r; NULL means h = 0) and the token's input row x,
 * h[i] = bf16(value_i) with value_i formed in fp64 from p_i = M[i, :] . hprev.
 * Gated / RNN: M is bf16 bits [r, r] and x the token's W1 row (r).  GRU: M is
 * [3r, r] (the r-, z- and n-gate matrices) and x holds the token's rows of
 * the three tables one after another (3r).  exact (optional, r) receives
 * value_i.
 */
void orc_cell_update(int cell, const uint16_t *M, int r, const uint16_t *hprev,
                     const uint16_t *x, uint16_t *h, double *exact)
{
    for (int i = 0; i < r; ++i) {
        const double hp = hprev ? orc_bf16_to_f64(hprev[i]) : 0.0;
        const double xi = orc_bf16_to_f64(x[i]);
        double val;
        if (cell == ORC_CELL_GRU) {
            double pg[3] = {0.0, 0.0, 0.0};              /* M_g[i, :] . h_{k-1} */
            if (hprev)
                for (int g = 0; g < 3; ++g)
                    pg[g] = orc_row_dot(M + ((int64_t)g * r + i) * r, 1, hprev, r);
            const double rg = orc_sigmoid(xi + pg[0]);                       /* reset */
            const double zg = orc_sigmoid(orc_bf16_to_f64(x[r + i]) + pg[1]); /* update */
            const double ng = tanh(orc_bf16_to_f64(x[2 * r + i]) + rg * pg[2]);
            val = (1.0 - zg) * ng + zg * hp;
        } else {
            const double p = hprev ? orc_row_dot(M + (int64_t)i * r, 1, hprev, r) : 0.0;
            if (cell == ORC_CELL_GATED) {
                const double z = 1.0 / (1.0 + exp(-p)); /* update gate */
                val = (1.0 - z) * hp + z * xi;
            } else if (cell == ORC_CELL_RNN) {
                val = tanh(p + xi);
            } else {
                val = xi;                                /* Markov: u = W1[prev] */
            }
        }
        h[i] = orc_bf16_rne(val);
        if (exact)
            exact[i] = val;
    }
}

/* ---------------------------------------------------------------- walk --- */

/*
 * One walk per request (the Markov head, or a recurrent head's state walk).
 *
 *   W1, W2     bf16 bits, [V, r] row-major
 *   base       bf16 bits, [B, gamma, V]
 *   anchor     [B] int32, each in [0, V)
 *   T          [B] fp32 temperatures (0 = greedy)
 *   req0       request index of batch row 0: row i draws the noise of request
 *              req0 + i (so one request can be replayed on its own)
 *   forced     optional [B, gamma] int32: when given, step k > 0 uses
 *              prev = forced[b, k-1] instead of this walk's own token
 *              (teacher forcing; lets a test check each step of another
 *              walk on its own)
 *   out_tokens [B, gamma] int32
 *   out_logits optional [B, gamma, V] bf16 bits
 *   sampler    0: per-token Gumbel-max; 1: group inverse-CDF (see the header)
 *   out_scores optional [B, gamma, V] fp32 selection scores (the bf16 logit
 *              itself when T == 0, and for every token under sampler 1)
 *   out_gscore, out_gpick, out_gmargin  optional [B, gamma, ceil(V / 8)]:
 *              under sampler 1 with T > 0, each group's score, in-group pick
 *              and the pick's margin (see orc_group_sample)
 *   cell       0: Markov (u = W1[prev]); 1: gated; 2: RNN; 3: GRU (see the header)
 *   M          the recurrent matrix, bf16 bits [r, r] (cells 1 and 2), [3r, r] (GRU)
 *   X          the GRU's token tables, bf16 bits [3, V, r] (cell 3 only)
 *   forced_state  optional [B, gamma, r] bf16 bits: when given (with a
 *              cell), step k updates the state from forced_state[b, k-1]
 *              and projects forced_state[b, k] (teacher forcing of the
 *              state; out_state still receives this oracle's own update)
 *   out_state  optional [B, gamma, r] bf16 bits: each step's state h_k
 *   out_state_exact  optional [B, gamma, r] fp64: its value before rounding
 *   nthreads   OpenMP threads for the loop over tokens (<= 0: all)
 *
 * Returns 0, or a negative code (invalid sizes, sampler, cell, anchor or
 * temperature).
 */
int orc_walk3(const uint16_t *W1, const uint16_t *W2, int64_t V, int r,
              const uint16_t *base, const int32_t *anchor, const float *T,
              uint64_t seed, int B, int gamma, int req0, const int32_t *forced,
              int sampler, int cell, const uint16_t *M, const uint16_t *X,
              const uint16_t *forced_state,
              int32_t *out_tokens, uint16_t *out_logits, float *out_scores,
              float *out_gscore, int32_t *out_gpick, float *out_gmargin,
              uint16_t *out_state, double *out_state_exact, int nthreads)
{
    if (sampler != 0 && sampler != 1)
        return ORC_EINVAL;
    if (cell < ORC_CELL_MARKOV || cell > ORC_CELL_GRU)
        return ORC_EINVAL;
    if (cell != ORC_CELL_MARKOV && !M)
        return ORC_EINVAL;
    if (cell == ORC_CELL_GRU && !X)
        return ORC_EINVAL;
    if (V <= 0 || r <= 0 || B < 0 || gamma < 0 || req0 < 0)
        return ORC_EINVAL;
    for (int b = 0; b < B; ++b) {
        if (anchor[b] < 0 || anchor[b] >= V)
            return ORC_EANCHOR;
        if (!(T[b] >= 0.0f) || isinf(T[b]))
            return ORC_ETEMP;
    }
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif
    /* scratch rows, one vocabulary wide */
    uint16_t *logit = (uint16_t *)malloc((size_t)V * sizeof *logit);
    double *score = (double *)malloc((size_t)V * sizeof *score);
    uint16_t *hbuf = (uint16_t *)malloc(2 * (size_t)r * sizeof *hbuf);   /* h_{k-1}, h_k */
    double *hex = (double *)malloc((size_t)r * sizeof *hex);
    uint16_t *xin = (uint16_t *)malloc(3 * (size_t)r * sizeof *xin);      /* GRU rows */
    if (!logit || !score || !hbuf || !hex || !xin) {
        free(logit);
        free(score);
        free(hbuf);
        free(hex);
        free(xin);
        return ORC_EINVAL;
    }
    for (int b = 0; b < B; ++b) {
        int64_t prev = anchor[b];
        for (int k = 0; k < gamma; ++k) {
            if (forced && k > 0)
                prev = forced[(int64_t)b * gamma + (k - 1)];
            const uint16_t *u = W1 + prev * r;            /* u = W1[prev] */
            if (cell != ORC_CELL_MARKOV) {
                /* h_{k-1}: this walk's own, or the forced one; h_{-1} = 0 */
                const uint16_t *hprev = NULL;
                if (k > 0)
                    hprev = forced_state ? forced_state + ((int64_t)b * gamma + (k - 1)) * r
                                         : hbuf;
                uint16_t *hk = hbuf + r;
                const uint16_t *x = u;                     /* the token's input row(s) */
                if (cell == ORC_CELL_GRU) {
                    for (int g = 0; g < 3; ++g)
                        memcpy(xin + (size_t)g * r, X + ((int64_t)g * V + prev) * r,
                               (size_t)r * sizeof *xin);
                    x = xin;
                }
                orc_cell_update(cell, M, r, hprev, x, hk, hex);
                if (out_state)
                    memcpy(out_state + ((int64_t)b * gamma + k) * r, hk, (size_t)r * sizeof *hk);
                if (out_state_exact)
                    memcpy(out_state_exact + ((int64_t)b * gamma + k) * r, hex,
                           (size_t)r * sizeof *hex);
                memcpy(hbuf, hk, (size_t)r * sizeof *hk);  /* h_k becomes h_{k-1} */
                /* the projected state: h_k, or the forced walk's own h_k */
                u = forced_state ? forced_state + ((int64_t)b * gamma + k) * r : hbuf;
            }
            const uint16_t *bk = base + ((int64_t)b * gamma + k) * V;
            const float Tb = T[b];
#pragma omp parallel for num_threads(nthreads) schedule(static)
            for (int64_t v = 0; v < V; ++v) {
                const uint16_t *w = W2 + v * r;
                double acc = 0.0;                          /* W2[v,:] . u */
                for (int j = 0; j < r; ++j)
                    acc += orc_bf16_to_f64(w[j]) * orc_bf16_to_f64(u[j]);
                uint16_t bias = orc_bf16_rne(acc);         /* first rounding */
                uint16_t lg = orc_bf16_rne(orc_bf16_to_f64(bk[v]) +
                                           orc_bf16_to_f64(bias)); /* second */
                logit[v] = lg;
                if (Tb == 0.0f || sampler == 1) {
                    score[v] = orc_bf16_to_f64(lg);
                } else {
                    float U = orc_uniform(orc_noise_bits(seed, req0 + b, k, v));
                    score[v] = (double)orc_sample_score(lg, Tb, orc_gumbel(U));
                }
            }
            int64_t best = 0;                              /* ties: lowest v */
            if (sampler == 1 && Tb > 0.0f) {
                const int64_t ng = (V + 7) / 8;
                const int64_t go = ((int64_t)b * gamma + k) * ng;
                best = orc_group_sample(logit, V, Tb, seed, req0 + b, k,
                                        out_gscore ? out_gscore + go : NULL,
                                        out_gpick ? out_gpick + go : NULL,
                                        out_gmargin ? out_gmargin + go : NULL);
            } else {
                for (int64_t v = 1; v < V; ++v)
                    if (score[v] > score[best])
                        best = v;
            }
            out_tokens[(int64_t)b * gamma + k] = (int32_t)best;
            if (out_logits)
                memcpy(out_logits + ((int64_t)b * gamma + k) * V, logit,
                       (size_t)V * sizeof *logit);
            if (out_scores)
                for (int64_t v = 0; v < V; ++v)
                    out_scores[((int64_t)b * gamma + k) * V + v] = (float)score[v];
            prev = best;
        }
    }
    free(logit);
    free(score);
    free(hbuf);
    free(hex);
    free(xin);
    return ORC_OK;
}

/* The Markov walk with either sampler (the argument list before the cells). */
int orc_walk2(const uint16_t *W1, const uint16_t *W2, int64_t V, int r,
              const uint16_t *base, const int32_t *anchor, const float *T,
              uint64_t seed, int B, int gamma, int req0, const int32_t *forced,
              int sampler, int32_t *out_tokens, uint16_t *out_logits, float *out_scores,
              float *out_gscore, int32_t *out_gpick, float *out_gmargin, int nthreads)
{
    return orc_walk3(W1, W2, V, r, base, anchor, T, seed, B, gamma, req0, forced, sampler,
                     ORC_CELL_MARKOV, NULL, NULL, NULL, out_tokens, out_logits, out_scores,
                     out_gscore, out_gpick, out_gmargin, NULL, NULL, nthreads);
}

/* Batch helpers used by the tests to pin the pieces one by one. */
void orc_bf16_rne_many(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_rne(x[i]);
}

void orc_philox_many(const uint32_t *ctr, const uint32_t *key, uint32_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        orc_philox4x32_10(ctr + 4 * i, key + 2 * i, out + 4 * i);
}

/* The per-token Gumbel-max walk (sampler 0) with the original argument list. */
int orc_walk(const uint16_t *W1, const uint16_t *W2, int64_t V, int r,
             const uint16_t *base, const int32_t *anchor, const float *T,
             uint64_t seed, int B, int gamma, int req0, const int32_t *forced,
             int32_t *out_tokens, uint16_t *out_logits, float *out_scores,
             int nthreads)
{
    return orc_walk2(W1, W2, V, r, base, anchor, T, seed, B, gamma, req0, forced, 0,
                     out_tokens, out_logits, out_scores, NULL, NULL, NULL, nthreads);
}
