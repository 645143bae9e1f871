/*
 * dust_oracle.c -- plain, slow fp64 CPU oracle of the Dust virtual-population
 * gradient estimator.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load this library.  The CUDA library never
 * calls it, and the two share no source, header, table or helper.
 *
 * What is computed, and where the pages define it:
 *   - Activation-space noise y_t + sigma*a_t, a_t ~ N(0, I), independent per
 *     token and per linear layer: laoyaoba.com "抛弃反向传播预训练大模型"
 *     section 机制拆解; hn.213312.xyz Dust translation §2 and §2.2;
 *     linlog.top article "Dust 的核心：虚拟种群".
 *   - Centred per-token loss decrease c_s, reward
 *     r_t = sum_{s>=t} gamma^(s-t) c_s (gamma = 0: own token only), error
 *     estimate g_t = -(1/(K sigma)) sum_i r_t^(i) a_t^(i), weight gradient
 *     G_W = sum_t g_t x_t^T, embedding one-hot outer product = scatter-add:
 *     hn.213312.xyz Dust translation §2.2 (信用分配).
 *   - LM head perturbed directly on cached logits, only the cross-entropy
 *     recomputed; interior layers re-run only the part after the perturbed
 *     layer: laoyaoba.com section 机制拆解; hn.213312.xyz §2.3.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - Noise: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
 *     numbers: as easy as 1, 2, 3", SC'11) with counter
 *     (channel/4, token, draw, layer) and key (seed low word, seed high word);
 *     uniform u(w) = ((w >> 9) + 0.5) * 2^-23; Box-Muller (Box & Muller 1958):
 *     rho = sqrt(-2 ln u(w0)), theta = 2 pi u(w1), channel 4j gets
 *     rho cos theta and 4j+1 gets rho sin theta; words w2, w3 give 4j+2, 4j+3.
 *   - Loss: natural-log cross-entropy over the full vocabulary, per token.
 *   - c = clean loss - perturbed loss, centred by its mean over the K draws of
 *     the same token (self included).
 *   - Credit never crosses a sequence boundary.
 *   - GELU(u) = u * Phi(u) with the exact error function.
 *   - Interior downstream: GELU -> W2 -> causal per-sequence EMA
 *     e_t = lam e_{t-1} + (1 - lam) u_t, e_{-1} = 0 -> W_head -> CE.
 *
 * Everything is double precision.  Inputs given as fp32 are widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 as defined in the SC'11 paper: two 32x32->64 multiplies per */
/* round, the high halves xored with the other two words and the round key, */
/* the key bumped by the Weyl constants after every round.                  */
/* ------------------------------------------------------------------------ */
static const uint32_t PHILOX_M4x32_0 = 0xD2511F53u;
static const uint32_t PHILOX_M4x32_1 = 0xCD9E8D57u;
static const uint32_t PHILOX_W32_0 = 0x9E3779B9u; /* golden ratio */
static const uint32_t PHILOX_W32_1 = 0xBB67AE85u; /* sqrt(3) - 1  */

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t prod0 = (uint64_t)PHILOX_M4x32_0 * (uint64_t)x0;
        uint64_t prod1 = (uint64_t)PHILOX_M4x32_1 * (uint64_t)x2;
        uint32_t n0 = (uint32_t)(prod1 >> 32) ^ x1 ^ k0;
        uint32_t n1 = (uint32_t)prod1;
        uint32_t n2 = (uint32_t)(prod0 >> 32) ^ x3 ^ k1;
        uint32_t n3 = (uint32_t)prod0;
        x0 = n0; x1 = n1; x2 = n2; x3 = n3;
        k0 += PHILOX_W32_0;
        k1 += PHILOX_W32_1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* n counters given as n x 4 words, one key: n x 4 output words. */
void orc_philox_batch(const uint32_t* ctrs, int64_t n, uint32_t key0, uint32_t key1,
                      uint32_t* out)
{
    const uint32_t key[2] = {key0, key1};
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) orc_philox4x32_10(ctrs + 4 * i, key, out + 4 * i);
}

double orc_uniform(uint32_t w) { return ((double)(w >> 9) + 0.5) * 0x1p-23; }

/* Raw words for one token: words[c] is word (c % 4) of block c / 4. */
static void token_words(uint64_t seed, uint32_t layer, uint32_t draw, uint32_t token,
                        int64_t nchan, uint32_t* words)
{
    const uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t blk[4];
    for (int64_t j = 0; 4 * j < nchan; ++j) {
        const uint32_t ctr[4] = {(uint32_t)j, token, draw, layer};
        orc_philox4x32_10(ctr, key, blk);
        for (int q = 0; q < 4 && 4 * j + q < nchan; ++q) words[4 * j + q] = blk[q];
    }
}

/* Standard normals a[c], c < nchan, for one (seed, layer, draw, token). */
static void token_normals(uint64_t seed, uint32_t layer, uint32_t draw, uint32_t token,
                          int64_t nchan, double* a)
{
    const uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t w[4];
    for (int64_t j = 0; 4 * j < nchan; ++j) {
        const uint32_t ctr[4] = {(uint32_t)j, token, draw, layer};
        orc_philox4x32_10(ctr, key, w);
        double vals[4];
        for (int pair = 0; pair < 2; ++pair) {
            double rho = sqrt(-2.0 * log(orc_uniform(w[2 * pair])));
            double theta = 2.0 * M_PI * orc_uniform(w[2 * pair + 1]);
            vals[2 * pair] = rho * cos(theta);
            vals[2 * pair + 1] = rho * sin(theta);
        }
        for (int q = 0; q < 4 && 4 * j + q < nchan; ++q) a[4 * j + q] = vals[q];
    }
}

/* words / normals for tokens token0 .. token0+ntok-1, row-major ntok x nchan */
void orc_noise_words(uint64_t seed, uint32_t layer, uint32_t draw, int64_t token0,
                     int64_t ntok, int64_t nchan, uint32_t* words)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < ntok; ++t)
        token_words(seed, layer, draw, (uint32_t)(token0 + t), nchan, words + t * nchan);
}

void orc_noise_normals(uint64_t seed, uint32_t layer, uint32_t draw, int64_t token0,
                       int64_t ntok, int64_t nchan, double* a)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < ntok; ++t)
        token_normals(seed, layer, draw, (uint32_t)(token0 + t), nchan, a + t * nchan);
}

/* ------------------------------------------------------------------------ */
/* Cross-entropy pieces                                                     */
/* ------------------------------------------------------------------------ */
static double logsumexp(const double* v, int64_t n)
{
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) if (v[i] > m) m = v[i];
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += exp(v[i] - m);
    return m + log(s);
}

/* Per-token CE of a logit row: lse(z) - z_y. */
static double token_ce(const double* zrow, int64_t V, int32_t y)
{
    return logsumexp(zrow, V) - zrow[y];
}

/*
 * LM head, perturbed on the cached logits (hn.213312.xyz §2.3; laoyaoba.com
 * 机制拆解): for draw i and token t,
 *     dl[i][t] = CE(z_t + sigma a_{i,t}) - CE(z_t),
 * the change of the per-token loss.  z is T x V row-major; dl is K x T.
 */
void orc_head_delta_loss(const double* z, const int32_t* y, int64_t T, int64_t V, double sigma,
                         uint64_t seed, uint32_t layer, uint32_t draw0, int64_t token0,
                         int64_t K, double* dl)
{
#pragma omp parallel
    {
        double* zc = (double*)malloc(sizeof(double) * V);
        double* a = (double*)malloc(sizeof(double) * V);
        double* zp = (double*)malloc(sizeof(double) * V);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t v = 0; v < V; ++v) zc[v] = z[t * V + v];
            const double ce_clean = token_ce(zc, V, y[t]);
            for (int64_t i = 0; i < K; ++i) {
                token_normals(seed, layer, draw0 + (uint32_t)i, (uint32_t)(token0 + t), V, a);
                for (int64_t v = 0; v < V; ++v) zp[v] = zc[v] + sigma * a[v];
                dl[i * T + t] = token_ce(zp, V, y[t]) - ce_clean;
            }
        }
        free(zc); free(a); free(zp);
    }
}

/* c[i][t] = -(dl[i][t] - mean_j dl[j][t]): the centred loss decrease. */
void orc_center(const double* dl, int64_t K, int64_t T, double* c)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double mean = 0.0;
        for (int64_t i = 0; i < K; ++i) mean += dl[i * T + t];
        mean /= (double)K;
        for (int64_t i = 0; i < K; ++i) c[i * T + t] = -(dl[i * T + t] - mean);
    }
}

/*
 * Reward, literal double sum: r[i][t] = sum_{s=t}^{end of t's sequence}
 * gamma^(s-t) c[i][s], with gamma^0 = 1 (so gamma = 0 keeps the own token).
 */
void orc_reward_literal(const double* c, int64_t K, int64_t T, int64_t seq_len, double gamma,
                        double* r)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < K; ++i) {
        for (int64_t t = 0; t < T; ++t) {
            const int64_t end = (t / seq_len + 1) * seq_len; /* exclusive */
            double acc = 0.0;
            for (int64_t s = t; s < end; ++s) acc += pow(gamma, (double)(s - t)) * c[i * T + s];
            r[i * T + t] = acc;
        }
    }
}

/* Same reward by the backward recurrence r_t = c_t + gamma r_{t+1}. */
void orc_reward_recurrence(const double* c, int64_t K, int64_t T, int64_t seq_len,
                           double gamma, double* r)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < K; ++i) {
        for (int64_t seq = 0; seq < T / seq_len; ++seq) {
            double acc = 0.0;
            for (int64_t t = (seq + 1) * seq_len - 1; t >= seq * seq_len; --t) {
                acc = c[i * T + t] + gamma * acc;
                r[i * T + t] = acc;
            }
        }
    }
}

/*
 * Error estimate g[t][c] = -(1/(K sigma)) sum_i r[i][t] a_{i,t}[c], the noise
 * regenerated from its counters.  r is K x T, g is T x C.
 */
void orc_ghat(const double* r, int64_t K, int64_t T, int64_t C, double sigma, uint64_t seed,
              uint32_t layer, uint32_t draw0, int64_t token0, double* g)
{
#pragma omp parallel
    {
        double* a = (double*)malloc(sizeof(double) * C);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            double* gt = g + t * C;
            for (int64_t c = 0; c < C; ++c) gt[c] = 0.0;
            for (int64_t i = 0; i < K; ++i) {
                token_normals(seed, layer, draw0 + (uint32_t)i, (uint32_t)(token0 + t), C, a);
                const double ri = r[i * T + t];
                for (int64_t c = 0; c < C; ++c) gt[c] += ri * a[c];
            }
            const double scale = -1.0 / ((double)K * sigma);
            for (int64_t c = 0; c < C; ++c) gt[c] *= scale;
        }
        free(a);
    }
}

/* Weight gradient G[c][k] = sum_t g[t][c] x[t][k]  (g: T x C, x: T x d). */
void orc_outer(const double* g, const double* x, int64_t T, int64_t C, int64_t d, double* G)
{
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t k = 0; k < d; ++k) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t) acc += g[t * C + c] * x[t * d + k];
            G[c * d + k] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Embedding: with one-hot inputs the outer product is a scatter-add.        */
/* ------------------------------------------------------------------------ */
typedef struct { int32_t id; int64_t t; } id_pos;

static int cmp_id_pos(const void* pa, const void* pb)
{
    const id_pos* a = (const id_pos*)pa;
    const id_pos* b = (const id_pos*)pb;
    if (a->id != b->id) return a->id < b->id ? -1 : 1;
    return a->t < b->t ? -1 : (a->t > b->t ? 1 : 0);
}

/*
 * perm: tokens ordered by (id, t); G_E[v] = sum over tokens with id v, in
 * ascending t, of g[t]; rows no token hits are zero.  g: T x d, G_E: V x d.
 */
void orc_embed_scatter(const double* g, const int32_t* ids, int64_t T, int64_t d, int64_t V,
                       int64_t* perm, double* G_E)
{
    id_pos* keys = (id_pos*)malloc(sizeof(id_pos) * (T > 0 ? T : 1));
    for (int64_t t = 0; t < T; ++t) { keys[t].id = ids[t]; keys[t].t = t; }
    qsort(keys, (size_t)T, sizeof(id_pos), cmp_id_pos);
    for (int64_t n = 0; n < T; ++n) perm[n] = keys[n].t;
    memset(G_E, 0, sizeof(double) * (size_t)(V * d));
    for (int64_t n = 0; n < T; ++n) {
        const int64_t t = keys[n].t;
        double* row = G_E + (int64_t)keys[n].id * d;
        for (int64_t k = 0; k < d; ++k) row[k] += g[t * d + k];
    }
    free(keys);
}

/* ------------------------------------------------------------------------ */
/* Interior linear layer: only the part after the perturbed layer re-runs.   */
/* ------------------------------------------------------------------------ */
static double gelu(double u) { return 0.5 * u * (1.0 + erf(u / sqrt(2.0))); }

void orc_gelu(const double* u, int64_t n, double* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = gelu(u[i]);
}

/* dh[t][c] = GELU(y1[t][c] + sigma a_{draw,t}[c]) - GELU(y1[t][c]), T x C. */
void orc_interior_dh(const float* y1, int64_t T, int64_t C, double sigma, uint64_t seed,
                     uint32_t layer, uint32_t draw, int64_t token0, double* dh)
{
#pragma omp parallel
    {
        double* a = (double*)malloc(sizeof(double) * C);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            token_normals(seed, layer, draw, (uint32_t)(token0 + t), C, a);
            for (int64_t c = 0; c < C; ++c) {
                const double y = (double)y1[t * C + c];
                dh[t * C + c] = gelu(y + sigma * a[c]) - gelu(y);
            }
        }
        free(a);
    }
}

/* Causal EMA per sequence: e_t = lam e_{t-1} + (1 - lam) u_t, e = 0 before
 * each sequence start.  u, e: T x n. */
void orc_ema(const double* u, int64_t T, int64_t n, int64_t seq_len, double lam, double* e)
{
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < n; ++k) {
        double prev = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            if (t % seq_len == 0) prev = 0.0;
            prev = lam * prev + (1.0 - lam) * u[t * n + k];
            e[t * n + k] = prev;
        }
    }
}

/* dl[t] = CE(z_t + dz_t) - CE(z_t) for cached clean logits z and the
 * downstream logit change dz; T x V row-major. */
void orc_ce_delta(const double* z, const double* dz, const int32_t* y, int64_t T, int64_t V,
                  double* dl)
{
#pragma omp parallel
    {
        double* zc = (double*)malloc(sizeof(double) * V);
        double* zp = (double*)malloc(sizeof(double) * V);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t v = 0; v < V; ++v) {
                zc[v] = z[t * V + v];
                zp[v] = zc[v] + dz[t * V + v];
            }
            dl[t] = token_ce(zp, V, y[t]) - token_ce(zc, V, y[t]);
        }
        free(zc); free(zp);
    }
}
