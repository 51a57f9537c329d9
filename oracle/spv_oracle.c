/*
 * spv_oracle.c -- ORACLE for the speculative-sampling verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, double-precision CPU
 * restatement of what the verify step computes.  It exists so that the tests,
 * the smoke check and the benchmark's CPU-baseline leg can check the CUDA
 * library against something written independently of it.  It shares no code,
 * header, table or constant generator with the CUDA library, and nothing in
 * the library links, loads or calls it.
 *
 * Sources (web pages this follows; the section names are the pages' own):
 *   [SD]  "Speculative Decoding: How Draft-Model Parallelism Cuts LLM
 *         Inference Latency" -- sections "The four-phase loop" (steps 2-4),
 *         "The acceptance criterion and why it is exact", "The proof of
 *         exactness", "Acceptance rate equals 1 minus total variation
 *         distance" (Theorem 3.5).
 *   [SPD] "Speculative Pipeline Decoding: Higher-Accuracy Drafting with Hidden
 *         Latency via Pipeline Parallelism" -- the streaming-verification
 *         section (at T = 0 a draft token stands only if it is the target's
 *         most likely token; at T > 0 the usual rejection rule decides) and
 *         "Evaluation" (temperature T).
 *   [SSD] "Speculative Speculative Decoding" (review of arXiv 2603.03251) --
 *         Figure 2 / "Core Technical Barrier" (geometric fan-out
 *         F_k = F_0 * a_p^(k/(1+r)), top-ranked draft tokens excluding the
 *         token already sent for verification).
 *
 * Readings where the pages leave a step open:
 *   - Accept test: accept x_i iff p_i(x_i) > 0 and r_i * q_i(x_i) <= p_i(x_i),
 *     r_i in (0,1].  This is [SD] step 3 "r_i <= min(1, p/q)" without the
 *     division; p = 0 always rejects, q == p always accepts.
 *   - "Sample from" ([SD] step 4) is realised by an exponential race, which
 *     draws exactly from the stated distribution:
 *       * ids are grouped in blocks of SPVO_BLOCK ids and each block in
 *         sub-blocks of SPVO_SUB ids.  The block with the smallest
 *         E_beta / W_beta wins (W_beta = the block's probability mass,
 *         E_beta ~ Exp(1)); inside it the sub-block with the smallest
 *         E_s / W_s; inside that the id with the smallest E_x / P(x).
 *         P(x) = W_beta/Z * W_s/W_beta * P(x)/W_s.
 *       * The residual norm(max(0, p - q)) is drawn by rejection: draw x from
 *         p by the race above, accept it with probability max(0, 1 - q/p)
 *         (i.e. iff q(x) <= (1 - v) p(x)); accepted draws have density
 *         proportional to p * (1 - q/p)+ = (p - q)+.  After SPVO_MAX_TRIALS
 *         failed trials the residual is drawn directly by the same race over
 *         the residual masses, so the output stays exact.
 *     Every exponential comes from E = -ln U, U = ((w >> 8) + 1) * 2^-24,
 *     w one 32-bit word of Philox4x32-10 keyed by the sequence's 64-bit key,
 *     counter (n / 4, stream, trial, 0), word n % 4, where n is the block
 *     index, the sub-block's index within its block, or the id's offset
 *     within its sub-block.  The position of the draw is not in the counter
 *     (a sequence makes one draw), and given the winning block the sub-block
 *     and id variates are fresh, so every level stays exact.
 *   - Ties in a race, in an argmax and in the fan-out order go to the lower
 *     index; -0.0 ranks equal to +0.0.
 *   - NaN or +inf in any row read, a row without a finite entry (in the
 *     greedy case too), or a draft token outside [0, V) make the sequence a
 *     bad row (status 4).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SPVO_BLOCK 1024
#define SPVO_SUB 32
#define SPVO_MAX_TRIALS 64

/* Stream tags: the second counter word of every Philox draw. */
#define SPVO_STREAM_BLOCK 1u
#define SPVO_STREAM_SUB 2u
#define SPVO_STREAM_TOKEN 3u
#define SPVO_STREAM_ACCEPT 4u
#define SPVO_STREAM_FB_BLOCK 5u
#define SPVO_STREAM_FB_SUB 6u
#define SPVO_STREAM_FB_TOKEN 7u
#define SPVO_STREAM_FILTERED 8u

#define SPVO_OK 0
#define SPVO_BAD_ROW 4

/* ------------------------------------------------------------------------ */
/* Philox4x32-10, from its published definition (Salmon, Moraes, Dror, Shaw,
 * "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): ten rounds; each
 * multiplies counter words 0 and 2 by two 32-bit constants (64-bit products)
 * and mixes the halves with the other words and the key, which is bumped by
 * two Weyl constants between rounds. */
void spvo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Uniform in (0,1] for draw n of (stream, trial, position) of one sequence:
 * counter = (n / 4, stream, trial, position), key = (low, high 32 bits of the
 * sequence key), word n % 4, U = ((w >> 8) + 1) * 2^-24. */
double spvo_uniform(uint64_t seq_key, uint32_t stream, uint32_t trial, uint32_t pos, uint64_t n)
{
    uint32_t ctr[4] = { (uint32_t)(n >> 2), stream, trial, pos };
    uint32_t key[2] = { (uint32_t)seq_key, (uint32_t)(seq_key >> 32) };
    uint32_t out[4];
    spvo_philox4x32_10(ctr, key, out);
    uint32_t w = out[n & 3u];
    return (double)((w >> 8) + 1u) * ldexp(1.0, -24);
}

/* Test hook (tests only; NULL in every other use): when set, every uniform a
 * draw consumes comes from this function instead of Philox, with the same
 * arguments.  The tests use it to enumerate a draw's variates on a grid and
 * to build decisions whose margin is known in advance.  spvo_uniform itself
 * is never overridden. */
typedef double (*spvo_uniform_fn)(uint64_t seq_key, uint32_t stream, uint32_t trial, uint32_t pos, uint64_t n);
static spvo_uniform_fn uniform_override = NULL;
void spvo_set_uniform_override(spvo_uniform_fn fn) { uniform_override = fn; }

/* The uniform of draw n of (stream, trial) for a draw made at position pos.
 * The counter's fourth word is 0, not the position: a sequence makes exactly
 * one draw (the residual at its first rejection, or the bonus), so the
 * variates it uses are i.i.d. whatever the position, and they can be
 * generated before the position is known. */
static double draw_uniform(uint64_t seq_key, uint32_t stream, uint32_t trial, uint32_t pos, uint64_t n)
{
    if (uniform_override) return uniform_override(seq_key, stream, trial, pos, n);
    return spvo_uniform(seq_key, stream, trial, 0, n);
}

/* Exp(1) variate from the same draw: E = -ln U. */
static double expo(uint64_t seq_key, uint32_t stream, uint32_t trial, uint32_t pos, uint64_t n)
{
    return -log(draw_uniform(seq_key, stream, trial, pos, n));
}

/* ------------------------------------------------------------------------ */
/* Compensated (Neumaier) running sum. */
typedef struct { double s, c; } ksum;
static void ksum_add(ksum *k, double x)
{
    double t = k->s + x;
    if (fabs(k->s) >= fabs(x)) k->c += (k->s - t) + x;
    else k->c += (x - t) + k->s;
    k->s = t;
}
static double ksum_val(const ksum *k) { return k->s + k->c; }

/* Temperature softmax of one row, [SD] step 2 ("probability distributions
 * p_1 ... p_{gamma+1}") with [SPD] "Evaluation" temperature T > 0:
 * y = z / T, M = max y, S = sum exp(y - M), P(x) = exp(y_x - M) / S.
 * Returns 0, or SPVO_BAD_ROW if the row holds NaN or +inf or no finite entry. */
int spvo_softmax_stats(const float *z, int V, double T, double *M_out, double *S_out)
{
    double M = -INFINITY;
    for (int x = 0; x < V; ++x) {
        double zx = (double)z[x];
        if (isnan(zx) || (isinf(zx) && zx > 0)) return SPVO_BAD_ROW;
        double y = zx / T;
        if (y > M) M = y;
    }
    if (isinf(M)) return SPVO_BAD_ROW; /* every entry is -inf */
    ksum S = { 0, 0 };
    for (int x = 0; x < V; ++x) ksum_add(&S, exp((double)z[x] / T - M));
    *M_out = M;
    *S_out = ksum_val(&S);
    return SPVO_OK;
}

static double prob(const float *z, int x, double T, double M, double S)
{
    return exp((double)z[x] / T - M) / S;
}

/* Margin bookkeeping: the smallest decision margin seen for a sequence. */
static void note_margin(double *margin, double m)
{
    if (m < *margin) *margin = m;
}

/* Race winner among arrivals a[0..n): smallest arrival, ties to the lower
 * index.  Records ln(second) - ln(first) as the decision margin. */
static int race_winner(const double *a, int n, double *margin)
{
    int best = -1;
    double a1 = INFINITY, a2 = INFINITY;
    for (int i = 0; i < n; ++i) {
        if (a[i] < a1) { a2 = a1; a1 = a[i]; best = i; }
        else if (a[i] < a2) a2 = a[i];
    }
    double m;
    if (isinf(a2)) m = INFINITY;
    else if (a1 == 0.0) m = (a2 == 0.0) ? 0.0 : INFINITY;
    else m = log(a2) - log(a1);
    note_margin(margin, m);
    return best;
}

/* Draw one token from the distribution with (unnormalised) masses w[0..V)
 * by the three-level exponential race described in the header.  The three
 * stream tags name the block, sub-block and token races. */
static int race_sample(const double *w, int V, uint64_t key, uint32_t s_block, uint32_t s_sub, uint32_t s_tok,
                       uint32_t trial, uint32_t pos, double *margin)
{
    int nb = (V + SPVO_BLOCK - 1) / SPVO_BLOCK;
    double *arr = (double *)malloc(sizeof(double) * (size_t)(nb > SPVO_BLOCK ? nb : SPVO_BLOCK));
    /* level 1: blocks */
    for (int b = 0; b < nb; ++b) {
        int lo = b * SPVO_BLOCK, hi = lo + SPVO_BLOCK < V ? lo + SPVO_BLOCK : V;
        ksum W = { 0, 0 };
        for (int x = lo; x < hi; ++x) ksum_add(&W, w[x]);
        double Wb = ksum_val(&W);
        arr[b] = Wb > 0 ? expo(key, s_block, trial, pos, (uint64_t)b) / Wb : INFINITY;
    }
    int bw = race_winner(arr, nb, margin);
    int lo = bw * SPVO_BLOCK, hi = lo + SPVO_BLOCK < V ? lo + SPVO_BLOCK : V;
    /* level 2: sub-blocks of the winning block; variate n = j, the sub-block's
     * index within the block (given the block, i.i.d. whichever block won) */
    int ns = (hi - lo + SPVO_SUB - 1) / SPVO_SUB;
    for (int j = 0; j < ns; ++j) {
        int s0 = lo + j * SPVO_SUB, s1 = s0 + SPVO_SUB < hi ? s0 + SPVO_SUB : hi;
        ksum W = { 0, 0 };
        for (int x = s0; x < s1; ++x) ksum_add(&W, w[x]);
        double Ws = ksum_val(&W);
        arr[j] = Ws > 0 ? expo(key, s_sub, trial, pos, (uint64_t)j) / Ws : INFINITY;
    }
    int sw = race_winner(arr, ns, margin);
    int s0 = lo + sw * SPVO_SUB, s1 = s0 + SPVO_SUB < hi ? s0 + SPVO_SUB : hi;
    /* level 3: ids of the winning sub-block; variate n = the id's offset in it */
    for (int x = s0; x < s1; ++x)
        arr[x - s0] = w[x] > 0 ? expo(key, s_tok, trial, pos, (uint64_t)(x - s0)) / w[x] : INFINITY;
    int xw = s0 + race_winner(arr, s1 - s0, margin);
    free(arr);
    return xw;
}

/* ------------------------------------------------------------------------ */
/* Greedy verify (T = 0), [SPD] streaming verification: a draft token stands
 * only if it is the target's most likely token.  a_i = argmax z_i (lowest id on
 * ties), accept x_i iff x_i == a_i, stop at the first mismatch and emit a_k
 * there, or the bonus a_gamma when every draft matched. */
static int argmax_row(const float *z, int V, int *a)
{
    int best = -1;
    double bv = -INFINITY;
    for (int x = 0; x < V; ++x) {
        double v = (double)z[x];
        if (isnan(v) || (isinf(v) && v > 0)) return SPVO_BAD_ROW;
        if (best < 0 || v > bv) { best = x; bv = v; }
    }
    if (isinf(bv)) return SPVO_BAD_ROW; /* every entry is -inf */
    *a = best;
    return SPVO_OK;
}

int spvo_verify_greedy_seq(const float *tgt, const int32_t *tok, int gamma, int V,
                           int32_t *k_out, int32_t *tokens_out)
{
    for (int i = 0; i <= gamma; ++i) tokens_out[i] = -1;
    *k_out = -1;
    int a[64 + 1];
    for (int i = 0; i < gamma; ++i)
        if (tok[i] < 0 || tok[i] >= V) return SPVO_BAD_ROW;
    for (int i = 0; i <= gamma; ++i)
        if (argmax_row(tgt + (size_t)i * V, V, &a[i]) != SPVO_OK) return SPVO_BAD_ROW;
    int k = 0;
    while (k < gamma && tok[k] == a[k]) ++k;
    for (int i = 0; i < k; ++i) tokens_out[i] = tok[i];
    tokens_out[k] = a[k];
    *k_out = k;
    return SPVO_OK;
}

/* ------------------------------------------------------------------------ */
/* Chain verify for one sequence, T > 0.  [SD] "The four-phase loop":
 *   step 3: draft token x_i stands when its uniform r_i is at most the
 *           ratio p_i(x_i)/q_i(x_i) capped at 1; the chain ends at the first
 *           token that fails.
 *   step 4: with every token standing, one more token is drawn from
 *           p_{gamma+1}; after a failure at j the replacement is drawn from
 *           norm(max(0, p_j - q_j)).
 * Inputs : tgt [(gamma+1) * V], drf [gamma * V] (row-major), tok [gamma],
 *          r [gamma], seq_key, T > 0.
 * Outputs: k, tokens [gamma+1] (k+1 ids then -1), pq [2*gamma] (p_i(x_i),
 *          q_i(x_i)), Z (sum of the residual at the rejected position, or 1
 *          for the bonus; only if Z_out != NULL), margin (smallest decision
 *          margin along the decisive path), trials (residual trials used;
 *          SPVO_MAX_TRIALS + 1 means the direct fallback ran).
 * Returns SPVO_OK or SPVO_BAD_ROW. */
int spvo_verify_chain_seq(const float *tgt, const float *drf, const int32_t *tok, const float *r,
                          uint64_t seq_key, int gamma, int V, double T,
                          int32_t *k_out, int32_t *tokens_out, double *pq_out, double *Z_out,
                          double *margin_out, int32_t *trials_out)
{
    for (int i = 0; i <= gamma; ++i) tokens_out[i] = -1;
    for (int i = 0; i < 2 * gamma; ++i) pq_out[i] = NAN;
    *k_out = -1;
    *margin_out = INFINITY;
    *trials_out = 0;
    if (Z_out) *Z_out = NAN;
    for (int i = 0; i < gamma; ++i)
        if (tok[i] < 0 || tok[i] >= V) return SPVO_BAD_ROW;

    /* step 2: the gamma+1 target distributions and the gamma draft ones */
    double Mt[65], St[65], Md[64], Sd[64];
    for (int i = 0; i <= gamma; ++i)
        if (spvo_softmax_stats(tgt + (size_t)i * V, V, T, &Mt[i], &St[i]) != SPVO_OK) return SPVO_BAD_ROW;
    for (int i = 0; i < gamma; ++i)
        if (spvo_softmax_stats(drf + (size_t)i * V, V, T, &Md[i], &Sd[i]) != SPVO_OK) return SPVO_BAD_ROW;

    /* step 3: accept / reject, stop at the first rejection */
    int k = gamma;
    double margin = INFINITY;
    for (int i = 0; i < gamma; ++i) {
        const float *ti = tgt + (size_t)i * V, *di = drf + (size_t)i * V;
        double p = prob(ti, tok[i], T, Mt[i], St[i]);
        double q = prob(di, tok[i], T, Md[i], Sd[i]);
        pq_out[2 * i] = p;
        pq_out[2 * i + 1] = q;
        int acc = (p > 0) && ((double)r[i] * q <= p);
        if (i < k) { /* decisions up to the first rejection decide the output */
            double m = (q > 0) ? fabs((double)r[i] - p / q) : INFINITY;
            note_margin(&margin, m);
            if (!acc) k = i;
        }
    }

    /* step 4 */
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    int emitted;
    if (k == gamma) {
        const float *tb = tgt + (size_t)gamma * V;
        for (int x = 0; x < V; ++x) w[x] = prob(tb, x, T, Mt[gamma], St[gamma]);
        emitted = race_sample(w, V, seq_key, SPVO_STREAM_BLOCK, SPVO_STREAM_SUB, SPVO_STREAM_TOKEN, 0,
                              (uint32_t)gamma, &margin);
        if (Z_out) *Z_out = 1.0;
    } else {
        const float *tj = tgt + (size_t)k * V, *dj = drf + (size_t)k * V;
        for (int x = 0; x < V; ++x) w[x] = prob(tj, x, T, Mt[k], St[k]);
        emitted = -1;
        int t;
        for (t = 0; t < SPVO_MAX_TRIALS; ++t) {
            int x = race_sample(w, V, seq_key, SPVO_STREAM_BLOCK, SPVO_STREAM_SUB, SPVO_STREAM_TOKEN, (uint32_t)t,
                                (uint32_t)k, &margin);
            double v = draw_uniform(seq_key, SPVO_STREAM_ACCEPT, (uint32_t)t, (uint32_t)k, 0);
            double p = w[x], q = prob(dj, x, T, Md[k], Sd[k]);
            note_margin(&margin, fabs((1.0 - v) - q / p));
            if (q <= (1.0 - v) * p) { emitted = x; break; }
        }
        *trials_out = (emitted >= 0) ? t + 1 : SPVO_MAX_TRIALS + 1;
        /* residual masses max(0, p - q) (also the fallback's race weights) */
        for (int x = 0; x < V; ++x) {
            double d = w[x] - prob(dj, x, T, Md[k], Sd[k]);
            w[x] = d > 0 ? d : 0.0;
        }
        ksum Z = { 0, 0 };
        for (int x = 0; x < V; ++x) ksum_add(&Z, w[x]);
        if (emitted < 0) {
            /* No positive residual mass: impossible when x_k was drawn from
             * q_k (then sum (p-q)+ = sum (q-p)+ >= q(x_k) - p(x_k) > 0), but a
             * caller may pass a token outside q's support; the row is bad. */
            if (!(ksum_val(&Z) > 0)) {
                free(w);
                for (int i = 0; i < 2 * gamma; ++i) pq_out[i] = NAN;
                return SPVO_BAD_ROW;
            }
            emitted = race_sample(w, V, seq_key, SPVO_STREAM_FB_BLOCK, SPVO_STREAM_FB_SUB, SPVO_STREAM_FB_TOKEN, 0,
                                  (uint32_t)k, &margin);
        }
        if (Z_out) *Z_out = ksum_val(&Z);
    }
    free(w);
    for (int i = 0; i < k; ++i) tokens_out[i] = tok[i];
    tokens_out[k] = emitted;
    *k_out = k;
    *margin_out = margin;
    return SPVO_OK;
}

/* ------------------------------------------------------------------------ */
/* Fan-out, [SSD] Figure 2: at each position k the F_k top-ranked draft
 * tokens by draft logit, excluding the token already sent for verification
 * there.  Order: logit descending (-0.0 equal to +0.0), then id ascending. */
typedef struct { double v; int id; } vid;
static int cmp_vid(const void *a, const void *b)
{
    const vid *x = (const vid *)a, *y = (const vid *)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->id > y->id) - (x->id < y->id);
}

int spvo_fanout_row(const float *d, int V, int exclude, int F, int32_t *ids_out)
{
    for (int i = 0; i < F; ++i) ids_out[i] = -1;
    vid *all = (vid *)malloc(sizeof(vid) * (size_t)V);
    int n = 0;
    for (int x = 0; x < V; ++x) {
        double v = (double)d[x];
        if (isnan(v)) { free(all); return SPVO_BAD_ROW; }
        if (x == exclude) continue;
        all[n].v = v + 0.0; /* -0.0 + 0.0 == +0.0 */
        all[n].id = x;
        ++n;
    }
    qsort(all, (size_t)n, sizeof(vid), cmp_vid);
    for (int i = 0; i < F && i < n; ++i) ids_out[i] = all[i].id;
    free(all);
    return SPVO_OK;
}

/* [SSD] "Core Technical Barrier" (Theorem 12): F_k = F_0 * a_p^(k/(1+r)). */
double spvo_fanout_size(int F0, double a, double r, int k)
{
    return (double)F0 * pow(a, (double)k / (1.0 + r));
}

/* ------------------------------------------------------------------------ */
/* Top-k / top-p filtered rows, [SPD] "Evaluation": the sampled runs (T = 1)
 * draw from the target and draft distributions restricted by top-k = 50 and
 * top-p = 1.0.  The filter of one row at temperature T > 0:
 *   1. rank the ids by logit (descending, -0.0 equal to +0.0, ties to the
 *      lower id) and keep the first top_k;
 *   2. give them the probabilities renormalised over the kept ids,
 *      P(x) = exp(y_x - y_max) / sum_kept exp(y_j - y_max), y = z / T;
 *   3. if top_p < 1, keep only the shortest prefix (in rank order) whose
 *      probability sum reaches top_p, and renormalise over that prefix.
 * Every other id has probability 0.  Writes the kept ids and probabilities
 * in rank order and returns their count, or -1 for a bad row (NaN or +inf
 * anywhere, or no finite logit among the kept ids).  The top-p cut is the
 * only floating-point decision; its margin min(top_p - C_{n-1}, C_n - top_p)
 * (C_j = probability sum of the first j kept ids) is recorded. */
int spvo_filter_row(const float *z, int V, double T, int top_k, double top_p, int32_t *ids_out,
                    double *probs_out, double *margin)
{
    vid *all = (vid *)malloc(sizeof(vid) * (size_t)V);
    for (int x = 0; x < V; ++x) {
        double v = (double)z[x];
        if (isnan(v) || (isinf(v) && v > 0)) { free(all); return -1; }
        all[x].v = v + 0.0;
        all[x].id = x;
    }
    qsort(all, (size_t)V, sizeof(vid), cmp_vid);
    int n = top_k < V ? top_k : V;
    if (isinf(all[0].v)) { free(all); return -1; } /* no finite logit at all */
    double ymax = all[0].v / T;
    ksum S = { 0, 0 };
    for (int j = 0; j < n; ++j) {
        ids_out[j] = all[j].id;
        probs_out[j] = exp(all[j].v / T - ymax);
        ksum_add(&S, probs_out[j]);
    }
    free(all);
    double s = ksum_val(&S);
    for (int j = 0; j < n; ++j) probs_out[j] /= s;
    if (top_p < 1.0) {
        ksum C = { 0, 0 };
        int cut = n;
        for (int j = 0; j < n; ++j) {
            double before = ksum_val(&C);
            ksum_add(&C, probs_out[j]);
            double after = ksum_val(&C);
            if (after >= top_p) {
                note_margin(margin, top_p - before);
                note_margin(margin, after - top_p);
                cut = j + 1;
                break;
            }
        }
        n = cut;
        ksum S2 = { 0, 0 };
        for (int j = 0; j < n; ++j) ksum_add(&S2, probs_out[j]);
        double s2 = ksum_val(&S2);
        for (int j = 0; j < n; ++j) probs_out[j] /= s2;
    }
    return n;
}

/* Probability of id x under a filtered row (0 when x is not kept). */
static double filtered_prob(const int32_t *ids, const double *probs, int n, int x)
{
    for (int j = 0; j < n; ++j)
        if (ids[j] == x) return probs[j];
    return 0.0;
}

/* Chain verify of one sequence on the filtered distributions p'_i, q'_i of
 * spvo_filter_row (the same top_k, top_p for target and draft): [SD] steps
 * 3 and 4 unchanged -- accept x_i iff p'_i(x_i) > 0 and r_i q'_i(x_i) <=
 * p'_i(x_i), stop at the first rejection, then one draw from
 * norm(max(0, p'_k - q'_k)) (rejection at k) or from p'_gamma (bonus).  The
 * draw is an exponential race over the kept target ids: the id x with the
 * smallest E_x / w(x) wins (E_x = -ln U for draw n = x of stream
 * SPVO_STREAM_FILTERED, trial 0, position k; ties to the lower id), which is
 * exactly distributed as w / sum w.  Outputs as spvo_verify_chain_seq (pq
 * holds p'_i(x_i), q'_i(x_i)); the margin also covers the top-p cuts of the
 * rows read. */
int spvo_verify_filtered_seq(const float *tgt, const float *drf, const int32_t *tok, const float *r,
                             uint64_t seq_key, int gamma, int V, double T, int top_k, double top_p,
                             int32_t *k_out, int32_t *tokens_out, double *pq_out, double *Z_out,
                             double *margin_out)
{
    for (int i = 0; i <= gamma; ++i) tokens_out[i] = -1;
    for (int i = 0; i < 2 * gamma; ++i) pq_out[i] = NAN;
    *k_out = -1;
    *margin_out = INFINITY;
    if (Z_out) *Z_out = NAN;
    for (int i = 0; i < gamma; ++i)
        if (tok[i] < 0 || tok[i] >= V) return SPVO_BAD_ROW;
    int K = top_k < V ? top_k : V;
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)K * (size_t)(2 * gamma + 1));
    double *pr = (double *)malloc(sizeof(double) * (size_t)K * (size_t)(2 * gamma + 1));
    int n[129];
    double margin = INFINITY;
    int bad = 0;
    /* rows 0..gamma: target; gamma+1..2gamma: draft */
    for (int row = 0; row <= 2 * gamma && !bad; ++row) {
        const float *z = row <= gamma ? tgt + (size_t)row * V : drf + (size_t)(row - gamma - 1) * V;
        n[row] = spvo_filter_row(z, V, T, top_k, top_p, ids + (size_t)row * K, pr + (size_t)row * K, &margin);
        if (n[row] < 0) bad = 1;
    }
    if (bad) { free(ids); free(pr); return SPVO_BAD_ROW; }

    int k = gamma;
    for (int i = 0; i < gamma; ++i) {
        double p = filtered_prob(ids + (size_t)i * K, pr + (size_t)i * K, n[i], tok[i]);
        double q = filtered_prob(ids + (size_t)(gamma + 1 + i) * K, pr + (size_t)(gamma + 1 + i) * K,
                                 n[gamma + 1 + i], tok[i]);
        pq_out[2 * i] = p;
        pq_out[2 * i + 1] = q;
        int stands = (p > 0) && ((double)r[i] * q <= p);
        if (i < k) {
            note_margin(&margin, (q > 0) ? fabs((double)r[i] - p / q) : INFINITY);
            if (!stands) k = i;
        }
    }
    /* draw over the kept target ids of row k, taken in ascending id order */
    const int32_t *ti = ids + (size_t)k * K;
    const double *tp = pr + (size_t)k * K;
    int m = n[k];
    int order[64 + 1];
    double w[64 + 1], arr[64 + 1];
    for (int j = 0; j < m; ++j) order[j] = j;
    for (int a = 1; a < m; ++a)          /* insertion sort by id */
        for (int b2 = a; b2 > 0 && ti[order[b2 - 1]] > ti[order[b2]]; --b2) {
            int t = order[b2]; order[b2] = order[b2 - 1]; order[b2 - 1] = t;
        }
    ksum Z = { 0, 0 };
    for (int j = 0; j < m; ++j) {
        int x = ti[order[j]];
        double wx = tp[order[j]];
        if (k < gamma) {
            double qx = filtered_prob(ids + (size_t)(gamma + 1 + k) * K, pr + (size_t)(gamma + 1 + k) * K,
                                      n[gamma + 1 + k], x);
            wx = wx - qx > 0 ? wx - qx : 0.0;
        }
        w[j] = wx;
        ksum_add(&Z, wx);
        arr[j] = wx > 0 ? expo(seq_key, SPVO_STREAM_FILTERED, 0, (uint32_t)k, (uint64_t)x) / wx : INFINITY;
    }
    if (!(ksum_val(&Z) > 0)) { /* no positive residual mass (token outside q's support): bad row */
        free(ids);
        free(pr);
        for (int i = 0; i < 2 * gamma; ++i) pq_out[i] = NAN;
        return SPVO_BAD_ROW;
    }
    int jw = race_winner(arr, m, &margin);
    int emitted = ti[order[jw]];
    if (Z_out) *Z_out = (k == gamma) ? 1.0 : ksum_val(&Z);
    free(ids);
    free(pr);
    for (int i = 0; i < k; ++i) tokens_out[i] = tok[i];
    tokens_out[k] = emitted;
    *k_out = k;
    *margin_out = margin;
    return SPVO_OK;
}

/* ------------------------------------------------------------------------ */
/* Saguaro sampling, [SSD] "Key Innovations" / Table 7b (logit bonus C,
 * Theorem 15: the cache hit rate grows with C, C = 1 being plain sampling).
 * Reading: at draft position i the draft samples from
 *   q_C(x) = q(x) w(x) / sum_y q(y) w(y),   w(x) = 1/C if x is one of the
 * position's cached candidates S_i, else 1,
 * i.e. the cached candidates' draft logits are lowered by T ln C.  The verify
 * step is [SD] steps 3 and 4 with q_C in place of q -- exact for the draft
 * tokens drawn from q_C -- so a rejection's residual max(0, p - q_C) leans
 * towards the cached candidates.  S_i = the ids of cache_ids[off_i ..
 * off_i + F_i) (k-major lists, as for the cache lookup) that lie in [0, V),
 * counted once.  Same outputs, sampling rule and streams as
 * spvo_verify_chain_seq; pq holds p_i(x_i), q_C,i(x_i). */
static double sag_prob(const float *z, const unsigned char *inS, int x, double T, double M, double S, double invC)
{
    return exp((double)z[x] / T - M) * (inS[x] ? invC : 1.0) / S;
}

int spvo_verify_saguaro_seq(const float *tgt, const float *drf, const int32_t *tok, const float *r, uint64_t seq_key,
                            int gamma, int V, double T, const int32_t *cache_ids, const int32_t *fanout, double C,
                            int32_t *k_out, int32_t *tokens_out, double *pq_out, double *Z_out, double *margin_out,
                            int32_t *trials_out)
{
    for (int i = 0; i <= gamma; ++i) tokens_out[i] = -1;
    for (int i = 0; i < 2 * gamma; ++i) pq_out[i] = NAN;
    *k_out = -1;
    *margin_out = INFINITY;
    *trials_out = 0;
    if (Z_out) *Z_out = NAN;
    for (int i = 0; i < gamma; ++i)
        if (tok[i] < 0 || tok[i] >= V) return SPVO_BAD_ROW;
    const double invC = 1.0 / C;
    double Mt[65], St[65], Md[64], Sd[64];
    for (int i = 0; i <= gamma; ++i)
        if (spvo_softmax_stats(tgt + (size_t)i * V, V, T, &Mt[i], &St[i]) != SPVO_OK) return SPVO_BAD_ROW;
    /* membership of each draft position's cached candidates, and q_C's normaliser */
    unsigned char *inS = (unsigned char *)calloc((size_t)gamma * (size_t)V, 1);
    int off = 0;
    for (int i = 0; i < gamma; ++i) {
        for (int j = 0; j < fanout[i]; ++j) {
            int x = cache_ids[off + j];
            if (x >= 0 && x < V) inS[(size_t)i * V + x] = 1;
        }
        off += fanout[i];
    }
    for (int i = 0; i < gamma; ++i) {
        const float *d = drf + (size_t)i * V;
        double M = -INFINITY;
        for (int x = 0; x < V; ++x) {
            double v = (double)d[x];
            if (isnan(v) || (isinf(v) && v > 0)) { free(inS); return SPVO_BAD_ROW; }
            if (v / T > M) M = v / T;
        }
        if (isinf(M)) { free(inS); return SPVO_BAD_ROW; }
        ksum S = { 0, 0 };
        for (int x = 0; x < V; ++x) ksum_add(&S, exp((double)d[x] / T - M) * (inS[(size_t)i * V + x] ? invC : 1.0));
        Md[i] = M;
        Sd[i] = ksum_val(&S);
    }

    int k = gamma;
    double margin = INFINITY;
    for (int i = 0; i < gamma; ++i) {
        double p = prob(tgt + (size_t)i * V, tok[i], T, Mt[i], St[i]);
        double q = sag_prob(drf + (size_t)i * V, inS + (size_t)i * V, tok[i], T, Md[i], Sd[i], invC);
        pq_out[2 * i] = p;
        pq_out[2 * i + 1] = q;
        int holds = (p > 0) && ((double)r[i] * q <= p);
        if (i < k) {
            note_margin(&margin, (q > 0) ? fabs((double)r[i] - p / q) : INFINITY);
            if (!holds) k = i;
        }
    }
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    int emitted;
    if (k == gamma) {
        const float *last = tgt + (size_t)gamma * V;
        for (int x = 0; x < V; ++x) w[x] = prob(last, x, T, Mt[gamma], St[gamma]);
        emitted = race_sample(w, V, seq_key, SPVO_STREAM_BLOCK, SPVO_STREAM_SUB, SPVO_STREAM_TOKEN, 0,
                              (uint32_t)gamma, &margin);
        if (Z_out) *Z_out = 1.0;
    } else {
        const float *tj = tgt + (size_t)k * V, *dj = drf + (size_t)k * V;
        const unsigned char *sj = inS + (size_t)k * V;
        for (int x = 0; x < V; ++x) w[x] = prob(tj, x, T, Mt[k], St[k]);
        emitted = -1;
        int t;
        for (t = 0; t < SPVO_MAX_TRIALS; ++t) {
            int x = race_sample(w, V, seq_key, SPVO_STREAM_BLOCK, SPVO_STREAM_SUB, SPVO_STREAM_TOKEN, (uint32_t)t,
                                (uint32_t)k, &margin);
            double v = draw_uniform(seq_key, SPVO_STREAM_ACCEPT, (uint32_t)t, (uint32_t)k, 0);
            double p = w[x], q = sag_prob(dj, sj, x, T, Md[k], Sd[k], invC);
            note_margin(&margin, fabs((1.0 - v) - q / p));
            if (q <= (1.0 - v) * p) {
                emitted = x;
                break;
            }
        }
        *trials_out = (emitted >= 0) ? t + 1 : SPVO_MAX_TRIALS + 1;
        for (int x = 0; x < V; ++x) {
            double d = w[x] - sag_prob(dj, sj, x, T, Md[k], Sd[k], invC);
            w[x] = d > 0 ? d : 0.0;
        }
        ksum Z = { 0, 0 };
        for (int x = 0; x < V; ++x) ksum_add(&Z, w[x]);
        if (emitted < 0) {
            if (!(ksum_val(&Z) > 0)) {
                free(w);
                free(inS);
                for (int i = 0; i < 2 * gamma; ++i) pq_out[i] = NAN;
                return SPVO_BAD_ROW;
            }
            emitted = race_sample(w, V, seq_key, SPVO_STREAM_FB_BLOCK, SPVO_STREAM_FB_SUB, SPVO_STREAM_FB_TOKEN, 0,
                                  (uint32_t)k, &margin);
        }
        if (Z_out) *Z_out = ksum_val(&Z);
    }
    free(w);
    free(inS);
    for (int i = 0; i < k; ++i) tokens_out[i] = tok[i];
    tokens_out[k] = emitted;
    *k_out = k;
    *margin_out = margin;
    return SPVO_OK;
}

void spvo_verify_saguaro_batch(const float *tgt, const float *drf, const int32_t *tok, const float *r,
                               const uint64_t *keys, int b0, int b1, int gamma, int V, double T,
                               const int32_t *cache_ids, const int32_t *fanout, int sumF, double C,
                               int32_t *k_out, int32_t *tokens_out, double *pq_out, double *Z_out,
                               double *margin_out, int32_t *trials_out, int32_t *status_out)
{
    for (int b = b0; b < b1; ++b) {
        status_out[b] = spvo_verify_saguaro_seq(
            tgt + (size_t)b * (size_t)(gamma + 1) * (size_t)V, drf + (size_t)b * (size_t)gamma * (size_t)V,
            tok + (size_t)b * gamma, r + (size_t)b * gamma, keys[b], gamma, V, T, cache_ids + (size_t)b * sumF,
            fanout, C, &k_out[b], tokens_out + (size_t)b * (gamma + 1), pq_out + (size_t)b * 2 * gamma,
            Z_out ? &Z_out[b] : 0, &margin_out[b], &trials_out[b]);
    }
}

/* ------------------------------------------------------------------------ */
/* Tree verify.  The pages name draft trees ([SPD] tree drafting of width 4;
 * tree-style verification with k = 21 in the benchmark study the survey
 * page cites) but give no verification rule.  This follows the published
 * multi-round speculative sampling for token trees (Miao et al., SpecInfer,
 * stochastic verification), restated: the children of node u were drawn
 * i.i.d. from q_u and are tested in index order against a residual that
 * shrinks with every rejection,
 *   P_0 = p_u,  P_m(x) = max(0, p_u(x) - s_m q_u(x)) / N_m,
 *   s_0 = 0, s_{m+1} = s_m + N_m, N_0 = 1, N_m = sum_x max(0, p_u - s_m q_u),
 * child c (token x) being accepted iff P_m(x) > 0 and r_c q_u(x) <= P_m(x).
 * The walk descends into the first accepted child; when every child of u is
 * rejected (m = number of children) one token is drawn from P_m, and at a
 * leaf the bonus token from p_u.  With one child per node this is [SD]
 * steps 3 and 4 exactly (s_1 = 1: the residual max(0, p - q)).
 * Draws use the race and rejection trials of the chain (trial t accepts x ~
 * p_u iff s_m q_u(x) <= (1 - v) p_u(x)), position = the node's index.
 * Inputs: tgt, drf [N * V] (row v: p, q at node v), parent [N] (parent[0] =
 * -1, 0 <= parent[v] < v), tok [N] (token of node v >= 1), r [N].
 * Outputs: k (accepted nodes), tokens_out [N] (their tokens, then the drawn
 * one, then -1), nodes_out [N] (the accepted nodes, then -1). */
static int tree_trials(const double *w, const float *dj, int V, double T, double Md, double Sd, double sres,
                       uint64_t key, uint32_t pos, double *margin, int *trials)
{
    int t;
    for (t = 0; t < SPVO_MAX_TRIALS; ++t) {
        int x = race_sample(w, V, key, SPVO_STREAM_BLOCK, SPVO_STREAM_SUB, SPVO_STREAM_TOKEN, (uint32_t)t, pos, margin);
        double v = draw_uniform(key, SPVO_STREAM_ACCEPT, (uint32_t)t, pos, 0);
        double p = w[x], q = sres * prob(dj, x, T, Md, Sd);
        note_margin(margin, fabs((1.0 - v) - q / p));
        if (q <= (1.0 - v) * p) { *trials = t + 1; return x; }
    }
    *trials = SPVO_MAX_TRIALS + 1;
    return -1;
}

int spvo_verify_tree_seq(const float *tgt, const float *drf, const int32_t *parent, const int32_t *tok, const float *r,
                         uint64_t seq_key, int N, int V, double T, int32_t *k_out, int32_t *tokens_out,
                         int32_t *nodes_out, double *margin_out, int32_t *trials_out)
{
    for (int i = 0; i < N; ++i) { tokens_out[i] = -1; nodes_out[i] = -1; }
    *k_out = -1;
    *margin_out = INFINITY;
    *trials_out = 0;
    if (N < 1 || parent[0] != -1) return SPVO_BAD_ROW;
    for (int v = 1; v < N; ++v)
        if (parent[v] < 0 || parent[v] >= v || tok[v] < 0 || tok[v] >= V) return SPVO_BAD_ROW;
    /* Every target row, and the draft row of every node with children, must
     * be a distribution, whether or not the walk reaches it: the outcome of a
     * sequence does not depend on where its bad rows sit. */
    for (int v = 0; v < N; ++v) {
        double M, S;
        if (spvo_softmax_stats(tgt + (size_t)v * V, V, T, &M, &S) != SPVO_OK) return SPVO_BAD_ROW;
    }
    for (int v = 1; v < N; ++v) {
        double M, S;
        if (spvo_softmax_stats(drf + (size_t)parent[v] * V, V, T, &M, &S) != SPVO_OK) return SPVO_BAD_ROW;
    }
    double margin = INFINITY;
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    int u = 0, k = 0, emitted = -1, total_trials = 0;
    for (;;) {
        const float *tu = tgt + (size_t)u * V, *du = drf + (size_t)u * V;
        double Mt, St;
        if (spvo_softmax_stats(tu, V, T, &Mt, &St) != SPVO_OK) { free(w); return SPVO_BAD_ROW; }
        int nkids = 0;
        for (int c = u + 1; c < N; ++c) nkids += parent[c] == u;
        for (int x = 0; x < V; ++x) w[x] = prob(tu, x, T, Mt, St);
        if (nkids == 0) { /* leaf: the bonus token from p_u */
            emitted = race_sample(w, V, seq_key, SPVO_STREAM_BLOCK, SPVO_STREAM_SUB, SPVO_STREAM_TOKEN, 0,
                                  (uint32_t)u, &margin);
            break;
        }
        double Md, Sd;
        if (spvo_softmax_stats(du, V, T, &Md, &Sd) != SPVO_OK) { free(w); return SPVO_BAD_ROW; }
        double s = 0.0, Nm = 1.0;
        int next = -1;
        for (int c = u + 1; c < N && next < 0; ++c) {
            if (parent[c] != u) continue;
            const int x = tok[c];
            const double px = w[x], qx = prob(du, x, T, Md, Sd);
            const double Pm = (s == 0.0) ? px : (px - s * qx > 0 ? (px - s * qx) / Nm : 0.0);
            note_margin(&margin, (qx > 0) ? fabs((double)r[c] - Pm / qx) : INFINITY);
            if (Pm > 0 && (double)r[c] * qx <= Pm) { next = c; break; }
            /* rejected: the next residual */
            s += Nm;
            ksum Z = { 0, 0 };
            for (int y = 0; y < V; ++y) {
                double d = w[y] - s * prob(du, y, T, Md, Sd);
                if (d > 0) ksum_add(&Z, d);
            }
            Nm = ksum_val(&Z);
            if (!(Nm > 0)) { free(w); return SPVO_BAD_ROW; } /* no residual mass (token outside q's support) */
        }
        if (next >= 0) {
            tokens_out[k] = tok[next];
            nodes_out[k] = next;
            ++k;
            u = next;
            continue;
        }
        /* every child rejected: one draw from P_m = max(0, p - s q) / N_m */
        int tr = 0;
        emitted = tree_trials(w, du, V, T, Md, Sd, s, seq_key, (uint32_t)u, &margin, &tr);
        total_trials = tr;
        if (emitted < 0) {
            for (int y = 0; y < V; ++y) {
                double d = w[y] - s * prob(du, y, T, Md, Sd);
                w[y] = d > 0 ? d : 0.0;
            }
            emitted = race_sample(w, V, seq_key, SPVO_STREAM_FB_BLOCK, SPVO_STREAM_FB_SUB, SPVO_STREAM_FB_TOKEN, 0,
                                  (uint32_t)u, &margin);
        }
        break;
    }
    free(w);
    tokens_out[k] = emitted;
    *k_out = k;
    *margin_out = margin;
    *trials_out = total_trials;
    return SPVO_OK;
}

/* Greedy tree verify (T = 0): descend into the first child whose token is
 * the argmax of p_u (lowest id on ties); emit the argmax of the last node. */
int spvo_verify_tree_greedy_seq(const float *tgt, const int32_t *parent, const int32_t *tok, int N, int V,
                                int32_t *k_out, int32_t *tokens_out, int32_t *nodes_out)
{
    for (int i = 0; i < N; ++i) { tokens_out[i] = -1; nodes_out[i] = -1; }
    *k_out = -1;
    int a;
    if (N < 1 || parent[0] != -1) return SPVO_BAD_ROW;
    for (int v = 1; v < N; ++v)
        if (parent[v] < 0 || parent[v] >= v || tok[v] < 0 || tok[v] >= V) return SPVO_BAD_ROW;
    for (int v = 0; v < N; ++v) /* every target row, reached or not (as in the sampled walk) */
        if (argmax_row(tgt + (size_t)v * V, V, &a) != SPVO_OK) return SPVO_BAD_ROW;
    int u = 0, k = 0;
    for (;;) {
        if (argmax_row(tgt + (size_t)u * V, V, &a) != SPVO_OK) return SPVO_BAD_ROW;
        int next = -1;
        for (int c = u + 1; c < N; ++c)
            if (parent[c] == u && tok[c] == a) { next = c; break; }
        if (next < 0) break;
        tokens_out[k] = tok[next];
        nodes_out[k] = next;
        ++k;
        u = next;
    }
    tokens_out[k] = a;
    *k_out = k;
    return SPVO_OK;
}

void spvo_verify_tree_batch(const float *tgt, const float *drf, const int32_t *parent, const int32_t *tok,
                            const float *r, const uint64_t *keys, int b0, int b1, int N, int V, double T,
                            int32_t *k_out, int32_t *tokens_out, int32_t *nodes_out, double *margin_out,
                            int32_t *trials_out, int32_t *status_out)
{
    for (int b = b0; b < b1; ++b) {
        const size_t o = (size_t)b * N;
        if (T == 0.0) {
            status_out[b] = spvo_verify_tree_greedy_seq(tgt + o * V, parent + o, tok + o, N, V, &k_out[b],
                                                        tokens_out + o, nodes_out + o);
            margin_out[b] = INFINITY;
            trials_out[b] = 0;
        } else {
            status_out[b] = spvo_verify_tree_seq(tgt + o * V, drf + o * V, parent + o, tok + o, r + o, keys[b], N, V, T,
                                                 &k_out[b], tokens_out + o, nodes_out + o, &margin_out[b],
                                                 &trials_out[b]);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Speculation-cache lookup, [SSD] Algorithm 1 ("if verify_outcome in cache")
 * and Figure 2: the cache holds one branch per (k, t) pair, for every
 * position k = 0..K and each of the F_k fan-out candidates t listed for it,
 * in k-major order.  The verify outcome (k accepted, emitted token t*) hits
 * when one of the entries is the pair (k, t*); the result is that entry's
 * index in the row of cache ids, else -1.  A bad row (k < 0) never hits. */
int spvo_cache_slot(int k, int32_t t_star, const int32_t *cache_ids, const int32_t *fanout, int K)
{
    if (k < 0) return -1;
    int slot = 0;
    for (int pos = 0; pos <= K; ++pos) {
        for (int j = 0; j < fanout[pos]; ++j, ++slot) {
            if (pos == k && cache_ids[slot] == t_star) return slot;
        }
    }
    return -1;
}

/* ------------------------------------------------------------------------ */
/* Batch loops over sequences [b0, b1): the same per-sequence functions, so a
 * caller can split a batch across threads without per-sequence overhead. */
void spvo_verify_chain_batch(const float *tgt, const float *drf, const int32_t *tok, const float *r,
                             const uint64_t *keys, int b0, int b1, int gamma, int V, double T,
                             int32_t *k_out, int32_t *tokens_out, double *pq_out, double *Z_out,
                             double *margin_out, int32_t *trials_out, int32_t *status_out)
{
    for (int b = b0; b < b1; ++b) {
        status_out[b] = spvo_verify_chain_seq(
            tgt + (size_t)b * (size_t)(gamma + 1) * (size_t)V, drf + (size_t)b * (size_t)gamma * (size_t)V,
            tok + (size_t)b * gamma, r + (size_t)b * gamma, keys[b], gamma, V, T, &k_out[b],
            tokens_out + (size_t)b * (gamma + 1), pq_out + (size_t)b * 2 * gamma, Z_out ? &Z_out[b] : 0,
            &margin_out[b], &trials_out[b]);
    }
}

void spvo_verify_filtered_batch(const float *tgt, const float *drf, const int32_t *tok, const float *r,
                                const uint64_t *keys, int b0, int b1, int gamma, int V, double T, int top_k,
                                double top_p, int32_t *k_out, int32_t *tokens_out, double *pq_out, double *Z_out,
                                double *margin_out, int32_t *status_out)
{
    for (int b = b0; b < b1; ++b) {
        status_out[b] = spvo_verify_filtered_seq(
            tgt + (size_t)b * (size_t)(gamma + 1) * (size_t)V, drf + (size_t)b * (size_t)gamma * (size_t)V,
            tok + (size_t)b * gamma, r + (size_t)b * gamma, keys[b], gamma, V, T, top_k, top_p, &k_out[b],
            tokens_out + (size_t)b * (gamma + 1), pq_out + (size_t)b * 2 * gamma, Z_out ? &Z_out[b] : 0,
            &margin_out[b]);
    }
}

void spvo_verify_greedy_batch(const float *tgt, const int32_t *tok, int b0, int b1, int gamma, int V,
                              int32_t *k_out, int32_t *tokens_out, int32_t *status_out)
{
    for (int b = b0; b < b1; ++b)
        status_out[b] = spvo_verify_greedy_seq(tgt + (size_t)b * (size_t)(gamma + 1) * (size_t)V,
                                               tok + (size_t)b * gamma, gamma, V, &k_out[b],
                                               tokens_out + (size_t)b * (gamma + 1));
}
