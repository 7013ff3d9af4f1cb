/*
 * dspark_oracle.c -- plain, slow, double-precision CPU oracle for the DSpark
 * draft-sample / schedule / verify path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA kernels.  Every loop is written in the order the method states it, with
 * no blocking, fusion or reordering, so that it can be checked against the
 * sources by eye.
 *
 * Sources (web pages describing the method):
 *  [DSP-IT]  "DSpark, la bozza che sa quando fermarsi: lo speculative decoding
 *            di DeepSeek-V4" (paithon.it), sections "Un po' di autoregressione
 *            basta" (equation for p_k) and "Verificare meglio, non di piu'"
 *            (equations for c_k*, a_j and Theta).
 *  [MATH-FR] "Les mathematiques derriere l'acceleration : comment le decodage
 *            speculatif masque la latence sans modifier les sorties"
 *            (seventnews.com), section "La garantie de l'echantillonnage par
 *            rejet".
 *  [DSP-ZH]  "DeepSeek发布DSpark" (learnblockchain.cn), section "DSpark 是什么？"
 *            (bonus token) and "工作原理：半自回归生成".
 *  [PHILOX]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *            1, 2, 3", SC'11 -- the Philox4x32-10 bijection.
 *
 * Readings where the pages are silent (each one is also listed in the design
 * notes):
 *  R1  Random stream: key = (seed mod 2^32, seed >> 32); counter =
 *      (v >> 2, j, request_id, stream); output word v & 3.  Draws that are not
 *      per-token use v = 0.  Streams: 0 draft Gumbel, 1 accept uniform,
 *      2 residual Gumbel, 3 bonus Gumbel.
 *  R2  u = ((w >> 9) + 1/2) * 2^-23, an exact fp32 value in (0, 1);
 *      Gumbel noise g = -ln(-ln u).
 *  R3  One low-rank factorisation B = E_in * W_out^T serves every block
 *      position; the bias at position j depends only on the previous token
 *      (the anchor for j = 0).
 *  R4  z = U + bias is rounded to fp32 (the value the kernels hold); all later
 *      arithmetic here is double.
 *  R5  Temperature T > 0 divides draft and target logits alike; T = 0 is the
 *      greedy limit (argmax, lowest id on exact ties).
 *  R6  Residual distribution = normalise(max(0, p - q)).  If no entry has
 *      p > q (impossible in exact arithmetic after a rejection) the token is
 *      drawn from p with stream 2.
 *  R7  Confidence calibration c = sigmoid(l / T_pos[j]) (sequential
 *      temperature scaling applied with given per-position temperatures).
 *  R8  Scheduler: B counts batch tokens sum_b (L_b + 1); tau = sum_b
 *      (1 + sum_{j < L_b} a_{b,j}); candidates sorted by (a desc, j asc,
 *      b asc); admit while tau' * SPS(B + 1) > tau * SPS(B); stop at the first
 *      candidate that does not raise Theta.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* [PHILOX] Philox4x32-10: two 32x32->64 multiplies per round, round keys    */
/* bumped by the Weyl constants (golden ratio and sqrt(3)-1).                */
/* ------------------------------------------------------------------------ */
void or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t prod0 = (uint64_t)M0 * (uint64_t)x0;
        uint64_t prod1 = (uint64_t)M1 * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* R1: the 32-bit word for (seed, request, position, token, stream). */
uint32_t or_random_word(uint64_t seed, uint32_t request_id, uint32_t j, uint32_t v, uint32_t stream)
{
    uint32_t key[2] = { (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32) };
    uint32_t ctr[4] = { v >> 2, j, request_id, stream };
    uint32_t out[4];
    or_philox4x32_10(ctr, key, out);
    return out[v & 3u];
}

/* R2: uniform in (0, 1). */
double or_uniform(uint64_t seed, uint32_t request_id, uint32_t j, uint32_t v, uint32_t stream)
{
    uint32_t w = or_random_word(seed, request_id, j, v, stream);
    return ((double)(w >> 9) + 0.5) * (1.0 / 8388608.0); /* 2^-23 */
}

/* R2: standard Gumbel noise. */
double or_gumbel(uint64_t seed, uint32_t request_id, uint32_t j, uint32_t v, uint32_t stream)
{
    double u = or_uniform(seed, request_id, j, v, stream);
    return -log(-log(u));
}

/* Bulk form of or_uniform for tokens v0 .. v0 + n - 1 (used by statistical
 * tests of the stream). */
void or_uniforms(uint64_t seed, uint32_t request_id, uint32_t j, uint32_t v0, int n,
                 uint32_t stream, double *out)
{
    for (int i = 0; i < n; ++i) out[i] = or_uniform(seed, request_id, j, v0 + (uint32_t)i, stream);
}

/* ------------------------------------------------------------------------ */
/* Helpers on one row of V doubles.                                          */
/* ------------------------------------------------------------------------ */

/* log sum_v exp(s_v), max-shifted. */
static double row_logsumexp(const double *s, int V)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) if (s[v] > m) m = s[v];
    double sum = 0.0;
    for (int v = 0; v < V; ++v) sum += exp(s[v] - m);
    return m + log(sum);
}

/* argmax with lowest index on exact ties; also reports the top-two gap. */
static int row_argmax(const double *s, int V, double *gap, double *top)
{
    int best = 0;
    double b1 = s[0], b2 = -INFINITY;
    for (int v = 1; v < V; ++v) {
        if (s[v] > b1) { b2 = b1; b1 = s[v]; best = v; }
        else if (s[v] > b2) { b2 = s[v]; }
    }
    if (gap) *gap = b1 - b2;
    if (top) *top = b1;
    return best;
}

/* Gumbel-max draw with one random word per token, keyed on (seed, request,
 * position, token, stream) (reading R1):
 *   x = argmax_v ( w_v + g(u_{stream, j, v}) ),  g(u) = -log(-log u),
 * over the entries with w_v > -inf, the lowest id on exact ties.  With w the
 * logits s = z / T this draws x with probability softmax(s)_x exactly; with
 * w_v = log r_v it draws from r normalised.  Every token takes its own word
 * (or_uniform at token v).  gap / top: the difference of the two largest keys
 * and the largest key (how close the draw came to a tie). */
static int gumbel_max(const double *w, int V, uint64_t seed, uint32_t rid, uint32_t j, uint32_t stream,
                      double *gap, double *top)
{
    int best = -1;
    double k1 = -INFINITY, k2 = -INFINITY;
    for (int v = 0; v < V; ++v) {
        if (w[v] == -INFINITY) continue;
        double key = w[v] + or_gumbel(seed, rid, j, (uint32_t)v, stream);
        if (best < 0 || key > k1) { k2 = k1; k1 = key; best = v; }
        else if (key > k2) { k2 = key; }
    }
    if (gap) *gap = k1 - k2;
    if (top) *top = k1;
    return best;
}

/* [DSP-IT] "Un po' di autoregressione basta", equation for p_k, with the
 * Markov head B = W1 W2 (R3, R4).  W1 = E_in is stored [V][r]; W2 is stored
 * transposed as W_out [V][r] (row v scores token v), so
 *   z_v = fp32( U[v] + sum_k E_in[prev, k] * W_out[v, k] ). */
static void markov_logits(const double *U_row, const double *E_in, const double *W_out,
                          int prev, int V, int r, double *z)
{
    const double *e = E_in + (size_t)prev * (size_t)r;
    for (int v = 0; v < V; ++v) {
        const double *w = W_out + (size_t)v * (size_t)r;
        double bias = 0.0;
        for (int k = 0; k < r; ++k) bias += e[k] * w[k];
        z[v] = (double)(float)(U_row[v] + bias);
    }
}

/* ------------------------------------------------------------------------ */
/* Draft sampling, left to right over the block ([DSP-IT] "Un po' di         */
/* autoregressione basta": each draft token keeps an explicit softmax         */
/* probability; the sampled token feeds the next position's bias).            */
/*                                                                           */
/* U [B][G][V], E_in [V][r], W_out [V][r], anchor [B], temp [B], rid [B]      */
/* (NULL = 0..B-1).  Outputs [B][G]: tokens (Gumbel-max on stream 0), lse     */
/* (T = 0: max z), logq (T = 0: 0), gap / top of the two largest keys (T = 0: */
/* of the logits); z_out [B][G][V] optional.                                  */
/* Returns 0, or -1 on an out-of-range anchor.                                */
/* ------------------------------------------------------------------------ */
int or_draft_sample(const double *U, const double *E_in, const double *W_out,
                    const int32_t *anchor, const double *temp, const uint32_t *rid,
                    int B, int G, int V, int r, uint64_t seed,
                    int32_t *tokens, double *lse, double *logq, double *gap, double *top,
                    double *z_out)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    double *s = (double *)malloc(sizeof(double) * (size_t)V);
    if (!z || !s) { free(z); free(s); return -2; }
    for (int b = 0; b < B; ++b) {
        uint32_t id = rid ? rid[b] : (uint32_t)b;
        double T = temp[b];
        int prev = anchor[b];
        if (prev < 0 || prev >= V) { free(z); free(s); return -1; }
        for (int j = 0; j < G; ++j) {
            size_t o = (size_t)b * (size_t)G + (size_t)j;
            const double *U_row = U + o * (size_t)V;
            markov_logits(U_row, E_in, W_out, prev, V, r, z);
            if (z_out) memcpy(z_out + o * (size_t)V, z, sizeof(double) * (size_t)V);
            int x;
            if (T > 0.0) {
                for (int v = 0; v < V; ++v) s[v] = z[v] / T;
                double l = row_logsumexp(s, V);
                x = gumbel_max(s, V, seed, id, (uint32_t)j, 0u, &gap[o], &top[o]);
                lse[o] = l;
                logq[o] = s[x] - l;
            } else {
                x = row_argmax(z, V, &gap[o], &top[o]);
                lse[o] = z[x];
                logq[o] = 0.0;
            }
            tokens[o] = x;
            prev = x;
        }
    }
    free(z); free(s);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The recurrent (RNN) head, the second sequential head the pages set beside  */
/* the Markov head ([DSP-IT] "Un po' di autoregressione basta"; the aitalk   */
/* overview "Un drafter...").  The pages do not give the cell; reading R12:   */
/*   h_{-1} = 0, x_{-1} = anchor,                                             */
/*   h_j = bf16( tanh( E_in[x_{j-1}] + W_h h_{j-1} ) )   (an Elman cell whose */
/*         input term is the embedding of the previous token; the state is   */
/*         kept in bf16, the storage type of the head's weights),           */
/*   bias_j[v] = sum_k h_j[k] W_out[v][k],  z = fp32(U + bias).              */
/* W_h is [r][r] with row n the weights of output unit n.  Everything else   */
/* (temperature, Gumbel-max, streams) is as in or_draft_sample.             */
/* h_out [B][G][r] receives the states; h_margin [B][G] the smallest relative */
/* distance of a pre-rounding state value to a bf16 rounding boundary (a      */
/* value on a boundary may round either way under another summation order). */
/* ------------------------------------------------------------------------ */
static double bf16_rne(double x, double *margin)
{
    if (x == 0.0 || !isfinite(x)) { if (margin) *margin = INFINITY; return x; }
    int e;
    double m = frexp(x, &e);          /* x = m 2^e, 0.5 <= |m| < 1 */
    double sc = ldexp(m, 8);          /* 8 significant bits */
    double fl = floor(sc);
    if (margin) *margin = fabs((sc - fl) - 0.5) / fabs(sc);
    double rn = nearbyint(sc);        /* round half to even (default mode) */
    return ldexp(rn, e - 8);
}

int or_draft_sample_rnn(const double *U, const double *E_in, const double *W_h, const double *W_out,
                        const int32_t *anchor, const double *temp, const uint32_t *rid,
                        int B, int G, int V, int r, uint64_t seed,
                        int32_t *tokens, double *lse, double *logq, double *gap, double *top,
                        double *h_out, double *h_margin, double *z_out)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    double *s = (double *)malloc(sizeof(double) * (size_t)V);
    double *h = (double *)malloc(sizeof(double) * (size_t)r);
    double *hn = (double *)malloc(sizeof(double) * (size_t)r);
    if (!z || !s || !h || !hn) { free(z); free(s); free(h); free(hn); return -2; }
    for (int b = 0; b < B; ++b) {
        uint32_t id = rid ? rid[b] : (uint32_t)b;
        double T = temp[b];
        int prev = anchor[b];
        if (prev < 0 || prev >= V) { free(z); free(s); free(h); free(hn); return -1; }
        for (int k = 0; k < r; ++k) h[k] = 0.0;
        for (int j = 0; j < G; ++j) {
            size_t o = (size_t)b * (size_t)G + (size_t)j;
            /* the state update */
            double mm = INFINITY;
            for (int n = 0; n < r; ++n) {
                double a = E_in[(size_t)prev * (size_t)r + n];
                for (int k = 0; k < r; ++k) a += W_h[(size_t)n * (size_t)r + k] * h[k];
                double mg;
                hn[n] = bf16_rne(tanh(a), &mg);
                if (mg < mm) mm = mg;
            }
            memcpy(h, hn, sizeof(double) * (size_t)r);
            if (h_out) memcpy(h_out + o * (size_t)r, h, sizeof(double) * (size_t)r);
            if (h_margin) h_margin[o] = mm;
            /* the bias and the logits of this position */
            const double *U_row = U + o * (size_t)V;
            for (int v = 0; v < V; ++v) {
                const double *w = W_out + (size_t)v * (size_t)r;
                double bias = 0.0;
                for (int k = 0; k < r; ++k) bias += h[k] * w[k];
                z[v] = (double)(float)(U_row[v] + bias);
            }
            if (z_out) memcpy(z_out + o * (size_t)V, z, sizeof(double) * (size_t)V);
            int x;
            if (T > 0.0) {
                for (int v = 0; v < V; ++v) s[v] = z[v] / T;
                double l = row_logsumexp(s, V);
                x = gumbel_max(s, V, seed, id, (uint32_t)j, 0u, &gap[o], &top[o]);
                lse[o] = l;
                logq[o] = s[x] - l;
            } else {
                x = row_argmax(z, V, &gap[o], &top[o]);
                lse[o] = z[x];
                logq[o] = 0.0;
            }
            tokens[o] = x;
            prev = x;
        }
    }
    free(z); free(s); free(h); free(hn);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Confidence calibration and prefix scheduler ([DSP-IT] "Verificare meglio, */
/* non di piu'": c_k, a_j = prod_{i<=j} c_i, Theta = tau * SPS(B), greedy     */
/* admission in a-order with the early stop), readings R7 and R8.             */
/*                                                                           */
/* conf_logits [B][G], pos_temp [G], sps [sps_len] (SPS of n batch tokens).   */
/* Outputs: conf, cum_conf [B][G], verify_len [B], theta (final Theta),       */
/* n_admitted, min_margin = smallest |Theta' - Theta| / Theta over the        */
/* decisions taken, min_tie = smallest relative gap between consecutive a in  */
/* the sorted candidate list (both for the parity exemption).                 */
/* Returns 0, or -1 on invalid sizes.                                         */
/* ------------------------------------------------------------------------ */
typedef struct { double a; int j; int b; } or_cand;

static int cand_order(const void *pa, const void *pb)
{
    const or_cand *x = (const or_cand *)pa, *y = (const or_cand *)pb;
    if (x->a > y->a) return -1;
    if (x->a < y->a) return 1;
    if (x->j != y->j) return x->j < y->j ? -1 : 1;
    if (x->b != y->b) return x->b < y->b ? -1 : 1;
    return 0;
}

int or_schedule(const double *conf_logits, const double *pos_temp, const double *sps, int sps_len,
                int B, int G, int L_min, int L_max,
                double *conf, double *cum_conf, int32_t *verify_len, double *theta,
                int32_t *n_admitted, double *min_margin, double *min_tie)
{
    if (B < 0 || G < 1 || L_min < 0 || L_min > L_max || L_max > G) return -1;
    if (sps_len < B * (L_max + 1) + 1) return -1;
    for (int b = 0; b < B; ++b) {
        double prod = 1.0;
        for (int j = 0; j < G; ++j) {
            double l = conf_logits[(size_t)b * G + j];
            double c = 1.0 / (1.0 + exp(-l / pos_temp[j]));
            prod *= c;
            conf[(size_t)b * G + j] = c;
            cum_conf[(size_t)b * G + j] = prod;
        }
    }
    double tau = 0.0;
    long btok = 0;
    for (int b = 0; b < B; ++b) {
        verify_len[b] = L_min;
        double t = 1.0;
        for (int j = 0; j < L_min; ++j) t += cum_conf[(size_t)b * G + j];
        tau += t;
        btok += L_min + 1;
    }
    int nc = B * (L_max - L_min);
    or_cand *cand = (or_cand *)malloc(sizeof(or_cand) * (size_t)(nc > 0 ? nc : 1));
    if (!cand) return -2;
    int n = 0;
    for (int b = 0; b < B; ++b)
        for (int j = L_min; j < L_max; ++j) {
            cand[n].a = cum_conf[(size_t)b * G + j];
            cand[n].j = j;
            cand[n].b = b;
            ++n;
        }
    qsort(cand, (size_t)nc, sizeof(or_cand), cand_order);
    double mt = INFINITY;
    for (int i = 0; i + 1 < nc; ++i) {
        double d = fabs(cand[i].a - cand[i + 1].a) / fmax(fabs(cand[i].a), 1e-300);
        if (d < mt) mt = d;
    }
    double th = tau * sps[btok];
    double mm = INFINITY;
    int admitted = 0;
    for (int i = 0; i < nc; ++i) {
        double tau2 = tau + cand[i].a;
        double th2 = tau2 * sps[btok + 1];
        double margin = fabs(th2 - th) / fmax(fabs(th), 1e-300);
        if (margin < mm) mm = margin;
        if (th2 > th) {
            verify_len[cand[i].b] = cand[i].j + 1;
            tau = tau2;
            btok += 1;
            th = th2;
            ++admitted;
        } else {
            break; /* early stop: the first candidate that does not raise Theta */
        }
    }
    free(cand);
    if (theta) *theta = th;
    if (n_admitted) *n_admitted = admitted;
    if (min_margin) *min_margin = mm;
    if (min_tie) *min_tie = mt;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Other verify-length policies the pages describe next to the early-stop    */
/* scheduler ([DSP-IT] "Che cosa resta da verificare": production schedules  */
/* from confidences two rounds old and drops the early stop; "Verificare     */
/* meglio, non di piu'" and [DSP-ZH] "置信度调度的验证": a fixed confidence     */
/* threshold as the simpler comparator).  Readings:                           */
/*  policy 0  the early stop above (or_schedule);                             */
/*  policy 1  no early stop: over the same candidate order, admit the count   */
/*            n in 0..ncand whose Theta(n) = tau_n * SPS(B_tok + n) is        */
/*            largest (the first such n);                                    */
/*  policy 2  threshold on the prefix survival: L_b grows from L_min while    */
/*            a_{b,L_b} > threshold (a is non-increasing in j);              */
/*  policy 3  threshold on the per-position confidence: L_b grows from L_min  */
/*            while c_{b,L_b} > threshold (the leading run).                  */
/* Theta is reported for the chosen lengths in every policy.  min_margin is   */
/* the smallest relative gap on which a decision turned: policy 1, the best  */
/* Theta against the runner-up; policies 2-3, |value - threshold| / threshold. */
/* The lag itself is the caller's: the confidences passed in are the ones     */
/* the policy is applied to.                                                  */
/* ------------------------------------------------------------------------ */
int or_schedule_policy(const double *conf_logits, const double *pos_temp, const double *sps, int sps_len,
                       int B, int G, int L_min, int L_max, int policy, double threshold,
                       double *conf, double *cum_conf, int32_t *verify_len, double *theta,
                       int32_t *n_admitted, double *min_margin, double *min_tie)
{
    if (policy == 0)
        return or_schedule(conf_logits, pos_temp, sps, sps_len, B, G, L_min, L_max, conf, cum_conf, verify_len,
                           theta, n_admitted, min_margin, min_tie);
    if (policy < 1 || policy > 3) return -1;
    if (B < 0 || G < 1 || L_min < 0 || L_min > L_max || L_max > G) return -1;
    if (sps_len < B * (L_max + 1) + 1) return -1;
    for (int b = 0; b < B; ++b) {
        double prod = 1.0;
        for (int j = 0; j < G; ++j) {
            double l = conf_logits[(size_t)b * G + j];
            double c = 1.0 / (1.0 + exp(-l / pos_temp[j]));
            prod *= c;
            conf[(size_t)b * G + j] = c;
            cum_conf[(size_t)b * G + j] = prod;
        }
    }
    double mm = INFINITY, mt = INFINITY;
    int admitted = 0;
    if (policy == 1) {
        double tau = 0.0;
        long btok = 0;
        for (int b = 0; b < B; ++b) {
            verify_len[b] = L_min;
            double t = 1.0;
            for (int j = 0; j < L_min; ++j) t += cum_conf[(size_t)b * G + j];
            tau += t;
            btok += L_min + 1;
        }
        int nc = B * (L_max - L_min);
        or_cand *cand = (or_cand *)malloc(sizeof(or_cand) * (size_t)(nc > 0 ? nc : 1));
        if (!cand) return -2;
        int n = 0;
        for (int b = 0; b < B; ++b)
            for (int j = L_min; j < L_max; ++j) {
                cand[n].a = cum_conf[(size_t)b * G + j];
                cand[n].j = j;
                cand[n].b = b;
                ++n;
            }
        qsort(cand, (size_t)nc, sizeof(or_cand), cand_order);
        for (int i = 0; i + 1 < nc; ++i) {
            double d = fabs(cand[i].a - cand[i + 1].a) / fmax(fabs(cand[i].a), 1e-300);
            if (d < mt) mt = d;
        }
        /* Theta after admitting the first n candidates, n = 0..nc */
        double best = tau * sps[btok], second = -INFINITY, run = tau;
        int nbest = 0;
        for (int i = 0; i < nc; ++i) {
            run += cand[i].a;
            double th = run * sps[btok + i + 1];
            if (th > best) {
                second = best;
                best = th;
                nbest = i + 1;
            } else if (th > second) {
                second = th;
            }
        }
        for (int i = 0; i < nbest; ++i) verify_len[cand[i].b] = cand[i].j + 1;
        admitted = nbest;
        if (second > -INFINITY) mm = fabs(best - second) / fmax(fabs(best), 1e-300);
        free(cand);
    } else {
        for (int b = 0; b < B; ++b) {
            int L = L_min;
            for (int j = L_min; j < L_max; ++j) {
                double x = (policy == 2) ? cum_conf[(size_t)b * G + j] : conf[(size_t)b * G + j];
                double d = fabs(x - threshold) / fmax(fabs(threshold), 1e-300);
                if (d < mm) mm = d;
                if (!(x > threshold)) break;
                L = j + 1;
            }
            verify_len[b] = L;
            admitted += L - L_min;
        }
    }
    /* Theta of the chosen lengths */
    double tau = 0.0;
    long btok = 0;
    for (int b = 0; b < B; ++b) {
        double t = 1.0;
        for (int j = 0; j < verify_len[b]; ++j) t += cum_conf[(size_t)b * G + j];
        tau += t;
        btok += verify_len[b] + 1;
    }
    if (theta) *theta = tau * sps[btok];
    if (n_admitted) *n_admitted = admitted;
    if (min_margin) *min_margin = mm;
    if (min_tie) *min_tie = mt;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Verification by rejection sampling ([MATH-FR] "La garantie de            */
/* l'echantillonnage par rejet": accept x with probability min(1, p/q), stop */
/* at the first rejection and resample from the residual distribution;       */
/* [DSP-ZH] "DSpark 是什么？": append a bonus token when the whole block is   */
/* accepted), readings R5 and R6; the residual, fallback and bonus draws    */
/* are Gumbel-max draws on streams 2, 2 and 3.                               */
/*                                                                           */
/* target [B][G+1][V]: row j is the target's logits for draft position j,    */
/* row L_b gives the bonus.  The draft side is recomputed here from U, E_in, */
/* W_out, anchor and the draft tokens.  verify_len [B] (NULL = G).           */
/* Outputs: accept_len [B], out_tokens [B][G+1] (-1 padded), num_out [B],    */
/* target_lse [B][G+1] (NaN where not read; T = 0: max t), logp / logq       */
/* [B][G] (NaN where not tested), accept_margin [B][G] = |u - min(1, p/q)|   */
/* (NaN where not tested), final_gap / final_top [B] for the last draw (the  */
/* two largest Gumbel keys' gap and the largest; greedy: of the logits),     */
/* final_kind [B] = 0 bonus, 1 residual, 2 residual fell back to p,          */
/* 3 greedy correction.  Returns 0, -1 on invalid input.                     */
/* ------------------------------------------------------------------------ */
int or_verify(const double *target, const double *U, const double *E_in, const double *W_out,
              const int32_t *anchor, const int32_t *draft_tokens, const int32_t *verify_len,
              const double *temp, const uint32_t *rid,
              int B, int G, int V, int r, uint64_t seed,
              int32_t *accept_len, int32_t *out_tokens, int32_t *num_out,
              double *target_lse, double *logp, double *logq, double *accept_margin,
              double *final_gap, double *final_top, int32_t *final_kind)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    double *s = (double *)malloc(sizeof(double) * (size_t)V);
    double *st = (double *)malloc(sizeof(double) * (size_t)V);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    unsigned char *allowed = (unsigned char *)malloc((size_t)V);
    if (!z || !s || !st || !w || !allowed) {
        free(z); free(s); free(st); free(w); free(allowed);
        return -2;
    }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        uint32_t id = rid ? rid[b] : (uint32_t)b;
        double T = temp[b];
        int L = verify_len ? verify_len[b] : G;
        if (L < 0 || L > G || anchor[b] < 0 || anchor[b] >= V) { rc = -1; break; }
        for (int j = 0; j < G; ++j) {
            size_t o = (size_t)b * G + j;
            logp[o] = NAN; logq[o] = NAN; accept_margin[o] = NAN;
        }
        for (int j = 0; j <= G; ++j) target_lse[(size_t)b * (G + 1) + j] = NAN;
        for (int j = 0; j <= G; ++j) out_tokens[(size_t)b * (G + 1) + j] = -1;
        for (int j = 0; j < L; ++j) {
            int x = draft_tokens[(size_t)b * G + j];
            if (x < 0 || x >= V) { rc = -1; break; }
        }
        if (rc) break;

        int k = 0;         /* number of accepted draft tokens */
        int y = -1;        /* the final (resampled or bonus) token */
        int kind = 0;
        double fgap = NAN, ftop = NAN;
        for (int j = 0; j < L; ++j) {
            const double *t_row = target + ((size_t)b * (G + 1) + j) * (size_t)V;
            int x = draft_tokens[(size_t)b * G + j];
            size_t o = (size_t)b * G + j;
            if (T > 0.0) {
                for (int v = 0; v < V; ++v) st[v] = t_row[v] / T;
                double lt = row_logsumexp(st, V);
                target_lse[(size_t)b * (G + 1) + j] = lt;
                int prev = (j == 0) ? anchor[b] : draft_tokens[(size_t)b * G + j - 1];
                markov_logits(U + o * (size_t)V, E_in, W_out, prev, V, r, z);
                for (int v = 0; v < V; ++v) s[v] = z[v] / T;
                double lq = row_logsumexp(s, V);
                double lp_x = st[x] - lt;
                double lq_x = s[x] - lq;
                logp[o] = lp_x;
                logq[o] = lq_x;
                double u = or_uniform(seed, id, (uint32_t)j, 0u, 1u);
                double ratio = exp(lp_x - lq_x);
                double thr = ratio < 1.0 ? ratio : 1.0;
                accept_margin[o] = fabs(u - thr);
                if (u < thr) { ++k; continue; }
                /* rejected at j: residual max(0, p - q), R6 */
                int any = 0;
                for (int v = 0; v < V; ++v) {
                    double pv = exp(st[v] - lt), qv = exp(s[v] - lq);
                    allowed[v] = (unsigned char)(pv > qv);
                    w[v] = allowed[v] ? log(pv - qv) : -INFINITY;
                    any |= allowed[v];
                }
                if (any) {
                    y = gumbel_max(w, V, seed, id, (uint32_t)j, 2u, &fgap, &ftop);
                    kind = 1;
                } else {
                    y = gumbel_max(st, V, seed, id, (uint32_t)j, 2u, &fgap, &ftop);
                    kind = 2;
                }
                break;
            } else {
                double gap, top;
                int a = row_argmax(t_row, V, &gap, &top);
                target_lse[(size_t)b * (G + 1) + j] = top;
                logp[o] = (a == x) ? 0.0 : -INFINITY;
                logq[o] = 0.0;
                if (a == x) { ++k; continue; }
                y = a; kind = 3; fgap = gap; ftop = top;
                break;
            }
        }
        if (y < 0) {
            /* all L draft tokens accepted: bonus token from row L */
            const double *t_row = target + ((size_t)b * (G + 1) + L) * (size_t)V;
            if (T > 0.0) {
                for (int v = 0; v < V; ++v) st[v] = t_row[v] / T;
                y = gumbel_max(st, V, seed, id, (uint32_t)L, 3u, &fgap, &ftop);
            } else {
                double top;
                y = row_argmax(t_row, V, &fgap, &top);
                ftop = top;
                target_lse[(size_t)b * (G + 1) + L] = top;
            }
            kind = 0;
        }
        accept_len[b] = k;
        for (int j = 0; j < k; ++j) out_tokens[(size_t)b * (G + 1) + j] = draft_tokens[(size_t)b * G + j];
        out_tokens[(size_t)b * (G + 1) + k] = y;
        num_out[b] = k + 1;
        final_gap[b] = fgap;
        final_top[b] = ftop;
        final_kind[b] = kind;
    }
    free(z); free(s); free(st); free(w); free(allowed);
    return rc;
}
