/*
 * moe_oracle.c -- plain, slow, fp64 CPU definition of one sparse MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library.  It shares
 * no code, header, table or constant with the CUDA library; neither includes
 * or loads the other.
 *
 * Sources (the four web pages this layer is specified by):
 *   [LLaMA4-MoE]  "Hand-building a LLaMA4-MoE" guide (nxmr.cn/news/140631)
 *   [ZeRO3-MoE]   "DeepSpeed ZeRO-3 and MoE memory accounting" guide
 *                 (nlpx.cn/news/237350)
 *   [Twinkle]     "Twinkle adapts DeepSeek-V4 training" notes (wmrh.cn/news/44033)
 *
 * Every step is written as the plain definition, token by token, in the
 * order the pages state the layer; no blocking, fusion or reordering.
 * OpenMP is used only on loops whose iterations are independent (each
 * writes its own output rows), so results do not depend on thread count.
 *
 * Readings taken where the pages are silent or inconsistent:
 *   - top-k is taken on the logits (softmax is monotone), ties broken by the
 *     lowest expert id; a NaN logit ranks below every number.
 *   - gates are the softmax over the k selected logits (they sum to 1 before
 *     capacity drops); normalize_gates = 0 keeps the raw softmax probability.
 *   - capacity C = ceil(capacity_factor * T * k / E) evaluated in IEEE double
 *     from the given (fp32) factor, clamped to T; assignments are kept in
 *     ascending token order while an expert has fewer than C kept.
 *   - dropped slots contribute nothing; surviving gates are not renormalised.
 *   - aux loss = lambda * sum_i (pbar_i - 1/E)^2 with pbar the mean softmax
 *     probability (the [ZeRO3-MoE] §3.2 form, its 1/k read as 1/E).
 *   - each expert is a two-layer FFN without biases: SiLU-MLP, or SwiGLU.
 */
#include <math.h>
#include <omp.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int T, d, f, E, k;
    double capacity_factor; /* <= 0 : no capacity limit */
    int swiglu;             /* 0: y = Wd^T silu(Wu^T x); 1: y = Wd^T (silu(Wg^T x) * Wu^T x) */
    int normalize_gates;    /* 1: softmax over the k selected logits; 0: raw probabilities */
    double aux_coef;        /* lambda of the variance-form aux loss */
    int pad_m;              /* segment padding of the expert-contiguous layout (>= 1) */
    double temperature;     /* softmax temperature tau (<= 0 means 1) */
    int straight_through;   /* 1: select on logits + noise, gates 1, gradient through
                               softmax(logits / tau) (Gumbel top-k, straight-through) */
    int f_shared;           /* hidden width of the shared experts' FFN (0: none) */
} oracle_cfg;

static double tau_of(const oracle_cfg* c) { return c->temperature > 0.0 ? c->temperature : 1.0; }

/* Layout of the statistics vector written by oracle_stats (length 9 + E). */
enum {
    OST_AUX_LOSS = 0,   /* lambda * sum_i (pbar_i - 1/E)^2                         */
    OST_AUX_SWITCH = 1, /* E * sum_i f_i pbar_i, f_i = counts_i / (T k)             */
    OST_ENTROPY = 2,    /* mean over tokens of -sum_e p log p                      */
    OST_NONFINITE = 3,  /* number of tokens with a non-finite logit                */
    OST_DROPPED = 4,    /* assignments dropped by the capacity limit               */
    OST_MAX_OVER_MEAN_KEPT = 5, /* max_e kept_e / mean_e kept_e                   */
    OST_COUNT_CV = 6,   /* std/mean of counts over experts                         */
    OST_MAX_OVER_MEAN_COUNT = 7,
    OST_TOKENS = 8,     /* tokens that take part in routing (not masked)           */
    OST_PBAR = 9        /* pbar[0..E), mean over those tokens                      */
};

static double silu(double z) { return z / (1.0 + exp(-z)); }
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }
/* d/dz silu(z) = s(z) (1 + z (1 - s(z))) */
static double dsilu(double z) { double s = sigmoid(z); return s * (1.0 + z * (1.0 - s)); }

/* ---- Step 1: router logits  [LLaMA4-MoE] §2.4; noise [LLaMA4-MoE] §3.2 ----
 * logits[t,e] = sum_i x[t,i] W_r[i,e] + b[e] + noise[t,e]                      */
void oracle_router_logits(const oracle_cfg* c, const double* x, const double* Wr,
                          const double* bias, const double* noise, double* logits)
{
    const int T = c->T, d = c->d, E = c->E;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += x[(size_t)t * d + i] * Wr[(size_t)i * E + e];
            if (bias) s += bias[e];
            if (noise) s += noise[(size_t)t * E + e];
            logits[(size_t)t * E + e] = s;
        }
    }
}

/* a ranks above b in the top-k order: larger logit, NaN lowest, then lower id */
static int ranks_above(double la, int a, double lb, int b)
{
    int na = isnan(la), nb = isnan(lb);
    if (na != nb) return nb;          /* the number ranks above the NaN */
    if (!na && la != lb) return la > lb;
    return a < b;
}

/* ---- Steps 2-4: softmax, top-k, gates  [LLaMA4-MoE] §2.4; [Twinkle] §3.1 ----
 * probs  [T,E] softmax of logits / tau (max subtracted)   [Twinkle] §3.1, [ZeRO3-MoE] §3.2
 * topk   [T,k] experts in rank order; gate [T,k]; counts [E] selections.
 * noise_sel (straight-through mode only, may be NULL): selection key =
 *   logits + noise, summed in fp32 (the precision the kernel decides in);
 *   gates are 1 ([Twinkle] §3.1, Gumbel top-k with straight-through).
 * mask (may be NULL): tokens with mask 0 are padding and take no part in
 *   routing ([LLaMA4-MoE] §4.1): topk -1, gates 0, probs 0.
 * Returns the number of routed tokens that had a non-finite logit.            */
int oracle_route(const oracle_cfg* c, const double* logits, const double* noise_sel,
                 const unsigned char* mask, double* probs, int* topk, double* gate, int* counts)
{
    const int T = c->T, E = c->E, k = c->k;
    const double tau = tau_of(c);
    double* key = (double*)malloc(sizeof(double) * (size_t)E);
    int nonfinite = 0;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int t = 0; t < T; ++t) {
        const double* l = logits + (size_t)t * E;
        int* sel = topk + (size_t)t * k;
        double* g = gate + (size_t)t * k;
        if (mask && !mask[t]) {
            for (int e = 0; e < E; ++e) probs[(size_t)t * E + e] = 0.0;
            for (int j = 0; j < k; ++j) { sel[j] = -1; g[j] = 0.0; }
            continue;
        }
        double m = -INFINITY;
        int bad = 0;
        for (int e = 0; e < E; ++e) {
            if (!isfinite(l[e])) bad = 1;
            if (l[e] > m) m = l[e];
            key[e] = l[e];
            if (c->straight_through && noise_sel)
                key[e] = (double)((float)l[e] + (float)noise_sel[(size_t)t * E + e]);
        }
        nonfinite += bad;
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp((l[e] - m) / tau);
        for (int e = 0; e < E; ++e) probs[(size_t)t * E + e] = exp((l[e] - m) / tau) / z;

        /* selection: k passes, each taking the best expert not yet taken */
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                int taken = 0;
                for (int q = 0; q < j; ++q) taken |= (sel[q] == e);
                if (taken) continue;
                if (best < 0 || ranks_above(key[e], e, key[best], best)) best = e;
            }
            sel[j] = best;
            counts[best] += 1;
        }
        /* gates: 1 (straight-through), softmax over the selected, or raw probs */
        if (c->straight_through) {
            for (int j = 0; j < k; ++j) g[j] = 1.0;
        } else if (c->normalize_gates) {
            double ms = l[sel[0]], zs = 0.0;
            for (int j = 0; j < k; ++j) ms = l[sel[j]] > ms ? l[sel[j]] : ms;
            for (int j = 0; j < k; ++j) zs += exp((l[sel[j]] - ms) / tau);
            for (int j = 0; j < k; ++j) g[j] = exp((l[sel[j]] - ms) / tau) / zs;
        } else {
            for (int j = 0; j < k; ++j) g[j] = probs[(size_t)t * E + sel[j]];
        }
    }
    free(key);
    return nonfinite;
}

/* ---- Capacity C  [ZeRO3-MoE] §3.1, §3.4 (capacity_factor 1.2) ---- */
int oracle_capacity(const oracle_cfg* c)
{
    if (!(c->capacity_factor > 0.0)) return c->T; /* no limit: an expert sees each token once at most */
    double v = ceil(c->capacity_factor * (double)c->T * (double)c->k / (double)c->E);
    if (v > (double)c->T) v = (double)c->T;
    return (int)v;
}

/* ---- Steps 5-6: capacity dropping and the expert-contiguous permutation ----
 * Sort-by-expert then split into per-expert intervals  [LLaMA4-MoE] §2.4.
 * kept[E]; offsets[E+1] (segment e = rows offsets[e] .. offsets[e+1], its
 * length kept[e] rounded up to pad_m); perm_token[rows] (-1 on padding rows);
 * slot_of[T,k] (row of assignment (t,j), or -1 when dropped).
 * perm_token must hold offsets[E] entries (at most T*k + E*(pad_m-1)).       */
void oracle_permute(const oracle_cfg* c, const int* topk, int* kept, int* offsets,
                    int* perm_token, int* slot_of)
{
    const int T = c->T, E = c->E, k = c->k, pm = c->pad_m;
    const int C = oracle_capacity(c);
    int* taken = (int*)calloc((size_t)E, sizeof(int));
    int* rank = (int*)malloc(sizeof(int) * (size_t)T * k);
    /* walk tokens in order; keep while the expert has room */
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = topk[(size_t)t * k + j];
            if (e < 0) { rank[(size_t)t * k + j] = -1; continue; }   /* masked token */
            if (taken[e] < C) { rank[(size_t)t * k + j] = taken[e]; taken[e]++; }
            else rank[(size_t)t * k + j] = -1;
        }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        kept[e] = taken[e];
        int padded = (kept[e] + pm - 1) / pm * pm;
        offsets[e + 1] = offsets[e] + padded;
    }
    for (int r = 0; r < offsets[E]; ++r) perm_token[r] = -1;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = topk[(size_t)t * k + j];
            int q = rank[(size_t)t * k + j];
            if (e < 0 || q < 0) { slot_of[(size_t)t * k + j] = -1; continue; }
            slot_of[(size_t)t * k + j] = offsets[e] + q;
            perm_token[offsets[e] + q] = t;
        }
    free(taken);
    free(rank);
}

/* ---- Step 7: one expert FFN on one token  [LLaMA4-MoE] §2.4 ("two-layer FFN") ----
 * SiLU-MLP : h = Wu^T x, a = silu(h), y = Wd^T a
 * SwiGLU   : g = Wg^T x, u = Wu^T x, a = silu(g) * u, y = Wd^T a
 * Wu, Wg point at expert e's [d,f] block, Wd at its [f,d] block.
 * h_out receives h (SiLU) or g (SwiGLU); u_out receives u (SwiGLU only).    */
static void expert_ffn(const oracle_cfg* c, int f, const double* x, const double* Wu,
                       const double* Wg, const double* Wd, double* h_out,
                       double* u_out, double* a_out, double* y)
{
    const int d = c->d;
    for (int j = 0; j < f; ++j) { h_out[j] = 0.0; if (c->swiglu) u_out[j] = 0.0; }
    for (int i = 0; i < d; ++i) {
        const double xi = x[i];
        const double* wu = Wu + (size_t)i * f;
        if (c->swiglu) {
            const double* wg = Wg + (size_t)i * f;
            for (int j = 0; j < f; ++j) { h_out[j] += xi * wg[j]; u_out[j] += xi * wu[j]; }
        } else {
            for (int j = 0; j < f; ++j) h_out[j] += xi * wu[j];
        }
    }
    for (int j = 0; j < f; ++j) a_out[j] = c->swiglu ? silu(h_out[j]) * u_out[j] : silu(h_out[j]);
    for (int i = 0; i < d; ++i) y[i] = 0.0;
    for (int j = 0; j < f; ++j) {
        const double aj = a_out[j];
        const double* wd = Wd + (size_t)j * d;
        for (int i = 0; i < d; ++i) y[i] += aj * wd[i];
    }
}

/* One expert on one token with its intermediates: h (SiLU: W_up^T x; SwiGLU:
 * g = W_gate^T x), u (SwiGLU only; may be NULL), act, y.                      */
void oracle_expert_forward(const oracle_cfg* c, int e, const double* x, const double* Wup,
                           const double* Wgate, const double* Wdown, double* h, double* u,
                           double* act, double* y)
{
    const size_t df = (size_t)c->d * c->f;
    double* tmp = NULL;
    if (c->swiglu && !u) u = tmp = (double*)malloc(sizeof(double) * (size_t)c->f);
    expert_ffn(c, c->f, x, Wup + e * df, c->swiglu ? Wgate + e * df : NULL, Wdown + e * df, h, u,
               act, y);
    free(tmp);
}

/* One expert's FFN output on one token (for sampled checks and special cases). */
void oracle_expert_apply(const oracle_cfg* c, int e, const double* x, const double* Wup,
                         const double* Wgate, const double* Wdown, double* y)
{
    const size_t df = (size_t)c->d * c->f;
    double* h = (double*)malloc(sizeof(double) * 3 * (size_t)c->f);
    expert_ffn(c, c->f, x, Wup + e * df, c->swiglu ? Wgate + e * df : NULL, Wdown + e * df,
               h, h + c->f, h + 2 * (size_t)c->f, y);
    free(h);
}

/* ---- Step 8: gate-weighted combine  [LLaMA4-MoE] §2.4 ----
 * out[t] = sum over kept slots j (ascending) of gate[t,j] * FFN_{e_j}(x_t);
 * a token whose slots were all dropped outputs zeros.                         */
void oracle_combine(const oracle_cfg* c, const double* x, const int* topk,
                    const double* gate, const int* slot_of, const double* Wup,
                    const double* Wgate, const double* Wdown, double* out)
{
    const int T = c->T, d = c->d, f = c->f, k = c->k;
    const size_t df = (size_t)d * f;
#pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * (3 * (size_t)f + d));
        double* y = h + 3 * (size_t)f;
#pragma omp for schedule(dynamic, 4)
        for (int t = 0; t < T; ++t) {
            double* o = out + (size_t)t * d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            for (int j = 0; j < k; ++j) {
                if (slot_of[(size_t)t * k + j] < 0) continue;
                int e = topk[(size_t)t * k + j];
                expert_ffn(c, f, x + (size_t)t * d, Wup + e * df, c->swiglu ? Wgate + e * df : NULL,
                           Wdown + e * df, h, h + f, h + 2 * (size_t)f, y);
                const double g = gate[(size_t)t * k + j];
                for (int i = 0; i < d; ++i) o[i] += g * y[i];
            }
        }
        free(h);
    }
}

/* ---- Shared experts  [LLaMA4-MoE] §5.2 ----
 * A fixed set of experts joins every token's computation.  They form one
 * dense FFN of hidden width f_shared (several shared experts of width f_e are
 * the same FFN with their weight blocks side by side, f_shared = n f_e), of
 * the routed experts' kind (SiLU-MLP or SwiGLU), added with weight 1:
 *   out[t] += FFN_shared(x_t)   for every token, masked or not.
 * Wup_s, Wgate_s [d, f_shared], Wdown_s [f_shared, d].                        */
void oracle_shared_forward(const oracle_cfg* c, const double* x, const double* Wup_s,
                           const double* Wgate_s, const double* Wdown_s, double* h, double* u,
                           double* act, double* y)
{
    double* tmp = NULL;
    if (c->swiglu && !u) u = tmp = (double*)malloc(sizeof(double) * (size_t)c->f_shared);
    expert_ffn(c, c->f_shared, x, Wup_s, c->swiglu ? Wgate_s : NULL, Wdown_s, h, u, act, y);
    free(tmp);
}

void oracle_shared_add(const oracle_cfg* c, const double* x, const double* Wup_s,
                       const double* Wgate_s, const double* Wdown_s, double* out)
{
    const int T = c->T, d = c->d, fs = c->f_shared;
#pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * (3 * (size_t)fs + d));
        double* y = h + 3 * (size_t)fs;
#pragma omp for schedule(dynamic, 4)
        for (int t = 0; t < T; ++t) {
            expert_ffn(c, fs, x + (size_t)t * d, Wup_s, c->swiglu ? Wgate_s : NULL, Wdown_s, h,
                       h + fs, h + 2 * (size_t)fs, y);
            double* o = out + (size_t)t * d;
            for (int i = 0; i < d; ++i) o[i] += y[i];
        }
        free(h);
    }
}

/* ---- Step 9: aux statistics  [ZeRO3-MoE] §3.2; [LLaMA4-MoE] §3.2, §3.3 ----
 * Means run over the routed tokens (those with topk[t][0] >= 0).
 * stats has 9 + E entries (layout OST_*).                                     */
void oracle_stats(const oracle_cfg* c, const double* probs, const int* topk, const int* counts,
                  const int* kept, int nonfinite, double* stats)
{
    const int T = c->T, E = c->E, k = c->k;
    double* pbar = stats + OST_PBAR;
    for (int e = 0; e < E; ++e) pbar[e] = 0.0;
    double ent = 0.0;
    int real = 0;
    for (int t = 0; t < T; ++t) {
        if (topk[(size_t)t * k] < 0) continue;
        ++real;
        double h = 0.0;
        for (int e = 0; e < E; ++e) {
            double p = probs[(size_t)t * E + e];
            pbar[e] += p;
            if (p > 0.0) h -= p * log(p);
        }
        ent += h;
    }
    const double Tr = real > 0 ? (double)real : 1.0;
    double aux = 0.0, sw = 0.0;
    for (int e = 0; e < E; ++e) {
        pbar[e] /= Tr;
        aux += (pbar[e] - 1.0 / E) * (pbar[e] - 1.0 / E);
        sw += ((double)counts[e] / (Tr * k)) * pbar[e];
    }
    stats[OST_AUX_LOSS] = c->aux_coef * aux;
    stats[OST_AUX_SWITCH] = (double)E * sw;
    stats[OST_ENTROPY] = ent / Tr;
    stats[OST_NONFINITE] = (double)nonfinite;
    stats[OST_TOKENS] = (double)real;
    long dropped = 0, kmax = 0, ksum = 0, cmax = 0, csum = 0;
    for (int e = 0; e < E; ++e) {
        dropped += counts[e] - kept[e];
        if (kept[e] > kmax) kmax = kept[e];
        ksum += kept[e];
        if (counts[e] > cmax) cmax = counts[e];
        csum += counts[e];
    }
    double cmean = (double)csum / E, var = 0.0;
    for (int e = 0; e < E; ++e) var += (counts[e] - cmean) * (counts[e] - cmean);
    stats[OST_DROPPED] = (double)dropped;
    stats[OST_MAX_OVER_MEAN_KEPT] = ksum > 0 ? (double)kmax / ((double)ksum / E) : 0.0;
    stats[OST_COUNT_CV] = cmean > 0 ? sqrt(var / E) / cmean : 0.0;
    stats[OST_MAX_OVER_MEAN_COUNT] = cmean > 0 ? (double)cmax / cmean : 0.0;
}

/* ---- Whole forward: steps 1-9.  If logits_in is given, step 1 is skipped and
 * those logits are routed instead (the "conditioned" oracle).  Gate noise is
 * added to the logits, except in straight-through mode, where it only enters
 * the selection key.  mask may be NULL.                                       */
void oracle_forward(const oracle_cfg* c, const double* x, const double* Wr, const double* bias,
                    const double* noise, const unsigned char* mask, const double* Wup,
                    const double* Wgate, const double* Wdown, const double* logits_in,
                    double* logits, double* probs, int* topk, double* gate, int* counts,
                    int* kept, int* offsets, int* perm_token, int* slot_of,
                    double* out, double* stats,
                    const double* Wup_s, const double* Wgate_s, const double* Wdown_s)
{
    if (logits_in) memcpy(logits, logits_in, sizeof(double) * (size_t)c->T * c->E);
    else oracle_router_logits(c, x, Wr, bias, c->straight_through ? NULL : noise, logits);
    int nf = oracle_route(c, logits, c->straight_through ? noise : NULL, mask, probs, topk, gate,
                          counts);
    oracle_permute(c, topk, kept, offsets, perm_token, slot_of);
    oracle_combine(c, x, topk, gate, slot_of, Wup, Wgate, Wdown, out);
    if (c->f_shared > 0) oracle_shared_add(c, x, Wup_s, Wgate_s, Wdown_s, out);
    oracle_stats(c, probs, topk, counts, kept, nf, stats);
}

/* Backward of one FFN application y = FFN(x_t) of width f, given its forward
 * intermediates h (SwiGLU: g), u (SwiGLU) and a, and dy = dL/dy:
 *   da = Wd dy; dWd += a dy^T;
 *   SiLU:   dh = da * silu'(h);                    dWu += x dh^T;  dx = Wu dh
 *   SwiGLU: du = da * silu(g), dg = da * u * silu'(g);
 *           dWu += x du^T, dWg += x dg^T;           dx = Wu du + Wg dg
 * dx is written; dh_out (nh*f: dh, or dg then du) is written when not NULL.
 * scratch holds 3f doubles.                                                   */
static void ffn_token_backward(const oracle_cfg* c, int f, const double* xt, const double* h,
                               const double* u, const double* a, const double* Wu,
                               const double* Wg, const double* Wd, const double* dy,
                               double* dWu, double* dWg, double* dWd, double* dx,
                               double* dh_out, double* scratch)
{
    const int d = c->d;
    double *da = scratch, *dh = scratch + f, *du = scratch + 2 * (size_t)f;
    /* y = Wd^T a */
    for (int q = 0; q < f; ++q) {
        const double* wd = Wd + (size_t)q * d;
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += wd[i] * dy[i];
        da[q] = acc;
        double* gw = dWd + (size_t)q * d;
        for (int i = 0; i < d; ++i) gw[i] += a[q] * dy[i];
    }
    /* activation */
    for (int q = 0; q < f; ++q) {
        if (c->swiglu) {
            du[q] = da[q] * silu(h[q]);          /* d/du (silu(g) u) */
            dh[q] = da[q] * u[q] * dsilu(h[q]);  /* d/dg             */
        } else {
            dh[q] = da[q] * dsilu(h[q]);
        }
    }
    if (dh_out)
        for (int q = 0; q < f; ++q) {
            dh_out[q] = dh[q];
            if (c->swiglu) dh_out[f + q] = du[q];
        }
    /* h = Wu^T x (SiLU) ; g = Wg^T x, u = Wu^T x (SwiGLU) */
    for (int i = 0; i < d; ++i) {
        const double xi = xt[i];
        double acc = 0.0;
        double* gu = dWu + (size_t)i * f;
        const double* wu = Wu + (size_t)i * f;
        if (c->swiglu) {
            double* gg = dWg + (size_t)i * f;
            const double* wg = Wg + (size_t)i * f;
            for (int q = 0; q < f; ++q) {
                gu[q] += xi * du[q];
                gg[q] += xi * dh[q];
                acc += wu[q] * du[q] + wg[q] * dh[q];
            }
        } else {
            for (int q = 0; q < f; ++q) { gu[q] += xi * dh[q]; acc += wu[q] * dh[q]; }
        }
        dx[i] = acc;
    }
}

/* ---- Step 10: backward of L = <dout, out> + aux loss ----
 * Gradients flow through the gate weights into the router; the selection
 * itself is piecewise constant  ([LLaMA4-MoE] §2.4: do not detach the
 * routing weights).  Outputs are written, not accumulated.
 * dx[T,d], dWr[d,E], db[E] (may be NULL), dWup/dWgate[E,d,f], dWdown[E,f,d],
 * dgate[T,k] and dlogits[T,E] (both may be NULL).  Optional per-slot views of
 * the expert path (NULL = not wanted): dh_slot[T,k,nh,f] holds dh (SiLU) or
 * dg then du (SwiGLU); dxp_slot[T,k,d] holds the slot's dx contribution.
 * pbar_in (E) and T_aux: when the T tokens given are a sample of a larger batch,
 * the aux-loss term uses that batch's mean probabilities and token count (NULL /
 * 0: computed from the tokens given).                                          */
void oracle_backward(const oracle_cfg* c, const double* x, const double* Wr,
                     const double* Wup, const double* Wgate, const double* Wdown,
                     const double* logits, const int* topk, const double* gate,
                     const int* slot_of, const double* dout,
                     double* dx, double* dWr, double* db, double* dWup, double* dWgate,
                     double* dWdown, double* dgate_out, double* dlogits_out,
                     double* dh_slot_out, double* dxp_slot_out,
                     const double* pbar_in, int T_aux,
                     const double* Wup_s, const double* Wgate_s, const double* Wdown_s,
                     double* dWup_s, double* dWgate_s, double* dWdown_s)
{
    const int T = c->T, d = c->d, f = c->f, E = c->E, k = c->k;
    const size_t df = (size_t)d * f;
    double* dgate = (double*)calloc((size_t)T * k, sizeof(double));
    double* dxp = (double*)calloc((size_t)T * k * d, sizeof(double)); /* per-slot dx */
    memset(dWup, 0, sizeof(double) * E * df);
    memset(dWdown, 0, sizeof(double) * E * df);
    if (c->swiglu) memset(dWgate, 0, sizeof(double) * E * df);

    /* expert FFN backward, expert by expert, tokens ascending (each expert's
     * weight gradients are its own; per-slot dx rows are disjoint)            */
#pragma omp parallel for schedule(dynamic, 1)
    for (int e = 0; e < E; ++e) {
        double* h = (double*)malloc(sizeof(double) * (6 * (size_t)f + 2 * (size_t)d));
        double *u = h + f, *a = h + 2 * (size_t)f, *tmp = h + 3 * (size_t)f;
        double *y = h + 6 * (size_t)f, *dy = y + d;
        const double* Wu = Wup + e * df;
        const double* Wg = c->swiglu ? Wgate + e * df : NULL;
        const double* Wd = Wdown + e * df;
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j) {
                if (topk[(size_t)t * k + j] != e || slot_of[(size_t)t * k + j] < 0) continue;  /* not e, dropped or masked */
                const double* xt = x + (size_t)t * d;
                const double* go = dout + (size_t)t * d;
                expert_ffn(c, f, xt, Wu, Wg, Wd, h, u, a, y);
                /* out += gate * y  =>  dgate = <dout, y>, dy = gate * dout */
                double s = 0.0;
                for (int i = 0; i < d; ++i) s += go[i] * y[i];
                dgate[(size_t)t * k + j] = s;
                const double gt = gate[(size_t)t * k + j];
                for (int i = 0; i < d; ++i) dy[i] = gt * go[i];
                ffn_token_backward(c, f, xt, h, u, a, Wu, Wg, Wd, dy, dWup + e * df,
                                   c->swiglu ? dWgate + e * df : NULL, dWdown + e * df,
                                   dxp + ((size_t)t * k + j) * d,
                                   dh_slot_out ? dh_slot_out + ((size_t)t * k + j) * (c->swiglu ? 2 : 1) * f
                                               : NULL,
                                   tmp);
            }
        free(h);
    }

    /* shared experts ([LLaMA4-MoE] §5.2): out[t] += FFN_shared(x_t) on every
     * token, weight 1, so dy = dout[t]; their input gradient joins dx below.  */
    double* dxs = NULL;
    if (c->f_shared > 0) {
        const int fs = c->f_shared;
        const size_t dfs = (size_t)d * fs;
        memset(dWup_s, 0, sizeof(double) * dfs);
        memset(dWdown_s, 0, sizeof(double) * dfs);
        if (c->swiglu) memset(dWgate_s, 0, sizeof(double) * dfs);
        dxs = (double*)calloc((size_t)T * d, sizeof(double));
        /* the weight gradients sum over all tokens: run tokens in order, one thread */
        double* h = (double*)malloc(sizeof(double) * (6 * (size_t)fs + (size_t)d));
        double *u = h + fs, *a = h + 2 * (size_t)fs, *tmp = h + 3 * (size_t)fs;
        double* y = h + 6 * (size_t)fs;
        for (int t = 0; t < T; ++t) {
            const double* xt = x + (size_t)t * d;
            expert_ffn(c, fs, xt, Wup_s, c->swiglu ? Wgate_s : NULL, Wdown_s, h, u, a, y);
            ffn_token_backward(c, fs, xt, h, u, a, Wup_s, c->swiglu ? Wgate_s : NULL, Wdown_s,
                               dout + (size_t)t * d, dWup_s, c->swiglu ? dWgate_s : NULL,
                               dWdown_s, dxs + (size_t)t * d, NULL, tmp);
        }
        free(h);
    }

    /* router: dL/dlogits from the gates and from the aux loss.  p = softmax(l/tau)
     * over the routed tokens; every derivative through it carries 1/tau.      */
    const double tau = tau_of(c);
    double* probs = (double*)malloc(sizeof(double) * (size_t)T * E);
    double* pbar = (double*)calloc((size_t)E, sizeof(double));
    double* dl = (double*)malloc(sizeof(double) * (size_t)T * E);
    int real = 0;
    for (int t = 0; t < T; ++t) {
        const double* l = logits + (size_t)t * E;
        double m = -INFINITY, z = 0.0;
        for (int e = 0; e < E; ++e) if (l[e] > m) m = l[e];
        for (int e = 0; e < E; ++e) z += exp((l[e] - m) / tau);
        for (int e = 0; e < E; ++e) probs[(size_t)t * E + e] = exp((l[e] - m) / tau) / z;
        if (topk[(size_t)t * k] < 0) continue;              /* masked token */
        ++real;
        for (int e = 0; e < E; ++e) pbar[e] += probs[(size_t)t * E + e];
    }
    for (int e = 0; e < E; ++e) pbar[e] /= real > 0 ? (double)real : 1.0;
    if (pbar_in)
        for (int e = 0; e < E; ++e) pbar[e] = pbar_in[e];
    const double Tn = T_aux > 0 ? (double)T_aux : (real > 0 ? (double)real : 1.0);
    double* cvec = (double*)malloc(sizeof(double) * (size_t)E); /* dL_aux / dp[t,e] */
    for (int e = 0; e < E; ++e) cvec[e] = c->aux_coef * 2.0 * (pbar[e] - 1.0 / E) / Tn;

    for (int t = 0; t < T; ++t) {
        const double* p = probs + (size_t)t * E;
        const double* g = gate + (size_t)t * k;
        const double* dg = dgate + (size_t)t * k;
        const int* sel = topk + (size_t)t * k;
        double* dlt = dl + (size_t)t * E;
        for (int e = 0; e < E; ++e) dlt[e] = 0.0;
        if (sel[0] < 0) continue;                            /* masked token: no gradient */
        if (c->normalize_gates && !c->straight_through) {
            /* gate_j = exp(l_j/tau) / sum_sel: d gate_j / d l_i = gate_j (delta_ji - gate_i) / tau */
            double s = 0.0;
            for (int j = 0; j < k; ++j) s += g[j] * dg[j];
            for (int j = 0; j < k; ++j) dlt[sel[j]] += g[j] * (dg[j] - s) / tau;
        } else {
            /* raw probabilities (gate_j = p_{e_j}), and the straight-through estimator
             * (forward gates 1, backward through p_{e_j}): d p_a / d l_b = p_a (delta_ab - p_b) / tau */
            double s = 0.0;
            for (int j = 0; j < k; ++j) s += dg[j] * p[sel[j]];
            for (int j = 0; j < k; ++j) dlt[sel[j]] += dg[j] * p[sel[j]] / tau;
            for (int e = 0; e < E; ++e) dlt[e] -= p[e] * s / tau;
        }
        /* aux: dL/dp[t,e] = cvec[e], through the full softmax */
        double s = 0.0;
        for (int e = 0; e < E; ++e) s += p[e] * cvec[e];
        for (int e = 0; e < E; ++e) dlt[e] += p[e] * (cvec[e] - s) / tau;
    }

    /* dx = sum over kept slots of the expert dx, plus the router term, plus the
     * shared experts' term */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double* o = dx + (size_t)t * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        for (int j = 0; j < k; ++j) {
            if (slot_of[(size_t)t * k + j] < 0) continue;
            const double* r = dxp + ((size_t)t * k + j) * d;
            for (int i = 0; i < d; ++i) o[i] += r[i];
        }
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int e = 0; e < E; ++e) acc += dl[(size_t)t * E + e] * Wr[(size_t)i * E + e];
            o[i] += acc;
        }
        if (dxs)
            for (int i = 0; i < d; ++i) o[i] += dxs[(size_t)t * d + i];
    }
    /* dW_r = x^T dlogits ; db = sum_t dlogits */
#pragma omp parallel for schedule(static)
    for (int i = 0; i < d; ++i)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t) acc += x[(size_t)t * d + i] * dl[(size_t)t * E + e];
            dWr[(size_t)i * E + e] = acc;
        }
    if (db)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t) acc += dl[(size_t)t * E + e];
            db[e] = acc;
        }
    if (dgate_out) memcpy(dgate_out, dgate, sizeof(double) * (size_t)T * k);
    if (dxp_slot_out) memcpy(dxp_slot_out, dxp, sizeof(double) * (size_t)T * k * d);
    if (dlogits_out) memcpy(dlogits_out, dl, sizeof(double) * (size_t)T * E);
    free(dgate); free(dxp); free(probs); free(pbar); free(dl); free(cvec); free(dxs);
}

/* ---- Single weight-gradient entries of one expert, from the definition ----
 * Only the <dout, out> part of the loss reaches the expert weights (the aux
 * loss depends on the router alone).  Expert e's kept tokens t, with
 * dy_t = gate_t dout_t ([LLaMA4-MoE] §2.4: output = gate-weighted sum), give
 *   dW_down[j][i] = sum_t act_j(x_t) dy_t[i]
 *   SiLU:   dW_up[i][j]   = sum_t x_t[i] dact_j silu'(h_j)
 *   SwiGLU: dW_up[i][j]   = sum_t x_t[i] dact_j silu(g_j)
 *           dW_gate[i][j] = sum_t x_t[i] dact_j u_j silu'(g_j)
 * where, for the one hidden unit j, h_j = x_t . W_up[:,j] (SwiGLU:
 * g_j = x_t . W_gate[:,j], u_j = x_t . W_up[:,j]), act_j = silu(h_j) or
 * silu(g_j) u_j, and dact_j = W_down[j,:] . dy_t.  So an entry needs one
 * column of W_up (W_gate) and one row of W_down: O(n d) per entry, which
 * lets single entries of a full-size layer be checked.
 *   xs[n][d], douts[n][d]: inputs and output gradients of the n kept tokens,
 *   gates[n] their gates for this expert (tokens in ascending order);
 *   Wu, Wg (SwiGLU, else NULL) [d][f] and Wd [f][d]: expert e's blocks;
 *   which[q] = 0: dW_down[rows[q]][cols[q]]; 1: dW_up[rows[q]][cols[q]];
 *   2: dW_gate[rows[q]][cols[q]] (SwiGLU).  out[q] receives the entry.       */
void oracle_expert_wgrad_entries(const oracle_cfg* c, int n, const double* xs,
                                 const double* gates, const double* douts, const double* Wu,
                                 const double* Wg, const double* Wd, int nq, const int* which,
                                 const int* rows, const int* cols, double* out)
{
    const int d = c->d, f = c->f;
#pragma omp parallel for schedule(dynamic, 1)
    for (int q = 0; q < nq; ++q) {
        const int kind = which[q];
        const int j = kind == 0 ? rows[q] : cols[q];    /* hidden unit */
        const int i = kind == 0 ? cols[q] : rows[q];    /* model-width index */
        /* the weights unit j touches: column j of W_up (and W_gate), row j of W_down */
        double* wcol = (double*)malloc(sizeof(double) * 2 * (size_t)d);
        double* gcol = wcol + d;
        for (int r = 0; r < d; ++r) {
            wcol[r] = Wu[(size_t)r * f + j];
            gcol[r] = c->swiglu ? Wg[(size_t)r * f + j] : 0.0;
        }
        const double* wdrow = Wd + (size_t)j * d;
        double acc = 0.0;
        for (int t = 0; t < n; ++t) {
            const double* x = xs + (size_t)t * d;
            const double* go = douts + (size_t)t * d;
            double pre = 0.0, u = 0.0;     /* h_j (SiLU) or g_j, and u_j (SwiGLU) */
            for (int r = 0; r < d; ++r) {
                if (c->swiglu) { pre += x[r] * gcol[r]; u += x[r] * wcol[r]; }
                else pre += x[r] * wcol[r];
            }
            if (kind == 0) {
                const double act = c->swiglu ? silu(pre) * u : silu(pre);
                acc += act * (gates[t] * go[i]);
                continue;
            }
            double dact = 0.0;
            for (int r = 0; r < d; ++r) dact += wdrow[r] * (gates[t] * go[r]);
            double dpre;
            if (!c->swiglu) dpre = dact * dsilu(pre);
            else if (kind == 1) dpre = dact * silu(pre);
            else dpre = dact * u * dsilu(pre);
            acc += x[i] * dpre;
        }
        out[q] = acc;
        free(wcol);
    }
}

/* Threads the OpenMP loops above use (results do not depend on it): the
 * benchmark times the oracle on all host cores and on one.                   */
void oracle_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
int oracle_max_threads(void) { return omp_get_max_threads(); }
