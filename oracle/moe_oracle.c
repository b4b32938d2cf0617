/*
 * moe_oracle.c -- the oracle: a plain, slow, obviously correct fp64 CPU model of the
 * sparse Mixture-of-Experts feed-forward layer (router, softmax, top-K with renormalised
 * weights, SwiGLU experts, sigmoid-gated shared expert, sum into the residual).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load this file's library. It shares no code, header, table or helper with the CUDA
 * library of the product path, and the product path never calls it.
 *
 * Conventions (all fixed by the pages):
 *   - Every weight is stored [Out, In] row-major ("Qwen3.6 35B-A3B", Blocks: Linear,
 *     `weight: Tensor[Out, In; T]`), so "x . W" in the expert equation is x times the
 *     transpose of the stored matrix.
 *   - Storage type T = bf16 ("Qwen3.6 35B-A3B", Generics: T bf16). Inputs arrive as the raw
 *     16-bit patterns and are widened exactly to double; nothing is rounded afterwards.
 *   - The merged gate_up tensor is [Experts, 2*ExpertInner, H] ("Qwen3.6 35B-A3B", Blocks:
 *     SparseMoe; "Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts). The pages
 *     do not say how the two halves are placed; this oracle reads rows [0, I) as the gate
 *     projection and rows [I, 2I) as the up projection (name order, not interleaved).
 *   - Router outputs: by default the router and shared-gate scores are kept exact (fp64).
 *     With ORACLE_BF16_SCORES in dims.flags they are typed T = bf16 as the pages' interface
 *     types them (`gate: Linear<H, Experts, T>`, `shared_expert_gate: Linear<H, 1, T>` and
 *     `ranks(logits: Tensor[R, Experts; T])` in "Qwen3.6 35B-A3B", Blocks: SparseMoe): each
 *     score, bias included, is rounded to the nearest bf16 (ties to even) before the softmax,
 *     the ranking and the sigmoid. Equal rounded scores are then common; the rank rule puts
 *     the lower expert index first.
 *
 * Each function follows one step of the pages and cites it. Work is split over tokens with
 * OpenMP only; tokens are independent, so the split changes no result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t T;  /* tokens (B*S flattened) */
    int32_t H;  /* hidden width */
    int32_t E;  /* routed experts */
    int32_t K;  /* experts chosen per token */
    int32_t I;  /* routed expert inner width */
    int32_t Is; /* shared expert inner width */
    int32_t flags; /* ORACLE_BF16_SCORES: router and shared-gate scores typed bf16 */
} oracle_dims;

#define ORACLE_BF16_SCORES 1

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an IEEE binary32. */
static double bf(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Round a double to the nearest bf16 (ties to even) and return the bit pattern.
 * Used only where the pages type a value as T = bf16 between two steps (the RMSNorm
 * output and the residual stream of a stack of layers). */
uint16_t oracle_round_bf16(double v) {
    float f = (float)v; /* first rounding: to the 24-bit significand */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t low = u & 0xffffu, hi = u >> 16; /* sign-magnitude: hi + 1 grows the magnitude */
    if (low > 0x8000u) {
        hi += 1u;
    } else if (low == 0x8000u) {
        /* f sits on a bf16 midpoint. If v itself is not f, the first rounding moved it
         * there and v lies strictly on one side: round to that side, not to even. */
        if ((double)f != v) {
            if (fabs(v) > fabs((double)f)) hi += 1u;
        } else if (hi & 1u) {
            hi += 1u;
        }
    }
    return (uint16_t)hi;
}

/* A score as the following steps see it: exact, or rounded to bf16 under ORACLE_BF16_SCORES. */
static double score_as_typed(const oracle_dims* d, double s) {
    return (d->flags & ORACLE_BF16_SCORES) ? bf(oracle_round_bf16(s)) : s;
}

/* Router projection: "A learned linear layer 2048 -> 256 scores all 256 experts for each
 * token" ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts, Router; the
 * router is `gate: Linear<H, Experts>` in "Qwen3.6 35B-A3B", Blocks: SparseMoe, with the
 * optional `bias: Tensor[Out; T]?` of Blocks: Linear).
 * logits[t*E + e] = sum_h x[t,h] * Wr[e,h] (+ br[e]), then typed (score_as_typed). */
void oracle_router_logits(const oracle_dims* d, const uint16_t* x, const uint16_t* router_w,
                          const uint16_t* router_b, double* logits) {
    const int T = d->T, H = d->H, E = d->E;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int h = 0; h < H; ++h) s += bf(x[(size_t)t * H + h]) * bf(router_w[(size_t)e * H + h]);
            if (router_b) s += bf(router_b[e]);
            logits[(size_t)t * E + e] = score_as_typed(d, s);
        }
    }
}

/* Softmax over the E router scores ("Softmax, then top-8 are selected",
 * "Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts, Router). */
static void softmax_row(int E, const double* l, double* p) {
    double m = l[0];
    for (int e = 1; e < E; ++e)
        if (l[e] > m) m = l[e];
    double s = 0.0;
    for (int e = 0; e < E; ++e) {
        p[e] = exp(l[e] - m);
        s += p[e];
    }
    for (int e = 0; e < E; ++e) p[e] /= s;
}

/* Rank of every expert, as the `ranks(logits) -> Tensor[R, Experts; i32]` function of
 * "Qwen3.6 35B-A3B" (Blocks: SparseMoe) returns it: rank 0 is the highest probability. The
 * pages give no tie rule; equal probabilities are ordered by the lower expert index.
 * rank[e] = #{ j : p[j] > p[e]  or  (p[j] == p[e] and j < e) }  (brute force, O(E^2)). */
static void ranks_row(int E, const double* p, int32_t* rank) {
    for (int e = 0; e < E; ++e) {
        int r = 0;
        for (int j = 0; j < E; ++j)
            if (p[j] > p[e] || (p[j] == p[e] && j < e)) ++r;
        rank[e] = r;
    }
}

/* Top-K selection and renormalisation ("top-8 are selected and their weights renormalized
 * to sum to 1", "Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts, Router;
 * "The router does not run all 256 experts", "One Token Through Qwen3.6", The Router).
 * The expert with rank k goes to slot k, so slots run from the highest probability down.
 * w[k] = p[id_k] / sum_{j<K} p[id_j]. */
static void select_row(int E, int K, const double* p, int32_t* rank_scratch, int32_t* ids, double* w) {
    ranks_row(E, p, rank_scratch);
    for (int e = 0; e < E; ++e)
        if (rank_scratch[e] < K) ids[rank_scratch[e]] = e;
    double s = 0.0;
    for (int k = 0; k < K; ++k) s += p[ids[k]];
    for (int k = 0; k < K; ++k) w[k] = p[ids[k]] / s;
}

/* Token dispatch: which rows each expert receives ("It determines which experts should
 * receive this token", "One Token Through Qwen3.6", The Router). The pages give no layout;
 * this is a plain stable counting sort of the (token, slot) pairs by expert:
 *   counts[e]  = number of pairs routed to e,
 *   offsets[e] = sum_{j<e} counts[j], offsets[E] = T*K,
 *   perm[j]    = t*K + k for the pairs in expert order, tokens ascending within an expert,
 *   inv[t*K+k] = the position j of that pair in perm. */
void oracle_permute(const oracle_dims* d, const int32_t* ids, int32_t* counts, int32_t* offsets,
                    int32_t* perm, int32_t* inv) {
    const int T = d->T, E = d->E, K = d->K;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int i = 0; i < T * K; ++i) counts[ids[i]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int pos = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int k = 0; k < K; ++k)
                if (ids[t * K + k] == e) {
                    perm[pos] = t * K + k;
                    if (inv) inv[t * K + k] = pos;
                    ++pos;
                }
}

/* Routing for all tokens: logits, softmax, ranks, top-K, renormalised weights, and the
 * dispatch of oracle_permute. probs (nullable) receives the full softmax row [T, E].
 * Returns 0, or -1 when the dims are unusable. */
int oracle_route(const oracle_dims* d, const uint16_t* x, const uint16_t* router_w, const uint16_t* router_b,
                 int32_t* ids, double* w, double* probs, int32_t* counts, int32_t* offsets, int32_t* perm,
                 int32_t* inv) {
    const int T = d->T, E = d->E, K = d->K;
    if (T < 0 || E <= 0 || K <= 0 || K > E || d->H <= 0) return -1;
    if (T == 0) {
        for (int e = 0; e < E; ++e) counts[e] = 0;
        for (int e = 0; e <= E; ++e) offsets[e] = 0;
        return 0;
    }
    double* logits = (double*)malloc(sizeof(double) * (size_t)T * E);
    if (!logits) return -1;
    oracle_router_logits(d, x, router_w, router_b, logits);
    int fail = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * E);
        int32_t* rk = (int32_t*)malloc(sizeof(int32_t) * E);
        if (!p || !rk) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(static)
            for (int t = 0; t < T; ++t) {
                softmax_row(E, logits + (size_t)t * E, p);
                select_row(E, K, p, rk, ids + (size_t)t * K, w + (size_t)t * K);
                if (probs) memcpy(probs + (size_t)t * E, p, sizeof(double) * E);
            }
        }
        free(p);
        free(rk);
    }
    free(logits);
    if (fail) return -1;
    oracle_permute(d, ids, counts, offsets, perm, inv);
    return 0;
}

/* Load-balancing statistics ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256
 * Experts, Load Balancing: an auxiliary loss with coefficient 0.001 penalises uneven expert
 * utilisation across the batch). The page names the loss but gives no formula; this oracle
 * computes the two per-expert quantities such a loss is built from, and the product form
 * that is smallest when routing is uniform:
 *   P_e  = (1/T) sum_t softmax(l_t)_e      mean router probability of expert e,
 *   f_e  = count_e / (T K)                 share of the T*K (token, slot) assignments,
 *   loss = 0.001 * E * sum_e f_e * P_e     (exactly 0.001 for uniform routing).
 * Sums run over t ascending and then e ascending. T = 0 gives zeros. Returns 0, or -1 when
 * the dims are unusable. */
int oracle_router_stats(const oracle_dims* d, const uint16_t* x, const uint16_t* router_w, const uint16_t* router_b,
                        double* P, double* f, double* loss) {
    const int T = d->T, E = d->E, K = d->K;
    if (T < 0 || E <= 0 || K <= 0 || K > E || d->H <= 0) return -1;
    for (int e = 0; e < E; ++e) P[e] = f[e] = 0.0;
    *loss = 0.0;
    if (T == 0) return 0;
    const size_t P_ = (size_t)T * K;
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * P_);
    double* w = (double*)malloc(sizeof(double) * P_);
    double* probs = (double*)malloc(sizeof(double) * (size_t)T * E);
    int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * E);
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (E + 1));
    int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * P_);
    int32_t* inv = (int32_t*)malloc(sizeof(int32_t) * P_);
    int rc = -1;
    if (ids && w && probs && counts && offsets && perm && inv &&
        oracle_route(d, x, router_w, router_b, ids, w, probs, counts, offsets, perm, inv) == 0) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int t = 0; t < T; ++t) s += probs[(size_t)t * E + e];
            P[e] = s / T;
            f[e] = (double)counts[e] / (double)P_;
        }
        double acc = 0.0;
        for (int e = 0; e < E; ++e) acc += f[e] * P[e];
        *loss = 0.001 * E * acc;
        rc = 0;
    }
    free(ids);
    free(w);
    free(probs);
    free(counts);
    free(offsets);
    free(perm);
    free(inv);
    return rc;
}

/* One SwiGLU feed-forward network applied to one token:
 *   expert(x) = SiLU(x . W_gate) (elementwise *) (x . W_up) . W_down
 * ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN: 256 Experts, Experts; the same
 * three projections as `SwiGlu<H, Inner>` with sub-blocks gate, up, down in
 * "Qwen3.6 35B-A3B", Blocks: SwiGlu; "One Token Through Qwen3.6", Inside One Expert).
 * gate_up is [2*Inner, H] (rows [0,Inner) gate, [Inner,2*Inner) up), down is [H, Inner].
 * SiLU(z) = z * sigmoid(z) = z / (1 + e^-z). Writes y[H]; hbuf[Inner] receives the gated
 * activation SiLU(g)*u. */
static void swiglu_token(int H, int Inner, const double* xrow, const uint16_t* gate_up, const uint16_t* down,
                         double* hbuf, double* y) {
    for (int i = 0; i < Inner; ++i) {
        double g = 0.0, u = 0.0;
        const uint16_t* wg = gate_up + (size_t)i * H;
        const uint16_t* wu = gate_up + (size_t)(Inner + i) * H;
        for (int h = 0; h < H; ++h) {
            g += xrow[h] * bf(wg[h]);
            u += xrow[h] * bf(wu[h]);
        }
        hbuf[i] = g / (1.0 + exp(-g)) * u;
    }
    for (int o = 0; o < H; ++o) {
        double s = 0.0;
        const uint16_t* wd = down + (size_t)o * Inner;
        for (int i = 0; i < Inner; ++i) s += hbuf[i] * bf(wd[i]);
        y[o] = s;
    }
}

/* The whole layer for every token ("Qwen3.6-35B-A3B -- Architecture Overview", MoE FFN:
 * 256 Experts: Router, Experts, Shared Expert; Stage 2: "RMSNorm -> MoE FFN -> +residual"):
 *   out[t] = residual[t] + sigmoid(x[t] . ws) * shared(x[t]) + sum_k w[t,k] * expert_{id[t,k]}(x[t])
 * shared_gate is the [1, H] weight of `shared_expert_gate: Linear<H, 1>` (no bias);
 * residual is nullable (then the layer output alone is returned).
 * Optional taps (each nullable):
 *   h_out   [T, K, I]  gated activation of each routed slot,
 *   y_out   [T, K, H]  each routed expert's output, before the routing weight,
 *   ys_out  [T, H]     the shared expert's output, before its gate,
 *   sg_out  [T]        the shared gate sigmoid(x . ws),
 *   ids/w   [T, K]     the routing of oracle_route (nullable together).
 * Returns 0, or -1 on unusable dims or allocation failure. */
int oracle_forward(const oracle_dims* d, const uint16_t* x, const uint16_t* router_w, const uint16_t* router_b,
                   const uint16_t* gate_up, const uint16_t* down, const uint16_t* shared_gate_up,
                   const uint16_t* shared_down, const uint16_t* shared_gate, const uint16_t* residual, double* out,
                   double* h_out, double* y_out, double* ys_out, double* sg_out, int32_t* ids_out, double* w_out) {
    const int T = d->T, H = d->H, E = d->E, K = d->K, I = d->I, Is = d->Is;
    if (T < 0 || H <= 0 || E <= 0 || K <= 0 || K > E || I <= 0 || Is <= 0) return -1;
    if (T == 0) return 0;
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * K);
    double* w = (double*)malloc(sizeof(double) * (size_t)T * K);
    int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * E);
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * (E + 1));
    int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * K);
    int rc = -1;
    if (!ids || !w || !counts || !offsets || !perm) goto done;
    if (oracle_route(d, x, router_w, router_b, ids, w, NULL, counts, offsets, perm, NULL) != 0) goto done;
    if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)T * K);
    if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)T * K);
    int fail = 0;
#pragma omp parallel
    {
        int Imax = I > Is ? I : Is;
        double* xrow = (double*)malloc(sizeof(double) * H);
        double* hb = (double*)malloc(sizeof(double) * Imax);
        double* y = (double*)malloc(sizeof(double) * H);
        double* acc = (double*)malloc(sizeof(double) * H);
        if (!xrow || !hb || !y || !acc) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(static)
            for (int t = 0; t < T; ++t) {
                for (int h = 0; h < H; ++h) xrow[h] = bf(x[(size_t)t * H + h]);
                for (int h = 0; h < H; ++h) acc[h] = residual ? bf(residual[(size_t)t * H + h]) : 0.0;
                /* Shared expert, always active, scaled by sigmoid(Linear(x, 1)). */
                double z = 0.0;
                for (int h = 0; h < H; ++h) z += xrow[h] * bf(shared_gate[h]);
                z = score_as_typed(d, z);
                double sg = 1.0 / (1.0 + exp(-z));
                swiglu_token(H, Is, xrow, shared_gate_up, shared_down, hb, y);
                for (int h = 0; h < H; ++h) acc[h] += sg * y[h];
                if (sg_out) sg_out[t] = sg;
                if (ys_out) memcpy(ys_out + (size_t)t * H, y, sizeof(double) * H);
                /* The K routed experts, each weighted by its renormalised routing weight. */
                for (int k = 0; k < K; ++k) {
                    int e = ids[(size_t)t * K + k];
                    swiglu_token(H, I, xrow, gate_up + (size_t)e * 2 * I * H, down + (size_t)e * H * I, hb, y);
                    double wk = w[(size_t)t * K + k];
                    for (int h = 0; h < H; ++h) acc[h] += wk * y[h];
                    if (h_out) memcpy(h_out + ((size_t)t * K + k) * I, hb, sizeof(double) * I);
                    if (y_out) memcpy(y_out + ((size_t)t * K + k) * H, y, sizeof(double) * H);
                }
                memcpy(out + (size_t)t * H, acc, sizeof(double) * H);
            }
        }
        free(xrow);
        free(hb);
        free(y);
        free(acc);
    }
    rc = fail ? -1 : 0;
done:
    free(ids);
    free(w);
    free(counts);
    free(offsets);
    free(perm);
    return rc;
}

/* RMSNorm before the MoE block ("RMSNorm -> MoE FFN -> +residual", "Qwen3.6-35B-A3B --
 * Architecture Overview", Stage 2; `RmsNorm<H, T>` with `weight: Tensor[H; T]` in
 * "Qwen3.6 35B-A3B", Blocks: RmsNorm):
 *   out[t,h] = x[t,h] / sqrt(mean_h(x[t,h]^2) + eps) * gamma[h]   (gamma nullable = ones). */
void oracle_rmsnorm(int32_t T, int32_t H, const uint16_t* x, const uint16_t* gamma, double eps, double* out) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            double v = bf(x[(size_t)t * H + h]);
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / H + eps);
        for (int h = 0; h < H; ++h)
            out[(size_t)t * H + h] = bf(x[(size_t)t * H + h]) * r * (gamma ? bf(gamma[h]) : 1.0);
    }
}
