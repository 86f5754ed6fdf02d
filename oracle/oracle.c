/*
 * CPU oracle for the expert-streaming MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no code with the CUDA library: it reads the
 * canonical weight layout directly, one element at a time, and follows the
 * plain definition of each step. Single-threaded, built with -O2
 * -ffp-contract=off so that every floating-point operation is the one written.
 *
 * Pages cited:
 *   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
 *        (the turbo-fieldfare port plan), by section number.
 *   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测", by section heading.
 *
 * What each function follows:
 *   - weights are MLX-style affine 4-bit in groups of 64, the router 8-bit
 *     affine in groups of 64: w = scale * q + bias  ([P1] §2.1 table, §2.5
 *     "量化方案");
 *   - per token and layer the router scores every expert, the top-k are chosen
 *     and their outputs are combined with gate weights, y = sum_j w_j E_j(x)
 *     ([P3] "每个 token、每层都要重新路由"; [P1] §2.4 cb1/cb2);
 *   - the shared expert is always resident and is added to the weighted routed
 *     output ([P1] §2.3, §6.2.3 "共享专家输出 + 路由专家输出加权融合");
 *   - the per-layer LFU expert cache: empty slot first, else the slot with the
 *     smallest use count, new entries start at 1, hits increment
 *     ([P1] §6.2.2, §6.2.3 ExpertCache, §8.3); the LRU variant keyed by
 *     (layer, expert) whose budget may be exceeded to protect the working set
 *     ([P3] "缓存管理的是专家工作集");
 *   - prefill groups a chunk's tokens by expert so one fetch serves every row
 *     of the chunk ([P1] §2.5, §8.4).
 *
 * Readings where the pages are silent (each listed with its reason in the
 * design notes): fp32 router logits in a fixed lane-strided order so that the
 * chosen ids are reproducible bit for bit; ties in top-k go to the lower expert
 * index; gates are the full softmax renormalised over the k chosen experts;
 * GELU uses the tanh form; one LFU increment per distinct expert per step,
 * distinct ids handled in ascending order, the step's slots pinned, and misses
 * beyond the free capacity bypass the cache.
 *
 * Precision: weights dequantise exactly in double; the FFNs and the combine
 * accumulate in double. Router logits are fp32 (the precision that decides the
 * integer expert ids on the device as well).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_SLOTS 1024
#define ORACLE_MAX_EXPERTS 4096

/* ---- storage formats (exact decoding) ----------------------------------- */

/* IEEE 754 binary16 -> double, exact. */
double oracle_f16(uint16_t h) {
    int sign = (h >> 15) & 1, ex = (h >> 10) & 0x1F, mant = h & 0x3FF;
    double v;
    if (ex == 0)
        v = ldexp((double)mant, -24);
    else if (ex == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), ex - 25);
    return sign ? -v : v;
}

/* bfloat16 -> float, exact (the upper half of a binary32). */
float oracle_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ---- dequantisation ([P1] §2.1, §2.5) ----------------------------------- */

/* 4-bit code of element (n, k) of a row-major [N][K] matrix: byte k/2 of row
 * n, low nibble for even k, high nibble for odd k. */
unsigned oracle_code_u4(const uint8_t* codes, int K, int n, int k) {
    uint8_t byte = codes[(size_t)n * (size_t)(K / 2) + (size_t)(k / 2)];
    return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 15u);
}

/* Dequantised 4-bit weight w[n][k] = scale[n][k/64] * q + bias[n][k/64]. The
 * product and sum are exact in double (11+4 and 11 significant bits). */
double oracle_w4(const uint8_t* codes, const uint16_t* scale, const uint16_t* bias, int K, int n, int k) {
    size_t g = (size_t)n * (size_t)(K / 64) + (size_t)(k / 64);
    return oracle_f16(scale[g]) * (double)oracle_code_u4(codes, K, n, k) + oracle_f16(bias[g]);
}

/* Dequantised 8-bit router weight, exact in double. */
double oracle_w8(const uint8_t* codes, const uint16_t* scale, const uint16_t* bias, int K, int n, int k) {
    size_t g = (size_t)n * (size_t)(K / 64) + (size_t)(k / 64);
    return oracle_f16(scale[g]) * (double)codes[(size_t)n * (size_t)K + (size_t)k] + oracle_f16(bias[g]);
}

/* ---- router ([P3] "每个 token、每层都要重新路由"; [P1] §2.4 cb1) ---------- */

/*
 * Router logits in fp32, in the fixed order that makes the selected ids
 * reproducible bit for bit:
 *   the d inputs are cut into runs of 16; run c belongs to lane c mod 32;
 *   each of the 32 lanes walks its runs in increasing c and, inside a run,
 *   the elements in increasing index, doing
 *       w = fmaf(scale, q, bias);   acc = fmaf(w, x, acc)   (acc starts at 0);
 *   then the 32 lane sums are combined pairwise at distances 16, 8, 4, 2, 1:
 *       s[l] <- s[l] + s[l ^ dist]  (all l at once),
 *   and lane 0's sum plus zbias[e] (when given) is the logit.
 * x is [T][d] bfloat16, codes [E][d], scale/bias [E][d/64]; out is [T][E].
 */
void oracle_router_logits(const uint16_t* x, int T, int d, int E, const uint8_t* codes, const uint16_t* scale,
                          const uint16_t* bias, const float* zbias, float* out) {
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float lane[32];
            for (int l = 0; l < 32; ++l) {
                float acc = 0.0f;
                for (int c = l; c * 16 < d; c += 32) {
                    for (int i = c * 16; i < c * 16 + 16; ++i) {
                        size_t g = (size_t)e * (size_t)(d / 64) + (size_t)(i / 64);
                        float s = (float)oracle_f16(scale[g]);
                        float b = (float)oracle_f16(bias[g]);
                        float w = fmaf(s, (float)codes[(size_t)e * (size_t)d + (size_t)i], b);
                        acc = fmaf(w, oracle_bf16(x[(size_t)t * (size_t)d + (size_t)i]), acc);
                    }
                }
                lane[l] = acc;
            }
            for (int dist = 16; dist >= 1; dist /= 2) {
                float nxt[32];
                for (int l = 0; l < 32; ++l) nxt[l] = lane[l] + lane[l ^ dist];
                memcpy(lane, nxt, sizeof lane);
            }
            float logit = lane[0];
            if (zbias) logit = logit + zbias[e];
            out[(size_t)t * (size_t)E + (size_t)e] = logit;
        }
    }
}

/* Router logits in double, plain sum in index order (for bounding the fp32 ones). */
void oracle_router_logits_f64(const uint16_t* x, int T, int d, int E, const uint8_t* codes, const uint16_t* scale,
                              const uint16_t* bias, const float* zbias, double* out) {
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += oracle_w8(codes, scale, bias, d, e, i) * (double)oracle_bf16(x[(size_t)t * (size_t)d + (size_t)i]);
            out[(size_t)t * (size_t)E + (size_t)e] = acc + (zbias ? (double)zbias[e] : 0.0);
        }
}

/* Does expert a rank before expert b? Larger logit first; equal logits go to
 * the lower index. */
static int ranks_before(const float* l, int a, int b) { return l[a] > l[b] || (l[a] == l[b] && a < b); }

/*
 * Top-k and gates for each token: ids[t][0..k) are the k experts with the
 * largest logits in rank order (ties to the lower index); gates are the
 * softmax over all E logits, renormalised over the k chosen (in double).
 * Selection is by selection sort on the fp32 logits.
 */
void oracle_topk_gates(const float* logits, int T, int E, int k, int32_t* ids, double* gates) {
    char* taken = (char*)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * (size_t)E;
        memset(taken, 0, (size_t)E);
        for (int r = 0; r < k; ++r) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || ranks_before(l, e, best))) best = e;
            taken[best] = 1;
            ids[(size_t)t * (size_t)k + (size_t)r] = best;
        }
        /* full softmax over all experts (shifted by the maximum) */
        double mx = -INFINITY;
        for (int e = 0; e < E; ++e) mx = fmax(mx, (double)l[e]);
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp((double)l[e] - mx);
        double sel = 0.0;
        for (int r = 0; r < k; ++r) sel += exp((double)l[ids[(size_t)t * (size_t)k + (size_t)r]] - mx) / z;
        for (int r = 0; r < k; ++r) {
            double p = exp((double)l[ids[(size_t)t * (size_t)k + (size_t)r]] - mx) / z;
            gates[(size_t)t * (size_t)k + (size_t)r] = p / sel;
        }
    }
    free(taken);
}

/* ---- expert FFN ([P1] §2.4 cb2; [P3] "每个 token、每层都要重新路由") ----- */

#define ACT_GELU_TANH 0
#define ACT_SILU 1

/* gelu_tanh(z) = z/2 (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))); silu(z) = z / (1 + e^-z). */
double oracle_act(double z, int act) {
    if (act == ACT_SILU) return z / (1.0 + exp(-z));
    const double c = 0.7978845608028654; /* sqrt(2/pi) */
    return 0.5 * z * (1.0 + tanh(c * (z + 0.044715 * z * z * z)));
}

/*
 * One gated FFN on one token: h[j] = act(Wg[j] . x) * (Wu[j] . x), then
 * out[n] = Wd[n] . h. Wg, Wu are [inter][d], Wd is [d][inter], canonical
 * 4-bit layout. x is d bfloat16 values. Double accumulation in index order.
 */
void oracle_ffn(const uint16_t* x, int d, int inter, int act, const uint8_t* gc, const uint16_t* gs,
                const uint16_t* gb, const uint8_t* uc, const uint16_t* us, const uint16_t* ub, const uint8_t* dc,
                const uint16_t* ds, const uint16_t* db, double* out) {
    double* h = (double*)malloc(sizeof(double) * (size_t)inter);
    for (int j = 0; j < inter; ++j) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < d; ++i) {
            double xi = (double)oracle_bf16(x[i]);
            g += oracle_w4(gc, gs, gb, d, j, i) * xi;
            u += oracle_w4(uc, us, ub, d, j, i) * xi;
        }
        h[j] = oracle_act(g, act) * u;
    }
    for (int n = 0; n < d; ++n) {
        double acc = 0.0;
        for (int j = 0; j < inter; ++j) acc += oracle_w4(dc, ds, db, inter, n, j) * h[j];
        out[n] = acc;
    }
    free(h);
}

/* Weights of one layer in the canonical layout. Routed arrays are stacked on a
 * leading expert axis: gate/up codes [E][I][d/2], scales [E][I][d/64], down
 * codes [E][d][I/2], scales [E][d][I/64]. */
typedef struct {
    int d, E, k, I, Is, act;
    const uint8_t* rc;
    const uint16_t *rs, *rb;
    const uint8_t *sgc, *suc, *sdc;
    const uint16_t *sgs, *sgb, *sus, *sub, *sds, *sdb;
    const uint8_t *gc, *uc, *dc;
    const uint16_t *gs, *gb, *us, *ub, *ds, *db;
} oracle_layer;

static void expert_ffn(const oracle_layer* L, int e, const uint16_t* x, double* out) {
    size_t gcs = (size_t)L->I * (size_t)(L->d / 2), gss = (size_t)L->I * (size_t)(L->d / 64);
    size_t dcs = (size_t)L->d * (size_t)(L->I / 2), dss = (size_t)L->d * (size_t)(L->I / 64);
    oracle_ffn(x, L->d, L->I, L->act, L->gc + e * gcs, L->gs + e * gss, L->gb + e * gss, L->uc + e * gcs,
               L->us + e * gss, L->ub + e * gss, L->dc + e * dcs, L->ds + e * dss, L->db + e * dss, out);
}

/* Shared expert output for one token. */
void oracle_shared_ffn(const oracle_layer* L, const uint16_t* x, double* out) {
    oracle_ffn(x, L->d, L->Is, L->act, L->sgc, L->sgs, L->sgb, L->suc, L->sus, L->sub, L->sdc, L->sds, L->sdb, out);
}

/* One routed expert's output for one token. */
void oracle_expert_ffn(const oracle_layer* L, int e, const uint16_t* x, double* out) { expert_ffn(L, e, x, out); }

/*
 * The MoE layer on T tokens: y[t] = shared(x_t) + sum_{r<k} gate[t][r] * FFN_{ids[t][r]}(x_t),
 * the routed terms added in rank order. Writes logits [T][E] (fp32), ids
 * [T][k], gates [T][k] and y [T][d] (double). zbias may be NULL.
 */
void oracle_moe_layer(const oracle_layer* L, const uint16_t* x, int T, const float* zbias, float* logits,
                      int32_t* ids, double* gates, double* y) {
    oracle_router_logits(x, T, L->d, L->E, L->rc, L->rs, L->rb, zbias, logits);
    oracle_topk_gates(logits, T, L->E, L->k, ids, gates);
    double* o = (double*)malloc(sizeof(double) * (size_t)L->d);
    for (int t = 0; t < T; ++t) {
        const uint16_t* xt = x + (size_t)t * (size_t)L->d;
        double* yt = y + (size_t)t * (size_t)L->d;
        oracle_shared_ffn(L, xt, yt);
        for (int r = 0; r < L->k; ++r) {
            expert_ffn(L, ids[(size_t)t * (size_t)L->k + (size_t)r], xt, o);
            double g = gates[(size_t)t * (size_t)L->k + (size_t)r];
            for (int n = 0; n < L->d; ++n) yt[n] += g * o[n];
        }
    }
    free(o);
}

/*
 * Brute force of the same layer for tiny inputs: evaluate every expert
 * densely, decide membership of the top-k by counting for each expert how
 * many others rank before it, take the renormalised softmax weight of the
 * members and zero for the rest, and sum over all experts in index order.
 */
void oracle_moe_layer_dense(const oracle_layer* L, const uint16_t* x, int T, const float* zbias, double* y) {
    float* logits = (float*)malloc(sizeof(float) * (size_t)L->E);
    double* w = (double*)malloc(sizeof(double) * (size_t)L->E);
    double* o = (double*)malloc(sizeof(double) * (size_t)L->d);
    for (int t = 0; t < T; ++t) {
        const uint16_t* xt = x + (size_t)t * (size_t)L->d;
        oracle_router_logits(xt, 1, L->d, L->E, L->rc, L->rs, L->rb, zbias, logits);
        double mx = -INFINITY, z = 0.0, sel = 0.0;
        for (int e = 0; e < L->E; ++e) mx = fmax(mx, (double)logits[e]);
        for (int e = 0; e < L->E; ++e) z += exp((double)logits[e] - mx);
        for (int e = 0; e < L->E; ++e) {
            int before = 0;
            for (int f = 0; f < L->E; ++f)
                if (f != e && ranks_before(logits, f, e)) ++before;
            w[e] = before < L->k ? exp((double)logits[e] - mx) / z : 0.0;
            sel += w[e];
        }
        double* yt = y + (size_t)t * (size_t)L->d;
        oracle_shared_ffn(L, xt, yt);
        for (int e = 0; e < L->E; ++e) {
            expert_ffn(L, e, xt, o);
            for (int n = 0; n < L->d; ++n) yt[n] += (w[e] / sel) * o[n];
        }
    }
    free(logits);
    free(w);
    free(o);
}

/* ---- expert cache ([P1] §6.2.2, §6.2.3, §8.3; [P3] "缓存管理的是专家工作集") -- */

#define POLICY_LFU 0
#define POLICY_LRU 1

typedef struct {
    int E, S, policy;
    int64_t step;
    int32_t slot_expert[ORACLE_MAX_SLOTS]; /* -1: empty */
    uint32_t count[ORACLE_MAX_SLOTS];      /* LFU use count */
    int64_t tick[ORACLE_MAX_SLOTS];        /* LRU: step of last use */
} oracle_cache;

int oracle_cache_init(oracle_cache* c, int E, int S, int policy) {
    if (S < 1 || S > ORACLE_MAX_SLOTS || E < 1 || E > ORACLE_MAX_EXPERTS) return -1;
    c->E = E;
    c->S = S;
    c->policy = policy;
    c->step = 0;
    for (int s = 0; s < S; ++s) {
        c->slot_expert[s] = -1;
        c->count[s] = 0;
        c->tick[s] = 0;
    }
    return 0;
}

static int find_slot(const oracle_cache* c, int e) {
    for (int s = 0; s < c->S; ++s)
        if (c->slot_expert[s] == e) return s;
    return -1;
}

/*
 * One lookup step over the ids of one call (n ids, duplicates allowed).
 * Distinct experts are visited in ascending id. Hits: LFU count += 1 (LRU:
 * tick = step) and the slot is pinned for this step. Misses, ascending: the
 * lowest-index empty slot, else the unpinned slot with the smallest count
 * (LRU: smallest tick), ties to the lowest slot index; the new entry starts at
 * count 1 (tick = step) and is pinned. A miss with no unpinned slot left
 * bypasses the cache (slot -1, not inserted).
 * Outputs: slot_of[i] for each input id (-1 = bypass); miss lists in ascending
 * expert order with their slot (-1 = bypass); counts of hits, misses (bypasses
 * included) and bypasses.
 */
int oracle_cache_step(oracle_cache* c, const int32_t* ids, int n, int32_t* slot_of, int32_t* miss_expert,
                      int32_t* miss_slot, int32_t* n_hit, int32_t* n_miss, int32_t* n_bypass) {
    char present[ORACLE_MAX_EXPERTS];
    char pinned[ORACLE_MAX_SLOTS];
    int32_t where[ORACLE_MAX_EXPERTS];
    memset(present, 0, (size_t)c->E);
    memset(pinned, 0, (size_t)c->S);
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= c->E) return -1;
        present[ids[i]] = 1;
    }
    *n_hit = *n_miss = *n_bypass = 0;
    for (int e = 0; e < c->E; ++e) {
        where[e] = -1;
        if (!present[e]) continue;
        int s = find_slot(c, e);
        if (s >= 0) {
            if (c->policy == POLICY_LFU)
                c->count[s] += 1;
            else
                c->tick[s] = c->step;
            pinned[s] = 1;
            where[e] = s;
            ++*n_hit;
        }
    }
    for (int e = 0; e < c->E; ++e) {
        if (!present[e] || where[e] >= 0) continue;
        int victim = -1;
        for (int s = 0; s < c->S && victim < 0; ++s)
            if (c->slot_expert[s] < 0) victim = s;
        if (victim < 0) {
            for (int s = 0; s < c->S; ++s) {
                if (pinned[s]) continue;
                if (victim < 0) {
                    victim = s;
                } else if (c->policy == POLICY_LFU ? c->count[s] < c->count[victim] : c->tick[s] < c->tick[victim]) {
                    victim = s;
                }
            }
        }
        miss_expert[*n_miss] = e;
        miss_slot[*n_miss] = victim;
        ++*n_miss;
        if (victim < 0) {
            ++*n_bypass;
            continue;
        }
        c->slot_expert[victim] = e;
        c->count[victim] = 1;
        c->tick[victim] = c->step;
        pinned[victim] = 1;
        where[e] = victim;
    }
    for (int i = 0; i < n; ++i) slot_of[i] = where[ids[i]];
    c->step += 1;
    return 0;
}

/* Slot table snapshot: expert per slot (-1 empty) and LFU counts. */
void oracle_cache_dump(const oracle_cache* c, int32_t* slot_expert, uint32_t* counts) {
    for (int s = 0; s < c->S; ++s) {
        slot_expert[s] = c->slot_expert[s];
        counts[s] = c->count[s];
    }
}

int oracle_cache_size(void) { return (int)sizeof(oracle_cache); }

/* ---- prefill grouping ([P1] §2.5, §8.4) --------------------------------- */

/*
 * Group the (token, rank) pairs of a chunk by expert: pair p = t*k + r has
 * expert ids[p]. perm lists the pairs of expert 0, then expert 1, ..., each in
 * increasing p (a stable sort by expert); offsets[e] .. offsets[e+1] is expert
 * e's range.
 */
void oracle_group_pairs(const int32_t* ids, int n_pairs, int E, int32_t* offsets, int32_t* perm) {
    int pos = 0;
    for (int e = 0; e < E; ++e) {
        offsets[e] = pos;
        for (int p = 0; p < n_pairs; ++p)
            if (ids[p] == e) perm[pos++] = p;
    }
    offsets[E] = pos;
}
