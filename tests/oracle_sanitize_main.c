/* The CPU oracle (oracle/oracle.c) and the input generator (synth/gen.c)
 * under AddressSanitizer and UBSan: both are compiled into this program and
 * run on small layers of several shapes (routing, the sparse layer against
 * its dense brute force, every cache policy through overflowing steps, pair
 * grouping). Built and run by test_oracle_sanitizers.py; any memory error or
 * undefined behaviour ends the run with a report. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include "../oracle/oracle.c"
#include "../synth/gen.c"

static void* xmalloc(size_t n) {
    void* p = malloc(n ? n : 1);
    if (!p) exit(3);
    return p;
}

static void fill4(uint64_t key, int E, int n, int k, uint8_t** c, uint16_t** s, uint16_t** b) {
    const size_t el = (size_t)E * (size_t)n * (size_t)k, g = el / 64;
    *c = (uint8_t*)xmalloc(el / 2);
    *s = (uint16_t*)xmalloc(g * 2);
    *b = (uint16_t*)xmalloc(g * 2);
    synth_codes_u4(key, el, *c);
    synth_scale_bias_f16(key + 1, g, 0.005, 0.02, 1.0, -8.0, *s, *b);
}

static int run(int d, int E, int k, int I, int Is, int act, int T) {
    oracle_layer L;
    uint8_t *rc, *sgc, *suc, *sdc, *gc, *uc, *dc;
    uint16_t *rs, *rb, *sgs, *sgb, *sus, *sub, *sds, *sdb, *gs, *gb, *us, *ub, *ds, *db;
    const size_t rel = (size_t)E * (size_t)d;
    rc = (uint8_t*)xmalloc(rel);
    rs = (uint16_t*)xmalloc(rel / 64 * 2);
    rb = (uint16_t*)xmalloc(rel / 64 * 2);
    synth_codes_u8(11, rel, rc);
    synth_scale_bias_f16(12, rel / 64, 0.005, 0.02, sqrt((double)d), -128.0, rs, rb);
    fill4(20, 1, Is, d, &sgc, &sgs, &sgb);
    fill4(30, 1, Is, d, &suc, &sus, &sub);
    fill4(40, 1, d, Is, &sdc, &sds, &sdb);
    fill4(50, E, I, d, &gc, &gs, &gb);
    fill4(60, E, I, d, &uc, &us, &ub);
    fill4(70, E, d, I, &dc, &ds, &db);
    L.d = d; L.E = E; L.k = k; L.I = I; L.Is = Is; L.act = act;
    L.rc = rc; L.rs = rs; L.rb = rb;
    L.sgc = sgc; L.suc = suc; L.sdc = sdc;
    L.sgs = sgs; L.sgb = sgb; L.sus = sus; L.sub = sub; L.sds = sds; L.sdb = sdb;
    L.gc = gc; L.uc = uc; L.dc = dc;
    L.gs = gs; L.gb = gb; L.us = us; L.ub = ub; L.ds = ds; L.db = db;

    uint16_t* x = (uint16_t*)xmalloc((size_t)T * (size_t)d * 2);
    double* scratch = (double*)xmalloc((size_t)d * sizeof(double));
    synth_normal_bf16(80, T, d, 1, x, scratch);
    float* zb = (float*)xmalloc((size_t)E * sizeof(float));
    int32_t* perm = (int32_t*)xmalloc((size_t)E * sizeof(int32_t));
    synth_permutation(90, E, perm);
    for (int r = 0; r < E; ++r) zb[perm[r]] = (float)(-1.1 * log(r + 1.0));
    float* logits = (float*)xmalloc((size_t)T * (size_t)E * sizeof(float));
    int32_t* ids = (int32_t*)xmalloc((size_t)T * (size_t)k * sizeof(int32_t));
    double* gates = (double*)xmalloc((size_t)T * (size_t)k * sizeof(double));
    double* y = (double*)xmalloc((size_t)T * (size_t)d * sizeof(double));
    double* yd = (double*)xmalloc((size_t)T * (size_t)d * sizeof(double));
    oracle_moe_layer(&L, x, T, zb, logits, ids, gates, y);
    oracle_moe_layer_dense(&L, x, T, zb, yd);
    double err = 0, mx = 0;
    for (size_t i = 0; i < (size_t)T * (size_t)d; ++i) {
        err = fmax(err, fabs(y[i] - yd[i]));
        mx = fmax(mx, fabs(y[i]));
    }
    if (!(err <= 1e-9 * mx)) return 1;

    /* the cache under both policies, through steps that overflow it */
    for (int policy = 0; policy < 2; ++policy) {
        oracle_cache* c = (oracle_cache*)xmalloc(sizeof(oracle_cache));
        const int S = E > 4 ? E / 4 : 1;
        if (oracle_cache_init(c, E, S, policy) != 0) return 2;
        int32_t* slot_of = (int32_t*)xmalloc((size_t)T * (size_t)k * sizeof(int32_t));
        int32_t* me = (int32_t*)xmalloc((size_t)T * (size_t)k * sizeof(int32_t));
        int32_t* ms = (int32_t*)xmalloc((size_t)T * (size_t)k * sizeof(int32_t));
        for (int step = 0; step < 6; ++step) {
            const int n = 1 + (step * 7) % (T * k);
            int32_t nh, nm, nb;
            oracle_cache_step(c, ids, n, slot_of, me, ms, &nh, &nm, &nb);
        }
        int32_t* se = (int32_t*)xmalloc((size_t)S * sizeof(int32_t));
        uint32_t* cnt = (uint32_t*)xmalloc((size_t)S * sizeof(uint32_t));
        oracle_cache_dump(c, se, cnt);
        free(se); free(cnt); free(slot_of); free(me); free(ms); free(c);
    }
    int32_t* off = (int32_t*)xmalloc((size_t)(E + 1) * sizeof(int32_t));
    int32_t* pp = (int32_t*)xmalloc((size_t)T * (size_t)k * sizeof(int32_t));
    oracle_group_pairs(ids, T * k, E, off, pp);
    if (off[E] != T * k) return 4;
    free(off); free(pp);
    free(rc); free(rs); free(rb); free(sgc); free(sgs); free(sgb); free(suc); free(sus); free(sub);
    free(sdc); free(sds); free(sdb); free(gc); free(gs); free(gb); free(uc); free(us); free(ub);
    free(dc); free(ds); free(db); free(x); free(scratch); free(zb); free(perm); free(logits); free(ids);
    free(gates); free(y); free(yd);
    return 0;
}

int main(void) {
    /* d, E, k, I, I_shared, act, tokens */
    const int cases[][7] = {{512, 16, 2, 256, 512, 0, 4}, {256, 5, 3, 64, 128, 1, 3}, {256, 1, 1, 128, 64, 0, 2},
                            {512, 32, 32, 64, 64, 1, 2}};
    for (size_t i = 0; i < sizeof cases / sizeof cases[0]; ++i) {
        const int* c = cases[i];
        const int r = run(c[0], c[1], c[2], c[3], c[4], c[5], c[6]);
        if (r) {
            printf("case %zu failed (%d)\n", i, r);
            return 1;
        }
    }
    printf("oracle ok\n");
    return 0;
}
