// Fused expert FFN for the decode path (sm_103a): gate/up, activation, down
// and the gate-weighted combine of a set of experts in one launch.
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
//
// FFN_e(x) = W_down,e (act(W_gate,e x) * (W_up,e x)) ([P1] §2.4 cb2) over int4
// affine group-64 weights ([P1] §2.1, §2.5), fp32 accumulation, for every
// (token, rank) pair routed to each expert; then y[t] += sum_r g[t][r] o[t][r]
// added in rank order ([P1] §6.2.3 fusion of shared and weighted routed
// outputs; [P3] "每个 token、每层都要重新路由": y = sum_j w_j Expert_j(x)).
//
// Items come in two families: the shared expert (always resident, its pairs
// are tokens) and the routed experts; one launch covers both, so the shared
// expert runs while misses are still streaming.
//
// Work: jobs are (expert item, 32-row tile, K-chunk). All gate/up jobs come
// before all down jobs in the job order, and each CTA takes jobs j = blockIdx.x,
// blockIdx.x + gridDim.x, ..., so a CTA finishes its gate/up jobs before it
// starts a down job. The launch is cooperative (every CTA resident), so a down
// job may wait for its expert's gate/up jobs without deadlock: gate/up jobs
// wait only on copies, never on other jobs.
//
// Ready state ([P3] "读取完成后，算子才可以使用切片"): an expert whose bytes are
// still being copied into its slot carries the index of a ready flag and the
// call's round number; the copy stream writes the round number into the flag
// after the copy, and the producer waits for that value before it streams the
// expert's weights. A hit needs no wait. A flag left over from an earlier round
// holds an older number and is never mistaken for ready.
//
// Pipeline per CTA: warp kCons is the producer (one thread issues 1-D bulk
// copies of codes and (scale, bias) words into a kStages-deep shared-memory
// ring); warps 0..kCons-1 are consumers, warp w taking group w of each stage.
// Cross-warp and cross-CTA sums are added in fixed orders, so results do not
// depend on scheduling. Every wait is bounded and reports into an error word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kCons = 8;  // consumer warps
constexpr int kEpi = 2;   // epilogue warps
constexpr int kThreads = (kCons + 1 + kEpi) * 32;
constexpr int kStages = 3;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kRecord = 1152;  // one group of 64 inputs x 32 rows: codes, then scale/bias words
constexpr int kStageBytes = 2 * kCons * kRecord;  // gate+up stage; a down stage uses half
constexpr int kMaxSplitJobs = 1024;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float2 unpack_sb(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

// 4-bit codes to floats: code q at nibble position p of a word becomes the
// float 2^23 + q * 16^p via (word & (15 << 4p)) | 0x4B000000 (exact), and
// subtracting 2^23 leaves q * 16^p. Nibbles 5..7 are taken from the word
// shifted right by 12, so the positions used are p = 0,1,2,3,4,2,3,4.
__device__ __forceinline__ void codes8(uint32_t v, float2 (&o)[4]) {
    const uint32_t M = 0x4B000000u;
    const uint32_t w = v >> 12;
    const float2 off = make_float2(-8388608.0f, -8388608.0f);
    o[0] = __fadd2_rn(make_float2(__uint_as_float((v & 0xFu) | M), __uint_as_float((v & 0xF0u) | M)), off);
    o[1] = __fadd2_rn(make_float2(__uint_as_float((v & 0xF00u) | M), __uint_as_float((v & 0xF000u) | M)), off);
    o[2] = __fadd2_rn(make_float2(__uint_as_float((v & 0xF0000u) | M), __uint_as_float((w & 0xF00u) | M)), off);
    o[3] = __fadd2_rn(make_float2(__uint_as_float((w & 0xF000u) | M), __uint_as_float((w & 0xF0000u) | M)), off);
}

// 16^-p for input index k mod 8 (p = 0,1,2,3,4,2,3,4), as the power of two 2^(-4p).
__device__ __forceinline__ float pos_scale(int k8) {
    const int p = k8 < 5 ? k8 : k8 - 3;
    return __int_as_float((127 - 4 * p) << 23);
}

__device__ __forceinline__ float act_fn(float z, int act) {
    if (act == 1) return z / (1.0f + expf(-z));
    return 0.5f * z * (1.0f + tanhf(0.7978845608028654f * (z + 0.044715f * z * z * z)));
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *p == want (or, with at_least, *p >= want).
__device__ __forceinline__ bool wait_value(const uint32_t* p, uint32_t want, volatile int* abort) {
    if (ld_acquire(p) == want) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t i = 0;; ++i) {
        if (ld_acquire(p) == want) return true;
        __nanosleep(64);
        if ((i & 15) == 15) {
            if (abort && *abort) return false;
            if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) return false;
        }
    }
}

// a[f] for a two-entry array without a runtime-indexed (local-memory) access
template <class T>
__device__ __forceinline__ T sel(const T (&a)[2], int f) {
    return f ? a[1] : a[0];
}

struct Plan {
    int tiles_d;             // 32-row tiles of down (d)
    int G1;                  // groups of 64 along K of gate/up (d)
    int first[kFfnFams];     // first item of each family
    int tiles_i[kFfnFams];   // 32-row tiles of gate/up (inter)
    int G2[kFfnFams];        // groups along K of down (inter)
    int kc1[kFfnFams], kc2[kFfnFams], gpc1[kFfnFams], gpc2[kFfnFams];
    int tpj[kFfnFams], groups2[kFfnFams];  // down tiles per job, down jobs per (item, chunk)
    int jobs1[kFfnFams], jobs2[kFfnFams];
    int jobs1_total;
    size_t part1[kFfnFams], part2[kFfnFams];  // partial-sum region offsets (floats)
    int cnt1[kFfnFams];                       // split-K counter region offsets
};

template <int NT>
__device__ __forceinline__ Plan make_plan(const FfnArgs& a) {
    Plan p;
    p.tiles_d = a.d >> 5;
    p.G1 = a.d >> 6;
    int first = 0, jobs1 = 0;
    size_t off = 0;
    int c1 = 0;
    for (int f = 0; f < kFfnFams; ++f) {
        const FfnFam& F = a.fam[f];
        p.first[f] = first;
        p.tiles_i[f] = F.inter >> 5;
        p.G2[f] = F.inter >> 6;
        p.kc1[f] = F.kc1;
        p.kc2[f] = F.kc2;
        p.tpj[f] = F.tpj;
        p.gpc1[f] = (p.G1 + F.kc1 - 1) / F.kc1;
        p.gpc2[f] = (p.G2[f] + F.kc2 - 1) / F.kc2;
        p.groups2[f] = (p.tiles_d + F.tpj - 1) / F.tpj;
        p.jobs1[f] = F.n_items * p.tiles_i[f] * F.kc1;
        p.jobs2[f] = F.n_items * p.groups2[f] * F.kc2;
        jobs1 += p.jobs1[f];
        first += F.n_items;
        p.part1[f] = off;
        off += (size_t)F.n_items * p.tiles_i[f] * F.kc1 * NT * 2 * 32;
        p.cnt1[f] = c1;
        c1 += F.n_items * p.tiles_i[f];
    }
    for (int f = 0; f < kFfnFams; ++f) {
        p.part2[f] = off;
        off += (size_t)a.fam[f].n_items * p.tiles_d * a.fam[f].kc2 * NT * 32;
    }
    p.jobs1_total = jobs1;
    return p;
}

// A job: phase 1 is one gate/up row tile of one item over one K-chunk; phase 2
// is ntiles consecutive down row tiles of one item over one K-chunk.
struct Job {
    int phase, fam, item, local, rt0, ntiles, kc, g0, ng;
};

__device__ __forceinline__ Job decode_job(const Plan& p, int j) {
    Job b;
    b.phase = j < p.jobs1_total ? 1 : 2;
    if (b.phase == 2) j -= p.jobs1_total;
    b.fam = 0;
    const int jobs0 = b.phase == 1 ? p.jobs1[0] : p.jobs2[0];
    if (j >= jobs0) {
        j -= jobs0;
        b.fam = 1;
    }
    const int f = b.fam;
    const int units = b.phase == 1 ? sel(p.tiles_i, f) : sel(p.groups2, f);
    const int kc = b.phase == 1 ? sel(p.kc1, f) : sel(p.kc2, f);
    const int gpc = b.phase == 1 ? sel(p.gpc1, f) : sel(p.gpc2, f);
    const int G = b.phase == 1 ? p.G1 : sel(p.G2, f);
    const int per = units * kc;
    b.local = j / per;
    b.item = sel(p.first, f) + b.local;
    const int r = j - b.local * per;
    const int u = r / kc;
    b.kc = r - u * kc;
    if (b.phase == 1) {
        b.rt0 = u;
        b.ntiles = 1;
    } else {
        b.rt0 = u * sel(p.tpj, f);
        b.ntiles = min(sel(p.tpj, f), p.tiles_d - b.rt0);
    }
    b.g0 = b.kc * gpc;
    b.ng = min(gpc, G - b.g0);
    return b;
}

// Sum over one group (two 16-byte chunks of 32 codes each, for M matrices
// that share the same inputs) of q * x for NT rows of x; xs points at the
// group's 64 inputs of the first row, rows `stride` apart. Each (matrix, row)
// pair keeps two partial sums so the fused multiply-add chains stay short.
template <int NT, int M>
__device__ __forceinline__ void group_dot(const uint4 (&c0)[M], const uint4 (&c1)[M], const float* xs, int stride,
                                          float (&out)[M][NT]) {
    float2 acc[M][NT][2];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[m][j][0] = acc[m][j][1] = make_float2(0.0f, 0.0f);
    // with several rows of x, a full unroll would keep every word's activations
    // live at once; two words at a time keeps the register count in bounds
#pragma unroll(NT <= 2 ? 8 : 2)
    for (int w = 0; w < 8; ++w) {
        float2 q[M][4];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint4& c = w < 4 ? c0[m] : c1[m];
            const int k = w & 3;
            codes8(k == 0 ? c.x : k == 1 ? c.y : k == 2 ? c.z : c.w, q[m]);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float4* xp = reinterpret_cast<const float4*>(xs + j * stride + w * 8);
            const float4 a = xp[0], b = xp[1];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                acc[m][j][0] = __ffma2_rn(q[m][0], make_float2(a.x, a.y), acc[m][j][0]);
                acc[m][j][1] = __ffma2_rn(q[m][1], make_float2(a.z, a.w), acc[m][j][1]);
                acc[m][j][0] = __ffma2_rn(q[m][2], make_float2(b.x, b.y), acc[m][j][0]);
                acc[m][j][1] = __ffma2_rn(q[m][3], make_float2(b.z, b.w), acc[m][j][1]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float2 s = __fadd2_rn(acc[m][j][0], acc[m][j][1]);
            out[m][j] = s.x + s.y;
        }
}

// Release increment of a counter: orders this thread's earlier writes
// before the increment for any thread that later observes it with acquire.
__device__ __forceinline__ void red_release(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// The epilogue of one finished tile: cross-warp sums -> split-K partials or
// the final values -> h / out -> the counters that publish them -> the combine.
template <int NT, class L>
__device__ void tile_epilogue(const FfnArgs& a, const L& list, const Plan& P, const Job& b, int rt,
                              const float (&v_in)[2][NT], unsigned* cnt_t1, unsigned* cnt_t2, unsigned* gu_done,
                              unsigned* dn_done, unsigned* comb, unsigned long long* tr) {
    const int lane = threadIdx.x & 31;
    const FfnFam& F = a.fam[b.fam];
    const FfnItem& it = list.item[b.item];
    const int nt = it.np;
    const int mats = b.phase == 1 ? 2 : 1;
    const int kcn = b.phase == 1 ? sel(P.kc1, b.fam) : sel(P.kc2, b.fam);
    const int tiles = b.phase == 1 ? sel(P.tiles_i, b.fam) : P.tiles_d;
    const int tile_local = b.local * tiles + rt;  // within the family
    float v[2][NT];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int q = 0; q < NT; ++q) v[m][q] = v_in[m][q];
    bool finish = kcn == 1;
    if (!finish) {
        const int stride = NT * mats * 32;
        float* pbase = a.partials + (b.phase == 1 ? sel(P.part1, b.fam) : sel(P.part2, b.fam));
        float* pp = pbase + ((size_t)tile_local * kcn + b.kc) * stride;
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int q = 0; q < NT; ++q)
                if (m < mats) pp[(q * mats + m) * 32 + lane] = v[m][q];
        __threadfence();
        __syncwarp();
        unsigned prev = 0;
        unsigned* c = b.phase == 1 ? cnt_t1 + sel(P.cnt1, b.fam) + tile_local : cnt_t2 + b.item * P.tiles_d + rt;
        if (lane == 0) prev = atomicAdd(c, 1u);
        prev = __shfl_sync(kFull, prev, 0);
        finish = prev == (unsigned)(kcn - 1);
        if (!finish) return;
        __threadfence();
        const float* pt = pbase + (size_t)tile_local * kcn * stride;
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int q = 0; q < NT; ++q) {
                if (m >= mats) continue;
                float acc = 0.0f;
                for (int cc = 0; cc < kcn; ++cc) acc += __ldcg(pt + (size_t)cc * stride + (q * mats + m) * 32 + lane);
                v[m][q] = acc;
            }
        if (lane == 0) *c = 0;
    }
    if (b.phase == 1) {
#pragma unroll
        for (int q = 0; q < NT; ++q)
            if (q < nt) {
                const int p = list.pair[it.pb + q];
                F.h[(size_t)p * F.inter + rt * 32 + lane] = act_fn(v[0][q], a.act) * v[1][q];
            }
        __threadfence();  // each lane's h writes, visible GPU-wide before the count that publishes them
        __syncwarp();
        if (lane == 0) red_release(gu_done + b.item, 1u);
        if (tr && lane == 0) tr[2] = ptx::globaltimer();
        return;
    }
#pragma unroll
    for (int q = 0; q < NT; ++q)
        if (q < nt) {
            const int p = list.pair[it.pb + q];
            F.out[(size_t)p * a.d + rt * 32 + lane] = v[0][q];
        }
    __threadfence();  // each lane's outputs, visible GPU-wide before the counts that publish them
    __syncwarp();
    unsigned prev_d = 0, prev_c = 0;
    if (lane == 0) {
        prev_d = atomicAdd(dn_done + b.item, 1u);
        if (a.combine) prev_c = atom_add_acq_rel(comb + rt, 1u);
    }
    prev_d = __shfl_sync(kFull, prev_d, 0);
    prev_c = __shfl_sync(kFull, prev_c, 0);
    if (tr && lane == 0) tr[4] = ptx::globaltimer();
    if (prev_d == (unsigned)(P.tiles_d - 1) && lane == 0) {
        // every down tile of this item is done: nobody waits on its counters any more
        gu_done[b.item] = 0;
        dn_done[b.item] = 0;
    }
    if (a.combine && prev_c == (unsigned)(list.n_items - 1)) {
        // every item finished output tile rt: y[t] = base[t] + sum_r g[t][r] o[t*k + r], ranks in order
        __threadfence();
        const int n = rt * 32 + lane;
        const float* ro = a.fam[1].out;
        for (int t2 = 0; t2 < a.T; ++t2) {
            float acc = a.combine_base ? __ldcg(a.combine_base + (size_t)t2 * a.d + n) : a.y[(size_t)t2 * a.d + n];
            for (int r = 0; r < a.k; ++r)
                acc = fmaf(__ldg(a.gates + t2 * a.k + r), __ldcg(ro + ((size_t)t2 * a.k + r) * a.d + n), acc);
            a.y[(size_t)t2 * a.d + n] = acc;
        }
        if (lane == 0) comb[rt] = 0;
    }
}

template <int NT, class L>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 2 : 1) ffn_kernel(const __grid_constant__ FfnArgs a,
                                                                        const __grid_constant__ L list) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* red_full = empty + kStages;  // [2]: a tile's cross-warp partials are ready
    uint64_t* red_empty = red_full + 2;    // [2]: the epilogue warp has taken them
    const int xs_stride = a.xs_stride;     // staged inputs per warp and row
    const int cw_max = xs_stride / 64;     // groups per warp and job
    float* xsw = reinterpret_cast<float*>(red_empty + 2);  // [kCons][NT][xs_stride]
    float* xsumw = xsw + kCons * NT * xs_stride;            // [kCons][NT][cw_max]
    float* red = xsumw + kCons * NT * cw_max;              // [2][kCons][NT][2][32]
    int* meta = reinterpret_cast<int*>(red + 2 * kCons * NT * 2 * 32);  // [2][2]: job, tile
    __shared__ int abort_flag;
    __shared__ int staged_key[kCons][4 + kFfnMaxNT];  // per warp: (phase, family or item, g0, count, rows...)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Plan P = make_plan<NT>(a);
    const int n_jobs = P.jobs1_total + P.jobs2[0] + P.jobs2[1];

    // counters (all zero between launches): split-K arrivals per gate/up tile
    // (per family), per down tile, gate/up tiles done per item, down tiles
    // done per item, items done per output tile (for the combine)
    unsigned* cnt_t1 = a.counters;
    unsigned* cnt_t2 = cnt_t1 + P.cnt1[1] + a.fam[1].n_items * P.tiles_i[1];
    unsigned* gu_done = cnt_t2 + list.n_items * P.tiles_d;
    unsigned* dn_done = gu_done + list.n_items;
    unsigned* comb = dn_done + list.n_items;

    unsigned long long* tr = a.trace ? a.trace + (size_t)blockIdx.x * kFfnTracePoints : nullptr;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(full + i, 1);
            ptx::mbar_init(empty + i, kCons);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(red_full + i, kCons);
            ptx::mbar_init(red_empty + i, 1);
        }
        abort_flag = 0;
        ptx::fence_mbar_init();
        if (tr) {
            tr[0] = ptx::globaltimer();
            for (int i = 1; i < kFfnTracePoints; ++i) tr[i] = 0;
        }
    }
    if (threadIdx.x < kCons * 32 && lane == 0) staged_key[warp][0] = -1;
    __syncthreads();
    volatile int* abortp = &abort_flag;

    if (warp == kCons) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int slot = 0;
            uint32_t phase = 1;  // a fresh "empty" barrier counts as released
            int issued = 0;
            bool ok = true;
            int ready_item = -1;  // last item whose ready flag was confirmed
            for (int j = blockIdx.x; j < n_jobs && ok; j += gridDim.x) {
                const Job b = decode_job(P, j);
                const FfnItem& it = list.item[b.item];
                if (it.ready >= 0 && ready_item != b.item) {
                    if (!wait_value(a.ready + it.ready, list.epoch, abortp)) {
                        ok = false;
                        break;
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    ready_item = b.item;
                }
                const int inter = a.fam[b.fam].inter;
                const size_t mat = qmat_bytes(inter, a.d);  // bytes of one of gate, up, down
                const int two = b.phase == 1 ? 2 : 1;
                const int K = b.phase == 1 ? a.d : inter;
                const unsigned char* A = it.w + (b.phase == 1 ? 0 : 2 * mat);
                for (int t = 0; t < b.ntiles && ok; ++t) {
                    const int rt = b.rt0 + t;
                    const unsigned char* ra = A + (size_t)rt * (K >> 6) * kRecord;  // the row tile's records
                    // a gate/up stage holds kCons groups of both matrices, a down
                    // stage 2 kCons groups of one
                    const int gps = two == 2 ? kCons : 2 * kCons;
                    for (int s0 = 0; s0 < b.ng; s0 += gps) {
                        const int ng = min(gps, b.ng - s0);
                        const size_t g = (size_t)(b.g0 + s0);
                        if (!ptx::mbar_wait_bounded(empty + slot, phase, abortp)) {
                            ok = false;
                            break;
                        }
                        unsigned char* st = ring + slot * kStageBytes;
                        ptx::mbar_arrive_expect_tx(full + slot, (uint32_t)(two * ng * kRecord));
                        ptx::bulk_g2s(st, ra + g * kRecord, ng * kRecord, full + slot);
                        if (two == 2) ptx::bulk_g2s(st + kCons * kRecord, ra + mat + g * kRecord, ng * kRecord, full + slot);
                        ++issued;
                        if (++slot == kStages) {
                            slot = 0;
                            phase ^= 1;
                        }
                    }
                }
            }
            if (!ok) {
                atomicOr(a.err, 1u);
                abort_flag = 1;
                // Let every copy already issued land before the CTA can exit.
                // Round r of a slot is waited on by consumers with parity r & 1;
                // `phase` is (r & 1) ^ 1 for the round at `slot`.
                for (int i = 0; i < kStages && i < issued; ++i) {
                    int sl = slot - 1 - i;
                    uint32_t full_parity = phase ^ 1;
                    if (sl < 0) {
                        sl += kStages;
                        full_parity ^= 1;
                    }
                    ptx::mbar_wait_bounded(full + sl, full_parity, nullptr);
                }
            }
        }
        return;
    }

    if (warp > kCons) {
        // ---------------- epilogue warps ----------------
        // Epilogue warp e takes the tiles handed off through buffer e.
        const int e = warp - kCons - 1;
        for (uint32_t uses = 0;; ++uses) {
            // a warp-uniform decision: the tile epilogue uses full-warp shuffles
            if (!__all_sync(kFull, ptx::mbar_wait_bounded(red_full + e, uses & 1, abortp))) {
                if (lane == 0 && !*abortp) {
                    atomicOr(a.err, 8u);
                    abort_flag = 1;
                }
                break;
            }
            const int j = meta[e * 2], t = meta[e * 2 + 1];
            if (j < 0) break;
            const Job b = decode_job(P, j);
            const float* rb = red + e * (kCons * NT * 2 * 32);
            float v[2][NT];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int q = 0; q < NT; ++q) {
                    float acc = 0.0f;
#pragma unroll
                    for (int w = 0; w < kCons; ++w) acc += rb[((w * NT + q) * 2 + m) * 32 + lane];  // warp order
                    v[m][q] = acc;
                }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(red_empty + e);
            tile_epilogue<NT>(a, list, P, b, b.rt0 + t, v, cnt_t1, cnt_t2, gu_done, dn_done, comb, tr);
        }
        return;
    }

    // ---------------- consumers ----------------
    int slot = 0;
    uint32_t phase = 0;
    uint32_t handoffs = 0;  // tiles handed to the epilogue warps so far
    float* xme = xsw + warp * NT * xs_stride;
    float* xsme = xsumw + warp * NT * cw_max;
    int* key = staged_key[warp];
    auto handoff = [&](int j, int t, const float (&tot)[2][NT]) {
        const int rbuf = handoffs & 1;
        ++handoffs;
        // wait until the epilogue warp has taken this buffer's previous tile;
        // after an abort the epilogue warps may be gone, so hand off nothing
        if (!__all_sync(kFull, ptx::mbar_wait_bounded(red_empty + rbuf, (((handoffs - 1) >> 1) & 1) ^ 1, abortp))) {
            if (lane == 0 && !*abortp) {
                atomicOr(a.err, 16u);
                abort_flag = 1;
            }
            return;
        }
        float* rb = red + rbuf * (kCons * NT * 2 * 32);
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int q = 0; q < NT; ++q) rb[((warp * NT + q) * 2 + m) * 32 + lane] = tot[m][q];
        if (warp == 0 && lane == 0) {
            meta[rbuf * 2] = j;
            meta[rbuf * 2 + 1] = t;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(red_full + rbuf);
    };
    for (int j = blockIdx.x; j < n_jobs; j += gridDim.x) {
        const Job b = decode_job(P, j);
        const FfnFam& F = a.fam[b.fam];
        const FfnItem& it = list.item[b.item];
        const int nt = it.np;
        const int mats = b.phase == 1 ? 2 : 1;
        const int K = b.phase == 1 ? a.d : F.inter;
        if (b.phase == 2) {
            // h of this item must be complete: all its gate/up tiles done
            if (lane == 0 && !wait_value(gu_done + b.item, (uint32_t)sel(P.tiles_i, b.fam), abortp)) {
                atomicOr(a.err, 4u);
                abort_flag = 1;
            }
            if (tr && warp == 0 && lane == 0) tr[3] = ptx::globaltimer();
            __syncwarp();
        }
        // this warp's groups of the job (b.g0 + warp + kCons c), staged once per
        // job unless the same rows and range are already staged
        const int my_groups = b.ng > warp ? (b.ng - warp + kCons - 1) / kCons : 0;
        bool same = key[0] == b.phase && key[1] == (b.phase == 1 ? b.fam : b.item) && key[2] == b.g0 && key[3] == nt;
        for (int q = 0; q < nt && same; ++q) {
            const int p = list.pair[it.pb + q];
            same = key[4 + q] == (b.phase == 1 ? p / F.x_div : p);
        }
        if (!same) {
            for (int c = 0; c < my_groups; ++c) {
                const int g = b.g0 + warp + kCons * c;
                for (int q = 0; q < nt; ++q) {
                    const int p = list.pair[it.pb + q];
                    float v0, v1;
                    if (b.phase == 1) {
                        const size_t e = (size_t)(p / F.x_div) * K + (size_t)g * 64 + 2 * lane;
                        const uint32_t r = *reinterpret_cast<const uint32_t*>(a.x + e);
                        v0 = bf16_lo(r);
                        v1 = bf16_hi(r);
                    } else {
                        const size_t e = (size_t)p * K + (size_t)g * 64 + 2 * lane;
                        const float2 r = __ldcg(reinterpret_cast<const float2*>(F.h + e));
                        v0 = r.x;
                        v1 = r.y;
                    }
                    float sum = v0 + v1;
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
                    // elements 2m and 2m+1 of each run of 8 sit at nibbles m and 4+m of the code word
                    float* xo = xme + q * xs_stride + c * 64 + 8 * (lane >> 2);
                    const int m = lane & 3;
                    xo[m] = v0 * pos_scale(m);
                    xo[4 + m] = v1 * pos_scale(4 + m);
                    if (lane == 0) xsme[q * cw_max + c] = sum;
                }
            }
            if (lane == 0) {
                key[0] = b.phase;
                key[1] = b.phase == 1 ? b.fam : b.item;
                key[2] = b.g0;
                key[3] = nt;
                for (int q = 0; q < nt; ++q) {
                    const int p = list.pair[it.pb + q];
                    key[4 + q] = b.phase == 1 ? p / F.x_div : p;
                }
            }
            __syncwarp();
        }
        for (int t = 0; t < b.ntiles; ++t) {
            float tot[2][NT];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int q = 0; q < NT; ++q) tot[m][q] = 0.0f;
            const int gps = mats == 2 ? kCons : 2 * kCons;  // groups per stage
            for (int s0 = 0; s0 < b.ng; s0 += gps) {
                const bool active = s0 + warp < b.ng;
                const int c = s0 / kCons;  // this warp's staged group slot (down: c and c + 1)
                const bool ok = ptx::mbar_wait_bounded(full + slot, phase, abortp);
                if (tr && warp == 0 && lane == 0 && tr[1] == 0) tr[1] = ptx::globaltimer();
                if (!ok && lane == 0) {
                    atomicOr(a.err, 2u);
                    abort_flag = 1;
                }
                if (ok && active) {
                    const unsigned char* st = ring + slot * kStageBytes;
                    const float* xg = xme + c * 64;
                    const unsigned char* cb = st + warp * kRecord + lane * 16;  // this warp's record
                    const unsigned char* sbp = st + warp * kRecord + 1024 + lane * 4;
                    if (mats == 2) {
                        const uint4 c0[2] = {*reinterpret_cast<const uint4*>(cb),
                                             *reinterpret_cast<const uint4*>(cb + kCons * kRecord)};
                        const uint4 c1[2] = {*reinterpret_cast<const uint4*>(cb + 512),
                                             *reinterpret_cast<const uint4*>(cb + kCons * kRecord + 512)};
                        const float2 fg = unpack_sb(*reinterpret_cast<const uint32_t*>(sbp));
                        const float2 fu = unpack_sb(*reinterpret_cast<const uint32_t*>(sbp + kCons * kRecord));
                        float pr[2][NT];
                        group_dot<NT, 2>(c0, c1, xg, xs_stride, pr);
#pragma unroll
                        for (int q = 0; q < NT; ++q) {
                            const float xq = xsme[q * cw_max + c];
                            tot[0][q] += fmaf(fg.x, pr[0][q], fg.y * xq);
                            tot[1][q] += fmaf(fu.x, pr[1][q], fu.y * xq);
                        }
                    } else {
                        // this warp's groups of the stage: s0 + warp and s0 + kCons + warp
                        for (int hh = 0; hh < 2 && s0 + hh * kCons + warp < b.ng; ++hh) {
                            const unsigned char* cbh = cb + hh * kCons * kRecord;
                            const uint4 c0[1] = {*reinterpret_cast<const uint4*>(cbh)};
                            const uint4 c1[1] = {*reinterpret_cast<const uint4*>(cbh + 512)};
                            const float2 f = unpack_sb(*reinterpret_cast<const uint32_t*>(sbp + hh * kCons * kRecord));
                            float pr[1][NT];
                            group_dot<NT, 1>(c0, c1, xg + hh * 64, xs_stride, pr);
#pragma unroll
                            for (int q = 0; q < NT; ++q)
                                tot[0][q] += fmaf(f.x, pr[0][q], f.y * xsme[q * cw_max + c + hh]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(empty + slot);
                if (++slot == kStages) {
                    slot = 0;
                    phase ^= 1;
                }
            }
            handoff(j, t, tot);
        }
    }
    // tell both epilogue warps that no tiles follow
    float zero[2][NT];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int q = 0; q < NT; ++q) zero[m][q] = 0.0f;
    handoff(-1, 0, zero);
    handoff(-1, 0, zero);
    if (tr && warp == 0 && lane == 0) tr[5] = ptx::globaltimer();
}

int sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    }
    return n;
}

// Shared memory: ring, barriers, per-warp staged inputs (NT rows of
// `xs_stride` inputs plus group sums), the two hand-off buffers and their tags.
template <int NT>
size_t ffn_smem(int xs_stride) {
    return (size_t)kStages * kStageBytes + (2 * kStages + 4) * sizeof(uint64_t) +
           sizeof(float) * ((size_t)kCons * NT * xs_stride + (size_t)kCons * NT * (xs_stride / 64) +
                            2 * (size_t)kCons * NT * 2 * 32) +
           4 * sizeof(int);
}

// K-chunks of a row tile whose weights take `tile` bytes, aiming at jobs of
// about `target` bytes: at least one chunk, at most one per two groups, at
// least enough that a chunk's inputs fit the staged-input buffer (gmax
// groups), and no chunk empty (with gpc = ceil(G / kc) groups per chunk,
// ceil(G / gpc) chunks cover 0..G-1).
int choose_kc(int G, double tile, double target, int gmax) {
    int kc = std::max(1, (int)std::lround(tile / std::max(target, 1.0)));
    kc = std::min(kc, std::max(1, G / 2));
    kc = std::max(kc, (G + gmax - 1) / gmax);
    const int gpc = (G + kc - 1) / kc;
    return (G + gpc - 1) / gpc;
}

size_t partial_floats_for(const FfnArgs& a, int nt) {
    size_t f = 0;
    for (int i = 0; i < kFfnFams; ++i) {
        const FfnFam& F = a.fam[i];
        f += (size_t)F.n_items * (F.inter / 32) * F.kc1 * nt * 2 * 32;
        f += (size_t)F.n_items * (a.d / 32) * F.kc2 * nt * 32;
    }
    return f;
}

size_t counters_for(int d, int n_shared, int inter_shared, int n_routed, int inter_routed) {
    const int n = n_shared + n_routed;
    return (size_t)n_shared * (inter_shared / 32) + (size_t)n_routed * (inter_routed / 32) + (size_t)n * (d / 32) +
           2 * (size_t)n + (size_t)(d / 32);
}

// inputs one staged buffer may hold per row: 64 KB of smem over NT rows
constexpr int staged_inputs_cap(int nt) { return (64 * 1024 / 4) / nt; }

template <int NT, class L>
cudaError_t ffn_launch(FfnArgs a, const L& list, cudaStream_t s) {
    static int per_sm = 0;
    static size_t attr_smem = 0;
    const int gmax = staged_inputs_cap(NT) / 64;  // groups per K-chunk
    // K-splits sized so that gate/up fills about one wave; a split never covers
    // more than kMaxSplitJobs (tile, chunk) pairs, which bounds the partials
    const size_t worst = ffn_smem<NT>(((std::min(kMaxDModel / 64, gmax) + kCons - 1) / kCons) * 64);
    if (worst > attr_smem) {
        cudaError_t e = cudaFuncSetAttribute(ffn_kernel<NT, L>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)worst);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ffn_kernel<NT, L>, kThreads, worst);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        attr_smem = worst;
    }
    // Jobs sized by bytes: each phase's weight bytes spread over about one
    // wave of CTAs. Gate/up tiles are K-split only when a tile is well above
    // the target; down tiles are grouped (or, when large, K-split) per family.
    const int cap = std::min(per_sm * sms(), kMaxSplitJobs);
    double bytes1 = 0, bytes2 = 0;
    for (int f = 0; f < kFfnFams; ++f) {
        const double n = a.fam[f].n_items;
        bytes1 += n * (a.fam[f].inter / 32) * (double)(2 * 32) * a.d * 9 / 16;
        bytes2 += n * (a.d / 32) * (double)32 * a.fam[f].inter * 9 / 16;
    }
    const double target1 = bytes1 / cap, target2 = bytes2 / cap;
    int jobs = 0, stride = 64;
    for (int f = 0; f < kFfnFams; ++f) {
        FfnFam& F = a.fam[f];
        const double tile1 = 2.0 * 32 * a.d * 9 / 16, tile2 = 32.0 * F.inter * 9 / 16;
        F.kc1 = choose_kc(a.d / 64, tile1, target1, gmax);
        if (tile2 >= target2) {
            F.kc2 = choose_kc(F.inter / 64, tile2, target2, gmax);
            F.tpj = 1;
        } else {
            F.kc2 = choose_kc(F.inter / 64, 0.0, 1.0, gmax);
            F.tpj = std::max(1, std::min(a.d / 32, (int)std::lround(target2 / tile2)));
        }
        const int gpc1 = (a.d / 64 + F.kc1 - 1) / F.kc1, gpc2 = (F.inter / 64 + F.kc2 - 1) / F.kc2;
        // each consumer warp stages ceil(gpc / kCons) groups of a job
        stride = std::max({stride, (gpc1 + kCons - 1) / kCons * 64, (gpc2 + kCons - 1) / kCons * 64});
        jobs += F.n_items * (F.inter / 32) * F.kc1 + F.n_items * ((a.d / 32 + F.tpj - 1) / F.tpj) * F.kc2;
    }
    a.xs_stride = stride;
    if (partial_floats_for(a, NT) > a.partial_floats ||
        counters_for(a.d, a.fam[0].n_items, a.fam[0].inter, a.fam[1].n_items, a.fam[1].inter) > a.n_counters ||
        a.fam[0].n_items + a.fam[1].n_items != list.n_items || stride > (gmax + kCons - 1) / kCons * 64)
        return cudaErrorInvalidValue;
    const int grid = std::min(jobs, per_sm * sms());
    void* args[] = {&a, const_cast<L*>(&list)};
    return cudaLaunchCooperativeKernel((const void*)ffn_kernel<NT, L>, dim3(grid), dim3(kThreads), args,
                                       ffn_smem<NT>(stride), s);
}

}  // namespace

size_t ffn_max_partial_floats(int d, int n_shared, int inter_shared, int n_routed, int inter_routed) {
    // A phase's chunk count per tile is max(round(tile / target), ceil(G / gmax))
    // with target = phase bytes / at most kMaxSplitJobs CTAs and gmax >= 32
    // groups: summed over tiles, the first term is at most kMaxSplitJobs plus
    // a half per tile, the second at most ceil(G / 32) per tile.
    const size_t tiles1 = (size_t)n_shared * (inter_shared / 32) + (size_t)n_routed * (inter_routed / 32);
    const size_t tiles2 = (size_t)(n_shared + n_routed) * (d / 32);
    const size_t g1 = (size_t)(d / 64 + 31) / 32, g2 = (size_t)(std::max(inter_shared, inter_routed) / 64 + 31) / 32;
    return (tiles1 * (1 + g1) + kMaxSplitJobs) * kFfnMaxNT * 64 + (tiles2 * (1 + g2) + kMaxSplitJobs) * kFfnMaxNT * 32;
}

size_t ffn_max_counters(int d, int n_shared, int inter_shared, int n_routed, int inter_routed) {
    return counters_for(d, n_shared, inter_shared, n_routed, inter_routed);
}

template <class L>
cudaError_t launch_ffn(const FfnArgs& a, const L& list, cudaStream_t s) {
    if (list.n_items == 0) return cudaSuccess;
    int m = 0;
    for (int i = 0; i < list.n_items; ++i) m = std::max(m, (int)list.item[i].np);
    if (m <= 1) return ffn_launch<1>(a, list, s);
    if (m <= 2) return ffn_launch<2>(a, list, s);
    if (m <= 4) return ffn_launch<4>(a, list, s);
    if (m <= kFfnMaxNT) return ffn_launch<8>(a, list, s);
    return cudaErrorInvalidValue;
}

template cudaError_t launch_ffn<FfnSmall>(const FfnArgs&, const FfnSmall&, cudaStream_t);
template cudaError_t launch_ffn<FfnLarge>(const FfnArgs&, const FfnLarge&, cudaStream_t);

}  // namespace moe
