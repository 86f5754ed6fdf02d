// Fused expert FFN for the decode path (sm_103a): gate/up, activation, down
// and the gate-weighted sum into y of a set of experts in one launch.
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
//
// FFN_e(x) = W_down,e (act(W_gate,e x) * (W_up,e x)) ([P1] §2.4 cb2) over int4
// affine group-64 weights ([P1] §2.1, §2.5), fp32 accumulation, for every
// (token, rank) pair routed to each expert, and y[t] = shared(x_t) +
// sum_r g[t][r] FFN_{e_r}(x_t) ([P1] §6.2.3 fusion of the shared and the
// weighted routed outputs; [P3] "每个 token、每层都要重新路由": y = sum_j w_j
// Expert_j(x)).
//
// Work unit: 32 consecutive intermediate rows c of one item (an expert with
// up to kFfnMaxNT of its pairs). A unit computes its slice of h,
//   h_j = act(W_gate[j] . x) * (W_up[j] . x),   j = 32c .. 32c + 31,
// then multiplies the matching 32 columns of W_down by that slice and adds
// gate * partial into y with fp32 atomic adds (y is zero on entry). Units
// never wait on one another: a unit's down columns stream through the same
// shared-memory ring right behind its gate/up rows, and its h never leaves the
// SM. The down matrix is stored column-sliced so that those columns are one
// contiguous run of codes plus one of scales. The sum over units lands in y
// in whatever order the atomics arrive, so y can differ between calls in the
// last bits of fp32.
//
// Ready state ([P3] "读取完成后，算子才可以使用切片"): an expert whose bytes are
// still being copied into its slot carries the index of a ready flag and the
// call's round number; the copy stream writes the round number into the flag
// after the copy, and the producer waits for that value before it streams the
// expert's weights. A hit needs no wait. A flag left over from an earlier round
// holds an older number and is never mistaken for ready.
//
// Pipeline per CTA: warp kCons is the producer (one thread issues 1-D bulk
// copies into a kStages-deep ring); warps 0..kCons-1 are consumers. In a
// gate/up stage warp w takes group w (64 inputs) of both matrices; in a down
// stage it takes row tiles w, w + kCons, ... Cross-warp sums of a unit are
// added in warp order. Every wait is bounded and reports into an error word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRecord = 1152;                     // gate/up: 64 inputs x 32 rows of codes, then 32 scale/bias words
constexpr int kHalf = 512;                        // down: codes of 32 rows x 32 inputs
constexpr int kSbBlock = 128;                     // down: scale/bias words of 32 rows
constexpr int kBarCons = 1;                       // named barrier of the consumer warps
constexpr int kStageCap = 64 * 1024;              // bytes of staged inputs per CTA

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float2 unpack_sb(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

// 4-bit codes to floats without a conversion: the word masked to the nibble
// at position p, read as an fp32 bit pattern, is the subnormal q * 16^p *
// 2^-149 (exact; nibbles 0..5 lie in the mantissa field). The inputs it
// multiplies are staged as x * 2^(kStageExp - 4p), so the fused multiply-add
// forms q * x * 2^(kStageExp - 149) exactly before its one rounding, a normal
// number for any |q x| above 2^-77; the sums are scaled back by the exact
// power of two kDotUnscale. Nibbles 5..7 are taken from the word shifted
// right by 12, so the positions used are p = 0,1,2,3,4,2,3,4.
constexpr int kStageExp = 100;  // staged |x| may reach 2^27 before overflow
constexpr float kDotUnscale = 562949953421312.0f;  // 2^(149 - kStageExp) = 2^49

template <uint32_t kMask>
__device__ __forceinline__ float nibble_code(uint32_t v) {
    return __uint_as_float(v & kMask);
}

__device__ __forceinline__ void codes8(uint32_t v, float2 (&o)[4]) {
    // v >> 12 as the high word of v * 2^20: an integer multiply-add, which
    // runs beside the logic unit that the eight extractions keep busy
    const uint32_t w = __umulhi(v, 1u << 20);
    o[0] = make_float2(nibble_code<0xFu>(v), nibble_code<0xF0u>(v));
    o[1] = make_float2(nibble_code<0xF00u>(v), nibble_code<0xF000u>(v));
    o[2] = make_float2(nibble_code<0xF0000u>(v), nibble_code<0xF00u>(w));
    o[3] = make_float2(nibble_code<0xF000u>(w), nibble_code<0xF0000u>(w));
}

// The staging factor 2^(kStageExp - 4p) for slot s of a run of 8 (p = 0,1,2,3,4,2,3,4).
__device__ __forceinline__ float pos_scale(int s) {
    const int p = s < 5 ? s : s - 3;
    return __int_as_float((127 + kStageExp - 4 * p) << 23);
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

// Bounded wait until *p == want.
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

// Word w of C 16-byte chunks (C = 1 or 2), by selects rather than an indexed
// (local-memory) access when w is not a compile-time constant.
template <int C>
__device__ __forceinline__ uint32_t word_at(const uint4 (&c)[C], int w) {
    const uint4 v = (C == 1 || w < 4) ? c[0] : c[C - 1];
    const int k = w & 3;
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

// Sum over the 8 C code words of C chunks (8 inputs each, for M matrices that
// share the same inputs) of q * x for NT rows of x; xs points at the staged
// inputs of the first word of the first row, rows `stride` apart. Each
// (matrix, row) pair keeps two partial sums so the fused multiply-add chains
// stay short.
template <int NT, int M, int C>
__device__ __forceinline__ void words_dot(const uint4 (&c)[M][C], const float* xs, int stride,
                                          float (&out)[M][NT]) {
    constexpr int W = 4 * C;
    constexpr int A = 2;  // independent accumulators per (matrix, row); four measured no faster
    float2 acc[M][NT][A];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int u = 0; u < A; ++u) acc[m][j][u] = make_float2(0.0f, 0.0f);
    // with several rows of x, a full unroll would keep every word's activations
    // live at once; two words at a time keeps the register count in bounds
#pragma unroll(NT <= 2 ? W : 2)
    for (int w = 0; w < W; ++w) {
        float2 q[M][4];
#pragma unroll
        for (int m = 0; m < M; ++m) codes8(word_at<C>(c[m], w), q[m]);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const uint32_t xp = ptx::smem_addr(xs + j * stride + w * 8);
            const float4 a = ptx::lds_f4(xp), b = ptx::lds_f4(xp + 16);
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
            out[m][j] = (s.x + s.y) * kDotUnscale;
        }
}

// As words_dot for one matrix and one 16-byte chunk (32 inputs), with the
// position-scaled inputs already in registers (few rows of x only).
template <int NT>
__device__ __forceinline__ void chunk_dot_reg(const uint4 c, const float (&h)[NT][32], float (&out)[NT]) {
    float2 acc[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = make_float2(0.0f, 0.0f);
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float2 q[4];
        codes8(words[w], q);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float* x = h[j] + 8 * w;
            acc[j][0] = __ffma2_rn(q[0], make_float2(x[0], x[1]), acc[j][0]);
            acc[j][1] = __ffma2_rn(q[1], make_float2(x[2], x[3]), acc[j][1]);
            acc[j][0] = __ffma2_rn(q[2], make_float2(x[4], x[5]), acc[j][0]);
            acc[j][1] = __ffma2_rn(q[3], make_float2(x[6], x[7]), acc[j][1]);
        }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const float2 s = __fadd2_rn(acc[j][0], acc[j][1]);
        out[j] = (s.x + s.y) * kDotUnscale;
    }
}

// The weights of an item: its blob, or for a pair resolved on the device the
// slot holding its expert, or null when that expert is not resident (the
// unit is skipped). Reads what the router wrote: call after the wait for the
// previous kernel.
__device__ __forceinline__ const uint8_t* item_weights(const FfnArgs& a, const FfnItem& it, int pair) {
    if (it.w) return it.w;
    const int s = __ldg(a.slot_of + __ldg(a.ids + pair));
    return s >= 0 ? a.slots + (size_t)s * a.ebytes : nullptr;
}

struct Unit {
    int fam, item, c;  // family, item index in the list, 32-row slice of the intermediate dim
};

__device__ __forceinline__ Unit unit_of(const FfnArgs& a, int u) {
    Unit r;
    const int t0 = a.fam[0].inter >> 5;
    const int n0 = a.fam[0].n_items * t0;
    if (u < n0) {
        r.fam = 0;
        r.item = u / t0;
        r.c = u - r.item * t0;
    } else {
        u -= n0;
        const int t1 = a.fam[1].inter >> 5;
        const int li = u / t1;
        r.fam = 1;
        r.item = a.fam[0].n_items + li;
        r.c = u - li * t1;
    }
    return r;
}

// C consumer warps (8 or 16) and one producer warp per CTA.
template <int C>
struct Shape {
    static constexpr int kThreads = (C + 1) * 32;
    // ring depth: one CTA of 16 consumer warps per SM has room for five stages
    static constexpr int kStages = C >= 16 ? 5 : 4;
    static constexpr int kStageBytes = 2 * C * kRecord;  // gate/up stage: C groups of gate and of up
    static constexpr int kDnTiles = kStageBytes / (kHalf + kSbBlock);  // down row tiles a stage can hold
};

template <int NT, int C, class L>
__global__ void __launch_bounds__(Shape<C>::kThreads, (C <= 11 && NT == 1) ? 2 : 1)
    ffn_kernel(const __grid_constant__ FfnArgs a, const __grid_constant__ L list) {
    constexpr int kCons = C;
    constexpr int kStages = Shape<C>::kStages;
    constexpr int kStageBytes = Shape<C>::kStageBytes;
    constexpr int kDnTiles = Shape<C>::kDnTiles;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    const int xs_stride = a.xs_stride;  // staged inputs per warp and row (a multiple of 64)
    const int cpw = xs_stride / 64;     // staged groups per warp
    float* xsw = reinterpret_cast<float*>(empty + kStages);  // [kCons][NT][xs_stride], position-scaled x
    float* red = xsw + kCons * NT * xs_stride;               // [kCons][NT][2][32] per-warp gate/up sums
    float* hs = red + kCons * NT * 2 * 32;                   // [NT][32] position-scaled h of the unit
    float* xsumw = hs + NT * 32;                             // [kCons][NT][cpw] sums of staged groups
    float* hsum = xsumw + kCons * NT * cpw;                  // [NT] sums of the unit's h
    __shared__ int abort_flag;
    __shared__ int staged_key[kCons][2 + kFfnMaxNT];  // per warp: first group, rows, row indices

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G1 = a.d >> 6, tiles_d = a.d >> 5;
    const int n_units = a.fam[0].n_items * (a.fam[0].inter >> 5) + a.fam[1].n_items * (a.fam[1].inter >> 5);
    const int dn_stages = (tiles_d + kDnTiles - 1) / kDnTiles;
    const int dn_per = (tiles_d + dn_stages - 1) / dn_stages;  // down row tiles per stage

    unsigned long long* tr = a.trace ? a.trace + (size_t)blockIdx.x * kFfnTracePoints : nullptr;
    if (a.span && threadIdx.x == 0) atomicMin(a.span, (unsigned long long)ptx::globaltimer());
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(full + i, 1);
            ptx::mbar_init(empty + i, kCons);
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
    // the next kernel may start now: it waits for this one before it writes
    // anything this one reads
    ptx::pdl_launch_dependents();

    if (warp == kCons) {
        // this call's slot-table changes (by an otherwise idle lane), once the
        // launch that read the table has finished
        if (lane == 1 && blockIdx.x == 0 && a.n_upd > 0) {
            ptx::pdl_wait();
            for (int i = 0; i < a.n_upd; ++i) const_cast<int32_t*>(a.slot_of)[a.upd_expert[i]] = a.upd_slot[i];
        }
        // ---------------- producer ----------------
        if (lane == 0) {
            int slot = 0;
            uint32_t phase = 1;  // a fresh "empty" barrier counts as released
            int issued = 0;
            bool ok = true;
            int ready_gu = -1, ready_dn = -1;  // last items whose gate/up (down) flag was confirmed
            auto next_stage = [&](uint32_t bytes) -> unsigned char* {
                if (!ptx::mbar_wait_sleep(empty + slot, phase, abortp)) return nullptr;
                ptx::mbar_arrive_expect_tx(full + slot, bytes);
                return ring + slot * kStageBytes;
            };
            auto advance = [&]() {
                ++issued;
                if (++slot == kStages) {
                    slot = 0;
                    phase ^= 1;
                }
            };
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit un = unit_of(a, u);
                const FfnItem& it = list.item[un.item];
                if (!it.w) ptx::pdl_wait();  // the router's ids (a no-op once passed)
                const uint8_t* wts = item_weights(a, it, list.pair[it.pb]);
                if (!wts) continue;  // a miss: done by a later launch
                if (it.ready >= 0 && ready_gu != un.item) {
                    if (!wait_value(a.ready + it.ready, list.epoch, abortp)) {
                        ok = false;
                        break;
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    ready_gu = un.item;
                }
                const int inter = a.fam[un.fam].inter;
                const size_t mat = qmat_bytes(inter, a.d);  // bytes of each of gate, up, down
                // gate/up: row tile c of both matrices, kCons groups per stage
                const unsigned char* gw = wts + (size_t)un.c * G1 * kRecord;
                for (int s0 = 0; s0 < G1; s0 += kCons) {
                    const int ng = min(kCons, G1 - s0);
                    unsigned char* st = next_stage((uint32_t)(2 * ng * kRecord));
                    if (!st) {
                        ok = false;
                        break;
                    }
                    ptx::bulk_g2s(st, gw + (size_t)s0 * kRecord, ng * kRecord, full + slot);
                    ptx::bulk_g2s(st + kCons * kRecord, gw + mat + (size_t)s0 * kRecord, ng * kRecord, full + slot);
                    advance();
                }
                // down: input chunk c of every row tile, and the scale blocks of group c / 2
                if (ok && it.ready_dn >= 0 && ready_dn != un.item) {
                    if (!wait_value(a.ready + it.ready_dn, list.epoch, abortp)) {
                        ok = false;
                        break;
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    ready_dn = un.item;
                }
                const unsigned char* dn = wts + 2 * mat;
                const unsigned char* dc = dn + (size_t)un.c * tiles_d * kHalf;
                const unsigned char* ds = dn + down_codes_bytes(a.d, inter) + (size_t)(un.c >> 1) * tiles_d * kSbBlock;
                for (int r0 = 0; r0 < tiles_d && ok; r0 += dn_per) {
                    const int n = min(dn_per, tiles_d - r0);
                    unsigned char* st = next_stage((uint32_t)(n * (kHalf + kSbBlock)));
                    if (!st) {
                        ok = false;
                        break;
                    }
                    ptx::bulk_g2s(st, dc + (size_t)r0 * kHalf, n * kHalf, full + slot);
                    ptx::bulk_g2s(st + kDnTiles * kHalf, ds + (size_t)r0 * kSbBlock, n * kSbBlock, full + slot);
                    advance();
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

    // ---------------- consumers ----------------
    // Every consumer warp walks the same units and stages, whatever fails, so
    // the named barriers always see all of them.
    int slot = 0;
    uint32_t phase = 0;
    float* xme = xsw + warp * NT * xs_stride;
    float* xsme = xsumw + warp * NT * cpw;
    int* key = staged_key[warp];
    const int kchunk = a.kchunk;  // groups per staging pass, a multiple of kCons
    auto take_stage = [&]() -> const unsigned char* {
        // a sleeping wait: spinning would take issue slots from the warps
        // (of this and the other resident CTA) that have data to work on
        const bool ok = ptx::mbar_wait_sleep(full + slot, phase, abortp);
        if (tr && warp == 0 && lane == 0 && tr[1] == 0) tr[1] = ptx::globaltimer();
        if (!ok && lane == 0 && !*abortp) {
            atomicOr(a.err, 2u);
            abort_flag = 1;
        }
        return __all_sync(kFull, ok) ? ring + slot * kStageBytes : nullptr;
    };
    auto release_stage = [&]() {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty + slot);
        if (++slot == kStages) {
            slot = 0;
            phase ^= 1;
        }
    };
    bool first_unit = true;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit un = unit_of(a, u);
        const FfnItem& it = list.item[un.item];
        if (!it.w) {
            ptx::pdl_wait();  // the router's ids (a no-op once passed)
            if (!item_weights(a, it, list.pair[it.pb])) continue;  // the producer skips it too
        }
        const int nt = it.np;
        const int x_div = a.fam[un.fam].x_div;
        int row[NT];
#pragma unroll
        for (int q = 0; q < NT; ++q) row[q] = (q < nt ? list.pair[it.pb + q] : 0) / x_div;
        // ---- gate/up of rows 32c .. 32c+31 ----
        float tot[2][NT];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int q = 0; q < NT; ++q) tot[m][q] = 0.0f;
        // this warp's offsets within a stage, and its staged group of the pass
        const uint32_t cb0 = ptx::smem_addr(ring) + warp * kRecord + lane * 16;
        const uint32_t sb0 = ptx::smem_addr(ring) + warp * kRecord + 1024 + lane * 4;
        int g0 = 0, i = 0;  // first group of the current staging pass, and the stage's index in it
        for (int s0 = 0; s0 < G1; s0 += kCons, ++i) {
            if (s0 == g0 + kchunk) {
                g0 = s0;
                i = 0;
            }
            if (i == 0) {
                // this warp's groups of the pass, g0 + warp + kCons i, staged as
                // position-scaled fp32 unless the same rows and pass are staged already
                bool same = key[0] == g0 && key[1] == nt;
#pragma unroll
                for (int q = 0; q < NT; ++q) same = same && (q >= nt || key[2 + q] == row[q]);
                if (!same) {
                    const int gend = min(g0 + kchunk, G1);
                    const int ngw = gend > g0 + warp ? (gend - g0 - warp + kCons - 1) / kCons : 0;
#pragma unroll
                    for (int q = 0; q < NT; ++q) {
                        if (q >= nt) continue;
                        const uint16_t* xr = a.x + (size_t)row[q] * a.d + 2 * lane;
                        // up to 8 groups' loads in flight at once, then their sums and stores
                        for (int i0 = 0; i0 < ngw; i0 += 8) {
                            uint32_t r[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (i0 + j < ngw)
                                    r[j] = __ldg(reinterpret_cast<const uint32_t*>(xr + (size_t)(g0 + warp + kCons * (i0 + j)) * 64));
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                if (i0 + j >= ngw) continue;
                                const int i = i0 + j;
                                const float v0 = bf16_lo(r[j]), v1 = bf16_hi(r[j]);
                                float sum = v0 + v1;
#pragma unroll
                                for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
                                // elements 2m and 2m+1 of each run of 8 sit at nibbles m and 4+m of the code word
                                float* xo = xme + q * xs_stride + i * 64 + 8 * (lane >> 2);
                                const int m = lane & 3;
                                xo[m] = v0 * pos_scale(m);
                                xo[4 + m] = v1 * pos_scale(4 + m);
                                if (lane == 0) xsme[q * cpw + i] = sum;
                            }
                        }
                    }
                    if (lane == 0) {
                        key[0] = g0;
                        key[1] = nt;
#pragma unroll
                        for (int q = 0; q < NT; ++q)
                            if (q < nt) key[2 + q] = row[q];
                    }
                    __syncwarp();
                }
            }
            const unsigned char* st = take_stage();
            if (st && s0 + warp < G1) {
                const uint32_t so = (uint32_t)(st - ring);  // the stage's offset in the ring
                const uint32_t cb = cb0 + so, sbp = sb0 + so;
                const uint4 words[2][2] = {{ptx::lds_u4(cb), ptx::lds_u4(cb + 512)},
                                           {ptx::lds_u4(cb + kCons * kRecord), ptx::lds_u4(cb + kCons * kRecord + 512)}};
                const float2 fg = unpack_sb(ptx::lds_u32(sbp));
                const float2 fu = unpack_sb(ptx::lds_u32(sbp + kCons * kRecord));
                float pr[2][NT];
                words_dot<NT, 2, 2>(words, xme + i * 64, xs_stride, pr);
#pragma unroll
                for (int q = 0; q < NT; ++q) {
                    const float xq = ptx::lds_f32(ptx::smem_addr(xsme + q * cpw + i));
                    tot[0][q] += fmaf(fg.x, pr[0][q], fg.y * xq);
                    tot[1][q] += fmaf(fu.x, pr[1][q], fu.y * xq);
                }
            }
            release_stage();
        }
        // ---- h = act(gate) * up: cross-warp sums in warp order, warp q takes token q ----
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int q = 0; q < NT; ++q) red[((warp * NT + q) * 2 + m) * 32 + lane] = tot[m][q];
        ptx::named_sync(kBarCons, kCons * 32);
        if (warp < NT) {
            const int q = warp;
            float vg = 0.0f, vu = 0.0f;
#pragma unroll
            for (int w = 0; w < kCons; ++w) {
                vg += red[((w * NT + q) * 2 + 0) * 32 + lane];
                vu += red[((w * NT + q) * 2 + 1) * 32 + lane];
            }
            const float h = q < nt ? act_fn(vg, a.act) * vu : 0.0f;
            float sum = h;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
            // input lane of the down chunk: run lane / 8, element e = lane % 8 at slot e / 2 (+4 if odd)
            const int e = lane & 7;
            const int sl = (e >> 1) + 4 * (e & 1);
            hs[q * 32 + 8 * (lane >> 3) + sl] = h * pos_scale(sl);
            if (lane == 0) hsum[q] = sum;
        }
        ptx::named_sync(kBarCons, kCons * 32);
        if (tr && first_unit && warp == 0 && lane == 0) tr[2] = ptx::globaltimer();
        // ---- down: columns 32c .. 32c+31 of every row, added into y ----
        // y was zeroed by an earlier kernel on the stream: before the first
        // add, wait until the previous kernel (and so everything before it)
        // has finished
        if (first_unit) ptx::pdl_wait();
        // the gates were written by the router launch: read after the wait
        float gate[NT];
#pragma unroll
        for (int q = 0; q < NT; ++q)
            gate[q] = q < nt ? (un.fam == 0 ? 1.0f : __ldg(a.gates + list.pair[it.pb + q])) : 0.0f;
        constexpr bool kHReg = NT <= 2;  // h of the unit in registers for the whole down pass
        float hq[NT];
        float hr[kHReg ? NT : 1][32];
#pragma unroll
        for (int q = 0; q < NT; ++q) hq[q] = hsum[q];
        if (kHReg) {
#pragma unroll
            for (int q = 0; q < (kHReg ? NT : 1); ++q)
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(hs + q * 32 + j);
                    hr[q][j] = v.x;
                    hr[q][j + 1] = v.y;
                    hr[q][j + 2] = v.z;
                    hr[q][j + 3] = v.w;
                }
        }
        // this lane's output element of row tile 0 in each token's y row
        float* yq[NT];
#pragma unroll
        for (int q = 0; q < NT; ++q) yq[q] = a.y + (size_t)row[q] * a.d + lane;
        const uint32_t dc0 = ptx::smem_addr(ring) + lane * 16;
        const uint32_t ds0 = ptx::smem_addr(ring) + kDnTiles * kHalf + lane * 4;
        for (int r0 = 0; r0 < tiles_d; r0 += dn_per) {
            const int n = min(dn_per, tiles_d - r0);
            const unsigned char* st = take_stage();
            if (st) {
                const uint32_t so = (uint32_t)(st - ring);
                for (int i = warp; i < n; i += kCons) {
                    const uint4 words[1][1] = {{ptx::lds_u4(dc0 + so + i * kHalf)}};
                    const float2 f = unpack_sb(ptx::lds_u32(ds0 + so + i * kSbBlock));
                    float pr[1][NT];
                    if constexpr (kHReg) {
                        chunk_dot_reg<NT>(words[0][0], hr, pr[0]);
                    } else {
                        words_dot<NT, 1, 1>(words, hs, 32, pr);
                    }
                    const int col = 32 * (r0 + i);
#pragma unroll
                    for (int q = 0; q < NT; ++q)
                        if (q < nt) atomicAdd(yq[q] + col, gate[q] * fmaf(f.x, pr[0][q], f.y * hq[q]));
                }
            }
            release_stage();
        }
        if (tr && first_unit && warp == 0 && lane == 0) tr[3] = ptx::globaltimer();
        first_unit = false;
    }
    if (tr && warp == 0 && lane == 0) tr[4] = ptx::globaltimer();
    if (a.span && warp == 0 && lane == 0) atomicMax(a.span + 1, (unsigned long long)ptx::globaltimer());
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
// `xs_stride` inputs), the cross-warp sums, h, and the group and h sums.
template <int NT, int C>
size_t ffn_smem(int xs_stride) {
    return (size_t)Shape<C>::kStages * Shape<C>::kStageBytes + 2 * Shape<C>::kStages * sizeof(uint64_t) +
           sizeof(float) * ((size_t)C * NT * xs_stride + (size_t)C * NT * 64 + NT * 32 +
                            (size_t)C * NT * (xs_stride / 64) + NT);
}

// Staged groups per warp and pass: all of a row's when they fit kStageCap.
constexpr int groups_per_warp_cap(int nt, int c) { return kStageCap / (4 * 64 * nt * c); }

template <int NT, int C, class L>
cudaError_t ffn_launch(FfnArgs a, const L& list, cudaStream_t s, bool pdl) {
    constexpr int kThreads = Shape<C>::kThreads;
    const int cap = groups_per_warp_cap(NT, C);
    static bool attr = false;
    if (!attr) {
        const int worst = ffn_smem<NT, C>(std::min(cap, (kMaxDModel / 64 + C - 1) / C) * 64);
        cudaError_t e = cudaFuncSetAttribute(ffn_kernel<NT, C, L>, cudaFuncAttributeMaxDynamicSharedMemorySize, worst);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int G1 = a.d / 64;
    const int gpw = std::min((G1 + C - 1) / C, cap);
    a.xs_stride = gpw * 64;
    a.kchunk = gpw * C;
    int units = 0;
    for (int f = 0; f < kFfnFams; ++f) {
        if (a.fam[f].n_items && (a.fam[f].inter % 32 || a.fam[f].x_div < 1)) return cudaErrorInvalidValue;
        units += a.fam[f].n_items * (a.fam[f].inter / 32);
    }
    if (a.fam[0].n_items + a.fam[1].n_items != list.n_items || a.d % 256 || units == 0) return cudaErrorInvalidValue;
    // resident CTAs per SM at this launch's shared memory (cached per size)
    const size_t smem = ffn_smem<NT, C>(a.xs_stride);
    static size_t occ_smem[4] = {0, 0, 0, 0};
    static int occ_val[4] = {0, 0, 0, 0};
    int per_sm = 0;
    for (int i = 0; i < 4 && !per_sm; ++i)
        if (occ_smem[i] == smem) per_sm = occ_val[i];
    if (!per_sm) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ffn_kernel<NT, C, L>, kThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        for (int i = 3; i > 0; --i) {
            occ_smem[i] = occ_smem[i - 1];
            occ_val[i] = occ_val[i - 1];
        }
        occ_smem[0] = smem;
        occ_val[0] = per_sm;
    }
    const int grid = std::min(units, per_sm * sms());
    cudaLaunchAttribute la;
    const cudaLaunchConfig_t c = launch_config(dim3(grid), dim3(kThreads), smem, s, pdl, &la);
    return cudaLaunchKernelEx(&c, ffn_kernel<NT, C, L>, a, list);
}

}  // namespace

template <class L>
cudaError_t launch_ffn(const FfnArgs& a, const L& list, cudaStream_t s, bool pdl) {
    if (list.n_items == 0) return cudaSuccess;
    int m = 0;
    for (int i = 0; i < list.n_items; ++i) m = std::max(m, (int)list.item[i].np);
    // one row per item: 16 consumer warps (one CTA per SM); more rows need more
    // registers per thread than 17 warps leave (at most 96 when one SM
    // sub-partition holds five of them), and get 8
    if (m <= 1) return ffn_launch<1, 16>(a, list, s, pdl);
    if (m <= 2) return ffn_launch<2, 8>(a, list, s, pdl);
    if (m <= 4) return ffn_launch<4, 8>(a, list, s, pdl);
    if (m <= kFfnMaxNT) return ffn_launch<8, 8>(a, list, s, pdl);
    return cudaErrorInvalidValue;
}

template cudaError_t launch_ffn<FfnSmall>(const FfnArgs&, const FfnSmall&, cudaStream_t, bool);
template cudaError_t launch_ffn<FfnLarge>(const FfnArgs&, const FfnLarge&, cudaStream_t, bool);

}  // namespace moe
