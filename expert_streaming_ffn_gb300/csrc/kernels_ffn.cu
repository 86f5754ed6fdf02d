// Fused expert FFN for the decode path (sm_103a): gate/up, activation, down
// and the gate-weighted sum into y of a set of experts in one launch.
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
//
// FFN_e(x) = W_down,e (act(W_gate,e x) * (W_up,e x)) ([P1] §2.4 cb2) over int4
// affine group-64 weights ([P1] §2.1, §2.5), for every (token, rank) pair
// routed to each expert, and y[t] = shared(x_t) + sum_r g[t][r] FFN_{e_r}(x_t)
// ([P1] §6.2.3 fusion of the shared and the weighted routed outputs; [P3]
// "每个 token、每层都要重新路由": y = sum_j w_j Expert_j(x)).
//
// Work unit: 32 consecutive intermediate rows c of one item (an expert with
// up to kFfnMaxNT of its pairs). A unit computes its slice of h,
//   h_j = act(W_gate[j] . x) * (W_up[j] . x),   j = 32c .. 32c + 31,
// then multiplies the matching 32 columns of W_down by that slice and adds
// its gate-weighted share into y with fp32 atomic adds (y is zero on entry).
// Units never wait on one another: a unit's down columns stream through the
// same shared-memory ring right behind its gate/up rows, and its h never
// leaves the SM. The down matrix is stored column-sliced so that those
// columns are one contiguous run of codes plus one of scales. The sum over
// units lands in y in whatever order the atomics arrive, so y can differ
// between calls in the last bits of fp32.
//
// Dot products on the tensor cores, with the 4-bit codes exact. A word of 8
// codes masked into the mantissa of fp16 1024.0 gives, per 16-bit half,
// 1024 + q (nibble in bits 0-3) or 1024 + 16 q (nibble in bits 4-7): one
// logic op per two codes, no conversion and no rounding. Those halves are the
// A operand of mma.sync m16n8k16 (16 weight rows x 16 inputs); the B operand
// holds the token rows (8 columns: up to 8 tokens) in fp16, scaled per row by
// a power of two 2^s so that the largest magnitude lands in [2^14, 2^15), and
// divided by 16 where the codes carry the factor 16. The products are exact
// and accumulate in fp32. Per group of 64 inputs the accumulator starts at
// -1024 * (sum of the group's B values), which removes the offset, so it ends
// at sum_i q_i x~_i; the affine part is then s * that + b * sum_i x~_i, and
// 2^-s undoes the scaling. For the down projection the B operand is h in two
// fp16 parts, h~ = hi + lo (22 significant bits), in neighbouring columns.
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
#include <type_traits>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRecord = 1152;  // gate/up: 64 inputs x 32 rows of codes, then 32 scale/bias words
constexpr int kHalf = 512;     // down: codes of 32 rows x 32 inputs
constexpr int kSbBlock = 128;  // down: scale/bias words of 32 rows
constexpr int kBarCons = 1;    // named barrier of the consumer warps

__device__ __forceinline__ float2 unpack_sb(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

// Two codes as an fp16 pair: (w & mask) | 0x64006400.
__device__ __forceinline__ uint32_t magic_pair(uint32_t w, uint32_t mask) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(0x64006400u));
    return r;
}

// The 8 codes of a word (nibble i holds element [0,2,4,6,1,3,5,7][i] of its
// run of 8) as four fp16 pairs of consecutive elements: p[0] = elements 0,1
// as 1024 + q; p[1] = 2,3 as 1024 + 16 q; p[2] = 4,5 as 1024 + q; p[3] = 6,7
// as 1024 + 16 q.
__device__ __forceinline__ void codes16(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t w8 = w >> 8;
    p[0] = magic_pair(w, 0x000F000Fu);
    p[1] = magic_pair(w, 0x00F000F0u);
    p[2] = magic_pair(w8, 0x000F000Fu);
    p[3] = magic_pair(w8, 0x00F000F0u);
}

// d += A * B, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A * B + c, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, float c0, float c1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %10, %11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}

// 16 weight rows x 32 inputs: lane (g, t) = (lane / 4, lane % 4) brings word t
// (inputs 8t .. 8t+7) of rows g and g + 8; b is its 16-byte B fragment, the
// 8 inputs of column g at word t as [x0, x1, x2/16, x3/16, x4, x5, x6/16, x7/16].
// Two MMAs: inputs 8t + {0,1,2,3} of every t, then 8t + {4,5,6,7}. The
// accumulators start at (c0, c1) for the columns 2t, 2t + 1 of both rows.
__device__ __forceinline__ void dot16x32c(float (&d)[4], uint32_t wg, uint32_t wg8, const uint4& b, float c0,
                                          float c1) {
    uint32_t pg[4], ph[4];
    codes16(wg, pg);
    codes16(wg8, ph);
    mma_f16c(d, pg[0], ph[0], pg[1], ph[1], b.x, b.y, c0, c1);
    mma_f16(d, pg[2], ph[2], pg[3], ph[3], b.z, b.w);
}
__device__ __forceinline__ void dot16x32(float (&d)[4], uint32_t wg, uint32_t wg8, const uint4& b) {
    uint32_t pg[4], ph[4];
    codes16(wg, pg);
    codes16(wg8, ph);
    mma_f16(d, pg[0], ph[0], pg[1], ph[1], b.x, b.y);
    mma_f16(d, pg[2], ph[2], pg[3], ph[3], b.z, b.w);
}

// Four 8x8 matrices of 16-bit elements (rows of 16 bytes; lanes 8j..8j+7 give
// the row addresses of matrix j): lane (g, t) receives word t of row g of
// each, i.e. the MMA fragment words of 8 weight rows per matrix.
template <int OFF>
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4+%5];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr), "n"(OFF)
                 : "memory");
}
template <int OFF>
__device__ __forceinline__ uint4 lds4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4+%5];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr), "n"(OFF)
                 : "memory");
    return v;
}

// 2^e as a float (|e| <= 126).
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// The power of two that brings a largest magnitude m (m >= 0, as fp32 bits)
// into [2^14, 2^15): fp16 then holds every value, below 65504.
__device__ __forceinline__ int range_shift(uint32_t mbits) {
    if (mbits == 0) return 0;
    const int e = (int)(mbits >> 23) - 127;  // floor(log2 m) for normal m
    return max(-100, min(100, 14 - e));
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
    // ring depth: one CTA of 16 consumer warps per SM has room for five stages
    static constexpr int kStages = C >= 16 ? 5 : 4;
    static constexpr int kStageBytes = 2 * C * kRecord;  // gate/up stage: C groups of gate and of up
    static constexpr int kDnTiles = kStageBytes / (kHalf + kSbBlock);  // down row tiles a stage can hold
};

// Shared memory after the ring and its barriers, for d_model d:
//   xs   [NT][2d + 64 bytes]   token rows as B fragments (fp16), rows 64 bytes
//                              apart modulo 128 so that a warp's loads of
//                              eight rows meet no bank conflict
//   kx   [d/64][4] float4      per group and lane t: -1024 * B sum and the
//                              sum of x~ for tokens 2t and 2t+1
//   red  [C][2][32][NT] f32    per-warp gate and up sums of the unit
//   hb   [NPASS][8][4] uint4   B fragments of the unit's h (hi, lo columns)
//   kh   [8] float4            per token: -1024 * B sum of hi, of lo, the
//                              sum of h~ times 2^-s, and 2^-s
//   wmax [C][NT] u32           per-warp largest |x| (bf16 magnitude bits)
//   xinv [NT] f32              2^-s of each staged token row
template <int NT, int C>
struct Smem {
    static constexpr int kPass = (NT + 3) / 4;
    static constexpr size_t ring = (size_t)Shape<C>::kStages * Shape<C>::kStageBytes + 16 * Shape<C>::kStages;
    static __host__ __device__ size_t xstride(int d) { return 2 * (size_t)d + 64; }
    static __host__ __device__ size_t xs(int) { return ring; }
    static __host__ __device__ size_t kx(int d) { return xs(d) + NT * xstride(d); }
    static __host__ __device__ size_t red(int d) { return kx(d) + (size_t)(d / 64) * 64; }
    static __host__ __device__ size_t hb(int d) { return red(d) + (size_t)C * 2 * 32 * NT * 4; }
    static __host__ __device__ size_t kh(int d) { return hb(d) + (size_t)kPass * 512; }
    static __host__ __device__ size_t wmax(int d) { return kh(d) + 8 * 16; }
    static __host__ __device__ size_t xinv(int d) { return wmax(d) + (size_t)C * NT * 4; }
    static __host__ __device__ size_t total(int d) { return xinv(d) + NT * 4; }
};

// Stages the unit's token rows (rows row[0..nt-1] of x) as B fragments, with
// the per-group sums, for every consumer thread (tid < 32 C). Pass 1 copies
// the raw bf16 rows into shared memory and finds each row's largest
// magnitude; pass 2 converts in place to fp16 at the row's scale.
template <int NT, int C>
__device__ __forceinline__ void stage_rows(const FfnArgs& a, const int (&row)[NT], int nt, unsigned char* smem,
                                           int warp, int lane) {
    using S = Smem<NT, C>;
    const int d = a.d, nf = d >> 3;  // 16-byte fragments per row
    const size_t xstride = S::xstride(d);
    unsigned char* xs = smem + S::xs(d);
    float* kx = reinterpret_cast<float*>(smem + S::kx(d));
    uint32_t* wmax = reinterpret_cast<uint32_t*>(smem + S::wmax(d));
    float* xinv = reinterpret_cast<float*>(smem + S::xinv(d));
    const int tid = warp * 32 + lane;
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        if (q >= nt) continue;
        const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)row[q] * d);
        const uint32_t dst = ptx::smem_addr(xs + q * xstride);
        uint32_t m2 = 0;  // two bf16 magnitudes, maxed lane-wise
        for (int f = tid; f < nf; f += 32 * C) {
            const uint4 v = __ldg(src + f);
            ptx::sts_u4(dst + 16 * f, v);
            m2 = __vmaxu2(m2, v.x & 0x7fff7fffu);
            m2 = __vmaxu2(m2, v.y & 0x7fff7fffu);
            m2 = __vmaxu2(m2, v.z & 0x7fff7fffu);
            m2 = __vmaxu2(m2, v.w & 0x7fff7fffu);
        }
        uint32_t m = max(m2 & 0xffffu, m2 >> 16);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(kFull, m, off));
        if (lane == 0) wmax[warp * NT + q] = m;
    }
    ptx::named_sync(kBarCons, C * 32);
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        if (q >= nt) continue;
        uint32_t m = 0;
        for (int w = 0; w < C; ++w) m = max(m, wmax[w * NT + q]);
        const int sh = range_shift(m << 16);  // bf16 bits -> fp32 bits
        const float sc = exp2i(sh), sc16 = exp2i(sh - 4);
        if (tid == 0) xinv[q] = exp2i(-sh);
        const uint32_t base = ptx::smem_addr(xs + q * xstride);
        // one fragment per lane; the 8 fragments of a group sit in 8 neighbouring lanes
        for (int f0 = warp * 32; f0 < nf; f0 += 32 * C) {
            const int f = f0 + lane;
            float bsum = 0.0f, xsum = 0.0f;
            if (f < nf) {
                const uint4 v = ptx::lds_u4(base + 16 * f);
                const uint32_t in[4] = {v.x, v.y, v.z, v.w};
                uint32_t out[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // slots 2j, 2j+1; slots 2,3 and 6,7 (j odd) carry the factor 1/16
                    const float lo = __uint_as_float(in[j] << 16), hi = __uint_as_float(in[j] & 0xffff0000u);
                    const float s = (j & 1) ? sc16 : sc;
                    const __half2 h = __floats2half2_rn(lo * s, hi * s);
                    const float2 hf = __half22float2(h);
                    bsum += hf.x + hf.y;
                    xsum += (j & 1) ? 16.0f * (hf.x + hf.y) : hf.x + hf.y;
                    out[j] = *reinterpret_cast<const uint32_t*>(&h);
                }
                ptx::sts_u4(base + 16 * f, make_uint4(out[0], out[1], out[2], out[3]));
            }
#pragma unroll
            for (int off = 4; off >= 1; off >>= 1) {
                bsum += __shfl_xor_sync(kFull, bsum, off);
                xsum += __shfl_xor_sync(kFull, xsum, off);
            }
            if (f < nf && (f & 7) == 0) {
                float* e = kx + ((f >> 3) * 4 + (q >> 1)) * 4 + (q & 1);
                e[0] = -1024.0f * bsum;
                e[2] = xsum;
            }
        }
    }
}

template <int NT, int C, class L>
__global__ void __launch_bounds__(Shape<C>::kThreads, 1)
    ffn_kernel(const __grid_constant__ FfnArgs a, const __grid_constant__ L list) {
    constexpr int kCons = C;
    constexpr int kStages = Shape<C>::kStages;
    constexpr int kStageBytes = Shape<C>::kStageBytes;
    constexpr int kDnTiles = Shape<C>::kDnTiles;
    using S = Smem<NT, C>;
    constexpr int kPass = S::kPass;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    __shared__ int abort_flag;
    __shared__ int staged_key[1 + kFfnMaxNT];  // rows staged in xs: count, then row indices

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G1 = a.d >> 6, tiles_d = a.d >> 5;
    const int n_units = a.fam[0].n_items * (a.fam[0].inter >> 5) + a.fam[1].n_items * (a.fam[1].inter >> 5);
    const int dn_stages = (tiles_d + kDnTiles - 1) / kDnTiles;
    const int dn_per = (tiles_d + dn_stages - 1) / dn_stages;  // down row tiles per stage
    // This CTA's units: round robin for one token (every SM streams in the
    // first wave); for several, a contiguous run, so that consecutive units
    // share an item and the token rows it staged (measured 12 % faster at 8
    // tokens, 5 % slower at one)
    const int per_cta = NT == 1 ? 1 : (n_units + gridDim.x - 1) / gridDim.x;
    const int u_begin = NT == 1 ? (int)blockIdx.x : (int)blockIdx.x * per_cta;
    const int u_end = NT == 1 ? n_units : min(n_units, u_begin + per_cta);
    const int u_step = NT == 1 ? (int)gridDim.x : 1;

    unsigned long long* tr = a.trace ? a.trace + (size_t)blockIdx.x * kFfnTracePoints : nullptr;
    if (a.span && threadIdx.x == 0) atomicMin(a.span, (unsigned long long)ptx::globaltimer());
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(full + i, 1);
            ptx::mbar_init(empty + i, kCons);
        }
        abort_flag = 0;
        staged_key[0] = -1;
        ptx::fence_mbar_init();
        if (tr) {
            tr[0] = ptx::globaltimer();
            for (int i = 1; i < kFfnTracePoints; ++i) tr[i] = 0;
        }
    }
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
            for (int u = u_begin; u < u_end && ok; u += u_step) {
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
    const int g = lane >> 2, t = lane & 3;  // MMA fragment coordinates
    // this lane's ldmatrix row in a gate/up record: matrix lane / 8 is (chunk
    // lane / 16, rows 0-7 or 8-15), row lane % 8 of it
    const uint32_t lm_off = (lane >> 4) * 512 + ((lane >> 3) & 1) * 128 + (lane & 7) * 16;
    const size_t xstride = S::xstride(a.d);
    const uint32_t xs_a = ptx::smem_addr(smem + S::xs(a.d));
    const uint32_t kx_a = ptx::smem_addr(smem + S::kx(a.d));
    float* red = reinterpret_cast<float*>(smem + S::red(a.d));
    unsigned char* hb = smem + S::hb(a.d);
    float4* kh = reinterpret_cast<float4*>(smem + S::kh(a.d));
    const float* xinv = reinterpret_cast<const float*>(smem + S::xinv(a.d));
    int slot = 0;
    uint32_t phase = 0;
    auto take_stage = [&]() -> const unsigned char* {
        // a sleeping wait: spinning would take issue slots from the warps
        // that have data to work on
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
    for (int u = u_begin; u < u_end; u += u_step) {
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
        // ---- the unit's token rows as B fragments, unless staged already ----
        {
            bool same = staged_key[0] == nt;
#pragma unroll
            for (int q = 0; q < NT; ++q) same = same && (q >= nt || staged_key[1 + q] == row[q]);
            if (!same) {
                stage_rows<NT, C>(a, row, nt, smem, warp, lane);
                if (warp == 0 && lane == 0) {
                    staged_key[0] = nt;
#pragma unroll
                    for (int q = 0; q < NT; ++q)
                        if (q < nt) staged_key[1 + q] = row[q];
                }
                ptx::named_sync(kBarCons, kCons * 32);
            }
        }
        // ---- gate/up of rows 32c .. 32c+31 ----
        // tot[m][rb][.]: matrix m, rows 16 rb + g (0, 1) and 16 rb + g + 8
        // (2, 3), tokens 2t (0, 2) and 2t + 1 (1, 3)
        float tot[2][2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int rb = 0; rb < 2; ++rb)
#pragma unroll
                for (int v = 0; v < 4; ++v) tot[m][rb][v] = 0.0f;
        const uint32_t xrow = xs_a + (uint32_t)(min(g, nt - 1) * xstride) + t * 16;
        for (int s0 = 0; s0 < G1; s0 += kCons) {
            const unsigned char* st = take_stage();
            const int grp = s0 + warp;
            if (st && grp < G1) {
                // this warp's gate and up records: the code words of rows
                // 16 rb + g and 16 rb + g + 8 of both chunks (ldmatrix), and
                // the scale words of rows g, g + 8, g + 16, g + 24
                const uint32_t rec = ptx::smem_addr(st) + warp * kRecord;
                uint32_t wd[2][2][4];
                uint4 sbv[2];
                ldsm4<0>(rec + lm_off, wd[0][0]);
                ldsm4<256>(rec + lm_off, wd[0][1]);
                ldsm4<kCons * kRecord>(rec + lm_off, wd[1][0]);
                ldsm4<kCons * kRecord + 256>(rec + lm_off, wd[1][1]);
                sbv[0] = lds4<1024>(rec + 16 * g);
                sbv[1] = lds4<kCons * kRecord + 1024>(rec + 16 * g);
                const uint32_t xa = xrow + grp * 128;
                const uint4 xb0 = lds4<0>(xa), xb1 = lds4<64>(xa);
                const float4 k4 = ptx::lds_f4(kx_a + (grp * 4 + t) * 16);  // -K(2t), -K(2t+1), X(2t), X(2t+1)
#pragma unroll
                for (int m = 0; m < 2; ++m) {
#pragma unroll
                    for (int rb = 0; rb < 2; ++rb) {
                        float dd[4];
                        dot16x32c(dd, wd[m][rb][0], wd[m][rb][1], xb0, k4.x, k4.y);
                        dot16x32(dd, wd[m][rb][2], wd[m][rb][3], xb1);
                        const float2 f0 = unpack_sb(rb ? sbv[m].z : sbv[m].x);
                        const float2 f1 = unpack_sb(rb ? sbv[m].w : sbv[m].y);
                        tot[m][rb][0] = fmaf(f0.x, dd[0], fmaf(f0.y, k4.z, tot[m][rb][0]));
                        tot[m][rb][2] = fmaf(f1.x, dd[2], fmaf(f1.y, k4.z, tot[m][rb][2]));
                        if (NT > 1) {
                            tot[m][rb][1] = fmaf(f0.x, dd[1], fmaf(f0.y, k4.w, tot[m][rb][1]));
                            tot[m][rb][3] = fmaf(f1.x, dd[3], fmaf(f1.y, k4.w, tot[m][rb][3]));
                        }
                    }
                }
            }
            release_stage();
        }
        // ---- h = act(gate) * up: cross-warp sums in warp order, warp q takes token q ----
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int rb = 0; rb < 2; ++rb)
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int tok = 2 * t + (v & 1);
                    const int r = 16 * rb + g + 8 * (v >> 1);
                    if ((NT > 1 || (v & 1) == 0) && tok < nt) red[((warp * 2 + m) * 32 + r) * NT + tok] = tot[m][rb][v];
                }
        ptx::named_sync(kBarCons, kCons * 32);
        if (warp < nt) {
            const int q = warp;
            float vg = 0.0f, vu = 0.0f;
#pragma unroll
            for (int w = 0; w < kCons; ++w) {
                vg += red[((w * 2 + 0) * 32 + lane) * NT + q];
                vu += red[((w * 2 + 1) * 32 + lane) * NT + q];
            }
            float gw = 1.0f;
            if (un.fam != 0) {
                ptx::pdl_wait();  // the gates were written by the router launch
                gw = __ldg(a.gates + list.pair[it.pb + q]);
            }
            const float xi = xinv[q];
            const float h = act_fn(vg * xi, a.act) * (vu * xi) * gw;
            const int sh = range_shift(__reduce_max_sync(kFull, __float_as_uint(fabsf(h))));
            const float ht = h * exp2i(sh);
            const __half hi = __float2half_rn(ht);
            const __half lo = __float2half_rn(ht - __half2float(hi));
            const int e = lane & 7;
            const bool scaled = (e & 2) != 0;  // slots 2, 3, 6, 7 carry the factor 1/16
            const __half bhi = scaled ? __float2half_rn(__half2float(hi) * 0.0625f) : hi;
            const __half blo = scaled ? __float2half_rn(__half2float(lo) * 0.0625f) : lo;
            // column 2 (q % 4) holds hi, the next one lo, in pass q / 4
            __half* frag = reinterpret_cast<__half*>(hb) + (((q >> 2) * 8 + 2 * (q & 3)) * 4 + (lane >> 3)) * 8 + e;
            frag[0] = bhi;
            frag[32] = blo;  // next column: 4 fragments of 8 halves further
            float shi = __half2float(bhi), slo = __half2float(blo), hs = __half2float(hi) + __half2float(lo);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                shi += __shfl_xor_sync(kFull, shi, off);
                slo += __shfl_xor_sync(kFull, slo, off);
                hs += __shfl_xor_sync(kFull, hs, off);
            }
            if (lane == 0) kh[q] = make_float4(-1024.0f * shi, -1024.0f * slo, hs * exp2i(-sh), exp2i(-sh));
        }
        ptx::named_sync(kBarCons, kCons * 32);
        if (tr && first_unit && warp == 0 && lane == 0) tr[2] = ptx::globaltimer();
        // ---- down: columns 32c .. 32c+31 of every row, added into y ----
        // y was zeroed by an earlier kernel on the stream: before the first
        // add, wait until the previous kernel (and so everything before it)
        // has finished
        if (first_unit) ptx::pdl_wait();
        uint4 hbv[kPass];
        float4 khv[kPass];
        float* yp[kPass];  // this lane's output row: y, or the unit's partial row
        const bool ordered = a.part[un.fam] != nullptr;
#pragma unroll
        for (int p = 0; p < kPass; ++p) {
            hbv[p] = ptx::lds_u4(ptx::smem_addr(hb) + ((p * 8 + g) * 4 + t) * 16);
            const int tok = 4 * p + t;
            khv[p] = kh[tok];
            yp[p] = nullptr;
            if (tok < nt) {
                const int pv = list.pair[it.pb + tok];
                yp[p] = ordered ? a.part[un.fam] + ((size_t)pv * a.part_c[un.fam] + un.c) * a.d
                                : a.y + (size_t)(pv / x_div) * a.d;
            }
        }
        // (two copies of the loop: adds into y, or stores into partial rows)
        auto down = [&](auto ordered_c) {
            constexpr bool kOrdered = decltype(ordered_c)::value;
            for (int r0 = 0; r0 < tiles_d; r0 += dn_per) {
                const int n = min(dn_per, tiles_d - r0);
                const unsigned char* st = take_stage();
                if (st) {
                    const uint32_t so = ptx::smem_addr(st);
                    for (int i = warp; i < n; i += kCons) {
                        // rows 0-7, 8-15, 16-23, 24-31 of the tile: 16 bytes per row
                        uint32_t wd[4];
                        ldsm4<0>(so + i * kHalf + lane * 16, wd);
                        const uint4 sbv = lds4<0>(so + kDnTiles * kHalf + i * kSbBlock + 16 * g);
#pragma unroll
                        for (int rb = 0; rb < 2; ++rb) {
                            uint32_t pg[4], ph[4];
                            codes16(wd[2 * rb], pg);
                            codes16(wd[2 * rb + 1], ph);
                            const float2 f0 = unpack_sb(rb ? sbv.z : sbv.x);
                            const float2 f1 = unpack_sb(rb ? sbv.w : sbv.y);
                            const int col = 32 * (r0 + i) + 16 * rb + g;
#pragma unroll
                            for (int p = 0; p < kPass; ++p) {
                                float dd[4];
                                mma_f16c(dd, pg[0], ph[0], pg[1], ph[1], hbv[p].x, hbv[p].y, khv[p].x, khv[p].y);
                                mma_f16(dd, pg[2], ph[2], pg[3], ph[3], hbv[p].z, hbv[p].w);
                                if (yp[p]) {
                                    const float v0 = fmaf(f0.x * khv[p].w, dd[0] + dd[1], f0.y * khv[p].z);
                                    const float v1 = fmaf(f1.x * khv[p].w, dd[2] + dd[3], f1.y * khv[p].z);
                                    if constexpr (kOrdered) {
                                        __stcg(yp[p] + col, v0);
                                        __stcg(yp[p] + col + 8, v1);
                                    } else {
                                        atomicAdd(yp[p] + col, v0);
                                        atomicAdd(yp[p] + col + 8, v1);
                                    }
                                }
                            }
                        }
                    }
                }
                release_stage();
            }
        };
        if (ordered)
            down(std::true_type{});
        else
            down(std::false_type{});
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

template <int NT, int C>
size_t ffn_smem(int d) {
    return Smem<NT, C>::total(d);
}

template <int NT, int C, class L>
cudaError_t ffn_launch(FfnArgs a, const L& list, cudaStream_t s, bool pdl) {
    constexpr int kThreads = Shape<C>::kThreads;
    cudaError_t e = ensure_smem_attr((const void*)ffn_kernel<NT, C, L>, ffn_smem<NT, C>(kMaxDModel));
    if (e != cudaSuccess) return e;
    int units = 0;
    for (int f = 0; f < kFfnFams; ++f) {
        if (a.fam[f].n_items && (a.fam[f].inter % 32 || a.fam[f].x_div < 1)) return cudaErrorInvalidValue;
        units += a.fam[f].n_items * (a.fam[f].inter / 32);
    }
    if (a.fam[0].n_items + a.fam[1].n_items != list.n_items || a.d % 256 || units == 0 ||
        (reinterpret_cast<uintptr_t>(a.x) & 15))
        return cudaErrorInvalidValue;
    // resident CTAs per SM at this launch's shared memory (cached per size)
    const size_t smem = ffn_smem<NT, C>(a.d);
    static size_t occ_smem[4] = {0, 0, 0, 0};
    static int occ_val[4] = {0, 0, 0, 0};
    int per_sm = 0;
    for (int i = 0; i < 4 && !per_sm; ++i)
        if (occ_smem[i] == smem) per_sm = occ_val[i];
    if (!per_sm) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ffn_kernel<NT, C, L>, kThreads, smem);
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
    int m = a.min_nt;  // the shape (and so the cross-warp order of the sums) for at least min_nt rows
    for (int i = 0; i < list.n_items; ++i) m = std::max(m, (int)list.item[i].np);
    // one row per item: 16 consumer warps (one CTA per SM); more rows stage
    // more token rows in shared memory and get 8 (a smaller ring)
    if (m <= 1) return ffn_launch<1, 16>(a, list, s, pdl);
    if (m <= 2) return ffn_launch<2, 8>(a, list, s, pdl);
    if (m <= 4) return ffn_launch<4, 8>(a, list, s, pdl);
    if (m <= kFfnMaxNT) return ffn_launch<8, 8>(a, list, s, pdl);
    return cudaErrorInvalidValue;
}

template cudaError_t launch_ffn<FfnSmall>(const FfnArgs&, const FfnSmall&, cudaStream_t, bool);
template cudaError_t launch_ffn<FfnLarge>(const FfnArgs&, const FfnLarge&, cudaStream_t, bool);

}  // namespace moe
