// Router and combine kernels of the expert-streaming MoE layer (sm_103a).
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
//
// router_kernel   8-bit router GEMV, one warp per expert row, fp32 in a fixed
//                 order, followed, in the last block to finish a token block,
//                 by a warp-reduction top-k (ties to the lower expert index) and
//                 the softmax over the k chosen logits ([P3]
//                 "每个 token、每层都要重新路由"; [P1] §2.4 cb1). Each id is
//                 also written to mapped host memory as one 64-bit word
//                 (call number << 32 | id), so the host sees the routing as
//                 soon as it lands, without a copy, an event or a fence
//                 ([P1] §2.4: the ids go to the CPU for the cache lookup).
// router_wide_kernel  the same routing for 64 tokens or more (prefill), with
//                 the block's token rows staged once as fp32 and each warp
//                 taking several expert rows: the same logits, bit for bit.
// combine_kernel  y += sum_r gate_r * o_r in rank order ([P1] §6.2.3 fusion).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRouterWarps = 4;  // expert rows per block (decode and short inputs)
constexpr int kRouterTB = 8;     // tokens per block
constexpr int kRouterBatch = 8;  // runs per lane whose loads are issued together
// Long inputs (prefill, T >= 64): router_wide_kernel, 8 warps by 8 tokens a
// block with the token rows staged once as fp32, each warp taking 2 or 4
// expert rows, two at a time (see there).
constexpr int kRouterWideWarps = 8, kRouterWideTB = 8, kRouterWideBatch = 4;
constexpr int kRouterWideMinT = 64, kRouterWideMaxD = 6144;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float2 unpack_sb(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

__device__ __forceinline__ float bf16_at(const uint4& r, int i) {
    const uint32_t w = i < 2 ? r.x : i < 4 ? r.y : i < 6 ? r.z : r.w;
    return (i & 1) ? bf16_hi(w) : bf16_lo(w);
}

// Monotonic map of floats to unsigned keys (a < b iff key(a) < key(b)), with
// -0 taken as +0 so that the two compare equal as floats do.
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.0f);
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Top-k of one token's logits by one warp. Lane l holds the candidates of
// experts l + 32 j as 64-bit words (key << 32 | ~e), so that a larger word is
// a larger logit or, for equal logits, a lower expert index; it sorts them
// once, descending. Each of the k rounds then takes the warp-wide maximum of
// the lanes' heads with two single-instruction reductions (the largest key,
// then the largest index part, i.e. the lowest expert id, among the lanes
// holding that key), and the lane that owned it moves to its next candidate
// (measured faster than a butterfly merge of the lanes' sorted lists). Lane r
// ends up with rank r. Then gates = softmax over the k chosen logits.
template <int MAXV>
__device__ void topk_warp(const float* logits, int E, int k, int lane, int32_t* ids, float* gates,
                          unsigned long long* host_ids, uint32_t seq) {
    const int k_all = k;
    unsigned long long c[MAXV];
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int e = lane + 32 * j;
        // beyond E: 0, below every real candidate (whose index part is nonzero)
        c[j] = e < E ? ((unsigned long long)order_key(__ldcg(logits + e)) << 32) | (uint32_t)~e : 0ull;
    }
    // odd-even transposition sort, descending (MAXV passes)
#pragma unroll
    for (int pass = 0; pass < MAXV; ++pass)
#pragma unroll
        for (int j = pass & 1; j + 1 < MAXV; j += 2)
            if (c[j] < c[j + 1]) {
                const unsigned long long t = c[j];
                c[j] = c[j + 1];
                c[j + 1] = t;
            }
    float mine_v = -INFINITY;
    int mine_i = 0;
    for (int r = 0; r < k; ++r) {
        const uint32_t hk = (uint32_t)(c[0] >> 32), hi = (uint32_t)c[0];
        const uint32_t top = __reduce_max_sync(kFull, hk);
        const uint32_t win = __reduce_max_sync(kFull, hk == top ? hi : 0u);  // ~e: the lowest index
        if (hk == top && hi == win) {
            // this lane's head was taken: move up its remaining candidates
#pragma unroll
            for (int j = 0; j + 1 < MAXV; ++j) c[j] = c[j + 1];
            c[MAXV - 1] = 0ull;
        }
        if (lane == r) {
            mine_v = key_value(top);
            mine_i = (int)~win;
        }
    }
    const float top = __shfl_sync(kFull, mine_v, 0);
    const float ex = lane < k_all ? expf(mine_v - top) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (lane < k_all) {
        ids[lane] = mine_i;
        gates[lane] = ex / sum;
        if (host_ids)
            *reinterpret_cast<volatile unsigned long long*>(host_ids + lane) =
                ((unsigned long long)seq << 32) | (uint32_t)mine_i;
    }
}

// The top-k for more than 256 experts, out of line: its 32 candidates per
// lane would otherwise set the register budget of every router launch.
__device__ __noinline__ void topk_warp_large(const float* logits, int E, int k, int lane, int32_t* ids, float* gates,
                                             unsigned long long* host_ids, uint32_t seq) {
    topk_warp<32>(logits, E, k, lane, ids, gates, host_ids, seq);
}

// Code byte m of a word as the float q (exact): 2^23 + q from a byte permute
// into the magic word 0x4B000000, minus 2^23.
__device__ __forceinline__ float byte_code(uint32_t w, int m) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | (uint32_t)m)) - 8388608.0f;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// The end of a router launch: the last block of each token block to finish
// (counted on the token block's arrival counter) runs the top-k of its tokens
// with its W warps and resets the counter. Each block's arrival is a release
// of its logits, and the count the last one reads an acquire of all of them.
template <int W>
__device__ __forceinline__ void router_finish(const RouterParams& p, int t0, int nt, int warp, int lane) {
    __shared__ int is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atom_add_acq_rel(p.counters + blockIdx.y, 1u);
        is_last = prev == gridDim.x - 1;
    }
    __syncthreads();
    if (!is_last) {
        if (p.span && threadIdx.x == 0) atomicMax(p.span + 1, (unsigned long long)ptx::globaltimer());
        return;
    }
    for (int j = warp; j < nt; j += W) {
        const int t = t0 + j;
        unsigned long long* hid = p.host_ids ? p.host_ids + (size_t)t * p.k : nullptr;
        if (p.E <= 256)
            topk_warp<8>(p.logits + (size_t)t * p.E, p.E, p.k, lane, p.ids + (size_t)t * p.k,
                         p.gates + (size_t)t * p.k, hid, p.seq);
        else
            topk_warp_large(p.logits + (size_t)t * p.E, p.E, p.k, lane, p.ids + (size_t)t * p.k,
                            p.gates + (size_t)t * p.k, hid, p.seq);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        p.counters[blockIdx.y] = 0;
        if (p.span) atomicMax(p.span + 1, (unsigned long long)ptx::globaltimer());
    }
}

template <int TB, int W, int KB>
__global__ void __launch_bounds__(W * 32, TB == 1 ? 5 : 1) router_kernel(const RouterParams p) {
    extern __shared__ uint4 xsm[];  // the block's token rows, [nt][d / 8] of 8 bf16 each
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e_first = blockIdx.x * W + warp;  // this warp's expert row
    const int t0 = blockIdx.y * TB;
    const int nt = min(TB, p.T - t0);
    const int runs = p.d >> 4;
    const int vec = p.d >> 3;
    // the next kernel may start now; this one reads x and writes y only
    // after the previous kernel has finished (griddepcontrol.wait below)
    ptx::pdl_launch_dependents();
    if (p.span && threadIdx.x == 0) atomicMin(p.span, (unsigned long long)ptx::globaltimer());
    if (e_first < p.E) {
        const uint8_t* row0 = p.codes + (size_t)e_first * p.d;
        for (int c = lane; c < runs && c < 32 * KB; c += 32)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(row0 + (size_t)c * 16));
    }
    ptx::pdl_wait();
    if (p.zero) {
        const int nb = gridDim.x * gridDim.y * blockDim.x;
        for (int i = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x; i < p.zero_n; i += nb)
            p.zero[i] = 0.0f;
    }
    // Lane l owns runs c = l + 32 i (16 inputs each), walked in increasing c.
    // A batch's KB loads are all in flight together; the first batch of the
    // first row is issued before the token rows are staged, so the two
    // latencies overlap.
    uint4 q[KB];
    uint32_t sbw[KB];
    const uint8_t* row = nullptr;
    const uint32_t* sbrow = nullptr;
    bool has_row = false;
    auto load_batch = [&](int b0) {
#pragma unroll
        for (int i = 0; i < KB; ++i) {
            const int c = lane + 32 * (b0 + i);
            if (has_row && c < runs) {
                q[i] = ld_stream(row + (size_t)c * 16);
                sbw[i] = __ldg(sbrow + (c >> 2));
            }
        }
    };
    auto set_row = [&](int e) {
        has_row = e < p.E;
        row = p.codes + (size_t)(has_row ? e : 0) * p.d;
        sbrow = p.sb + (size_t)(has_row ? e : 0) * (p.d >> 6);
    };
    set_row(e_first);
    load_batch(0);
    {
        // the token rows, eight loads per thread in flight at a time
        const uint4* xg = reinterpret_cast<const uint4*>(p.x + (size_t)t0 * p.d);
        const int n = nt * vec;
        for (int i0 = threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (i0 + u * (int)blockDim.x < n) v[u] = __ldg(xg + i0 + u * blockDim.x);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (i0 + u * (int)blockDim.x < n) xsm[i0 + u * blockDim.x] = v[u];
        }
    }
    __syncthreads();
    if (has_row) {
        const int e = e_first;
        float acc[TB];
#pragma unroll
        for (int j = 0; j < TB; ++j) acc[j] = 0.0f;
        for (int b0 = 0; 32 * b0 < runs; b0 += KB) {
            if (b0 > 0) load_batch(b0);
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                const int c = lane + 32 * (b0 + i);
                if (c >= runs) continue;
                const float2 f = unpack_sb(sbw[i]);
                const uint32_t qw[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
                float w[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) w[m] = __fmaf_rn(f.x, byte_code(qw[m >> 2], m & 3), f.y);
#pragma unroll
                for (int j = 0; j < TB; ++j) {
                    if (j < nt) {
                        const uint4 xa = xsm[j * vec + 2 * c], xb = xsm[j * vec + 2 * c + 1];
#pragma unroll
                        for (int m = 0; m < 8; ++m) acc[j] = __fmaf_rn(w[m], bf16_at(xa, m), acc[j]);
#pragma unroll
                        for (int m = 0; m < 8; ++m) acc[j] = __fmaf_rn(w[8 + m], bf16_at(xb, m), acc[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            if (j < nt) {
                float v = acc[j];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
                if (lane == 0) p.logits[(size_t)(t0 + j) * p.E + e] = p.zbias ? __fadd_rn(v, p.zbias[e]) : v;
            }
        }
    }
    router_finish<W>(p, t0, nt, warp, lane);
}

// One block per (token, 32 output columns). Term j < ns is the j-th group of
// cr shared-expert chunks, term ns + r the routed pair of rank r; warp w sums
// terms w, w + warps, ... (each over its chunks in order), and one warp then
// adds the terms in order.
__global__ void part_reduce_kernel(const float* __restrict__ part0, const float* __restrict__ part1, int cs, int cr,
                                   int k, int d, float* __restrict__ y) {
    extern __shared__ float terms[];  // [ns + k][32]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.y, n = blockIdx.x * 32 + lane;
    const int ns = (cs + cr - 1) / cr, nterm = ns + k;
    // the partials were written by the previous kernels of the call
    ptx::pdl_wait();
    for (int j = warp; j < nterm; j += blockDim.x >> 5) {
        const float* src;
        int c0, c1, cstride;
        if (j < ns) {
            src = part0 + (size_t)t * cs * d;
            c0 = j * cr;
            c1 = min(cs, c0 + cr);
        } else {
            src = part1 + ((size_t)t * k + (j - ns)) * cr * d;
            c0 = 0;
            c1 = cr;
        }
        cstride = d;
        float acc = 0.0f;
        if (n < d) {
            int c = c0;
            for (; c + 4 <= c1; c += 4) {
                const float v0 = __ldcg(src + (size_t)c * cstride + n), v1 = __ldcg(src + (size_t)(c + 1) * cstride + n);
                const float v2 = __ldcg(src + (size_t)(c + 2) * cstride + n), v3 = __ldcg(src + (size_t)(c + 3) * cstride + n);
                acc = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(acc, v0), v1), v2), v3);
            }
            for (; c < c1; ++c) acc = __fadd_rn(acc, __ldcg(src + (size_t)c * cstride + n));
        }
        terms[j * 32 + lane] = acc;
    }
    __syncthreads();
    if (warp == 0 && n < d) {
        float v = 0.0f;
        for (int j = 0; j < nterm; ++j) v = __fadd_rn(v, terms[j * 32 + lane]);
        y[(size_t)t * d + n] = v;
    }
}

__global__ void combine_kernel(const float* __restrict__ o, const float* __restrict__ gates, int k, int d,
                               float* __restrict__ y) {
    const int t = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= d) return;
    float acc = y[(size_t)t * d + n];
    for (int r = 0; r < k; ++r) acc = fmaf(gates[t * k + r], o[((size_t)t * k + r) * d + n], acc);
    y[(size_t)t * d + n] = acc;
}

// The router over a long input. The block's token rows are staged once as
// fp32 (the exact values of the bf16 inputs), laid out so that the 16 inputs
// of lane l's run slot i are four float4 at [token][i][quad][l]: a warp's
// loads are conflict-free and the loop does no unpacking. Each warp takes R
// expert rows, two at a time, so that every input it loads from shared memory
// feeds two FMAs (one input per FMA would need four times the SM's
// shared-memory bandwidth); a staged token row serves 8 R rows (R = 4 for long
// prompts, 2 for a chunk, whose fewer token blocks need more blocks across
// the experts). Every logit is one warp's sum over the same runs in the same
// order, with the same butterfly, as in router_kernel: the same bits.
template <int R>
__global__ void __launch_bounds__(kRouterWideWarps * 32, 2) router_wide_kernel(const RouterParams p) {
    constexpr int TB = kRouterWideTB, W = kRouterWideWarps, KB = kRouterWideBatch, RP = 2;
    static_assert(R % RP == 0, "rows in pairs");
    extern __shared__ float4 xw[];  // [nt][NI][4][32]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e_first = (blockIdx.x * W + warp) * R;
    const int t0 = blockIdx.y * TB;
    const int nt = min(TB, p.T - t0);
    const int runs = p.d >> 4, NI = (runs + 31) >> 5;
    ptx::pdl_launch_dependents();
    if (p.span && threadIdx.x == 0) atomicMin(p.span, (unsigned long long)ptx::globaltimer());
    for (int r = 0; r < RP; ++r)
        if (e_first + r < p.E) {
            const uint8_t* row0 = p.codes + (size_t)(e_first + r) * p.d;
            for (int c = lane; c < runs && c < 32 * KB; c += 32)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(row0 + (size_t)c * 16));
        }
    ptx::pdl_wait();
    if (p.zero) {
        const int nb = gridDim.x * gridDim.y * blockDim.x;
        for (int i = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x; i < p.zero_n; i += nb)
            p.zero[i] = 0.0f;
    }
    uint4 q[RP][KB];
    uint32_t sbw[RP][KB];
    const uint8_t* row[RP];
    const uint32_t* sbrow[RP];
    bool has[RP];
    auto load_batch = [&](int b0) {
#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                const int c = lane + 32 * (b0 + i);
                if (has[r] && c < runs) {
                    q[r][i] = ld_stream(row[r] + (size_t)c * 16);
                    sbw[r][i] = __ldg(sbrow[r] + (c >> 2));
                }
            }
    };
    auto set_rows = [&](int e0) {
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            has[r] = e0 + r < p.E;
            row[r] = p.codes + (size_t)(has[r] ? e0 + r : 0) * p.d;
            sbrow[r] = p.sb + (size_t)(has[r] ? e0 + r : 0) * (p.d >> 6);
        }
    };
    set_rows(e_first);
    load_batch(0);
    {
        // 8-input chunk k of token j: run k / 2, quads 2 (k & 1) and 2 (k & 1) + 1
        const int per_row = p.d >> 3;
        const uint4* xg = reinterpret_cast<const uint4*>(p.x + (size_t)t0 * p.d);
        const int n = nt * per_row;
        for (int i0 = threadIdx.x; i0 < n; i0 += 4 * blockDim.x) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (i0 + u * (int)blockDim.x < n) v[u] = __ldg(xg + i0 + u * blockDim.x);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int idx = i0 + u * (int)blockDim.x;
                if (idx < n) {
                    const int j = idx / per_row, k = idx - j * per_row;
                    const int c = k >> 1, base = ((j * NI + (c >> 5)) * 4 + 2 * (k & 1)) * 32 + (c & 31);
                    xw[base] = make_float4(bf16_lo(v[u].x), bf16_hi(v[u].x), bf16_lo(v[u].y), bf16_hi(v[u].y));
                    xw[base + 32] = make_float4(bf16_lo(v[u].z), bf16_hi(v[u].z), bf16_lo(v[u].w), bf16_hi(v[u].w));
                }
            }
        }
    }
    __syncthreads();
    for (int rr = 0; rr < R; rr += RP) {
        const int e0 = e_first + rr;
        if (rr > 0) {
            set_rows(e0);
            load_batch(0);
        }
        if (!has[0]) break;
        float acc[RP][TB];
#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
            for (int j = 0; j < TB; ++j) acc[r][j] = 0.0f;
        for (int b0 = 0; 32 * b0 < runs; b0 += KB) {
            if (b0 > 0) load_batch(b0);
#pragma unroll
            for (int i = 0; i < KB; ++i) {
                const int c = lane + 32 * (b0 + i);
                if (c >= runs) continue;
                float w[RP][16];
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    const float2 f = unpack_sb(sbw[r][i]);
                    const uint32_t qw[4] = {q[r][i].x, q[r][i].y, q[r][i].z, q[r][i].w};
#pragma unroll
                    for (int m = 0; m < 16; ++m) w[r][m] = __fmaf_rn(f.x, byte_code(qw[m >> 2], m & 3), f.y);
                }
                const float4* xs = xw + (size_t)(b0 + i) * 4 * 32 + lane;
#pragma unroll
                for (int j = 0; j < TB; ++j) {
                    if (j < nt) {
                        const float4* xj = xs + (size_t)j * NI * 4 * 32;
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            const float4 xv = xj[qq * 32];
#pragma unroll
                            for (int r = 0; r < RP; ++r) {
                                acc[r][j] = __fmaf_rn(w[r][4 * qq + 0], xv.x, acc[r][j]);
                                acc[r][j] = __fmaf_rn(w[r][4 * qq + 1], xv.y, acc[r][j]);
                                acc[r][j] = __fmaf_rn(w[r][4 * qq + 2], xv.z, acc[r][j]);
                                acc[r][j] = __fmaf_rn(w[r][4 * qq + 3], xv.w, acc[r][j]);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            if (!has[r]) continue;
            const int e = e0 + r;
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                if (j < nt) {
                    float v = acc[r][j];
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
                    if (lane == 0) p.logits[(size_t)(t0 + j) * p.E + e] = p.zbias ? __fadd_rn(v, p.zbias[e]) : v;
                }
            }
        }
    }
    router_finish<W>(p, t0, nt, warp, lane);
}

}  // namespace

cudaError_t launch_router(const RouterParams& p, cudaStream_t s, bool pdl) {
    cudaError_t e =
        ensure_smem_attr((const void*)router_kernel<kRouterTB, kRouterWarps, kRouterBatch>, (size_t)kRouterTB * kMaxDModel * 2);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr((const void*)router_kernel<1, kRouterWarps, 6>, (size_t)kMaxDModel * 2);
    if (e != cudaSuccess) return e;
    const auto wide_smem = [](int d) { return (size_t)kRouterWideTB * (((d >> 4) + 31) >> 5) * 4 * 32 * 16; };
    e = ensure_smem_attr((const void*)router_wide_kernel<2>, wide_smem(kRouterWideMaxD));
    if (e == cudaSuccess) e = ensure_smem_attr((const void*)router_wide_kernel<4>, wide_smem(kRouterWideMaxD));
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute la;
    if (p.T == 1) {
        const cudaLaunchConfig_t c = launch_config(dim3((p.E + kRouterWarps - 1) / kRouterWarps, 1),
                                                   dim3(kRouterWarps * 32), (size_t)p.d * 2, s, pdl, &la);
        return cudaLaunchKernelEx(&c, router_kernel<1, kRouterWarps, 6>, p);
    }
    if (p.T >= kRouterWideMinT && p.d <= kRouterWideMaxD) {
        // four expert rows a warp once there are enough token blocks to fill the GPU
        const int R = p.T >= 512 ? 4 : 2;
        const int rows = kRouterWideWarps * R;
        const cudaLaunchConfig_t c =
            launch_config(dim3((p.E + rows - 1) / rows, (p.T + kRouterWideTB - 1) / kRouterWideTB),
                          dim3(kRouterWideWarps * 32), wide_smem(p.d), s, pdl, &la);
        return R == 4 ? cudaLaunchKernelEx(&c, router_wide_kernel<4>, p) : cudaLaunchKernelEx(&c, router_wide_kernel<2>, p);
    }
    const size_t sm = (size_t)std::min(kRouterTB, p.T) * p.d * 2;
    const cudaLaunchConfig_t c = launch_config(
        dim3((p.E + kRouterWarps - 1) / kRouterWarps, (p.T + kRouterTB - 1) / kRouterTB), dim3(kRouterWarps * 32), sm, s,
        pdl, &la);
    return cudaLaunchKernelEx(&c, router_kernel<kRouterTB, kRouterWarps, kRouterBatch>, p);
}

cudaError_t launch_part_reduce(const float* part0, const float* part1, int cs, int cr, int k, int d, int T, float* y,
                               cudaStream_t s, bool pdl) {
    if (cs < 1 || cr < 1 || k < 1 || d % 32 || T < 1) return cudaErrorInvalidValue;
    const int nterm = (cs + cr - 1) / cr + k;
    const int warps = std::min(nterm, 16);
    cudaLaunchAttribute la;
    const cudaLaunchConfig_t c =
        launch_config(dim3(d / 32, T), dim3(32 * warps), sizeof(float) * 32 * nterm, s, pdl, &la);
    return cudaLaunchKernelEx(&c, part_reduce_kernel, part0, part1, cs, cr, k, d, y);
}

cudaError_t launch_combine(const float* o, const float* gates, int T, int k, int d, float* y, cudaStream_t s) {
    dim3 grid((d + 255) / 256, T);
    combine_kernel<<<grid, 256, 0, s>>>(o, gates, k, d, y);
    return cudaGetLastError();
}

}  // namespace moe
