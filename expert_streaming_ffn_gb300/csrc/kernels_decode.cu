// Decode-path kernels of the expert-streaming MoE layer (sm_103a).
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
//
// router_kernel   8-bit router GEMV (warp per expert row, fp32 in a fixed order)
//                 followed, in the last block to finish a token block, by a
//                 warp-shuffle top-k and the renormalised softmax gates
//                 ([P3] "每个 token、每层都要重新路由"; [P1] §2.4 cb1).
// gateup_kernel   fused int4 dequant GEMV of gate and up for every (token, rank)
//                 pair of every selected expert, h = act(gate) * up
//                 ([P1] §2.4 cb2; int4 affine group 64, [P1] §2.1, §2.5).
// down_kernel     fused int4 dequant GEMV of the down projection.
// combine_kernel  y += sum_r gate_r * o_r in rank order ([P1] §6.2.3 fusion).
//
// The GEMVs are bound by HBM bandwidth. Lane l of a warp owns one weight row,
// so a warp-wide 16-byte load reads 512 contiguous bytes of the tiled layout,
// and the K dimension is split over the block's four warps. The activations
// sit in shared memory, pre-scaled so that 4-bit codes can be turned into
// floats with one bitwise op each: code q at nibble position p of a 32-bit
// word becomes the float 2^23 + q * 16^p via (word & (15 << 4p)) | 0x4B000000,
// and subtracting 2^23 (exact) leaves q * 16^p; the matching activation is
// stored multiplied by 16^-p (exact), so every product equals q * x. The
// affine dequantisation is applied per group afterwards:
//   sum_k x_k (s q_k + b) = s * sum_k q_k x_k + b * sum_k x_k.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// scale (low half) and bias (high half) of one group
__device__ __forceinline__ float2 unpack_sb(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

// The eight 4-bit codes of a word as q * 16^p pairs, p = 0,1 | 2,3 | 4,2 | 3,4
// (codes 5..7 are read from the word shifted right by 12).
__device__ __forceinline__ void codes8(uint32_t v, float2 (&o)[4]) {
    const uint32_t M = 0x4B000000u;
    const uint32_t w = v >> 12;
    const float2 off = make_float2(-8388608.0f, -8388608.0f);
    o[0] = __fadd2_rn(make_float2(__uint_as_float((v & 0xFu) | M), __uint_as_float((v & 0xF0u) | M)), off);
    o[1] = __fadd2_rn(make_float2(__uint_as_float((v & 0xF00u) | M), __uint_as_float((v & 0xF000u) | M)), off);
    o[2] = __fadd2_rn(make_float2(__uint_as_float((v & 0xF0000u) | M), __uint_as_float((w & 0xF00u) | M)), off);
    o[3] = __fadd2_rn(make_float2(__uint_as_float((w & 0xF000u) | M), __uint_as_float((w & 0xF0000u) | M)), off);
}

// 16^-p for the nibble positions above, indexed by k mod 8.
__device__ __forceinline__ float pos_scale(int k8) {
    const float t[8] = {1.0f, 0.0625f, 0.00390625f, 0.000244140625f, 1.52587890625e-05f, 0.00390625f,
                        0.000244140625f, 1.52587890625e-05f};
    return t[k8];
}

__device__ __forceinline__ float act_fn(float z, int act) {
    if (act == 1) return z / (1.0f + expf(-z));
    return 0.5f * z * (1.0f + tanhf(0.7978845608028654f * (z + 0.044715f * z * z * z)));
}

// Stage rows of activations into shared memory: xs[j][k] = v * 16^-p(k),
// xsum[j][g] = sum of the unscaled values of group g. Rows come from bf16 x
// (row stride d) or from fp32 h. 8 values per thread per step; 8 consecutive
// threads cover one group of 64.
template <bool F32>
__device__ __forceinline__ void stage_rows(const void* src, int d, const int16_t* pairs, int nt, int x_div,
                                           float* xs, float* xsum) {
    const int G = d >> 6;
    for (int j = 0; j < nt; ++j) {
        const size_t row = (size_t)(pairs[j] / x_div) * (size_t)d;
        for (int base = 0; base < d; base += kThreads * 8) {
            const int i = base + (int)threadIdx.x * 8;
            float f[8];
            if (i < d) {
                if (F32) {
                    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + row + i);
                    float4 a = p[0], b = p[1];
                    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
                    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
                } else {
                    uint4 r = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + row + i);
                    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x); f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
                    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z); f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
                }
            } else {
#pragma unroll
                for (int m = 0; m < 8; ++m) f[m] = 0.0f;
            }
            float s = ((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]));
            s += __shfl_xor_sync(kFull, s, 1);
            s += __shfl_xor_sync(kFull, s, 2);
            s += __shfl_xor_sync(kFull, s, 4);
            if (i < d) {
                float4* o = reinterpret_cast<float4*>(xs + (size_t)j * d + i);
                o[0] = make_float4(f[0] * pos_scale(0), f[1] * pos_scale(1), f[2] * pos_scale(2), f[3] * pos_scale(3));
                o[1] = make_float4(f[4] * pos_scale(4), f[5] * pos_scale(5), f[6] * pos_scale(6), f[7] * pos_scale(7));
                if ((threadIdx.x & 7) == 0) xsum[j * G + (i >> 6)] = s;
            }
        }
    }
}

// sum over one group (64 codes = two 16-byte chunks) of q * x for NT rows of x.
template <int NT>
__device__ __forceinline__ void group_dot(const uint4& c0, const uint4& c1, const float* xs, int d, int g,
                                          float2 (&acc)[NT]) {
    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        float2 q[4];
        codes8(words[w], q);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)j * d + g * 64 + w * 8);
            const float4 a = xp[0], b = xp[1];
            acc[j] = __ffma2_rn(q[0], make_float2(a.x, a.y), acc[j]);
            acc[j] = __ffma2_rn(q[1], make_float2(a.z, a.w), acc[j]);
            acc[j] = __ffma2_rn(q[2], make_float2(b.x, b.y), acc[j]);
            acc[j] = __ffma2_rn(q[3], make_float2(b.z, b.w), acc[j]);
        }
    }
}

// ---------------------------------------------------------------------------
// gate/up

template <int NT, class L>
__global__ void __launch_bounds__(kThreads) gateup_kernel(const uint16_t* __restrict__ x, int d, int inter, int act,
                                                          int x_div, const __grid_constant__ L list,
                                                          float* __restrict__ h) {
    const int tiles = inter >> 5;
    const int item = blockIdx.x / tiles;
    const int rt = blockIdx.x - item * tiles;
    const int G = d >> 6;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g_lo = warp * G / kWarps, g_hi = (warp + 1) * G / kWarps;

    const uint8_t* blob = list.w[item];
    const size_t mat = qmat_bytes(inter, d);
    const size_t codes_bytes = (size_t)inter * (size_t)d / 2;
    // lane-owned row: chunk c at ((rt*K/32 + c)*32 + lane)*16
    const uint8_t* gc = blob + ((size_t)rt * (d >> 5) * 32 + lane) * 16;
    const uint8_t* uc = gc + mat;
    const uint8_t* gs = blob + codes_bytes + ((size_t)rt * G * 32 + lane) * 4;
    const uint8_t* us = gs + mat;

    extern __shared__ float smem[];
    float* xs = smem;             // [NT][d]
    float* xsum = xs + NT * d;    // [NT][G]
    float* red = xsum + NT * G;   // [kWarps][NT][2][32]

    const int pb = list.begin[item], pe = list.begin[item + 1];
    for (int p0 = pb; p0 < pe; p0 += NT) {
        const int nt = min(NT, pe - p0);
        stage_rows<false>(x, d, list.pair + p0, nt, x_div, xs, xsum);
        __syncthreads();

        float accg[NT], accu[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) accg[j] = accu[j] = 0.0f;

        if (g_lo < g_hi) {
            uint4 g0 = ld_stream(gc + (size_t)(2 * g_lo) * 512), g1 = ld_stream(gc + (size_t)(2 * g_lo + 1) * 512);
            uint4 u0 = ld_stream(uc + (size_t)(2 * g_lo) * 512), u1 = ld_stream(uc + (size_t)(2 * g_lo + 1) * 512);
            uint32_t sg = ld_stream_u32(gs + (size_t)g_lo * 128), su = ld_stream_u32(us + (size_t)g_lo * 128);
            for (int g = g_lo; g < g_hi; ++g) {
                uint4 ng0 = g0, ng1 = g1, nu0 = u0, nu1 = u1;
                uint32_t nsg = sg, nsu = su;
                if (g + 1 < g_hi) {  // prefetch the next group
                    ng0 = ld_stream(gc + (size_t)(2 * g + 2) * 512);
                    ng1 = ld_stream(gc + (size_t)(2 * g + 3) * 512);
                    nu0 = ld_stream(uc + (size_t)(2 * g + 2) * 512);
                    nu1 = ld_stream(uc + (size_t)(2 * g + 3) * 512);
                    nsg = ld_stream_u32(gs + (size_t)(g + 1) * 128);
                    nsu = ld_stream_u32(us + (size_t)(g + 1) * 128);
                }
                float2 pg[NT], pu[NT];
#pragma unroll
                for (int j = 0; j < NT; ++j) pg[j] = pu[j] = make_float2(0.0f, 0.0f);
                group_dot<NT>(g0, g1, xs, d, g, pg);
                group_dot<NT>(u0, u1, xs, d, g, pu);
                const float2 fg = unpack_sb(sg), fu = unpack_sb(su);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const float xsg = xsum[j * G + g];
                    accg[j] = fmaf(fg.x, pg[j].x + pg[j].y, fmaf(fg.y, xsg, accg[j]));
                    accu[j] = fmaf(fu.x, pu[j].x + pu[j].y, fmaf(fu.y, xsg, accu[j]));
                }
                g0 = ng0; g1 = ng1; u0 = nu0; u1 = nu1; sg = nsg; su = nsu;
            }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            red[((warp * NT + j) * 2 + 0) * 32 + lane] = accg[j];
            red[((warp * NT + j) * 2 + 1) * 32 + lane] = accu[j];
        }
        __syncthreads();
        if (warp < NT && warp < nt) {  // warp j finishes pair j
            const int j = warp;
            float gsum = 0.0f, usum = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                gsum += red[((w * NT + j) * 2 + 0) * 32 + lane];
                usum += red[((w * NT + j) * 2 + 1) * 32 + lane];
            }
            h[(size_t)list.pair[p0 + j] * inter + rt * 32 + lane] = act_fn(gsum, act) * usum;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// down

template <int NT, class L>
__global__ void __launch_bounds__(kThreads) down_kernel(const float* __restrict__ hin, int inter, int d,
                                                        const __grid_constant__ L list, float* __restrict__ out) {
    const int tiles = d >> 5;
    const int item = blockIdx.x / tiles;
    const int rt = blockIdx.x - item * tiles;
    const int G = inter >> 6;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g_lo = warp * G / kWarps, g_hi = (warp + 1) * G / kWarps;

    const uint8_t* blob = list.w[item] + 2 * qmat_bytes(inter, d);
    const uint8_t* dc = blob + ((size_t)rt * (inter >> 5) * 32 + lane) * 16;
    const uint8_t* ds = blob + (size_t)d * (size_t)inter / 2 + ((size_t)rt * G * 32 + lane) * 4;

    extern __shared__ float smem[];
    float* xs = smem;              // [NT][inter]
    float* xsum = xs + NT * inter; // [NT][G]
    float* red = xsum + NT * G;    // [kWarps][NT][32]

    const int pb = list.begin[item], pe = list.begin[item + 1];
    for (int p0 = pb; p0 < pe; p0 += NT) {
        const int nt = min(NT, pe - p0);
        stage_rows<true>(hin, inter, list.pair + p0, nt, 1, xs, xsum);
        __syncthreads();
        float acc[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j] = 0.0f;
        if (g_lo < g_hi) {
            uint4 c0 = ld_stream(dc + (size_t)(2 * g_lo) * 512), c1 = ld_stream(dc + (size_t)(2 * g_lo + 1) * 512);
            uint32_t sb = ld_stream_u32(ds + (size_t)g_lo * 128);
            for (int g = g_lo; g < g_hi; ++g) {
                uint4 n0 = c0, n1 = c1;
                uint32_t nsb = sb;
                if (g + 1 < g_hi) {
                    n0 = ld_stream(dc + (size_t)(2 * g + 2) * 512);
                    n1 = ld_stream(dc + (size_t)(2 * g + 3) * 512);
                    nsb = ld_stream_u32(ds + (size_t)(g + 1) * 128);
                }
                float2 p[NT];
#pragma unroll
                for (int j = 0; j < NT; ++j) p[j] = make_float2(0.0f, 0.0f);
                group_dot<NT>(c0, c1, xs, inter, g, p);
                const float2 f = unpack_sb(sb);
#pragma unroll
                for (int j = 0; j < NT; ++j) acc[j] = fmaf(f.x, p[j].x + p[j].y, fmaf(f.y, xsum[j * G + g], acc[j]));
                c0 = n0; c1 = n1; sb = nsb;
            }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) red[(warp * NT + j) * 32 + lane] = acc[j];
        __syncthreads();
        if (warp < NT && warp < nt) {
            const int j = warp;
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += red[(w * NT + j) * 32 + lane];
            out[(size_t)list.pair[p0 + j] * d + rt * 32 + lane] = s;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// combine

__global__ void combine_kernel(const float* __restrict__ o, const float* __restrict__ gates, int k, int d,
                               float* __restrict__ y) {
    const int t = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= d) return;
    float acc = y[(size_t)t * d + n];
    for (int r = 0; r < k; ++r) acc = fmaf(gates[t * k + r], o[((size_t)t * k + r) * d + n], acc);
    y[(size_t)t * d + n] = acc;
}

// ---------------------------------------------------------------------------
// router + top-k

constexpr int kRouterWarps = 4;
constexpr int kRouterTB = 8;  // tokens per block

__device__ __forceinline__ float bf16_at(const uint4& r, int i) {
    const uint32_t w = i < 2 ? r.x : i < 4 ? r.y : i < 6 ? r.z : r.w;
    return (i & 1) ? bf16_hi(w) : bf16_lo(w);
}

// Top-k of one token's logits by one warp: k rounds of a warp-wide argmax
// ordered by (logit descending, expert index ascending); lane r ends up with
// rank r. Then gates = softmax over the k chosen logits.
template <int MAXV>
__device__ void topk_warp(const float* logits, int E, int k, int lane, int32_t* ids, float* gates) {
    float v[MAXV];
    uint32_t taken = 0;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int e = lane + 32 * j;
        if (e < E)
            v[j] = __ldcg(logits + e);
        else {
            v[j] = -INFINITY;
            taken |= 1u << j;
        }
    }
    float mine_v = -INFINITY;
    int mine_i = 0;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int e = lane + 32 * j;
            if (!((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < bi))) {
                bv = v[j];
                bi = e;
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, off);
            const int oi = __shfl_xor_sync(kFull, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == r) {
            mine_v = bv;
            mine_i = bi;
        }
    }
    const float top = __shfl_sync(kFull, mine_v, 0);
    float ex = lane < k ? expf(mine_v - top) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (lane < k) {
        ids[lane] = mine_i;
        gates[lane] = ex / sum;
    }
}

__global__ void __launch_bounds__(kRouterWarps * 32) router_kernel(const RouterParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRouterWarps + warp;
    const int t0 = blockIdx.y * kRouterTB;
    const int nt = min(kRouterTB, p.T - t0);
    const int runs = p.d >> 4;
    if (e < p.E) {
        float acc[kRouterTB];
#pragma unroll
        for (int j = 0; j < kRouterTB; ++j) acc[j] = 0.0f;
        const uint8_t* row = p.codes + (size_t)e * p.d;
        const uint32_t* sbrow = p.sb + (size_t)e * (p.d >> 6);
        for (int c = lane; c < runs; c += 32) {
            const uint4 q = ld_stream(row + (size_t)c * 16);
            const float2 f = unpack_sb(__ldg(sbrow + (c >> 2)));
            float w[16];
            const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __fmaf_rn(f.x, (float)((qw[i >> 2] >> (8 * (i & 3))) & 0xFFu), f.y);
#pragma unroll
            for (int j = 0; j < kRouterTB; ++j) {
                if (j < nt) {
                    const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)(t0 + j) * p.d + (size_t)c * 16);
                    const uint4 xa = __ldg(xr), xb = __ldg(xr + 1);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[j] = __fmaf_rn(w[i], bf16_at(xa, i), acc[j]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[j] = __fmaf_rn(w[8 + i], bf16_at(xb, i), acc[j]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kRouterTB; ++j) {
            if (j < nt) {
                float v = acc[j];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
                if (lane == 0) p.logits[(size_t)(t0 + j) * p.E + e] = p.zbias ? __fadd_rn(v, p.zbias[e]) : v;
            }
        }
    }
    // The last block of this token block to finish runs the top-k.
    __shared__ int is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(p.counters + blockIdx.y, 1u);
        is_last = prev == gridDim.x - 1;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int j = warp; j < nt; j += kRouterWarps) {
        const int t = t0 + j;
        if (p.E <= 256)
            topk_warp<8>(p.logits + (size_t)t * p.E, p.E, p.k, lane, p.ids + (size_t)t * p.k, p.gates + (size_t)t * p.k);
        else
            topk_warp<32>(p.logits + (size_t)t * p.E, p.E, p.k, lane, p.ids + (size_t)t * p.k, p.gates + (size_t)t * p.k);
    }
    if (threadIdx.x == 0) p.counters[blockIdx.y] = 0;
}

template <int NT>
size_t gateup_smem(int d) {
    return sizeof(float) * ((size_t)NT * d + (size_t)NT * (d / 64) + (size_t)kWarps * NT * 2 * 32);
}
template <int NT>
size_t down_smem(int inter) {
    return sizeof(float) * ((size_t)NT * inter + (size_t)NT * (inter / 64) + (size_t)kWarps * NT * 32);
}

template <int NT, class L>
cudaError_t gateup_nt(const uint16_t* x, int d, int inter, int act, int x_div, const L& list, float* h,
                      cudaStream_t s) {
    const size_t sm = gateup_smem<NT>(d);
    static bool attr_set = false;  // per template instance
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gateup_kernel<NT, L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)gateup_smem<NT>(kMaxDModel));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    gateup_kernel<NT, L><<<list.n_items * (inter / 32), kThreads, sm, s>>>(x, d, inter, act, x_div, list, h);
    return cudaGetLastError();
}

template <int NT, class L>
cudaError_t down_nt(const float* h, int inter, int d, const L& list, float* out, cudaStream_t s) {
    const size_t sm = down_smem<NT>(inter);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(down_kernel<NT, L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)down_smem<NT>(kMaxDModel));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    down_kernel<NT, L><<<list.n_items * (d / 32), kThreads, sm, s>>>(h, inter, d, list, out);
    return cudaGetLastError();
}

// Largest pair count of any item: picks how many rows one pass stages.
template <class L>
int max_pairs(const L& list) {
    int m = 0;
    for (int i = 0; i < list.n_items; ++i) m = list.begin[i + 1] - list.begin[i] > m ? list.begin[i + 1] - list.begin[i] : m;
    return m;
}

}  // namespace

cudaError_t launch_router(const RouterParams& p, cudaStream_t s) {
    dim3 grid((p.E + kRouterWarps - 1) / kRouterWarps, (p.T + kRouterTB - 1) / kRouterTB);
    router_kernel<<<grid, kRouterWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

template <class L>
cudaError_t launch_gateup(const uint16_t* x, int d, int inter, int act, int x_div, const L& list, float* h,
                          cudaStream_t s) {
    if (list.n_items == 0) return cudaSuccess;
    const int m = max_pairs(list);
    if (m <= 1) return gateup_nt<1>(x, d, inter, act, x_div, list, h, s);
    if (m <= 2) return gateup_nt<2>(x, d, inter, act, x_div, list, h, s);
    return gateup_nt<4>(x, d, inter, act, x_div, list, h, s);
}

template <class L>
cudaError_t launch_down(const float* h, int inter, int d, const L& list, float* out, cudaStream_t s) {
    if (list.n_items == 0) return cudaSuccess;
    const int m = max_pairs(list);
    if (m <= 1) return down_nt<1>(h, inter, d, list, out, s);
    if (m <= 2) return down_nt<2>(h, inter, d, list, out, s);
    return down_nt<4>(h, inter, d, list, out, s);
}

cudaError_t launch_combine(const float* o, const float* gates, int T, int k, int d, float* y, cudaStream_t s) {
    dim3 grid((d + 255) / 256, T);
    combine_kernel<<<grid, 256, 0, s>>>(o, gates, k, d, y);
    return cudaGetLastError();
}

template cudaError_t launch_gateup<SmallList>(const uint16_t*, int, int, int, int, const SmallList&, float*, cudaStream_t);
template cudaError_t launch_gateup<LargeList>(const uint16_t*, int, int, int, int, const LargeList&, float*, cudaStream_t);
template cudaError_t launch_down<SmallList>(const float*, int, int, const SmallList&, float*, cudaStream_t);
template cudaError_t launch_down<LargeList>(const float*, int, int, const LargeList&, float*, cudaStream_t);

}  // namespace moe
