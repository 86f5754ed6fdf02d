// Internal declarations of libmoe: host cache manager, weight layout and the
// kernel launchers. Not part of the public ABI (include/moe.h).
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/moe.h"

#ifdef __CUDACC__
#define MOE_HD __host__ __device__
#else
#define MOE_HD
#endif

namespace moe {

constexpr int kLFU = 0, kLRU = 1;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxDModel = 8192;
constexpr int kDecodeMaxT = 64;     // T above this runs the prefill path
constexpr int kPrefillChunk = 128;  // tokens per prefill chunk ([P1] §2.5, §8.4)

// Records a message for moe_last_error() (thread-local) and returns s.
moe_status set_error(moe_status s, const char* fmt, ...);

// ---- expert cache ----------------------------------------------------------

struct StepResult {
    std::vector<int> distinct;      // the step's distinct experts, ascending
    std::vector<int> miss_experts;  // ascending
    std::vector<int> miss_slots;    // -1 = bypass
    int hits = 0, bypass = 0;
};

class HostCache {
   public:
    HostCache(int n_experts, int slots, int policy);
    bool step(const int32_t* ids, int n, StepResult& r);  // false: id out of range
    void reset();
    void evict(int slot);  // leaves the slot empty (failed copy)
    int slot_of(int expert) const;

    int E, S, policy;
    int64_t step_index;
    std::vector<int32_t> slot_expert;
    std::vector<uint32_t> use_count;
    std::vector<int64_t> stamp;

   private:
    int pick_victim() const;
    std::vector<int32_t> expert_slot;
    std::vector<uint8_t> pinned;
};

void group_pairs(const int32_t* ids, int n_pairs, int n_experts, int32_t* offsets, int32_t* perm);

// ---- weight layout on the device -------------------------------------------
//
// A quantised matrix W[N][K] (N % 32 == 0, K % 64 == 0) is stored as a blob of
// two regions, tiled so that lane l of a warp owns row 32*rt + l of row tile rt
// and every warp-wide 16-byte load is 512 contiguous bytes:
//   codes: 16-byte chunk c (codes 32c..32c+31 of the row, canonical nibble
//          order) of row n at ((rt * K/32 + c) * 32 + lane) * 16;
//   sb:    (scale, bias) of group g as one 32-bit word (scale in the low half)
//          at N*K/2 + ((rt * K/64 + g) * 32 + lane) * 4.
// An expert blob is [gate (I x d)][up (I x d)][down (d x I)]; its size equals
// the canonical byte count, 27 * I * d / 16.

MOE_HD inline size_t qmat_bytes(int N, int K) { return (size_t)N * (size_t)K / 2 + (size_t)N * (size_t)K / 16; }
MOE_HD inline size_t expert_blob_bytes(int d, int inter) { return 2 * qmat_bytes(inter, d) + qmat_bytes(d, inter); }

// Repack one canonical matrix into the tiled blob format at dst.
void repack_qmatrix(const moe_qmatrix& m, int N, int K, uint8_t* dst);

// ---- kernel work lists -------------------------------------------------------
//
// A list of distinct experts ("items") and, per item, the (token, rank) pairs
// it serves. Pair p reads input row p / x_div (x_div is a launch argument:
// k for the routed gate/up, 1 otherwise) and writes output row p.

template <int MAXI, int MAXP>
struct WorkList {
    int n_items;
    const uint8_t* w[MAXI];   // expert blob base (slot, staging or shared)
    int16_t begin[MAXI + 1];  // pair ranges within pair[]
    int16_t pair[MAXP];
};
using SmallList = WorkList<16, 64>;
using LargeList = WorkList<256, 1024>;

struct RouterParams {
    const uint16_t* x;  // [T][d] bf16
    int T, d, E, k;
    const uint8_t* codes;  // [E][d]
    const uint32_t* sb;    // [E][d/64] (scale | bias << 16)
    const float* zbias;    // [E] or null
    float* logits;         // scratch [T][E]
    unsigned* counters;    // scratch, one per token block, zero between launches
    int32_t* ids;          // [T][k]
    float* gates;          // [T][k]
};

cudaError_t launch_router(const RouterParams& p, cudaStream_t s);

// h[pair][inter] = act(Wg x) * (Wu x) for every pair of every item.
template <class L>
cudaError_t launch_gateup(const uint16_t* x, int d, int inter, int act, int x_div, const L& list, float* h,
                          cudaStream_t s);

// out[pair][d] = Wd h[pair] for every pair of every item (down region of the blob).
template <class L>
cudaError_t launch_down(const float* h, int inter, int d, const L& list, float* out, cudaStream_t s);

// y[t][n] += sum_{r<k} gates[t][r] * o[t*k + r][n], added in rank order.
cudaError_t launch_combine(const float* o, const float* gates, int T, int k, int d, float* y, cudaStream_t s);

}  // namespace moe
