// Internal declarations of libmoe: host cache manager, weight layout and the
// kernel launchers. Not part of the public ABI (include/moe.h).
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
#pragma once

#include <cuda_fp16.h>
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
constexpr int kPromptMaxT = 4096;   // tokens of one layer-major prompt call

// Records a message for moe_last_error() (thread-local) and returns s.
moe_status set_error(moe_status s, const char* fmt, ...);

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device); thread-safe. The limit is a per-device
// property of a kernel, so every device that launches it needs its own call.
cudaError_t ensure_smem_attr(const void* kernel, size_t bytes);

// MOE_OK if the shapes are ones the library supports, else MOE_EINVAL.
moe_status check_shapes(const moe_shapes* s);

// ---- storage tier (store.cpp) ------------------------------------------------
//
// An expert file read into a host tier of H expert buffers. store_acquire
// returns the expert's bytes (reading them first if needed) and pins its
// entry; store_release unpins it. store_readahead queues reads for experts not
// in the tier, into entries nobody pins (never taking an entry read ahead and
// not yet fetched); with predicted (a guess from history) only into entries
// whose experts were fetched no more often, behind every fetch's read; without
// it (the reads of a call's own misses) never displacing an expert of the
// list. It returns how many it queued.

moe_status store_acquire(moe_expert_store* s, int expert, const uint8_t** out);
moe_status store_release(moe_expert_store* s, int expert);
int store_readahead(moe_expert_store* s, const int32_t* experts, int n, bool predicted);
bool store_contains(moe_expert_store* s, int expert);  // ready or being read
bool store_ready(moe_expert_store* s, int expert);
uint8_t* store_buffer(moe_expert_store* s, size_t* bytes);
int store_host_slots(const moe_expert_store* s);
const moe_shapes& store_shapes(const moe_expert_store* s);
bool store_attach(moe_expert_store* s, bool on);  // false: already attached

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
    std::vector<uint8_t> seen;  // scratch of step(), all zero between calls
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
//          at N*K/2 + ((rt * K/64 + g) * 32 + sb_pos(lane)) * 4.
// An expert blob is [gate (I x d)][up (I x d)][down (d x I)]; its size equals
// the canonical byte count, 27 * I * d / 16. Gate and up use this tiled
// format, down the column-sliced one below.

// Within each block of 32 scale/bias words (one per row of a 32-row tile),
// row r's word sits at position 4 (r % 8) + r / 8, so that rows g, g + 8,
// g + 16 and g + 24 (the rows of one MMA fragment lane) are 16 contiguous bytes.
MOE_HD inline int sb_pos(int r) { return 4 * (r & 7) + (r >> 3); }

MOE_HD inline size_t qmat_bytes(int N, int K) { return (size_t)N * (size_t)K / 2 + (size_t)N * (size_t)K / 16; }
MOE_HD inline size_t expert_blob_bytes(int d, int inter) { return 2 * qmat_bytes(inter, d) + qmat_bytes(d, inter); }

// Repack one canonical matrix into the tiled blob format at dst.
void repack_qmatrix(const moe_qmatrix& m, int N, int K, uint8_t* dst);

// The down matrix W[N][K] (N = d, K = intermediate) is column-sliced instead,
// so that the 32 columns one decode work unit needs are contiguous:
//   codes: 16-byte chunk c of row n at ((c * N/32 + rt) * 32 + lane) * 16,
//          i.e. 512-byte half-records ordered by (chunk, row tile);
//   sb:    the word of group g of row n at N*K/2 + ((g * N/32 + rt) * 32 + sb_pos(lane)) * 4,
//          i.e. 128-byte blocks ordered by (group, row tile).
// Same size as the tiled format.
void repack_down(const moe_qmatrix& m, int N, int K, uint8_t* dst);

// ---- router -----------------------------------------------------------------

struct RouterParams {
    const uint16_t* x;  // [T][d] bf16
    int T, d, E, k;
    const uint8_t* codes;  // [E][d]
    const uint32_t* sb;    // [E][d/64] (scale | bias << 16)
    const float* zbias;    // [E] or null
    float* logits;         // scratch [T][E]
    unsigned* counters;    // scratch, ceil(T/8) entries, zero between launches
    int32_t* ids;          // [T][k] device
    float* gates;          // [T][k] device
    unsigned long long* host_ids;  // [T][k] mapped pinned host memory (seq << 32 | id), or null
    uint32_t seq;
    float* zero;  // optional: zero_n floats set to zero by the launch (the decode output, which
    int zero_n;   // the expert FFN then adds into)
    // optional diagnostics: {earliest block start, latest block end} in
    // %globaltimer nanoseconds, merged with atomicMin / atomicMax; null = off
    unsigned long long* span;
};

// pdl: launch as a programmatic dependent of the previous kernel on the
// stream. The router then only prefetches its weights before it waits for
// that kernel to finish; it lets the next kernel start early as well.
cudaError_t launch_router(const RouterParams& p, cudaStream_t s, bool pdl = false);

// The ordered decode combine: y[t][n] = S + O_0 + ... + O_{k-1}, where S is
// the shared expert's share of token t (its cs chunk partials part0[t][c][n]
// summed in groups of cr chunks, the groups then added in order) and O_r the
// routed share of pair t*k + r (its cr chunk partials part1[t*k+r][c][n]
// summed in chunk order). The order depends on nothing but the shapes.
cudaError_t launch_part_reduce(const float* part0, const float* part1, int cs, int cr, int k, int d, int T, float* y,
                               cudaStream_t s, bool pdl);

// y[t][n] += sum_{r<k} gates[t][r] * o[t*k + r][n], added in rank order.
cudaError_t launch_combine(const float* o, const float* gates, int T, int k, int d, float* y, cudaStream_t s);

// ---- fused expert FFN (decode) --------------------------------------------------
//
// A list of expert "items", each with at most kFfnMaxNT (token, rank) pairs.
// Items come in two families, family 0 first: the shared expert (its pairs
// are token indices, gate 1) and the routed experts (pair p = t * k + r, gate
// gates[p]). Pair p of family f reads x row p / x_div and adds its
// gate-weighted FFN output into y row p / x_div. An item whose bytes are still
// being copied names a ready flag (index into `ready`) that must reach the
// list's epoch before its weights are read (the gate/up bytes and the down
// bytes have a flag each); -1 means resident.
//
// Device layout of an expert blob (see repack_qmatrix / repack_down):
// gate | up (records by 32-row tile, then group of 64 inputs) | down
// (column-sliced: the codes of 32 output rows x 32 intermediate inputs as
// 512-byte half-records ordered by (input slice, row tile), then the
// scale/bias words as 128-byte blocks ordered by (group, row tile)).

constexpr int kFfnMaxNT = 8;
constexpr int kFfnFams = 2;
constexpr int kFfnMaxUpd = 64;  // slot-table changes one launch can carry

struct FfnItem {
    const uint8_t* w;  // expert blob; null: a routed pair resolved on the device (see FfnArgs::ids)
    int16_t pb, np;    // pair range within pair[]
    int16_t ready;     // ready-flag index of the gate and up bytes, -1 if resident
    int16_t ready_dn;  // ready-flag index of the down bytes, -1 if resident
};

template <int MAXI, int MAXP>
struct FfnList {
    int n_items;
    uint32_t epoch;
    FfnItem item[MAXI];
    int16_t pair[MAXP];
};
using FfnSmall = FfnList<24, 96>;
using FfnLarge = FfnList<256, 1024>;

struct FfnFam {
    int n_items;  // consecutive items of the list; family 0 first
    int inter;    // intermediate size
    int x_div;    // x (and y) row of pair p is p / x_div
};

struct FfnArgs {
    const uint16_t* x;  // [T][d] bf16
    int d, act;
    FfnFam fam[kFfnFams];
    const float* gates;  // [T * k], pair p's gate (family 1)
    float* y;            // [T][d] fp32, zero on entry: every unit adds its share
    const uint32_t* ready;
    unsigned* err;
    // optional diagnostics: per CTA, %globaltimer at kFfnTracePoints moments
    // (start, first weights landed, first unit's h ready, first unit done,
    // end); null = off
    unsigned long long* trace;
    // optional diagnostics: {earliest CTA start, latest CTA end}, as for the router
    unsigned long long* span;
    // Items with w == null name one routed pair p (pair[pb]) whose expert is
    // ids[p], written by the router launch before this one: if the expert's
    // slot (slot_of[expert], -1 = not resident) holds it at the start of the
    // call, the item's weights are slots + slot * ebytes; otherwise the item is
    // skipped (its expert is a miss, done by a later launch).
    const int32_t* ids;
    const int32_t* slot_of;
    const uint8_t* slots;
    size_t ebytes;
    // Ordered combine (null: every unit adds into y with fp32 atomics). Unit
    // (item, c) of family f stores its gate-weighted share of row q (pair
    // value p = pair[pb + q]: a token for family 0, a pair t*k + r for family
    // 1) at part[f] + (p * part_c[f] + c) * d, where part_c[f] = inter / 32;
    // launch_part_reduce then sums them per token in a fixed order.
    float* part[kFfnFams];
    int part_c[kFfnFams];
    // The launch takes the kernel shape for at least min_nt rows per item.
    // The shape sets how a unit's gate/up group sums are split over warps, so
    // the ordered combine gives every launch of a multi-token call the same
    // one (its items can fall into the hit and miss launches differently on
    // another call).
    int min_nt;
    // Slot-table changes of this call's cache step, written into slot_of once
    // the previous kernel on the stream (the launch that read the table) has
    // finished: slot_of[upd_expert[i]] = upd_slot[i].
    int n_upd;
    int16_t upd_expert[kFfnMaxUpd];
    int16_t upd_slot[kFfnMaxUpd];
};
constexpr int kFfnTracePoints = 5;

// One launch computing, for every item, unit by unit (32 intermediate rows at
// a time), h = act(W_g x) * (W_u x) and the matching slice of W_d h, added
// gate-weighted into y.
// pdl: launch as a programmatic dependent of the previous kernel on the
// stream: the weights stream and gate/up run as soon as SMs are free, and
// each CTA waits for that kernel to finish before its first add into y.
template <class L>
cudaError_t launch_ffn(const FfnArgs& a, const L& list, cudaStream_t s, bool pdl = false);

// Launch configuration with the programmatic-dependent-launch attribute set
// when pdl (attr must outlive the launch call).
inline cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                                        cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t c{};
    c.gridDim = grid;
    c.blockDim = block;
    c.dynamicSmemBytes = smem;
    c.stream = s;
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = pdl ? 1 : 0;
    return c;
}

// Bytes of the down matrix of one expert in the column-sliced layout (equal to
// qmat_bytes(d, inter)).
MOE_HD inline size_t down_codes_bytes(int d, int inter) { return (size_t)d * (size_t)inter / 2; }

// ---- prefill grouped GEMM (tcgen05) -------------------------------------------
//
// A prefill chunk's experts as two grouped GEMMs on the tensor cores:
// gate/up (h = act(W_g x) * W_u x for every item and token) and down
// (o = W_d h). Weights are dequantised to fp16 by producer warps; the token
// rows (x converted to fp16, or h in fp16) are loaded by TMA; accumulators
// are fp32 in tensor memory. An item is one expert and up to kPfMaxN rows:
// family 0 is the shared expert over every token (rows 0..T-1), family 1 a
// routed expert over its pairs, which occupy the sorted positions
// pb..pb+np-1 (sorted position -> pair index in `pair`).

constexpr int kPfMaxN = 128;

struct PfItem {
    const uint8_t* w;  // expert blob: gate | up | down in the tiled layout
    int32_t pb, np;    // first row and row count (sorted positions, or tokens for family 0)
    int32_t ready;     // ready-flag index of the gate and up bytes, -1 if resident
    int32_t ready_dn;  // ready-flag index of the down bytes, -1 if resident
};

struct PfArgs {
    const PfItem* items;  // device, n_items entries, family 0 first
    int n_items, n_fam0;
    int d, act, T, k;
    int inter[2];         // intermediate size per family
    const int32_t* pair;  // device [P]: sorted position -> pair index t*k + r
    __half* h[2];         // gate/up output, fp16: family 0 [T][inter0], family 1 [P][inter1]
    float* out[2];        // down output, fp32: family 0 -> [T][d] by token, family 1 -> [T*k][d] by pair
    const uint32_t* ready;
    uint32_t epoch;
    unsigned* err;
    // K split of the tiles of a launch that has too few to fill the GPU (the
    // shared expert's 128-row tiles alone leave most SMs idle): each of a
    // tile's ks[fam] parts covers a slice of K and writes its fp32 sums to
    // `part` ([split tile][part][kPfMaxN columns][128 rows], family 0's split
    // tiles first); a second kernel adds them in part order and runs the
    // epilogue. part_cap is the buffer's size in floats; with a null buffer no
    // tile is split. ks is set by launch_pf_gemm.
    float* part;
    size_t part_cap;
    int ks[2];
    // optional diagnostics: a count, then the first kPfFailRecords waits of
    // the launch that expired (block, warp, which wait, job, K-block); null = off
    unsigned long long* trace;
};
constexpr int kPfFailRecords = 31;

// Converts the chunk's token rows to fp16 for the gate/up B operand:
// xs[t] = x[t] for t < T and xg[i] = x[pair[i] / k] for i < P.
cudaError_t launch_pf_gather(const uint16_t* x, int T, int d, const int32_t* pair, int P, int k, __half* xs,
                             __half* xg, cudaStream_t s);

// phase 1: gate/up (B rows from xs / xg, K = d); phase 2: down (B rows from
// h[0] / h[1], K = inter). `rows[f]` is the number of rows of family f's B
// matrix (T for family 0, P for family 1).
// Floats of K-split partial sums a layer with these shapes needs for its
// prefill GEMMs on the current device.
size_t pf_part_floats(int d, int inter0);

// One phase of the grouped GEMM: the GEMM launch, and the K-split epilogue
// launch when tiles are split; *launched (if given) gets the launch count.
cudaError_t launch_pf_gemm(const PfArgs& a, int phase, const void* b0, const void* b1, const int rows[2],
                           cudaStream_t s, int* launched = nullptr);

}  // namespace moe
