// libmoe C ABI: contexts, layers, weight loading, routing, the expert cache
// step with miss streaming, and the layer forward.
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
//
// One decode call maps the three phases of [P1] §2.4 / §8.2 onto the GPU:
//   cb1  the router kernel publishes each id to mapped host memory as it is
//        chosen, tagged with the call number;
//   io   host LFU/LRU step; one cudaMemcpyAsync per miss from the pinned pool
//        into its HBM slot (or, for a bypass, into the staging arena) on the
//        context's copy stream, each followed by a stream write of the call's
//        round number into that slot's ready flag ([P3] "读取完成后，算子才可以
//        使用切片": a hit is ready at once, a miss when its read completes, and
//        the round number keeps a stale "ready" from being reused);
//   cb2  one fused kernel runs the shared expert and every routed expert -
//        the shared expert and the hits at once, each miss as soon as its flag
//        shows the current round, so the shared branch overlaps the reads
//        ([P1] §2.4: it does not depend on the routed experts) - and writes
//        y = shared + the gate-weighted routed outputs in rank order.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <type_traits>
#include <vector>

#include "moe_internal.h"

namespace moe {

static thread_local char g_err[512] = "";

moe_status set_error(moe_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

cudaError_t ensure_smem_attr(const void* kernel, size_t bytes) {
    struct Done {
        const void* kernel;
        int device;
    };
    static std::mutex mu;
    static std::vector<Done> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const Done& x : done)
        if (x.kernel == kernel && x.device == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done.push_back(Done{kernel, dev});
    return e;
}

// One 32-bit word of 8 codes (elements k0..k7 of the canonical row, byte j =
// k_2j | k_2j+1 << 4) in the device order: nibble i holds element
// [0,2,4,6,1,3,5,7][i], so that masking with 0x000F000F (and the same on the
// word shifted by 4, 8, 12) yields the consecutive pairs (k0,k1), (k2,k3),
// (k4,k5), (k6,k7) in the two halves of a 32-bit register.
uint32_t device_nibble_order(const uint8_t* b) {
    uint32_t k[8];
    for (int j = 0; j < 4; ++j) {
        k[2 * j] = b[j] & 15u;
        k[2 * j + 1] = b[j] >> 4;
    }
    static const int order[8] = {0, 2, 4, 6, 1, 3, 5, 7};
    uint32_t w = 0;
    for (int i = 0; i < 8; ++i) w |= k[order[i]] << (4 * i);
    return w;
}

// Device layout of one [N][K] int4 matrix: 32-row tiles, each a run of K/64
// records, one per group of 64 inputs. Record (rt, g), at (rt * K/64 + g) *
// 1152: the codes of chunk 2g for rows rt*32 + lane (16 bytes per lane), the
// codes of chunk 2g+1 likewise, then one word per row: fp16 scale | fp16 bias
// << 16, row `lane` at position sb_pos(lane). So a row tile's consecutive
// groups are one contiguous copy.
void repack_qmatrix(const moe_qmatrix& m, int N, int K, uint8_t* dst) {
    const int G = K / 64;
    for (int n = 0; n < N; ++n) {
        const int rt = n >> 5, lane = n & 31;
        const uint8_t* src = m.codes + (size_t)n * (size_t)(K / 2);
        for (int g = 0; g < G; ++g) {
            uint8_t* rec = dst + ((size_t)rt * G + g) * 1152;
            for (int h = 0; h < 2; ++h) {
                uint32_t* o = reinterpret_cast<uint32_t*>(rec + h * 512 + lane * 16);
                for (int w = 0; w < 4; ++w) o[w] = device_nibble_order(src + (size_t)(2 * g + h) * 16 + 4 * w);
            }
            const size_t i = (size_t)n * G + g;
            reinterpret_cast<uint32_t*>(rec + 1024)[sb_pos(lane)] = (uint32_t)m.scale[i] | ((uint32_t)m.bias[i] << 16);
        }
    }
}

void repack_down(const moe_qmatrix& m, int N, int K, uint8_t* dst) {
    const int G = K / 64, RT = N / 32;
    uint8_t* sb = dst + down_codes_bytes(N, K);
    for (int n = 0; n < N; ++n) {
        const int rt = n >> 5, lane = n & 31;
        const uint8_t* src = m.codes + (size_t)n * (size_t)(K / 2);
        for (int c = 0; c < K / 32; ++c) {
            uint32_t* o = reinterpret_cast<uint32_t*>(dst + (((size_t)c * RT + rt) * 32 + lane) * 16);
            for (int w = 0; w < 4; ++w) o[w] = device_nibble_order(src + (size_t)c * 16 + 4 * w);
        }
        for (int g = 0; g < G; ++g) {
            const size_t i = (size_t)n * G + g;
            reinterpret_cast<uint32_t*>(sb)[((size_t)g * RT + rt) * 32 + sb_pos(lane)] =
                (uint32_t)m.scale[i] | ((uint32_t)m.bias[i] << 16);
        }
    }
}

}  // namespace moe

using namespace moe;

#define CUDA_TRY(call)                                                                                 \
    do {                                                                                               \
        cudaError_t e_ = (call);                                                                       \
        if (e_ != cudaSuccess)                                                                         \
            return set_error(MOE_ECUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, \
                             __LINE__);                                                                \
    } while (0)

namespace {

constexpr int kKinds = 8;
enum Kind { K_ROUTER = 0, K_FFN = 1, K_COMBINE = 2, K_GEMM_GU = 3, K_GEMM_DN = 4, K_GATHER = 5, K_FFN_MISS = 6 };
constexpr double kHostWaitLimitS = 10.0;  // longest the host waits for the routing of one call
// Rounds of ready-word source values kept in pinned memory. A round's entry is
// rewritten kEpochRing calls later, long after its copies ran: every call
// waits, on the host, for routing that follows the previous call's kernels.
constexpr uint32_t kEpochRing = 4096;


struct ProfRec {
    int kind;
    cudaEvent_t a, b;
    double bytes, flops;
};

struct WaitRec {
    cudaEvent_t ffn_start, copies_done;
};

// Timeline diagnostics, on when the environment variable MOE_TRACE_FILE
// names an output file at context creation: every launch gets a device span
// {earliest block start, latest block end} in %globaltimer nanoseconds, and
// the host records its own steps in CLOCK_REALTIME nanoseconds; the file is
// written when the context is destroyed.
constexpr int kTraceSpans = 1 << 18;

struct TraceLaunch {
    int kind, layer;
    uint32_t seq;
    int slot;
    uint64_t t_host;
};
struct TraceHost {
    const char* what;
    int layer;
    uint32_t seq;
    uint64_t t;
};

uint64_t realtime_ns() {
    timespec ts;
    clock_gettime(CLOCK_REALTIME, &ts);
    return (uint64_t)ts.tv_sec * 1000000000ull + (uint64_t)ts.tv_nsec;
}

__global__ void read_globaltimer(unsigned long long* out) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    *out = t;
}

}  // namespace

struct moe_ctx {
    int device = 0;
    cudaStream_t copy_stream = nullptr;
    uint8_t* staging = nullptr;  // transient arena for bypassed experts
    size_t staging_bytes = 0;
    cudaEvent_t staging_free = nullptr;  // after the last kernels that read staging
    bool profiling = false;
    std::vector<ProfRec> prof;
    struct Acc {
        uint64_t n = 0;
        double ms = 0, bytes = 0, flops = 0;
    } acc[kKinds];
    std::vector<cudaEvent_t> timing_pool;
    uint64_t launches = 0;          // kernels launched by this context's layers
    unsigned* err_host = nullptr;   // mapped pinned word that kernels report expired waits into
    unsigned* err_dev = nullptr;
    uint32_t err_generation = 0;  // bumped whenever a kernel reported an expired wait
    long fail_copy_at = -1;  // test hook: the n-th miss copy from now reports failure
    long copies_issued = 0;
    // timeline diagnostics (see TraceLaunch)
    std::string trace_path;
    unsigned long long* trace_spans = nullptr;  // device [kTraceSpans][2]
    std::vector<TraceLaunch> trace_launches;
    std::vector<TraceHost> trace_host;

    unsigned long long* trace_span(int kind, int layer, uint32_t seq) {
        if (!trace_spans || (int)trace_launches.size() >= kTraceSpans) return nullptr;
        const int slot = (int)trace_launches.size();
        trace_launches.push_back(TraceLaunch{kind, layer, seq, slot, realtime_ns()});
        return trace_spans + 2 * slot;
    }
    void trace_mark(const char* what, int layer, uint32_t seq) {
        if (trace_spans) trace_host.push_back(TraceHost{what, layer, seq, realtime_ns()});
    }

    cudaEvent_t timing_event() {
        if (!timing_pool.empty()) {
            cudaEvent_t e = timing_pool.back();
            timing_pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
};

struct moe_layer {
    moe_ctx* ctx = nullptr;
    int id = 0;  // creation order within the process (diagnostics)
    moe_shapes sh{};
    int S = 0, policy = 0;
    size_t ebytes = 0, shared_bytes = 0, router_bytes = 0;
    uint8_t* d_router_codes = nullptr;
    uint32_t* d_router_sb = nullptr;
    uint8_t* d_shared = nullptr;
    uint8_t* d_slots = nullptr;
    int32_t* d_slot_of = nullptr;  // device copy of the cache's expert -> slot map (-1 = not resident)
    std::vector<int32_t> slot_before;  // slot table before the current step (host)
    uint8_t* h_pool = nullptr;    // pinned, E * ebytes
    uint32_t* d_ready = nullptr;  // ready flags: slots, then staging entries
    uint32_t epoch = 0;           // round number of the current call
    // pinned source words of the ready-word copies: entry e % kEpochRing holds
    // epoch e while that round's copies may still be queued
    uint32_t* h_epochs = nullptr;
    uint32_t seq = 0;             // routing publication number
    HostCache cache;
    StepResult step;
    cudaEvent_t ev_done = nullptr;     // end of the layer's last call
    cudaEvent_t ev_pending = nullptr;  // copies issued by moe_cache_step
    bool pending = false;              // ev_pending recorded since the last forward
    cudaStream_t last_stream = nullptr;  // stream of the last call that recorded ev_done
    bool have_last_stream = false;
    bool loaded = false;
    // scratch, sized for cap_T tokens per call
    int cap_T = 0;
    float* d_logits = nullptr;
    unsigned* d_rcount = nullptr;  // router block counters
    int32_t* d_ids = nullptr;
    float* d_gates = nullptr;
    float* d_o = nullptr;      // prefill: routed-expert outputs by pair [cap_T * k][d]
    unsigned long long* h_pub = nullptr;  // mapped pinned [cap_T * k]: seq << 32 | id
    unsigned long long* h_pub_dev = nullptr;
    std::vector<int32_t> h_ids;           // ids of the current call, read from h_pub
    // prefill (T > kDecodeMaxT): fp16 token rows (x of the shared expert
    // [cap_T][d], then x gathered per sorted pair [pairs][d]), fp16 h (shared
    // [cap_T][d_ff_shared], then routed [pairs][d_ff]), and the item/pair
    // table (pinned host copy and its device twin)
    __half* d_x16 = nullptr;
    __half* d_h16 = nullptr;
    // prefill: K-split partial sums (the shared expert's tiles)
    float* d_part = nullptr;
    size_t part_floats = 0;
    uint8_t* d_pf = nullptr;
    uint8_t* h_pf = nullptr;
    size_t pf_bytes = 0;
    uint32_t err_generation = 0;  // the context's value when the counters were last known zero
    std::vector<int32_t> offsets, perm;
    moe_stats stats{};
    std::vector<WaitRec> waits;
    // storage tier (moe_layer_create_streamed): misses are fetched from the
    // store's host tier instead of h_pool; an entry stays pinned until the
    // copy that reads it has finished (the event recorded behind it on the
    // copy stream). route_hist counts, per expert, the steps that routed to it.
    moe_expert_store* store = nullptr;
    uint8_t* store_pinned = nullptr;  // the tier buffer registered with CUDA
    struct StorePin {
        std::vector<int> experts;
        cudaEvent_t ev;
    };
    std::deque<StorePin> store_pins;  // in copy-stream order
    std::vector<cudaEvent_t> store_events;  // free events for store_pins
    std::vector<uint32_t> route_hist;
    // predictive prefetch into HBM (moe_layer_set_prefetch): one spare expert
    // buffer, refilled after each call's misses with the most-routed expert
    // that is not resident; a later miss of that expert copies from it
    bool prefetch = false;
    uint8_t* d_spare = nullptr;
    int spare_expert = -1;           // the expert the spare buffer holds (or is being filled with)
    int spare_miss_expert = -1;      // this call's miss served from the spare buffer, or -1
    int spare_miss_slot = -1;        // ... and the slot it goes into (-1: it bypasses)
    bool spare_call = false;         // the current call may serve a miss from the spare buffer
    cudaEvent_t ev_spare_ready = nullptr;  // copy stream: the last prefetch into the spare landed
    cudaEvent_t ev_spare_free = nullptr;   // compute stream: the last reads of the spare are done
    bool spare_free_recorded = false;
    uint64_t prefetch_issued = 0, prefetch_used = 0;
    // ordered (deterministic) decode combine: per-unit partial rows, then a
    // reduce in a fixed order (moe_layer_set_deterministic)
    bool deterministic = false;
    float* d_dpart = nullptr;
    size_t dpart_floats = 0;
    // the last one-token call's resident FFN launch, for moe_layer_replay_resident
    bool record_resident = false;
    bool have_resident = false;
    FfnArgs resident_args{};
    FfnSmall resident_list{};

    moe_layer(int E, int S_, int pol) : cache(E, S_, pol) {}
};

moe_status moe::check_shapes(const moe_shapes* s) {
    if (!s) return set_error(MOE_EINVAL, "shapes is NULL");
    if (s->d_model < 256 || s->d_model > kMaxDModel || s->d_model % 256 != 0)
        return set_error(MOE_EINVAL, "d_model %d must be a multiple of 256 in [256, %d]", s->d_model, kMaxDModel);
    if (s->d_ff < 64 || s->d_ff % 64 != 0 || s->d_ff > kMaxDModel)
        return set_error(MOE_EINVAL, "d_ff %d must be a multiple of 64 in [64, %d]", s->d_ff, kMaxDModel);
    if (s->d_ff_shared < 64 || s->d_ff_shared % 64 != 0 || s->d_ff_shared > kMaxDModel)
        return set_error(MOE_EINVAL, "d_ff_shared %d must be a multiple of 64 in [64, %d]", s->d_ff_shared,
                         kMaxDModel);
    if (s->n_experts < 1 || s->n_experts > kMaxExperts)
        return set_error(MOE_EINVAL, "n_experts %d out of [1, %d]", s->n_experts, kMaxExperts);
    if (s->top_k < 1 || s->top_k > kMaxTopK || s->top_k > s->n_experts)
        return set_error(MOE_EINVAL, "top_k %d out of [1, min(%d, n_experts)]", s->top_k, kMaxTopK);
    if (s->act != 0 && s->act != 1) return set_error(MOE_EINVAL, "act %d must be 0 (GELU tanh) or 1 (SiLU)", s->act);
    return MOE_OK;
}

namespace {

// Items of one prefill call of T tokens: the shared expert per block of
// kPfMaxN tokens, and each routed expert's pairs in pieces of at most kPfMaxN.
size_t pf_max_items(const moe_shapes& s, int T) {
    const size_t pairs = (size_t)T * s.top_k;
    return (T + kPfMaxN - 1) / kPfMaxN + std::min<size_t>(s.n_experts, pairs) + pairs / kPfMaxN;
}

void free_scratch(moe_layer* L) {
    cudaFree(L->d_logits);
    cudaFree(L->d_rcount);
    cudaFree(L->d_ids);
    cudaFree(L->d_gates);
    cudaFree(L->d_o);
    cudaFree(L->d_x16);
    cudaFree(L->d_h16);
    cudaFree(L->d_part);
    L->d_part = nullptr;
    L->part_floats = 0;
    cudaFree(L->d_pf);
    cudaFreeHost(L->h_pf);
    L->d_x16 = L->d_h16 = nullptr;
    L->d_pf = L->h_pf = nullptr;
    L->pf_bytes = 0;
    cudaFreeHost(L->h_pub);
    L->d_logits = nullptr;
    L->d_rcount = nullptr;
    L->d_ids = nullptr;
    L->d_gates = nullptr;
    L->d_o = nullptr;
    L->h_pub = L->h_pub_dev = nullptr;
    L->cap_T = 0;
}

// Scratch for up to T tokens per call (grows; never shrinks).
moe_status ensure_scratch(moe_layer* L, int T) {
    if (T <= L->cap_T) return MOE_OK;
    if (L->ev_done) CUDA_TRY(cudaEventSynchronize(L->ev_done));  // the old buffers may still be in use
    free_scratch(L);
    const moe_shapes& s = L->sh;
    const size_t pairs = (size_t)T * s.top_k;
    const int blocks = (T + 7) / 8;
    bool ok = cudaMalloc(&L->d_logits, sizeof(float) * T * s.n_experts) == cudaSuccess &&
              cudaMalloc(&L->d_rcount, sizeof(unsigned) * blocks) == cudaSuccess &&
              cudaMemset(L->d_rcount, 0, sizeof(unsigned) * blocks) == cudaSuccess &&
              cudaMalloc(&L->d_ids, sizeof(int32_t) * pairs) == cudaSuccess &&
              cudaMalloc(&L->d_gates, sizeof(float) * pairs) == cudaSuccess &&
              cudaMalloc(&L->d_o, sizeof(float) * pairs * s.d_model) == cudaSuccess &&
              cudaHostAlloc(&L->h_pub, sizeof(unsigned long long) * pairs, cudaHostAllocMapped) == cudaSuccess &&
              cudaHostGetDevicePointer(&L->h_pub_dev, L->h_pub, 0) == cudaSuccess;
    if (ok && T > kDecodeMaxT) {
        const size_t items = pf_max_items(s, T);
        L->pf_bytes = items * sizeof(PfItem) + pairs * sizeof(int32_t);
        ok = cudaMalloc(&L->d_x16, sizeof(__half) * ((size_t)T + pairs) * s.d_model) == cudaSuccess &&
             cudaMalloc(&L->d_h16, sizeof(__half) * ((size_t)T * s.d_ff_shared + pairs * s.d_ff)) == cudaSuccess &&
             cudaMalloc(&L->d_pf, L->pf_bytes) == cudaSuccess &&
             cudaHostAlloc(&L->h_pf, L->pf_bytes, cudaHostAllocDefault) == cudaSuccess;
        L->part_floats = pf_part_floats(s.d_model, s.d_ff_shared);
        if (ok && L->part_floats) ok = cudaMalloc(&L->d_part, sizeof(float) * L->part_floats) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        free_scratch(L);
        return set_error(MOE_ENOMEM, "scratch allocation for %d tokens failed", T);
    }
    memset(L->h_pub, 0, sizeof(unsigned long long) * pairs);
    L->h_ids.assign(pairs, 0);
    L->cap_T = T;
    return MOE_OK;
}

// Partial rows of the ordered decode combine for T tokens: the shared
// expert's chunks per token, then the routed chunks per pair.
size_t det_part_floats(const moe_shapes& s, int T) {
    return (size_t)T * ((size_t)(s.d_ff_shared / 32) + (size_t)s.top_k * (s.d_ff / 32)) * s.d_model;
}

moe_status ensure_det_scratch(moe_layer* L, int T) {
    const size_t need = det_part_floats(L->sh, T);
    if (need <= L->dpart_floats) return MOE_OK;
    if (L->ev_done) CUDA_TRY(cudaEventSynchronize(L->ev_done));  // the old buffer may still be in use
    cudaFree(L->d_dpart);
    L->d_dpart = nullptr;
    L->dpart_floats = 0;
    if (cudaMalloc(&L->d_dpart, sizeof(float) * need) != cudaSuccess) {
        cudaGetLastError();
        return set_error(MOE_ENOMEM, "ordered-combine scratch for %d tokens (%zu floats) failed", T, need);
    }
    L->dpart_floats = need;
    return MOE_OK;
}

// Staging arena for bypassed experts, shared by the context's layers.
moe_status ensure_staging(moe_ctx* C, size_t bytes) {
    if (bytes <= C->staging_bytes) return MOE_OK;
    CUDA_TRY(cudaEventSynchronize(C->staging_free));
    cudaFree(C->staging);
    C->staging = nullptr;
    C->staging_bytes = 0;
    if (cudaMalloc(&C->staging, bytes) != cudaSuccess) {
        cudaGetLastError();
        return set_error(MOE_ENOMEM, "staging arena of %zu bytes failed", bytes);
    }
    C->staging_bytes = bytes;
    return MOE_OK;
}

struct Prof {
    moe_ctx* C;
    cudaStream_t s;
    ProfRec r{};
    Prof(moe_ctx* c, cudaStream_t st, int kind, double bytes, double flops) : C(c), s(st) {
        ++C->launches;
        if (!C->profiling) return;
        r.kind = kind;
        r.bytes = bytes;
        r.flops = flops;
        r.a = C->timing_event();
        r.b = C->timing_event();
        cudaEventRecord(r.a, s);
    }
    ~Prof() {
        if (!C->profiling) return;
        cudaEventRecord(r.b, s);
        C->prof.push_back(r);
    }
};

void drain_prof(moe_ctx* C) {
    for (ProfRec& r : C->prof) {
        cudaEventSynchronize(r.b);
        float ms = 0;
        cudaEventElapsedTime(&ms, r.a, r.b);
        C->acc[r.kind].n += 1;
        C->acc[r.kind].ms += ms;
        C->acc[r.kind].bytes += r.bytes;
        C->acc[r.kind].flops += r.flops;
        C->timing_pool.push_back(r.a);
        C->timing_pool.push_back(r.b);
    }
    C->prof.clear();
}

// Exposed copy time: how long the routed-expert kernel had misses still
// landing after it started (zero when every copy finished before it).
void drain_waits(moe_layer* L) {
    for (WaitRec& w : L->waits) {
        cudaEventSynchronize(w.copies_done);
        cudaEventSynchronize(w.ffn_start);
        float ms = 0;
        if (cudaEventElapsedTime(&ms, w.ffn_start, w.copies_done) == cudaSuccess && ms > 0)
            L->stats.exposed_copy_us += 1000.0 * ms;
        cudaGetLastError();
        L->ctx->timing_pool.push_back(w.ffn_start);
        L->ctx->timing_pool.push_back(w.copies_done);
    }
    L->waits.clear();
}

moe_status check_err_word(moe_ctx* C) {
    if (const unsigned ew = *(volatile unsigned*)C->err_host) {
        *(volatile unsigned*)C->err_host = 0;
        ++C->err_generation;  // a kernel that gave up may have left counters non-zero
        return set_error(MOE_ETIMEOUT, "a bounded device wait expired in an earlier kernel (code %u)", ew);
    }
    return MOE_OK;
}

// The ready flags of one miss: its gate/up bytes and its down bytes land
// separately, so that its gate/up work can run while its down bytes are still
// being copied.
struct MissFlags {
    int gu = -1, dn = -1;
};

// Misses per ready-flag group: a group's flag is written after the group's
// copies, so a small call (decode) waits on one flag per part and a large one
// (a prefill chunk) can start on its first experts while the rest still copy.
constexpr int kFlagGroup = 8;

// Issue the copies of one cache step's misses. A slot miss lands in its slot,
// a bypass in the next staging entry. With flags wanted (ready_of_miss),
// after each group of kFlagGroup misses the copy stream writes `epoch` into
// that group's flags. With split, each expert is copied in two parts, every
// miss's gate and up matrices first and then every miss's down matrix, each
// part with its own flag (group g: 2g for gate/up, 2g + 1 for down), so that
// gate/up work overlaps the down copies; a copy costs a few microseconds on
// top of its bytes, so calls with many misses (prefill) copy each expert
// whole and flag 2g covers both parts. On failure every slot this step
// filled but whose copy is not known good is emptied, so the table never
// claims bytes that are missing.
// Release the tier entries whose copies have finished (all of them, waiting
// for each copy, with wait_all).
moe_status release_store_pins(moe_layer* L, bool wait_all) {
    while (!L->store_pins.empty()) {
        moe_layer::StorePin& p = L->store_pins.front();
        if (wait_all) {
            CUDA_TRY(cudaEventSynchronize(p.ev));
        } else {
            const cudaError_t q = cudaEventQuery(p.ev);
            if (q == cudaErrorNotReady) break;
            if (q != cudaSuccess) CUDA_TRY(q);
        }
        for (int e : p.experts) store_release(L->store, e);
        L->store_events.push_back(p.ev);
        L->store_pins.pop_front();
    }
    return MOE_OK;
}

// Record an event on the copy stream behind the copies issued so far; the
// listed experts' tier entries are released once it completes.
moe_status pin_until_copied(moe_layer* L, std::vector<int> experts) {
    if (experts.empty()) return MOE_OK;
    cudaEvent_t ev = nullptr;
    if (!L->store_events.empty()) {
        ev = L->store_events.back();
        L->store_events.pop_back();
    } else {
        CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    }
    const cudaError_t e = cudaEventRecord(ev, L->ctx->copy_stream);
    if (e != cudaSuccess) {
        L->store_events.push_back(ev);
        CUDA_TRY(e);
    }
    L->store_pins.push_back(moe_layer::StorePin{std::move(experts), ev});
    return MOE_OK;
}

// issue_miss_copies for a layer that streams from an expert store: the same
// destinations, flags, parts and failure handling, but each expert's source
// is its entry in the store's host tier. Misses already in the tier are
// copied first; the reads of the others are queued at once (as many as the
// tier has entries to give), and each copy is issued as soon as its read
// lands, so reads, copies and the kernels waiting on the flags overlap. An
// entry stays pinned until its last copy has finished. Nothing is merged:
// tier entries are not consecutive experts.
moe_status issue_store_copies(moe_layer* L, const StepResult& r, bool with_bypass, uint32_t epoch,
                              std::vector<MissFlags>* ready_of_miss, bool split) {
    moe_ctx* C = L->ctx;
    L->h_epochs[epoch % kEpochRing] = epoch;
    moe_status st = release_store_pins(L, false);
    if (st != MOE_OK) return st;
    if (with_bypass && r.bypass > 0) {
        st = ensure_staging(C, (size_t)r.bypass * L->ebytes);
        if (st != MOE_OK) return st;
        CUDA_TRY(cudaStreamWaitEvent(C->copy_stream, C->staging_free, 0));
    }
    if (ready_of_miss) ready_of_miss->assign(r.miss_experts.size(), MissFlags{});
    struct Copy {
        size_t i;
        uint8_t* dst;
        const uint8_t* src;
    };
    std::vector<Copy> copies;
    int nb = 0;
    for (size_t i = 0; i < r.miss_experts.size(); ++i) {
        const int slot = r.miss_slots[i];
        if (slot < 0 && !with_bypass) continue;
        uint8_t* dst = slot >= 0 ? L->d_slots + (size_t)slot * L->ebytes : C->staging + (size_t)(nb++) * L->ebytes;
        copies.push_back(Copy{i, dst, nullptr});
    }
    std::stable_partition(copies.begin(), copies.end(),
                          [&](const Copy& c) { return store_ready(L->store, r.miss_experts[c.i]); });
    std::vector<int32_t> wanted;
    for (const Copy& c : copies) wanted.push_back(r.miss_experts[c.i]);
    store_readahead(L->store, wanted.data(), (int)wanted.size(), false);
    const bool flags = ready_of_miss != nullptr;
    // a split copy reads its entry twice, so every entry of the call stays
    // pinned across both parts: only when the tier can hold them all
    split = split && flags && copies.size() <= (size_t)store_host_slots(L->store);
    const int parts = split ? 2 : 1;
    const size_t gu_bytes = 2 * qmat_bytes(L->sh.d_ff, L->sh.d_model);
    auto set_flag = [&](int flag) {
        return cudaMemcpyAsync(L->d_ready + flag, L->h_epochs + epoch % kEpochRing, sizeof(uint32_t),
                               cudaMemcpyHostToDevice, C->copy_stream);
    };
    std::vector<int> held;  // entries fetched but not yet behind a recorded event
    int cur_part = 0;
    auto fail_from = [&](size_t k, moe_status code, const char* why) {
        // the copies not known good: from k on, or all of them while the
        // first part of a split copy is still being issued (none has its down bytes)
        for (size_t j = split && cur_part == 0 ? 0 : k; j < copies.size(); ++j)
            if (r.miss_slots[copies[j].i] >= 0) L->cache.evict(r.miss_slots[copies[j].i]);
        pin_until_copied(L, held);  // the copies already issued may still read them
        return set_error(code, "copy of expert %d (slot %d) failed: %s", r.miss_experts[copies[k].i],
                         r.miss_slots[copies[k].i], why);
    };
    for (int part = 0; part < parts; ++part) {
        cur_part = part;
        const size_t off = part == 0 ? 0 : gu_bytes;
        const size_t len = !split ? L->ebytes : part == 0 ? gu_bytes : L->ebytes - gu_bytes;
        for (size_t k = 0; k < copies.size(); ++k) {
            const int e = r.miss_experts[copies[k].i];
            bool injected = false;
            if (part == 0) {
                for (;;) {  // the expert's bytes in the tier
                    st = store_acquire(L->store, e, &copies[k].src);
                    if (st != MOE_EBUSY || L->store_pins.empty()) break;
                    // every entry is pinned by copies still in flight: wait for the oldest
                    st = release_store_pins(L, false);
                    if (st == MOE_OK && !L->store_pins.empty()) {
                        const cudaError_t we = cudaEventSynchronize(L->store_pins.front().ev);
                        st = we == cudaSuccess ? release_store_pins(L, false)
                                               : set_error(MOE_ECUDA, "%s", cudaGetErrorString(we));
                    }
                    if (st != MOE_OK) break;
                }
                if (st != MOE_OK) {
                    const std::string why = moe_last_error();
                    return fail_from(k, MOE_ECOPY, why.c_str());
                }
                held.push_back(e);
                if (C->fail_copy_at >= 0 && C->copies_issued == C->fail_copy_at) {
                    injected = true;
                    C->fail_copy_at = -1;
                }
                C->copies_issued += 1;
            }
            const cudaError_t ce = injected ? cudaErrorUnknown
                                            : cudaMemcpyAsync(copies[k].dst + off, copies[k].src + off, len,
                                                              cudaMemcpyHostToDevice, C->copy_stream);
            if (ce != cudaSuccess) {
                if (!injected) cudaGetLastError();
                return fail_from(k, MOE_ECOPY, injected ? "injected failure" : cudaGetErrorString(ce));
            }
            if (part == parts - 1) {
                st = pin_until_copied(L, {e});
                if (st != MOE_OK) return st;
                held.erase(std::find(held.begin(), held.end(), e));
            }
            if (flags) {
                const int g = (int)(k / kFlagGroup);
                (*ready_of_miss)[copies[k].i] = MissFlags{2 * g, split ? 2 * g + 1 : 2 * g};
                if (k + 1 == copies.size() || (k + 1) % kFlagGroup == 0) {
                    const cudaError_t fe = set_flag(2 * g + part);
                    if (fe != cudaSuccess) {
                        cudaGetLastError();
                        return fail_from(k, MOE_ECOPY, cudaGetErrorString(fe));
                    }
                }
            }
        }
    }
    L->stats.bytes_h2d += (uint64_t)copies.size() * L->ebytes;
    return MOE_OK;
}

moe_status issue_miss_copies(moe_layer* L, const StepResult& r, bool with_bypass, uint32_t epoch,
                             std::vector<MissFlags>* ready_of_miss, bool split = false) {
    if (L->store) return issue_store_copies(L, r, with_bypass, epoch, ready_of_miss, split);
    moe_ctx* C = L->ctx;
    L->h_epochs[epoch % kEpochRing] = epoch;
    if (with_bypass && r.bypass > 0) {
        moe_status st = ensure_staging(C, (size_t)r.bypass * L->ebytes);
        if (st != MOE_OK) return st;
        CUDA_TRY(cudaStreamWaitEvent(C->copy_stream, C->staging_free, 0));
    }
    if (ready_of_miss) ready_of_miss->assign(r.miss_experts.size(), MissFlags{});
    // the copies to make, in miss order
    struct Copy {
        size_t i;
        uint8_t* dst;
        const uint8_t* src;
    };
    std::vector<Copy> copies;
    int nb = 0;
    for (size_t i = 0; i < r.miss_experts.size(); ++i) {
        const int slot = r.miss_slots[i];
        if (slot < 0 && !with_bypass) continue;
        uint8_t* dst = slot >= 0 ? L->d_slots + (size_t)slot * L->ebytes : C->staging + (size_t)(nb++) * L->ebytes;
        if (L->spare_call && r.miss_experts[i] == L->spare_expert) {
            // prefetched: no copy over the host link; the call's kernels read
            // the spare buffer, and the compute stream then copies it into the
            // slot (run_experts)
            if (slot < 0) --nb;  // it takes no staging entry
            L->spare_miss_expert = r.miss_experts[i];
            L->spare_miss_slot = slot;
            L->spare_expert = -1;
            ++L->prefetch_used;
            continue;
        }
        copies.push_back(Copy{i, dst, L->h_pool + (size_t)r.miss_experts[i] * L->ebytes});
    }
    const bool flags = ready_of_miss != nullptr;
    const size_t gu_bytes = 2 * qmat_bytes(L->sh.d_ff, L->sh.d_model);
    // a flag is set by a 4-byte copy queued behind the data on the same
    // stream: on this stream it costs ~1.5 us, a stream write of the value
    // ~3.3 us (measured)
    auto set_flag = [&](int flag) {
        return cudaMemcpyAsync(L->d_ready + flag, L->h_epochs + epoch % kEpochRing, sizeof(uint32_t),
                               cudaMemcpyHostToDevice, C->copy_stream);
    };
    int cur_part = 0;
    auto fail_from = [&](size_t k, cudaError_t ce, bool injected) {
        if (!injected) cudaGetLastError();
        // the copies not known good: from k on, or all of them while the first
        // part of a split copy is still being issued (none has its down bytes)
        const size_t first = split && flags && cur_part == 0 ? 0 : copies[k].i;
        for (size_t j = first; j < r.miss_experts.size(); ++j)
            if (r.miss_slots[j] >= 0) L->cache.evict(r.miss_slots[j]);
        return set_error(MOE_ECOPY, "copy of expert %d (slot %d) failed: %s", r.miss_experts[copies[k].i],
                         r.miss_slots[copies[k].i], injected ? "injected failure" : cudaGetErrorString(ce));
    };
    split = split && flags;
    const int parts = split ? 2 : 1;
    // Whole-expert copies of consecutive experts into consecutive places (the
    // staging arena's bypass entries, or a fresh cache's slots) go as one copy,
    // within a flag group: fewer, larger copies keep the copy engine fed at the
    // link's rate rather than at the host's issue rate. Not with an injected
    // failure armed, which names one expert's copy.
    const bool merge = !split && C->fail_copy_at < 0;
    for (int part = 0; part < parts; ++part) {
        cur_part = part;
        const size_t off = part == 0 ? 0 : gu_bytes;
        const size_t len = !split ? L->ebytes : part == 0 ? gu_bytes : L->ebytes - gu_bytes;
        for (size_t k = 0; k < copies.size();) {
            size_t e = k + 1;  // the run [k, e)
            while (merge && e < copies.size() && e % kFlagGroup != 0 &&
                   copies[e].dst == copies[e - 1].dst + L->ebytes && copies[e].src == copies[e - 1].src + L->ebytes)
                ++e;
            bool injected = false;
            if (part == 0) {
                if (C->fail_copy_at >= 0 && C->copies_issued == C->fail_copy_at) {
                    injected = true;
                    C->fail_copy_at = -1;
                }
                C->copies_issued += (long)(e - k);
            }
            const size_t bytes = (e - k - 1) * L->ebytes + len;
            const cudaError_t ce = injected ? cudaErrorUnknown
                                            : cudaMemcpyAsync(copies[k].dst + off, copies[k].src + off, bytes,
                                                              cudaMemcpyHostToDevice, C->copy_stream);

            if (ce != cudaSuccess) return fail_from(k, ce, injected);
            if (flags) {
                const int g = (int)(k / kFlagGroup);
                for (size_t j = k; j < e; ++j) (*ready_of_miss)[copies[j].i] = MissFlags{2 * g, split ? 2 * g + 1 : 2 * g};
                if (e == copies.size() || e % kFlagGroup == 0) {
                    const cudaError_t fe = set_flag(2 * g + part);
                    if (fe != cudaSuccess) return fail_from(k, fe, false);
                }
            }
            k = e;
        }
    }
    L->stats.bytes_h2d += (uint64_t)copies.size() * L->ebytes;
    return MOE_OK;
}

struct Item {
    const uint8_t* w;
    int b, e;              // pair range in perm, or pair ids themselves when perm is null
    const int32_t* perm;
    int ready, ready_dn;   // ready-flag indices of the gate/up and down bytes, -1 if resident
    int fam;               // 0 shared expert, 1 routed expert
};

template <class List>
bool add_item(List& l, const Item& x) {
    constexpr int MAXI = sizeof(l.item) / sizeof(l.item[0]);
    constexpr int MAXP = sizeof(l.pair) / sizeof(l.pair[0]);
    if (l.n_items >= MAXI) return false;
    int pb = l.n_items ? l.item[l.n_items - 1].pb + l.item[l.n_items - 1].np : 0;
    if (pb + (x.e - x.b) > MAXP) return false;
    FfnItem& it = l.item[l.n_items++];
    it.w = x.w;
    it.pb = (int16_t)pb;
    it.np = (int16_t)(x.e - x.b);
    it.ready = (int16_t)x.ready;
    it.ready_dn = (int16_t)x.ready_dn;
    for (int i = x.b; i < x.e; ++i) l.pair[pb++] = x.perm ? (int16_t)x.perm[i] : (int16_t)i;
    return true;
}

// Fused FFN launches covering `items` (family 0 first), each adding its
// experts' gate-weighted outputs into y; timed as `kind` when profiling.
template <class List>
moe_status launch_items(moe_layer* L, const std::vector<Item>& items, FfnArgs a, int kind, cudaStream_t s) {
    const moe_shapes& sh = L->sh;
    size_t i = 0;
    while (i < items.size()) {
        List l{};
        l.epoch = L->epoch;
        size_t j = i;
        int n_fam[2] = {0, 0};
        double bytes = 0, flops = 0;
        while (j < items.size() && add_item(l, items[j])) {
            ++n_fam[items[j].fam];
            bytes += items[j].fam == 0 ? (double)L->shared_bytes : (double)L->ebytes;
            flops += 6.0 * (items[j].e - items[j].b) * sh.d_model * (items[j].fam == 0 ? sh.d_ff_shared : sh.d_ff);
            ++j;
        }
        if (j == i) return set_error(MOE_EINVAL, "an expert with too many pairs for one work list");
        a.fam[0].n_items = n_fam[0];
        a.fam[1].n_items = n_fam[1];
        a.span = L->ctx->trace_span(kind, L->id, L->seq);
        if constexpr (std::is_same<List, FfnSmall>::value) {
            if (L->record_resident && i == 0 && j == items.size()) {
                L->resident_args = a;
                L->resident_args.span = nullptr;
                L->resident_list = l;
                L->have_resident = true;
            }
        }
        {
            Prof p(L->ctx, s, kind, bytes, flops);
            CUDA_TRY(launch_ffn(a, l, s, true));
        }
        L->stats.bytes_resident += (uint64_t)bytes;
        i = j;
    }
    return MOE_OK;
}

moe_status launch_items_any(moe_layer* L, const std::vector<Item>& items, const FfnArgs& a, int kind,
                            cudaStream_t s) {
    if (items.empty()) return MOE_OK;
    int pairs = 0;
    for (const Item& it : items) pairs += it.e - it.b;
    if ((int)items.size() <= 24 && pairs <= 96) return launch_items<FfnSmall>(L, items, a, kind, s);
    return launch_items<FfnLarge>(L, items, a, kind, s);
}

FfnArgs decode_args(moe_layer* L, const uint16_t* x, float* y) {
    const moe_shapes& sh = L->sh;
    FfnArgs a{};
    a.x = x;
    a.d = sh.d_model;
    a.act = sh.act;
    a.fam[0] = FfnFam{0, sh.d_ff_shared, 1};
    a.fam[1] = FfnFam{0, sh.d_ff, sh.top_k};
    a.gates = L->d_gates;
    a.y = y;  // zeroed by the router launch of this call
    a.ready = L->d_ready;
    a.err = L->ctx->err_dev;
    a.trace = nullptr;
    if (L->deterministic && L->d_dpart) {
        // partial rows: the shared expert's by token, then the routed by pair
        const int cs = sh.d_ff_shared / 32, cr = sh.d_ff / 32;
        const size_t cap = L->dpart_floats / ((size_t)(cs + sh.top_k * cr) * sh.d_model);
        a.part[0] = L->d_dpart;
        a.part[1] = L->d_dpart + cap * cs * sh.d_model;
        a.part_c[0] = cs;
        a.part_c[1] = cr;
    }
    return a;
}

// The ordered combine of a decode call: y = shared + ranks 0..k-1, from the
// partial rows the call's FFN launches wrote.
moe_status reduce_parts(moe_layer* L, int T, float* y, cudaStream_t s) {
    const moe_shapes& sh = L->sh;
    const FfnArgs a = decode_args(L, nullptr, y);
    Prof p(L->ctx, s, K_COMBINE, 4.0 * (double)det_part_floats(sh, T) + 4.0 * T * sh.d_model,
           (double)det_part_floats(sh, T));
    CUDA_TRY(launch_part_reduce(a.part[0], a.part[1], a.part_c[0], a.part_c[1], sh.top_k, sh.d_model, T, y, s, true));
    return MOE_OK;
}

// The shared expert of a decode call on every token. It needs no routing, so
// it is queued right behind the router and runs while the host reads the
// routing, steps the cache and issues the miss copies ([P1] §8.2: the copies
// overlap the shared expert's compute).
moe_status run_shared(moe_layer* L, const uint16_t* x, int T, float* y, cudaStream_t s) {
    std::vector<Item> items;
    for (int t0 = 0; t0 < T; t0 += kFfnMaxNT)
        items.push_back(Item{L->d_shared, t0, std::min(T, t0 + kFfnMaxNT), nullptr, -1, -1, 0});
    FfnArgs a = decode_args(L, x, y);
    if (L->deterministic && T > 1) a.min_nt = 2;
    return launch_items_any(L, items, a, K_FFN, s);
}

// `zero_y`, when given, is the call's [T][d] fp32 output, zeroed by the same launch.
moe_status route_into(moe_layer* L, const uint16_t* x, int T, const float* zbias, int32_t* ids, float* gates,
                      bool publish, cudaStream_t s, float* zero_y = nullptr) {
    RouterParams p{x, T, L->sh.d_model, L->sh.n_experts, L->sh.top_k, L->d_router_codes, L->d_router_sb, zbias,
                   L->d_logits, L->d_rcount, ids, gates, publish ? L->h_pub_dev : nullptr, L->seq,
                   zero_y, zero_y ? T * L->sh.d_model : 0, L->ctx->trace_span(K_ROUTER, L->id, L->seq)};
    Prof pr(L->ctx, s, K_ROUTER, (double)L->router_bytes + 2.0 * T * L->sh.d_model,
            2.0 * T * L->sh.n_experts * L->sh.d_model);
    CUDA_TRY(launch_router(p, s, true));
    L->stats.bytes_resident += L->router_bytes;
    return MOE_OK;
}

// A one-token decode call's resident work in one launch queued right behind
// the router, before the host has read the routing: the shared expert, and
// each routed pair whose expert the device slot table shows resident (the
// kernel looks the experts up itself once the router has finished). Misses
// are skipped there and launched after the cache step. *prof_index is the
// launch's timing record (profiling), whose bytes the caller corrects once
// the misses are known.
moe_status run_resident_on_device(moe_layer* L, const uint16_t* x, float* y, cudaStream_t s, long* prof_index) {
    std::vector<Item> items;
    items.push_back(Item{L->d_shared, 0, 1, nullptr, -1, -1, 0});
    for (int p = 0; p < L->sh.top_k; ++p) items.push_back(Item{nullptr, p, p + 1, nullptr, -1, -1, 1});
    FfnArgs a = decode_args(L, x, y);
    a.ids = L->d_ids;
    a.slot_of = L->d_slot_of;
    a.slots = L->d_slots;
    a.ebytes = L->ebytes;
    *prof_index = L->ctx->profiling ? (long)L->ctx->prof.size() : -1;
    L->record_resident = true;
    const moe_status st = launch_items_any(L, items, a, K_FFN, s);
    L->record_resident = false;
    return st;
}

// The routed experts of a decode call, added into y (which already holds the
// shared expert's output): one launch over the hits, whose weights are
// resident, then one over the misses in miss order, whose producers wait for
// each expert's ready flag.
// The slot-table changes of the last cache step (removals first), from the
// table before the step and the cache after it.
void table_changes(const moe_layer* L, std::vector<std::pair<int, int>>& out) {
    out.clear();
    for (int sl = 0; sl < L->S; ++sl)
        if (L->slot_before[sl] != L->cache.slot_expert[sl] && L->slot_before[sl] >= 0)
            out.push_back({L->slot_before[sl], -1});
    for (int sl = 0; sl < L->S; ++sl)
        if (L->slot_before[sl] != L->cache.slot_expert[sl] && L->cache.slot_expert[sl] >= 0)
            out.push_back({L->cache.slot_expert[sl], sl});
}

// The whole device slot table, from the cache, ordered on `s` (the source
// is staged by the copy call, so it may change as soon as the call returns).
moe_status table_upload(moe_layer* L, cudaStream_t s) {
    std::vector<int32_t> t(L->sh.n_experts, -1);
    for (int sl = 0; sl < L->S; ++sl)
        if (L->cache.slot_expert[sl] >= 0) t[L->cache.slot_expert[sl]] = sl;
    CUDA_TRY(cudaMemcpyAsync(L->d_slot_of, t.data(), t.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s));
    return MOE_OK;
}

// The same outside any call: after the layer's earlier work, synchronously.
moe_status table_upload_sync(moe_layer* L) {
    if (L->ev_done) CUDA_TRY(cudaEventSynchronize(L->ev_done));
    moe_status st = table_upload(L, L->ctx->copy_stream);
    if (st != MOE_OK) return st;
    CUDA_TRY(cudaStreamSynchronize(L->ctx->copy_stream));
    return MOE_OK;
}

// device_hits: the hits were already launched before the cache step, resolved
// on the device (see launch_routed_on_device); launch the misses only, which
// also carry the step's slot-table changes.
moe_status run_experts(moe_layer* L, const uint16_t* x, int T, float* y, const std::vector<MissFlags>& ready_of_miss,
                       cudaEvent_t copies_done, cudaStream_t s, bool device_hits = false) {
    moe_ctx* C = L->ctx;
    const moe_shapes& sh = L->sh;
    const int npairs = T * sh.top_k;
    L->offsets.resize(sh.n_experts + 1);
    L->perm.resize(npairs);
    group_pairs(L->h_ids.data(), npairs, sh.n_experts, L->offsets.data(), L->perm.data());
    std::vector<Item> items, miss;
    int nb = 0;
    size_t mi = 0;
    for (int e : L->step.distinct) {
        while (mi < L->step.miss_experts.size() && L->step.miss_experts[mi] < e) ++mi;
        const bool is_miss = mi < L->step.miss_experts.size() && L->step.miss_experts[mi] == e;
        const int slot = is_miss ? L->step.miss_slots[mi] : L->cache.slot_of(e);
        const uint8_t* w;
        if (is_miss && e == L->spare_miss_expert) {
            w = L->d_spare;  // prefetched into HBM
        } else if (slot >= 0) {
            w = L->d_slots + (size_t)slot * L->ebytes;
        } else {
            w = C->staging + (size_t)nb * L->ebytes;
            ++nb;
        }
        const MissFlags f = is_miss ? ready_of_miss[mi] : MissFlags{};
        for (int b = L->offsets[e]; b < L->offsets[e + 1]; b += kFfnMaxNT)
            (is_miss ? miss : items)
                .push_back(Item{w, b, std::min(b + kFfnMaxNT, (int)L->offsets[e + 1]), L->perm.data(), f.gu, f.dn, 1});
    }
    FfnArgs a = decode_args(L, x, y);
    if (L->deterministic && T > 1) a.min_nt = 2;  // one kernel shape for every launch of the call
    moe_status st = device_hits ? MOE_OK : launch_items_any(L, items, a, K_FFN, s);
    if (st != MOE_OK) return st;
    std::vector<std::pair<int, int>> upd;
    table_changes(L, upd);
    if (!upd.empty()) {
        if (miss.empty() || (int)upd.size() > kFfnMaxUpd) {
            st = table_upload(L, s);
            if (st != MOE_OK) return st;
        } else {
            a.slot_of = L->d_slot_of;
            a.n_upd = (int)upd.size();
            for (size_t i = 0; i < upd.size(); ++i) {
                a.upd_expert[i] = (int16_t)upd[i].first;
                a.upd_slot[i] = (int16_t)upd[i].second;
            }
        }
    }
    // exposed copy time: from the end of the resident work to the last copy
    WaitRec w{};
    if (copies_done) {
        w.ffn_start = C->timing_event();
        w.copies_done = copies_done;
        CUDA_TRY(cudaEventRecord(w.ffn_start, s));
    }
    // a miss served from the spare buffer: its kernels wait for the prefetch
    // copy (an event, not a flag: no kernel spins on it)
    if (L->spare_miss_expert >= 0) CUDA_TRY(cudaStreamWaitEvent(s, L->ev_spare_ready, 0));
    st = launch_items_any(L, miss, a, K_FFN_MISS, s);
    if (copies_done) L->waits.push_back(w);
    if (st == MOE_OK && L->spare_miss_expert >= 0) {
        // then the spare's bytes go into the expert's slot, on this stream,
        // after the kernels that read the spare; the next prefetch into the
        // spare waits for this copy
        if (L->spare_miss_slot >= 0)
            CUDA_TRY(cudaMemcpyAsync(L->d_slots + (size_t)L->spare_miss_slot * L->ebytes, L->d_spare, L->ebytes,
                                     cudaMemcpyDeviceToDevice, s));
        CUDA_TRY(cudaEventRecord(L->ev_spare_free, s));
        L->spare_free_recorded = true;
    }
    L->spare_miss_expert = -1;
    L->spare_miss_slot = -1;
    return st;
}

// The experts of a prefill call (T > kDecodeMaxT: a 128-token chunk, or a
// whole prompt run layer-major) as grouped GEMMs on the tensor cores. An item
// is up to kPfMaxN token rows of one expert: the shared expert over each block
// of kPfMaxN tokens, each routed expert over its pairs (sorted by expert) in
// pieces of at most kPfMaxN. Then gate/up, down into y (shared) and o
// (routed), and the combine y += sum_r g_r o_r. Hits come before misses in
// the job order, so the resident experts run while the copies land.
moe_status run_experts_prefill(moe_layer* L, const uint16_t* x, int T, float* y,
                               const std::vector<MissFlags>& ready_of_miss, cudaEvent_t copies_done, cudaStream_t s) {
    moe_ctx* C = L->ctx;
    const moe_shapes& sh = L->sh;
    const int k = sh.top_k, d = sh.d_model, P = T * k;
    if (T > L->cap_T || !L->d_pf) return set_error(MOE_EINVAL, "prefill call of %d tokens (scratch for %d)", T, L->cap_T);
    L->offsets.resize(sh.n_experts + 1);
    L->perm.resize(P);
    group_pairs(L->h_ids.data(), P, sh.n_experts, L->offsets.data(), L->perm.data());
    PfItem* items = reinterpret_cast<PfItem*>(L->h_pf);
    const size_t max_items = pf_max_items(sh, T);
    int n = 0;
    const int n_shared = (T + kPfMaxN - 1) / kPfMaxN;
    for (int t0 = 0; t0 < T; t0 += kPfMaxN) items[n++] = PfItem{L->d_shared, t0, std::min(kPfMaxN, T - t0), -1, -1};
    std::vector<PfItem> miss;
    int nb = 0;
    size_t mi = 0;
    double bytes = (double)L->shared_bytes * n_shared;  // the shared weights, read once per token block
    for (int e : L->step.distinct) {
        while (mi < L->step.miss_experts.size() && L->step.miss_experts[mi] < e) ++mi;
        const bool is_miss = mi < L->step.miss_experts.size() && L->step.miss_experts[mi] == e;
        const int slot = is_miss ? L->step.miss_slots[mi] : L->cache.slot_of(e);
        const uint8_t* w = slot >= 0 ? L->d_slots + (size_t)slot * L->ebytes : C->staging + (size_t)(nb++) * L->ebytes;
        const MissFlags f = is_miss ? ready_of_miss[mi] : MissFlags{};
        for (int p0 = L->offsets[e]; p0 < L->offsets[e + 1]; p0 += kPfMaxN) {
            const PfItem it{w, p0, std::min(kPfMaxN, L->offsets[e + 1] - p0), f.gu, f.dn};
            if ((size_t)n + miss.size() >= max_items) return set_error(MOE_ESTATE, "prefill item list overflow");
            if (is_miss)
                miss.push_back(it);
            else
                items[n++] = it;
            bytes += (double)L->ebytes;  // each piece reads the expert's weights
        }
    }
    for (const PfItem& it : miss) items[n++] = it;
    const size_t item_bytes = sizeof(PfItem) * max_items;
    int32_t* pair_h = reinterpret_cast<int32_t*>(L->h_pf + item_bytes);
    std::copy(L->perm.begin(), L->perm.end(), pair_h);
    CUDA_TRY(cudaMemcpyAsync(L->d_pf, L->h_pf, L->pf_bytes, cudaMemcpyHostToDevice, s));

    PfArgs a{};
    a.items = reinterpret_cast<const PfItem*>(L->d_pf);
    a.n_items = n;
    a.n_fam0 = n_shared;
    a.d = d;
    a.act = sh.act;
    a.T = T;
    a.k = k;
    a.inter[0] = sh.d_ff_shared;
    a.inter[1] = sh.d_ff;
    a.pair = reinterpret_cast<const int32_t*>(L->d_pf + item_bytes);
    __half* xs = L->d_x16;
    __half* xg = xs + (size_t)T * d;
    a.h[0] = L->d_h16;
    a.h[1] = L->d_h16 + (size_t)T * sh.d_ff_shared;
    a.out[0] = y;
    a.out[1] = L->d_o;
    a.ready = L->d_ready;
    a.epoch = L->epoch;
    a.err = C->err_dev;
    a.part = L->d_part;
    a.part_cap = L->d_part ? L->part_floats : 0;
    const int rows[2] = {T, P};
    WaitRec wr{};
    if (copies_done) {
        wr.ffn_start = C->timing_event();
        wr.copies_done = copies_done;
        CUDA_TRY(cudaEventRecord(wr.ffn_start, s));
    }
    {
        Prof p(C, s, K_GATHER, 2.0 * (T + P) * d * 2, 0);
        CUDA_TRY(launch_pf_gather(x, T, d, a.pair, P, k, xs, xg, s));
    }
    const double rows_shared = T, rows_routed = P;
    const double fl_gu = 4.0 * d * (rows_shared * sh.d_ff_shared + rows_routed * sh.d_ff);
    const double fl_dn = 2.0 * d * (rows_shared * sh.d_ff_shared + rows_routed * sh.d_ff);
    const double by_gu = (double)L->shared_bytes * 2 / 3 + (bytes - L->shared_bytes) * 2 / 3;
    const double by_dn = bytes - by_gu;
    {
        Prof p(C, s, K_GEMM_GU, by_gu, fl_gu);
        int n_launch = 1;
        CUDA_TRY(launch_pf_gemm(a, 1, xs, xg, rows, s, &n_launch));
        C->launches += n_launch - 1;  // the K-split epilogue launch
    }
    {
        Prof p(C, s, K_GEMM_DN, by_dn, fl_dn);
        int n_launch = 1;
        CUDA_TRY(launch_pf_gemm(a, 2, a.h[0], a.h[1], rows, s, &n_launch));
        C->launches += n_launch - 1;  // the K-split epilogue launch
    }
    {
        Prof p(C, s, K_COMBINE, 4.0 * ((double)P * d + 2.0 * T * d), 2.0 * P * d);
        CUDA_TRY(launch_combine(L->d_o, L->d_gates, T, k, d, y, s));
    }
    L->stats.bytes_resident += (uint64_t)bytes;
    if (copies_done) L->waits.push_back(wr);
    return MOE_OK;
}

// Wait on the host until the router of the current call has published all
// n ids (each word carries the call number in its high half).
moe_status wait_published(moe_layer* L, int n) {
    volatile unsigned long long* pub = L->h_pub;
    const auto t0 = std::chrono::steady_clock::now();
    int done = 0;
    for (uint32_t i = 0;; ++i) {
        while (done < n) {
            const unsigned long long v = pub[done];
            if ((uint32_t)(v >> 32) != L->seq) break;
            L->h_ids[done] = (int32_t)(uint32_t)v;
            ++done;
        }
        if (done == n) return MOE_OK;
        if ((i & 1023) == 1023) {
            const double el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
            if (el > kHostWaitLimitS) return set_error(MOE_ETIMEOUT, "routing was not published within %.0f s", el);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return set_error(MOE_ECUDA, "while waiting for routing: %s", cudaGetErrorString(e));
        }
    }
}

double us_since(std::chrono::steady_clock::time_point t) {
    return std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t).count();
}

// One call: at most kPrefillChunk tokens from moe_forward, or a whole
// layer-major prompt from moe_forward_prompt.
// The prefetch of a decode call, queued on the copy stream after the call's
// kernels were enqueued: the expert routed in the most steps so far (ties to the lower id)
// that is neither in a slot nor already in the spare buffer goes into the
// spare buffer ([P1] §9.2 item 3, §9.5 item 2: predict the next experts from
// routing history and read them ahead). The cache trace does not change: a
// later miss of that expert is still a miss, copied from the spare buffer.
moe_status issue_prefetch(moe_layer* L) {
    int best = -1;
    uint32_t best_n = 0;
    for (int e = 0; e < L->sh.n_experts; ++e) {
        const uint32_t n = L->route_hist[(size_t)e];
        if (n > best_n && L->cache.slot_of(e) < 0) {
            best = e;
            best_n = n;
        }
    }
    if (best < 0 || best == L->spare_expert) return MOE_OK;
    // the spare buffer may still be read by earlier kernels or copied into a slot
    if (L->spare_free_recorded) CUDA_TRY(cudaStreamWaitEvent(L->ctx->copy_stream, L->ev_spare_free, 0));
    CUDA_TRY(cudaMemcpyAsync(L->d_spare, L->h_pool + (size_t)best * L->ebytes, L->ebytes, cudaMemcpyHostToDevice,
                             L->ctx->copy_stream));
    CUDA_TRY(cudaEventRecord(L->ev_spare_ready, L->ctx->copy_stream));
    L->spare_expert = best;
    ++L->prefetch_issued;
    L->stats.bytes_h2d += L->ebytes;
    return MOE_OK;
}

moe_status forward_chunk(moe_layer* L, const uint16_t* x, int T, const float* zbias, float* y, int32_t* ids_out,
                         float* gates_out, cudaStream_t s) {
    moe_ctx* C = L->ctx;
    const moe_shapes& sh = L->sh;
    const int npairs = T * sh.top_k;
    auto t0 = std::chrono::steady_clock::now();
    C->trace_mark("call", L->id, L->seq + 1);
    // the layer's previous call and any copies moe_cache_step issued come first;
    // a call on the stream that recorded ev_done is already ordered after it
    if (!L->have_last_stream || L->last_stream != s) CUDA_TRY(cudaStreamWaitEvent(s, L->ev_done, 0));
    if (L->pending) {
        CUDA_TRY(cudaStreamWaitEvent(s, L->ev_pending, 0));
        L->pending = false;
    }
    if (L->err_generation != C->err_generation) {
        // an earlier kernel abandoned a wait: restore the all-zero counters
        CUDA_TRY(cudaMemsetAsync(L->d_rcount, 0, sizeof(unsigned) * ((L->cap_T + 7) / 8), s));
        L->err_generation = C->err_generation;
    }
    ++L->seq;
    // a decode call's experts add into y, which the router launch zeroes
    const bool decode = T <= kDecodeMaxT;
    if (decode && L->deterministic) {
        moe_status st = ensure_det_scratch(L, std::max(T, L->cap_T));
        if (st != MOE_OK) return st;
    }
    // one token: the hits are found on the device (the work list holds the
    // shared item and the k pairs)
    const bool device_routed = T == 1 && 1 + sh.top_k <= (int)(sizeof(FfnSmall::item) / sizeof(FfnItem));
    moe_status st = route_into(L, x, T, zbias, L->d_ids, L->d_gates, true, s, decode ? y : nullptr);
    if (st != MOE_OK) return st;
    long r_prof = -1;
    if (device_routed) {
        st = run_resident_on_device(L, x, y, s, &r_prof);
        if (st != MOE_OK) return st;
    } else if (decode) {
        st = run_shared(L, x, T, y, s);
        if (st != MOE_OK) return st;
    }
    L->stats.host_issue_us += us_since(t0);
    t0 = std::chrono::steady_clock::now();
    st = wait_published(L, npairs);
    L->stats.host_wait_us += us_since(t0);
    C->trace_mark("ids", L->id, L->seq);
    if (st != MOE_OK) return st;
    t0 = std::chrono::steady_clock::now();
    st = check_err_word(C);
    if (st != MOE_OK) return st;
    L->slot_before = L->cache.slot_expert;
    if (!L->cache.step(L->h_ids.data(), npairs, L->step))
        return set_error(MOE_ESTATE, "router produced an invalid id");
    if (L->store || L->prefetch)
        for (int e : L->step.distinct) ++L->route_hist[(size_t)e];
    if (device_routed) {
        // the resident launch counted every routed pair as a hit
        const size_t n_miss = L->step.miss_experts.size();
        const double mb = (double)n_miss * L->ebytes;
        L->stats.bytes_resident -= (uint64_t)mb;
        if (r_prof >= 0 && r_prof < (long)C->prof.size()) {
            C->prof[r_prof].bytes -= mb;
            C->prof[r_prof].flops -= 6.0 * n_miss * sh.d_model * sh.d_ff;
        }
    }
    L->stats.steps += 1;
    L->stats.hits += L->step.hits;
    L->stats.misses += L->step.miss_experts.size();
    L->stats.bypass += L->step.bypass;
    const uint32_t epoch = ++L->epoch;
    std::vector<MissFlags> ready_of_miss;
    L->spare_call = L->prefetch && T <= kDecodeMaxT;
    st = issue_miss_copies(L, L->step, true, epoch, &ready_of_miss, L->step.miss_experts.size() <= kFlagGroup);
    L->spare_call = false;
    C->trace_mark("copies", L->id, L->seq);
    if (st != MOE_OK) {
        table_upload(L, s);  // the failed slots were emptied: the device table follows
        return st;
    }
    cudaEvent_t copies_done = nullptr;
    if (!L->step.miss_experts.empty() && C->profiling) {  // exposed copy time: profiling only
        copies_done = C->timing_event();
        CUDA_TRY(cudaEventRecord(copies_done, C->copy_stream));
    }
    if (T > kDecodeMaxT) {
        st = run_experts_prefill(L, x, T, y, ready_of_miss, copies_done, s);
        if (st == MOE_OK && L->slot_before != L->cache.slot_expert) st = table_upload(L, s);
    } else {
        st = run_experts(L, x, T, y, ready_of_miss, copies_done, s, device_routed);
        if (st == MOE_OK && L->deterministic) st = reduce_parts(L, T, y, s);
        if (st == MOE_OK && L->prefetch) st = issue_prefetch(L);
    }
    if (st != MOE_OK) return st;
    if (ids_out) CUDA_TRY(cudaMemcpyAsync(ids_out, L->d_ids, sizeof(int32_t) * npairs, cudaMemcpyDeviceToDevice, s));
    if (gates_out)
        CUDA_TRY(cudaMemcpyAsync(gates_out, L->d_gates, sizeof(float) * npairs, cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaEventRecord(L->ev_done, s));
    L->last_stream = s;
    L->have_last_stream = true;
    if (L->step.bypass > 0) CUDA_TRY(cudaEventRecord(C->staging_free, s));
    L->stats.host_issue_us += us_since(t0);
    C->trace_mark("end", L->id, L->seq);
    return MOE_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI

extern "C" const char* moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_EINVAL: return "MOE_EINVAL";
        case MOE_ENOMEM: return "MOE_ENOMEM";
        case MOE_ECUDA: return "MOE_ECUDA";
        case MOE_ECOPY: return "MOE_ECOPY";
        case MOE_ETIMEOUT: return "MOE_ETIMEOUT";
        case MOE_ESTATE: return "MOE_ESTATE";
        case MOE_EBUSY: return "MOE_EBUSY";
        case MOE_EIO: return "MOE_EIO";
    }
    return "MOE_UNKNOWN";
}

extern "C" const char* moe_last_error(void) { return g_err; }

extern "C" moe_status moe_ctx_create(int device, moe_ctx** out) {
    if (!out) return set_error(MOE_EINVAL, "out is NULL");
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) {
        cudaGetLastError();
        return set_error(MOE_EINVAL, "no CUDA device %d (%d present)", device, n);
    }
    CUDA_TRY(cudaSetDevice(device));
    moe_ctx* C = new (std::nothrow) moe_ctx();
    if (!C) return set_error(MOE_ENOMEM, "out of host memory");
    C->device = device;
    if (cudaStreamCreateWithFlags(&C->copy_stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&C->staging_free, cudaEventDisableTiming) != cudaSuccess ||
        cudaHostAlloc(&C->err_host, sizeof(unsigned), cudaHostAllocMapped) != cudaSuccess ||
        cudaHostGetDevicePointer(&C->err_dev, C->err_host, 0) != cudaSuccess) {
        cudaGetLastError();
        delete C;
        return set_error(MOE_ECUDA, "stream/event creation failed");
    }
    *C->err_host = 0;
    if (const char* tp = getenv("MOE_TRACE_FILE")) {
        if (*tp && cudaMalloc(&C->trace_spans, sizeof(unsigned long long) * 2 * kTraceSpans) == cudaSuccess) {
            std::vector<unsigned long long> init(2 * kTraceSpans, 0ull);
            for (int i = 0; i < kTraceSpans; ++i) init[2 * i] = ~0ull;
            cudaMemcpy(C->trace_spans, init.data(), init.size() * sizeof(unsigned long long), cudaMemcpyHostToDevice);
            C->trace_path = tp;
        }
        cudaGetLastError();
    }
    *out = C;
    return MOE_OK;
}

namespace {

// Writes the timeline: a calibration line (host clock before and after a
// one-thread kernel that reads %globaltimer, and the value it read), then one
// line per launch and per host step.
void write_trace(moe_ctx* C) {
    cudaDeviceSynchronize();
    std::vector<unsigned long long> spans(2 * C->trace_launches.size());
    if (!spans.empty())
        cudaMemcpy(spans.data(), C->trace_spans, spans.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    unsigned long long* d = C->trace_spans;  // reuse slot 0's words for the calibration read
    const uint64_t h0 = realtime_ns();
    read_globaltimer<<<1, 1>>>(d);
    unsigned long long g = 0;
    cudaMemcpy(&g, d, sizeof(g), cudaMemcpyDeviceToHost);
    const uint64_t h1 = realtime_ns();
    FILE* f = fopen(C->trace_path.c_str(), "w");
    if (!f) return;
    fprintf(f, "cal %llu %llu %llu\n", (unsigned long long)h0, (unsigned long long)h1, g);
    for (const TraceLaunch& t : C->trace_launches)
        fprintf(f, "launch %d %d %u %llu %llu %llu\n", t.kind, t.layer, t.seq, (unsigned long long)t.t_host,
                spans[2 * t.slot], spans[2 * t.slot + 1]);
    for (const TraceHost& t : C->trace_host)
        fprintf(f, "host %s %d %u %llu\n", t.what, t.layer, t.seq, (unsigned long long)t.t);

    fclose(f);
    cudaGetLastError();
}

}  // namespace

extern "C" void moe_ctx_destroy(moe_ctx* C) {
    if (!C) return;
    cudaSetDevice(C->device);
    cudaStreamSynchronize(C->copy_stream);
    drain_prof(C);
    if (C->trace_spans) {
        write_trace(C);
        cudaFree(C->trace_spans);
    }
    for (cudaEvent_t e : C->timing_pool) cudaEventDestroy(e);
    cudaFree(C->staging);
    cudaFreeHost(C->err_host);
    cudaEventDestroy(C->staging_free);
    cudaStreamDestroy(C->copy_stream);
    delete C;
}

extern "C" size_t moe_expert_bytes(const moe_shapes* s) {
    if (!s) return 0;
    return expert_blob_bytes(s->d_model, s->d_ff);
}

extern "C" void moe_layer_destroy(moe_layer* L) {
    if (!L) return;
    cudaSetDevice(L->ctx->device);
    if (L->ev_done) cudaEventSynchronize(L->ev_done);
    cudaStreamSynchronize(L->ctx->copy_stream);
    drain_waits(L);
    free_scratch(L);
    cudaFree(L->d_dpart);
    cudaFree(L->d_spare);
    if (L->ev_spare_ready) cudaEventDestroy(L->ev_spare_ready);
    if (L->ev_spare_free) cudaEventDestroy(L->ev_spare_free);
    if (L->store) {
        release_store_pins(L, true);
        for (cudaEvent_t e : L->store_events) cudaEventDestroy(e);
        if (L->store_pinned) cudaHostUnregister(L->store_pinned);
        store_attach(L->store, false);
    }
    cudaFree(L->d_router_codes);
    cudaFree(L->d_router_sb);
    cudaFree(L->d_shared);
    cudaFree(L->d_slots);
    cudaFree(L->d_slot_of);
    cudaFree(L->d_ready);
    cudaFreeHost(L->h_pool);
    cudaFreeHost(L->h_epochs);
    if (L->ev_done) cudaEventDestroy(L->ev_done);
    if (L->ev_pending) cudaEventDestroy(L->ev_pending);
    delete L;
}

namespace {

// moe_layer_create, with the pinned pool of every routed expert (with_pool)
// or without it (a layer that streams from an expert store).
moe_status create_layer(moe_ctx* C, const moe_shapes* s, const moe_quant_layout* q, int32_t slots, int32_t policy,
                        bool with_pool, moe_layer** out) {
    if (!C || !out) return set_error(MOE_EINVAL, "ctx or out is NULL");
    moe_status st = check_shapes(s);
    if (st != MOE_OK) return st;
    if (!q || q->w_bits != 4 || q->w_group != 64 || q->r_bits != 8 || q->r_group != 64)
        return set_error(MOE_EINVAL, "only the {4, 64, 8, 64} quantisation layout is supported");
    if (slots < 1 || slots > s->n_experts) return set_error(MOE_EINVAL, "cache_slots %d out of [1, n_experts]", slots);
    if (policy != kLFU && policy != kLRU) return set_error(MOE_EINVAL, "policy %d must be 0 (LFU) or 1 (LRU)", policy);
    CUDA_TRY(cudaSetDevice(C->device));
    moe_layer* L = new (std::nothrow) moe_layer(s->n_experts, slots, policy);
    if (!L) return set_error(MOE_ENOMEM, "out of host memory");
    L->ctx = C;
    {
        static std::atomic<int> next_id{0};
        L->id = next_id++;
    }
    L->sh = *s;
    L->S = slots;
    L->policy = policy;
    L->ebytes = expert_blob_bytes(s->d_model, s->d_ff);
    L->shared_bytes = expert_blob_bytes(s->d_model, s->d_ff_shared);
    L->router_bytes = (size_t)s->n_experts * s->d_model + (size_t)s->n_experts * (s->d_model / 64) * 4;
    const size_t n_flags = (size_t)slots + s->n_experts;
    bool ok = cudaMalloc(&L->d_router_codes, (size_t)s->n_experts * s->d_model) == cudaSuccess &&
              cudaMalloc(&L->d_router_sb, (size_t)s->n_experts * (s->d_model / 64) * 4) == cudaSuccess &&
              cudaMalloc(&L->d_shared, L->shared_bytes) == cudaSuccess &&
              cudaMalloc(&L->d_slots, (size_t)slots * L->ebytes) == cudaSuccess &&
              cudaMalloc(&L->d_slot_of, (size_t)s->n_experts * sizeof(int32_t)) == cudaSuccess &&
              cudaMemset(L->d_slot_of, 0xFF, (size_t)s->n_experts * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&L->d_ready, n_flags * sizeof(uint32_t)) == cudaSuccess &&
              cudaMemset(L->d_ready, 0, n_flags * sizeof(uint32_t)) == cudaSuccess &&
              (!with_pool ||
               cudaHostAlloc(&L->h_pool, (size_t)s->n_experts * L->ebytes, cudaHostAllocDefault) == cudaSuccess) &&
              cudaHostAlloc(&L->h_epochs, kEpochRing * sizeof(uint32_t), cudaHostAllocDefault) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        moe_layer_destroy(L);
        return set_error(MOE_ENOMEM, "layer allocation failed (%zu B pinned pool, %zu B slots)",
                         with_pool ? (size_t)s->n_experts * L->ebytes : (size_t)0, (size_t)slots * L->ebytes);
    }
    ok = cudaEventCreateWithFlags(&L->ev_done, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&L->ev_pending, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        moe_layer_destroy(L);
        return set_error(MOE_ECUDA, "event creation failed");
    }
    *out = L;
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_layer_create(moe_ctx* C, const moe_shapes* s, const moe_quant_layout* q, int32_t slots,
                                       int32_t policy, moe_layer** out) {
    return create_layer(C, s, q, slots, policy, true, out);
}

extern "C" moe_status moe_layer_create_streamed(moe_ctx* C, const moe_shapes* s, const moe_quant_layout* q,
                                                int32_t slots, int32_t policy, moe_expert_store* store,
                                                moe_layer** out) {
    if (!store) return set_error(MOE_EINVAL, "store is NULL");
    moe_status st = check_shapes(s);
    if (st != MOE_OK) return st;
    if (memcmp(&store_shapes(store), s, sizeof(moe_shapes)) != 0)
        return set_error(MOE_EINVAL, "the store holds experts of other shapes");
    if (!store_attach(store, true)) return set_error(MOE_EINVAL, "the store already serves a layer");
    moe_layer* L = nullptr;
    st = create_layer(C, s, q, slots, policy, false, &L);
    if (st != MOE_OK) {
        store_attach(store, false);
        return st;
    }
    size_t bytes = 0;
    uint8_t* buf = store_buffer(store, &bytes);
    const cudaError_t e = cudaHostRegister(buf, bytes, cudaHostRegisterDefault);
    if (e != cudaSuccess) {
        cudaGetLastError();
        moe_layer_destroy(L);
        store_attach(store, false);
        return set_error(MOE_ECUDA, "page-locking the store's %zu B tier failed: %s", bytes, cudaGetErrorString(e));
    }
    L->store = store;
    L->store_pinned = buf;
    L->route_hist.assign((size_t)s->n_experts, 0);
    *out = L;
    return MOE_OK;
}

extern "C" moe_status moe_layer_prefetch(moe_layer* L, int32_t n, int32_t* queued) {
    if (queued) *queued = 0;
    if (!L || n < 0) return set_error(MOE_EINVAL, "moe_layer_prefetch: bad arguments");
    if (!L->store) return set_error(MOE_ESTATE, "moe_layer_prefetch: the layer does not stream from a store");
    if (n == 0) return MOE_OK;
    // entries whose copies have finished may take the reads
    moe_status st = release_store_pins(L, false);
    if (st != MOE_OK) return st;
    // experts by routing count, highest first, ties to the lower id
    std::vector<int32_t> order;
    for (int e = 0; e < L->sh.n_experts; ++e)
        if (L->route_hist[(size_t)e] > 0 && L->cache.slot_of(e) < 0 && !store_contains(L->store, e))
            order.push_back(e);
    const size_t take = std::min(order.size(), (size_t)n);
    std::partial_sort(order.begin(), order.begin() + (long)take, order.end(), [&](int32_t a, int32_t b) {
        const uint32_t ca = L->route_hist[(size_t)a], cb = L->route_hist[(size_t)b];
        return ca != cb ? ca > cb : a < b;
    });
    const int q = store_readahead(L->store, order.data(), (int)take, true);
    if (queued) *queued = q;
    return MOE_OK;
}

extern "C" moe_status moe_layer_set_weights(moe_layer* L, const moe_host_weights* w) {
    L->spare_expert = -1;  // the spare buffer holds weights of the old set
    if (!L || !w) return set_error(MOE_EINVAL, "layer or weights is NULL");
    const moe_qmatrix* all[] = {&w->router, &w->shared_gate, &w->shared_up, &w->shared_down, &w->gate, &w->up,
                                &w->down};
    const int n_needed = L->store ? 4 : 7;  // a streamed layer's routed experts come from its store
    for (int i = 0; i < n_needed; ++i)
        if (!all[i]->codes || !all[i]->scale || !all[i]->bias) return set_error(MOE_EINVAL, "a weight pointer is NULL");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    const moe_shapes& s = L->sh;
    const int d = s.d_model, I = s.d_ff, Is = s.d_ff_shared, E = s.n_experts;
    CUDA_TRY(cudaEventSynchronize(L->ev_done));
    CUDA_TRY(cudaStreamSynchronize(L->ctx->copy_stream));
    // router: codes as they are, (scale, bias) interleaved
    std::vector<uint32_t> sb((size_t)E * (d / 64));
    for (size_t i = 0; i < sb.size(); ++i) sb[i] = (uint32_t)w->router.scale[i] | ((uint32_t)w->router.bias[i] << 16);
    CUDA_TRY(cudaMemcpy(L->d_router_codes, w->router.codes, (size_t)E * d, cudaMemcpyHostToDevice));
    CUDA_TRY(cudaMemcpy(L->d_router_sb, sb.data(), sb.size() * 4, cudaMemcpyHostToDevice));
    // shared expert blob
    std::vector<uint8_t> blob(L->shared_bytes);
    repack_qmatrix(w->shared_gate, Is, d, blob.data());
    repack_qmatrix(w->shared_up, Is, d, blob.data() + qmat_bytes(Is, d));
    repack_down(w->shared_down, d, Is, blob.data() + 2 * qmat_bytes(Is, d));
    CUDA_TRY(cudaMemcpy(L->d_shared, blob.data(), blob.size(), cudaMemcpyHostToDevice));
    // routed experts into the pinned pool, expert-major
    const size_t gc = (size_t)I * (d / 2), gs = (size_t)I * (d / 64), dc = (size_t)d * (I / 2), ds = (size_t)d * (I / 64);
    auto one = [&](int e) {
        uint8_t* dst = L->h_pool + (size_t)e * L->ebytes;
        moe_qmatrix g{w->gate.codes + e * gc, w->gate.scale + e * gs, w->gate.bias + e * gs};
        moe_qmatrix u{w->up.codes + e * gc, w->up.scale + e * gs, w->up.bias + e * gs};
        moe_qmatrix dn{w->down.codes + e * dc, w->down.scale + e * ds, w->down.bias + e * ds};
        repack_qmatrix(g, I, d, dst);
        repack_qmatrix(u, I, d, dst + qmat_bytes(I, d));
        repack_down(dn, d, I, dst + 2 * qmat_bytes(I, d));
    };
    if (L->h_pool) {
        unsigned nth = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
        std::vector<std::thread> pool;
        for (unsigned t = 0; t < nth; ++t)
            pool.emplace_back([&, t] {
                for (int e = (int)t; e < E; e += (int)nth) one(e);
            });
        for (auto& th : pool) th.join();
    }
    L->cache.reset();
    moe_status st = table_upload_sync(L);
    if (st != MOE_OK) return st;
    L->loaded = true;
    return MOE_OK;
}

extern "C" moe_status moe_route(moe_layer* L, const void* x, int32_t T, const float* zbias, int32_t* ids,
                                float* gates, void* stream) {
    if (!L || !x || !ids || !gates || T < 1) return set_error(MOE_EINVAL, "moe_route: bad arguments");
    if (reinterpret_cast<uintptr_t>(x) & 15) return set_error(MOE_EINVAL, "moe_route: x must be 16-byte aligned");
    if (!L->loaded) return set_error(MOE_ESTATE, "moe_route before moe_layer_set_weights");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    cudaStream_t s = (cudaStream_t)stream;
    for (int t0 = 0; t0 < T; t0 += kPrefillChunk) {
        const int tc = std::min(kPrefillChunk, T - t0);
        moe_status st = ensure_scratch(L, std::max(tc, L->cap_T));
        if (st != MOE_OK) return st;
        CUDA_TRY(cudaStreamWaitEvent(s, L->ev_done, 0));
        st = route_into(L, static_cast<const uint16_t*>(x) + (size_t)t0 * L->sh.d_model, tc, zbias,
                        ids + (size_t)t0 * L->sh.top_k, gates + (size_t)t0 * L->sh.top_k, false, s);
        if (st != MOE_OK) return st;
        CUDA_TRY(cudaEventRecord(L->ev_done, s));
        L->last_stream = s;
        L->have_last_stream = true;
    }
    return MOE_OK;
}

extern "C" moe_status moe_cache_step(moe_layer* L, const int32_t* ids, int32_t n_ids, int32_t* slot_of,
                                     int32_t* miss_experts, int32_t* miss_slots, int32_t* n_miss) {
    if (!L || (!ids && n_ids > 0) || n_ids < 0) return set_error(MOE_EINVAL, "moe_cache_step: bad arguments");
    if (!L->loaded) return set_error(MOE_ESTATE, "moe_cache_step before moe_layer_set_weights");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    L->slot_before = L->cache.slot_expert;
    if (!L->cache.step(ids, n_ids, L->step)) return set_error(MOE_EINVAL, "moe_cache_step: expert id out of range");
    if (L->store)
        for (int e : L->step.distinct) ++L->route_hist[(size_t)e];
    L->stats.steps += 1;
    L->stats.hits += L->step.hits;
    L->stats.misses += L->step.miss_experts.size();
    L->stats.bypass += L->step.bypass;
    // slots being overwritten may still be read by this layer's earlier kernels
    CUDA_TRY(cudaStreamWaitEvent(L->ctx->copy_stream, L->ev_done, 0));
    moe_status st = issue_miss_copies(L, L->step, false, ++L->epoch, nullptr);
    // the device slot table follows the cache, behind the copies
    if (L->slot_before != L->cache.slot_expert) {
        moe_status tu = table_upload(L, L->ctx->copy_stream);
        if (st == MOE_OK) st = tu;
    }
    // the next forward treats these experts as resident: it waits for the copies first
    cudaError_t e = cudaEventRecord(L->ev_pending, L->ctx->copy_stream);
    L->pending = true;
    if (slot_of)
        for (int i = 0; i < n_ids; ++i) slot_of[i] = L->cache.slot_of(ids[i]);
    for (size_t i = 0; i < L->step.miss_experts.size(); ++i) {
        if (miss_experts) miss_experts[i] = L->step.miss_experts[i];
        if (miss_slots) miss_slots[i] = L->step.miss_slots[i];
    }
    if (n_miss) *n_miss = (int32_t)L->step.miss_experts.size();
    if (st == MOE_OK && e != cudaSuccess) return set_error(MOE_ECUDA, "event record failed: %s", cudaGetErrorString(e));
    return st;
}

extern "C" moe_status moe_forward(moe_layer* L, const void* x, int32_t T, const float* zbias, float* y,
                                  int32_t* ids_out, float* gates_out, void* stream) {
    if (!L || !x || !y || T < 1) return set_error(MOE_EINVAL, "moe_forward: bad arguments");
    if (reinterpret_cast<uintptr_t>(x) & 15) return set_error(MOE_EINVAL, "moe_forward: x must be 16-byte aligned");
    if (!L->loaded) return set_error(MOE_ESTATE, "moe_forward before moe_layer_set_weights");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    cudaStream_t s = (cudaStream_t)stream;
    const moe_shapes& sh = L->sh;
    const int chunk = T <= kDecodeMaxT ? T : kPrefillChunk;
    moe_status st = ensure_scratch(L, std::max(chunk, L->cap_T));
    if (st != MOE_OK) return st;
    for (int t0 = 0; t0 < T; t0 += chunk) {
        const int tc = std::min(chunk, T - t0);
        const uint16_t* xc = static_cast<const uint16_t*>(x) + (size_t)t0 * sh.d_model;
        float* yc = y + (size_t)t0 * sh.d_model;
        int32_t* io = ids_out ? ids_out + (size_t)t0 * sh.top_k : nullptr;
        float* go = gates_out ? gates_out + (size_t)t0 * sh.top_k : nullptr;
        st = forward_chunk(L, xc, tc, zbias, yc, io, go, s);
        if (st != MOE_OK) return st;
    }
    return MOE_OK;
}

extern "C" moe_status moe_forward_prompt(moe_layer* L, const void* x, int32_t T, const float* zbias, float* y,
                                         int32_t* ids_out, float* gates_out, void* stream) {
    if (!L || !x || !y || T < 1 || T > kPromptMaxT) return set_error(MOE_EINVAL, "moe_forward_prompt: bad arguments");
    if (reinterpret_cast<uintptr_t>(x) & 15)
        return set_error(MOE_EINVAL, "moe_forward_prompt: x must be 16-byte aligned");
    if (!L->loaded) return set_error(MOE_ESTATE, "moe_forward_prompt before moe_layer_set_weights");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    moe_status st = ensure_scratch(L, std::max(T, L->cap_T));
    if (st != MOE_OK) return st;
    return forward_chunk(L, static_cast<const uint16_t*>(x), T, zbias, y, ids_out, gates_out, (cudaStream_t)stream);
}

extern "C" moe_status moe_cache_reset(moe_layer* L) {
    if (!L) return set_error(MOE_EINVAL, "layer is NULL");
    if (!L->loaded) return set_error(MOE_ESTATE, "moe_cache_reset before moe_layer_set_weights");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    L->cache.reset();
    return table_upload_sync(L);
}

extern "C" moe_status moe_layer_stats(moe_layer* L, moe_stats* out) {
    if (!L || !out) return set_error(MOE_EINVAL, "moe_layer_stats: bad arguments");
    cudaSetDevice(L->ctx->device);
    drain_waits(L);
    *out = L->stats;
    return MOE_OK;
}

extern "C" moe_status moe_layer_reset_stats(moe_layer* L) {
    if (!L) return set_error(MOE_EINVAL, "layer is NULL");
    cudaSetDevice(L->ctx->device);
    drain_waits(L);
    L->stats = moe_stats{};
    return MOE_OK;
}

extern "C" moe_status moe_cache_dump(const moe_layer* L, int32_t* slot_expert, uint32_t* counts) {
    if (!L) return set_error(MOE_EINVAL, "layer is NULL");
    for (int s = 0; s < L->S; ++s) {
        if (slot_expert) slot_expert[s] = L->cache.slot_expert[s];
        if (counts) counts[s] = L->cache.use_count[s];
    }
    return MOE_OK;
}

extern "C" moe_status moe_ctx_set_profiling(moe_ctx* C, int32_t on) {
    if (!C) return set_error(MOE_EINVAL, "ctx is NULL");
    C->profiling = on != 0;
    return MOE_OK;
}

extern "C" moe_status moe_ctx_kernel_times(moe_ctx* C, int32_t kind, uint64_t* launches, double* total_ms,
                                           double* bytes, double* flops) {
    if (!C || kind < 0 || kind >= kKinds) return set_error(MOE_EINVAL, "moe_ctx_kernel_times: bad arguments");
    cudaSetDevice(C->device);
    drain_prof(C);
    if (launches) *launches = C->acc[kind].n;
    if (total_ms) *total_ms = C->acc[kind].ms;
    if (bytes) *bytes = C->acc[kind].bytes;
    if (flops) *flops = C->acc[kind].flops;
    return MOE_OK;
}

extern "C" moe_status moe_ctx_reset_kernel_times(moe_ctx* C) {
    if (!C) return set_error(MOE_EINVAL, "ctx is NULL");
    cudaSetDevice(C->device);
    drain_prof(C);
    for (auto& a : C->acc) a = moe_ctx::Acc{};
    return MOE_OK;
}

extern "C" moe_status moe_ctx_launches(moe_ctx* C, uint64_t* out) {
    if (!C || !out) return set_error(MOE_EINVAL, "moe_ctx_launches: bad arguments");
    *out = C->launches;
    return MOE_OK;
}

extern "C" moe_status moe_ctx_inject_copy_failure(moe_ctx* C, int64_t nth) {
    if (!C) return set_error(MOE_EINVAL, "ctx is NULL");
    C->fail_copy_at = nth < 0 ? -1 : C->copies_issued + nth;
    return MOE_OK;
}

extern "C" moe_status moe_layer_set_prefetch(moe_layer* L, int32_t on) {
    if (!L || (on != 0 && on != 1)) return set_error(MOE_EINVAL, "moe_layer_set_prefetch: bad arguments");
    if (L->store) return set_error(MOE_EINVAL, "moe_layer_set_prefetch: a streamed layer reads ahead into its tier");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    if (L->ev_done) CUDA_TRY(cudaEventSynchronize(L->ev_done));
    CUDA_TRY(cudaStreamSynchronize(L->ctx->copy_stream));
    if (on && !L->d_spare && cudaMalloc(&L->d_spare, L->ebytes) != cudaSuccess) {
        cudaGetLastError();
        return set_error(MOE_ENOMEM, "prefetch buffer of %zu bytes failed", L->ebytes);
    }
    if (on && !L->ev_spare_ready) {
        CUDA_TRY(cudaEventCreateWithFlags(&L->ev_spare_ready, cudaEventDisableTiming));
        CUDA_TRY(cudaEventCreateWithFlags(&L->ev_spare_free, cudaEventDisableTiming));
    }
    L->spare_free_recorded = false;
    if (!on) {
        cudaFree(L->d_spare);
        L->d_spare = nullptr;
    }
    L->prefetch = on != 0;
    L->spare_expert = -1;
    if ((int)L->route_hist.size() != L->sh.n_experts) L->route_hist.assign(L->sh.n_experts, 0);
    return MOE_OK;
}

extern "C" moe_status moe_layer_prefetch_stats(const moe_layer* L, uint64_t* issued, uint64_t* used) {
    if (!L) return set_error(MOE_EINVAL, "layer is NULL");
    if (issued) *issued = L->prefetch_issued;
    if (used) *used = L->prefetch_used;
    return MOE_OK;
}

extern "C" moe_status moe_layer_set_deterministic(moe_layer* L, int32_t on) {
    if (!L || (on != 0 && on != 1)) return set_error(MOE_EINVAL, "moe_layer_set_deterministic: bad arguments");
    if (L->ev_done) {
        CUDA_TRY(cudaSetDevice(L->ctx->device));
        CUDA_TRY(cudaEventSynchronize(L->ev_done));  // calls in flight keep the mode they started with
    }
    L->deterministic = on != 0;
    return MOE_OK;
}

extern "C" moe_status moe_layers_replay_resident(moe_layer* const* layers, int32_t n_layers, int32_t rounds,
                                                 void* stream, double* bytes) {
    if (!layers || n_layers < 1 || rounds < 1) return set_error(MOE_EINVAL, "moe_layers_replay_resident: bad arguments");
    double by = 0;
    for (int i = 0; i < n_layers; ++i) {
        moe_layer* L = layers[i];
        if (!L) return set_error(MOE_EINVAL, "layer %d is NULL", i);
        if (!L->have_resident || (int)L->h_ids.size() < L->sh.top_k)
            return set_error(MOE_ESTATE, "moe_layers_replay_resident: layer %d made no one-token call yet", i);
        if (L->ctx->device != layers[0]->ctx->device)
            return set_error(MOE_EINVAL, "moe_layers_replay_resident: layers on different devices");
        // the routed items read the experts of the last routing that are resident now
        double b = (double)L->shared_bytes;
        for (int p = 0; p < L->sh.top_k; ++p)
            if (L->cache.slot_of(L->h_ids[p]) >= 0) b += (double)L->ebytes;
        by += b;
    }
    CUDA_TRY(cudaSetDevice(layers[0]->ctx->device));
    // the routed items resolved on the host (slot addresses of the recorded
    // routing), so that no unit waits for the previous kernel before it
    // starts: what is timed is the launch's own work
    std::vector<FfnSmall> lists(n_layers);
    std::vector<FfnArgs> args(n_layers);
    for (int i = 0; i < n_layers; ++i) {
        moe_layer* L = layers[i];
        const FfnSmall& src = L->resident_list;
        FfnSmall& l = lists[i];
        l = FfnSmall{};
        l.epoch = src.epoch;
        int n0 = 0, n1 = 0;
        for (int it = 0; it < src.n_items; ++it) {
            FfnItem x = src.item[it];
            const int fam = it < L->resident_args.fam[0].n_items ? 0 : 1;
            if (!x.w) {
                const int e = L->h_ids[src.pair[x.pb]];
                const int slot = L->cache.slot_of(e);
                if (slot < 0) continue;
                x.w = L->d_slots + (size_t)slot * L->ebytes;
            }
            x.pb = (int16_t)(n0 + n1);
            l.pair[n0 + n1] = src.pair[src.item[it].pb];
            l.item[n0 + n1] = x;
            if (fam == 0) ++n0; else ++n1;
        }
        l.n_items = n0 + n1;
        args[i] = L->resident_args;
        args[i].fam[0].n_items = n0;
        args[i].fam[1].n_items = n1;
        args[i].ids = nullptr;
        args[i].slot_of = nullptr;
    }
    for (int r = 0; r < rounds; ++r)
        for (int i = 0; i < n_layers; ++i) {
            CUDA_TRY(launch_ffn(args[i], lists[i], (cudaStream_t)stream, true));
            ++layers[i]->ctx->launches;
        }
    if (bytes) *bytes = by * rounds;
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// moe_route_noalloc: the router with library-owned static scratch.
//
// For callers that cannot allocate: a decode loop on a fixed memory budget,
// or one that cannot take the device-wide synchronisation of the cudaFree in
// ensure_scratch's growth path. The scratch below is sized once at compile
// time; the entry point never calls cudaMalloc, cudaFree or any routine that
// allocates. Every layer on a device shares it, so overlapping calls race.

namespace {

constexpr int kNoAllocMaxT = 64;
constexpr int kNoAllocLogits = 16384;                                // fp32 logits, T * n_experts
constexpr int kNoAllocCounters = (kNoAllocMaxT + 7) / 8;            // one per block of 8 tokens
constexpr int kNoAllocMaxDevices = 64;

// Zero at load; the router's last block per token block puts its counter back to zero.
static __device__ __align__(256) float g_noalloc_logits[kNoAllocLogits];
static __device__ __align__(256) unsigned g_noalloc_counters[kNoAllocCounters];

struct NoAllocScratch {
    float* logits = nullptr;
    unsigned* counters = nullptr;
};
std::mutex g_noalloc_mu;
NoAllocScratch g_noalloc[kNoAllocMaxDevices];

// Device addresses of the scratch on `device`, looked up once per device with
// that device current.
moe_status noalloc_scratch(int device, NoAllocScratch* out) {
    if (device < 0 || device >= kNoAllocMaxDevices)
        return set_error(MOE_EINVAL, "moe_route_noalloc: device %d out of [0, %d)", device, kNoAllocMaxDevices);
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    NoAllocScratch& sc = g_noalloc[device];
    if (!sc.logits) {
        void* l = nullptr;
        void* c = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&l, g_noalloc_logits);
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&c, g_noalloc_counters);
        if (e != cudaSuccess)
            return set_error(MOE_ECUDA, "moe_route_noalloc: scratch lookup failed: %s", cudaGetErrorString(e));
        sc.logits = static_cast<float*>(l);
        sc.counters = static_cast<unsigned*>(c);
    }
    *out = sc;
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_route_noalloc(moe_layer* L, const void* x, int32_t T, const float* zbias, int32_t* ids,
                                        float* gates, void* stream) {
    if (!L || !x || !ids || !gates || T < 1) return set_error(MOE_EINVAL, "moe_route_noalloc: bad arguments");
    if (reinterpret_cast<uintptr_t>(x) & 15)
        return set_error(MOE_EINVAL, "moe_route_noalloc: x must be 16-byte aligned");
    if (!L->loaded) return set_error(MOE_ESTATE, "moe_route_noalloc before moe_layer_set_weights");
    if (T > kNoAllocMaxT || (long)T * L->sh.n_experts > kNoAllocLogits)
        return set_error(MOE_EINVAL,
                         "moe_route_noalloc: T = %d with %d experts exceeds the static scratch "
                         "(T <= %d and T * n_experts <= %d)",
                         T, L->sh.n_experts, kNoAllocMaxT, kNoAllocLogits);
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    NoAllocScratch sc;
    moe_status st = noalloc_scratch(L->ctx->device, &sc);
    if (st != MOE_OK) return st;
    RouterParams p{static_cast<const uint16_t*>(x), T, L->sh.d_model, L->sh.n_experts, L->sh.top_k,
                   L->d_router_codes, L->d_router_sb, zbias, sc.logits, sc.counters, ids, gates, nullptr, 0};
    CUDA_TRY(launch_router(p, (cudaStream_t)stream));
    // counted, but never timed: a timing record would create CUDA events
    ++L->ctx->launches;
    return MOE_OK;
}
