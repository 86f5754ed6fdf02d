// libmoe C ABI: contexts, layers, weight loading, routing, the expert cache
// step with miss streaming, and the layer forward.
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
//
// Per layer and call (decode), the three phases of [P1] §2.4 / §8.2 map to:
//   cb1  router kernel on the caller's stream, ids copied to pinned host memory;
//        the shared expert is enqueued behind it, so it runs while the host
//        waits and while misses stream ([P1] §2.4: "meanwhile the GPU can start
//        the shared-expert branch");
//   io   host LFU/LRU step; one cudaMemcpyAsync per miss from the pinned pool
//        into its HBM slot on the context's copy stream, each followed by that
//        slot's ready event ([P3] "读取完成后，算子才可以使用切片": a hit is
//        ready at once, a miss when its read completes);
//   cb2  routed experts that hit run at once; the compute stream then waits on
//        the ready events of the misses and runs them; the combine adds the
//        gate-weighted expert outputs to the shared output in rank order.
// Ready state is an event per slot, re-recorded by every copy into the slot,
// so a later wait can never observe a stale "ready" from an earlier round.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <new>
#include <thread>
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

void repack_qmatrix(const moe_qmatrix& m, int N, int K, uint8_t* dst) {
    const int C = K / 32, G = K / 64;
    uint8_t* codes = dst;
    uint32_t* sb = reinterpret_cast<uint32_t*>(dst + (size_t)N * (size_t)K / 2);
    for (int n = 0; n < N; ++n) {
        const int rt = n >> 5, lane = n & 31;
        const uint8_t* src = m.codes + (size_t)n * (size_t)(K / 2);
        for (int c = 0; c < C; ++c) memcpy(codes + (((size_t)rt * C + c) * 32 + lane) * 16, src + (size_t)c * 16, 16);
        for (int g = 0; g < G; ++g) {
            const size_t i = (size_t)n * G + g;
            sb[((size_t)rt * G + g) * 32 + lane] = (uint32_t)m.scale[i] | ((uint32_t)m.bias[i] << 16);
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
enum Kind { K_ROUTER = 0, K_SHARED_GU, K_SHARED_DN, K_ROUTED_GU, K_ROUTED_DN, K_COMBINE, K_GEMM_GU, K_GEMM_DN };

struct ProfRec {
    int kind;
    cudaEvent_t a, b;
    double bytes, flops;
};

struct WaitRec {
    cudaEvent_t a, b;
};

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
    long fail_copy_at = -1;  // test hook: the n-th miss copy from now reports failure
    long copies_issued = 0;
    std::mutex mu;

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
    moe_shapes sh{};
    int S = 0, policy = 0;
    size_t ebytes = 0, shared_bytes = 0, router_bytes = 0;
    uint8_t* d_router_codes = nullptr;
    uint32_t* d_router_sb = nullptr;
    uint8_t* d_shared = nullptr;
    uint8_t* d_slots = nullptr;
    uint8_t* h_pool = nullptr;  // pinned, E * ebytes
    HostCache cache;
    StepResult step;
    std::vector<cudaEvent_t> slot_ready;
    cudaEvent_t ev_ids = nullptr, ev_done = nullptr, ev_bypass = nullptr;
    bool loaded = false;
    // scratch, sized for cap_T tokens
    int cap_T = 0;
    float* d_logits = nullptr;
    unsigned* d_counters = nullptr;
    int32_t* d_ids = nullptr;
    float* d_gates = nullptr;
    float* d_h = nullptr;
    float* d_hs = nullptr;
    float* d_o = nullptr;
    int32_t* h_ids = nullptr;  // pinned
    std::vector<int32_t> offsets, perm;
    moe_stats stats{};
    std::vector<WaitRec> waits;

    moe_layer(int E, int S_, int pol) : cache(E, S_, pol) {}
};

namespace {

moe_status check_shapes(const moe_shapes* s) {
    if (!s) return set_error(MOE_EINVAL, "shapes is NULL");
    if (s->d_model < 64 || s->d_model > kMaxDModel || s->d_model % 256 != 0)
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

void free_scratch(moe_layer* L) {
    cudaFree(L->d_logits);
    cudaFree(L->d_counters);
    cudaFree(L->d_ids);
    cudaFree(L->d_gates);
    cudaFree(L->d_h);
    cudaFree(L->d_hs);
    cudaFree(L->d_o);
    cudaFreeHost(L->h_ids);
    L->d_logits = nullptr;
    L->d_counters = nullptr;
    L->d_ids = nullptr;
    L->d_gates = nullptr;
    L->d_h = L->d_hs = L->d_o = nullptr;
    L->h_ids = nullptr;
    L->cap_T = 0;
}

// Scratch for up to T tokens per call (grows; never shrinks).
moe_status ensure_scratch(moe_layer* L, int T) {
    if (T <= L->cap_T) return MOE_OK;
    if (L->ev_done) CUDA_TRY(cudaEventSynchronize(L->ev_done));  // old buffers may still be in use
    free_scratch(L);
    const moe_shapes& s = L->sh;
    const size_t pairs = (size_t)T * s.top_k;
    const int blocks = (T + 7) / 8;
    bool ok = cudaMalloc(&L->d_logits, sizeof(float) * T * s.n_experts) == cudaSuccess &&
              cudaMalloc(&L->d_counters, sizeof(unsigned) * blocks) == cudaSuccess &&
              cudaMemset(L->d_counters, 0, sizeof(unsigned) * blocks) == cudaSuccess &&
              cudaMalloc(&L->d_ids, sizeof(int32_t) * pairs) == cudaSuccess &&
              cudaMalloc(&L->d_gates, sizeof(float) * pairs) == cudaSuccess &&
              cudaMalloc(&L->d_h, sizeof(float) * pairs * s.d_ff) == cudaSuccess &&
              cudaMalloc(&L->d_hs, sizeof(float) * (size_t)T * s.d_ff_shared) == cudaSuccess &&
              cudaMalloc(&L->d_o, sizeof(float) * pairs * s.d_model) == cudaSuccess &&
              cudaHostAlloc(&L->h_ids, sizeof(int32_t) * pairs, cudaHostAllocDefault) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        free_scratch(L);
        return set_error(MOE_ENOMEM, "scratch allocation for %d tokens failed", T);
    }
    L->cap_T = T;
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

void drain_waits(moe_layer* L) {
    for (WaitRec& w : L->waits) {
        cudaEventSynchronize(w.b);
        float ms = 0;
        cudaEventElapsedTime(&ms, w.a, w.b);
        L->stats.exposed_copy_us += 1000.0 * ms;
        L->ctx->timing_pool.push_back(w.a);
        L->ctx->timing_pool.push_back(w.b);
    }
    L->waits.clear();
}

double qbytes(int N, int K) { return (double)qmat_bytes(N, K); }

// Issue the copies of one cache step's misses. Slot misses land in their
// slots and record the slot's ready event; bypassed experts land in staging,
// in miss order, and share one ready event. On failure the failed slot is
// emptied so that the table never claims an expert whose bytes are missing.
moe_status issue_miss_copies(moe_layer* L, const StepResult& r, bool with_bypass, int* n_bypass_staged) {
    moe_ctx* C = L->ctx;
    int nb = 0;
    if (with_bypass && r.bypass > 0) {
        moe_status st = ensure_staging(C, (size_t)r.bypass * L->ebytes);
        if (st != MOE_OK) return st;
        CUDA_TRY(cudaStreamWaitEvent(C->copy_stream, C->staging_free, 0));
    }
    for (size_t i = 0; i < r.miss_experts.size(); ++i) {
        const int e = r.miss_experts[i], slot = r.miss_slots[i];
        if (slot < 0 && !with_bypass) continue;
        uint8_t* dst = slot >= 0 ? L->d_slots + (size_t)slot * L->ebytes : C->staging + (size_t)nb * L->ebytes;
        bool fail = false;
        if (C->fail_copy_at >= 0 && C->copies_issued == C->fail_copy_at) {
            fail = true;
            C->fail_copy_at = -1;
        }
        ++C->copies_issued;
        cudaError_t ce = fail ? cudaErrorUnknown
                              : cudaMemcpyAsync(dst, L->h_pool + (size_t)e * L->ebytes, L->ebytes,
                                                cudaMemcpyHostToDevice, C->copy_stream);
        if (ce != cudaSuccess) {
            if (!fail) cudaGetLastError();
            // empty every slot this step filled but whose copy is not known good
            for (size_t j = i; j < r.miss_experts.size(); ++j)
                if (r.miss_slots[j] >= 0) L->cache.evict(r.miss_slots[j]);
            return set_error(MOE_ECOPY, "copy of expert %d (slot %d) failed: %s", e, slot,
                             fail ? "injected failure" : cudaGetErrorString(ce));
        }
        L->stats.bytes_h2d += L->ebytes;
        if (slot >= 0)
            CUDA_TRY(cudaEventRecord(L->slot_ready[slot], C->copy_stream));
        else
            ++nb;
    }
    if (nb > 0) CUDA_TRY(cudaEventRecord(L->ev_bypass, C->copy_stream));
    if (n_bypass_staged) *n_bypass_staged = nb;
    return MOE_OK;
}

template <class List>
bool add_item(List& l, const uint8_t* w, const int32_t* perm, int b, int e_) {
    constexpr int MAXI = sizeof(l.w) / sizeof(l.w[0]);
    constexpr int MAXP = sizeof(l.pair) / sizeof(l.pair[0]);
    if (l.n_items >= MAXI || l.begin[l.n_items] + (e_ - b) > MAXP) return false;
    l.w[l.n_items] = w;
    int p = l.begin[l.n_items];
    for (int i = b; i < e_; ++i) l.pair[p++] = (int16_t)perm[i];
    ++l.n_items;
    l.begin[l.n_items] = (int16_t)p;
    return true;
}

struct Item {
    const uint8_t* w;
    int b, e;  // pair range in perm
};

// Gate/up and down for a set of experts, packed into as few work lists as fit.
template <class List>
moe_status launch_items(moe_layer* L, const uint16_t* x, const std::vector<Item>& items, cudaStream_t s) {
    moe_ctx* C = L->ctx;
    const moe_shapes& sh = L->sh;
    const double egu = 2 * qbytes(sh.d_ff, sh.d_model), edn = qbytes(sh.d_model, sh.d_ff);
    size_t i = 0;
    while (i < items.size()) {
        List l{};
        l.begin[0] = 0;
        while (i < items.size() && add_item(l, items[i].w, L->perm.data(), items[i].b, items[i].e)) ++i;
        if (l.n_items == 0) return set_error(MOE_EINVAL, "expert with too many pairs for one work list");
        const double np = l.begin[l.n_items];
        {
            Prof p(C, s, K_ROUTED_GU, l.n_items * egu, 2.0 * np * 2 * sh.d_ff * sh.d_model);
            CUDA_TRY(launch_gateup(x, sh.d_model, sh.d_ff, sh.act, sh.top_k, l, L->d_h, s));
        }
        {
            Prof p(C, s, K_ROUTED_DN, l.n_items * edn, 2.0 * np * sh.d_ff * sh.d_model);
            CUDA_TRY(launch_down(L->d_h, sh.d_ff, sh.d_model, l, L->d_o, s));
        }
        L->stats.bytes_resident += (uint64_t)(l.n_items * (egu + edn));
    }
    return MOE_OK;
}

moe_status launch_items_any(moe_layer* L, const uint16_t* x, const std::vector<Item>& items, cudaStream_t s) {
    if (items.empty()) return MOE_OK;
    int pairs = 0;
    for (const Item& it : items) pairs += it.e - it.b;
    if ((int)items.size() <= 16 && pairs <= 64) return launch_items<SmallList>(L, x, items, s);
    return launch_items<LargeList>(L, x, items, s);
}

// Routed experts: hits first, then (after the ready events) misses.
moe_status run_routed(moe_layer* L, const uint16_t* x, int T, int nb_staged, cudaStream_t s) {
    moe_ctx* C = L->ctx;
    const moe_shapes& sh = L->sh;
    const int npairs = T * sh.top_k;
    L->offsets.resize(sh.n_experts + 1);
    L->perm.resize(npairs);
    group_pairs(L->h_ids, npairs, sh.n_experts, L->offsets.data(), L->perm.data());
    std::vector<Item> hit, miss;
    std::vector<int> miss_slots;
    int bypass_i = 0;
    size_t mi = 0;
    for (int e : L->step.distinct) {
        int slot = -1;
        bool is_miss = false;
        while (mi < L->step.miss_experts.size() && L->step.miss_experts[mi] < e) ++mi;
        if (mi < L->step.miss_experts.size() && L->step.miss_experts[mi] == e) {
            is_miss = true;
            slot = L->step.miss_slots[mi];
        } else {
            slot = L->cache.slot_of(e);
        }
        const uint8_t* w;
        if (slot >= 0) {
            w = L->d_slots + (size_t)slot * L->ebytes;
        } else {
            if (bypass_i >= nb_staged) return set_error(MOE_ESTATE, "bypassed expert %d has no staging", e);
            w = C->staging + (size_t)bypass_i * L->ebytes;
            ++bypass_i;
        }
        (is_miss ? miss : hit).push_back(Item{w, L->offsets[e], L->offsets[e + 1]});
        if (is_miss && slot >= 0) miss_slots.push_back(slot);
    }
    moe_status st = launch_items_any(L, x, hit, s);
    if (st != MOE_OK) return st;
    if (!miss.empty()) {
        WaitRec w{C->timing_event(), C->timing_event()};
        CUDA_TRY(cudaEventRecord(w.a, s));
        for (int slot : miss_slots) CUDA_TRY(cudaStreamWaitEvent(s, L->slot_ready[slot], 0));
        if (nb_staged > 0) CUDA_TRY(cudaStreamWaitEvent(s, L->ev_bypass, 0));
        CUDA_TRY(cudaEventRecord(w.b, s));
        L->waits.push_back(w);
        st = launch_items_any(L, x, miss, s);
        if (st != MOE_OK) return st;
    }
    return MOE_OK;
}

moe_status route_into(moe_layer* L, const uint16_t* x, int T, const float* zbias, int32_t* ids, float* gates,
                      cudaStream_t s) {
    RouterParams p{x, T, L->sh.d_model, L->sh.n_experts, L->sh.top_k, L->d_router_codes, L->d_router_sb, zbias,
                   L->d_logits, L->d_counters, ids, gates};
    Prof pr(L->ctx, s, K_ROUTER, (double)L->router_bytes + 2.0 * T * L->sh.d_model,
            2.0 * T * L->sh.n_experts * L->sh.d_model);
    CUDA_TRY(launch_router(p, s));
    L->stats.bytes_resident += L->router_bytes;
    return MOE_OK;
}

template <class List>
moe_status shared_expert_t(moe_layer* L, const uint16_t* x, int T, float* y, cudaStream_t s) {
    const moe_shapes& sh = L->sh;
    List l{};
    l.n_items = 1;
    l.w[0] = L->d_shared;
    l.begin[0] = 0;
    l.begin[1] = (int16_t)T;
    for (int t = 0; t < T; ++t) l.pair[t] = (int16_t)t;
    {
        Prof p(L->ctx, s, K_SHARED_GU, 2 * qbytes(sh.d_ff_shared, sh.d_model), 4.0 * T * sh.d_ff_shared * sh.d_model);
        CUDA_TRY(launch_gateup(x, sh.d_model, sh.d_ff_shared, sh.act, 1, l, L->d_hs, s));
    }
    {
        Prof p(L->ctx, s, K_SHARED_DN, qbytes(sh.d_model, sh.d_ff_shared), 2.0 * T * sh.d_ff_shared * sh.d_model);
        CUDA_TRY(launch_down(L->d_hs, sh.d_ff_shared, sh.d_model, l, y, s));
    }
    L->stats.bytes_resident += L->shared_bytes;
    return MOE_OK;
}

moe_status shared_expert(moe_layer* L, const uint16_t* x, int T, float* y, cudaStream_t s) {
    return T <= 64 ? shared_expert_t<SmallList>(L, x, T, y, s) : shared_expert_t<LargeList>(L, x, T, y, s);
}

// One call of at most kPrefillChunk tokens.
moe_status forward_chunk(moe_layer* L, const uint16_t* x, int T, const float* zbias, float* y, int32_t* ids_out,
                         float* gates_out, cudaStream_t s) {
    moe_ctx* C = L->ctx;
    const moe_shapes& sh = L->sh;
    const int npairs = T * sh.top_k;
    CUDA_TRY(cudaStreamWaitEvent(s, L->ev_done, 0));
    moe_status st = route_into(L, x, T, zbias, L->d_ids, L->d_gates, s);
    if (st != MOE_OK) return st;
    CUDA_TRY(cudaMemcpyAsync(L->h_ids, L->d_ids, sizeof(int32_t) * npairs, cudaMemcpyDeviceToHost, s));
    CUDA_TRY(cudaEventRecord(L->ev_ids, s));
    st = shared_expert(L, x, T, y, s);  // overlaps the host step and the miss copies
    if (st != MOE_OK) return st;
    CUDA_TRY(cudaEventSynchronize(L->ev_ids));
    if (!L->cache.step(L->h_ids, npairs, L->step)) return set_error(MOE_ESTATE, "router produced an invalid id");
    L->stats.steps += 1;
    L->stats.hits += L->step.hits;
    L->stats.misses += L->step.miss_experts.size();
    L->stats.bypass += L->step.bypass;
    int nb = 0;
    st = issue_miss_copies(L, L->step, true, &nb);
    if (st != MOE_OK) return st;
    st = run_routed(L, x, T, nb, s);
    if (st != MOE_OK) return st;
    {
        Prof p(C, s, K_COMBINE, 4.0 * npairs * sh.d_model + 8.0 * T * sh.d_model, 2.0 * npairs * sh.d_model);
        CUDA_TRY(launch_combine(L->d_o, L->d_gates, T, sh.top_k, sh.d_model, y, s));
    }
    if (ids_out) CUDA_TRY(cudaMemcpyAsync(ids_out, L->d_ids, sizeof(int32_t) * npairs, cudaMemcpyDeviceToDevice, s));
    if (gates_out)
        CUDA_TRY(cudaMemcpyAsync(gates_out, L->d_gates, sizeof(float) * npairs, cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaEventRecord(L->ev_done, s));
    if (nb > 0) CUDA_TRY(cudaEventRecord(C->staging_free, s));
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
        cudaEventCreateWithFlags(&C->staging_free, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        delete C;
        return set_error(MOE_ECUDA, "stream/event creation failed");
    }
    *out = C;
    return MOE_OK;
}

extern "C" void moe_ctx_destroy(moe_ctx* C) {
    if (!C) return;
    cudaSetDevice(C->device);
    cudaStreamSynchronize(C->copy_stream);
    drain_prof(C);
    for (cudaEvent_t e : C->timing_pool) cudaEventDestroy(e);
    cudaFree(C->staging);
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
    cudaFree(L->d_router_codes);
    cudaFree(L->d_router_sb);
    cudaFree(L->d_shared);
    cudaFree(L->d_slots);
    cudaFreeHost(L->h_pool);
    for (cudaEvent_t e : L->slot_ready) cudaEventDestroy(e);
    if (L->ev_ids) cudaEventDestroy(L->ev_ids);
    if (L->ev_done) cudaEventDestroy(L->ev_done);
    if (L->ev_bypass) cudaEventDestroy(L->ev_bypass);
    delete L;
}

extern "C" moe_status moe_layer_create(moe_ctx* C, const moe_shapes* s, const moe_quant_layout* q, int32_t slots,
                                       int32_t policy, moe_layer** out) {
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
    L->sh = *s;
    L->S = slots;
    L->policy = policy;
    L->ebytes = expert_blob_bytes(s->d_model, s->d_ff);
    L->shared_bytes = expert_blob_bytes(s->d_model, s->d_ff_shared);
    L->router_bytes = (size_t)s->n_experts * s->d_model + (size_t)s->n_experts * (s->d_model / 64) * 4;
    bool ok = cudaMalloc(&L->d_router_codes, (size_t)s->n_experts * s->d_model) == cudaSuccess &&
              cudaMalloc(&L->d_router_sb, (size_t)s->n_experts * (s->d_model / 64) * 4) == cudaSuccess &&
              cudaMalloc(&L->d_shared, L->shared_bytes) == cudaSuccess &&
              cudaMalloc(&L->d_slots, (size_t)slots * L->ebytes) == cudaSuccess &&
              cudaHostAlloc(&L->h_pool, (size_t)s->n_experts * L->ebytes, cudaHostAllocDefault) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        moe_layer_destroy(L);
        return set_error(MOE_ENOMEM, "layer allocation failed (%zu B pinned pool, %zu B slots)",
                         (size_t)s->n_experts * L->ebytes, (size_t)slots * L->ebytes);
    }
    L->slot_ready.resize(slots, nullptr);
    for (int i = 0; i < slots; ++i)
        if (cudaEventCreateWithFlags(&L->slot_ready[i], cudaEventDisableTiming) != cudaSuccess) ok = false;
    ok = ok && cudaEventCreateWithFlags(&L->ev_ids, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&L->ev_done, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&L->ev_bypass, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        moe_layer_destroy(L);
        return set_error(MOE_ECUDA, "event creation failed");
    }
    *out = L;
    return MOE_OK;
}

extern "C" moe_status moe_layer_set_weights(moe_layer* L, const moe_host_weights* w) {
    if (!L || !w) return set_error(MOE_EINVAL, "layer or weights is NULL");
    const moe_qmatrix* all[] = {&w->router, &w->shared_gate, &w->shared_up, &w->shared_down, &w->gate, &w->up,
                                &w->down};
    for (const moe_qmatrix* m : all)
        if (!m->codes || !m->scale || !m->bias) return set_error(MOE_EINVAL, "a weight pointer is NULL");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    const moe_shapes& s = L->sh;
    const int d = s.d_model, I = s.d_ff, Is = s.d_ff_shared, E = s.n_experts;
    if (L->ev_done) CUDA_TRY(cudaEventSynchronize(L->ev_done));
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
    repack_qmatrix(w->shared_down, d, Is, blob.data() + 2 * qmat_bytes(Is, d));
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
        repack_qmatrix(dn, d, I, dst + 2 * qmat_bytes(I, d));
    };
    unsigned nth = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
    std::vector<std::thread> pool;
    for (unsigned t = 0; t < nth; ++t)
        pool.emplace_back([&, t] {
            for (int e = (int)t; e < E; e += (int)nth) one(e);
        });
    for (auto& th : pool) th.join();
    L->cache.reset();
    L->loaded = true;
    return MOE_OK;
}

extern "C" moe_status moe_route(moe_layer* L, const void* x, int32_t T, const float* zbias, int32_t* ids,
                                float* gates, void* stream) {
    if (!L || !x || !ids || !gates || T < 1) return set_error(MOE_EINVAL, "moe_route: bad arguments");
    if (!L->loaded) return set_error(MOE_ESTATE, "moe_route before moe_layer_set_weights");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    cudaStream_t s = (cudaStream_t)stream;
    for (int t0 = 0; t0 < T; t0 += kPrefillChunk) {
        const int tc = std::min(kPrefillChunk, T - t0);
        moe_status st = ensure_scratch(L, std::max(tc, L->cap_T));
        if (st != MOE_OK) return st;
        CUDA_TRY(cudaStreamWaitEvent(s, L->ev_done, 0));
        st = route_into(L, static_cast<const uint16_t*>(x) + (size_t)t0 * L->sh.d_model, tc, zbias,
                        ids + (size_t)t0 * L->sh.top_k, gates + (size_t)t0 * L->sh.top_k, s);
        if (st != MOE_OK) return st;
        CUDA_TRY(cudaEventRecord(L->ev_done, s));
    }
    return MOE_OK;
}

extern "C" moe_status moe_cache_step(moe_layer* L, const int32_t* ids, int32_t n_ids, int32_t* slot_of,
                                     int32_t* miss_experts, int32_t* miss_slots, int32_t* n_miss) {
    if (!L || (!ids && n_ids > 0) || n_ids < 0) return set_error(MOE_EINVAL, "moe_cache_step: bad arguments");
    if (!L->loaded) return set_error(MOE_ESTATE, "moe_cache_step before moe_layer_set_weights");
    CUDA_TRY(cudaSetDevice(L->ctx->device));
    if (!L->cache.step(ids, n_ids, L->step)) return set_error(MOE_EINVAL, "moe_cache_step: expert id out of range");
    L->stats.steps += 1;
    L->stats.hits += L->step.hits;
    L->stats.misses += L->step.miss_experts.size();
    L->stats.bypass += L->step.bypass;
    // slots being overwritten may still be read by this layer's earlier kernels
    CUDA_TRY(cudaStreamWaitEvent(L->ctx->copy_stream, L->ev_done, 0));
    moe_status st = issue_miss_copies(L, L->step, false, nullptr);
    if (slot_of)
        for (int i = 0; i < n_ids; ++i) slot_of[i] = L->cache.slot_of(ids[i]);
    for (size_t i = 0; i < L->step.miss_experts.size(); ++i) {
        if (miss_experts) miss_experts[i] = L->step.miss_experts[i];
        if (miss_slots) miss_slots[i] = L->step.miss_slots[i];
    }
    if (n_miss) *n_miss = (int32_t)L->step.miss_experts.size();
    return st;
}

extern "C" moe_status moe_forward(moe_layer* L, const void* x, int32_t T, const float* zbias, float* y,
                                  int32_t* ids_out, float* gates_out, void* stream) {
    if (!L || !x || !y || T < 1) return set_error(MOE_EINVAL, "moe_forward: bad arguments");
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

extern "C" moe_status moe_ctx_inject_copy_failure(moe_ctx* C, int64_t nth) {
    if (!C) return set_error(MOE_EINVAL, "ctx is NULL");
    C->fail_copy_at = nth < 0 ? -1 : C->copies_issued + nth;
    return MOE_OK;
}
