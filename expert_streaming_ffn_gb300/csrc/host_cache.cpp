// Host-side expert cache manager and prefill pair grouping.
//
// The per-layer expert cache of expert-streaming inference ([P1] §6.2.2
// LayerExpertCache with lookup / allocate / touch, §6.2.3 ExpertCache, §8.3
// hit/miss flow) with the LFU policy of [P1] §2.3 and §9.5, and the LRU
// variant keyed by (layer, expert) of [P3] "缓存管理的是专家工作集", whose
// budget may be exceeded temporarily to protect the working set.
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
//
// Rules (the pages leave the details open; these are the readings the library
// implements):
//   * one lookup per distinct expert per step; distinct ids in ascending order;
//   * a hit increments the use count (LRU: stamps the step index) and pins its
//     slot for the rest of the step;
//   * a miss takes the lowest-index empty slot, else the unpinned slot with the
//     smallest count (LRU: the oldest stamp), ties to the lowest slot index;
//     the new entry starts at count 1 and is pinned;
//   * a miss with no unpinned slot left bypasses the cache (slot -1): it is
//     streamed to a transient buffer and not inserted.
#include "moe_internal.h"

#include <algorithm>
#include <new>

namespace moe {

HostCache::HostCache(int n_experts, int slots, int policy)
    : E(n_experts), S(slots), policy(policy), step_index(0), slot_expert(slots, -1), use_count(slots, 0),
      stamp(slots, 0), expert_slot(n_experts, -1), pinned(slots, 0), seen(n_experts, 0) {}

void HostCache::reset() {
    std::fill(slot_expert.begin(), slot_expert.end(), -1);
    std::fill(use_count.begin(), use_count.end(), 0u);
    std::fill(stamp.begin(), stamp.end(), 0);
    std::fill(expert_slot.begin(), expert_slot.end(), -1);
    step_index = 0;
}

int HostCache::pick_victim() const {
    int best = -1;
    for (int s = 0; s < S; ++s) {
        if (slot_expert[s] < 0) return s;  // empty slots first, lowest index
    }
    for (int s = 0; s < S; ++s) {
        if (pinned[s]) continue;
        if (best < 0) {
            best = s;
            continue;
        }
        bool better = policy == kLFU ? use_count[s] < use_count[best] : stamp[s] < stamp[best];
        if (better) best = s;
    }
    return best;
}

bool HostCache::step(const int32_t* ids, int n, StepResult& r) {
    r.distinct.clear();
    r.miss_experts.clear();
    r.miss_slots.clear();
    r.hits = r.bypass = 0;
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= E) return false;
    if (n <= 64) {
        r.distinct.assign(ids, ids + n);
        std::sort(r.distinct.begin(), r.distinct.end());
        r.distinct.erase(std::unique(r.distinct.begin(), r.distinct.end()), r.distinct.end());
    } else {
        // a prefill step's thousands of ids: mark, then list in ascending order
        for (int i = 0; i < n; ++i) seen[ids[i]] = 1;
        for (int e = 0; e < E; ++e)
            if (seen[e]) {
                r.distinct.push_back(e);
                seen[e] = 0;
            }
    }
    std::fill(pinned.begin(), pinned.end(), 0);
    // hits: touch and pin
    for (int e : r.distinct) {
        int s = expert_slot[e];
        if (s < 0) continue;
        if (policy == kLFU)
            ++use_count[s];
        else
            stamp[s] = step_index;
        pinned[s] = 1;
        ++r.hits;
    }
    // misses, ascending: allocate (evicting) or bypass
    for (int e : r.distinct) {
        if (expert_slot[e] >= 0) continue;
        int v = pick_victim();
        r.miss_experts.push_back(e);
        r.miss_slots.push_back(v);
        if (v < 0) {
            ++r.bypass;
            continue;
        }
        if (slot_expert[v] >= 0) expert_slot[slot_expert[v]] = -1;
        slot_expert[v] = e;
        expert_slot[e] = v;
        use_count[v] = 1;
        stamp[v] = step_index;
        pinned[v] = 1;
    }
    ++step_index;
    return true;
}

void HostCache::evict(int slot) {
    if (slot < 0 || slot >= S) return;
    if (slot_expert[slot] >= 0) expert_slot[slot_expert[slot]] = -1;
    slot_expert[slot] = -1;
    use_count[slot] = 0;
    stamp[slot] = 0;
}

int HostCache::slot_of(int expert) const { return expert_slot[expert]; }

// Stable grouping of (token, rank) pairs by expert: a counting sort.
void group_pairs(const int32_t* ids, int n_pairs, int n_experts, int32_t* offsets, int32_t* perm) {
    std::fill(offsets, offsets + n_experts + 1, 0);
    for (int p = 0; p < n_pairs; ++p) ++offsets[ids[p] + 1];
    for (int e = 0; e < n_experts; ++e) offsets[e + 1] += offsets[e];
    std::vector<int32_t> cursor(offsets, offsets + n_experts);
    for (int p = 0; p < n_pairs; ++p) perm[cursor[ids[p]]++] = p;
}

}  // namespace moe

using moe::set_error;

struct moe_host_cache {
    moe::HostCache cache;
    moe::StepResult last;
    moe_host_cache(int E, int S, int policy) : cache(E, S, policy) {}
};

extern "C" moe_status moe_host_cache_create(int32_t n_experts, int32_t slots, int32_t policy, moe_host_cache** out) {
    if (!out || n_experts < 1 || n_experts > moe::kMaxExperts || slots < 1 || slots > n_experts ||
        (policy != moe::kLFU && policy != moe::kLRU))
        return set_error(MOE_EINVAL, "moe_host_cache_create: bad arguments");
    moe_host_cache* c = new (std::nothrow) moe_host_cache(n_experts, slots, policy);
    if (!c) return set_error(MOE_ENOMEM, "moe_host_cache_create: out of host memory");
    *out = c;
    return MOE_OK;
}

extern "C" moe_status moe_host_cache_step(moe_host_cache* c, const int32_t* ids, int32_t n_ids, int32_t* slot_of,
                                          int32_t* miss_experts, int32_t* miss_slots, int32_t* n_miss,
                                          int32_t* n_hit, int32_t* n_bypass) {
    if (!c || (!ids && n_ids > 0) || n_ids < 0) return set_error(MOE_EINVAL, "moe_host_cache_step: bad arguments");
    if (!c->cache.step(ids, n_ids, c->last)) return set_error(MOE_EINVAL, "moe_host_cache_step: expert id out of range");
    const moe::StepResult& r = c->last;
    if (slot_of)
        for (int i = 0; i < n_ids; ++i) slot_of[i] = c->cache.slot_of(ids[i]);
    for (size_t i = 0; i < r.miss_experts.size(); ++i) {
        if (miss_experts) miss_experts[i] = r.miss_experts[i];
        if (miss_slots) miss_slots[i] = r.miss_slots[i];
    }
    if (n_miss) *n_miss = (int32_t)r.miss_experts.size();
    if (n_hit) *n_hit = r.hits;
    if (n_bypass) *n_bypass = r.bypass;
    return MOE_OK;
}

extern "C" moe_status moe_host_cache_dump(const moe_host_cache* c, int32_t* slot_expert, uint32_t* counts) {
    if (!c) return set_error(MOE_EINVAL, "moe_host_cache_dump: NULL cache");
    for (int s = 0; s < c->cache.S; ++s) {
        if (slot_expert) slot_expert[s] = c->cache.slot_expert[s];
        if (counts) counts[s] = c->cache.use_count[s];
    }
    return MOE_OK;
}

extern "C" void moe_host_cache_destroy(moe_host_cache* c) { delete c; }

extern "C" moe_status moe_group_pairs(const int32_t* ids, int32_t n_pairs, int32_t n_experts, int32_t* offsets,
                                      int32_t* perm) {
    if (n_pairs < 0 || n_experts < 1 || !offsets || (n_pairs > 0 && (!ids || !perm)))
        return set_error(MOE_EINVAL, "moe_group_pairs: bad arguments");
    for (int p = 0; p < n_pairs; ++p)
        if (ids[p] < 0 || ids[p] >= n_experts) return set_error(MOE_EINVAL, "moe_group_pairs: id out of range");
    moe::group_pairs(ids, n_pairs, n_experts, offsets, perm);
    return MOE_OK;
}
