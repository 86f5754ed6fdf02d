// A check of the expert store (csrc/store.cpp) and the host cache manager
// (csrc/host_cache.cpp) under the sanitizers: several
// threads fetch, release and read ahead at random against one store, while
// its reader threads fill the tier, and every fetched expert is compared with
// the file's bytes. Built with g++ -fsanitize=thread, and with
// -fsanitize=address,undefined, by test_store_sanitizers.py together with
// store.cpp and host_cache.cpp alone, so the few library functions they call
// are defined here (the file is written by the library beforehand; nothing here repacks
// weights).
//
//   store_sanitize <expert file> <read chunk bytes>
#include <fcntl.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include <atomic>
#include <random>
#include <thread>
#include <vector>

#include "../expert_streaming_ffn_gb300/csrc/moe_internal.h"

namespace moe {
static thread_local char g_msg[512];
moe_status set_error(moe_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}
moe_status check_shapes(const moe_shapes* s) { return s ? MOE_OK : MOE_EINVAL; }
void repack_qmatrix(const moe_qmatrix&, int, int, uint8_t*) { abort(); }
void repack_down(const moe_qmatrix&, int, int, uint8_t*) { abort(); }
}  // namespace moe

// The host cache manager (host_cache.cpp, built in as well) on random steps
// of up to 512 ids under both policies, checking the invariants every step
// must keep: each id's slot holds that id (or it bypassed), a slot holds at
// most one expert, and hits + misses count the distinct ids.
static int host_cache_check() {
    std::mt19937 rng(7);
    for (int policy = 0; policy < 2; ++policy)
        for (int S : {1, 3, 16, 64}) {
            const int E = 256;
            moe_host_cache* c = nullptr;
            if (moe_host_cache_create(E, S, policy, &c) != MOE_OK) return 10;
            std::vector<int32_t> ids(512), slot_of(512), me(512), ms(512), se((size_t)S), off(E + 1), perm(512);
            std::vector<uint32_t> cnt((size_t)S);
            for (int step = 0; step < 200; ++step) {
                const int n = 1 + (int)(rng() % 512u);
                for (int i = 0; i < n; ++i) ids[(size_t)i] = (int32_t)(rng() % (step % 3 ? 24u : 256u));
                int32_t nm = 0, nh = 0, nb = 0;
                if (moe_host_cache_step(c, ids.data(), n, slot_of.data(), me.data(), ms.data(), &nm, &nh, &nb) !=
                    MOE_OK)
                    return 11;
                if (moe_host_cache_dump(c, se.data(), cnt.data()) != MOE_OK) return 12;
                std::vector<int> seen(E, 0);
                int distinct = 0;
                for (int i = 0; i < n; ++i) {
                    distinct += !seen[(size_t)ids[(size_t)i]];
                    seen[(size_t)ids[(size_t)i]] = 1;
                    const int32_t sl = slot_of[(size_t)i];
                    if (sl >= S || (sl >= 0 && se[(size_t)sl] != ids[(size_t)i])) return 13;
                }
                if (nh + nm != distinct || nb > nm) return 14;
                std::vector<int> held(E, 0);
                for (int t = 0; t < S; ++t)
                    if (se[(size_t)t] >= 0 && held[(size_t)se[(size_t)t]]++) return 15;
                if (moe_group_pairs(ids.data(), n, E, off.data(), perm.data()) != MOE_OK || off[E] != n) return 16;
                for (int e = 0; e < E; ++e)
                    for (int q = off[(size_t)e]; q < off[(size_t)e + 1]; ++q)
                        if (ids[(size_t)perm[(size_t)q]] != e || (q > off[(size_t)e] && perm[(size_t)q] <= perm[(size_t)q - 1]))
                            return 17;
            }
            moe_host_cache_destroy(c);
        }
    return 0;
}

int main(int argc, char** argv) {
    if (argc < 3) return 2;
    if (const int hc = host_cache_check()) {
        printf("host cache check failed (%d)\n", hc);
        return 1;
    }
    const moe_shapes sh = {512, 8, 2, 192, 512, 0};
    const size_t eb = moe::expert_blob_bytes(sh.d_model, sh.d_ff);
    const size_t stride = moe_store_expert_stride(&sh);
    // the file's bytes, read plainly, to check every fetch against
    std::vector<std::vector<uint8_t>> want((size_t)sh.n_experts, std::vector<uint8_t>(eb));
    const int fd = open(argv[1], O_RDONLY);
    if (fd < 0) return 3;
    for (int e = 0; e < sh.n_experts; ++e)
        if (pread(fd, want[(size_t)e].data(), eb, (off_t)(4096 + (size_t)e * stride)) != (ssize_t)eb) return 4;
    close(fd);
    moe_expert_store* st = nullptr;
    if (moe_store_open(argv[1], &sh, 3, 4, 0, &st) != MOE_OK) return 5;
    if (moe_store_set_read_chunk(st, (size_t)atol(argv[2])) != MOE_OK) return 6;
    std::atomic<int> bad{0}, busy{0}, ok{0};
    std::vector<std::thread> th;
    for (int t = 0; t < 4; ++t)
        th.emplace_back([&, t] {
            std::mt19937 rng(1234u + (unsigned)t);
            for (int i = 0; i < 400; ++i) {
                const int e = (int)(rng() % (unsigned)sh.n_experts);
                if (rng() % 4 == 0) {
                    int32_t ask[2] = {e, (int32_t)(rng() % (unsigned)sh.n_experts)};
                    int32_t q = 0;
                    if (moe_store_prefetch(st, ask, 2, &q) != MOE_OK) ++bad;
                    continue;
                }
                const uint8_t* p = nullptr;
                const moe_status s = moe_store_fetch(st, e, &p);
                if (s == MOE_EBUSY) {
                    ++busy;
                    continue;
                }
                if (s != MOE_OK || memcmp(p, want[(size_t)e].data(), eb) != 0) ++bad;
                ++ok;
                if (moe_store_release(st, e) != MOE_OK) ++bad;
            }
        });
    for (auto& x : th) x.join();
    if (moe_store_wait_idle(st) != MOE_OK) ++bad;
    moe_store_stats ss{};
    moe_store_get_stats(st, &ss);
    if (moe_store_close(st) != MOE_OK) ++bad;
    printf("ok %d busy %d bad %d reads %llu\n", ok.load(), busy.load(), bad.load(), (unsigned long long)ss.reads);
    return bad.load() == 0 && ss.fetches == (uint64_t)ok.load() ? 0 : 1;
}
