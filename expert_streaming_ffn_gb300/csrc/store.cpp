// The storage tier of the expert stream: one file per layer holding its
// routed experts, read on demand by a pool of threads into a small host tier.
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//
// The pages' system streams the routed experts from SSD: the CPU reads the
// experts the next layer needs with pread while the accelerator computes
// ([P1] §2.3 "流式部分" and "流水线"), through an asynchronous reader with
// request / wait_all ([P1] §6.2.2 AsyncExpertReader). Its I/O notes ([P1]
// §9.2) ask for one file per layer with an [offset, size] per expert (item
// 2), readahead of the experts that routing history says are likely (item
// 3), and O_DIRECT, since an expert read once is not worth the page cache
// (item 4).
//
// Here the file holds each expert as the library's device blob (the layout
// the slots use), so a read lands bytes that go to HBM unchanged:
//   [0, 4096)               header (StoreHeader, zero padded)
//   4096 + e * stride       expert e: expert_blob_bytes bytes, zero padded to
//                           stride = the blob size rounded up to 4096
// Every read is one pread of `stride` bytes at a 4096-aligned offset into a
// 4096-aligned buffer, which O_DIRECT requires; with a read chunk set
// (moe_store_set_read_chunk, a multiple of 4096), one pread per chunk of it,
// taken by as many readers as are free, and the entry is ready when the last
// piece lands.
//
// The host tier is H entries of `stride` bytes. An entry is empty, being
// read, ready, or failed. The store counts every expert's fetches (its
// history, kept across evictions). A fetch of an expert that is not in the
// tier takes an empty entry, else, among the entries nobody pins and nobody
// is reading, the one whose expert has the fewest fetches (ties: the least
// recently used), and queues its read. Readahead takes an entry only if its
// expert has no more fetches than the expert read ahead, never one read ahead
// and not yet fetched, and its reads wait behind every read a fetch needs.
// A fetch that finds a failed read it did not ask for (readahead's) reads
// once more; a read that fails for the fetch that asked for it is reported
// (MOE_EIO) and its entry freed. A fetched entry stays pinned until released:
// the layer releases it once the host-to-device copy that reads it has
// finished.
//
// Reads run on the reader threads. The tier's table is guarded by one mutex;
// a reader writes only the piece of the entry's buffer it was given, outside
// the mutex, and no one else touches that buffer until the entry is ready.
#include <errno.h>
#include <fcntl.h>
#include <stdlib.h>
#include <string.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kAlign = 4096;
constexpr uint32_t kVersion = 1;
const char kMagic[8] = {'M', 'O', 'E', 'X', 'P', 'R', 'T', 'S'};

struct StoreHeader {
    char magic[8];
    uint32_t version;
    uint32_t header_bytes;
    moe_shapes shapes;
    uint32_t pad;
    uint64_t ebytes, stride, data_offset;
};
static_assert(sizeof(StoreHeader) <= kAlign, "the header fits its block");

enum { kEmpty = 0, kReading = 1, kReady = 2, kFailed = 3 };

struct Entry {
    int expert = -1;
    int state = kEmpty;
    int pins = 0;
    uint64_t used = 0;        // tick of the last fetch (or of the read's start)
    bool predicted = false;   // read by a readahead request and not fetched since
    bool demand = false;      // queued ahead for a fetch that follows (not a tier hit)
    int err = 0;              // errno of a failed read (the first failed piece's)
    int pending = 0;          // pieces of the read not yet finished
    size_t piece = 0;         // bytes per piece of the read in flight
    bool started = false;     // a piece has started (t0 is set)
    std::chrono::steady_clock::time_point t0;
};

// One piece of an expert's read: bytes [piece * chunk, ...) of entry `entry`.
struct Job {
    int entry;
    int piece;
};

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

double us_between(std::chrono::steady_clock::time_point a, std::chrono::steady_clock::time_point b) {
    return std::chrono::duration<double, std::micro>(b - a).count();
}

}  // namespace
}  // namespace moe

struct moe_expert_store {
    std::string path;
    int fd = -1;
    bool direct = false;
    moe_shapes sh{};
    int E = 0, H = 0;
    size_t ebytes = 0, stride = 0, data_offset = 0;
    uint8_t* buf = nullptr;  // H * stride, 4096-aligned
    std::vector<moe::Entry> ent;
    std::vector<int> where;  // expert -> entry, -1 if not in the tier
    std::mutex mu;
    std::condition_variable cv_job, cv_done;
    std::deque<moe::Job> jobs;     // pieces to read for fetches, in request order
    std::deque<moe::Job> jobs_ra;  // pieces to read ahead, taken only when `jobs` is empty
    size_t chunk = 0;              // bytes per piece of a read (a multiple of 4096); 0 = whole expert
    std::vector<uint32_t> freq;  // fetches per expert
    std::vector<uint8_t> keep;   // experts whose entries must not be taken (during one readahead call)
    std::vector<std::thread> readers;
    bool stop = false;
    uint64_t tick = 0;
    bool attached = false;  // a layer streams from this store
    moe_store_stats st{};
};

namespace moe {
namespace {

void reader_loop(moe_expert_store* s) {
    for (;;) {
        Job job;
        int e;
        size_t begin, len;
        {
            std::unique_lock<std::mutex> lk(s->mu);
            s->cv_job.wait(lk, [&] { return s->stop || !s->jobs.empty() || !s->jobs_ra.empty(); });
            std::deque<Job>& q = !s->jobs.empty() ? s->jobs : s->jobs_ra;
            if (q.empty()) return;  // stop, and nothing left to read
            job = q.front();
            q.pop_front();
            Entry& en = s->ent[(size_t)job.entry];
            e = en.expert;
            begin = (size_t)job.piece * en.piece;
            len = std::min(en.piece, s->stride - begin);
            if (!en.started) {
                en.started = true;
                en.t0 = std::chrono::steady_clock::now();
            }
        }
        uint8_t* dst = s->buf + (size_t)job.entry * s->stride + begin;
        const off_t off = (off_t)(s->data_offset + (size_t)e * s->stride + begin);
        size_t done = 0;
        int err = 0;
        while (done < len) {
            const ssize_t r = pread(s->fd, dst + done, len - done, off + (off_t)done);
            if (r < 0) {
                if (errno == EINTR) continue;
                err = errno;
                break;
            }
            if (r == 0) {
                err = EIO;  // the file ends inside the expert
                break;
            }
            done += (size_t)r;
        }
        bool finished = false;
        {
            std::lock_guard<std::mutex> g(s->mu);
            Entry& en = s->ent[(size_t)job.entry];
            if (err && !en.err) en.err = err;
            if (--en.pending == 0) {
                finished = true;
                en.state = en.err ? kFailed : kReady;
                s->st.reads += 1;
                s->st.read_us += us_between(en.t0, std::chrono::steady_clock::now());
                if (!en.err) s->st.bytes_read += s->stride;
                else s->st.read_errors += 1;
            }
        }
        if (finished) s->cv_done.notify_all();
    }
}

// Queue the read of entry i (state already kReading) as its pieces. Caller
// holds the mutex.
void queue_read(moe_expert_store* s, int i, bool predicted) {
    Entry& en = s->ent[(size_t)i];
    en.piece = s->chunk ? s->chunk : s->stride;
    const int pieces = (int)((s->stride + en.piece - 1) / en.piece);
    en.pending = pieces;
    en.started = false;
    en.err = 0;
    std::deque<Job>& q = predicted ? s->jobs_ra : s->jobs;
    for (int p = 0; p < pieces; ++p) q.push_back(Job{i, p});
    if (pieces == 1) s->cv_job.notify_one();
    else s->cv_job.notify_all();
}

// An entry to (re)use: the lowest empty one, else, among the ready or failed
// entries nobody pins, the one whose expert has the fewest fetches, ties to
// the least recently used. For readahead of expert `ahead` (>= 0), entries
// read ahead and not yet fetched are kept, and an entry whose expert has more
// fetches than `ahead` is not taken; with keep_predicted, entries read ahead
// and not yet fetched are kept too. Entries of experts marked in `keep` are
// never taken. -1 if none. Caller holds the mutex.
int pick_entry(const moe_expert_store* s, int ahead, bool keep_predicted) {
    int best = -1;
    for (int i = 0; i < s->H; ++i) {
        const Entry& en = s->ent[(size_t)i];
        if (en.state == kEmpty) return i;
        if (en.state == kReading || en.pins > 0) continue;
        if ((ahead >= 0 || keep_predicted) && en.predicted) continue;
        if (s->keep[(size_t)en.expert]) continue;
        if (best < 0) {
            best = i;
            continue;
        }
        const Entry& b = s->ent[(size_t)best];
        const uint32_t fi = s->freq[(size_t)en.expert], fb = s->freq[(size_t)b.expert];
        if (fi < fb || (fi == fb && en.used < b.used)) best = i;
    }
    if (best >= 0 && ahead >= 0 && s->freq[(size_t)s->ent[(size_t)best].expert] > s->freq[(size_t)ahead]) return -1;
    return best;
}

// Give entry i to expert e and queue its read. Caller holds the mutex.
void assign(moe_expert_store* s, int i, int e, bool predicted) {
    Entry& en = s->ent[(size_t)i];
    if (en.expert >= 0) s->where[(size_t)en.expert] = -1;
    en.expert = e;
    en.state = kReading;
    en.pins = 0;
    en.used = ++s->tick;
    en.predicted = predicted;
    en.demand = !predicted;
    s->where[(size_t)e] = i;
    queue_read(s, i, predicted);
}

bool any_reading(const moe_expert_store* s) {
    for (const Entry& en : s->ent)
        if (en.state == kReading) return true;
    return false;
}

}  // namespace

moe_status store_acquire(moe_expert_store* s, int e, const uint8_t** out) {
    std::unique_lock<std::mutex> lk(s->mu);
    bool queued = false;
    for (;;) {
        const int i = s->where[(size_t)e];
        if (i >= 0) {
            Entry& en = s->ent[(size_t)i];
            if (en.state == kReady) {
                if (!queued && !en.demand) s->st.tier_hits += 1;
                if (en.predicted) s->st.prefetch_used += 1;
                en.predicted = false;
                en.demand = false;
                en.pins += 1;
                s->st.fetches += 1;
                s->freq[(size_t)e] += 1;
                en.used = ++s->tick;
                *out = s->buf + (size_t)i * s->stride;
                return MOE_OK;
            }
            if (en.state == kFailed && !queued) {
                // a read queued earlier (readahead) failed: read again for this fetch
                en.state = kReading;
                en.predicted = false;
                queue_read(s, i, false);
                queued = true;
                continue;
            }
            if (en.state == kFailed) {
                s->st.fetches += 1;
                const int err = en.err;
                en.state = kEmpty;
                en.expert = -1;
                en.predicted = false;
                s->where[(size_t)e] = -1;
                return set_error(MOE_EIO, "read of expert %d from %s failed: %s", e, s->path.c_str(), strerror(err));
            }
            // being read: wait for it
            const auto t0 = std::chrono::steady_clock::now();
            s->cv_done.wait(lk);
            s->st.wait_us += us_between(t0, std::chrono::steady_clock::now());
            continue;
        }
        const int v = pick_entry(s, -1, false);
        if (v >= 0) {
            assign(s, v, e, false);
            queued = true;
            continue;
        }
        if (any_reading(s)) {  // a read in flight will free an entry
            const auto t0 = std::chrono::steady_clock::now();
            s->cv_done.wait(lk);
            s->st.wait_us += us_between(t0, std::chrono::steady_clock::now());
            continue;
        }
        return set_error(MOE_EBUSY, "every one of the %d host-tier entries is pinned", s->H);
    }
}

moe_status store_release(moe_expert_store* s, int e) {
    std::lock_guard<std::mutex> g(s->mu);
    const int i = s->where[(size_t)e];
    if (i < 0 || s->ent[(size_t)i].pins < 1) return set_error(MOE_EINVAL, "expert %d is not pinned in the tier", e);
    s->ent[(size_t)i].pins -= 1;
    return MOE_OK;
}

int store_readahead(moe_expert_store* s, const int32_t* experts, int n, bool predicted) {
    std::lock_guard<std::mutex> g(s->mu);
    int queued = 0;
    // reads for fetches that follow must not displace one another (or an
    // expert of the list already in the tier)
    if (!predicted)
        for (int j = 0; j < n; ++j)
            if (experts[j] >= 0 && experts[j] < s->E) s->keep[(size_t)experts[j]] = 1;
    for (int j = 0; j < n; ++j) {
        const int e = experts[j];
        if (e < 0 || e >= s->E || s->where[(size_t)e] >= 0) continue;
        const int v = pick_entry(s, predicted ? e : -1, true);
        if (v < 0) {
            if (predicted) continue;  // the next expert may still find an entry it is worth
            break;
        }
        assign(s, v, e, predicted);
        ++queued;
    }
    if (!predicted)
        for (int j = 0; j < n; ++j)
            if (experts[j] >= 0 && experts[j] < s->E) s->keep[(size_t)experts[j]] = 0;
    if (predicted) s->st.prefetch_reads += (uint64_t)queued;
    return queued;
}

bool store_ready(moe_expert_store* s, int e) {
    std::lock_guard<std::mutex> g(s->mu);
    const int i = s->where[(size_t)e];
    return i >= 0 && s->ent[(size_t)i].state == kReady;
}

bool store_contains(moe_expert_store* s, int e) {
    std::lock_guard<std::mutex> g(s->mu);
    const int i = s->where[(size_t)e];
    return i >= 0 && (s->ent[(size_t)i].state == kReady || s->ent[(size_t)i].state == kReading);
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_store_expert_stride(const moe_shapes* s) {
    if (!s) return 0;
    return round_up(expert_blob_bytes(s->d_model, s->d_ff), kAlign);
}

extern "C" moe_status moe_store_write(const char* path, const moe_shapes* s, const moe_host_weights* w) {
    if (!path || !w) return set_error(MOE_EINVAL, "moe_store_write: path or weights is NULL");
    moe_status st = check_shapes(s);
    if (st != MOE_OK) return st;
    for (const moe_qmatrix* m : {&w->gate, &w->up, &w->down})
        if (!m->codes || !m->scale || !m->bias) return set_error(MOE_EINVAL, "moe_store_write: a routed weight is NULL");
    const int d = s->d_model, I = s->d_ff, E = s->n_experts;
    StoreHeader h{};
    memcpy(h.magic, kMagic, sizeof(kMagic));
    h.version = kVersion;
    h.header_bytes = (uint32_t)kAlign;
    h.shapes = *s;
    h.ebytes = expert_blob_bytes(d, I);
    h.stride = round_up(h.ebytes, kAlign);
    h.data_offset = kAlign;
    const int fd = open(path, O_WRONLY | O_CREAT | O_TRUNC, 0644);
    if (fd < 0) return set_error(MOE_EIO, "moe_store_write: cannot create %s: %s", path, strerror(errno));
    std::vector<uint8_t> head(kAlign, 0);
    memcpy(head.data(), &h, sizeof(h));
    std::atomic<int> err{0};
    auto put = [&](const uint8_t* p, size_t n, off_t off) {
        size_t done = 0;
        while (done < n) {
            const ssize_t r = pwrite(fd, p + done, n - done, off + (off_t)done);
            if (r < 0 && errno == EINTR) continue;
            if (r <= 0) {
                int zero = 0;
                err.compare_exchange_strong(zero, r < 0 ? errno : EIO);
                return;
            }
            done += (size_t)r;
        }
    };
    put(head.data(), head.size(), 0);
    // routed experts, one padded blob each, repacked by a few threads
    const size_t gc = (size_t)I * (d / 2), gs = (size_t)I * (d / 64), dc = (size_t)d * (I / 2), ds = (size_t)d * (I / 64);
    const unsigned nth = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
    std::vector<std::thread> pool;
    for (unsigned t = 0; t < nth; ++t)
        pool.emplace_back([&, t] {
            std::vector<uint8_t> blob(h.stride, 0);
            for (int e = (int)t; e < E && err.load() == 0; e += (int)nth) {
                moe_qmatrix g{w->gate.codes + e * gc, w->gate.scale + e * gs, w->gate.bias + e * gs};
                moe_qmatrix u{w->up.codes + e * gc, w->up.scale + e * gs, w->up.bias + e * gs};
                moe_qmatrix dn{w->down.codes + e * dc, w->down.scale + e * ds, w->down.bias + e * ds};
                repack_qmatrix(g, I, d, blob.data());
                repack_qmatrix(u, I, d, blob.data() + qmat_bytes(I, d));
                repack_down(dn, d, I, blob.data() + 2 * qmat_bytes(I, d));
                put(blob.data(), blob.size(), (off_t)(h.data_offset + (size_t)e * h.stride));
            }
        });
    for (auto& th : pool) th.join();
    const int rc = close(fd);
    if (err.load() != 0)
        return set_error(MOE_EIO, "moe_store_write: writing %s failed: %s", path, strerror(err.load()));
    if (rc != 0) return set_error(MOE_EIO, "moe_store_write: closing %s failed: %s", path, strerror(errno));
    return MOE_OK;
}

extern "C" moe_status moe_store_open(const char* path, const moe_shapes* s, int32_t host_slots, int32_t readers,
                                     int32_t flags, moe_expert_store** out) {
    if (!path || !out) return set_error(MOE_EINVAL, "moe_store_open: path or out is NULL");
    moe_status st = check_shapes(s);
    if (st != MOE_OK) return st;
    if (host_slots < 1 || host_slots > s->n_experts)
        return set_error(MOE_EINVAL, "host_slots %d out of [1, n_experts]", host_slots);
    if (readers < 1 || readers > 64) return set_error(MOE_EINVAL, "readers %d out of [1, 64]", readers);
    if (flags & ~MOE_STORE_DIRECT) return set_error(MOE_EINVAL, "unknown flags 0x%x", (unsigned)flags);
    bool direct = (flags & MOE_STORE_DIRECT) != 0;
    int fd = -1;
#ifdef O_DIRECT
    if (direct) {
        fd = open(path, O_RDONLY | O_DIRECT);
        if (fd < 0 && errno == EINVAL) direct = false;  // the file system has no direct I/O
    }
#else
    direct = false;
#endif
    if (fd < 0) fd = open(path, O_RDONLY);
    if (fd < 0) return set_error(MOE_EIO, "moe_store_open: cannot open %s: %s", path, strerror(errno));
    auto fail = [&](moe_status code, const char* fmt, auto... a) {
        close(fd);
        return set_error(code, fmt, a...);
    };
    // the header, through an aligned buffer (direct I/O needs one)
    void* hb = nullptr;
    if (posix_memalign(&hb, kAlign, kAlign) != 0) return fail(MOE_ENOMEM, "moe_store_open: out of host memory");
    const ssize_t got = pread(fd, hb, kAlign, 0);
    StoreHeader h{};
    if (got == (ssize_t)kAlign) memcpy(&h, hb, sizeof(h));
    free(hb);
    if (got != (ssize_t)kAlign) return fail(MOE_EIO, "moe_store_open: %s: short or failed header read", path);
    if (memcmp(h.magic, kMagic, sizeof(kMagic)) != 0 || h.version != kVersion)
        return fail(MOE_EINVAL, "moe_store_open: %s is not an expert file of this library", path);
    if (memcmp(&h.shapes, s, sizeof(moe_shapes)) != 0)
        return fail(MOE_EINVAL, "moe_store_open: %s holds other shapes (d %d, E %d, I %d)", path, h.shapes.d_model,
                    h.shapes.n_experts, h.shapes.d_ff);
    const size_t eb = expert_blob_bytes(s->d_model, s->d_ff);
    if (h.ebytes != eb || h.stride != round_up(eb, kAlign) || h.data_offset != kAlign)
        return fail(MOE_EINVAL, "moe_store_open: %s has an inconsistent layout", path);
    struct stat sb{};
    if (fstat(fd, &sb) != 0 || (uint64_t)sb.st_size < h.data_offset + (uint64_t)s->n_experts * h.stride)
        return fail(MOE_EINVAL, "moe_store_open: %s is shorter than its %d experts", path, s->n_experts);
    moe_expert_store* S = new (std::nothrow) moe_expert_store();
    if (!S) return fail(MOE_ENOMEM, "moe_store_open: out of host memory");
    void* buf = nullptr;
    if (posix_memalign(&buf, kAlign, (size_t)host_slots * h.stride) != 0) {
        delete S;
        return fail(MOE_ENOMEM, "moe_store_open: cannot allocate %d host-tier entries of %zu B", host_slots,
                    (size_t)h.stride);
    }
    S->path = path;
    S->fd = fd;
    S->direct = direct;
    S->sh = *s;
    S->E = s->n_experts;
    S->H = host_slots;
    S->ebytes = eb;
    S->stride = h.stride;
    S->data_offset = h.data_offset;
    S->buf = (uint8_t*)buf;
    S->ent.assign((size_t)host_slots, Entry{});
    S->where.assign((size_t)s->n_experts, -1);
    S->freq.assign((size_t)s->n_experts, 0);
    S->keep.assign((size_t)s->n_experts, 0);
    S->st.direct = direct ? 1 : 0;
    S->st.host_slots = host_slots;
    S->st.readers = readers;
    try {
        for (int r = 0; r < readers; ++r) S->readers.emplace_back(reader_loop, S);
    } catch (...) {
        moe_store_close(S);
        return set_error(MOE_ENOMEM, "moe_store_open: cannot start %d reader threads", readers);
    }
    *out = S;
    return MOE_OK;
}

extern "C" moe_status moe_store_close(moe_expert_store* S) {
    if (!S) return MOE_OK;
    {
        std::lock_guard<std::mutex> g(S->mu);
        if (S->attached) return set_error(MOE_ESTATE, "moe_store_close: a layer still streams from this store");
        S->stop = true;
    }
    S->cv_job.notify_all();
    for (auto& th : S->readers) th.join();
    if (S->fd >= 0) close(S->fd);
    free(S->buf);
    delete S;
    return MOE_OK;
}

extern "C" moe_status moe_store_fetch(moe_expert_store* S, int32_t expert, const uint8_t** out) {
    if (!S || !out) return set_error(MOE_EINVAL, "moe_store_fetch: store or out is NULL");
    if (expert < 0 || expert >= S->E) return set_error(MOE_EINVAL, "expert %d out of [0, %d)", expert, S->E);
    return store_acquire(S, expert, out);
}

extern "C" moe_status moe_store_release(moe_expert_store* S, int32_t expert) {
    if (!S) return set_error(MOE_EINVAL, "moe_store_release: store is NULL");
    if (expert < 0 || expert >= S->E) return set_error(MOE_EINVAL, "expert %d out of [0, %d)", expert, S->E);
    return store_release(S, expert);
}

extern "C" moe_status moe_store_prefetch(moe_expert_store* S, const int32_t* experts, int32_t n, int32_t* queued) {
    if (!S || (!experts && n > 0) || n < 0) return set_error(MOE_EINVAL, "moe_store_prefetch: bad arguments");
    const int q = store_readahead(S, experts, n, true);
    if (queued) *queued = q;
    return MOE_OK;
}

extern "C" moe_status moe_store_set_read_chunk(moe_expert_store* S, size_t bytes) {
    if (!S) return set_error(MOE_EINVAL, "moe_store_set_read_chunk: store is NULL");
    if (bytes % kAlign != 0) return set_error(MOE_EINVAL, "read chunk %zu is not a multiple of 4096", bytes);
    std::lock_guard<std::mutex> g(S->mu);
    S->chunk = bytes >= S->stride ? 0 : bytes;
    return MOE_OK;
}

extern "C" moe_status moe_store_wait_idle(moe_expert_store* S) {
    if (!S) return set_error(MOE_EINVAL, "moe_store_wait_idle: store is NULL");
    std::unique_lock<std::mutex> lk(S->mu);
    S->cv_done.wait(lk, [&] { return S->jobs.empty() && S->jobs_ra.empty() && !any_reading(S); });
    return MOE_OK;
}

extern "C" moe_status moe_store_get_stats(moe_expert_store* S, moe_store_stats* out) {
    if (!S || !out) return set_error(MOE_EINVAL, "moe_store_get_stats: bad arguments");
    std::lock_guard<std::mutex> g(S->mu);
    *out = S->st;
    return MOE_OK;
}

extern "C" moe_status moe_store_reset_stats(moe_expert_store* S) {
    if (!S) return set_error(MOE_EINVAL, "moe_store_reset_stats: store is NULL");
    std::lock_guard<std::mutex> g(S->mu);
    const moe_store_stats keep = S->st;
    S->st = moe_store_stats{};
    S->st.direct = keep.direct;
    S->st.host_slots = keep.host_slots;
    S->st.readers = keep.readers;
    return MOE_OK;
}

extern "C" moe_status moe_store_tier(moe_expert_store* S, int32_t* entry_expert, int32_t* entry_state) {
    if (!S) return set_error(MOE_EINVAL, "moe_store_tier: store is NULL");
    std::lock_guard<std::mutex> g(S->mu);
    for (int i = 0; i < S->H; ++i) {
        if (entry_expert) entry_expert[i] = S->ent[(size_t)i].expert;
        if (entry_state) entry_state[i] = S->ent[(size_t)i].state;
    }
    return MOE_OK;
}

namespace moe {

// The layer side (api.cu) pins the tier's buffer for DMA and marks the store
// attached; these give it the pieces it needs.
uint8_t* store_buffer(moe_expert_store* s, size_t* bytes) {
    *bytes = (size_t)s->H * s->stride;
    return s->buf;
}
int store_host_slots(const moe_expert_store* s) { return s->H; }
const moe_shapes& store_shapes(const moe_expert_store* s) { return s->sh; }
bool store_attach(moe_expert_store* s, bool on) {
    std::lock_guard<std::mutex> g(s->mu);
    if (on && s->attached) return false;
    s->attached = on;
    return true;
}

}  // namespace moe
