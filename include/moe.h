/*
 * libmoe: the expert-streaming MoE layer on one NVIDIA GB300 (sm_103a).
 *
 * One MoE layer of expert-streaming inference: an 8-bit router with top-k and
 * renormalised gates, a per-layer expert cache whose slots live in HBM and
 * whose misses are streamed from pinned host memory, int4-affine expert FFNs,
 * an always-resident shared expert and the gate-weighted combine.
 *
 * Pages cited (by title and section):
 *   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
 *   [P3] "BigMoeOnEdge：端侧 MoE 专家流式推理原理与实测"
 *
 * Conventions for every call:
 *   - Return value: a moe_status. No call throws or aborts. On failure the
 *     outputs are unspecified and moe_last_error() (thread-local) describes
 *     the cause. CUDA errors map to MOE_ECUDA.
 *   - Pointers marked "device" must be device memory of the layer's device;
 *     pointers marked "host" are ordinary host memory (pageable is fine).
 *     The caller owns every pointer it passes; the library never frees them
 *     and keeps none beyond the call, except where a call says otherwise.
 *   - stream: a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Device work is enqueued on it; calls that must read device
 *     results on the host (moe_forward) synchronise internally on events.
 *   - One host thread at a time per moe_layer. Different layers may be used
 *     from different threads.
 *   - Numeric formats: bf16 = bfloat16 bit patterns, f16 = IEEE binary16 bit
 *     patterns, both as uint16_t.
 *   - Token rows x (bf16, device) must start on a 16-byte boundary (the
 *     kernels read them 16 bytes at a time); a misaligned x gives MOE_EINVAL.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_EINVAL = 1,   /* bad argument: shape, pointer, id out of range */
    MOE_ENOMEM = 2,   /* device or pinned host allocation failed */
    MOE_ECUDA = 3,    /* a CUDA runtime call failed */
    MOE_ECOPY = 4,    /* a miss copy failed; the slot is left empty */
    MOE_ETIMEOUT = 5, /* a bounded device wait expired */
    MOE_ESTATE = 6,   /* call out of order (e.g. forward before set_weights) */
    MOE_EBUSY = 7,    /* every host-tier entry of an expert store is pinned */
    MOE_EIO = 8       /* a file of the storage tier could not be read or written */
} moe_status;

typedef struct moe_ctx moe_ctx;
typedef struct moe_layer moe_layer;
typedef struct moe_host_cache moe_host_cache;
typedef struct moe_expert_store moe_expert_store;

/* Layer shapes. d_model, d_ff and d_ff_shared are multiples of 64 (the
 * quantisation group) and of 32; n_experts <= 1024; 1 <= top_k <= min(32,
 * n_experts); d_model <= 8192. act: 0 = GELU (tanh form), 1 = SiLU. */
typedef struct {
    int32_t d_model, n_experts, top_k, d_ff, d_ff_shared, act;
} moe_shapes;

/* Quantisation layout. Only {4, 64, 8, 64} is accepted: experts are 4-bit
 * affine in groups of 64 along the input dimension, the router 8-bit affine
 * in groups of 64 ([P1] §2.1 table, §2.5 "量化方案"). */
typedef struct {
    int32_t w_bits, w_group, r_bits, r_group;
} moe_quant_layout;

/* One quantised matrix W[N][K] in the canonical layout (host memory):
 *   codes: row-major; 4-bit: K/2 bytes per row, element 2j in the low nibble
 *          of byte j and 2j+1 in the high nibble, unsigned 0..15;
 *          8-bit: K bytes per row, unsigned 0..255;
 *   scale, bias: f16 [N][K/64];  w[n][k] = scale[n][k/64] * q + bias[n][k/64]. */
typedef struct {
    const uint8_t* codes;
    const uint16_t* scale;
    const uint16_t* bias;
} moe_qmatrix;

/* All weights of one layer, canonical layout, host memory. Routed experts are
 * stacked on a leading expert axis (expert-major, [P3] "从实际路由找到 GGUF 权重切片":
 * slice = base + expert_id * stride):
 *   gate, up:  codes [E][d_ff][d_model/2],  scale/bias [E][d_ff][d_model/64]
 *   down:      codes [E][d_model][d_ff/2],  scale/bias [E][d_model][d_ff/64]
 *   shared_gate/up: [d_ff_shared][d_model], shared_down: [d_model][d_ff_shared]
 *   router:    codes [E][d_model] (8-bit), scale/bias [E][d_model/64] */
typedef struct {
    moe_qmatrix router;
    moe_qmatrix shared_gate, shared_up, shared_down;
    moe_qmatrix gate, up, down;
} moe_host_weights;

/* Cumulative counters of one layer since creation (or the last reset).
 * Lookups count distinct experts per cache step; bypasses are misses that
 * found no unpinned slot ([P3] "缓存管理的是专家工作集": the budget may be
 * exceeded temporarily) and are included in misses. exposed_copy_us is the
 * time the compute stream spent waiting for miss copies ([P3]
 * "读取完成后，算子才可以使用切片": overlap hides only part of the reads): for
 * each call with misses, how long after the expert kernel started the last
 * copy finished. It is measured only while kernel profiling is on
 * (moe_ctx_set_profiling), since it needs two timed events per call. */
typedef struct {
    uint64_t steps, hits, misses, bypass;
    uint64_t bytes_h2d;      /* bytes copied host -> device for misses */
    uint64_t bytes_resident; /* weight bytes the layer's kernels read from HBM */
    double exposed_copy_us;
    double host_wait_us;     /* host time spent waiting for the routing to be published */
    double host_issue_us;    /* host time in the cache step, copy issue and kernel launches */
} moe_stats;

/* ---- context ------------------------------------------------------------ */

/* Create a context on CUDA device `device` (made current on the calling
 * thread). Owns a copy stream and the transient staging arena shared by its
 * layers. If the environment variable MOE_TRACE_FILE names a file when the
 * context is created, the context records a timeline (diagnostics): for each
 * launch of its layers, the host's issue time (CLOCK_REALTIME ns) and the
 * device span from the earliest block start to the latest block end
 * (%globaltimer ns); for each call, the host's steps (call, routing seen,
 * copies issued, end). moe_ctx_destroy writes it as text lines
 * "cal <host ns before> <host ns after> <device ns>" (a one-thread kernel
 * read between the two host reads), "launch <kind> <layer> <call> <host ns>
 * <device start> <device end>" (kind as for moe_ctx_kernel_times) and
 * "host <step> <layer> <call> <host ns>".
 * Errors: MOE_EINVAL (no such device), MOE_ECUDA. */
moe_status moe_ctx_create(int device, moe_ctx** out);
void moe_ctx_destroy(moe_ctx* ctx); /* after all its layers are destroyed */

/* ---- layer -------------------------------------------------------------- */

/* Create one MoE layer with `cache_slots` HBM expert slots and a replacement
 * policy (0 = LFU, [P1] §6.2.2-§6.2.3 and §8.3; 1 = LRU, [P3]
 * "缓存管理的是专家工作集"). Allocates: router, shared expert and slot arena in
 * device memory; the routed-expert pool (all experts) in pinned host memory.
 * Nothing is loaded until moe_layer_set_weights.
 * Errors: MOE_EINVAL (shapes, layout, slots < 1 or > n_experts, policy),
 * MOE_ENOMEM (allocation failed; nothing is leaked). */
moe_status moe_layer_create(moe_ctx* ctx, const moe_shapes* shapes, const moe_quant_layout* layout,
                            int32_t cache_slots, int32_t policy, moe_layer** out);

/* Load weights from canonical host arrays (read during the call only). The
 * router and shared expert are repacked and copied to HBM; the routed experts
 * are repacked into the library's pinned host pool, one contiguous blob per
 * expert at base + e * expert_bytes ([P1] §9.2 item 2: one region per layer,
 * [offset, size] per expert). Resets the cache to empty.
 * Blocking. Errors: MOE_EINVAL (NULL pointer), MOE_ECUDA. */
moe_status moe_layer_set_weights(moe_layer* layer, const moe_host_weights* w);

/* Bytes of one routed expert in the library's blob (gate + up + down codes,
 * scales and biases); equals the canonical byte count. */
size_t moe_expert_bytes(const moe_shapes* shapes);

/* Router, top-k and gates ([P3] "每个 token、每层都要重新路由"; [P1] §2.4 cb1):
 *   logit[t][e] = sum_i x[t][i] * (scale * q + bias)[e][i] + zbias[e]  (fp32)
 *   ids[t][0..k)  = the k largest logits, descending, ties -> lower expert id
 *   gates[t][r]   = softmax over the k chosen logits (= the full softmax
 *                   renormalised over them).
 * The fp32 sum runs in a fixed order (runs of 16 inputs dealt round-robin to
 * 32 lanes, each lane sequential with fused multiply-adds, lanes combined by a
 * butterfly at distances 16, 8, 4, 2, 1), so ids are reproducible bit for bit.
 * x: device bf16 [T][d_model]; zbias: device f32 [E] or NULL; ids: device
 * int32 [T][k]; gates: device f32 [T][k]. T >= 1. Asynchronous on `stream`.
 * Errors: MOE_EINVAL, MOE_ESTATE (no weights), MOE_ECUDA. */
moe_status moe_route(moe_layer* layer, const void* x_bf16, int32_t T, const float* zbias, int32_t* ids,
                     float* gates, void* stream);

/* Predictive prefetch into HBM ([P1] §9.2 item 3 and §9.5 item 2: predict
 * the experts the next steps will need from routing history and read them
 * ahead). With on = 1 the layer keeps one spare expert buffer in device
 * memory. After each decode call, the copy stream fills it with the expert
 * that the layer's steps have routed to most often (ties to the lower id)
 * among those in no cache slot. A later miss of that expert then costs no
 * copy over the host link: the call's kernels read the spare buffer (after
 * an event wait for the prefetch copy), and the call's stream copies it into
 * the expert's slot behind them. The cache and its hit/miss trace do not
 * change (a prefetched expert still counts as a miss and enters the cache by
 * the LFU/LRU rules); only where a miss's bytes come from does. The prefetch
 * copies share the host link with the misses and count in bytes_h2d. Not for layers created
 * with moe_layer_create_streamed (they read ahead into their host tier).
 * Waits for the layer's calls and copies in flight. Errors: MOE_EINVAL,
 * MOE_ENOMEM, MOE_ECUDA. */
moe_status moe_layer_set_prefetch(moe_layer* layer, int32_t on);

/* Prefetches issued, and misses served from the spare buffer, since the
 * layer was created. Either pointer may be NULL. Errors: MOE_EINVAL. */
moe_status moe_layer_prefetch_stats(const moe_layer* layer, uint64_t* issued, uint64_t* used);

/* Ordered combine for decode calls (T <= 64): with on = 1, a decode call
 * sums its output in a fixed order, y[t] = S_t + O_{t,0} + ... + O_{t,k-1}
 * ([P1] §6.2.3: the shared expert's output plus the routed outputs weighted
 * by their gates, here in rank order r = 0..k-1), where S_t is the shared
 * expert's share and O_{t,r} the gate-weighted output of the rank-r expert.
 * The expert FFN kernels then store each work unit's share (32 intermediate
 * rows of one expert) in a partial row fixed by (token or pair, rows) instead
 * of adding it into y with fp32 atomics, and one more kernel adds the partial
 * rows in that order. Two calls on the same x give bit-identical y, whatever
 * the cache state (which experts were hits, misses or bypasses). Cost: one
 * kernel launch per call, and T * (d_ff_shared/32 + top_k * d_ff/32) *
 * d_model floats of layer-owned device memory (3 MB at T = 1 for d_model =
 * 2816, d_ff = 704, d_ff_shared = 2816, top_k = 8), allocated on the next
 * call, written and read once per call. With on = 0 (the default) the shares
 * are added with atomics in arrival order, so y may differ between calls in
 * the last bits. Prefill calls (T > 64) always combine in rank order. Waits
 * for the layer's calls in flight. Errors: MOE_EINVAL, MOE_ECUDA. */
moe_status moe_layer_set_deterministic(moe_layer* layer, int32_t on);

/* Kernel-timing diagnostic (the pages have no counterpart). Enqueues on
 * `stream`, `rounds` times over, for each of the n_layers layers in turn, the
 * expert-FFN launch that the layer's last one-token moe_forward call made for
 * its resident experts: the shared expert and each routed pair of that call's
 * routing, looked up in the device slot table as it stands now (every expert
 * the call copied in is resident by then). Each launch adds into its call's y
 * again, so those y are garbage afterwards; nothing else changes (caches,
 * statistics, routing). Every launch is a programmatic dependent of the
 * previous kernel, as in a pipelined decode loop, and one host call enqueues
 * them all, so a pair of events around this call times the kernel rather
 * than the host. *bytes (may be NULL) gets the weight bytes all the launches
 * read. All layers must be on one device.
 * Errors: MOE_EINVAL, MOE_ESTATE (a layer made no one-token call yet),
 * MOE_ECUDA. */
moe_status moe_layers_replay_resident(moe_layer* const* layers, int32_t n_layers, int32_t rounds, void* stream,
                                      double* bytes);

/* moe_route without any device allocation. The pages have no counterpart:
 * this entry point exists for callers that must not allocate, such as a
 * decode loop that holds a fixed memory budget, or one that cannot afford the
 * device-wide synchronisation that a cudaFree inside moe_route's scratch
 * growth would add. It computes exactly what moe_route computes, with the
 * same kernel and the same fixed summation order, but its scratch (the fp32
 * logits and the per-token-block arrival counters) lives in a statically
 * sized device array of the library instead of the layer's own buffers.
 * Limits: 1 <= T <= 64 and T * n_experts <= 16384 (64 KiB of fp32 logits);
 * larger calls fail with MOE_EINVAL before anything is enqueued.
 * Zero state: the counters must be zero when a call starts. They are zero
 * when the library is loaded, and every call leaves them at zero.
 * The first call on a device looks up the scratch's device address and
 * sets the router kernel's shared-memory attribute, so make it before any
 * stream capture. Later calls only enqueue the one router kernel.
 * Overlapping calls race: the scratch is shared by every layer on a device,
 * so two calls that may run at the same time (other streams, other threads)
 * corrupt each other's logits. Calls ordered on one stream are safe.
 * Not timed: with moe_ctx_set_profiling on, these launches are counted by
 * moe_ctx_launches but get no timing record in moe_ctx_kernel_times (a
 * record would create CUDA events, and the call creates nothing).
 * Arguments, layouts and outputs as for moe_route.
 * Errors: MOE_EINVAL (bad arguments or over the limits), MOE_ESTATE (no
 * weights), MOE_ECUDA (the set-up lookup or the launch failed). */
moe_status moe_route_noalloc(moe_layer* layer, const void* x_bf16, int32_t T, const float* zbias, int32_t* ids,
                             float* gates, void* stream);

/* One expert-cache step over n_ids expert ids (host int32, duplicates
 * allowed): LFU/LRU lookup ([P1] §8.3 flow) in which distinct ids are taken
 * in ascending order; hits are counted (LFU: use_count += 1; LRU: stamped
 * with the step index) and their slots pinned for the step; each miss takes
 * the lowest empty slot, else the unpinned slot with the smallest count (LRU:
 * oldest stamp), ties to the lowest slot index, and starts at count 1; a miss
 * that finds no unpinned slot bypasses the cache (slot -1).
 * For every miss that got a slot, the library enqueues the copy of that
 * expert from its pinned pool into the slot on its copy stream, ordered after
 * the layer's previous kernels; the slot's ready event is recorded after the
 * copy ([P3] "读取完成后，算子才可以使用切片").
 * Outputs (host): slot_of[n_ids] = slot holding ids[i] after the step or -1;
 * miss_experts[n_miss] and miss_slots[n_miss] in ascending expert order
 * (capacity n_ids each); *n_miss. Any output pointer may be NULL.
 * Errors: MOE_EINVAL (id out of range), MOE_ESTATE, MOE_ECOPY, MOE_ECUDA. */
moe_status moe_cache_step(moe_layer* layer, const int32_t* ids, int32_t n_ids, int32_t* slot_of,
                          int32_t* miss_experts, int32_t* miss_slots, int32_t* n_miss);

/* The whole layer on T tokens ([P1] §2.4 cb1 -> io -> cb2, §8.2):
 *   route -> (host) cache step + miss copies on the copy stream, while the
 *   shared expert runs on `stream` -> routed expert FFNs (hits first, misses
 *   after their ready events) -> y[t] = shared(x_t) + sum_{r<k} gate[t][r] *
 *   FFN_{ids[t][r]}(x_t).
 *   FFN_e(x) = W_down,e (act(W_gate,e x) * (W_up,e x)); fp32 accumulation.
 * T <= 64 runs the decode path (fused dequant GEMV kernels, fp32 arithmetic),
 * which adds each expert's share of y with fp32 atomic adds: the order of
 * those additions is not fixed, so y may differ between calls in the last
 * bits. Larger T runs as prefill in chunks of 128 tokens, each chunk routed, cached
 * and grouped by expert before the grouped expert GEMMs on the tensor cores
 * ([P1] §2.5, §8.4), whose operands are fp16 (weights fp16(s*q + b), x, and h
 * rounded to fp16) with fp32 accumulation. Bypassed experts are streamed into
 * the context's staging arena.
 * x: device bf16 [T][d_model]; zbias: device f32 [E] or NULL; y: device f32
 * [T][d_model]. Optional ids_out (device int32 [T][k]) and gates_out (device
 * f32 [T][k]) receive the routing; pass NULL to skip.
 * Blocks the calling thread once per chunk until the routing is known on the
 * host; y is complete when `stream` reaches the end of the call's work.
 * Errors: MOE_EINVAL, MOE_ESTATE, MOE_ECOPY (the cache is consistent and the
 * failed expert's slot is empty), MOE_ECUDA. */
moe_status moe_forward(moe_layer* layer, const void* x_bf16, int32_t T, const float* zbias, float* y,
                       int32_t* ids_out, float* gates_out, void* stream);

/* The whole layer on a prompt of T tokens run layer-major (a widening of the
 * prefill path: [P1] §8.4 runs a prompt as chunks so that one fetch of an
 * expert serves every row of the chunk; here the chunk is the whole prompt):
 * one routing of all T tokens, one cache step over all T*k pairs (so each
 * distinct expert is fetched at most once per call, and the cache trajectory
 * is that of one step, not of one step per 128 tokens), the grouped expert
 * GEMMs over every token routed to each expert (items of up to 128 token
 * rows; the shared expert per block of 128 tokens), and the combine. Same
 * arithmetic as moe_forward's prefill path. T <= 64 runs the decode path, as
 * moe_forward does.
 * x: device bf16 [T][d_model], 1 <= T <= 4096; zbias: device f32 [E] or NULL;
 * y: device f32 [T][d_model]; ids_out / gates_out as for moe_forward.
 * Blocks the calling thread once until the routing is known on the host.
 * Errors: MOE_EINVAL (bad arguments, T > 4096), MOE_ENOMEM (scratch for T
 * tokens), MOE_ESTATE, MOE_ECOPY, MOE_ECUDA. */
moe_status moe_forward_prompt(moe_layer* layer, const void* x_bf16, int32_t T, const float* zbias, float* y,
                              int32_t* ids_out, float* gates_out, void* stream);

/* Empties the layer's expert cache: every slot becomes free and every count
 * zero, as the per-layer slot cache of [P1] §6.2.2 is when created (and
 * after moe_layer_set_weights). Slot contents are not touched; the next calls
 * refill them. Waits for the layer's earlier calls to finish on the device
 * (the device copy of the slot table is rewritten), so call it between calls,
 * not while another thread uses the layer.
 * Errors: MOE_EINVAL (layer NULL), MOE_ESTATE (no weights), MOE_ECUDA. */
moe_status moe_cache_reset(moe_layer* layer);

/* Counters (see moe_stats). Waits for the layer's outstanding timing events. */
moe_status moe_layer_stats(moe_layer* layer, moe_stats* out);
moe_status moe_layer_reset_stats(moe_layer* layer);

/* Slot table snapshot (host): expert per slot (-1 = empty) and LFU counts,
 * arrays of cache_slots entries. */
moe_status moe_cache_dump(const moe_layer* layer, int32_t* slot_expert, uint32_t* counts);

void moe_layer_destroy(moe_layer* layer);

/* ---- host cache manager (no GPU needed) -------------------------------- */

/* The replacement policy that moe_cache_step runs, as a stand-alone host
 * object, so that its trace can be checked on any machine. Same rules and
 * outputs as moe_cache_step, without copies. Errors: MOE_EINVAL, MOE_ENOMEM. */
moe_status moe_host_cache_create(int32_t n_experts, int32_t slots, int32_t policy, moe_host_cache** out);
moe_status moe_host_cache_step(moe_host_cache* c, const int32_t* ids, int32_t n_ids, int32_t* slot_of,
                               int32_t* miss_experts, int32_t* miss_slots, int32_t* n_miss, int32_t* n_hit,
                               int32_t* n_bypass);
moe_status moe_host_cache_dump(const moe_host_cache* c, int32_t* slot_expert, uint32_t* counts);
void moe_host_cache_destroy(moe_host_cache* c);

/* Stable grouping of n_pairs (token, rank) pairs by expert, as the prefill
 * path does it ([P1] §2.5, §8.4: one fetched expert serves all rows of the
 * chunk): perm lists pair indices of expert 0, then 1, ..., each ascending;
 * offsets[e]..offsets[e+1] is expert e's range. Host arrays: ids [n_pairs],
 * offsets [n_experts + 1], perm [n_pairs]. Errors: MOE_EINVAL. */
moe_status moe_group_pairs(const int32_t* ids, int32_t n_pairs, int32_t n_experts, int32_t* offsets,
                           int32_t* perm);

/* ---- storage tier (expert files) ------------------------------------------ */

/* The tier below the pinned host pool: the pages stream routed experts from
 * SSD, reading the experts a layer needs with pread while the accelerator
 * computes ([P1] §2.3 "流式部分", "流水线"; §6.2.2 AsyncExpertReader with
 * request / wait_all), and their I/O notes ([P1] §9.2) ask for one file per
 * layer with an [offset, size] per expert (item 2), readahead of the experts
 * routing history makes likely (item 3), and O_DIRECT (item 4).
 *
 * File layout (one file per layer, written by moe_store_write):
 *   bytes [0, 4096): a header (magic "MOEXPRTS", version 1, the layer's
 *   moe_shapes, the expert blob size, the stride, the data offset 4096);
 *   expert e at 4096 + e * stride: the expert's blob as the library's slots
 *   hold it (the repacked layout; moe_expert_bytes(shapes) bytes), zero padded
 *   to stride = moe_store_expert_stride(shapes), a multiple of 4096.
 * A store reads such a file into a host tier of host_slots expert buffers
 * (4096-aligned; page-locked while a layer streams from it) with `readers`
 * threads, one pread of `stride` bytes per expert (or one per piece, see
 * moe_store_set_read_chunk). The store counts each expert's fetches, across
 * evictions. A fetched expert not in the tier takes an empty entry, else, of
 * the entries neither pinned nor being read, the one whose expert was
 * fetched least often (ties: least recently used) ([P1] §9.5 item 1 prefers
 * frequency to recency for MoE experts). */

/* Bytes between consecutive experts in an expert file (the blob size rounded
 * up to 4096); 0 if shapes is NULL. */
size_t moe_store_expert_stride(const moe_shapes* shapes);

/* Write one layer's routed experts (w->gate, w->up, w->down in the canonical
 * layout of moe_host_weights; the other matrices are not read) to `path`,
 * replacing the file. Blocking; uses a few host threads.
 * Errors: MOE_EINVAL (shapes, NULL pointers), MOE_EIO (create/write failed). */
moe_status moe_store_write(const char* path, const moe_shapes* shapes, const moe_host_weights* w);

#define MOE_STORE_DIRECT 1 /* open with O_DIRECT; plain reads if the file system refuses it */

/* Open an expert file for a layer of these shapes (they must equal the
 * file's). host_slots in [1, n_experts]; readers in [1, 64]; flags: 0 or
 * MOE_STORE_DIRECT (moe_store_get_stats reports whether direct I/O is on).
 * Errors: MOE_EINVAL (arguments, not an expert file, other shapes, short
 * file), MOE_EIO (open/read failed), MOE_ENOMEM. */
moe_status moe_store_open(const char* path, const moe_shapes* shapes, int32_t host_slots, int32_t readers,
                          int32_t flags, moe_expert_store** out);

/* Stop the readers (after the reads already queued) and free the tier.
 * Errors: MOE_ESTATE if a layer still streams from the store (destroy the
 * layer first); the store is then left open. */
moe_status moe_store_close(moe_expert_store* store);

/* The expert's bytes in the host tier (*out points at moe_expert_bytes
 * bytes), reading them first if needed (blocking). The entry stays pinned
 * (it is never reused) until a matching moe_store_release.
 * Errors: MOE_EINVAL, MOE_EBUSY (every entry is pinned), MOE_EIO (the read
 * failed; the entry is freed, and a later fetch retries). */
moe_status moe_store_fetch(moe_expert_store* store, int32_t expert, const uint8_t** out);
moe_status moe_store_release(moe_expert_store* store, int32_t expert); /* MOE_EINVAL if not pinned */

/* Readahead ([P1] §9.2 item 3): for each listed expert not in the tier, in
 * list order, queue its read into an entry that is empty, or else neither
 * pinned, being read, nor read ahead and not yet fetched, and whose expert
 * was fetched no more often than the listed one (an expert with no such
 * entry is skipped). These reads start only when no read a fetch needs is
 * waiting. Does not wait. *queued (may be NULL) receives the number queued. */
moe_status moe_store_prefetch(moe_expert_store* store, const int32_t* experts, int32_t n, int32_t* queued);

/* Read each expert as pieces of `bytes` (a multiple of 4096), which the
 * reader threads take in parallel, instead of as one pread of the whole
 * padded expert (bytes = 0, the default, or bytes >= the stride). Applies to
 * reads queued after the call. Errors: MOE_EINVAL (NULL, not a multiple of
 * 4096). */
moe_status moe_store_set_read_chunk(moe_expert_store* store, size_t bytes);

/* Block until no read is queued or running. */
moe_status moe_store_wait_idle(moe_expert_store* store);

typedef struct {
    uint64_t fetches;        /* fetches (moe_store_fetch and a streamed layer's misses) that returned
                                the bytes or a read error (not those refused with MOE_EBUSY) */
    uint64_t tier_hits;      /* fetches that found the expert in the tier, or being read ahead by a
                                readahead request (a streamed layer's reads of its own call's misses,
                                queued before their fetches, are not hits) */
    uint64_t reads;          /* reads finished (fetch-driven and readahead) */
    uint64_t prefetch_reads; /* reads queued by readahead requests */
    uint64_t prefetch_used;  /* experts read ahead that a fetch then used */
    uint64_t bytes_read;
    uint64_t read_errors;
    double read_us;          /* summed duration of the reads (they overlap across readers) */
    double wait_us;          /* time fetches spent blocked on reads */
    int32_t direct;          /* 1 if the file is read with O_DIRECT */
    int32_t host_slots, readers;
} moe_store_stats;

moe_status moe_store_get_stats(moe_expert_store* store, moe_store_stats* out);
moe_status moe_store_reset_stats(moe_expert_store* store);

/* The tier's table: per entry the expert it holds (-1 = none) and its state
 * (0 empty, 1 being read, 2 ready, 3 failed); arrays of host_slots entries,
 * either may be NULL. */
moe_status moe_store_tier(moe_expert_store* store, int32_t* entry_expert, int32_t* entry_state);

/* A layer whose routed experts stream from `store` instead of a pinned pool
 * holding all of them: as moe_layer_create, but no pool is allocated; the
 * store's tier is page-locked (cudaHostRegister) for the layer's lifetime,
 * and the store may serve no other layer until this one is destroyed. Each
 * miss copy first fetches the expert from the store (the call queues the
 * reads of all its misses at once, then copies each one as its read lands);
 * the entry is released once its copy has finished. moe_layer_set_weights
 * then loads the router and the shared expert only (the routed pointers may
 * be NULL). A read that fails ends the call with MOE_ECOPY, the expert's slot
 * left empty, as a failed copy does.
 * Errors: as moe_layer_create, plus MOE_EINVAL (the store's shapes differ, or
 * it already serves a layer) and MOE_ECUDA (page-locking the tier failed). */
moe_status moe_layer_create_streamed(moe_ctx* ctx, const moe_shapes* shapes, const moe_quant_layout* layout,
                                     int32_t cache_slots, int32_t policy, moe_expert_store* store,
                                     moe_layer** out);

/* Readahead from routing history ([P1] §9.2 item 3, §9.5 item 2): a streamed
 * layer counts, per expert, the cache steps that routed to it; this offers
 * the store's readahead (moe_store_prefetch) up to n experts with the highest
 * counts (ties to the lower id) that are routed at least once, not in the
 * layer's HBM slots and not in the store's tier. Meant to be called for layer
 * l+1 while layer l runs. Does not wait. *queued (may be NULL) receives the
 * number of reads queued.
 * Errors: MOE_EINVAL (NULL layer, n < 0), MOE_ESTATE (not a streamed layer). */
moe_status moe_layer_prefetch(moe_layer* layer, int32_t n, int32_t* queued);

/* ---- diagnostics -------------------------------------------------------- */

const char* moe_status_str(moe_status s);
const char* moe_last_error(void);

/* Per-kernel device time, measured with CUDA events recorded around each
 * launch on the launching stream while profiling is on (off by default; it
 * adds event records to the stream). kind: 0 router + top-k, 1 decode expert
 * FFN over resident weights (the shared expert, and the routed experts that
 * hit), 2 combine, 3 prefill grouped GEMM gate/up, 4 prefill grouped GEMM
 * down, 5 prefill token-row conversion to fp16, 6 decode expert FFN over the
 * experts copied in by the call (its duration includes the wait for the
 * copies). Returns launches, total
 * milliseconds and the algorithmic bytes and flops of those launches. Waits
 * for the events. */
moe_status moe_ctx_set_profiling(moe_ctx* ctx, int32_t on);
moe_status moe_ctx_kernel_times(moe_ctx* ctx, int32_t kind, uint64_t* launches, double* total_ms,
                                double* bytes, double* flops);
moe_status moe_ctx_reset_kernel_times(moe_ctx* ctx);

/* Number of kernels the context's layers have launched since its creation
 * (every launch is counted, profiling or not). */
moe_status moe_ctx_launches(moe_ctx* ctx, uint64_t* out);

/* Fault injection on the host, for tests of the failure path: the nth miss
 * copy issued from now on (0 = the next one) is reported as failed instead of
 * being issued, exactly as if cudaMemcpyAsync had returned an error. The call
 * that hits it returns MOE_ECOPY and leaves the affected slots empty; later
 * calls proceed normally. nth < 0 disarms. No device fault is involved. */
moe_status moe_ctx_inject_copy_failure(moe_ctx* ctx, int64_t nth);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
