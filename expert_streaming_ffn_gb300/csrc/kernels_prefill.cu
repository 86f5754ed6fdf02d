// Prefill grouped GEMM of the expert-streaming MoE layer on the 5th-generation
// tensor cores (sm_103a): tcgen05.mma with fp16 operands in shared memory and
// fp32 accumulators in tensor memory.
//
//   [P1] "在 Rockchip NPU 上实现 turbo-fieldfare 风格 MoE 大模型流式推理的技术方案"
//        §2.5 and §8.4: a prefill chunk's tokens are grouped per expert, so one
//        fetch of an expert's weights serves every row of the chunk routed to it.
//
// One launch per phase. A job is one 128-row tile of one item's weight matrix
// over all of K (or, when a launch has too few tiles to fill the GPU, over a
// slice of K, the slices' sums added by pf_reduce_kernel), against all of the
// item's token rows (N <= 128, padded to a multiple of 16):
//   phase 1 (gate/up): the tile interleaves 64 gate rows and the same 64 up
//     rows (in each 32-row quarter, even rows gate and odd rows up), so the
//     epilogue forms h = act(gate) * up from neighbouring lanes;
//   phase 2 (down): 128 consecutive output rows.
// Warp roles in a CTA of 832 threads (one CTA per SM, persistent over jobs):
//   warps 0-3   MMA issue, one thread each, K-block kb of a job going to
//               issuer kb mod nI (one thread issues a tcgen05.mma only about
//               every 60-125 cycles, whatever N, so several issue in
//               parallel); warp 0 also allocates TMEM;
//   warps 4-7   epilogue, one TMEM lane quarter each;
//   warps 8-23  dequantisation in four groups of 4 warps, group g taking the
//               K-blocks whose running index is g mod 4 (A stages g and
//               g + 4 in turn); a thread turns one A row of 64 codes into fp16
//               w = fp16(s q + b) in the 128B-swizzled K-major A tile;
//   warp 24     bulk copies of the weight codes and scales of 4 K-blocks of
//               the job's row tiles at a time, into a raw ring (gate/up in
//               the tiled record format, down column-sliced);
//   warp 25     TMA loads of the token rows (128B-swizzled fp16): a routed
//               expert's rows, padded to 16, 32, 64 or 128, one 3-D box of a
//               whole B slot's K-blocks at a time; the shared expert's token
//               block, one 2-D box per K-block.
// Copies are few and large (a bulk copy costs its issuing thread tens of
// nanoseconds whatever its size), and the two producers issue in parallel.
// The single-thread roles (the issuers above all) sit on sub-partitions
// shared with busy dequantising warps, where every dependent instruction
// waits its turn: their loops do only the work of their own K-blocks, with
// stage and phase taken from running counts by masks, not divisions.
// Every wait is bounded; on expiry the kernel records an error bit, raises an
// abort flag that makes every other wait give up, drains its asynchronous work
// and frees its tensor memory before it exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 832;
// warps 0-3 issue MMAs (one thread each), 4-7 epilogue, 8-23 dequantise (four
// groups of 4, group g owning A stages g and g + 4), 24 and 25 load
constexpr int kIssuers = 4, kWarpEpi = 4, kWarpDq = 8, kDqWarps = 4, kDqGroups = 4, kWarpLoad = 24, kWarpB = 25;
constexpr int kUnit = 4;
constexpr int kTileM = 128;
constexpr int kRecord = 1152;           // 32 rows x 64 codes, then 32 scale/bias words
constexpr int kABytes = kTileM * 128;   // 128 rows x 64 fp16, 128B-swizzled
constexpr int kBBytes = kPfMaxN * 128;  // up to 128 token rows x 64 fp16
constexpr int kRawBytes = 4 * kUnit * kRecord;  // 4 row tiles x kUnit records
// Two accumulator buffers of 256 fp32 columns. A job's K-blocks are dealt to
// nI issuers in turn (nI = 4 for up to 64 token rows, else 2), each issuer
// accumulating into its own 256/nI columns of the buffer; the epilogue sums them.
constexpr int kTmemCols = 512;
// Ring sizes of a launch's layout. A stage holds one K-block (64) of the A
// tile; a B slot as many K-blocks of the job's token rows as fit in 16 KB; a
// raw stage kUnit K-blocks of codes and scales. Within a job every round of an
// A stage has the same issuer (kStages is a multiple of nI); between jobs the
// issuers hand off (see the MMA issue loop).
template <int A, int B, int R, bool D>
struct PfRings {
    static constexpr int kStages = A, kSlotsB = B, kRawStages = R;
    // routed token rows padded to a power of two and loaded one 3-D box per B
    // slot (else padded to a multiple of 16, 2-D boxes of 16, 64 or 128 rows)
    static constexpr bool kRows3d = D;
    static constexpr int kStageShift = A == 8 ? 3 : A == 4 ? 2 : A == 2 ? 1 : 0;
    static constexpr int kSlotShift = B == 8 ? 3 : B == 4 ? 2 : B == 2 ? 1 : 0;
    static_assert((1 << kStageShift) == A && (1 << kSlotShift) == B, "rings indexed by masks");
    static_assert(A % kIssuers == 0, "an A stage keeps its issuer within a job");
    static_assert(A % kDqGroups == 0, "each dequantising group owns whole A stages");
    // A ring, B ring, raw ring, barriers, TMEM address; +1 KB to align
    static constexpr int kSmemBytes = 1024 + A * kABytes + B * kBBytes + R * kRawBytes + 320;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};
// Chunks, whose routed experts have few rows each: most of shared memory to
// the A ring, whose loop dequantise -> MMA -> release then bounds the kernel,
// two stages per dequantising group; two B slots hold up to 16 K-blocks of
// 16-row items. Long prompts (~32 rows an expert, often more): four B slots,
// as two would hold only four K-blocks of 48- or 64-row items.
using RingsChunk = PfRings<8, 2, 3, true>;
using RingsPrompt = PfRings<4, 4, 4, false>;

// Shared-memory matrix descriptor of a K-major operand tile whose rows are 128
// bytes apart with the 128-byte swizzle (8-row atoms of 1024 bytes).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4)  // start address
           | ((uint64_t)1 << 16)                // leading byte offset (unused for swizzled K-major)
           | ((uint64_t)(1024 >> 4) << 32)      // stride byte offset: 8 rows
           | ((uint64_t)1 << 46)                // descriptor version
           | ((uint64_t)2 << 61);               // 128-byte swizzle
}

// Instruction descriptor: fp16 A and B, both K-major, fp32 D, M x N.
__device__ __forceinline__ uint32_t f16_idesc(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Eight codes of one word (device nibble order: nibble i holds element
// [0,2,4,6,1,3,5,7][i]) to eight fp16 weights fp16(s * q + b), elements in
// order. (w & 0x000F000F) | 0x6400_6400 is the fp16 pair (1024 + q, 1024 + q')
// exactly; with the mask 0x00F000F0 it is (1024 + 16 q, ...), brought back to
// q by one exact fused multiply-add.
__device__ __forceinline__ uint4 dequant8(uint32_t v, __half2 s2, __half2 b2) {
    const uint32_t M = 0x64006400u;
    const __half2 c1024 = as_h2(0x64006400u);  // (1024, 1024)
    const __half2 inv16 = as_h2(0x2C002C00u);  // (1/16, 1/16)
    const __half2 m64 = as_h2(0xD400D400u);    // (-64, -64)
    const uint32_t u = v >> 8;
    const __half2 q0 = __hsub2(as_h2((v & 0x000F000Fu) | M), c1024);
    const __half2 q1 = __hfma2(as_h2((v & 0x00F000F0u) | M), inv16, m64);
    const __half2 q2 = __hsub2(as_h2((u & 0x000F000Fu) | M), c1024);
    const __half2 q3 = __hfma2(as_h2((u & 0x00F000F0u) | M), inv16, m64);
    uint4 r;
    r.x = as_u32(__hfma2(q0, s2, b2));
    r.y = as_u32(__hfma2(q1, s2, b2));
    r.z = as_u32(__hfma2(q2, s2, b2));
    r.w = as_u32(__hfma2(q3, s2, b2));
    return r;
}

__device__ __forceinline__ float act_fn(float z, int act) {
    if (act == 1) return z / (1.0f + expf(-z));
    return 0.5f * z * (1.0f + tanhf(0.7978845608028654f * (z + 0.044715f * z * z * z)));
}

// A job: one M tile of one item over K-blocks kb0 .. kb0 + nkb - 1, part
// `part` of the tile's ks[fam] parts.
// The routed experts' token rows. Maps 0-3 see them as [K-block][row][64]
// and load boxes of 16 << i rows by min(8 >> i, K-blocks) K-blocks, a whole B
// slot at once; maps 4-6 load 2-D boxes of 16, 64 and 128 rows by one K-block.
struct PfRowMaps {
    CUtensorMap r[7];
};

struct Job {
    int item, fam, tile, part, kb0, nkb;
};

struct Plan {
    int phase;
    int tiles[2];    // M tiles per item
    int kblocks[2];  // K blocks of 64
    int ks[2];       // K parts of a tile
    int n_jobs, jobs0;
};

__device__ __forceinline__ Plan make_plan(const PfArgs& a, int phase) {
    Plan p;
    p.phase = phase;
    for (int f = 0; f < 2; ++f) {
        p.tiles[f] = phase == 1 ? a.inter[f] / 64 : a.d / kTileM;
        p.kblocks[f] = phase == 1 ? a.d / 64 : a.inter[f] / 64;
    }
    for (int f = 0; f < 2; ++f) p.ks[f] = a.ks[f] > 1 ? a.ks[f] : 1;
    p.jobs0 = a.n_fam0 * p.tiles[0] * p.ks[0];
    p.n_jobs = p.jobs0 + (a.n_items - a.n_fam0) * p.tiles[1] * p.ks[1];
    return p;
}

// A tile's parts are consecutive jobs, so they run at once on neighbouring
// CTAs.
__device__ __forceinline__ Job decode_job(const Plan& p, const PfArgs& a, int j) {
    Job b;
    // (selects, not indexing: an indexed Plan array would live in local memory)
    b.fam = j < p.jobs0 ? 0 : 1;
    if (b.fam) j -= p.jobs0;
    const int ks = b.fam ? p.ks[1] : p.ks[0];
    const int per_item = (b.fam ? p.tiles[1] : p.tiles[0]) * ks;
    const int i = j / per_item;
    const int r = j - i * per_item;
    b.item = b.fam ? a.n_fam0 + i : i;
    const int K = b.fam ? p.kblocks[1] : p.kblocks[0];
    if (ks == 1) {
        b.tile = r;
        b.part = 0;
        b.kb0 = 0;
        b.nkb = K;
    } else {
        b.tile = r / ks;
        b.part = r - b.tile * ks;
        b.kb0 = b.part * K / ks;
        b.nkb = (b.part + 1) * K / ks - b.kb0;
    }
    return b;
}

__device__ __forceinline__ int pad16(int n) { return n <= 16 ? 16 : (n + 15) & ~15; }

// Token rows of a job's B operand (the MMA's N): a routed expert's rows padded
// to a multiple of 16, or to a power of two from 16 where they are loaded one
// 3-D box per B slot; the shared expert's
// token block padded to a multiple of 16, or all kPfMaxN when there are several
// blocks (rows past the last token read as zeros).
__device__ __forceinline__ int job_rows(const PfArgs& a, int fam, int np, bool rows3d) {
    if (fam == 0) return a.n_fam0 > 1 ? kPfMaxN : pad16(np);
    if (!rows3d) return pad16(np);
    int n = 16;
    while (n < np) n <<= 1;
    return n;
}

__device__ __forceinline__ bool wait_flag(const uint32_t* p, uint32_t want, volatile int* abort) {
    for (uint64_t t0 = 0;;) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v == want) return true;
        if (*abort) return false;
        const uint64_t now = ptx::globaltimer();
        if (t0 == 0) t0 = now;
        if (now - t0 > ptx::kWaitLimitNs) return false;
        __nanosleep(128);
    }
}

template <class Rg>
__global__ void __launch_bounds__(kThreads, 1)
    pf_gemm_kernel(const __grid_constant__ PfArgs a, const int phase, const __grid_constant__ CUtensorMap map0,
                   const __grid_constant__ PfRowMaps rmaps) {
    constexpr int kStages = Rg::kStages, kSlotsB = Rg::kSlotsB, kRawStages = Rg::kRawStages;
    constexpr int kStageShift = Rg::kStageShift, kSlotShift = Rg::kSlotShift;
    constexpr bool kRows3d = Rg::kRows3d;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char* ringA = smem;
    unsigned char* ringB = ringA + kStages * kABytes;
    unsigned char* ringR = ringB + kSlotsB * kBBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ringR + kRawStages * kRawBytes);
    uint64_t* raw_full = bars;                    // [kRawStages] records landed
    uint64_t* raw_empty = raw_full + kRawStages;  // [kRawStages] records dequantised
    uint64_t* b_full = raw_empty + kRawStages;    // [kSlotsB] token rows landed
    uint64_t* b_empty = b_full + kSlotsB;         // [kSlotsB] MMAs reading the slot done
    uint64_t* a_full = b_empty + kSlotsB;         // [kStages] A tile dequantised
    uint64_t* a_empty = a_full + kStages;         // [kStages] MMAs reading the stage done
    uint64_t* acc_full = a_empty + kStages;       // [2] accumulator complete
    uint64_t* acc_empty = acc_full + 2;           // [2] accumulator read out
    uint64_t* drain = acc_empty + 2;              // [1] every MMA of the CTA done
    uint64_t* handoff = drain + 1;                // [1] every issuer done with a job's A stages
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(handoff + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Plan P = make_plan(a, phase);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRawStages; ++i) {
            ptx::mbar_init(raw_full + i, 1);
            ptx::mbar_init(raw_empty + i, kDqGroups * kDqWarps);
        }
        for (int i = 0; i < kSlotsB; ++i) {
            ptx::mbar_init(b_full + i, 1);
            ptx::mbar_init(b_empty + i, kIssuers);
        }
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(a_full + i, kDqWarps);
            ptx::mbar_init(a_empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(acc_full + i, kIssuers);
            ptx::mbar_init(acc_empty + i, 4);
        }
        ptx::mbar_init(drain, kIssuers);
        ptx::mbar_init(handoff, kIssuers);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* abortp = &abort_flag;
    auto fail = [&](unsigned bit) {
        atomicOr(a.err, bit);
        abort_flag = 1;
    };
    // diagnostics: the first kPfFailRecords expired waits of the launch, as
    // (block << 48 | warp << 40 | what << 32 | job << 16 | K-block), what =
    // 1 raw_empty, 2 b_empty, 3 acc_empty, 4 b_full, 5 a_full, 6 acc_full, 7 raw_full, 8 a_empty,
    // 9 handoff
    auto record = [&](int what, int job, int kb) {
        if (!a.trace) return;
        unsigned long long* rec = a.trace;
        const unsigned k = atomicAdd(reinterpret_cast<unsigned*>(rec), 1u);
        if (k < kPfFailRecords)
            rec[1 + k] = ((unsigned long long)blockIdx.x << 48) | ((unsigned long long)warp << 40) |
                         ((unsigned long long)what << 32) | ((unsigned long long)(job & 0xFFFF) << 16) | (kb & 0xFFFF);
    };

    if (warp == kWarpLoad) {
        // ---------------- weight records ----------------
        // Lane 0 waits and arms the stage; the copies of a stage are issued by
        // several lanes at once (a bulk copy costs its thread tens of ns).
        int r = 0;
        uint32_t ph = 0;
        int issued = 0;
        bool ok = true;
        for (int j = blockIdx.x; j < P.n_jobs && ok; j += gridDim.x) {
            const Job b = decode_job(P, a, j);
            const PfItem it = a.items[b.item];
            // the part of the expert this phase reads: gate/up bytes, or down bytes
            const int flag = phase == 1 ? it.ready : it.ready_dn;
            if (lane == 0 && flag >= 0 && !wait_flag(a.ready + flag, a.epoch, abortp)) {
                if (!*abortp) fail(32u);
                ok = false;
            }
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok) break;
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const int I = a.inter[b.fam];
            const size_t mat = qmat_bytes(I, a.d);
            const int nkb = b.nkb;
            for (int kb0 = 0; kb0 < nkb; kb0 += kUnit) {
                const int kbA = b.kb0 + kb0;  // the unit's first K-block within the matrix
                const int nu = min(kUnit, nkb - kb0);
                bool w = true;
                if (lane == 0) {
                    w = ptx::mbar_wait_sleep(raw_empty + r, ph ^ 1, abortp);
                    if (!w) {
                        record(1, j, kb0);
                        if (!*abortp) fail(32u);
                    } else {
                        ptx::mbar_arrive_expect_tx(raw_full + r, (uint32_t)(4 * nu * kRecord));
                    }
                }
                w = __shfl_sync(kFull, w, 0);
                if (!w) {
                    ok = false;
                    break;
                }
                unsigned char* raw = ringR + r * kRawBytes;
                if (phase == 1) {
                    // lane t < 4: row tile t of the job (gate 2i, gate 2i+1, up 2i, up 2i+1),
                    // records kb0 .. kb0+nu-1, into raw + t * kUnit * kRecord
                    if (lane < 4) {
                        const int G = a.d / 64;
                        const unsigned char* m = it.w + (size_t)(lane >> 1) * mat;
                        const int rt = 2 * b.tile + (lane & 1);
                        ptx::bulk_g2s(raw + lane * kUnit * kRecord, m + ((size_t)rt * G + kbA) * kRecord,
                                      nu * kRecord, raw_full + r);
                    }
                } else {
                    // down, column-sliced: the job's 4 row tiles are contiguous within each
                    // 32-input chunk (2 KB of codes) and each group's scale block (512 B).
                    // Lane c < 2 nu copies chunk 2 kb0 + c to raw + c * 2048; lane 16 + u
                    // (u < nu) the scale block of group kb0 + u to raw + kUnit * 4096 + u * 512.
                    const int RT = a.d / 32;
                    const unsigned char* dn = it.w + 2 * mat;
                    if (lane < 2 * nu)
                        ptx::bulk_g2s(raw + lane * 2048, dn + ((size_t)(2 * kbA + lane) * RT + 4 * b.tile) * 512, 2048,
                                      raw_full + r);
                    else if (lane >= 16 && lane - 16 < nu)
                        ptx::bulk_g2s(raw + kUnit * 4096 + (lane - 16) * 512,
                                      dn + down_codes_bytes(a.d, I) + ((size_t)(kbA + lane - 16) * RT + 4 * b.tile) * 128,
                                      512, raw_full + r);
                }
                __syncwarp();
                ++issued;
                if (++r == kRawStages) {
                    r = 0;
                    ph ^= 1;
                }
            }
        }
        if (!ok && lane == 0) {
            // let the copies already issued land before the CTA can exit
            for (int i = 0; i < kRawStages && i < issued; ++i) {
                int sl = r - 1 - i;
                uint32_t par = ph;
                if (sl < 0) {
                    sl += kRawStages;
                    par ^= 1;
                }
                ptx::mbar_wait_bounded(raw_full + sl, par, nullptr);
            }
        }
    } else if (warp == kWarpB) {
        // ---------------- token rows ----------------
        if (lane == 0) {
            ptx::prefetch_tensormap(&map0);
            for (int q = kRows3d ? 0 : 4; q < (kRows3d ? 4 : 5); ++q) ptx::prefetch_tensormap(&rmaps.r[q]);
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int j = blockIdx.x; j < P.n_jobs && ok; j += gridDim.x) {
                const Job b = decode_job(P, a, j);
                const PfItem it = a.items[b.item];
                const int nb = job_rows(a, b.fam, it.np, kRows3d);
                const int kpb = kPfMaxN / nb;  // K-blocks per slot
                const int nkb = b.nkb;
                for (int kb0 = 0; kb0 < nkb; kb0 += kpb) {
                    const int nk = min(kpb, nkb - kb0);
                    if (!ptx::mbar_wait_sleep(b_empty + s, ph ^ 1, abortp)) {
                        record(2, j, kb0);
                        if (!*abortp) fail(512u);
                        ok = false;
                        break;
                    }
                    unsigned char* bt = ringB + s * kBBytes;
                    if (b.fam == 1 && !kRows3d && (nb == 128 || nb == 64)) {
                        // a routed expert of 64 or 128 rows: one box per K-block
                        // (a box load costs its issuing thread ~100 ns)
                        const CUtensorMap* m = &rmaps.r[nb == 128 ? 6 : 5];
                        ptx::mbar_arrive_expect_tx(b_full + s, (uint32_t)(nk * nb * 128));
                        for (int kk = 0; kk < nk; ++kk)
                            ptx::tma_load_2d(bt + kk * nb * 128, m, (b.kb0 + kb0 + kk) * 64, it.pb, b_full + s);
                    } else if (b.fam == 1 && !kRows3d) {
                        // a routed expert: 16-row boxes, one K-block each
                        ptx::mbar_arrive_expect_tx(b_full + s, (uint32_t)(nk * nb * 128));
                        for (int kk = 0; kk < nk; ++kk)
                            for (int r0 = 0; r0 < nb; r0 += 16)
                                ptx::tma_load_2d(bt + (kk * nb + r0) * 128, &rmaps.r[4], (b.kb0 + kb0 + kk) * 64,
                                                 it.pb + r0, b_full + s);
                    } else if (b.fam == 1) {
                        // a routed expert: one box of the slot's kpb K-blocks
                        // (K-blocks past the job's last are loaded and not read)
                        const int q = nb == 16 ? 0 : nb == 32 ? 1 : nb == 64 ? 2 : 3;
                        const int depth = min(kpb, P.kblocks[1]);
                        ptx::mbar_arrive_expect_tx(b_full + s, (uint32_t)(depth * nb * 128));
                        ptx::tma_load_3d(bt, &rmaps.r[q], 0, it.pb, b.kb0 + kb0, b_full + s);
                    } else {
                        // the shared expert: one box of the token block's rows per
                        // K-block (rows past the last token read as zeros)
                        ptx::mbar_arrive_expect_tx(b_full + s, (uint32_t)(nk * nb * 128));
                        for (int kk = 0; kk < nk; ++kk)
                            ptx::tma_load_2d(bt + kk * nb * 128, &map0, (b.kb0 + kb0 + kk) * 64, it.pb, b_full + s);
                    }
                    ++issued;
                    if (++s == kSlotsB) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok) {
                for (int i = 0; i < kSlotsB && i < issued; ++i) {
                    int sl = s - 1 - i;
                    uint32_t par = ph;
                    if (sl < 0) {
                        sl += kSlotsB;
                        par ^= 1;
                    }
                    ptx::mbar_wait_bounded(b_full + sl, par, nullptr);
                }
            }
        }
    } else if (warp < kIssuers) {
        // ---------------- MMA issue ----------------
        // An issuer visits only its own K-blocks (kb mod nI == i): it waits on
        // and releases just their A stages, whose index and phase parity follow
        // from the CTA's running K-block count. Every issuer waits on every B
        // slot and arrives once per round on its release, after its own MMAs
        // that read it (a slot's K-blocks are spread over the issuers).
        if (lane == 0) {
            const int i = warp;  // this issuer
            const uint64_t a_desc0 = sw128_desc(ptx::smem_addr(ringA));
            const uint64_t b_desc0 = sw128_desc(ptx::smem_addr(ringB));
            uint32_t C = 0, SB = 0;  // K-blocks and B slots of this CTA's earlier jobs
            int njob = 0;
            for (int j = blockIdx.x; j < P.n_jobs; j += gridDim.x, ++njob) {
                const Job b = decode_job(P, a, j);
                const int nb = job_rows(a, b.fam, a.items[b.item].np, kRows3d);
                const int kpb = kPfMaxN / nb;
                const int nkb = b.nkb;
                const int nI = nb <= 64 ? 4 : 2;
                const int buf = njob & 1;
                const uint32_t idesc = f16_idesc(kTileM, nb);
                const uint32_t d_tmem = tmem + buf * 256 + i * (256 / nI);
                bool ok = ptx::mbar_wait_sleep(acc_empty + buf, ((njob >> 1) & 1) ^ 1, abortp);
                if (!ok) record(3, j, 0);
                ptx::tc_fence_after();
                uint32_t acc = 0;
                // K-block kb of the job is this issuer's when kb % nI == i
                int kb = i;
                for (int kb0 = 0; kb0 < nkb; kb0 += kpb, ++SB) {
                    const int kend = min(kb0 + kpb, nkb);
                    const int sl = (int)(SB & (kSlotsB - 1));
                    if (ok && !ptx::mbar_wait_sleep(b_full + sl, (SB >> kSlotShift) & 1, abortp)) {
                        ok = false;
                        record(4, j, kb0);
                    }
                    const uint64_t bslot = b_desc0 + (uint64_t)((sl * kBBytes) >> 4);
                    for (; ok && i < nI && kb < kend; kb += nI) {
                        const uint32_t c = C + (uint32_t)kb;
                        const int st = (int)(c & (kStages - 1));
                        if (!ptx::mbar_wait_sleep(a_full + st, (c >> kStageShift) & 1, abortp)) {
                            ok = false;
                            record(5, j, kb);
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint64_t ad = a_desc0 + (uint64_t)((st * kABytes) >> 4);
                        const uint64_t bd = bslot + (uint64_t)(((kb - kb0) * nb * 128) >> 4);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {  // K = 16 per MMA: +32 bytes in the swizzled row
                            ptx::mma_f16_ss(d_tmem, ad + 2 * k, bd + 2 * k, idesc, acc);
                            acc = 1;
                        }
                        ptx::mma_commit(a_empty + st);
                    }
                    // every issuer arrives once per round of every slot (after its own MMAs on it)
                    if (ok) ptx::mma_commit(b_empty + sl);
                }
                C += (uint32_t)nkb;
                if (ok) {
                    ptx::mma_commit(acc_full + buf);
                } else if (!*abortp) {
                    fail(128u);
                }
                // Hand-off: a stage's owner (kb % nI of the job's K-blocks) can change
                // between jobs; nobody waits on a stage of the next job before every
                // issuer has taken its last stage of this one.
                ptx::mbar_arrive(handoff);
                if (!ptx::mbar_wait_sleep(handoff, njob & 1, abortp)) {
                    record(9, j, nkb);
                    if (!*abortp) fail(128u);
                }
            }
            ptx::mma_commit(drain);
            ptx::mbar_wait_bounded(drain, 0, nullptr);
        }
    } else if (warp >= kWarpEpi && warp < kWarpEpi + 4) {
        // ---------------- epilogue ----------------
        const int q = warp - kWarpEpi;  // TMEM lanes 32q .. 32q + 31
        const int row = 32 * q + lane;  // this thread's row of the 128-row tile
        int njob = 0;
        for (int j = blockIdx.x; j < P.n_jobs; j += gridDim.x, ++njob) {
            const Job b = decode_job(P, a, j);
            const PfItem it = a.items[b.item];
            const int nb = job_rows(a, b.fam, it.np, kRows3d);
            const int buf = njob & 1;
            if (!__all_sync(kFull, ptx::mbar_wait_sleep(acc_full + buf, (njob >> 1) & 1, abortp))) {
                if (lane == 0) record(6, j, 0);
                if (lane == 0 && !*abortp) fail(256u);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * 256;
            const int nI = nb <= 64 ? 4 : 2;
            const int used = min(nI, b.nkb);  // issuers that accumulated anything
            // v = the sum of the issuers' accumulators for 16 columns from c, in issuer order
            auto load_sum = [&](int c, uint32_t (&v)[16]) {
                ptx::tmem_ld16(taddr + c, v);
                for (int i = 1; i < used; ++i) {
                    uint32_t w[16];
                    ptx::tmem_ld16(taddr + i * (256 / nI) + c, w);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int m = 0; m < 16; ++m) v[m] = __float_as_uint(__uint_as_float(v[m]) + __uint_as_float(w[m]));
                }
                ptx::tmem_ld_wait();
            };
            // K split: this part's sums go to the part buffer
            // ([split tile][part][column][row], so a warp's stores are whole
            // lines) and pf_reduce_kernel adds the parts and writes the tile
            const int ks = b.fam ? P.ks[1] : P.ks[0];
            if (ks > 1) {
                const size_t fam_tile =
                    (size_t)(b.item - (b.fam ? a.n_fam0 : 0)) * (b.fam ? P.tiles[1] : P.tiles[0]) + b.tile;
                const size_t n0 = P.ks[0] > 1 ? (size_t)a.n_fam0 * P.tiles[0] : 0;  // family 0's split tiles
                const size_t part = (b.fam ? n0 * P.ks[0] : 0) + fam_tile * ks + b.part;
                float* mine = a.part + part * kPfMaxN * kTileM + row;
                for (int c = 0; c < nb; c += 16) {
                    uint32_t v[16];
                    load_sum(c, v);
#pragma unroll
                    for (int m = 0; m < 16; ++m) mine[(size_t)(c + m) * kTileM] = __uint_as_float(v[m]);
                }
            } else if (phase == 1) {
                const int I = a.inter[b.fam];
                const int irow = 64 * b.tile + 16 * q + (lane >> 1);
                __half* hb = a.h[b.fam];
                for (int c = 0; c < nb; c += 16) {
                    uint32_t v[16];
                    load_sum(c, v);
                    // even lanes hold gate rows, odd lanes the matching up rows:
                    // the even lane finishes columns c..c+7, the odd lane c+8..c+15
                    const bool odd = lane & 1;
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const float mine = __uint_as_float(odd ? v[m + 8] : v[m]);
                        const float other = __shfl_xor_sync(kFull, __uint_as_float(odd ? v[m] : v[m + 8]), 1);
                        const float g = odd ? other : mine, u = odd ? mine : other;
                        const int col = c + m + (odd ? 8 : 0);
                        if (col < it.np) hb[(size_t)(it.pb + col) * I + irow] = __float2half_rn(act_fn(g, a.act) * u);
                    }
                }
            } else {
                const int n = kTileM * b.tile + row;
                // output row of each column: the token (family 0) or the pair
                // index (family 1); lane l holds that of columns l, 32 + l, ...
                int prow[kPfMaxN / 32];
#pragma unroll
                for (int q = 0; q < kPfMaxN / 32; ++q) {
                    const int col = 32 * q + lane;
                    prow[q] = col >= it.np ? 0 : b.fam == 0 ? it.pb + col : a.pair[it.pb + col];
                }
                for (int c = 0; c < nb; c += 16) {
                    uint32_t v[16];
                    load_sum(c, v);
                    const int pq = c < 32 ? prow[0] : c < 64 ? prow[1] : c < 96 ? prow[2] : prow[3];
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const int col = c + m;
                        const int orow = __shfl_sync(kFull, pq, col & 31);
                        if (col >= it.np) break;
                        a.out[b.fam][(size_t)orow * a.d + n] = __uint_as_float(v[m]);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acc_empty + buf);
        }
    } else if (warp >= kWarpDq && warp < kWarpDq + kDqGroups * kDqWarps) {
        // ---------------- dequantisation ----------------
        // group g takes the K-blocks whose running index c is g mod 4, into A
        // stage c mod kStages; thread t of a group dequantises A row t, all 64
        // inputs, from words it loads before it releases the raw stage
        const int grp = (warp - kWarpDq) / kDqWarps, wg = (warp - kWarpDq) % kDqWarps;
        const int rho = wg * 32 + lane;
        int tile_raw, rlane;
        if (phase == 1) {
            const int qq = rho >> 5, l = rho & 31;
            const int wrow = 16 * qq + (l >> 1);
            tile_raw = (l & 1) * 2 + (wrow >> 5);
            rlane = wrow & 31;
        } else {
            tile_raw = rho >> 5;
            rlane = rho & 31;
        }
        const int codes_off = phase == 1 ? tile_raw * kUnit * kRecord + rlane * 16 : tile_raw * 512 + rlane * 16;
        const int codes_hh = phase == 1 ? 512 : 2048;
        const int codes_step = phase == 1 ? kRecord : 4096;
        const int sb_off = phase == 1 ? tile_raw * kUnit * kRecord + 1024 + sb_pos(rlane) * 4
                                      : kUnit * 4096 + tile_raw * 128 + sb_pos(rlane) * 4;
        const int sb_step = phase == 1 ? kRecord : 512;
        const int swz = rho & 7;
        const uint32_t arow0 = ptx::smem_addr(ringA + rho * 128);
        int r = 0;
        uint32_t rph = 0, cb = 0;
        for (int j = blockIdx.x; j < P.n_jobs; j += gridDim.x) {
            const Job b = decode_job(P, a, j);
            const int nkb = b.nkb;
            for (int kb0 = 0; kb0 < nkb; kb0 += kUnit) {
                const int nu = min(kUnit, nkb - kb0);
                const bool have = ptx::mbar_wait_sleep(raw_full + r, rph, abortp);
                if (!have && lane == 0) record(7, j, kb0);
                if (!have && lane == 0 && !*abortp) fail(64u);
                const int u = (grp - (int)(cb & 3)) & 3;  // this group's K-block of the unit, if any
                const uint32_t c = cb + (uint32_t)u;
                const int st = (int)(c & (kStages - 1));
                const uint32_t arow = arow0 + st * kABytes;
                uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
                uint32_t w = 0;
                if (have && u < nu) {
                    const uint32_t raw_s = ptx::smem_addr(ringR + r * kRawBytes);
                    c0 = ptx::lds_u4(raw_s + codes_off + u * codes_step);
                    c1 = ptx::lds_u4(raw_s + codes_off + codes_hh + u * codes_step);
                    w = ptx::lds_u32(raw_s + sb_off + u * sb_step);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(raw_empty + r);
                if (u < nu) {
                    const bool free_a = have && ptx::mbar_wait_sleep(a_empty + st, ((c >> kStageShift) & 1) ^ 1, abortp);
                    if (free_a) {
                        const __half2 s2 = __half2half2(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
                        const __half2 b2 = __half2half2(__ushort_as_half((unsigned short)(w >> 16)));
                        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                        for (int q = 0; q < 8; ++q)  // 16-byte chunk q of the 128-byte row
                            ptx::sts_u4(arow + ((q ^ swz) << 4), dequant8(words[q], s2, b2));
                        ptx::fence_proxy_async_smem();
                    } else if (have && lane == 0) {
                        record(8, j, kb0 + u);
                        if (!*abortp) fail(64u);
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(a_full + st);
                }
                cb += (uint32_t)nu;
                if (++r == kRawStages) {
                    r = 0;
                    rph ^= 1;
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// The K-split tiles' epilogue: block (t, y) takes split tile t (family 0's
// first) and columns 16y .. 16y + 15, thread r row r of the tile; it adds the
// tile's parts in part order and writes h (gate/up) or the outputs (down)
// exactly as the GEMM's epilogue does for a whole tile.
__global__ void __launch_bounds__(kTileM) pf_reduce_kernel(const __grid_constant__ PfArgs a, const int phase) {
    const Plan P = make_plan(a, phase);
    const int row = threadIdx.x, lane = row & 31, q = row >> 5;
    const int n0 = P.ks[0] > 1 ? a.n_fam0 * P.tiles[0] : 0;
    int t = blockIdx.x, fam, item, tile, ks;
    size_t part0;
    if (t < n0) {
        fam = 0;
        item = t / P.tiles[0];
        tile = t - item * P.tiles[0];
        ks = P.ks[0];
        part0 = (size_t)t * ks;
    } else {
        t -= n0;
        fam = 1;
        const int i = t / P.tiles[1];
        tile = t - i * P.tiles[1];
        item = a.n_fam0 + i;
        ks = P.ks[1];
        part0 = (size_t)n0 * P.ks[0] + (size_t)t * ks;
    }
    const PfItem it = a.items[item];
    const int c = blockIdx.y * 16;
    if (c >= it.np) return;  // the whole block
    const size_t stride = (size_t)kPfMaxN * kTileM;
    const float* src = a.part + part0 * stride + (size_t)c * kTileM + row;
    float v[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) v[m] = src[(size_t)m * kTileM];
    for (int pp = 1; pp < ks; ++pp) {
        const float* sp = src + pp * stride;
        float w[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) w[m] = sp[(size_t)m * kTileM];
#pragma unroll
        for (int m = 0; m < 16; ++m) v[m] += w[m];
    }
    if (phase == 1) {
        const int I = a.inter[fam];
        const int irow = 64 * tile + 16 * q + (lane >> 1);
        __half* hb = a.h[fam];
        const bool odd = lane & 1;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const float mine = odd ? v[m + 8] : v[m];
            const float other = __shfl_xor_sync(kFull, odd ? v[m] : v[m + 8], 1);
            const float g = odd ? other : mine, u = odd ? mine : other;
            const int col = c + m + (odd ? 8 : 0);
            if (col < it.np) hb[(size_t)(it.pb + col) * I + irow] = __float2half_rn(act_fn(g, a.act) * u);
        }
    } else {
        const int n = kTileM * tile + row;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int col = c + m;
            if (col >= it.np) break;
            const size_t orow = fam == 0 ? (size_t)(it.pb + col) : (size_t)a.pair[it.pb + col];
            a.out[fam][orow * a.d + n] = v[m];
        }
    }
}

__global__ void pf_gather_kernel(const uint16_t* __restrict__ x, int T, int d, const int32_t* __restrict__ pair,
                                 int P, int k, __half* __restrict__ xs, __half* __restrict__ xg) {
    const int per_row = d / 8;
    const long n = (long)(T + P) * per_row;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int r = (int)(i / per_row), c = (int)(i - (long)r * per_row);
        const int tok = r < T ? r : pair[r - T] / k;
        const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)tok * d + c * 8);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float lo = __uint_as_float(w[m] << 16), hi = __uint_as_float(w[m] & 0xffff0000u);
            o[m] = as_u32(__floats2half2_rn(lo, hi));
        }
        __half* dst = r < T ? xs + (size_t)r * d : xg + (size_t)(r - T) * d;
        *reinterpret_cast<uint4*>(dst + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// fp16 [rows][cols] row-major, boxes of 64 columns x box_rows rows, 128-byte swizzle.
// fp16 [rows][cols] row-major seen as [cols / 64][rows][64]: boxes of 64
// columns x box_rows rows x box_kb K-blocks, 128-byte swizzle.
cudaError_t encode_rows3(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_kb) {
    EncodeTiled fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if ((reinterpret_cast<uintptr_t>(base) & 15) || cols % 64 || rows < 1) return cudaErrorInvalidValue;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_kb};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_rows(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
    EncodeTiled fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if ((reinterpret_cast<uintptr_t>(base) & 15) || cols % 64 || rows < 1) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

// K parts of a tile of `kblocks` K-blocks when a launch has `tiles` tiles in
// all: enough to give every SM a job, at most 8 and at least 4 K-blocks each.
// A launch with at least half as many tiles as SMs is not split (its tiles
// already fill the GPU, and the split costs a second launch).
int pf_split(int tiles, int kblocks) {
    if (2 * tiles >= num_sms()) return 1;
    int s = num_sms() / std::max(tiles, 1);
    s = std::min(s, 8);
    s = std::min(s, kblocks / 4);
    return std::max(s, 1);
}

}  // namespace

// pf_split keeps a launch's tiles x parts within the SM count.
size_t pf_part_floats(int d, int inter0) {
    (void)d;
    (void)inter0;
    return (size_t)num_sms() * kTileM * kPfMaxN;
}

cudaError_t launch_pf_gather(const uint16_t* x, int T, int d, const int32_t* pair, int P, int k, __half* xs,
                             __half* xg, cudaStream_t s) {
    const long n = (long)(T + P) * (d / 8);
    const int blocks = (int)std::min<long>((n + 255) / 256, 4L * num_sms());
    pf_gather_kernel<<<blocks, 256, 0, s>>>(x, T, d, pair, P, k, xs, xg);
    return cudaGetLastError();
}

cudaError_t launch_pf_gemm(const PfArgs& a, int phase, const void* b0, const void* b1, const int rows[2],
                           cudaStream_t s, int* launched) {
    if ((phase != 1 && phase != 2) || a.n_items < 1 || a.n_fam0 < 0 || a.n_fam0 > a.n_items || a.d % kTileM ||
        a.inter[0] % 64 || a.inter[1] % 64)
        return cudaErrorInvalidValue;
    CUtensorMap m0;
    const int k0 = phase == 1 ? a.d : a.inter[0], k1 = phase == 1 ? a.d : a.inter[1];
    // family 0 is the shared expert over every token row: one item per block
    // of kPfMaxN tokens (a single one loads all its rows as one box)
    if (rows[0] != a.T || a.T < 1 || a.n_fam0 != (a.T + kPfMaxN - 1) / kPfMaxN) return cudaErrorInvalidValue;
    const int box0 = a.n_fam0 > 1 ? kPfMaxN : a.T <= 16 ? 16 : (a.T + 15) & ~15;
    cudaError_t e = encode_rows(&m0, b0, rows[0], k0, box0);
    // the chunk layout when the routed experts average at most 24 rows
    const int n_routed = a.n_items - a.n_fam0;
    const bool chunk = (long)rows[1] <= 24L * n_routed;
    PfRowMaps rm{};
    if (chunk)
        for (int q = 0; q < 4 && e == cudaSuccess; ++q)
            e = encode_rows3(&rm.r[q], b1, std::max(rows[1], 1), k1, 16 << q, std::min(8 >> q, k1 / 64));
    else if (e == cudaSuccess)
        for (int q = 4; q < 7 && e == cudaSuccess; ++q)
            e = encode_rows(&rm.r[q], b1, std::max(rows[1], 1), k1, q == 4 ? 16 : q == 5 ? 64 : 128);
    if (e == cudaSuccess)
        e = chunk ? ensure_smem_attr((const void*)pf_gemm_kernel<RingsChunk>, RingsChunk::kSmemBytes)
                  : ensure_smem_attr((const void*)pf_gemm_kernel<RingsPrompt>, RingsPrompt::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int tiles0 = phase == 1 ? a.inter[0] / 64 : a.d / kTileM;
    const int tiles1 = phase == 1 ? a.inter[1] / 64 : a.d / kTileM;
    // K splits when the launch's tiles are too few to fill the GPU (the shared
    // expert alone has 44 or 22); a family whose parts would not fit the
    // buffer is not split
    PfArgs b = a;
    const int n_t[2] = {a.n_fam0 * tiles0, (a.n_items - a.n_fam0) * tiles1};
    const int kb[2] = {phase == 1 ? a.d / 64 : a.inter[0] / 64, phase == 1 ? a.d / 64 : a.inter[1] / 64};
    size_t parts = 0;
    int split_tiles = 0;
    for (int f = 0; f < 2; ++f) {
        b.ks[f] = a.part ? pf_split(n_t[0] + n_t[1], kb[f]) : 1;
        if (b.ks[f] > 1 && (parts + (size_t)n_t[f] * b.ks[f]) * kTileM * kPfMaxN > a.part_cap) b.ks[f] = 1;
        if (b.ks[f] > 1) {
            parts += (size_t)n_t[f] * b.ks[f];
            split_tiles += n_t[f];
        }
    }
    const int jobs = n_t[0] * b.ks[0] + n_t[1] * b.ks[1];
    const int grid = std::min(jobs, num_sms());
    if (chunk)
        pf_gemm_kernel<RingsChunk><<<grid, kThreads, RingsChunk::kSmemBytes, s>>>(b, phase, m0, rm);
    else
        pf_gemm_kernel<RingsPrompt><<<grid, kThreads, RingsPrompt::kSmemBytes, s>>>(b, phase, m0, rm);
    if (launched) *launched = 1;
    if (split_tiles > 0) {
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        pf_reduce_kernel<<<dim3(split_tiles, kPfMaxN / 16), kTileM, 0, s>>>(b, phase);
        if (launched) *launched = 2;
    }
    return cudaGetLastError();
}

}  // namespace moe
