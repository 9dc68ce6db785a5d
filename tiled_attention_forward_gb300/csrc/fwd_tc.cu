// fwd_tc.cu -- tensor-core attention forward for bf16 / fp16 on sm_103a.
//
// FlashAttention-2 structure (dandandamowang.xyz "Flash Attention (二) v2"
// page, §1.1-§1.4: Q tile outer, K/V tiles inner, running max/sum on chip,
// deferred 1/l, causal block skip + diagonal element mask), mapped onto
// Blackwell's tensor-core machinery in the way the hjcheng0602.cn
// "flashattn_G7" page describes for SM103 (1-CTA tcgen05, S and O in TMEM,
// P.V issued in the TS form with P in TMEM, V landed by TMA directly in the
// MN-major 128-byte-swizzled operand layout, persistent CTAs).
//
// One CTA per SM, persistent over tasks.  A task is one (batch*head, 256-row
// Q block): two 128-row Q tiles that share every K/V tile the CTA streams.
// CTAs take tasks from a per-launch counter as they run out of work
// (causal problems: heads in L2-sized groups, longest Q blocks first).
//
// Warp roles (384 threads = three warpgroups):
//   warps 0-3  softmax warpgroup 0: Q tile 0, thread t owns query row t
//              (TMEM lane t): S row and its max (one reducing TMEM load,
//              tcgen05.ld.red) -> mask -> exp2 -> P (16-bit) into
//              TMEM, conditional O rescale, epilogue (O/l, LSE, store)
//   warps 4-7  softmax warpgroup 1: same for Q tile 1
//   warp 8     MMA issue (one elected lane): S_i = Q_i K_j^T (SS form),
//              O_i += P_i V_j (TS form), tcgen05.commit -> mbarriers
//   warp 9     TMA producer (one elected lane): takes the CTA's next task
//              and publishes it to the other roles (task ring), Q tiles
//              once per task, K/V tiles through a ring of shared-memory stages
//   warp 10    the MMA warp's helper: does the MMA warp's barrier waits and
//              releases it on a named barrier
//   warp 11    idle
// The control warpgroup (warps 8-11) gives up registers (setmaxnreg) so the
// softmax warpgroups can hold a whole 128-score row per thread: 168 per
// thread at launch; 2 x 128 x kSoftmaxRegs + 128 x kControlRegs <= 384 x 168.
//
// TMEM (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256),
// O_0 [256,256+D), O_1 [256+D,256+2D).  P_i (two 16-bit values per column)
// overwrites the first 64 columns of S_i once its scores are in registers.
//
// MMA issue order per K/V tile j (tensor-core instructions of one CTA execute
// in issue order):  PV_0(j), S_0(j+1), PV_1(j), S_1(j+1).  So while softmax
// warpgroup 0 works on S_0(j+1), the tensor core runs PV_1(j) and S_1(j+1),
// and vice versa.  A commit after S_i(j+1) fires only once PV_i(j) is done,
// which is what lets the softmax warpgroup rescale O_i right after it sees
// S_i(j+1).
//
// That is the D = 128 layout.  At D = 64 the TMEM has room for a third S
// buffer, and the two tiles rotate through three buffers so that a tile's
// next scores are computed while its softmax still works on the current
// ones (mma_pair_role_rot below; softmax_role serves both layouts).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace fattn {

// Bit k set <=> a kernel on this device hit fattn_status k (only TIMEOUT today).
__device__ uint32_t g_error_word;

// Task counters of the persistent grid.  CTAs take their first task by
// index and every later one from a counter; a launch uses the slot its
// %gridid (the context's launch number, new for every launch, graph replays
// included) selects, so launches running at the same time use different
// slots unless 65536 other grids were launched on the context in between,
// and the last CTA to finish sets the slot back to zero.
//   [0]: tasks handed out beyond the first gridDim.x; [1]: CTAs finished.
constexpr uint32_t kSchedSlots = 1u << 16;
__device__ uint32_t g_sched[kSchedSlots][2];

namespace {

constexpr uint32_t kSoftmaxRegs = 216;
constexpr uint32_t kControlRegs = 72;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kTcThreads * 168,
              "register split must fit the launch allocation");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 2^8 while the max is stale
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct TcLayout {
    static constexpr int kAtoms = D / 64;               // 128-byte swizzle atoms along D
    static constexpr int kAtomRowBytes = 128;           // 64 x 16-bit
    static constexpr int kQTileBytes = kTcBM * D * 2;
    static constexpr int kKVTileBytes = kTcBN * D * 2;
    static constexpr int kStages = (D == 128) ? 5 : 8;  // K/V ring depth
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = kTcQTiles * kQTileBytes;
    static constexpr int kBarOff = kKVOff + kStages * kKVTileBytes;
    // D = 128: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] o_full[2] drain[1]
    // D = 64 (three S buffers): ... s_full[3][2] o_full[2] o_ready[2] drain[1]
    // (P is handed to the MMA warp on named barriers, see kPBar; the task
    // ring's words and barriers follow the misc words, see TaskRing.)
    static constexpr bool kRot = (D == 64);
    static constexpr int kSFull = kRot ? 6 : 2;
    static constexpr int kNumBars = 2 + 2 + 2 * kStages + kSFull + 2 + (kRot ? 2 : 0) + 1;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;   // TMEM base, abort flag
    static constexpr int kTaskOff = kMiscOff + 16;            // the task ring (TaskRing)
    static constexpr int kBytes = kTaskOff + 3 * 4 * 8;
    static constexpr int kAlloc = kBytes;  // the dynamic base is declared 1024-byte aligned
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kAlloc <= 227 * 1024, "shared memory budget");
    // The MMA warp holds two ring slots (V_j, K_{j+1}) until the end of an
    // iteration and then needs V_{j+1} and K_{j+2}: four slots at least.
    static_assert(kStages >= 4, "K/V ring depth");
    static_assert((kRot ? 384 : 256) + 2 * D <= 512, "TMEM budget");
};

struct Task {
    int bh;
    int q0;
    int nb[2];  // K/V tiles visited by Q tile 0 / 1 (0: tile has no valid row)
    int nbmax;
};

// Task order: non-causal, head-major (all Q blocks of one head are adjacent so
// concurrently running CTAs share that head's K/V in L2).  Causal: heads in
// groups of a.head_group (their K/V fits in L2 together), and within a group
// longest first: Q blocks nearest the end of the sequence (most K/V tiles)
// first, heads inner.  CTAs pull tasks in this order from a counter, so the
// short tasks at the end of the last group fill in the tail.
template <bool CAUSAL, bool EQUAL = false>
__device__ __forceinline__ Task decode_task(int t, const TcArgs& a) {
    Task k;
    int qblk;
    if (CAUSAL) {
        const int per_group = a.head_group * a.num_qblk;
        const int g = t / per_group;
        const int r = t - g * per_group;
        const int gsize = min(a.head_group, a.BH - g * a.head_group);
        qblk = a.num_qblk - 1 - r / gsize;
        k.bh = g * a.head_group + r % gsize;
    } else {
        qblk = t % a.num_qblk;
        k.bh = t / a.num_qblk;
    }
    k.q0 = qblk * (kTcBM * kTcQTiles);
    const int all = (a.N + kTcBN - 1) / kTcBN;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r0 = k.q0 + i * kTcBM;  // first row of tile i
        if (r0 >= a.N) {
            k.nb[i] = 0;
        } else if (CAUSAL) {
            const int kv_limit = min(r0 + kTcBM, a.N);  // keys beyond the tile's last row are never visible
            k.nb[i] = (kv_limit + kTcBN - 1) / kTcBN;
        } else {
            k.nb[i] = all;
        }
    }
    k.nbmax = max(k.nb[0], k.nb[1]);
    if (EQUAL) {
        // Both tiles visit nbmax blocks: under causal masking tile 0's extra
        // block lies wholly above its diagonal (every score masked, P = 0),
        // and a tile 1 past N computes rows that are never stored.
        k.nb[0] = k.nbmax;
        k.nb[1] = k.nbmax;
    }
    return k;
}

// The counter slot of this launch.
__device__ __forceinline__ uint32_t* sched_slot() {
    uint64_t id;
    asm volatile("mov.u64 %0, %%gridid;" : "=l"(id));
    return g_sched[id & (kSchedSlots - 1u)];
}

// The CTA's tasks go from the producer warp to the other roles through a
// ring of kTaskRing shared-memory words, each with a "published" and a "read
// by every reader" mbarrier.
// Word kt % kTaskRing holds (kt << 32) | task once the CTA's kt-th task is
// known; a task >= num_tasks ends the schedule.  Every role that meets
// another on a named barrier must see the same sequence (named-barrier waits
// are unbounded, see kPBar), also when a wait gives up: a reader whose wait
// for word kt gave up writes "end" into it with a compare-and-swap, the
// producer publishes with a compare-and-swap too, and whichever lands first
// is what every reader of the word gets.
constexpr int kTaskRing = 4;
constexpr uint32_t kTaskReaders = 8 + 1;  // the softmax warps, the issuing warp
constexpr uint32_t kEndOfSchedule = 0x7fffffffu;

// One shared-memory address locates the ring (a single register in the
// softmax warps, which hold a whole score row): kTaskRing words, then their
// "published" mbarriers, then their "read by every reader" mbarriers.
struct TaskRing {
    uint32_t base;
    __device__ __forceinline__ unsigned long long* word(int s) const {
        return static_cast<unsigned long long*>(__cvta_shared_to_generic(base + 8u * s));
    }
    __device__ __forceinline__ uint64_t* full(int s) const {
        return static_cast<uint64_t*>(__cvta_shared_to_generic(base + 8u * (kTaskRing + s)));
    }
    __device__ __forceinline__ uint64_t* empty(int s) const {
        return static_cast<uint64_t*>(__cvta_shared_to_generic(base + 8u * (2 * kTaskRing + s)));
    }
};

struct Bars {
    uint64_t* q_full;
    uint64_t* q_empty;
    uint64_t* kv_full;
    uint64_t* kv_empty;
    uint64_t* s_full;
    uint64_t* o_full;
    uint64_t* o_ready;  // D = 64: [tile], one phase per completed P.V product
    uint64_t* drain;
    TaskRing tasks;
};

template <int D>
__device__ __forceinline__ Bars carve_bars(uint8_t* smem) {
    using L = TcLayout<D>;
    uint64_t* b = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    Bars r;
    r.q_full = b;
    r.q_empty = b + 2;
    r.kv_full = b + 4;
    r.kv_empty = r.kv_full + L::kStages;
    r.s_full = r.kv_empty + L::kStages;
    r.o_full = r.s_full + L::kSFull;
    r.o_ready = r.o_full + 2;
    r.drain = r.o_ready + (L::kRot ? 2 : 0);
    r.tasks.base = smem_u32(smem + L::kTaskOff);
    return r;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// Every lane of a warp waits; the outcome is made warp-uniform so that the
// warp's control flow never diverges on a wait that gave up.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          volatile uint32_t* abort_flag, uint64_t timeout_ns) {
    return __all_sync(0xffffffffu,
                      mbar_wait_bounded(bar, parity, abort_flag, &g_error_word, timeout_ns));
}

__device__ __forceinline__ unsigned long long ring_word(int kt, uint32_t t) {
    return (static_cast<unsigned long long>(static_cast<uint32_t>(kt)) << 32) | t;
}
__device__ __forceinline__ unsigned long long ring_peek(const TaskRing& r, int kt) {
    return *reinterpret_cast<volatile unsigned long long*>(r.word(kt % kTaskRing));
}

// The CTA's kt-th task (whole warp; >= num_tasks: the schedule ended).
__device__ __forceinline__ int read_task(const TaskRing& r, int kt, volatile uint32_t* abort_flag,
                                         uint64_t timeout_ns) {
    const int slot = kt % kTaskRing;
    const bool arrived = warp_wait(r.full(slot), (kt / kTaskRing) & 1, abort_flag, timeout_ns);
    uint32_t t = 0u;
    if ((threadIdx.x % 32) == 0) {
        unsigned long long cur = ring_peek(r, kt);
        if (!arrived && (cur >> 32) != static_cast<uint32_t>(kt)) {
            const unsigned long long end = ring_word(kt, kEndOfSchedule);
            const unsigned long long prev = atomicCAS(r.word(slot), cur, end);
            cur = (prev == cur) ? end : prev;
        }
        t = static_cast<uint32_t>(cur);
    }
    return static_cast<int>(__shfl_sync(0xffffffffu, t, 0));
}
// A reader is done with word kt (the producer may reuse it for task kt + kTaskRing).
__device__ __forceinline__ void release_task(const TaskRing& r, int kt) {
    __syncwarp();
    if ((threadIdx.x % 32) == 0) mbar_arrive(r.empty(kt % kTaskRing));
    __syncwarp();
}

// ---------------------------------------------------------------------------
// TMA producer (one warp; one elected lane issues the copies)
// ---------------------------------------------------------------------------
template <int D, bool CAUSAL>
__device__ void producer_role(const TcArgs& a, uint8_t* smem, const Bars& bars,
                              volatile uint32_t* abort_flag) {
    using L = TcLayout<D>;
    uint32_t kv_it = 0;
    uint32_t qcnt[2] = {0u, 0u};
    bool ok = true;
    const uint64_t keep = l2_policy_evict_last();   // K/V: re-read by the other Q blocks of the head
    const uint64_t once = l2_policy_evict_first();  // Q: read once

    auto load_q = [&](int i, const Task& tk) {
        ok = warp_wait(&bars.q_empty[i], (qcnt[i] & 1u) ^ 1u, abort_flag, a.timeout_ns);
        if (!ok) return;
        if (elect_one_sync()) {
            mbar_arrive_expect_tx(&bars.q_full[i], L::kQTileBytes);
            uint8_t* dst = smem + L::kQOff + i * L::kQTileBytes;
#pragma unroll
            for (int at = 0; at < L::kAtoms; ++at)
                tma_load_3d_hint(dst + at * kTcBM * L::kAtomRowBytes, &a.tmap_q, &bars.q_full[i],
                                 at * 64, tk.q0 + i * kTcBM, tk.bh, once);
        }
        __syncwarp();
        ++qcnt[i];
    };
    auto load_kv = [&](const CUtensorMap* map, int j, int kvh) {
        const uint32_t slot = kv_it % L::kStages;
        const uint32_t round = kv_it / L::kStages;
        ok = warp_wait(&bars.kv_empty[slot], (round & 1u) ^ 1u, abort_flag, a.timeout_ns);
        if (!ok) return;
        if (elect_one_sync()) {
            mbar_arrive_expect_tx(&bars.kv_full[slot], L::kKVTileBytes);
            uint8_t* dst = smem + L::kKVOff + slot * L::kKVTileBytes;
#pragma unroll
            for (int at = 0; at < L::kAtoms; ++at)
                tma_load_3d_hint(dst + at * kTcBN * L::kAtomRowBytes, map, &bars.kv_full[slot],
                                 at * 64, j * kTcBN, kvh, keep);
        }
        __syncwarp();
        ++kv_it;
    };

    uint32_t* ctr = sched_slot();
    // Publish task t as the CTA's kt-th.  False: the wait for a free word
    // gave up, or a reader has already ended the schedule there.
    auto publish = [&](int kt, int t) -> bool {
        const int slot = kt % kTaskRing;
        if (kt >= kTaskRing &&
            !warp_wait(bars.tasks.empty(slot), ((kt / kTaskRing) - 1) & 1, abort_flag, a.timeout_ns))
            return false;
        uint32_t won = 0u;
        if ((threadIdx.x % 32) == 0) {
            const unsigned long long cur = ring_peek(bars.tasks, kt);
            if ((cur >> 32) != static_cast<uint32_t>(kt)) {
                won = atomicCAS(bars.tasks.word(slot), cur, ring_word(kt, static_cast<uint32_t>(t))) == cur;
                if (won) mbar_arrive(bars.tasks.full(slot));
            }
        }
        return __shfl_sync(0xffffffffu, won, 0) != 0u;
    };
    // The next task from this launch's counter (the first gridDim.x tasks
    // are the CTAs' own first ones).
    auto fetch = [&]() -> int {
        uint32_t v = 0u;
        if ((threadIdx.x % 32) == 0) v = atomicAdd(&ctr[0], 1u);
        v = __shfl_sync(0xffffffffu, v, 0);
        return static_cast<int>(gridDim.x + min(v, static_cast<uint32_t>(a.num_tasks)));
    };

    int t = static_cast<int>(blockIdx.x);
    for (int kt = 0; ok; ++kt) {
        if (t >= a.num_tasks) {
            publish(kt, static_cast<int>(kEndOfSchedule));
            break;
        }
        if (!publish(kt, t)) break;
        const Task tk = decode_task<CAUSAL, L::kRot>(t, a);
        const int kvh = kv_head_of(tk.bh, a.H, a.Hkv);
        load_q(0, tk);
        if (!ok) break;
        load_kv(&a.tmap_k, 0, kvh);
        if (!ok) break;
        if (tk.nb[1] > 0) {
            load_q(1, tk);
            if (!ok) break;
        }
        for (int j = 0; j < tk.nbmax && ok; ++j) {
            load_kv(&a.tmap_v, j, kvh);
            if (ok && j + 1 < tk.nbmax) load_kv(&a.tmap_k, j + 1, kvh);
        }
        if (!ok) break;
        // The next task is taken only now, a few K/V tiles before this CTA
        // runs out of work, so that the tasks still left go to the CTAs that
        // become free first.  Its Q tiles are read once, from DRAM, and their
        // loads can only start when this task's last score products are
        // done; fetched into L2 now, they land in shared memory at L2 latency.
        t = fetch();
        if (t < a.num_tasks && elect_one_sync()) {
            const Task nx = decode_task<CAUSAL, L::kRot>(t, a);
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (nx.q0 + i * kTcBM < a.N)
#pragma unroll
                    for (int at = 0; at < L::kAtoms; ++at)
                        tma_prefetch_3d(&a.tmap_q, at * 64, nx.q0 + i * kTcBM, nx.bh);
        }
        __syncwarp();
    }

    // Drain: every bulk copy this warp started has landed before the CTA can
    // retire (matters only when a wait gave up above).
    for (uint32_t s = 0; s < (uint32_t)L::kStages && s < kv_it; ++s) {
        const uint32_t last = s + ((kv_it - 1u - s) / L::kStages) * L::kStages;
        warp_wait(&bars.kv_full[s], (last / L::kStages) & 1u, nullptr, a.timeout_ns);
    }
    for (int i = 0; i < 2; ++i)
        if (qcnt[i] > 0u) warp_wait(&bars.q_full[i], (qcnt[i] - 1u) & 1u, nullptr, a.timeout_ns);
}

// ---------------------------------------------------------------------------
// MMA issue, two-buffer layout (D = 128): an issuing warp and its helper warp
// ---------------------------------------------------------------------------
// A barrier test (a shared-memory access) made by the warp that has just
// issued MMAs waits until those MMAs are taken by the tensor pipe, so every
// wait between two MMA groups left the pipe idle for the wake-up.  Here the
// issuing warp never touches a barrier inside its loop: a helper warp runs
// the same schedule, does every mbarrier wait, and meets the issuing warp on
// a named barrier (kMmaSync) before each group that depends on a wait.  The
// named barrier reduces the helper's "every wait succeeded" flag, so both
// warps leave the schedule at the same point when a wait gives up.
constexpr uint32_t kMmaSync = 1;          // named barrier id (0 is __syncthreads)
constexpr uint32_t kMmaSyncThreads = 64;  // the issuing warp and its helper
// P of Q tile i, K/V block j is handed from softmax warpgroup i to the
// issuing warp on named barrier kPBar + 2 i + (j & 1): the warpgroup arrives
// (no wait), the issuing warp waits.  A warpgroup can finish the P of the
// next block before the issuing warp has taken the current one (its next
// scores may already be computed), never the one after, so two barriers per
// tile alternate.  Ids 2..5.
constexpr uint32_t kPBar = 2;
constexpr uint32_t kPBarThreads = 128 + 32;  // one softmax warpgroup and the issuing warp

// Every wait on a named barrier is unbounded, so on an abort (an mbarrier
// wait that gave up) no role leaves early: each runs the rest of its
// schedule "dry" -- no mbarrier waits, MMAs, TMEM traffic or stores -- and
// still passes every named barrier, so that every named-barrier wait is met.
__device__ __forceinline__ uint32_t p_bar(int tile, int j) {
    return kPBar + 2u * static_cast<uint32_t>(tile) + (static_cast<uint32_t>(j) & 1u);
}

template <int D, bool BF16, bool CAUSAL, bool HELPER>
__device__ void mma_pair_role(const TcArgs& a, uint8_t* smem, const Bars& bars, uint32_t tmem_base,
                              volatile uint32_t* abort_flag) {
    using L = TcLayout<D>;
    static_assert(!L::kRot, "the three-buffer layout has its own MMA role");
    constexpr uint32_t kIdescQK = idesc_f16_f32(kTcBM, kTcBN, BF16 ? 1u : 0u, 0u, 0u);
    constexpr uint32_t kIdescPV = idesc_f16_f32(kTcBM, D, BF16 ? 1u : 0u, 0u, 1u);
    const uint32_t q_smem = smem_u32(smem + L::kQOff);
    const uint32_t kv_smem = smem_u32(smem + L::kKVOff);

    uint32_t kv_it = 0;               // ring positions consumed (both warps count alike)
    uint32_t qcnt[2] = {0u, 0u};
    bool ok = true;                   // false: dry run (see kPBar)

    // The helper's waits; the issuing warp only advances the same counters.
    auto wait_kv = [&](uint32_t& slot) {
        slot = kv_it % L::kStages;
        if (HELPER && ok)
            ok = warp_wait(&bars.kv_full[slot], (kv_it / L::kStages) & 1u, abort_flag, a.timeout_ns);
        ++kv_it;
    };
    auto wait_q = [&](int i) {
        if (HELPER && ok) ok = warp_wait(&bars.q_full[i], qcnt[i] & 1u, abort_flag, a.timeout_ns);
    };
    // Both warps pass here together; false (from then on) once a wait of the
    // helper gave up.
    auto sync = [&]() {
        ok = named_barrier_and(kMmaSync, kMmaSyncThreads, ok);
        if (!HELPER) tc_fence_after();
    };
    // The issuing warp takes P of tile i, block j from its softmax warpgroup.
    auto take_p = [&](int i, int j) {
        if (!HELPER) {
            named_barrier_sync(p_bar(i, j), kPBarThreads);
            tc_fence_after();
        }
    };
    // The CTA's kt-th task: the helper waits for it, the issuing warp reads
    // the same word after their meeting (also in a dry run).
    auto next_task = [&](int kt) -> int {
        int t = 0;
        if (HELPER) t = read_task(bars.tasks, kt, abort_flag, a.timeout_ns);
        sync();
        if (!HELPER) {
            t = static_cast<int>(static_cast<uint32_t>(ring_peek(bars.tasks, kt)));
            release_task(bars.tasks, kt);
        }
        return t;
    };

    // Descriptor templates with a zero start address.  A tile's descriptor is
    // the template plus (shared address >> 4): the start-address field is the
    // low 14 bits and every shared address is below 256 KB, so the add never
    // carries.  Per-MMA steps are compile-time offsets on top, which keeps the
    // issue loop to one 64-bit add per operand.
    const uint64_t kmaj_desc = smem_desc_sw128(0u, 16u, 1024u);             // Q, K: K-major
    const uint64_t vmn_desc = smem_desc_sw128(0u, kTcBN * 128u, 1024u);     // V: MN-major
    // S_i = Q_i K^T : M=128 rows, N=128 keys, K=D in steps of 16 (32 bytes
    // inside a 128-byte swizzle row; a new atom every 64 elements).
    auto issue_qk = [&](int i, uint32_t kslot) {
        const uint64_t adesc = kmaj_desc + ((q_smem + i * L::kQTileBytes) >> 4);
        const uint64_t bdesc = kmaj_desc + ((kv_smem + kslot * L::kKVTileBytes) >> 4);
        const uint32_t d_tmem = tmem_base + i * kTcBN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            constexpr uint32_t kAtomQ = kTcBM * 128, kAtomK = kTcBN * 128;
            const uint64_t off_q = ((kk / 4) * kAtomQ + (kk % 4) * 32) >> 4;
            const uint64_t off_k = ((kk / 4) * kAtomK + (kk % 4) * 32) >> 4;
            mma_ss(d_tmem, adesc + off_q, bdesc + off_k, kIdescQK, kk > 0 ? 1u : 0u);
        }
    };
    // O_i (+)= P_i V : A = P_i from TMEM (8 columns per 16 keys), B = V tile,
    // MN-major: 64-wide feature slabs of kTcBN rows x 128 bytes (leading
    // offset = slab size), 8-key groups 1024 bytes apart (stride offset).
    auto issue_pv = [&](int i, uint32_t vslot, bool accumulate) {
        const uint64_t bdesc = vmn_desc + ((kv_smem + vslot * L::kKVTileBytes) >> 4);
        const uint32_t d_tmem = tmem_base + 2 * kTcBN + i * D;
        const uint32_t a_tmem = tmem_base + i * kTcBN;
#pragma unroll
        for (int kk = 0; kk < kTcBN / 16; ++kk)
            mma_ts(d_tmem, a_tmem + kk * 8, bdesc + ((kk * 16 * 128) >> 4), kIdescPV,
                   (accumulate || kk > 0) ? 1u : 0u);
    };
    // S_i(j) with its signals (j = the K/V block of the score tile).
    auto qk_group = [&](int i, uint32_t kslot, int j, const Task& tk) {
        if (!HELPER && ok) {
            if (elect_one_sync()) {
                issue_qk(i, kslot);
                mma_commit(&bars.s_full[i]);
                if (j == tk.nb[i] - 1) mma_commit(&bars.q_empty[i]);
            }
            __syncwarp();
        }
    };
    auto pv_group = [&](int i, uint32_t vslot, int j, const Task& tk) {
        if (!HELPER && ok) {
            if (elect_one_sync()) {
                issue_pv(i, vslot, j > 0);
                if (j == tk.nb[i] - 1) mma_commit(&bars.o_full[i]);
            }
            __syncwarp();
        }
    };

    for (int kt = 0;; ++kt) {
        const int t = next_task(kt);
        if (t >= a.num_tasks) break;
        const Task tk = decode_task<CAUSAL>(t, a);
        uint32_t kslot, vslot;
        // Prologue: S_0(0), S_1(0).
        wait_q(0);
        wait_kv(kslot);  // K_0
        sync();
        qk_group(0, kslot, 0, tk);
        if (tk.nb[0] == 1) ++qcnt[0];
        if (tk.nb[1] > 0) {
            wait_q(1);
            sync();
            qk_group(1, kslot, 0, tk);
            if (tk.nb[1] == 1) ++qcnt[1];
        }
        if (!HELPER && ok) {
            if (elect_one_sync()) mma_commit(&bars.kv_empty[kslot]);
            __syncwarp();
        }

        // Per K/V tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1).  The tensor
        // core runs one tile's P.V and next scores while the other tile's
        // softmax works.  V_j and K_{j+1} are waited for together: K_{j+1}
        // lands right after V_j, and one meeting per block is cheaper.
        for (int j = 0; j < tk.nbmax; ++j) {
            const bool has_next = j + 1 < tk.nbmax;
            wait_kv(vslot);                  // V_j
            if (has_next) wait_kv(kslot);    // K_{j+1}
            sync();
            if (j < tk.nb[0]) {
                take_p(0, j);
                pv_group(0, vslot, j, tk);
            }
            if (j + 1 < tk.nb[0]) {
                qk_group(0, kslot, j + 1, tk);
                if (j + 1 == tk.nb[0] - 1) ++qcnt[0];
            }
            if (j < tk.nb[1]) {
                take_p(1, j);
                pv_group(1, vslot, j, tk);
            }
            if (j + 1 < tk.nb[1]) {
                qk_group(1, kslot, j + 1, tk);
                if (j + 1 == tk.nb[1] - 1) ++qcnt[1];
            }
            // V_j and K_{j+1} are released once every MMA issued so far is done.
            if (!HELPER && ok) {
                if (elect_one_sync()) {
                    mma_commit(&bars.kv_empty[vslot]);
                    if (has_next) mma_commit(&bars.kv_empty[kslot]);
                }
                __syncwarp();
            }
        }
    }

    if (!HELPER) {
        // Drain: every MMA issued above has completed before TMEM is released.
        if (elect_one_sync()) mma_commit(bars.drain);
        __syncwarp();
        warp_wait(bars.drain, 0u, nullptr, a.timeout_ns);
    }
}

// ---------------------------------------------------------------------------
// Softmax + correction + epilogue (one warpgroup per Q tile)
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// D = 64: three S buffers shared by the two Q tiles
// ---------------------------------------------------------------------------
// At D = 64 the TMEM holds three 128-column S buffers next to the two O
// accumulators (3 x 128 + 2 x 64 = 512 columns).  Both Q tiles of a task visit
// the same nb blocks (decode_task<CAUSAL, true>), and product k = 2j + i of a
// task (tile i, K/V block j; counted on from the products of earlier tasks)
// uses buffer k mod 3.  Per block j the MMA warp issues
//     P.V_0(j), S_1(j+1), P.V_1(j), S_0(j+2),
// each S going into the buffer whose P was consumed by the P.V just before it
// (tensor-core instructions of a CTA execute in issue order).  So a tile's
// next scores are computed while its softmax warps still work on the current
// ones, and the MMAs leave the softmax's critical path.  Ordering facts the
// barriers rely on: S_i(j) is issued after P.V_i(j-2), so when a softmax
// warpgroup sees S_i(j) complete, P.V_i(j-2) is complete too, and its wait
// for P.V_i(j-1) on o_ready[i] (only to rescale O_i) is never two phases away;
// s_full[b * 2 + i] has one waiting warpgroup (tile i), which sees every phase;
// the MMA warp takes P in product order on the kPBar named barriers.

template <bool BF16, bool CAUSAL, bool HELPER>
__device__ void mma_pair_role_rot(const TcArgs& a, uint8_t* smem, const Bars& bars, uint32_t tmem_base,
                                  volatile uint32_t* abort_flag) {
    // Issuing warp and helper warp as in mma_pair_role: the helper does every
    // mbarrier wait and meets the issuing warp on the named barrier kMmaSync;
    // P comes from the softmax warpgroups on the kPBar named barriers.
    constexpr int D = 64;
    using L = TcLayout<D>;
    constexpr uint32_t kIdescQK = idesc_f16_f32(kTcBM, kTcBN, BF16 ? 1u : 0u, 0u, 0u);
    constexpr uint32_t kIdescPV = idesc_f16_f32(kTcBM, D, BF16 ? 1u : 0u, 0u, 1u);
    const uint32_t q_smem = smem_u32(smem + L::kQOff);
    const uint32_t kv_smem = smem_u32(smem + L::kKVOff);
    const uint64_t kmaj_desc = smem_desc_sw128(0u, 16u, 1024u);          // Q, K: K-major
    const uint64_t vmn_desc = smem_desc_sw128(0u, kTcBN * 128u, 1024u);  // V: MN-major

    uint32_t kv_base = 0;  // ring position of the task's K_0 (K_j at 2j, V_j at 2j + 1)
    uint32_t sbase = 0;    // products of earlier tasks
    uint32_t qcnt = 0;     // tasks started (q_full phases of both tiles)
    bool ok = true;        // false: dry run (see kPBar)

    // Ring slot of a position; the helper also waits for it to be filled.
    auto wait_pos = [&](uint32_t pos) -> uint32_t {
        const uint32_t slot = pos % L::kStages;
        if (HELPER && ok)
            ok = warp_wait(&bars.kv_full[slot], (pos / L::kStages) & 1u, abort_flag, a.timeout_ns);
        return slot;
    };
    auto wait_q = [&](int i) {
        if (HELPER && ok) ok = warp_wait(&bars.q_full[i], qcnt & 1u, abort_flag, a.timeout_ns);
    };
    auto sync = [&]() {
        ok = named_barrier_and(kMmaSync, kMmaSyncThreads, ok);
        if (!HELPER) tc_fence_after();
    };
    auto take_p = [&](int i, int j) {
        if (!HELPER) {
            named_barrier_sync(p_bar(i, j), kPBarThreads);
            tc_fence_after();
        }
    };
    auto next_task = [&](int kt) -> int {
        int t = 0;
        if (HELPER) t = read_task(bars.tasks, kt, abort_flag, a.timeout_ns);
        sync();
        if (!HELPER) {
            t = static_cast<int>(static_cast<uint32_t>(ring_peek(bars.tasks, kt)));
            release_task(bars.tasks, kt);
        }
        return t;
    };
    const bool issuer = !HELPER;
    // S product into buffer b: Q tile i against the K tile in ring slot ks.
    auto issue_s = [&](uint32_t b, int i, uint32_t ks) {
        const uint64_t adesc = kmaj_desc + ((q_smem + i * L::kQTileBytes) >> 4);
        const uint64_t bdesc = kmaj_desc + ((kv_smem + ks * L::kKVTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem_base + b * kTcBN, adesc + ((kk * 32) >> 4), bdesc + ((kk * 32) >> 4),
                   kIdescQK, kk > 0 ? 1u : 0u);
        mma_commit(&bars.s_full[b * 2 + i]);
    };
    // O_i (+)= P (buffer b) V (ring slot vs).
    auto issue_pv = [&](uint32_t b, int i, uint32_t vs, bool accumulate) {
        const uint64_t bdesc = vmn_desc + ((kv_smem + vs * L::kKVTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTcBN / 16; ++kk)
            mma_ts(tmem_base + 3 * kTcBN + i * D, tmem_base + b * kTcBN + kk * 8,
                   bdesc + ((kk * 16 * 128) >> 4), kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
        mma_commit(&bars.o_ready[i]);
    };

    for (int kt = 0;; ++kt) {
        const int t = next_task(kt);
        if (t >= a.num_tasks) break;
        const Task tk = decode_task<CAUSAL, true>(t, a);
        const int nb = tk.nbmax;
        // Prologue: S_0(0), S_1(0), S_0(1).
        wait_q(0);
        wait_q(1);
        const uint32_t ks = wait_pos(kv_base);
        uint32_t ks_next = 0;  // ring slot of K_{j+1}
        if (nb > 1) ks_next = wait_pos(kv_base + 2u);
        sync();
        if (issuer && ok) {
            if (elect_one_sync()) {
                issue_s(sbase % 3u, 0, ks);
                if (nb == 1) mma_commit(&bars.q_empty[0]);
                issue_s((sbase + 1u) % 3u, 1, ks);
                mma_commit(&bars.kv_empty[ks]);
                if (nb == 1) mma_commit(&bars.q_empty[1]);
                if (nb > 1) {
                    issue_s((sbase + 2u) % 3u, 0, ks_next);
                    if (nb == 2) mma_commit(&bars.q_empty[0]);
                }
            }
            __syncwarp();
        }
        for (int j = 0; j < nb; ++j) {
            const uint32_t k0 = sbase + 2u * j;
            const uint32_t vs = wait_pos(kv_base + 2u * j + 1u);  // V_j
            uint32_t ks2 = 0;                                     // K_{j+2}
            if (j + 2 < nb) ks2 = wait_pos(kv_base + 2u * (j + 2));
            sync();
            take_p(0, j);
            if (issuer && ok) {
                if (elect_one_sync()) {
                    issue_pv(k0 % 3u, 0, vs, j > 0);
                    if (j == nb - 1) mma_commit(&bars.o_full[0]);
                    if (j + 1 < nb) {  // S_1(j+1) into the buffer P_0(j) leaves
                        issue_s(k0 % 3u, 1, ks_next);
                        mma_commit(&bars.kv_empty[ks_next]);
                        if (j + 1 == nb - 1) mma_commit(&bars.q_empty[1]);
                    }
                }
                __syncwarp();
            }
            take_p(1, j);
            if (issuer && ok) {
                if (elect_one_sync()) {
                    issue_pv((k0 + 1u) % 3u, 1, vs, j > 0);
                    if (j == nb - 1) mma_commit(&bars.o_full[1]);
                    mma_commit(&bars.kv_empty[vs]);
                    if (j + 2 < nb) {  // S_0(j+2) into the buffer P_1(j) leaves
                        issue_s((k0 + 1u) % 3u, 0, ks2);
                        if (j + 2 == nb - 1) mma_commit(&bars.q_empty[0]);
                    }
                }
                __syncwarp();
            }
            if (j + 2 < nb) ks_next = ks2;
        }
        kv_base += 2u * nb;
        sbase += 2u * nb;
        ++qcnt;
    }

    if (!HELPER) {
        // Drain: every MMA issued above has completed before TMEM is released.
        if (elect_one_sync()) mma_commit(bars.drain);
        __syncwarp();
        warp_wait(bars.drain, 0u, nullptr, a.timeout_ns);
    }
}

// ---------------------------------------------------------------------------
// Softmax + correction + epilogue (one warpgroup per Q tile), both layouts
// ---------------------------------------------------------------------------
// After a wait of a softmax warpgroup gave up: pass the P named barrier of
// every block this tile has not handed over yet -- blocks j0 .. nb0 - 1 of
// the current task, then every block of the CTA's tasks from the kt1-th on
// as the ring delivers them -- waiting on nothing else, so that the issuing
// warp, which runs the same schedule to its end, meets every barrier it
// waits on (see kPBar).
template <bool CAUSAL, bool EQUAL>
__device__ __noinline__ void softmax_dry_tail(const TcArgs& a, TaskRing tasks, int tile, int j0,
                                              int nb0, int kt1, volatile uint32_t* abort_flag) {
    for (int j = j0; j < nb0; ++j) {
        __syncwarp();
        named_barrier_arrive(p_bar(tile, j), kPBarThreads);
    }
    for (int kt = kt1;; ++kt) {
        const int t = read_task(tasks, kt, abort_flag, a.timeout_ns);
        if (t >= a.num_tasks) break;
        release_task(tasks, kt);
        const Task tk = decode_task<CAUSAL, EQUAL>(t, a);
        for (int j = 0; j < tk.nb[tile]; ++j) {
            __syncwarp();
            named_barrier_arrive(p_bar(tile, j), kPBarThreads);
        }
    }
}

template <int D, bool BF16, bool CAUSAL>
__device__ void softmax_role(const TcArgs& a, const Bars& bars, uint32_t tmem_base,
                             volatile uint32_t* abort_flag) {
    constexpr bool kRot = TcLayout<D>::kRot;  // D = 64: three rotating S buffers
    const int warp = threadIdx.x / 32;
    const int tile = warp / 4;                  // which Q tile / O accumulator
    const int trow = threadIdx.x % kTcBM;       // row within the tile == TMEM lane
    const uint32_t lane_field = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t tO = tmem_base + lane_field + (kRot ? 3 : 2) * kTcBN + tile * D;
    const float sl2 = a.scale_log2;

    // Barrier phases: D = 128 counts the S products of this tile on
    // s_full[tile]; D = 64 counts them per buffer on s_full[b * 2 + tile].
    uint32_t scnt0 = 0, scnt1 = 0, scnt2 = 0;
    uint32_t ocnt = 0;     // tasks of this tile (o_full phases)
    uint32_t pv_base = 0;  // D = 64: P.V products of this tile in earlier tasks
    uint32_t sbase = 0;    // D = 64: S products of both tiles in earlier tasks
    for (int kt = 0;; ++kt) {
        const int t = read_task(bars.tasks, kt, abort_flag, a.timeout_ns);
        if (t >= a.num_tasks) break;
        release_task(bars.tasks, kt);
        const Task tk = decode_task<CAUSAL, kRot>(t, a);
        const int nb = tk.nb[tile];
        if constexpr (!kRot) {
            if (nb == 0) continue;  // tile past N (the three-buffer layout computes it anyway)
        }
        const int row0 = tk.q0 + tile * kTcBM;
        const int row = row0 + trow;
        const int lim = CAUSAL ? min(row + 1, a.N) : a.N;  // keys < lim are visible to this row

        float m_run = -INFINITY;  // running max of scale*log2(e)*s
        // bf16: O is normalised by the running sum of the 16-bit P values fed
        // to the MMA, l_run, and the LSE comes from that of the unrounded
        // values, l_exact.  fp16 rounds P 8x more finely, so one sum (of the
        // unrounded values) serves both and the sum of the rounded ones is
        // not formed.
        constexpr bool kRoundedSum = BF16;
        float l_run = 0.f;
        float l_exact = 0.f;

        for (int j = 0; j < nb; ++j) {
            uint32_t b, use;
            if constexpr (kRot) {
                b = (sbase + 2u * j + tile) % 3u;
                use = (b == 0u) ? scnt0 : ((b == 1u) ? scnt1 : scnt2);
                scnt0 += (b == 0u) ? 1u : 0u;
                scnt1 += (b == 1u) ? 1u : 0u;
                scnt2 += (b == 2u) ? 1u : 0u;
            } else {
                b = static_cast<uint32_t>(tile);
                use = scnt0++;
            }
            const uint32_t tS = tmem_base + lane_field + b * kTcBN;
            const bool ok = warp_wait(&bars.s_full[kRot ? b * 2 + tile : b], use & 1u, abort_flag,
                                      a.timeout_ns);
            if (!ok) {
                softmax_dry_tail<CAUSAL, kRot>(a, bars.tasks, tile, j, nb, kt + 1, abort_flag);
                return;
            }
            tc_fence_after();

            // The whole score row: four 32-column loads in flight, one wait.
            // The loads also reduce: cmx[c] = max of the 32 scores of chunk c
            // (tcgen05.ld.red), the row max of every tile without masked keys.
            uint32_t sr[kTcBN / 32][32];
            float cmx[kTcBN / 32];
#pragma unroll
            for (int c = 0; c < kTcBN / 32; ++c) tmem_ld32_max(tS + c * 32, sr[c], cmx[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < kTcBN / 32; ++c) {
                reg_fence(sr[c]);
                reg_fence(cmx[c]);
            }
            float s[kTcBN];
#pragma unroll
            for (int c = 0; c < kTcBN; ++c) s[c] = __uint_as_float(sr[c / 32][c % 32]);

            const int kb = j * kTcBN;
            const bool need_mask = (kb + kTcBN > a.N) || (CAUSAL && kb + kTcBN - 1 > row0);
            float mblk = fmaxf(fmaxf(cmx[0], cmx[1]), fmaxf(cmx[2], cmx[3]));
            if (need_mask) {
                // Keys past N or past the row: masked here, and the row max
                // taken over the visible scores only.
                const int vis = lim - kb;
#pragma unroll
                for (int c = 0; c < kTcBN; ++c)
                    if (c >= vis) s[c] = -INFINITY;
                float mx[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mx[u] = s[u];
#pragma unroll
                for (int c = 8; c < kTcBN; c += 2)
                    mx[(c / 2) % 8] = fmax3f(mx[(c / 2) % 8], s[c], s[c + 1]);
                mblk = fmax3f(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], mx[5]),
                              fmaxf(mx[6], mx[7]));
            }
            const float m_new = fmaxf(m_run, mblk * sl2);

            if (j == 0) {
                m_run = m_new;
            } else {
                // Rescale O and l only when some row of the warp saw its max
                // rise by more than the threshold; otherwise keep the stale
                // max for P and l alike (exact in exact arithmetic, P <= 2^8).
                const bool grow = (m_new - m_run) > kRescaleThreshold;
                if (__any_sync(0xffffffffu, grow)) {
                    if (kRot) {
                        // O_i holds P.V_i(j-1) only once that product is done
                        // (at D = 128 the commit of S_i(j) already implies it).
                        if (!warp_wait(&bars.o_ready[tile], (pv_base + j - 1) & 1u, abort_flag,
                                       a.timeout_ns)) {
                            softmax_dry_tail<CAUSAL, kRot>(a, bars.tasks, tile, j, nb, kt + 1,
                                                           abort_flag);
                            return;
                        }
                        tc_fence_after();
                    }
                    const float alpha = ex2_approx(m_run - m_new);
                    if constexpr (kRoundedSum) l_run *= alpha;
                    l_exact *= alpha;
                    m_run = m_new;
                    uint32_t r[32];
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        tmem_ld32(tO + c * 32, r);
                        tmem_wait_ld();
                        reg_fence(r);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        tmem_st32(tO + c * 32, r);
                    }
                }
            }
            const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;

            // P = exp2(s*scale*log2e - m) rounded to the operand type, written
            // over the first half of S.  l_run sums exactly the rounded values
            // the P.V product consumes, so O is normalised by the weights it
            // was built from; l_exact sums the unrounded ones for the LSE (on
            // the way; l_run after the hand-off).
            uint32_t pk[kTcBN / 32][16];
            float le[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) le[u] = 0.f;
#pragma unroll
            for (int c = 0; c < kTcBN / 32; ++c) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float x0, x1;
                    ffma2(x0, x1, s[c * 32 + 2 * e], s[c * 32 + 2 * e + 1], sl2, sl2, neg_m, neg_m);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    pk[c][e] = pack2(p0, p1, BF16);
                    fadd2(le[(e % 4) * 2], le[(e % 4) * 2 + 1], p0, p1);
                }
                tmem_st16(tS + c * 16, pk[c]);
            }
            // P stored: hand it to the issuing warp once every lane's stores
            // have completed.
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            named_barrier_arrive(p_bar(tile, j), kPBarThreads);
            // The sum of the rounded P (which normalises O) feeds nothing the
            // MMA warp waits for, so it is formed after the hand-off.
            if constexpr (kRoundedSum) {
                float la[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) la[u] = 0.f;
#pragma unroll
                for (int c = 0; c < kTcBN / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        add_packed16_to_f32<BF16>(la[(e % 4) * 2], la[(e % 4) * 2 + 1], pk[c][e]);
                l_run += ((la[0] + la[1]) + (la[2] + la[3])) + ((la[4] + la[5]) + (la[6] + la[7]));
            }
            l_exact += ((le[0] + le[1]) + (le[2] + le[3])) + ((le[4] + le[5]) + (le[6] + le[7]));
        }

        // Epilogue: O = O~ / l, LSE = (m + log2 l) ln 2, rows < N only.
        const bool ok = warp_wait(&bars.o_full[tile], ocnt & 1u, abort_flag, a.timeout_ns);
        ++ocnt;
        if (!ok) {
            softmax_dry_tail<CAUSAL, kRot>(a, bars.tasks, tile, 0, 0, kt + 1, abort_flag);
            return;
        }
        tc_fence_after();
        const float inv_l = 1.f / (kRoundedSum ? l_run : l_exact);
        const bool valid = row < a.N;
        uint8_t* orow = reinterpret_cast<uint8_t*>(a.o) +
                        ((static_cast<int64_t>(tk.bh) * a.N + row) * D) * 2;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tO + c * 32, r);
            tmem_wait_ld();
            reg_fence(r);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                pk[e] = pack2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l,
                              BF16);
            if (valid) {
                uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
        }
        if (valid && a.lse != nullptr)
            a.lse[static_cast<int64_t>(tk.bh) * a.N + row] = (m_run + log2f(l_exact)) * kLn2;
        tc_fence_before();
        if constexpr (kRot) {
            pv_base += static_cast<uint32_t>(nb);
            sbase += static_cast<uint32_t>(tk.nb[0] + tk.nb[1]);
        }
    }
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kTcThreads, 1) attn_fwd_tc_kernel(const __grid_constant__ TcArgs a) {
    using L = TcLayout<D>;
    // 128-byte-swizzled TMA destinations and MMA operands need 1024-byte
    // aligned tiles.  Should the runtime ever place the dynamic window
    // differently, report it and leave before touching anything.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if ((smem_u32(smem_raw) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicOr(&g_error_word, 1u << kDevErrInternal);
        return;
    }
    uint8_t* smem = smem_raw;
    const Bars bars = carve_bars<D>(smem);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile uint32_t* abort_flag = misc + 1;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.q_full[i], 1);
            mbar_init(&bars.q_empty[i], 1);
            mbar_init(&bars.o_full[i], 1);
            if (L::kRot) mbar_init(&bars.o_ready[i], 1);
        }
        for (int b = 0; b < L::kSFull; ++b) mbar_init(&bars.s_full[b], 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&bars.kv_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        mbar_init(bars.drain, 1);
        for (int s = 0; s < kTaskRing; ++s) {
            mbar_init(bars.tasks.full(s), 1);
            mbar_init(bars.tasks.empty(s), kTaskReaders);
            *bars.tasks.word(s) = ring_word(-1, 0u);  // a tag no task index has
        }
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(misc, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 9 && lane == 0) {
        tma_prefetch_desc(&a.tmap_q);
        tma_prefetch_desc(&a.tmap_k);
        tma_prefetch_desc(&a.tmap_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];

    if (warp < 8) {
        regs_increase<kSoftmaxRegs>();
        softmax_role<D, BF16, CAUSAL>(a, bars, tmem_base, abort_flag);
    } else {
        regs_decrease<kControlRegs>();
        if (warp == 8 || warp == 10) {  // the issuing warp and its helper
            if constexpr (L::kRot) {
                if (warp == 8)
                    mma_pair_role_rot<BF16, CAUSAL, false>(a, smem, bars, tmem_base, abort_flag);
                else
                    mma_pair_role_rot<BF16, CAUSAL, true>(a, smem, bars, tmem_base, abort_flag);
            } else {
                if (warp == 8)
                    mma_pair_role<D, BF16, CAUSAL, false>(a, smem, bars, tmem_base, abort_flag);
                else
                    mma_pair_role<D, BF16, CAUSAL, true>(a, smem, bars, tmem_base, abort_flag);
            }
        } else if (warp == 9) {
            producer_role<D, CAUSAL>(a, smem, bars, abort_flag);
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::kTmemCols);
    }
    if (threadIdx.x == 0) {
        // The last CTA to finish puts the launch's counters back to zero
        // (every other CTA has taken its last task before counting itself).
        uint32_t* ctr = sched_slot();
        __threadfence();
        if (atomicAdd(&ctr[1], 1u) == gridDim.x - 1u) {
            atomicExch(&ctr[0], 0u);
            atomicExch(&ctr[1], 0u);
        }
    }
}

__global__ void wait_selftest_kernel(uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    // Nothing ever arrives on `bar`: the bounded wait must give up, record
    // the timeout in the error word and return.
    if (threadIdx.x == 0)
        (void)mbar_wait_bounded(&bar, 0u, &abort_flag, &g_error_word, timeout_ns);
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_one(const TcArgs& a, int grid, cudaStream_t stream) {
    using L = TcLayout<D>;
    auto* fn = attn_fwd_tc_kernel<D, BF16, CAUSAL>;
    // The opt-in above 48 KB of dynamic shared memory is per device: set it
    // once for every device this instantiation is launched on.
    static std::atomic<bool> done[kMaxDevices] = {};
    cudaError_t e = opt_in_smem_once(fn, L::kAlloc, done);
    if (e != cudaSuccess) return e;
    fn<<<grid, kTcThreads, L::kAlloc, stream>>>(a);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_causal(const TcArgs& a, bool causal, int grid, cudaStream_t s) {
    return causal ? launch_one<D, BF16, true>(a, grid, s) : launch_one<D, BF16, false>(a, grid, s);
}

}  // namespace

int tc_smem_bytes(int D) { return D == 128 ? TcLayout<128>::kAlloc : TcLayout<64>::kAlloc; }
int tc_num_stages(int D) { return D == 128 ? TcLayout<128>::kStages : TcLayout<64>::kStages; }

cudaError_t tc_launch(const TcArgs& a, int D, bool bf16, bool causal, int grid,
                      cudaStream_t stream) {
    if (D == 128)
        return bf16 ? launch_causal<128, true>(a, causal, grid, stream)
                    : launch_causal<128, false>(a, causal, grid, stream);
    return bf16 ? launch_causal<64, true>(a, causal, grid, stream)
                : launch_causal<64, false>(a, causal, grid, stream);
}

cudaError_t read_and_clear_error_word(uint32_t* out) {
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v));
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    *out = v;
    return e;
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns);
    return cudaGetLastError();
}

}  // namespace fattn
