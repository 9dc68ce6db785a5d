// bwd_tc.cu -- attention backward (dQ, dK, dV) on the tensor cores, bf16/fp16.
//
// The FA2 report of chang-wenbin.github.io (section "反向传播性能分析") keeps
// the forward's tiling for the backward pass and recomputes the scores
// instead of storing them.  Per (query i, key j) pair, with P_ij rebuilt from
// the LSE the forward emitted:
//   P_ij = exp(s_ij - LSE_i),  dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - Delta_i)
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j
// where Delta_i = dO_i . O_i.
//
// Three kernels:
//   prep : per row, -LSE_i * log2(e) and -Delta_i into a padded workspace
//          (-inf / 0 past N so that tail rows contribute nothing), negated so
//          that the elementwise steps are plain packed adds and FMAs;
//   dKdV : one CTA per (head, 128-key block): K and V stay in shared memory
//          while 128-query tiles of Q, dO and their row statistics stream
//          through a TMA ring; S^T = K Q^T and dP^T = V dO^T land in TMEM,
//          eight warps (one key row per thread, two warps per row range)
//          turn them into P^T and dS^T (16-bit, written back into TMEM) one
//          64-query half at a time, and dV += P^T dO, dK += dS^T Q
//          accumulate in TMEM, the first half's products running while the
//          warps work on the second, and the next tile's S^T while they
//          finish; dK and dV are written once at the end;
//   dQ   : one CTA per (head, 128-query tile), the mirror image: Q and dO
//          stay, K and V stream, S = Q K^T and dP = dO V^T, dS formed per
//          query row, dQ += dS K accumulates in TMEM.
// The page has the K/V gradients updated in place with atomics; here each
// gradient is owned by exactly one CTA (no atomics, a deterministic result),
// at the price of recomputing S and dP once more for dQ (7 products of
// 128 x 128 x D per tile pair instead of 5).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace fattn {
namespace {

// Error word of this translation unit's kernels (ORed into the status call).
__device__ uint32_t g_error_word;

constexpr int kBT = 128;            // tile edge: rows of every tile, keys / queries per tile
constexpr int kBwdThreads = 352;    // warps 0-7 elementwise, 8 MMA issue, 9 TMA, 10 MMA helper
constexpr int kMmaWarp = 8, kTmaWarp = 9, kHelperWarp = 10;
// Named barriers.  The issuing warp never tests an mbarrier inside its loop
// (a shared-memory access right after issued MMAs waits until they are
// taken by the tensor pipe): the helper warp does those waits and meets it on
// kSyncBar, with an AND of "every wait succeeded"; the elementwise warps hand
// their 16-bit tiles (dK/dV: kPBar + half of the 128-query tile; dQ: kPBar +
// tile parity, since they can run one tile ahead) and, for dQ, the dP columns
// they have read (kDpBar) over named barriers too.
constexpr uint32_t kSyncBar = 1, kSyncThreads = 64;
constexpr uint32_t kPBar = 2;        // 2, 3
constexpr uint32_t kDpBar = 4;
// dK/dV: the elementwise warps have loaded the last scores of a tile, so the
// issuing warp may overwrite them with the next tile's.
constexpr uint32_t kLdBar = 4;
constexpr uint32_t kEwThreads = 8 * 32 + 32;  // the elementwise warps and the issuing warp
constexpr uint32_t kTmemCols = 512;

// Shared memory: the two resident tiles, then ring A and ring B.
//   dK/dV: ring A slots hold a 128-query inner tile pair (Q, dO) and those
//          queries' LSE*log2e and Delta; ring B is empty (Q and dO are both
//          read until the tile's accumulating products).
//   dQ:    ring A holds K tiles, ring B V tiles: V is free once dP is done,
//          earlier than K (read again by dQ += dS K), so the two rings are
//          released separately and K gets the deeper one.

template <int D, bool KV>
struct BwdLayout {
    static constexpr int kTile = kBT * D * 2;               // one [128][D] 16-bit tile
    static constexpr int kTileIn = kTile;                   // one streamed inner tile (128 rows)
    static constexpr int kAtomIn = kBT * 128;               // bytes of one 64-wide swizzle atom of it
    static constexpr int kStats = KV ? 2 * kBT * 4 : 0;     // LSE*log2e and Delta of the tile's queries
    static constexpr int kSA = KV ? (D == 128 ? 2 : 5) : (D == 128 ? 3 : 4);
    static constexpr int kSB = KV ? 0 : (D == 128 ? 2 : 4);
    static constexpr int kSBm = kSB > 0 ? kSB : 1;          // divisor for ring B indices
    static constexpr int kSlotA = KV ? (2 * kTileIn + kStats + 1023) / 1024 * 1024 : kTile;
    static constexpr int kSlotB = kTile;
    static constexpr int kOuter = 0;                        // two resident tiles
    static constexpr int kRingA = 2 * kTile;
    static constexpr int kRingB = kRingA + kSA * kSlotA;
    static constexpr int kBar = kRingB + kSB * kSlotB;
    // barriers: outer_full, fullA/emptyA[SA], fullB/emptyB[SB], s_full[2],
    // done, r_free; abort flag; TMEM slot
    static constexpr int kBytes = kBar + (5 + 2 * kSA + 2 * kSB) * 8 + 16;
    static_assert(kBytes <= 227 * 1024, "shared memory");
};

struct BwdBars {
    uint64_t* outer_full;
    uint64_t* full_a;
    uint64_t* empty_a;
    uint64_t* full_b;
    uint64_t* empty_b;
    uint64_t* s_full;
    uint64_t* done;
    uint64_t* r_free;  // dK/dV at D = 64: a tile's second-half 16-bit results have been read
    uint32_t* abort_flag;
    uint32_t* tmem_slot;
};

template <int D, bool KV>
__device__ __forceinline__ BwdBars bwd_bars(uint8_t* smem) {
    using L = BwdLayout<D, KV>;
    BwdBars b;
    uint64_t* p = reinterpret_cast<uint64_t*>(smem + L::kBar);
    b.outer_full = p;
    b.full_a = p + 1;
    b.empty_a = b.full_a + L::kSA;
    b.full_b = b.empty_a + L::kSA;
    b.empty_b = b.full_b + L::kSB;
    b.s_full = b.empty_b + L::kSB;   // [2]: one per S buffer / tile parity
    b.done = b.s_full + 2;
    b.r_free = b.done + 1;
    b.abort_flag = reinterpret_cast<uint32_t*>(b.r_free + 1);
    b.tmem_slot = b.abort_flag + 1;
    return b;
}

// (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1), (a0 + b0, a1 + b1), (a0 * b0, a1 * b1):
// one packed fp32 instruction each, rounded as the scalar forms.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ uint32_t pack16(float lo, float hi, bool bf16) {
    if (bf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// One-dimensional bulk copy global -> shared, completion as tx bytes on `bar`
// (both addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* abort_flag,
                                          uint64_t timeout_ns) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort_flag, &g_error_word,
                                                     timeout_ns));
}

// Work unit of a CTA.  dKdV: key block kb of key/value head bh (B*Hkv of
// them); the inner tiles are the 128-query tiles j0 .. nt-1 (causal: from the
// tile on the block's diagonal) of each of the H/Hkv query heads that read
// this K/V head, head after head (n = group size x tiles per head).
// dQ: query tile qt of query head bh, key tiles 0 .. j_end-1 (causal: up to
// the diagonal) of its K/V head.  Causal grids run the longest units first
// (ascending kb, descending qt); otherwise head-major.
struct BwdTask {
    int bh, blk, j0, n, per_head;
};

template <bool KV, bool CAUSAL>
__device__ __forceinline__ BwdTask bwd_task(const BwdArgs& a) {
    BwdTask t;
    const int idx = blockIdx.x;
    const int heads = KV ? a.BHkv : a.BH;
    if (CAUSAL) {
        // longest first: across heads, by block
        t.bh = idx % heads;
        t.blk = KV ? idx / heads : a.num_tiles - 1 - idx / heads;
    } else {
        // head-major: CTAs running together stream the same head's tiles (L2 reuse)
        t.bh = idx / a.num_tiles;
        t.blk = idx % a.num_tiles;
    }
    if (KV) {
        t.j0 = CAUSAL ? t.blk : 0;
        t.per_head = a.num_tiles - t.j0;
        t.n = t.per_head * (a.H / a.Hkv);
    } else {
        t.j0 = 0;
        t.per_head = CAUSAL ? t.blk + 1 : a.num_tiles;
        t.n = t.per_head;
    }
    return t;
}

// Query head read by inner tile it of a dK/dV task: the group's query heads
// one after the other.
__device__ __forceinline__ int bwd_query_head(const BwdArgs& a, const BwdTask& tk, int it) {
    const int b = tk.bh / a.Hkv, hk = tk.bh % a.Hkv, G = a.H / a.Hkv;
    return b * a.H + hk * G + it / tk.per_head;
}

template <int D, bool BF16, bool KV, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_kernel(const __grid_constant__ BwdArgs a) {
    using L = BwdLayout<D, KV>;
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicOr(&g_error_word, 1u << kDevErrInternal);
        return;
    }
    const BwdBars bars = bwd_bars<D, KV>(smem);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const BwdTask tk = bwd_task<KV, CAUSAL>(a);

    if (threadIdx.x == 0) {
        mbar_init(bars.outer_full, 1);
        for (int s = 0; s < L::kSA; ++s) {
            mbar_init(&bars.full_a[s], 1);
            mbar_init(&bars.empty_a[s], 1);
        }
        for (int s = 0; s < L::kSB; ++s) {
            mbar_init(&bars.full_b[s], 1);
            mbar_init(&bars.empty_b[s], 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&bars.s_full[i], 1);
        mbar_init(bars.done, 1);
        mbar_init(bars.r_free, 1);
        *bars.abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(bars.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *bars.tmem_slot;
    // TMEM columns.  dK/dV: S^T [0,128) and dP^T [128,256) of one 128-query
    // tile; the 16-bit P^T and dS^T overwrite dP^T at D = 128 and have their
    // own columns [256,384) at D = 64; then dV and dK (D columns each).  dQ: S in two buffers [0,128) and [128,256) (then
    // the 16-bit dS), dP [256,384), dQ [384,384+D).  Within a 32-column chunk
    // the 16-bit results go to its first 16 columns (P^T, or dS for dQ) and,
    // for dK/dV, dS^T to the next 16.
    const uint32_t t_s = tmem;
    const uint32_t t_dp = KV ? tmem + 128 : tmem + 256;
    // dK/dV at D = 64: the 16-bit results in columns of their own, so the
    // next tile's S^T and dP^T need not wait for the products that read them.
    constexpr bool kOwnR = KV && D == 64;
    const uint32_t t_r = kOwnR ? tmem + 256 : t_dp;
    const uint32_t t_acc1 = KV ? tmem + (kOwnR ? 384 : 256) : tmem + 384;
    const uint32_t t_acc2 = t_acc1 + D;
    const int blk0 = tk.blk * kBT;  // first row of the resident tiles
    // K/V head of the task (dK/dV: the task's own head; dQ: the one its query head reads)
    const int kvh = KV ? tk.bh : kv_head_of(tk.bh, a.H, a.Hkv);

    if (warp == kTmaWarp) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const CUtensorMap* outer1 = KV ? &a.tmap_k : &a.tmap_q;
            const CUtensorMap* outer2 = KV ? &a.tmap_v : &a.tmap_do;
            const CUtensorMap* inner1 = KV ? &a.tmap_q : &a.tmap_k;
            const CUtensorMap* inner2 = KV ? &a.tmap_do : &a.tmap_v;
            mbar_arrive_expect_tx(bars.outer_full, 2 * L::kTile);
            const int oh = KV ? kvh : tk.bh;  // head of the resident tiles
            for (int at = 0; at < D / 64; ++at) {
                tma_load_3d(smem + L::kOuter + at * kBT * 128, outer1, bars.outer_full, at * 64, blk0, oh);
                tma_load_3d(smem + L::kOuter + L::kTile + at * kBT * 128, outer2, bars.outer_full, at * 64,
                            blk0, oh);
            }
            int issued_a = 0, issued_b = 0;
            bool ok = true;
            for (int it = 0; it < tk.n && ok; ++it) {
                const int row0 = (tk.j0 + it % tk.per_head) * kBT;
                const int qh = KV ? bwd_query_head(a, tk, it) : tk.bh;  // head of the Q / dO tiles
                const int sa = it % L::kSA;
                if (it >= L::kSA) {
                    ok = mbar_wait_bounded(&bars.empty_a[sa], ((it / L::kSA) - 1) & 1u, bars.abort_flag,
                                           &g_error_word, a.timeout_ns);
                    if (!ok) break;
                }
                uint8_t* st = smem + L::kRingA + sa * L::kSlotA;
                mbar_arrive_expect_tx(&bars.full_a[sa], KV ? 2 * L::kTileIn + L::kStats : L::kTile);
                for (int at = 0; at < D / 64; ++at) {
                    tma_load_3d(st + at * L::kAtomIn, inner1, &bars.full_a[sa], at * 64, row0, KV ? qh : kvh);
                    if (KV)
                        tma_load_3d(st + L::kTileIn + at * L::kAtomIn, inner2, &bars.full_a[sa], at * 64, row0,
                                    qh);
                }
                if (KV) {
                    const float* stats = a.ws + static_cast<int64_t>(qh) * 2 * a.Npad + row0;
                    bulk_load(st + 2 * L::kTileIn, stats, kBT * 4, &bars.full_a[sa]);
                    bulk_load(st + 2 * L::kTileIn + kBT * 4, stats + a.Npad, kBT * 4, &bars.full_a[sa]);
                }
                ++issued_a;
                if (!KV) {
                    const int sb = it % L::kSBm;
                    if (it >= L::kSB) {
                        ok = mbar_wait_bounded(&bars.empty_b[sb], ((it / L::kSBm) - 1) & 1u, bars.abort_flag,
                                               &g_error_word, a.timeout_ns);
                        if (!ok) break;
                    }
                    uint8_t* sv = smem + L::kRingB + sb * L::kSlotB;
                    mbar_arrive_expect_tx(&bars.full_b[sb], L::kTile);
                    for (int at = 0; at < D / 64; ++at)
                        tma_load_3d(sv + at * kBT * 128, inner2, &bars.full_b[sb], at * 64, row0, kvh);
                    ++issued_b;
                }
            }
            if (!ok) {
                // Let the copies already started land before the CTA leaves.
                for (int s = 0; s < L::kSA; ++s) {
                    int last = -1;
                    for (int i = 0; i < issued_a; ++i)
                        if (i % L::kSA == s) last = i;
                    if (last >= 0)
                        mbar_wait_bounded(&bars.full_a[s], (last / L::kSA) & 1u, nullptr, &g_error_word,
                                          a.timeout_ns);
                }
                for (int s = 0; s < L::kSB; ++s) {
                    int last = -1;
                    for (int i = 0; i < issued_b; ++i)
                        if (i % L::kSBm == s) last = i;
                    if (last >= 0)
                        mbar_wait_bounded(&bars.full_b[s], (last / L::kSBm) & 1u, nullptr, &g_error_word,
                                          a.timeout_ns);
                }
                mbar_wait_bounded(bars.outer_full, 0u, nullptr, &g_error_word, a.timeout_ns);
            }
        }
    } else if (warp == kMmaWarp || warp == kHelperWarp) {
        // ---------------- MMA issue (warp 8) and its helper (warp 10) ----------------
        // Both warps run the same schedule.  dK/dV: S^T and dP^T of 128-query
        // tile it (N = 128: the shared-memory operands at the tensor core's
        // full rate, where N = 64 products run at two thirds of it) go to
        // one TMEM buffer; the elementwise warps hand the 16-bit P^T and dS^T
        // (written over dP^T) over one 64-query half at a time (kPBar +
        // half), and the first half's accumulating products run while they
        // work on the second.  S^T of tile it+1 is issued as soon as they
        // have loaded the last scores of tile it (kLdBar), so it runs while
        // they work too; dP^T of tile it+1 follows the second half's
        // accumulating products, which read the columns it overwrites.  dQ: per
        // key tile it, S(it) and dP(it) -> s_full; the elementwise warps load
        // dP(it) and hand its columns back (kDpBar), so dP(it+1) (and
        // S(it+1), into the other buffer) run while they work, then dQ += dS K
        // once the 16-bit dS is in TMEM.  On an abort both warps run the rest
        // of the schedule dry (no waits, no MMAs) and still pass every named
        // barrier, which the elementwise warps then meet by arriving for
        // every remaining tile.
        const bool issuer = warp == kMmaWarp;
        constexpr uint32_t kIdescS = idesc_f16_f32(kBT, kBT, BF16 ? 1u : 0u, 0u, 0u);
        constexpr uint32_t kIdescAcc = idesc_f16_f32(kBT, D, BF16 ? 1u : 0u, 0u, 1u);
        constexpr int kInRows = kBT;
        const uint64_t kmaj = smem_desc_sw128(0u, 16u, 1024u);
        const uint64_t mnmaj = smem_desc_sw128(0u, kInRows * 128u, 1024u);  // leading offset = slab size
        const uint32_t outer1_s = smem_u32(smem + L::kOuter), outer2_s = outer1_s + L::kTile;
        auto inner1 = [&](int it) { return smem_u32(smem + L::kRingA + (it % L::kSA) * L::kSlotA); };
        auto inner2 = [&](int it) {
            return KV ? inner1(it) + L::kTileIn : smem_u32(smem + L::kRingB + (it % L::kSBm) * L::kSlotB);
        };
        // dK/dV: one S^T / dP^T buffer; dQ: S in two buffers by tile parity.
        auto s_buf = [&](int it) { return KV ? t_s : t_s + 128u * static_cast<uint32_t>(it & 1); };
        auto dp_buf = [&](int it) { return t_dp; };
        // S = outer1 inner1^T, dP = outer2 inner2^T: both operands K-major over D.
        auto issue_s = [&](int it) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off_a = ((kk / 4) * (kBT * 128) + (kk % 4) * 32) >> 4;
                const uint64_t off_b = ((kk / 4) * L::kAtomIn + (kk % 4) * 32) >> 4;
                mma_ss(s_buf(it), kmaj + (outer1_s >> 4) + off_a, kmaj + (inner1(it) >> 4) + off_b, kIdescS,
                       kk > 0 ? 1u : 0u);
            }
        };
        auto issue_dp = [&](int it) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off_a = ((kk / 4) * (kBT * 128) + (kk % 4) * 32) >> 4;
                const uint64_t off_b = ((kk / 4) * L::kAtomIn + (kk % 4) * 32) >> 4;
                mma_ss(dp_buf(it), kmaj + (outer2_s >> 4) + off_a, kmaj + (inner2(it) >> 4) + off_b, kIdescS,
                       kk > 0 ? 1u : 0u);
            }
        };
        // acc (+)= (16-bit tile in TMEM, 8 columns per 16 inner rows) x inner
        // tile as an MN-major operand (16 inner rows = 2048 bytes), over the
        // inner rows [64 h, 64 h + 64) (dQ: h = 0 and 1 in one go).  In each
        // 32-column chunk (of dP^T for dK/dV, of S for dQ) the elementwise
        // warp put its 16-bit results in the first 16 columns (P^T, or dS
        // for dQ) and dS^T in the next 16.
        auto issue_acc = [&](int it, int h, int halves) {
            const uint32_t in1 = inner1(it), in2 = inner2(it);
#pragma unroll
            for (int kk = 4 * h; kk < 4 * (h + halves); ++kk) {
                const uint64_t boff = (kk * 16 * 128) >> 4;
                const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                const uint32_t acol = (kk / 2) * 32 + (kk % 2) * 8;
                if (KV) {
                    mma_ts(t_acc1, t_r + acol, mnmaj + (in2 >> 4) + boff, kIdescAcc, acc);       // dV += P^T dO
                    mma_ts(t_acc2, t_r + acol + 16, mnmaj + (in1 >> 4) + boff, kIdescAcc, acc);  // dK += dS^T Q
                } else {
                    mma_ts(t_acc1, s_buf(it) + acol, mnmaj + (in1 >> 4) + boff, kIdescAcc, acc);       // dQ += dS K
                }
            }
        };
        bool ok = true;
        // The helper's waits for ring A (inner1; for dK/dV the whole slot) /
        // ring B (dQ: V) of tile it.
        auto wait_a = [&](int it) {
            if (!issuer && ok)
                ok = warp_wait(&bars.full_a[it % L::kSA], (it / L::kSA) & 1u, bars.abort_flag, a.timeout_ns);
        };
        auto wait_b = [&](int it) {
            if (!KV && !issuer && ok)
                ok = warp_wait(&bars.full_b[it % L::kSBm], (it / L::kSBm) & 1u, bars.abort_flag, a.timeout_ns);
        };
        auto sync = [&]() {
            ok = named_barrier_and(kSyncBar, kSyncThreads, ok);
            if (issuer) tc_fence_after();
        };
        // The issuing warp takes a tile from the elementwise warps.
        auto take = [&](uint32_t bar) {
            if (issuer) {
                named_barrier_sync(bar, kEwThreads);
                tc_fence_after();
            }
        };
        // One elected lane of the issuing warp runs f, unless dry.
        auto issue = [&](auto&& f) {
            if (issuer && ok) {
                if (elect_one_sync()) f();
                __syncwarp();
            }
        };
        if (!issuer && ok) ok = warp_wait(bars.outer_full, 0u, bars.abort_flag, a.timeout_ns);
        if (KV) {
            wait_a(0);
            sync();
            issue([&] {
                issue_s(0);
                issue_dp(0);
                mma_commit(&bars.s_full[0]);
            });
            for (int it = 0; it < tk.n; ++it) {
                const bool more = it + 1 < tk.n;
                take(kPBar);
                issue([&] { issue_acc(it, 0, 1); });
                take(kLdBar);
                if (more) {  // the next tile's scores over those just loaded
                    wait_a(it + 1);
                    sync();
                    issue([&] {
                        issue_s(it + 1);
                        if (kOwnR) {
                            issue_dp(it + 1);
                            mma_commit(&bars.s_full[0]);
                        }
                    });
                }
                take(kPBar + 1);
                issue([&] {
                    issue_acc(it, 1, 1);
                    mma_commit(&bars.empty_a[it % L::kSA]);
                    if (kOwnR) mma_commit(bars.r_free);
                    // D = 128: dP^T of tile it+1 in issue order after the
                    // products that read tile it's 16-bit results from its columns.
                    if (!kOwnR && more) {
                        issue_dp(it + 1);
                        mma_commit(&bars.s_full[0]);
                    }
                });
            }
        } else {
            wait_a(0);
            wait_b(0);
            sync();
            issue([&] {
                issue_s(0);
                issue_dp(0);
                mma_commit(&bars.s_full[0]);
                mma_commit(&bars.empty_b[0]);
            });
            for (int it = 0; it < tk.n; ++it) {
                const bool more = it + 1 < tk.n;
                if (more) {
                    wait_a(it + 1);
                    sync();
                    issue([&] { issue_s(it + 1); });
                }
                take(kDpBar);
                if (more) {
                    wait_b(it + 1);
                    sync();
                    issue([&] {
                        issue_dp(it + 1);
                        mma_commit(&bars.s_full[(it + 1) & 1]);
                        mma_commit(&bars.empty_b[(it + 1) % L::kSBm]);  // V slot free once dP is done
                    });
                }
                take(kPBar + (it & 1));
                issue([&] {
                    issue_acc(it, 0, 2);
                    mma_commit(&bars.empty_a[it % L::kSA]);
                });
            }
        }
        if (issuer) {
            if (elect_one_sync()) mma_commit(bars.done);  // fires once every MMA above has completed
            __syncwarp();
        }
    } else {
        // ---------------- elementwise warps 0-7 ----------------
        // Warps w and w+4 share TMEM lane quarter w % 4 (thread = lane =
        // resident row) and split the columns of S and dP between them (dK/dV:
        // 32 each of each 64-query half of a 128-query tile; dQ: 64 each of a
        // 128-key tile); each writes its 16-bit results into the S columns it
        // has already read.
        const int quarter = warp % 4, half = warp / 4;
        const int r = quarter * 32 + lane;
        const int row = blk0 + r;  // KV: key index; dQ: query index
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int c0 = half * 64;  // first column of this warp
        float nlse2_r = 0.f, ndelta_r = 0.f;  // -LSE*log2(e) and -Delta of this row
        if (!KV) {
            const float* stats = a.ws + static_cast<int64_t>(tk.bh) * 2 * a.Npad + row;
            nlse2_r = stats[0];        // -inf past N: the row's P is 0
            ndelta_r = stats[a.Npad];
        }
        bool ok = true;
        int failed_at = 0;  // first tile not handed over when a wait gave up
        if (KV) {
            // 128-query tile it, in two halves h: this warp's 32 columns
            // [64h + 32*half, 64h + 32*half + 32) of S^T and dP^T; P^T and
            // dS^T go to the first 16 and the next 16 of those dP^T columns,
            // and each half is handed to the issuing warp on kPBar + h; once
            // the second half's scores are in registers, S^T's columns are
            // free (kLdBar).
            for (int it = 0; it < tk.n && ok; ++it) {
                const int jq = tk.j0 + it % tk.per_head;  // 128-query tile index within its head
                const int sa = it % L::kSA;
                ok = warp_wait(&bars.s_full[0], it & 1u, bars.abort_flag, a.timeout_ns);
                if (ok)  // the slot's statistics: this phase is complete and not yet refilled
                    ok = warp_wait(&bars.full_a[sa], (it / L::kSA) & 1u, bars.abort_flag, a.timeout_ns);
                if (!ok) {
                    failed_at = it;
                    break;
                }
                tc_fence_after();
                const float* nlse2s = reinterpret_cast<const float*>(smem + L::kRingA + sa * L::kSlotA +
                                                                     2 * L::kTileIn);
                const float* ndeltas = nlse2s + kBT;
                // queries before this key row exist only in the tile on the block's diagonal
                const bool diag = CAUSAL && jq == tk.blk;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    const int cq = 64 * h + 32 * half;  // this warp's first query column
                    const uint32_t db = t_r + lane_off + cq;  // this warp's 16-bit results
                    uint32_t sv[32], dpv[32];
                    tmem_ld32(t_s + lane_off + cq, sv);
                    tmem_ld32(t_dp + lane_off + cq, dpv);
                    tmem_wait_ld();
                    reg_fence(sv);
                    reg_fence(dpv);
                    if (h == 1) {
                        tc_fence_before();
                        __syncwarp();
                        named_barrier_arrive(kLdBar, kEwThreads);
                    }
                    // P^T = exp2(s*scale*log2e - LSE2) and dS^T = P^T (dP^T - Delta),
                    // two queries per packed instruction; the statistics of the
                    // warp's 32 queries come as 16-byte broadcasts.
                    uint32_t pk[16], dsk[16];
#pragma unroll
                    for (int e4 = 0; e4 < 32; e4 += 4) {
                        const float4 nl = *reinterpret_cast<const float4*>(nlse2s + cq + e4);
                        const float4 nd = *reinterpret_cast<const float4*>(ndeltas + cq + e4);
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int e = e4 + 2 * h2;
                            const float nl0 = h2 ? nl.z : nl.x, nl1 = h2 ? nl.w : nl.y;
                            const float nd0 = h2 ? nd.z : nd.x, nd1 = h2 ? nd.w : nd.y;
                            float x0, x1, d0, d1;
                            fma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), a.sl2, a.sl2,
                                 nl0, nl1);
                            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            if (diag) {  // query cq + e of the tile against key r: hidden when before it
                                if (cq + e < r) p0 = 0.f;
                                if (cq + e + 1 < r) p1 = 0.f;
                            }
                            add2(d0, d1, __uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1]), nd0, nd1);
                            mul2(d0, d1, p0, p1, d0, d1);
                            pk[e / 2] = pack16(p0, p1, BF16);
                            dsk[e / 2] = pack16(d0, d1, BF16);
                        }
                    }
                    if (kOwnR && h == 1 && it > 0) {
                        // The previous tile's second-half products read these
                        // columns; they are issued after this tile's scores,
                        // so only this half can get here before they are done.
                        // (After a wait that gave up, the stores still go to
                        // TMEM; nothing reads them any more.)
                        ok = warp_wait(bars.r_free, (it - 1) & 1u, bars.abort_flag, a.timeout_ns);
                        tc_fence_after();
                    }
                    tmem_st16(db, pk);
                    tmem_st16(db + 16, dsk);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    named_barrier_arrive(kPBar + h, kEwThreads);
                }
                if (!ok) failed_at = it + 1;  // every barrier of this tile was met
            }
        }
        for (int it = 0; !KV && it < tk.n && ok; ++it) {
            const int j = tk.j0 + it;
            ok = warp_wait(&bars.s_full[it & 1], (it >> 1) & 1u, bars.abort_flag, a.timeout_ns);
            if (!ok) {
                failed_at = it;
                break;
            }
            tc_fence_after();
            const bool diag = CAUSAL && j == tk.blk;
            const uint32_t sb = t_s + 128u * static_cast<uint32_t>(it & 1) + lane_off + c0;
            // dP first, in full, so that its columns can be handed back at once.
            uint32_t dpv[2][32], sv[32];
            tmem_ld32(t_dp + lane_off + c0, dpv[0]);
            tmem_ld32(t_dp + lane_off + c0 + 32, dpv[1]);
            tmem_ld32(sb, sv);
            tmem_wait_ld();
            reg_fence(dpv[0]);
            reg_fence(dpv[1]);
            reg_fence(sv);
            tc_fence_before();
            __syncwarp();
            named_barrier_arrive(kDpBar, kEwThreads);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (c == 1) {
                    tmem_ld32(sb + 32, sv);
                    tmem_wait_ld();
                    reg_fence(sv);
                }
                // dS = exp2(s*scale*log2e - LSE2) (dP - Delta), two keys per
                // packed instruction; keys past N or (diagonal tile) past the
                // row are masked only in chunks that hold such keys.
                const int vis = min(a.N - j * kBT, diag ? r + 1 : kBT) - (c0 + c * 32);
                const bool masked = __any_sync(0xffffffffu, vis < 32);
                uint32_t dsk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float x0, x1, d0, d1;
                    fma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), a.sl2, a.sl2,
                         nlse2_r, nlse2_r);
                    float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    if (masked) {
                        if (e >= vis) p0 = 0.f;
                        if (e + 1 >= vis) p1 = 0.f;
                    }
                    add2(d0, d1, __uint_as_float(dpv[c][e]), __uint_as_float(dpv[c][e + 1]), ndelta_r,
                         ndelta_r);
                    mul2(d0, d1, p0, p1, d0, d1);
                    dsk[e / 2] = pack16(d0, d1, BF16);
                }
                // Only columns of this chunk, already read, are overwritten.
                tmem_st16(sb + c * 32, dsk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            named_barrier_arrive(kPBar + (it & 1), kEwThreads);
        }
        if (!ok) {
            // A wait gave up: hand over (nothing) for every tile not handed
            // over yet, so that the issuing warp, which runs its schedule to
            // the end, meets every named barrier it waits on.
            for (int it = failed_at; it < tk.n; ++it) {
                __syncwarp();
                if (KV) {
                    named_barrier_arrive(kPBar, kEwThreads);
                    named_barrier_arrive(kLdBar, kEwThreads);
                    named_barrier_arrive(kPBar + 1, kEwThreads);
                } else {
                    named_barrier_arrive(kDpBar, kEwThreads);
                    named_barrier_arrive(kPBar + (it & 1), kEwThreads);
                }
            }
        }
        // ---------------- epilogue: accumulators -> 16-bit rows ----------------
        // Each warp converts half of the D columns of its 32 rows.
        const bool fin = warp_wait(bars.done, 0u, nullptr, a.timeout_ns);
        tc_fence_after();
        const int64_t out_row = static_cast<int64_t>(tk.bh) * a.N + row;
#pragma unroll 1
        for (int acc = 0; acc < (KV ? 2 : 1); ++acc) {
            // KV: acc 0 = dV (no scale), acc 1 = dK (x scale); dQ: acc 0 = dQ (x scale)
            const uint32_t tacc = (acc == 0 ? t_acc1 : t_acc2) + lane_off;
            const float mul = (KV && acc == 0) ? 1.f : a.scale;
            void* base = KV ? (acc == 0 ? a.dv : a.dk) : a.dq;
            uint8_t* orow = reinterpret_cast<uint8_t*>(base) + out_row * D * 2;
#pragma unroll 1
            for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
                uint32_t v[32];
                tmem_ld32(tacc + c * 32, v);  // warp-collective: every lane, whatever its row
                tmem_wait_ld();
                reg_fence(v);
                if (fin && row < a.N) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack16(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul, BF16);
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// -LSE_i * log2(e) and -Delta_i, Delta_i = dO_i . O_i (fp32 over the 16-bit
// inputs), into the padded workspace [B*H][2][Npad]; rows past N get -inf
// and 0.  A row is read as 16-byte pieces by D/8 lanes, a warp covers
// 32/(D/8) rows per load and keeps kPrepLoads such loads of O and of dO in
// flight (kPrepRows rows per warp), so the kernel streams at memory rate.
constexpr int kPrepLoads = 4;
template <int D>
__host__ __device__ constexpr int prep_rows_per_warp() { return (32 / (D / 8)) * kPrepLoads; }

template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const void* __restrict__ o,
                                                            const void* __restrict__ dout,
                                                            const float* __restrict__ lse,
                                                            float* __restrict__ ws, int N, int Npad,
                                                            int64_t rows_padded) {
    constexpr int kLanesPerRow = D / 8;               // 16-byte pieces per row
    constexpr int kRowsPerLoad = 32 / kLanesPerRow;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    const int sub = lane / kLanesPerRow, piece = lane % kLanesPerRow;
    uint4 ov[kPrepLoads], dv[kPrepLoads];
    int64_t prow[kPrepLoads];
#pragma unroll
    for (int k = 0; k < kPrepLoads; ++k) {
        prow[k] = gw * prep_rows_per_warp<D>() + k * kRowsPerLoad + sub;  // padded row
        ov[k] = make_uint4(0u, 0u, 0u, 0u);
        dv[k] = ov[k];
        if (prow[k] < rows_padded) {
            const int64_t bh = prow[k] / Npad;
            const int i = static_cast<int>(prow[k] % Npad);
            if (i < N) {
                const int64_t off = ((bh * N + i) * D) * 2 + piece * 16;
                ov[k] = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(o) + off);
                dv[k] = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(dout) + off);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < kPrepLoads; ++k) {
        const uint32_t ow[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
        const uint32_t dw[4] = {dv[k].x, dv[k].y, dv[k].z, dv[k].w};
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            float x0, x1, y0, y1;
            if (BF16) {
                const __nv_bfloat162 xb = *reinterpret_cast<const __nv_bfloat162*>(&ow[w]);
                const __nv_bfloat162 yb = *reinterpret_cast<const __nv_bfloat162*>(&dw[w]);
                x0 = __low2float(xb); x1 = __high2float(xb);
                y0 = __low2float(yb); y1 = __high2float(yb);
            } else {
                const __half2 xh = *reinterpret_cast<const __half2*>(&ow[w]);
                const __half2 yh = *reinterpret_cast<const __half2*>(&dw[w]);
                x0 = __low2float(xh); x1 = __high2float(xh);
                y0 = __low2float(yh); y1 = __high2float(yh);
            }
            acc = fmaf(x0, y0, acc);
            acc = fmaf(x1, y1, acc);
        }
#pragma unroll
        for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off, kLanesPerRow);
        if (piece == 0 && prow[k] < rows_padded) {
            const int64_t bh = prow[k] / Npad;
            const int i = static_cast<int>(prow[k] % Npad);
            float nlse2 = -INFINITY, ndelta = 0.f;
            if (i < N) {
                ndelta = -acc;
                nlse2 = -lse[bh * N + i] * 1.4426950408889634f;
            }
            ws[bh * 2 * Npad + i] = nlse2;
            ws[(bh * 2 + 1) * Npad + i] = ndelta;
        }
    }
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t bwd_launch_all(const BwdArgs& a, const void* o, const void* dout, const float* lse,
                           cudaStream_t stream) {
    const int64_t rows_padded = static_cast<int64_t>(a.BH) * a.Npad;
    const int64_t prep_warps = (rows_padded + prep_rows_per_warp<D>() - 1) / prep_rows_per_warp<D>();
    attn_bwd_prep_kernel<D, BF16><<<static_cast<unsigned>((prep_warps + 7) / 8), 256, 0, stream>>>(
        o, dout, lse, a.ws, a.N, a.Npad, rows_padded);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned grid_kv = static_cast<unsigned>(static_cast<int64_t>(a.num_tiles) * a.BHkv);
    const unsigned grid_q = static_cast<unsigned>(static_cast<int64_t>(a.num_tiles) * a.BH);
    static std::atomic<bool> kv_done[kMaxDevices] = {};
    static std::atomic<bool> q_done[kMaxDevices] = {};
    auto* kkv = attn_bwd_kernel<D, BF16, true, CAUSAL>;
    if ((e = opt_in_smem_once(kkv, BwdLayout<D, true>::kBytes, kv_done)) != cudaSuccess) return e;
    kkv<<<grid_kv, kBwdThreads, BwdLayout<D, true>::kBytes, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    auto* kq = attn_bwd_kernel<D, BF16, false, CAUSAL>;
    if ((e = opt_in_smem_once(kq, BwdLayout<D, false>::kBytes, q_done)) != cudaSuccess) return e;
    kq<<<grid_q, kBwdThreads, BwdLayout<D, false>::kBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

int64_t bwd_padded_rows(int64_t N) { return (N + kBT - 1) / kBT * kBT; }

cudaError_t bwd_launch(const BwdArgs& a, const void* o, const void* dout, const float* lse, int D,
                       bool bf16, bool causal, cudaStream_t s) {
    if (D == 128) {
        if (bf16) return causal ? bwd_launch_all<128, true, true>(a, o, dout, lse, s)
                                : bwd_launch_all<128, true, false>(a, o, dout, lse, s);
        return causal ? bwd_launch_all<128, false, true>(a, o, dout, lse, s)
                      : bwd_launch_all<128, false, false>(a, o, dout, lse, s);
    }
    if (bf16) return causal ? bwd_launch_all<64, true, true>(a, o, dout, lse, s)
                            : bwd_launch_all<64, true, false>(a, o, dout, lse, s);
    return causal ? bwd_launch_all<64, false, true>(a, o, dout, lse, s)
                  : bwd_launch_all<64, false, false>(a, o, dout, lse, s);
}

cudaError_t bwd_read_and_clear_error_word(uint32_t* out) {
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v));
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    *out = v;
    return e;
}

}  // namespace fattn
