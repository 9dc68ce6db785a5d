// fwd_ffma.cu -- fp32 attention forward on CUDA cores (FFMA), sm_103a.
//
// The loop structure of the dandandamowang.xyz "Flash Attention (二) v2"
// page ([FA2-CUDA-core]: §1.1 grid = (ceil(N/Br), B*H) with Br = 128; §3.2
// double-buffered cp.async K/V tiles with zero fill past N; §3.3 S tile ->
// tile max -> P -> merge -> unnormalised O update; §3.4 causal KV loop cut at
// min(q_start+Br, N) plus the element mask on tiles crossing the diagonal;
// §3.5 one 1/l at the end), in two kernels that differ in how a CTA's work
// is spread over its threads:
//   * attn_fwd_ffma_tiled_kernel (fattn_fwd, fp32): 256 threads share the
//     128 x BC score tile and the 128 x D output tile as 8-row register
//     micro-tiles, so one 16-byte shared-memory read feeds about 11 FMAs at
//     D = 64, issued as packed fp32x2 FMAs; P passes through shared memory
//     to the lanes that own the same rows;
//   * attn_fwd_ffma_row_kernel (fattn_fwd_f32_rowwise): the page's one query
//     row per thread, where a read feeds 4 FMAs, which caps the FP32 pipe
//     near 40 % on this part.
// Both keep O~ in registers, fold the scale and log2(e) into one multiply
// for exp2, use the single-correction online-softmax form (chang-wenbin.
// github.io report §2: one rescale factor per tile instead of two), and
// under causal masking launch the Q blocks nearest the end of the sequence
// (most K/V tiles) first.
#include <cstdint>

#include "internal.h"

namespace fattn {
namespace {

constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1) in one packed fp32 FMA instruction:
// two FMAs per issue slot.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, bool valid) {
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    const int src_bytes = valid ? 16 : 0;  // 0: write 16 zero bytes, read nothing
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(gsrc),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// One query row per thread: the [FA2-CUDA-core] page's own design (§1.1
// block = Br = 128 threads, §3.2-§3.5), kept as fattn_fwd_f32_rowwise.
// Re-tuned for GB300: O~ accumulates in registers, not shared memory, so two
// CTAs fit per SM (the page's 97 KB layout allowed one); Q and the output
// tile are staged through shared memory with a padded row stride of D+4
// floats, so that the per-row 16-byte reads and writes of the 32 threads of a
// warp are bank-conflict free and the global traffic is coalesced; K/V rows
// are read as 16-byte warp broadcasts (every thread of the warp reads the same
// key), so the K/V tiles need no padding.  A broadcast feeds four FMAs per
// lane, which holds this form near 40 % of the FP32 pipe.
// ---------------------------------------------------------------------------
template <int D, int BC>
struct RowLayout {
    static constexpr int kBr = kFfmaBr;
    static constexpr int kQStride = D + 4;                // padded row stride (floats)
    static constexpr int kKVFloats = 2 * BC * D;          // double buffer of one tensor
    static constexpr int kBytes = (2 * kKVFloats + kBr * kQStride) * 4;
};

// One K/V tile (BC keys x D) of both tensors into buffer `buf` with cp.async;
// keys >= N are zero filled.
template <int D, int BC>
__device__ __forceinline__ void load_kv_tile(const float* kh, const float* vh, float* Ks, float* Vs,
                                             int kv_start, int N, int buf) {
    constexpr int kVec = BC * D / 4;  // 16-byte vectors per tile
    float* kd = Ks + buf * BC * D;
    float* vd = Vs + buf * BC * D;
#pragma unroll
    for (int i = threadIdx.x; i < kVec; i += kFfmaBr) {
        const int r = (i * 4) / D;
        const int key = kv_start + r;
        const bool ok = key < N;
        const int64_t src = static_cast<int64_t>(ok ? key : 0) * D + (i * 4) % D;
        cp_async16(kd + i * 4, kh + src, ok);
        cp_async16(vd + i * 4, vh + src, ok);
    }
}

template <int D, int BC, bool CAUSAL>
__global__ void __launch_bounds__(kFfmaBr, 2)
    attn_fwd_ffma_row_kernel(const float* __restrict__ q, const float* __restrict__ k,
                         const float* __restrict__ v, float* __restrict__ o,
                         float* __restrict__ lse, int N, int num_qblk, int H, int Hkv,
                         float scale_log2) {
    using L = RowLayout<D, BC>;
    extern __shared__ float4 smem4[];
    float* smem = reinterpret_cast<float*>(smem4);
    float* Ks = smem;                  // [2][BC][D]
    float* Vs = Ks + L::kKVFloats;     // [2][BC][D]
    float* Qs = Vs + L::kKVFloats;     // [Br][D+4]; reused for the output tile

    const int tid = threadIdx.x;
    const int qblk = CAUSAL ? (num_qblk - 1 - static_cast<int>(blockIdx.x)) : blockIdx.x;
    const int q_start = qblk * L::kBr;
    const int row = q_start + tid;
    const int64_t head = static_cast<int64_t>(blockIdx.y) * N * D;
    const int64_t kvhead = static_cast<int64_t>(kv_head_of(blockIdx.y, H, Hkv)) * N * D;
    const float* qh = q + head;
    const float* kh = k + kvhead;
    const float* vh = v + kvhead;

    const int kv_limit = CAUSAL ? min(q_start + L::kBr, N) : N;
    const int Tc = (kv_limit + BC - 1) / BC;

    // Prologue: K/V tile 0 in flight while Q is staged.
    load_kv_tile<D, BC>(kh, vh, Ks, Vs, 0, N, 0);
    cp_async_commit();

    // Q tile -> padded shared memory, coalesced (rows >= N read as zeros).
    for (int i = tid; i < L::kBr * D / 4; i += L::kBr) {
        const int r = i / (D / 4), c4 = i % (D / 4);
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q_start + r < N)
            val = *reinterpret_cast<const float4*>(qh + static_cast<int64_t>(q_start + r) * D + c4 * 4);
        *reinterpret_cast<float4*>(Qs + r * L::kQStride + c4 * 4) = val;
    }

    const int lim = CAUSAL ? min(row + 1, N) : N;  // keys < lim are visible to this row
    float m = -INFINITY;  // running max of scale*log2(e)*s
    float l = 0.f;
    float acc[D];
#pragma unroll
    for (int d = 0; d < D; ++d) acc[d] = 0.f;
    const float* qrow = Qs + tid * L::kQStride;

    for (int j = 0; j < Tc; ++j) {
        const int cur = j & 1;
        if (j + 1 < Tc) {
            load_kv_tile<D, BC>(kh, vh, Ks, Vs, (j + 1) * BC, N, cur ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float* Kt = Ks + cur * BC * D;
        const float* Vt = Vs + cur * BC * D;
        const int kv_start = j * BC;

        // S row: s_c = q . k_c  (K rows are warp-wide broadcasts)
        float s[BC];
#pragma unroll
        for (int c = 0; c < BC; ++c) s[c] = 0.f;
#pragma unroll
        for (int d4 = 0; d4 < D / 4; ++d4) {
            const float4 qv = *reinterpret_cast<const float4*>(qrow + d4 * 4);
#pragma unroll
            for (int c = 0; c < BC; ++c) {
                const float4 kv = *reinterpret_cast<const float4*>(Kt + c * D + d4 * 4);
                s[c] = fmaf(qv.x, kv.x, s[c]);
                s[c] = fmaf(qv.y, kv.y, s[c]);
                s[c] = fmaf(qv.z, kv.z, s[c]);
                s[c] = fmaf(qv.w, kv.w, s[c]);
            }
        }

        // Scale into the log2 domain; mask keys past N and (causal) past the row.
        const bool need_mask = (kv_start + BC > N) || (CAUSAL && kv_start + BC - 1 > q_start);
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < BC; ++c) {
            float x = s[c] * scale_log2;
            if (need_mask && kv_start + c >= lim) x = -INFINITY;
            s[c] = x;
            mt = fmaxf(mt, x);
        }

        // Online softmax, single-correction form.
        const float m_new = fmaxf(m, mt);
        const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
        const float corr = ex2f(m - m_sub);  // 0 on the first visible tile
        float ls = 0.f;
#pragma unroll
        for (int c = 0; c < BC; ++c) {
            s[c] = ex2f(s[c] - m_sub);  // P kept in registers
            ls += s[c];
        }
        l = fmaf(corr, l, ls);
        m = m_new;

        // O~ = corr * O~ + P V   (V rows are warp-wide broadcasts)
#pragma unroll
        for (int d = 0; d < D; ++d) acc[d] *= corr;
#pragma unroll
        for (int c = 0; c < BC; ++c) {
            const float p = s[c];
#pragma unroll
            for (int d4 = 0; d4 < D / 4; ++d4) {
                const float4 vv = *reinterpret_cast<const float4*>(Vt + c * D + d4 * 4);
                acc[d4 * 4 + 0] = fmaf(p, vv.x, acc[d4 * 4 + 0]);
                acc[d4 * 4 + 1] = fmaf(p, vv.y, acc[d4 * 4 + 1]);
                acc[d4 * 4 + 2] = fmaf(p, vv.z, acc[d4 * 4 + 2]);
                acc[d4 * 4 + 3] = fmaf(p, vv.w, acc[d4 * 4 + 3]);
            }
        }
        __syncthreads();  // everyone is done with buffer `cur` before it is refilled
    }

    // Epilogue: O = O~ / l staged through the padded tile, then coalesced stores.
    const float inv_l = 1.f / l;
    float* orow = Qs + tid * L::kQStride;  // this thread's own row: no other reader
#pragma unroll
    for (int d4 = 0; d4 < D / 4; ++d4)
        *reinterpret_cast<float4*>(orow + d4 * 4) =
            make_float4(acc[d4 * 4] * inv_l, acc[d4 * 4 + 1] * inv_l, acc[d4 * 4 + 2] * inv_l,
                        acc[d4 * 4 + 3] * inv_l);
    if (lse != nullptr && row < N)
        lse[static_cast<int64_t>(blockIdx.y) * N + row] = (m + log2f(l)) * kLn2;
    __syncthreads();
    float* oh = o + head;
    for (int i = tid; i < L::kBr * D / 4; i += L::kBr) {
        const int r = i / (D / 4), c4 = i % (D / 4);
        if (q_start + r < N)
            *reinterpret_cast<float4*>(oh + static_cast<int64_t>(q_start + r) * D + c4 * 4) =
                *reinterpret_cast<const float4*>(Qs + r * L::kQStride + c4 * 4);
    }
}

template <int D, int BC, bool CAUSAL>
cudaError_t launch_ffma_row(const float* q, const float* k, const float* v, float* o, float* lse,
                        int BH, int H, int Hkv, int N, float scale_log2, cudaStream_t stream) {
    using L = RowLayout<D, BC>;
    auto* fn = attn_fwd_ffma_row_kernel<D, BC, CAUSAL>;
    static std::atomic<bool> done[kMaxDevices] = {};
    cudaError_t e = opt_in_smem_once(fn, L::kBytes, done);
    if (e != cudaSuccess) return e;
    const int num_qblk = (N + L::kBr - 1) / L::kBr;
    dim3 grid(num_qblk, BH);
    fn<<<grid, L::kBr, L::kBytes, stream>>>(q, k, v, o, lse, N, num_qblk, H, Hkv, scale_log2);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// 256 threads, Br = 128 rows, BC keys per K/V tile.
//
// Thread (rg, cg) = (tid / 16, tid % 16) owns query rows rg + 16 i (i < 8),
// keys cg + 16 c of each K/V tile (c < BC / 16) and output columns
// 64 u + 4 cg .. +3 (u < D / 64).  A 16-byte shared-memory read then feeds
// 32/3 FMAs at D = 64 (6.4 for S and 16 for P.V at D = 128), against 4 with
// one row per thread:
//   S  = Q K^T : per 4 features, 8 Q reads (rows) + BC/16 K reads (keys);
//   O += P V   : P goes through shared memory (key-major, the thread's 8
//                rows contiguous) to the 16 lanes of the same half-warp,
//                which own the same rows; per key, 2 P reads + D/64 V reads.
// A row's 16 owners are the 16 lanes of one half-warp, so the row max is
// four xor-shuffles and the P hand-off needs only __syncwarp.  The row sums
// stay per-thread partial sums until the epilogue.  Padded strides (D + 4
// floats for Q, K, V; 128 + 4 for P) keep the reads conflict-free: the two
// half-warps read adjacent Q rows, the 16 lanes of a half-warp read 16
// consecutive K rows.
// ---------------------------------------------------------------------------
constexpr int kTiledThreads = 256;
constexpr int kTiledRows = 8;  // query rows per thread

template <int D, int BC>
struct TiledLayout {
    static constexpr int kBr = kFfmaBr;
    static constexpr int kKeys = BC / 16;       // keys per thread per tile
    static constexpr int kCols = D / 64;        // 4-wide output column groups per thread
    static constexpr int kStride = D + 4;       // Q, K, V row stride (floats)
    static constexpr int kPStride = kBr + 4;    // one key's P column (floats)
    static constexpr int kQFloats = kBr * kStride;
    static constexpr int kKVFloats = BC * kStride;  // one tile of one tensor
    static constexpr int kPFloats = BC * kPStride;
    static constexpr int kBytes = (kQFloats + 4 * kKVFloats + kPFloats) * 4;
    static_assert(kBr == 16 * kTiledRows, "16 row groups of 8 rows");
    static_assert(BC % 16 == 0 && D % 64 == 0, "tile shape");
    static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

template <int D, int BC>
__device__ __forceinline__ void tiled_load_rows(const float* src, float* dst, int row0, int rows,
                                                int N) {
    using L = TiledLayout<D, BC>;
    for (int i = threadIdx.x; i < rows * (D / 4); i += kTiledThreads) {
        const int r = i / (D / 4), c4 = i % (D / 4);
        const bool ok = row0 + r < N;
        const int64_t off = static_cast<int64_t>(ok ? row0 + r : 0) * D + c4 * 4;
        cp_async16(dst + r * L::kStride + c4 * 4, src + off, ok);
    }
}

template <int D, int BC, bool CAUSAL, int MIN_BLOCKS>
__global__ void __launch_bounds__(kTiledThreads, MIN_BLOCKS)
    attn_fwd_ffma_tiled_kernel(const float* __restrict__ q, const float* __restrict__ k,
                               const float* __restrict__ v, float* __restrict__ o,
                               float* __restrict__ lse, int N, int num_qblk, int H, int Hkv,
                               float scale_log2) {
    using L = TiledLayout<D, BC>;
    extern __shared__ float4 smem4[];
    float* Qs = reinterpret_cast<float*>(smem4);  // [Br][D+4]
    float* Ks = Qs + L::kQFloats;                  // [2][BC][D+4]
    float* Vs = Ks + 2 * L::kKVFloats;             // [2][BC][D+4]
    float* Ps = Vs + 2 * L::kKVFloats;             // [BC][Br+4], rows in (rg, i) order

    const int tid = threadIdx.x;
    const int rg = tid / 16, cg = tid % 16;
    const int qblk = CAUSAL ? (num_qblk - 1 - static_cast<int>(blockIdx.x)) : blockIdx.x;
    const int q_start = qblk * L::kBr;
    const int64_t head = static_cast<int64_t>(blockIdx.y) * N * D;
    const int64_t kvhead = static_cast<int64_t>(kv_head_of(blockIdx.y, H, Hkv)) * N * D;
    const float* kh = k + kvhead;
    const float* vh = v + kvhead;

    const int kv_limit = CAUSAL ? min(q_start + L::kBr, N) : N;
    const int Tc = (kv_limit + BC - 1) / BC;

    // Prologue: Q and K/V tile 0 in one cp.async group (rows >= N zero filled).
    tiled_load_rows<D, BC>(q + head, Qs, q_start, L::kBr, N);
    tiled_load_rows<D, BC>(kh, Ks, 0, BC, N);
    tiled_load_rows<D, BC>(vh, Vs, 0, BC, N);
    cp_async_commit();

    float m[kTiledRows], l[kTiledRows];
    float acc[kTiledRows][4 * L::kCols];
#pragma unroll
    for (int i = 0; i < kTiledRows; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int d = 0; d < 4 * L::kCols; ++d) acc[i][d] = 0.f;
    }

    for (int j = 0; j < Tc; ++j) {
        const int cur = j & 1;
        if (j + 1 < Tc) {
            tiled_load_rows<D, BC>(kh, Ks + (cur ^ 1) * L::kKVFloats, (j + 1) * BC, BC, N);
            tiled_load_rows<D, BC>(vh, Vs + (cur ^ 1) * L::kKVFloats, (j + 1) * BC, BC, N);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float* Kt = Ks + cur * L::kKVFloats;
        const float* Vt = Vs + cur * L::kKVFloats;
        const int kb = j * BC;

        // S micro-tile: rows rg + 16 i, keys cg + 16 c.  Even and odd
        // features accumulate in the two halves of packed FMAs and are added
        // at the end.
        float s[kTiledRows][L::kKeys], so[kTiledRows][L::kKeys];
#pragma unroll
        for (int i = 0; i < kTiledRows; ++i)
#pragma unroll
            for (int c = 0; c < L::kKeys; ++c) {
                s[i][c] = 0.f;
                so[i][c] = 0.f;
            }
#pragma unroll
        for (int d4 = 0; d4 < D / 4; ++d4) {
            float4 qf[kTiledRows], kf[L::kKeys];
#pragma unroll
            for (int i = 0; i < kTiledRows; ++i)
                qf[i] = *reinterpret_cast<const float4*>(Qs + (rg + 16 * i) * L::kStride + d4 * 4);
#pragma unroll
            for (int c = 0; c < L::kKeys; ++c)
                kf[c] = *reinterpret_cast<const float4*>(Kt + (cg + 16 * c) * L::kStride + d4 * 4);
#pragma unroll
            for (int i = 0; i < kTiledRows; ++i)
#pragma unroll
                for (int c = 0; c < L::kKeys; ++c) {
                    fma2(s[i][c], so[i][c], qf[i].x, qf[i].y, kf[c].x, kf[c].y, s[i][c], so[i][c]);
                    fma2(s[i][c], so[i][c], qf[i].z, qf[i].w, kf[c].z, kf[c].w, s[i][c], so[i][c]);
                }
        }
#pragma unroll
        for (int i = 0; i < kTiledRows; ++i)
#pragma unroll
            for (int c = 0; c < L::kKeys; ++c) s[i][c] += so[i][c];

        // Online softmax per row (single-correction form), P over the row's
        // 16 owners; keys past N and (causal) past the row are masked.
        const bool need_mask = (kb + BC > N) || (CAUSAL && kb + BC - 1 > q_start);
#pragma unroll
        for (int i = 0; i < kTiledRows; ++i) {
            const int row = q_start + rg + 16 * i;
            const int lim = CAUSAL ? min(row + 1, N) : N;
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < L::kKeys; ++c) {
                float x = s[i][c] * scale_log2;
                if (need_mask && kb + cg + 16 * c >= lim) x = -INFINITY;
                s[i][c] = x;
                mt = fmaxf(mt, x);
            }
#pragma unroll
            for (int off = 1; off < 16; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const float m_new = fmaxf(m[i], mt);
            const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
            const float corr = ex2f(m[i] - m_sub);  // 0 on the first visible tile
            float ls = 0.f;
#pragma unroll
            for (int c = 0; c < L::kKeys; ++c) {
                s[i][c] = ex2f(s[i][c] - m_sub);
                ls += s[i][c];
            }
            l[i] = fmaf(corr, l[i], ls);
            m[i] = m_new;
#pragma unroll
            for (int d = 0; d < 4 * L::kCols; ++d) acc[i][d] *= corr;
        }

        // P to shared memory: key-major, this thread's 8 rows contiguous.  Only
        // the 16 lanes of this half-warp read them back, so a warp barrier
        // orders both the previous tile's reads and this tile's reads.
        __syncwarp();
#pragma unroll
        for (int c = 0; c < L::kKeys; ++c) {
            float* dst = Ps + (cg + 16 * c) * L::kPStride + rg * kTiledRows;
            *reinterpret_cast<float4*>(dst) = make_float4(s[0][c], s[1][c], s[2][c], s[3][c]);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(s[4][c], s[5][c], s[6][c], s[7][c]);
        }
        __syncwarp();

        // O~ += P V
#pragma unroll 16
        for (int key = 0; key < BC; ++key) {
            const float4 pa = *reinterpret_cast<const float4*>(Ps + key * L::kPStride + rg * kTiledRows);
            const float4 pb = *reinterpret_cast<const float4*>(Ps + key * L::kPStride + rg * kTiledRows + 4);
            const float p[kTiledRows] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
            for (int u = 0; u < L::kCols; ++u) {
                const float4 vf = *reinterpret_cast<const float4*>(Vt + key * L::kStride + u * 64 + cg * 4);
#pragma unroll
                for (int i = 0; i < kTiledRows; ++i) {
                    fma2(acc[i][u * 4 + 0], acc[i][u * 4 + 1], p[i], p[i], vf.x, vf.y,
                         acc[i][u * 4 + 0], acc[i][u * 4 + 1]);
                    fma2(acc[i][u * 4 + 2], acc[i][u * 4 + 3], p[i], p[i], vf.z, vf.w,
                         acc[i][u * 4 + 2], acc[i][u * 4 + 3]);
                }
            }
        }
        __syncthreads();  // everyone is done with buffer `cur` before it is refilled
    }

    // Epilogue: row sums over the 16 owners, O = O~ / l (coalesced 16-byte
    // stores: a row's 16 owners cover 64 consecutive columns), LSE.
    float* oh = o + head;
#pragma unroll
    for (int i = 0; i < kTiledRows; ++i) {
        float lt = l[i];
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
        const int row = q_start + rg + 16 * i;
        if (row < N) {
            const float inv_l = 1.f / lt;
#pragma unroll
            for (int u = 0; u < L::kCols; ++u)
                *reinterpret_cast<float4*>(oh + static_cast<int64_t>(row) * D + u * 64 + cg * 4) =
                    make_float4(acc[i][u * 4] * inv_l, acc[i][u * 4 + 1] * inv_l,
                                acc[i][u * 4 + 2] * inv_l, acc[i][u * 4 + 3] * inv_l);
            if (cg == 0 && lse != nullptr)
                lse[static_cast<int64_t>(blockIdx.y) * N + row] = (m[i] + log2f(lt)) * kLn2;
        }
    }
}

template <int D, int BC, bool CAUSAL, int MIN_BLOCKS>
cudaError_t launch_ffma_tiled(const float* q, const float* k, const float* v, float* o, float* lse,
                              int BH, int H, int Hkv, int N, float scale_log2, cudaStream_t stream) {
    using L = TiledLayout<D, BC>;
    auto* fn = attn_fwd_ffma_tiled_kernel<D, BC, CAUSAL, MIN_BLOCKS>;
    static std::atomic<bool> done[kMaxDevices] = {};
    cudaError_t e = opt_in_smem_once(fn, L::kBytes, done);
    if (e != cudaSuccess) return e;
    const int num_qblk = (N + L::kBr - 1) / L::kBr;
    dim3 grid(num_qblk, BH);
    fn<<<grid, kTiledThreads, L::kBytes, stream>>>(q, k, v, o, lse, N, num_qblk, H, Hkv, scale_log2);
    return cudaGetLastError();
}

// K/V tile width and CTAs per SM of the register-tiled kernel.
constexpr int kTiledBc64 = 64, kTiledMinBlocks64 = 1;    // D = 64
constexpr int kTiledBc128 = 32, kTiledMinBlocks128 = 1;  // D = 128

}  // namespace

int ffma_bc(int D) { return D == 128 ? kTiledBc128 : kTiledBc64; }
int ffma_row_bc(int D) { return D == 128 ? 16 : 32; }
int ffma_threads(int) { return kTiledThreads; }
int ffma_smem_bytes(int D) {
    return D == 128 ? TiledLayout<128, kTiledBc128>::kBytes : TiledLayout<64, kTiledBc64>::kBytes;
}
int ffma_row_smem_bytes(int D) {
    return D == 128 ? RowLayout<128, 16>::kBytes : RowLayout<64, 32>::kBytes;
}

cudaError_t ffma_launch(const float* q, const float* k, const float* v, float* o, float* lse,
                        int64_t BH, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                        float scale_log2, bool causal, cudaStream_t stream) {
    const int bh = static_cast<int>(BH), n = static_cast<int>(N);
    const int h = static_cast<int>(H), hk = static_cast<int>(Hkv);
    if (D == 64)
        return causal ? launch_ffma_tiled<64, kTiledBc64, true, kTiledMinBlocks64>(
                            q, k, v, o, lse, bh, h, hk, n, scale_log2, stream)
                      : launch_ffma_tiled<64, kTiledBc64, false, kTiledMinBlocks64>(
                            q, k, v, o, lse, bh, h, hk, n, scale_log2, stream);
    return causal ? launch_ffma_tiled<128, kTiledBc128, true, kTiledMinBlocks128>(
                        q, k, v, o, lse, bh, h, hk, n, scale_log2, stream)
                  : launch_ffma_tiled<128, kTiledBc128, false, kTiledMinBlocks128>(
                        q, k, v, o, lse, bh, h, hk, n, scale_log2, stream);
}

cudaError_t ffma_row_launch(const float* q, const float* k, const float* v, float* o, float* lse,
                            int64_t BH, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                            float scale_log2, bool causal, cudaStream_t stream) {
    const int bh = static_cast<int>(BH), n = static_cast<int>(N);
    const int h = static_cast<int>(H), hk = static_cast<int>(Hkv);
    if (D == 64)
        return causal ? launch_ffma_row<64, 32, true>(q, k, v, o, lse, bh, h, hk, n, scale_log2, stream)
                      : launch_ffma_row<64, 32, false>(q, k, v, o, lse, bh, h, hk, n, scale_log2, stream);
    return causal ? launch_ffma_row<128, 16, true>(q, k, v, o, lse, bh, h, hk, n, scale_log2, stream)
                  : launch_ffma_row<128, 16, false>(q, k, v, o, lse, bh, h, hk, n, scale_log2, stream);
}

}  // namespace fattn
