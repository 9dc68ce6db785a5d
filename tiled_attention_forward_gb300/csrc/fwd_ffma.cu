// fwd_ffma.cu -- fp32 attention forward on CUDA cores (FFMA), sm_103a.
//
// The structure of the dandandamowang.xyz "Flash Attention (二) v2" page
// (§1.1 grid = (ceil(N/Br), B*H), one thread per query row, Br = 128; §3.2
// double-buffered cp.async K/V tiles with zero fill past N; §3.3 S row ->
// tile max -> P kept in registers -> merge -> unnormalised O update; §3.4
// causal KV loop cut at min(q_start+Br, N) plus the element mask on tiles
// crossing the diagonal; §3.5 one 1/l at the end), re-tuned for GB300:
//   * O~ accumulates in registers, not shared memory, so two CTAs fit per SM
//     (the page's 97 KB layout allowed one);
//   * exp2 with the scale and log2(e) folded into one multiply, and the
//     single-correction online-softmax form (chang-wenbin.github.io report
//     §2) -- one rescale factor per tile instead of two;
//   * Q and the output tile are staged through shared memory with a padded
//     row stride of D+4 floats, so that the per-row 16-byte reads and writes
//     of the 32 threads of a warp are bank-conflict free and the global
//     traffic is coalesced;
//   * K/V rows are read as 16-byte warp broadcasts (every thread of the warp
//     reads the same key), so the K/V tiles need no padding;
//   * under causal masking the Q blocks nearest the end of the sequence
//     (most K/V tiles) are launched first.
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

template <int D, int BC>
struct FfmaLayout {
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
    attn_fwd_ffma_kernel(const float* __restrict__ q, const float* __restrict__ k,
                         const float* __restrict__ v, float* __restrict__ o,
                         float* __restrict__ lse, int N, int num_qblk, int H, int Hkv,
                         float scale_log2) {
    using L = FfmaLayout<D, BC>;
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
cudaError_t launch_ffma(const float* q, const float* k, const float* v, float* o, float* lse,
                        int BH, int H, int Hkv, int N, float scale_log2, cudaStream_t stream) {
    using L = FfmaLayout<D, BC>;
    auto* fn = attn_fwd_ffma_kernel<D, BC, CAUSAL>;
    static bool done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !done[dev]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) done[dev] = true;
    }
    const int num_qblk = (N + L::kBr - 1) / L::kBr;
    dim3 grid(num_qblk, BH);
    fn<<<grid, L::kBr, L::kBytes, stream>>>(q, k, v, o, lse, N, num_qblk, H, Hkv, scale_log2);
    return cudaGetLastError();
}

}  // namespace

int ffma_bc(int D) { return D == 128 ? 16 : 32; }
int ffma_smem_bytes(int D) {
    return D == 128 ? FfmaLayout<128, 16>::kBytes : FfmaLayout<64, 32>::kBytes;
}

cudaError_t ffma_launch(const float* q, const float* k, const float* v, float* o, float* lse,
                        int64_t BH, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                        float scale_log2, bool causal, cudaStream_t stream) {
    const int bh = static_cast<int>(BH), n = static_cast<int>(N);
    const int h = static_cast<int>(H), hk = static_cast<int>(Hkv);
    if (D == 64)
        return causal ? launch_ffma<64, 32, true>(q, k, v, o, lse, bh, h, hk, n, scale_log2, stream)
                      : launch_ffma<64, 32, false>(q, k, v, o, lse, bh, h, hk, n, scale_log2, stream);
    return causal ? launch_ffma<128, 16, true>(q, k, v, o, lse, bh, h, hk, n, scale_log2, stream)
                  : launch_ffma<128, 16, false>(q, k, v, o, lse, bh, h, hk, n, scale_log2, stream);
}

}  // namespace fattn
