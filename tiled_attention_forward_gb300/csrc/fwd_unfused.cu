// fwd_unfused.cu -- the materialising (unfused) attention forward, kept as an
// in-library comparator for the fused kernel: S = scale Q K^T is written to
// HBM in fp32, a row softmax turns it into P (input dtype) and the LSE, and
// O = P V is a second contraction that reads P back.  This is the naive
// three-step algorithm of the cishoon.github.io "flashattention" page (§2:
// ScaledDotProduct -> Softmax -> PVMultiply, S and P materialised), whose HBM
// traffic the chang-wenbin.github.io FA2 report (§3) contrasts with the fused
// form.  Both contractions run on the tensor cores (tcgen05, operands by TMA)
// so that the comparison measures the memory traffic, not a slower math unit.
//
// Workspace layout (caller-owned): S fp32 [B*H][N][Np] then P 16-bit
// [B*H][N][Np], Np = N rounded up to a multiple of 8 (a TMA row pitch must be
// a multiple of 16 bytes).  Under causal masking S tiles wholly above the
// diagonal are neither computed nor read, and a row of P is written only up
// to the end of the last 128-key tile its Q tile reads (zeros for the hidden
// keys in that range).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace fattn {

namespace {

// Error word of this translation unit's kernels (device code is not linked
// across translation units, so each one keeps its own; the status call ORs
// them).  Same bit layout as the fused kernel's word.
__device__ uint32_t g_error_word;

constexpr int kUT = 128;                 // tile edge (rows, keys)
constexpr uint32_t kTmemCols = 128;

struct ScoreSmem {
    static constexpr int kQ = 0;                     // Q tile: D/64 atoms of [128][64]
    static constexpr int kK = 32 * 1024;             // K tile
    static constexpr int kBar = 64 * 1024;
    static constexpr int kBytes = kBar + 64;
};

// Kernel 1: S[bh][q0 + r][k0 + c] = scale * q . k for one 128 x 128 tile.
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(128, 1)
    unfused_scores_kernel(const __grid_constant__ UnfusedArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int kt = blockIdx.x, qt = blockIdx.y, bh = blockIdx.z;
    const int q0 = qt * kUT, k0 = kt * kUT;
    if (CAUSAL && k0 > q0 + kUT - 1) return;  // wholly above the diagonal: never read
    if ((smem_u32(smem) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicOr(&g_error_word, 1u << kDevErrInternal);
        return;
    }
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ScoreSmem::kBar);
    uint64_t* done = full + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(done, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    bool ok = true;
    if (threadIdx.x == 0) {
        constexpr int kAtoms = D / 64;
        mbar_arrive_expect_tx(full, 2 * kUT * D * 2);
        for (int at = 0; at < kAtoms; ++at) {
            tma_load_3d(smem + ScoreSmem::kQ + at * kUT * 128, &a.tmap_q, full, at * 64, q0, bh);
            tma_load_3d(smem + ScoreSmem::kK + at * kUT * 128, &a.tmap_k, full, at * 64, k0,
                        kv_head_of(bh, a.H, a.Hkv));
        }
        ok = mbar_wait_bounded(full, 0u, nullptr, &g_error_word, a.timeout_ns);
        if (ok) {
            tc_fence_after();
            const uint64_t desc = smem_desc_sw128(0u, 16u, 1024u);
            const uint64_t qd = desc + (smem_u32(smem + ScoreSmem::kQ) >> 4);
            const uint64_t kd = desc + (smem_u32(smem + ScoreSmem::kK) >> 4);
            constexpr uint32_t idesc = idesc_f16_f32(kUT, kUT, BF16 ? 1u : 0u, 0u, 0u);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = ((kk / 4) * (kUT * 128) + (kk % 4) * 32) >> 4;
                mma_ss(tmem, qd + off, kd + off, idesc, kk > 0 ? 1u : 0u);
            }
        }
        mma_commit(done);  // also when the load failed: the wait below must end
    }
    __syncwarp();
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(done, 0u, nullptr, &g_error_word, a.timeout_ns));
    tc_fence_after();
    if (ok) {
        // Each warp moves its 32 rows in 32 x 32 chunks through a 4 KB staging
        // buffer in the (now idle) Q tile, so that the global stores are
        // row-contiguous: 8 lanes write one row's 128 bytes, 4 rows per store.
        // Float4 slots are XOR-swizzled by row to keep both sides conflict-free.
        const int lane = threadIdx.x % 32;
        float4* stage = reinterpret_cast<float4*>(smem + ScoreSmem::kQ + warp * 4096);
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const int rsub = lane / 8, jsub = lane % 8;
#pragma unroll 1
        for (int c = 0; c < kUT / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(taddr + c * 32, v);
            tmem_wait_ld();
            reg_fence(v);
            __syncwarp();  // the previous chunk's reads of the staging buffer are done
#pragma unroll
            for (int j = 0; j < 8; ++j)
                stage[lane * 8 + (j ^ (lane & 7))] =
                    make_float4(__uint_as_float(v[4 * j]) * a.scale, __uint_as_float(v[4 * j + 1]) * a.scale,
                                __uint_as_float(v[4 * j + 2]) * a.scale, __uint_as_float(v[4 * j + 3]) * a.scale);
            __syncwarp();
            const int col = k0 + c * 32 + jsub * 4;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = it * 4 + rsub;
                const int row = q0 + warp * 32 + r;
                if (row < a.N && col < a.Np)
                    *reinterpret_cast<float4*>(a.s + (static_cast<int64_t>(bh) * a.N + row) * a.Np + col) =
                        stage[r * 8 + (jsub ^ (r & 7))];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
    if (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

constexpr int kSmThreads = 256;  // softmax: one CTA per row

// Maximum and sum over the CTA: warp shuffles, then the 8 warp results
// through shared memory.  Every thread returns the CTA-wide value.
__device__ __forceinline__ float cta_max(float x, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    __syncthreads();  // red is free (previous reduction fully read)
    if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = x;
    __syncthreads();
    x = red[0];
#pragma unroll
    for (int w = 1; w < kSmThreads / 32; ++w) x = fmaxf(x, red[w]);
    return x;
}

__device__ __forceinline__ float cta_sum(float x, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = x;
    __syncthreads();
    x = red[0];
#pragma unroll
    for (int w = 1; w < kSmThreads / 32; ++w) x += red[w];
    return x;
}

// Kernel 2: one CTA per row of S.  The visible scores are read once into
// registers (float4 i of the row goes to thread i % 256, slot i / 256; rows
// of up to kV * 1024 columns), the row maximum and the sum of exp(s - m)
// are CTA reductions, and P = exp(s - m) / l is written in the input dtype,
// with zeros for the hidden keys up to the last column the P V kernel reads
// for this row's Q tile.  LSE = m + ln(l).  Scores are handled in log2 units.
template <bool BF16, bool CAUSAL, int kV>
__global__ void __launch_bounds__(kSmThreads) unfused_softmax_kernel(const UnfusedArgs a) {
    __shared__ float red[kSmThreads / 32];
    const int64_t gr = blockIdx.x;  // row of [B*H*N]
    const int row = static_cast<int>(gr % a.N);
    const int nvis = CAUSAL ? row + 1 : a.N;
    // columns the P V kernel loads for this row's 128-row tile (a multiple of 8)
    const int ncols = CAUSAL ? min(a.Np, (row / kUT + 1) * kUT) : a.Np;
    const float* srow = a.s + gr * a.Np;
    constexpr float kLog2e = 1.4426950408889634f;

    float x[kV][4];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int j = (i * kSmThreads + static_cast<int>(threadIdx.x)) * 4;
        float4 x4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (j < nvis) x4 = *reinterpret_cast<const float4*>(srow + j);  // j+3 < Np: in the row
        x[i][0] = x4.x * kLog2e;
        x[i][1] = (j + 1 < nvis) ? x4.y * kLog2e : -INFINITY;
        x[i][2] = (j + 2 < nvis) ? x4.z * kLog2e : -INFINITY;
        x[i][3] = (j + 3 < nvis) ? x4.w * kLog2e : -INFINITY;
        m = fmaxf(m, fmaxf(fmaxf(x[i][0], x[i][1]), fmaxf(x[i][2], x[i][3])));
    }
    m = cta_max(m, red);  // finite: column 0 is visible to every row
    float l = 0.f;
#pragma unroll
    for (int i = 0; i < kV; ++i) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[i][e] = exp2f(x[i][e] - m);  // exp2(-inf) = 0 for the hidden ones
            l += x[i][e];
        }
    }
    l = cta_sum(l, red);
    const float inv_l = 1.f / l;
    uint2* prow = reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(a.p) + gr * a.Np * 2);
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int j = (i * kSmThreads + static_cast<int>(threadIdx.x)) * 4;
        if (j < ncols)
            prow[j / 4] = make_uint2(pack_p<BF16>(x[i][0] * inv_l, x[i][1] * inv_l),
                                     pack_p<BF16>(x[i][2] * inv_l, x[i][3] * inv_l));
    }
    if (threadIdx.x == 0 && a.lse != nullptr) a.lse[gr] = (m + log2f(l)) * 0.6931471805599453f;
}

// Kernel 2 for rows longer than the register cache holds (Np > 16384): the
// same result from two passes over S (maximum and sum with the online
// normaliser's rescaling, then P).
template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kSmThreads) unfused_softmax_long_kernel(const UnfusedArgs a) {
    __shared__ float red[kSmThreads / 32];
    const int64_t gr = blockIdx.x;
    const int row = static_cast<int>(gr % a.N);
    const int nvis = CAUSAL ? row + 1 : a.N;
    const int ncols = CAUSAL ? min(a.Np, (row / kUT + 1) * kUT) : a.Np;
    const float* srow = a.s + gr * a.Np;
    constexpr float kLog2e = 1.4426950408889634f;
    float m = -INFINITY, l = 0.f;
    for (int j = threadIdx.x; j < nvis; j += kSmThreads) {
        const float x = srow[j] * kLog2e;
        if (x > m) {
            l = l * exp2f(m - x) + 1.f;
            m = x;
        } else {
            l += exp2f(x - m);
        }
    }
    const float mt = cta_max(m, red);
    l = cta_sum(m == -INFINITY ? 0.f : l * exp2f(m - mt), red);
    m = mt;
    const float inv_l = 1.f / l;
    uint16_t* prow = reinterpret_cast<uint16_t*>(a.p) + gr * a.Np;
    for (int j = threadIdx.x; j < ncols; j += kSmThreads) {
        const float p = j < nvis ? exp2f(srow[j] * kLog2e - m) * inv_l : 0.f;
        prow[j] = static_cast<uint16_t>(pack_p<BF16>(p, 0.f) & 0xFFFFu);
    }
    if (threadIdx.x == 0 && a.lse != nullptr) a.lse[gr] = (m + log2f(l)) * 0.6931471805599453f;
}

template <int D>
struct PvSmem {
    static constexpr int kPTile = kUT * kUT * 2;   // 128 rows x 128 keys, 16-bit (2 atoms)
    static constexpr int kVTile = kUT * D * 2;     // 128 keys x D
    static constexpr int kStage = kPTile + kVTile;
    static constexpr int kStages = 2;
    static constexpr int kBar = kStages * kStage;
    static constexpr int kBytes = kBar + 64;
};

// Kernel 3: O[bh][q0..q0+127][:] = P[bh][q0.., :] V[kv head]: SS-form MMAs,
// A = P tile (K-major over keys), B = V tile (MN-major), two-stage TMA ring.
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(128, 1) unfused_pv_kernel(const __grid_constant__ UnfusedArgs a) {
    using L = PvSmem<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    if ((smem_u32(smem) & 1023u) != 0u) {
        if (threadIdx.x == 0) atomicOr(&g_error_word, 1u << kDevErrInternal);
        return;
    }
    const int qt = blockIdx.x, bh = blockIdx.y;
    const int q0 = qt * kUT;
    const int kv_limit = CAUSAL ? min(q0 + kUT, a.N) : a.N;
    const int nkb = (kv_limit + kUT - 1) / kUT;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);   // [2]
    uint64_t* empty = full + 2;                                      // [2]
    uint64_t* done = full + 4;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(full + 5);
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int kvh = kv_head_of(bh, a.H, a.Hkv);

    if (threadIdx.x == 0) {
        int issued = 0;  // loads started, in order 0, 1, ...
        auto load = [&](int kb) {
            const int s = kb % 2;
            uint8_t* st = smem + s * L::kStage;
            mbar_arrive_expect_tx(&full[s], L::kStage);
            for (int at = 0; at < 2; ++at)  // 128 keys of P = two 64-key atoms
                tma_load_3d(st + at * kUT * 128, &a.tmap_p, &full[s], kb * kUT + at * 64, q0, bh);
            for (int at = 0; at < D / 64; ++at)  // V: 64-wide feature slabs
                tma_load_3d(st + L::kPTile + at * kUT * 128, &a.tmap_v, &full[s], at * 64, kb * kUT, kvh);
            ++issued;
        };
        constexpr uint32_t idesc = idesc_f16_f32(kUT, D, BF16 ? 1u : 0u, 0u, 1u);
        const uint64_t pdesc0 = smem_desc_sw128(0u, 16u, 1024u);
        const uint64_t vdesc0 = smem_desc_sw128(0u, kUT * 128u, 1024u);
        bool ok = true;
        load(0);
        for (int kb = 0; kb < nkb && ok; ++kb) {
            const int s = kb % 2;
            if (kb + 1 < nkb) {
                if (kb >= 1)  // the other stage was last read by the MMAs of kb-1
                    ok = mbar_wait_bounded(&empty[(kb + 1) % 2], ((kb - 1) / 2) & 1u, nullptr,
                                           &g_error_word, a.timeout_ns);
                if (!ok) break;
                load(kb + 1);
            }
            ok = mbar_wait_bounded(&full[s], (kb / 2) & 1u, nullptr, &g_error_word, a.timeout_ns);
            if (!ok) break;
            tc_fence_after();
            const uint64_t pd = pdesc0 + (smem_u32(smem + s * L::kStage) >> 4);
            const uint64_t vd = vdesc0 + (smem_u32(smem + s * L::kStage + L::kPTile) >> 4);
#pragma unroll
            for (int kk = 0; kk < kUT / 16; ++kk) {
                const uint64_t poff = ((kk / 4) * (kUT * 128) + (kk % 4) * 32) >> 4;
                mma_ss(tmem, pd + poff, vd + ((kk * 16 * 128) >> 4), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&empty[s]);
        }
        if (!ok) {
            // Let every copy already started land before the CTA leaves.
            for (int s = 0; s < 2; ++s) {
                const int last = issued - 1 - ((issued - 1 - s) % 2 + 2) % 2;  // last load of stage s
                if (last >= 0)
                    mbar_wait_bounded(&full[s], (last / 2) & 1u, nullptr, &g_error_word, a.timeout_ns);
            }
        }
        mma_commit(done);
    }
    __syncwarp();
    mbar_wait_bounded(done, 0u, nullptr, &g_error_word, a.timeout_ns);
    tc_fence_after();
    // A failed wait has already set the error word; O is then undefined.
    const int row = q0 + warp * 32 + threadIdx.x % 32;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    uint8_t* orow = reinterpret_cast<uint8_t*>(a.o) + (static_cast<int64_t>(bh) * a.N + row) * D * 2;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(taddr + c * 32, v);  // warp-collective: every lane, whatever its row
        tmem_wait_ld();
        reg_fence(v);
        if (row < a.N) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = pack_p<BF16>(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
                dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_all(const UnfusedArgs& a, cudaStream_t stream) {
    const int nt = (a.N + kUT - 1) / kUT;
    auto* k1 = unfused_scores_kernel<D, BF16, CAUSAL>;
    static std::atomic<bool> k1_done[kMaxDevices] = {};
    static std::atomic<bool> k3_done[kMaxDevices] = {};
    cudaError_t e = opt_in_smem_once(k1, ScoreSmem::kBytes, k1_done);
    if (e != cudaSuccess) return e;
    k1<<<dim3(nt, nt, a.BH), 128, ScoreSmem::kBytes, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(a.BH) * a.N;
    const unsigned grid2 = static_cast<unsigned>(rows);
    const int need = (a.Np + 4 * kSmThreads - 1) / (4 * kSmThreads);  // float4 slots per thread
    if (need <= 1) unfused_softmax_kernel<BF16, CAUSAL, 1><<<grid2, kSmThreads, 0, stream>>>(a);
    else if (need <= 2) unfused_softmax_kernel<BF16, CAUSAL, 2><<<grid2, kSmThreads, 0, stream>>>(a);
    else if (need <= 4) unfused_softmax_kernel<BF16, CAUSAL, 4><<<grid2, kSmThreads, 0, stream>>>(a);
    else if (need <= 8) unfused_softmax_kernel<BF16, CAUSAL, 8><<<grid2, kSmThreads, 0, stream>>>(a);
    else if (need <= 16) unfused_softmax_kernel<BF16, CAUSAL, 16><<<grid2, kSmThreads, 0, stream>>>(a);
    else unfused_softmax_long_kernel<BF16, CAUSAL><<<grid2, kSmThreads, 0, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    auto* k3 = unfused_pv_kernel<D, BF16, CAUSAL>;
    e = opt_in_smem_once(k3, PvSmem<D>::kBytes, k3_done);
    if (e != cudaSuccess) return e;
    k3<<<dim3(nt, a.BH), 128, PvSmem<D>::kBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

// Fixed workspace of fattn_fwd_unfused_static: one array per device, in the
// module's static device memory, so that the call allocates nothing.  Every
// element a call reads is written earlier in the same call, so nothing in it
// has to start at zero.
static __device__ __align__(256) uint8_t g_unfused_static_scratch[kUnfusedStaticBytes];

cudaError_t unfused_static_scratch(void** ptr) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        e = cudaGetSymbolAddress(&addr[dev], g_unfused_static_scratch);
        if (e != cudaSuccess) {
            addr[dev] = nullptr;
            return e;
        }
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

cudaError_t unfused_read_and_clear_error_word(uint32_t* out) {
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v));
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    *out = v;
    return e;
}

int64_t unfused_row_pitch(int64_t N) { return (N + 7) / 8 * 8; }

size_t unfused_workspace_bytes(int64_t BH, int64_t N) {
    const int64_t np = unfused_row_pitch(N);
    return static_cast<size_t>(BH * N * np) * (4 + 2);
}

cudaError_t unfused_launch(const UnfusedArgs& a, int D, bool bf16, bool causal, cudaStream_t s) {
    if (D == 128) {
        if (bf16) return causal ? launch_all<128, true, true>(a, s) : launch_all<128, true, false>(a, s);
        return causal ? launch_all<128, false, true>(a, s) : launch_all<128, false, false>(a, s);
    }
    if (bf16) return causal ? launch_all<64, true, true>(a, s) : launch_all<64, true, false>(a, s);
    return causal ? launch_all<64, false, true>(a, s) : launch_all<64, false, false>(a, s);
}

}  // namespace fattn
