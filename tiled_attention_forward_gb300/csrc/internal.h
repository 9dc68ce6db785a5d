// internal.h -- declarations shared by the translation units of libfattn.
// Not part of the public ABI (see include/fattn.h).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fattn {

constexpr int kMaxDevices = 64;

// Raises one kernel's dynamic shared-memory limit once per device.  Each call
// site passes its own flag array; the flags are atomics, so host threads that
// launch at the same time never race on them (setting the attribute twice is
// harmless).
template <typename K>
inline cudaError_t opt_in_smem_once(K* fn, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool known = dev >= 0 && dev < kMaxDevices;
    if (known && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (known) done[dev].store(true, std::memory_order_release);
    return cudaSuccess;
}

// ---- tensor-core path (bf16 / fp16), fwd_tc.cu ------------------------------
constexpr int kTcBM = 128;        // Q rows per MMA tile (tcgen05 M)
constexpr int kTcQTiles = 2;      // Q tiles per task (rows per task = 256)
constexpr int kTcBN = 128;        // keys per K/V tile (N of S = Q K^T)
constexpr int kTcThreads = 384;   // 2 softmax warpgroups + 1 control warpgroup (MMA, TMA)

struct TcArgs {
    CUtensorMap tmap_q;  // 3-D {D, N, B*H}, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    void* o;             // [B,H,N,D] output, input dtype
    float* lse;          // [B,H,N] or nullptr
    int N;
    int BH;              // B * H query heads (task space)
    int H;               // query heads per batch
    int Hkv;             // key/value heads per batch (H % Hkv == 0)
    int num_qblk;        // ceil(N / 256)
    int num_tasks;       // BH * num_qblk
    int head_group;      // causal task order: query heads per group (K/V of a group stays in L2)
    float scale_log2;    // scale * log2(e)
    uint64_t timeout_ns; // bound of every barrier wait
};

int tc_smem_bytes(int D);
int tc_num_stages(int D);
// Encodes the three tensor maps of `a` for these buffers (host).
cudaError_t tc_encode_maps(TcArgs& a, const void* q, const void* k, const void* v, int64_t BH,
                           int64_t BHkv, int64_t N, int64_t D, bool bf16);
cudaError_t tc_launch(const TcArgs& a, int D, bool bf16, bool causal, int grid,
                      cudaStream_t stream);

// ---- CUDA-core path (fp32), fwd_ffma.cu --------------------------------------
constexpr int kFfmaBr = 128;      // Q rows per CTA
int ffma_bc(int D);               // keys per K/V tile
int ffma_threads(int D);          // threads per CTA
int ffma_smem_bytes(int D);
cudaError_t ffma_launch(const float* q, const float* k, const float* v, float* o, float* lse,
                        int64_t BH, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                        float scale_log2, bool causal, cudaStream_t stream);
// One query row per thread (Br = 128 threads), the page's own design.
int ffma_row_bc(int D);
int ffma_row_smem_bytes(int D);
cudaError_t ffma_row_launch(const float* q, const float* k, const float* v, float* o, float* lse,
                            int64_t BH, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                            float scale_log2, bool causal, cudaStream_t stream);

// ---- unfused comparator (bf16 / fp16), fwd_unfused.cu ----------------------
struct UnfusedArgs {
    CUtensorMap tmap_q;  // as TcArgs: 3-D {D, N, heads}, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    CUtensorMap tmap_p;  // 3-D {Np, N, B*H} over the P part of the workspace, same box
    float* s;            // workspace: S fp32 [B*H][N][Np]
    void* p;             // workspace: P 16-bit [B*H][N][Np]
    void* o;             // [B,H,N,D] output, input dtype
    float* lse;          // [B,H,N] or nullptr
    int N;
    int Np;              // row pitch of S and P in elements (N rounded up to 8)
    int BH;
    int H;
    int Hkv;
    float scale;         // natural-log units (S = scale Q K^T)
    uint64_t timeout_ns;
};

int64_t unfused_row_pitch(int64_t N);
size_t unfused_workspace_bytes(int64_t BH, int64_t N);
cudaError_t unfused_encode_p_map(UnfusedArgs& a, int64_t BH, int64_t N, bool bf16);
cudaError_t unfused_launch(const UnfusedArgs& a, int D, bool bf16, bool causal, cudaStream_t s);
cudaError_t unfused_read_and_clear_error_word(uint32_t* out);
// Device address of the fixed workspace of fattn_fwd_unfused_static on the
// current device (looked up once per device).
constexpr size_t kUnfusedStaticBytes = size_t(64) << 20;
cudaError_t unfused_static_scratch(void** ptr);

// ---- backward (bf16 / fp16), bwd_tc.cu --------------------------------------
struct BwdArgs {
    CUtensorMap tmap_q;   // 3-D {D, N, B*H}, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    CUtensorMap tmap_do;
    float* ws;            // [B*H][2][Npad]: LSE*log2(e) (+inf past N), Delta (0 past N)
    void* dq;             // [B,H,N,D] outputs, input dtype
    void* dk;
    void* dv;
    int N;
    int Npad;             // N rounded up to 128
    int BH;               // B * H query heads
    int H;                // query heads per batch
    int Hkv;              // key/value heads per batch (H % Hkv == 0)
    int BHkv;             // B * Hkv
    int num_tiles;        // Npad / 128
    float sl2;            // scale * log2(e)
    float scale;
    uint64_t timeout_ns;
};

int64_t bwd_padded_rows(int64_t N);
cudaError_t bwd_launch(const BwdArgs& a, const void* o, const void* dout, const float* lse, int D,
                       bool bf16, bool causal, cudaStream_t s);
cudaError_t bwd_read_and_clear_error_word(uint32_t* out);

// Key/value head read by query head bh = b*H + h: b*Hkv + h / (H/Hkv).
__host__ __device__ __forceinline__ int kv_head_of(int bh, int H, int Hkv) {
    return (bh / H) * Hkv + (bh % H) / (H / Hkv);
}

// ---- device error word (fwd_tc.cu) -----------------------------------------
cudaError_t read_and_clear_error_word(uint32_t* out);
cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t stream);

}  // namespace fattn
