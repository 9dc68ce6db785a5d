// fattn_api.cu -- the C ABI of libfattn (declared in include/fattn.h):
// argument validation, launch planning, TMA tensor-map encoding and dispatch
// to the tensor-core (bf16/fp16) or CUDA-core (fp32) kernel.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <cudaTypedefs.h>

#include "fattn.h"
#include "internal.h"

namespace fattn {
namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per barrier wait
constexpr int64_t kMaxElements = int64_t(1) << 52;      // bound of B*H*N*D accepted by validate()

// The fixed array behind fattn_fwd_unfused_static and the size the header
// promises are one number.
static_assert(static_cast<long long>(kUnfusedStaticBytes) == FATTN_UNFUSED_STATIC_BYTES,
              "static workspace size must match the public header");
constexpr float kLog2e = 1.4426950408889634f;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }

size_t elem_bytes(int dtype) { return dtype == FATTN_F32 ? 4u : 2u; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Validation shared by every compute entry point; returns FATTN_OK when the
// call may proceed (which includes the empty problem, flagged by *empty).
int validate(const void* q, const void* k, const void* v, const void* o, const float* lse,
             int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D, float scale, int dtype,
             bool* empty) {
    *empty = false;
    if (dtype != FATTN_F32 && dtype != FATTN_F16 && dtype != FATTN_BF16) return FATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || N < 0 || D < 0) return FATTN_ERR_INVALID_ARG;
    if (H > 0 && (Hkv <= 0 || H % Hkv != 0)) return FATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || scale < 0.f) return FATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0) {
        *empty = true;
        return FATTN_OK;
    }
    // Index ranges: N and B*H fit int32 (kernel indices, TMA coordinates,
    // grid.y <= 65535 on the FFMA path), and B*H*N*D is bounded by 2^52
    // elements, so that every byte count formed below stays far inside int64
    // (no device holds a problem anywhere near that size).
    if (N > (int64_t(1) << 30) || B > (int64_t(1) << 30) || H > (int64_t(1) << 30))
        return FATTN_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    if (BH > (int64_t(1) << 30)) return FATTN_ERR_UNSUPPORTED;
    if (BH * N > kMaxElements / D) return FATTN_ERR_UNSUPPORTED;  // BH*N <= 2^60: no overflow
    if (dtype == FATTN_F32 && BH > 65535) return FATTN_ERR_UNSUPPORTED;
    if (!q || !k || !v || !o) return FATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FATTN_ERR_MISALIGNED;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FATTN_ERR_MISALIGNED;
    const size_t bytes = static_cast<size_t>(BH * N * D) * elem_bytes(dtype);
    const size_t kvbytes = static_cast<size_t>(B * Hkv * N * D) * elem_bytes(dtype);
    if (overlaps(o, bytes, q, bytes) || overlaps(o, bytes, k, kvbytes) ||
        overlaps(o, bytes, v, kvbytes))
        return FATTN_ERR_INVALID_ARG;
    if (lse) {
        const size_t lb = static_cast<size_t>(BH * N) * sizeof(float);
        if (overlaps(lse, lb, o, bytes) || overlaps(lse, lb, q, bytes) ||
            overlaps(lse, lb, k, kvbytes) || overlaps(lse, lb, v, kvbytes))
            return FATTN_ERR_INVALID_ARG;
    }
    return FATTN_OK;
}

int current_sm_count(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FATTN_ERR_NO_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FATTN_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return FATTN_ERR_NO_DEVICE;  // built for sm_103a only
    return FATTN_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// K/V tiles one task visits: Q rows [r0, r0+rows) against keys, Bc-key tiles.
int64_t kv_tiles_for(int64_t r0, int64_t rows, int64_t N, int64_t bc, bool causal) {
    if (r0 >= N) return 0;
    const int64_t kv_limit = causal ? std::min(r0 + rows, N) : N;
    return ceil_div(kv_limit, bc);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    // Looked up once; a function-local static is initialised exactly once even
    // when several host threads make their first call at the same time.
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qres) == cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// Per-device helpers of fattn_fwd_host: a copy-in stream, a copy-out stream
// and the events that chain them to the caller's stream, created on the first
// call on the device and kept for the process lifetime.
constexpr int kHostChunks = 4;

struct HostPipe {
    cudaStream_t in = nullptr;
    cudaStream_t out = nullptr;
    cudaEvent_t fork = nullptr;
    cudaEvent_t join = nullptr;
    cudaEvent_t in_done[kHostChunks] = {};
    cudaEvent_t k_done[kHostChunks] = {};
    bool ready = false;
};

HostPipe g_host_pipes[kMaxDevices];
std::mutex g_host_mu;  // also serialises the enqueue sequence of fattn_fwd_host

cudaError_t host_pipe(HostPipe** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    HostPipe& p = g_host_pipes[dev];
    if (!p.ready) {
        const unsigned ev = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.fork, ev)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.join, ev)) != cudaSuccess)
            return e;
        for (int c = 0; c < kHostChunks; ++c)
            if ((e = cudaEventCreateWithFlags(&p.in_done[c], ev)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&p.k_done[c], ev)) != cudaSuccess)
                return e;
        p.ready = true;
    }
    *out = &p;
    return cudaSuccess;
}

// Causal task order: query heads per group.  A group's K/V (16-bit) is
// sized to stay in L2 while its tasks run (about 48 MB, so that the next
// group's first tasks fit beside the last ones of this group), whole K/V
// heads at a time (H / Hkv query heads share one), and the groups are made
// as equal as the head count allows.
int causal_head_group(int64_t BH, int64_t H, int64_t Hkv, int64_t N, int64_t D) {
    constexpr int64_t kL2Budget = 48ll << 20;
    const int64_t share = H / Hkv;
    const int64_t kv_bytes = 2 * N * D * 2;
    const int64_t kv_heads = std::max<int64_t>(1, kL2Budget / std::max<int64_t>(kv_bytes, 1));
    const int64_t cap = std::min<int64_t>(BH, kv_heads * share);
    const int64_t groups = ceil_div(BH, cap);
    int64_t hg = ceil_div(BH, groups);
    hg = ceil_div(hg, share) * share;  // whole K/V heads
    return static_cast<int>(std::min<int64_t>(hg, BH));
}

}  // namespace

cudaError_t tc_encode_maps(TcArgs& a, const void* q, const void* k, const void* v, int64_t BH,
                           int64_t BHkv, int64_t N, int64_t D, bool bf16) {
    auto encode = get_encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const CUtensorMapDataType dt =
        bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // [heads][N][D] row-major, 16-bit: innermost D, then rows, then heads
    // (B*H heads for Q, B*Hkv for K and V).
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2), static_cast<cuuint64_t>(N * D * 2)};
    const cuuint32_t box[3] = {64, 128, 1};  // one 128-byte swizzle atom wide, 128 rows
    const cuuint32_t estr[3] = {1, 1, 1};
    const void* ptrs[3] = {q, k, v};
    const int64_t heads[3] = {BH, BHkv, BHkv};
    CUtensorMap* maps[3] = {&a.tmap_q, &a.tmap_k, &a.tmap_v};
    for (int i = 0; i < 3; ++i) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                                    static_cast<cuuint64_t>(heads[i])};
        CUresult r = encode(maps[i], dt, 3, const_cast<void*>(ptrs[i]), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

cudaError_t unfused_encode_p_map(UnfusedArgs& a, int64_t BH, int64_t N, bool bf16) {
    auto encode = get_encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const int64_t np = unfused_row_pitch(N);
    const CUtensorMapDataType dt =
        bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // P: [B*H][N][Np] 16-bit; keys innermost, 64 keys (128 bytes) per box row
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(np), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(np * 2), static_cast<cuuint64_t>(N * np * 2)};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(&a.tmap_p, dt, 3, a.p, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace fattn

using namespace fattn;

extern "C" {

int fattn_version(void) { return 10000; }

const char* fattn_status_string(int status) {
    switch (status) {
        case FATTN_OK: return "FATTN_OK";
        case FATTN_ERR_INVALID_ARG: return "FATTN_ERR_INVALID_ARG";
        case FATTN_ERR_UNSUPPORTED: return "FATTN_ERR_UNSUPPORTED";
        case FATTN_ERR_MISALIGNED: return "FATTN_ERR_MISALIGNED";
        case FATTN_ERR_CUDA: return "FATTN_ERR_CUDA";
        case FATTN_ERR_TIMEOUT: return "FATTN_ERR_TIMEOUT";
        case FATTN_ERR_NO_DEVICE: return "FATTN_ERR_NO_DEVICE";
        case FATTN_ERR_INTERNAL: return "FATTN_ERR_INTERNAL";
        default: return "FATTN_ERR_UNKNOWN";
    }
}

int fattn_plan_head_group(int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                          int64_t* head_group) {
    if (!head_group) return FATTN_ERR_INVALID_ARG;
    *head_group = 0;
    if (B < 1 || H < 1 || Hkv < 1 || N < 1 || (D != 64 && D != 128) || H % Hkv != 0)
        return FATTN_ERR_INVALID_ARG;
    if (N > (int64_t(1) << 30) || B > (int64_t(1) << 30) || H > (int64_t(1) << 30) ||
        B * H > (int64_t(1) << 30))
        return FATTN_ERR_UNSUPPORTED;
    *head_group = causal_head_group(B * H, H, Hkv, N, D);
    return FATTN_OK;
}

int fattn_plan(int64_t B, int64_t H, int64_t N, int64_t D, int causal, int dtype, int num_sms,
               int64_t out[9]) {
    if (!out) return FATTN_ERR_INVALID_ARG;
    for (int i = 0; i < 9; ++i) out[i] = 0;
    if (dtype != FATTN_F32 && dtype != FATTN_F16 && dtype != FATTN_BF16) return FATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || N < 0 || D < 0) return FATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0) return FATTN_OK;
    if (N > (int64_t(1) << 30) || B > (int64_t(1) << 30) || H > (int64_t(1) << 30) ||
        B * H > (int64_t(1) << 30))
        return FATTN_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    const bool c = causal != 0;
    if (dtype == FATTN_F32) {
        const int64_t bc = ffma_bc(static_cast<int>(D));
        const int64_t nq = ceil_div(N, kFfmaBr);
        int64_t tiles = 0;
        for (int64_t qb = 0; qb < nq; ++qb) tiles += kv_tiles_for(qb * kFfmaBr, kFfmaBr, N, bc, c);
        out[0] = 1;
        out[1] = nq;
        out[2] = BH;
        out[3] = ffma_threads(static_cast<int>(D));
        out[4] = ffma_smem_bytes(static_cast<int>(D));
        out[5] = nq * BH;
        out[6] = tiles * BH;
        out[7] = kFfmaBr;
        out[8] = bc;
        return FATTN_OK;
    }
    if (num_sms <= 0) {
        int st = current_sm_count(&num_sms);
        if (st != FATTN_OK) return st;
    }
    const int64_t rows = int64_t(kTcBM) * kTcQTiles;
    const int64_t nq = ceil_div(N, rows);
    int64_t tiles = 0;
    for (int64_t qb = 0; qb < nq; ++qb) {
        const int64_t t0 = kv_tiles_for(qb * rows, kTcBM, N, kTcBN, c);
        const int64_t t1 = kv_tiles_for(qb * rows + kTcBM, kTcBM, N, kTcBN, c);
        tiles += std::max(t0, t1);  // the CTA streams each K/V tile once for both Q tiles
    }
    const int64_t tasks = nq * BH;
    out[0] = 2;
    out[1] = std::min<int64_t>(tasks, num_sms);
    out[2] = 1;
    out[3] = kTcThreads;
    out[4] = tc_smem_bytes(static_cast<int>(D));
    out[5] = tasks;
    out[6] = tiles * BH;
    out[7] = rows;
    out[8] = kTcBN;
    return FATTN_OK;
}

int fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
              int64_t N, int64_t D, float scale, int causal, int dtype, fattn_stream_t stream_h) {
    return fattn_fwd_gqa(q, k, v, o, lse, B, H, H, N, D, scale, causal, dtype, stream_h);
}

int fattn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                  int64_t H, int64_t Hkv, int64_t N, int64_t D, float scale, int causal, int dtype,
                  fattn_stream_t stream_h) {
    bool empty = false;
    int st = validate(q, k, v, o, lse, B, H, Hkv, N, D, scale, dtype, &empty);
    if (st != FATTN_OK || empty) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    const int64_t BH = B * H;
    const float scale_log2 = scale * kLog2e;

    if (dtype == FATTN_F32) {
        int sms = 0;
        st = current_sm_count(&sms);
        if (st != FATTN_OK) return st;
        cudaError_t e = ffma_launch(static_cast<const float*>(q), static_cast<const float*>(k),
                                    static_cast<const float*>(v), static_cast<float*>(o), lse, BH, H,
                                    Hkv, N, D, scale_log2, causal != 0, stream);
        return e == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
    }

    // Task indices (256-row Q blocks x heads) are ints in the kernel.
    if (ceil_div(N, int64_t(kTcBM) * kTcQTiles) * BH > (int64_t(1) << 30)) return FATTN_ERR_UNSUPPORTED;
    int sms = 0;
    st = current_sm_count(&sms);
    if (st != FATTN_OK) return st;
    TcArgs a;
    std::memset(&a, 0, sizeof(a));
    const bool bf16 = dtype == FATTN_BF16;
    if (tc_encode_maps(a, q, k, v, BH, B * Hkv, N, D, bf16) != cudaSuccess) return FATTN_ERR_CUDA;
    a.o = o;
    a.lse = lse;
    a.N = static_cast<int>(N);
    a.BH = static_cast<int>(BH);
    a.H = static_cast<int>(H);
    a.Hkv = static_cast<int>(Hkv);
    a.num_qblk = static_cast<int>(ceil_div(N, int64_t(kTcBM) * kTcQTiles));
    a.num_tasks = a.num_qblk * a.BH;
    a.head_group = causal_head_group(BH, H, Hkv, N, D);
    a.scale_log2 = scale_log2;
    a.timeout_ns = kDefaultTimeoutNs;
    const int grid = static_cast<int>(std::min<int64_t>(a.num_tasks, sms));
    cudaError_t e = tc_launch(a, static_cast<int>(D), bf16, causal != 0, grid, stream);
    return e == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

int fattn_fwd_f32_rowwise(const float* q, const float* k, const float* v, float* o, float* lse,
                          int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal,
                          fattn_stream_t stream_h) {
    bool empty = false;
    int st = validate(q, k, v, o, lse, B, H, H, N, D, scale, FATTN_F32, &empty);
    if (st != FATTN_OK || empty) return st;
    int sms = 0;
    st = current_sm_count(&sms);
    if (st != FATTN_OK) return st;
    cudaError_t e = ffma_row_launch(q, k, v, o, lse, B * H, H, H, N, D, scale * kLog2e, causal != 0,
                                    reinterpret_cast<cudaStream_t>(stream_h));
    return e == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

int fattn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                   float* lse_host, void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev,
                   int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal, int dtype,
                   fattn_stream_t stream_h) {
    bool empty = false;
    int st = validate(q_dev, k_dev, v_dev, o_dev, lse_dev, B, H, H, N, D, scale, dtype, &empty);
    if (st != FATTN_OK || empty) return st;
    if (!q_host || !k_host || !v_host || !o_host) return FATTN_ERR_INVALID_ARG;
    int sms = 0;
    st = current_sm_count(&sms);
    if (st != FATTN_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    std::lock_guard<std::mutex> lock(g_host_mu);
    HostPipe* p = nullptr;
    if (host_pipe(&p) != cudaSuccess) return FATTN_ERR_CUDA;
    // Heads in up to kHostChunks groups: the copies of group c+1 run on the
    // copy-in stream while the kernel of group c runs on `stream`, and O of
    // group c returns on the copy-out stream meanwhile.  The fp32 kernel runs
    // far longer than the copies and loses more to the partial last wave of
    // each group than the overlap gains, so it runs as one group.
    const int64_t BH = B * H;
    const int chunks = dtype == FATTN_F32 ? 1 : static_cast<int>(std::min<int64_t>(kHostChunks, BH));
    const size_t row = static_cast<size_t>(N * D) * elem_bytes(dtype);  // one head of Q, K, V or O
    const bool with_lse = lse_host && lse_dev;
    auto bptr = [](const void* base, size_t off) {
        return static_cast<void*>(static_cast<uint8_t*>(const_cast<void*>(base)) + off);
    };
    if (cudaEventRecord(p->fork, stream) != cudaSuccess || cudaStreamWaitEvent(p->in, p->fork, 0) != cudaSuccess)
        return FATTN_ERR_CUDA;
    for (int c = 0; c < chunks; ++c) {
        const int64_t h0 = BH * c / chunks, h1 = BH * (c + 1) / chunks;
        const size_t off = static_cast<size_t>(h0) * row, len = static_cast<size_t>(h1 - h0) * row;
        if (cudaMemcpyAsync(bptr(q_dev, off), bptr(q_host, off), len, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
            cudaMemcpyAsync(bptr(k_dev, off), bptr(k_host, off), len, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
            cudaMemcpyAsync(bptr(v_dev, off), bptr(v_host, off), len, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
            cudaEventRecord(p->in_done[c], p->in) != cudaSuccess ||
            cudaStreamWaitEvent(stream, p->in_done[c], 0) != cudaSuccess)
            return FATTN_ERR_CUDA;
        float* lse_c = lse_dev ? lse_dev + h0 * N : nullptr;
        st = fattn_fwd(bptr(q_dev, off), bptr(k_dev, off), bptr(v_dev, off), bptr(o_dev, off), lse_c, 1,
                       h1 - h0, N, D, scale, causal, dtype, stream_h);
        if (st != FATTN_OK) return st;
        if (cudaEventRecord(p->k_done[c], stream) != cudaSuccess ||
            cudaStreamWaitEvent(p->out, p->k_done[c], 0) != cudaSuccess ||
            cudaMemcpyAsync(bptr(o_host, off), bptr(o_dev, off), len, cudaMemcpyDeviceToHost, p->out) != cudaSuccess)
            return FATTN_ERR_CUDA;
        if (with_lse &&
            cudaMemcpyAsync(lse_host + h0 * N, lse_dev + h0 * N, static_cast<size_t>((h1 - h0) * N) * sizeof(float),
                            cudaMemcpyDeviceToHost, p->out) != cudaSuccess)
            return FATTN_ERR_CUDA;
    }
    if (cudaEventRecord(p->join, p->out) != cudaSuccess || cudaStreamWaitEvent(stream, p->join, 0) != cudaSuccess)
        return FATTN_ERR_CUDA;
    return FATTN_OK;
}

int64_t fattn_unfused_workspace_bytes(int64_t B, int64_t H, int64_t N) {
    if (B <= 0 || H <= 0 || N <= 0) return 0;
    if (B > (int64_t(1) << 30) || H > (int64_t(1) << 30) || N > (int64_t(1) << 30)) return 0;
    const int64_t BH = B * H;
    const int64_t np = unfused_row_pitch(N);
    // 6 * BH * N * np must stay below 2^62
    if (BH > (int64_t(1) << 30) || static_cast<double>(BH) * N * np * 6.0 > 4.0e18) return 0;
    return static_cast<int64_t>(unfused_workspace_bytes(BH, N));
}

int fattn_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse,
                      void* workspace, int64_t workspace_bytes, int64_t B, int64_t H, int64_t N,
                      int64_t D, float scale, int causal, int dtype, fattn_stream_t stream_h) {
    bool empty = false;
    int st = validate(q, k, v, o, lse, B, H, H, N, D, scale, dtype, &empty);
    if (st != FATTN_OK || empty) return st;
    if (dtype == FATTN_F32) return FATTN_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    if (BH > 65535 || ceil_div(N, 128) > 65535) return FATTN_ERR_UNSUPPORTED;
    const int64_t need = fattn_unfused_workspace_bytes(B, H, N);
    if (need <= 0) return FATTN_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < need) return FATTN_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return FATTN_ERR_MISALIGNED;
    const size_t bytes = static_cast<size_t>(BH * N * D) * 2u;
    const size_t ws = static_cast<size_t>(need);
    if (overlaps(workspace, ws, q, bytes) || overlaps(workspace, ws, k, bytes) ||
        overlaps(workspace, ws, v, bytes) || overlaps(workspace, ws, o, bytes) ||
        (lse && overlaps(workspace, ws, lse, static_cast<size_t>(BH * N) * sizeof(float))))
        return FATTN_ERR_INVALID_ARG;
    int sms = 0;
    st = current_sm_count(&sms);
    if (st != FATTN_OK) return st;
    UnfusedArgs a;
    std::memset(&a, 0, sizeof(a));
    const bool bf16 = dtype == FATTN_BF16;
    TcArgs t;
    std::memset(&t, 0, sizeof(t));
    if (tc_encode_maps(t, q, k, v, BH, BH, N, D, bf16) != cudaSuccess) return FATTN_ERR_CUDA;
    a.tmap_q = t.tmap_q;
    a.tmap_k = t.tmap_k;
    a.tmap_v = t.tmap_v;
    a.s = static_cast<float*>(workspace);
    a.p = static_cast<uint8_t*>(workspace) + static_cast<size_t>(BH * N * unfused_row_pitch(N)) * 4u;
    if (unfused_encode_p_map(a, BH, N, bf16) != cudaSuccess) return FATTN_ERR_CUDA;
    a.o = o;
    a.lse = lse;
    a.N = static_cast<int>(N);
    a.Np = static_cast<int>(unfused_row_pitch(N));
    a.BH = static_cast<int>(BH);
    a.H = static_cast<int>(H);
    a.Hkv = static_cast<int>(H);
    a.scale = scale;
    a.timeout_ns = kDefaultTimeoutNs;
    cudaError_t e = unfused_launch(a, static_cast<int>(D), bf16, causal != 0,
                                   reinterpret_cast<cudaStream_t>(stream_h));
    return e == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

int fattn_fwd_unfused_static(const void* q, const void* k, const void* v, void* o, float* lse,
                             int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal,
                             int dtype, fattn_stream_t stream_h) {
    bool empty = false;
    int st = validate(q, k, v, o, lse, B, H, H, N, D, scale, dtype, &empty);
    if (st != FATTN_OK || empty) return st;
    if (dtype == FATTN_F32) return FATTN_ERR_UNSUPPORTED;
    const int64_t need = fattn_unfused_workspace_bytes(B, H, N);
    if (need <= 0 || need > static_cast<int64_t>(kUnfusedStaticBytes)) return FATTN_ERR_UNSUPPORTED;
    int sms = 0;
    st = current_sm_count(&sms);
    if (st != FATTN_OK) return st;
    void* scratch = nullptr;
    if (unfused_static_scratch(&scratch) != cudaSuccess) return FATTN_ERR_CUDA;
    return fattn_fwd_unfused(q, k, v, o, lse, scratch, static_cast<int64_t>(kUnfusedStaticBytes), B, H,
                             N, D, scale, causal, dtype, stream_h);
}

int64_t fattn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N) {
    if (B <= 0 || H <= 0 || N <= 0) return 0;
    if (B > (int64_t(1) << 30) || H > (int64_t(1) << 30) || N > (int64_t(1) << 30) ||
        B * H > (int64_t(1) << 30))
        return 0;
    return B * H * 2 * bwd_padded_rows(N) * static_cast<int64_t>(sizeof(float));
}

int fattn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
              const float* lse, void* dq, void* dk, void* dv, void* workspace,
              int64_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t D, float scale,
              int causal, int dtype, fattn_stream_t stream_h) {
    return fattn_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, H, N, D,
                         scale, causal, dtype, stream_h);
}

int fattn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, void* workspace,
                  int64_t workspace_bytes, int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                  float scale, int causal, int dtype, fattn_stream_t stream_h) {
    bool empty = false;
    // q, k, v and dq share the forward's rules (dq plays O's part).
    int st = validate(q, k, v, dq, nullptr, B, H, Hkv, N, D, scale, dtype, &empty);
    if (st != FATTN_OK || empty) return st;
    if (dtype == FATTN_F32) return FATTN_ERR_UNSUPPORTED;
    if (!o || !dout || !lse || !dk || !dv || !workspace) return FATTN_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(dout) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return FATTN_ERR_MISALIGNED;
    const int64_t BH = B * H, BHkv = B * Hkv;
    const int64_t need = fattn_bwd_workspace_bytes(B, H, N);
    if (need <= 0) return FATTN_ERR_UNSUPPORTED;
    if (bwd_padded_rows(N) / 128 * BH > 0x7fffffffll) return FATTN_ERR_UNSUPPORTED;
    if (workspace_bytes < need) return FATTN_ERR_INVALID_ARG;
    const size_t bytes = static_cast<size_t>(BH * N * D) * 2u;
    const size_t kvbytes = static_cast<size_t>(BHkv * N * D) * 2u;
    const size_t lb = static_cast<size_t>(BH * N) * sizeof(float);
    const void* ins[6] = {q, k, v, o, dout, lse};
    const size_t in_sz[6] = {bytes, kvbytes, kvbytes, bytes, bytes, lb};
    void* outs[4] = {dq, dk, dv, workspace};
    const size_t out_sz[4] = {bytes, kvbytes, kvbytes, static_cast<size_t>(need)};
    for (int i = 0; i < 4; ++i) {
        for (int j = 0; j < 6; ++j)
            if (overlaps(outs[i], out_sz[i], ins[j], in_sz[j])) return FATTN_ERR_INVALID_ARG;
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(outs[i], out_sz[i], outs[j], out_sz[j])) return FATTN_ERR_INVALID_ARG;
    }
    int sms = 0;
    st = current_sm_count(&sms);
    if (st != FATTN_OK) return st;
    const bool bf16 = dtype == FATTN_BF16;
    BwdArgs a;
    std::memset(&a, 0, sizeof(a));
    TcArgs t;
    std::memset(&t, 0, sizeof(t));
    if (tc_encode_maps(t, q, k, v, BH, BHkv, N, D, bf16) != cudaSuccess) return FATTN_ERR_CUDA;
    a.tmap_q = t.tmap_q;
    a.tmap_k = t.tmap_k;
    a.tmap_v = t.tmap_v;
    if (tc_encode_maps(t, dout, dout, dout, BH, BH, N, D, bf16) != cudaSuccess) return FATTN_ERR_CUDA;
    a.tmap_do = t.tmap_q;
    a.ws = static_cast<float*>(workspace);
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.N = static_cast<int>(N);
    a.Npad = static_cast<int>(bwd_padded_rows(N));
    a.BH = static_cast<int>(BH);
    a.H = static_cast<int>(H);
    a.Hkv = static_cast<int>(Hkv);
    a.BHkv = static_cast<int>(BHkv);
    a.num_tiles = a.Npad / 128;
    a.sl2 = scale * kLog2e;
    a.scale = scale;
    a.timeout_ns = kDefaultTimeoutNs;
    cudaError_t e = bwd_launch(a, o, dout, lse, static_cast<int>(D), bf16, causal != 0,
                               reinterpret_cast<cudaStream_t>(stream_h));
    return e == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

int fattn_bwd_host(const void* q_host, const void* k_host, const void* v_host, const void* o_host,
                   const void* dout_host, const float* lse_host, void* dq_host, void* dk_host,
                   void* dv_host, void* q_dev, void* k_dev, void* v_dev, void* o_dev, void* dout_dev,
                   float* lse_dev, void* dq_dev, void* dk_dev, void* dv_dev, void* workspace,
                   int64_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t D, float scale,
                   int causal, int dtype, fattn_stream_t stream_h) {
    bool empty = false;
    int st = validate(q_dev, k_dev, v_dev, dq_dev, nullptr, B, H, H, N, D, scale, dtype, &empty);
    if (st != FATTN_OK || empty) return st;
    if (!q_host || !k_host || !v_host || !o_host || !dout_host || !lse_host || !dq_host || !dk_host ||
        !dv_host)
        return FATTN_ERR_INVALID_ARG;
    if (dtype == FATTN_F32) return FATTN_ERR_UNSUPPORTED;
    if (!o_dev || !dout_dev || !lse_dev || !dk_dev || !dv_dev || !workspace) return FATTN_ERR_INVALID_ARG;
    const int64_t need = fattn_bwd_workspace_bytes(B, H, N);
    if (need <= 0) return FATTN_ERR_UNSUPPORTED;
    if (workspace_bytes < need) return FATTN_ERR_INVALID_ARG;
    int sms = 0;
    st = current_sm_count(&sms);
    if (st != FATTN_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    std::lock_guard<std::mutex> lock(g_host_mu);
    HostPipe* p = nullptr;
    if (host_pipe(&p) != cudaSuccess) return FATTN_ERR_CUDA;
    // As fattn_fwd_host: groups of heads whose copies overlap the previous
    // group's three kernels.  A group's statistics use its own slice of the
    // workspace ([heads][2][Npad] floats).
    const int64_t BH = B * H;
    const int chunks = static_cast<int>(std::min<int64_t>(kHostChunks, BH));
    const size_t row = static_cast<size_t>(N * D) * 2u;  // one head of a 16-bit tensor
    const int64_t ws_head = need / BH;                   // bytes of workspace per head
    auto bptr = [](const void* base, size_t off) {
        return static_cast<void*>(static_cast<uint8_t*>(const_cast<void*>(base)) + off);
    };
    if (cudaEventRecord(p->fork, stream) != cudaSuccess || cudaStreamWaitEvent(p->in, p->fork, 0) != cudaSuccess)
        return FATTN_ERR_CUDA;
    for (int c = 0; c < chunks; ++c) {
        const int64_t h0 = BH * c / chunks, h1 = BH * (c + 1) / chunks;
        const size_t off = static_cast<size_t>(h0) * row, len = static_cast<size_t>(h1 - h0) * row;
        const size_t loff = static_cast<size_t>(h0 * N) * sizeof(float);
        const size_t llen = static_cast<size_t>((h1 - h0) * N) * sizeof(float);
        const void* hin[5] = {q_host, k_host, v_host, o_host, dout_host};
        void* din[5] = {q_dev, k_dev, v_dev, o_dev, dout_dev};
        for (int t = 0; t < 5; ++t)
            if (cudaMemcpyAsync(bptr(din[t], off), bptr(hin[t], off), len, cudaMemcpyHostToDevice, p->in) !=
                cudaSuccess)
                return FATTN_ERR_CUDA;
        if (cudaMemcpyAsync(bptr(lse_dev, loff), bptr(lse_host, loff), llen, cudaMemcpyHostToDevice, p->in) !=
                cudaSuccess ||
            cudaEventRecord(p->in_done[c], p->in) != cudaSuccess ||
            cudaStreamWaitEvent(stream, p->in_done[c], 0) != cudaSuccess)
            return FATTN_ERR_CUDA;
        st = fattn_bwd(bptr(q_dev, off), bptr(k_dev, off), bptr(v_dev, off), bptr(o_dev, off),
                       bptr(dout_dev, off), reinterpret_cast<const float*>(bptr(lse_dev, loff)),
                       bptr(dq_dev, off), bptr(dk_dev, off), bptr(dv_dev, off),
                       bptr(workspace, static_cast<size_t>(h0 * ws_head)), (h1 - h0) * ws_head, 1, h1 - h0,
                       N, D, scale, causal, dtype, stream_h);
        if (st != FATTN_OK) return st;
        if (cudaEventRecord(p->k_done[c], stream) != cudaSuccess ||
            cudaStreamWaitEvent(p->out, p->k_done[c], 0) != cudaSuccess)
            return FATTN_ERR_CUDA;
        void* hout[3] = {dq_host, dk_host, dv_host};
        void* dout3[3] = {dq_dev, dk_dev, dv_dev};
        for (int t = 0; t < 3; ++t)
            if (cudaMemcpyAsync(bptr(hout[t], off), bptr(dout3[t], off), len, cudaMemcpyDeviceToHost, p->out) !=
                cudaSuccess)
                return FATTN_ERR_CUDA;
    }
    if (cudaEventRecord(p->join, p->out) != cudaSuccess || cudaStreamWaitEvent(stream, p->join, 0) != cudaSuccess)
        return FATTN_ERR_CUDA;
    return FATTN_OK;
}

int fattn_get_device_status(fattn_stream_t stream_h) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FATTN_ERR_CUDA;
    uint32_t word = 0, word_unfused = 0, word_bwd = 0;
    if (read_and_clear_error_word(&word) != cudaSuccess ||
        unfused_read_and_clear_error_word(&word_unfused) != cudaSuccess ||
        bwd_read_and_clear_error_word(&word_bwd) != cudaSuccess)
        return FATTN_ERR_CUDA;
    word |= word_unfused | word_bwd;
    if (word & (1u << FATTN_ERR_INTERNAL)) return FATTN_ERR_INTERNAL;
    if (word & (1u << FATTN_ERR_TIMEOUT)) return FATTN_ERR_TIMEOUT;
    return FATTN_OK;
}

int fattn_selftest_wait_timeout(uint64_t timeout_ns, fattn_stream_t stream_h) {
    if (timeout_ns == 0 || timeout_ns > 1000000000ull) return FATTN_ERR_INVALID_ARG;
    int sms = 0;
    int st = current_sm_count(&sms);
    if (st != FATTN_OK) return st;
    cudaError_t e = launch_wait_selftest(timeout_ns, reinterpret_cast<cudaStream_t>(stream_h));
    return e == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

}  // extern "C"
