/*
 * fattn.h -- C ABI of libfattn: exact scaled-dot-product attention forward on
 * one NVIDIA GB300 (sm_103a), computed FlashAttention-2 style.
 *
 * Operation (the plain definition; cishoon.github.io "flashattention" page,
 * §1.1.2 "Attention公式拆解"):
 *
 *     O = softmax(scale * Q K^T  [+ causal mask]) V
 *     LSE[i] = ln sum_{j visible to i} exp(scale * q_i . k_j)
 *
 * computed without materialising S or P: Q tiles in the outer loop, K/V tiles
 * streamed in the inner loop, running row max m and row sum l (online
 * softmax), one 1/l normalisation at the end, and, under causal masking,
 * K/V tiles wholly above the diagonal skipped and the element mask applied
 * only on tiles that cross it (dandandamowang.xyz "Flash Attention (二) v2"
 * page, §1.1-§1.4 and §3.4; online-softmax recurrence: chang-wenbin.github.io
 * FA2 report, §2).  Causal masking is top-left aligned: key j is visible to
 * query row i iff j <= i.
 *
 * Data layout: every tensor is dense row-major [B, H, N, D] with no padding;
 * element (b,h,i,d) sits at ((b*H + h)*N + i)*D + d.  LSE is fp32 [B, H, N].
 * Q, K, V and O share one dtype; the output O has the input dtype.
 *
 * Paths: FATTN_BF16 / FATTN_F16 run the tensor-core kernel (TMA, tcgen05 MMA
 * with TMEM accumulators, fp32 accumulation and softmax, P rounded to the
 * input dtype for the P.V product).  FATTN_F32 runs a CUDA-core FFMA kernel
 * (register micro-tiles of 8 query rows per thread, fp32 throughout;
 * fattn_fwd_f32_rowwise runs the one-row-per-thread form).  Supported head
 * dims: 64, 128.
 *
 * Ownership: the caller owns every buffer.  No entry point allocates device
 * or pinned host memory, and nothing is retained after a call returns except
 * a per-device error word (see fattn_get_device_status).
 *
 * Streams: compute entry points are asynchronous on `stream` (a cudaStream_t;
 * NULL is the legacy default stream).  Argument errors are reported before
 * anything is enqueued.  An error detected inside a kernel (a bounded wait
 * that gave up) is recorded in the device error word and surfaces through
 * fattn_get_device_status.
 */
#ifndef FATTN_H
#define FATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the shared library are exported explicitly (it is built with
 * hidden default visibility). */
#if defined(__GNUC__)
#define FATTN_API __attribute__((visibility("default")))
#else
#define FATTN_API
#endif

/* A cudaStream_t (the same opaque handle type), without requiring CUDA headers. */
typedef struct CUstream_st* fattn_stream_t;

typedef enum {
    FATTN_F32 = 0,
    FATTN_F16 = 1,
    FATTN_BF16 = 2
} fattn_dtype;

typedef enum {
    FATTN_OK = 0,
    FATTN_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad dtype, non-finite or negative scale, overlapping O */
    FATTN_ERR_UNSUPPORTED = 2,   /* D not in {64, 128}; N or B*H above 2^30, or B*H*N*D above 2^52 */
    FATTN_ERR_MISALIGNED = 3,    /* a tensor pointer not 16-byte aligned (TMA / vector access requirement) */
    FATTN_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (launch, copy, tensor-map encode) */
    FATTN_ERR_TIMEOUT = 5,       /* a kernel's bounded wait expired (reported by fattn_get_device_status) */
    FATTN_ERR_NO_DEVICE = 6,     /* no usable sm_103 device is current */
    FATTN_ERR_INTERNAL = 7       /* a kernel found a broken launch invariant and did no work
                                    (reported by fattn_get_device_status) */
} fattn_status;

/*
 * fattn_fwd -- attention forward on device buffers.
 *
 *   q, k, v : device pointers, [B,H,N,D] of `dtype`, read only, 16-byte aligned.
 *   o       : device pointer, [B,H,N,D] of `dtype`, written; must not overlap q/k/v.
 *   lse     : device pointer to fp32 [B,H,N], written; may be NULL (not written).
 *   B,H,N,D : sizes; B,H,N >= 0 and D in {64, 128}.  B*H*N == 0 returns FATTN_OK
 *             with nothing enqueued.
 *   scale   : multiplier of q.k (typically 1/sqrt(D)); finite and >= 0.
 *   causal  : 0 = every key visible; nonzero = key j visible to row i iff j <= i.
 *   dtype   : a fattn_dtype.
 *   stream  : CUDA stream the single kernel launch is enqueued on.
 *
 * Returns FATTN_OK once the kernel is enqueued, or an error code (nothing
 * enqueued on argument errors).  Exactly one kernel is launched per call.
 */
FATTN_API int fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
              int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal,
              int dtype, fattn_stream_t stream);

/*
 * fattn_fwd_gqa -- grouped-query / multi-query attention forward.
 *
 * As fattn_fwd, except that k and v are [B, Hkv, N, D] with H a multiple of
 * Hkv, and query head h of batch b attends to key/value head
 * b*Hkv + h / (H/Hkv): consecutive groups of H/Hkv query heads share one
 * K/V head (Hkv == H is fattn_fwd; Hkv == 1 is multi-query attention).
 * Compatibility of the tiled method with GQA: the GQA reference (Ainslie et
 * al.) cited by the chang-wenbin.github.io FA2 report; the head mapping is the
 * usual consecutive grouping.  Hkv <= 0 or H % Hkv != 0 -> FATTN_ERR_INVALID_ARG.
 * o and lse keep the query shapes [B,H,N,D] and [B,H,N].
 */
FATTN_API int fattn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                  int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D, float scale,
                  int causal, int dtype, fattn_stream_t stream);

/*
 * fattn_fwd_f32_rowwise -- the fp32 forward in the CUDA-core layout of the
 * dandandamowang.xyz "Flash Attention (二) v2" page (§1.1, §3.2-§3.5): one
 * query row per thread, Br = 128 threads per CTA, Bc = 32 keys per K/V tile
 * at D = 64 (16 at D = 128), double-buffered cp.async K/V, padded shared
 * memory, grid (ceil(N/128), B*H).  Same arguments, results (to fp32
 * rounding), validation and error behaviour as fattn_fwd with dtype ==
 * FATTN_F32; one kernel launch per call.  fattn_fwd's own fp32 kernel
 * spreads each CTA's 128 rows over 256 threads as register micro-tiles and
 * is faster on this part; this entry point keeps the page's layout
 * available and measurable.
 */
FATTN_API int fattn_fwd_f32_rowwise(const float* q, const float* k, const float* v, float* o,
                          float* lse, int64_t B, int64_t H, int64_t N, int64_t D, float scale,
                          int causal, fattn_stream_t stream);

/*
 * fattn_fwd_host -- the same forward for callers holding the tensors in host
 * memory: the host->device copies of q, k, v into the caller's device buffers
 * q_dev, k_dev, v_dev, the forward kernel writing o_dev / lse_dev, and the
 * device->host copies of O (and LSE when both lse_host and lse_dev are
 * non-NULL) into o_host / lse_host.  For bf16 / fp16 the heads are split into
 * up to four groups so that the copies of one group overlap the kernel of
 * the previous one (fp32: one group).  Host->device copies run on an
 * internal copy-in stream, the kernels on `stream`, device->host copies on an
 * internal copy-out stream, chained with events; the work starts after
 * everything already enqueued on `stream`, and everything enqueued on
 * `stream` afterwards waits for all of it, so the caller synchronises
 * `stream` before reading o_host.  The first call on a device creates the two
 * streams and ten events (kept for the process lifetime; no memory is
 * allocated); enqueueing is serialised by a host mutex.  Host buffers should
 * be page-locked for the copies to overlap.  Argument rules are those of
 * fattn_fwd, applied to the device buffers; host pointers must be non-NULL.
 */
FATTN_API int fattn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                   void* o_host, float* lse_host,
                   void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev,
                   int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal,
                   int dtype, fattn_stream_t stream);

/*
 * fattn_bwd_workspace_bytes -- bytes of device workspace fattn_bwd needs:
 * fp32 [B*H][2][Npad] (per row -LSE*log2(e) and -Delta, Delta = dO.O,
 * Npad = N rounded up to 128), i.e. 8 * B*H*Npad.  0 for an empty or
 * invalid size.
 */
FATTN_API int64_t fattn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N);

/*
 * fattn_bwd -- attention backward: the gradients dQ, dK, dV of
 * L = sum(dO * O) for O = softmax(scale * Q K^T [+ causal mask]) V, given the
 * forward's output O and log-sum-exp LSE (as fattn_fwd writes them) and the
 * upstream gradient dO.  The FA2 report of chang-wenbin.github.io (section
 * "反向传播性能分析") sketches this pass: the forward's tiling, scores
 * recomputed rather than stored.  Per visible pair: P_ij = exp(s_ij - LSE_i),
 * dP_ij = dO_i.v_j, dS_ij = P_ij (dP_ij - Delta_i) with Delta_i = dO_i.O_i;
 * dV_j = sum_i P_ij dO_i, dK_j = scale sum_i dS_ij q_i, dQ_i = scale sum_j
 * dS_ij k_j.  P and dS are rounded to the input dtype before the products
 * that consume them; every sum accumulates in fp32.
 *
 *   q, k, v, o, dout : device, [B,H,N,D] of `dtype`, read only, 16-byte aligned.
 *   lse              : device, fp32 [B,H,N] (natural log), read only.
 *   dq, dk, dv       : device, [B,H,N,D] of `dtype`, written; 16-byte aligned;
 *                      overlapping no input and no other output.
 *   workspace        : caller-owned device scratch of at least
 *                      fattn_bwd_workspace_bytes(B, H, N) bytes, 16-byte
 *                      aligned, overlapping nothing else; contents ignored.
 *   dtype            : FATTN_BF16 or FATTN_F16 (FATTN_F32 -> FATTN_ERR_UNSUPPORTED).
 *   B,H,N,D,scale,causal : as fattn_fwd (multi-head: k and v have q's shape;
 *                      fattn_bwd_gqa below takes shared K/V heads).
 *
 * Three kernel launches on `stream` (row statistics, dK/dV, dQ); each
 * gradient row is produced by exactly one CTA, so the result is
 * deterministic.  Errors as fattn_fwd.
 */
FATTN_API int fattn_bwd(const void* q, const void* k, const void* v, const void* o,
              const void* dout, const float* lse, void* dq, void* dk, void* dv,
              void* workspace, int64_t workspace_bytes, int64_t B, int64_t H, int64_t N,
              int64_t D, float scale, int causal, int dtype, fattn_stream_t stream);

/*
 * fattn_bwd_gqa -- the backward of grouped-query / multi-query attention
 * (the forward is fattn_fwd_gqa): k, v, dk and dv are [B, Hkv, N, D] with H a
 * multiple of Hkv, query head h of batch b reads key/value head
 * b*Hkv + h/(H/Hkv), and the dK and dV rows of a shared head are the sums of
 * the gradients of the H/Hkv query heads that read it (the chain rule through
 * the shared rows).  q, o, dout, dq are [B, H, N, D], lse [B, H, N]; the
 * workspace is sized by fattn_bwd_workspace_bytes(B, H, N).  Each dK/dV
 * row is still produced by one CTA, which loops over the group's query
 * heads: no atomics, deterministic.  Hkv == H is fattn_bwd.  Other rules
 * and errors as fattn_bwd.
 */
FATTN_API int fattn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv,
                  void* workspace, int64_t workspace_bytes, int64_t B, int64_t H, int64_t Hkv,
                  int64_t N, int64_t D, float scale, int causal, int dtype,
                  fattn_stream_t stream);

/*
 * fattn_bwd_host -- the backward for callers holding the tensors in host
 * memory (multi-head, bf16 / fp16): host->device copies of q, k, v, o, dout
 * and lse into the caller's device buffers, the backward writing dq_dev,
 * dk_dev, dv_dev (with the caller's workspace, sized by
 * fattn_bwd_workspace_bytes), and device->host copies of the three
 * gradients, in up to four groups of heads whose copies overlap the previous
 * group's kernels, on the internal copy streams of fattn_fwd_host (same
 * ordering against `stream`, same first-call and mutex rules).  Argument
 * rules are those of fattn_bwd, applied to the device buffers; host pointers
 * must be non-NULL.
 */
FATTN_API int fattn_bwd_host(const void* q_host, const void* k_host, const void* v_host,
                   const void* o_host, const void* dout_host, const float* lse_host,
                   void* dq_host, void* dk_host, void* dv_host,
                   void* q_dev, void* k_dev, void* v_dev, void* o_dev, void* dout_dev,
                   float* lse_dev, void* dq_dev, void* dk_dev, void* dv_dev,
                   void* workspace, int64_t workspace_bytes,
                   int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal,
                   int dtype, fattn_stream_t stream);

/*
 * fattn_unfused_workspace_bytes -- bytes of device workspace fattn_fwd_unfused
 * needs for B*H heads of length N: S fp32 [B*H][N][Np] followed by P 16-bit
 * [B*H][N][Np], Np = N rounded up to a multiple of 8, i.e. 6 * B*H*N*Np.
 * Returns 0 for an empty or invalid (negative, overflowing) size.
 */
FATTN_API int64_t fattn_unfused_workspace_bytes(int64_t B, int64_t H, int64_t N);

/*
 * fattn_fwd_unfused -- the same O and LSE computed the materialising way, as
 * the comparator for the fused kernel's HBM traffic: three kernels, (1) S =
 * scale Q K^T written to the workspace in fp32 (tcgen05, 128x128 tiles; under
 * causal masking tiles wholly above the diagonal are skipped), (2) a row
 * softmax reading S and writing P in the input dtype and the LSE, (3) O = P V
 * (tcgen05) reading P back.  The three steps are the ScaledDotProduct ->
 * Softmax -> PVMultiply pipeline of the cishoon.github.io "flashattention"
 * page (§2), whose HBM traffic the chang-wenbin.github.io FA2 report (§3)
 * contrasts with the fused form.
 *
 *   q,k,v,o,lse,B,H,N,D,scale,causal : as fattn_fwd.
 *   dtype     : FATTN_BF16 or FATTN_F16 (FATTN_F32 -> FATTN_ERR_UNSUPPORTED).
 *   workspace : caller-owned device buffer of at least
 *               fattn_unfused_workspace_bytes(B, H, N) bytes, 16-byte aligned,
 *               overlapping none of q, k, v, o, lse; its contents on entry are
 *               ignored and on return are the S and P matrices (layout above;
 *               S entries of skipped tiles and P entries past the last tile a
 *               row's Q tile reads are left untouched).
 *   workspace_bytes : its size; smaller than needed -> FATTN_ERR_INVALID_ARG.
 *
 * B*H and ceil(N/128) must each be <= 65535 (grid limits), else
 * FATTN_ERR_UNSUPPORTED.  Three kernel launches per call on `stream`; no
 * allocation.  Errors as fattn_fwd.
 */
FATTN_API int fattn_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse,
                      void* workspace, int64_t workspace_bytes, int64_t B, int64_t H,
                      int64_t N, int64_t D, float scale, int causal, int dtype,
                      fattn_stream_t stream);

/*
 * fattn_fwd_unfused_static -- fattn_fwd_unfused with the workspace taken from
 * a fixed array of FATTN_UNFUSED_STATIC_BYTES in the library's own static
 * device memory (one per device) instead of from the caller, so that neither
 * the caller nor the library allocates anything for the call.  The pages have
 * no counterpart: it is an interface convenience around the same three
 * kernels, which give bit-identical O, LSE, S and P.
 *
 *   Arguments and errors as fattn_fwd_unfused without workspace /
 *   workspace_bytes.  A problem whose fattn_unfused_workspace_bytes(B, H, N)
 *   exceeds FATTN_UNFUSED_STATIC_BYTES -> FATTN_ERR_UNSUPPORTED, before any
 *   CUDA call.  Nothing in the array needs to start at zero: every element a
 *   call reads is written earlier in the same call.
 *
 * Races: the array is shared by every call on a device.  Calls on one device
 * must not overlap in time: enqueue them on one stream, or order them (events,
 * synchronisation).  Overlapping calls race on S and P and leave O undefined.
 * The first call on each device looks up the array's address
 * (cudaGetSymbolAddress, under a host mutex) and sets the kernels' shared
 * memory attributes; make that first call before any stream capture starts.
 */
#define FATTN_UNFUSED_STATIC_BYTES (64ll << 20)
FATTN_API int fattn_fwd_unfused_static(const void* q, const void* k, const void* v, void* o,
                             float* lse, int64_t B, int64_t H, int64_t N, int64_t D,
                             float scale, int causal, int dtype, fattn_stream_t stream);

/*
 * fattn_plan -- host-only description of the launch fattn_fwd would make for
 * these arguments (no CUDA call when num_sms > 0).  Fills `out` with:
 *   out[0] path       : 0 = none (empty problem), 1 = FFMA fp32, 2 = tcgen05 bf16/fp16
 *   out[1] grid_x     : CTAs launched (x)
 *   out[2] grid_y     : CTAs launched (y)
 *   out[3] threads    : threads per CTA
 *   out[4] smem_bytes : dynamic shared memory per CTA
 *   out[5] tasks      : work units (one Q tile of one head; BM = 256 rows on
 *                       the tcgen05 path, Br = 128 rows on the FFMA path)
 *   out[6] kv_tiles   : K/V tiles visited over all tasks (causal skip applied)
 *   out[7] rows_per_task, out[8] keys_per_kv_tile
 * num_sms <= 0 queries the current device.  Returns a fattn_status.
 */
FATTN_API int fattn_plan(int64_t B, int64_t H, int64_t N, int64_t D, int causal, int dtype,
               int num_sms, int64_t out[9]);

/*
 * fattn_plan_head_group -- host only, no CUDA call: the number of query heads
 * per group in fattn_fwd / fattn_fwd_gqa's causal task order.  The tensor-core
 * kernel runs the causal tasks (256-row Q blocks) head group by head group,
 * longest Q blocks first within a group, so that a group's K/V stays in L2;
 * a group is made of whole K/V heads (H / Hkv query heads share one), holds
 * about 48 MB of 16-bit K/V unless one K/V head is larger, and the groups are
 * as equal as the head count allows.  Writes the group size (1 .. B*H) to
 * *head_group.  Returns FATTN_ERR_INVALID_ARG for a null pointer, sizes < 1,
 * D not in {64, 128} or H not a multiple of Hkv, FATTN_ERR_UNSUPPORTED past
 * the kernels' index range, else FATTN_OK.
 */
FATTN_API int fattn_plan_head_group(int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                                    int64_t* head_group);

/*
 * fattn_get_device_status -- synchronises `stream`, then reads and clears the
 * current device's error word.  Returns FATTN_OK, FATTN_ERR_TIMEOUT if a
 * kernel gave up a bounded wait since the last call, FATTN_ERR_INTERNAL if a
 * kernel found a broken launch invariant (e.g. shared-memory alignment) and
 * returned without computing, or FATTN_ERR_CUDA if the synchronisation itself
 * failed.
 */
FATTN_API int fattn_get_device_status(fattn_stream_t stream);

/*
 * fattn_selftest_wait_timeout -- launches one tiny kernel whose single thread
 * waits, with the same bounded wait the forward kernels use, on a shared
 * memory barrier that nothing ever completes; after `timeout_ns` it records
 * FATTN_ERR_TIMEOUT in the device error word and returns.  Exists so the
 * timeout path can be exercised without hanging or faulting a GPU.
 * timeout_ns must be in (0, 10^9].  Asynchronous on `stream`.
 */
FATTN_API int fattn_selftest_wait_timeout(uint64_t timeout_ns, fattn_stream_t stream);

/* Human-readable name of a fattn_status (static string, never NULL). */
FATTN_API const char* fattn_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
FATTN_API int fattn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FATTN_H */
