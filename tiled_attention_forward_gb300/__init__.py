"""tiled_attention_forward_gb300 -- Python binding of libfattn.

Exact scaled-dot-product attention forward on one GB300 (sm_103a), computed
FlashAttention-2 style by hand-written CUDA kernels behind a C ABI
(``include/fattn.h``).  This module only marshals arguments: it turns torch
tensors into device pointers and the current CUDA stream into a
``cudaStream_t`` and calls the library.  Every step of the computation runs in
the library's kernels; there is no fallback of any kind.  If ``libfattn.so``
has not been built (``python -m tiled_attention_forward_gb300.build``), every
call raises ``FattnLibraryMissing``.

    import torch, tiled_attention_forward_gb300 as fattn
    o, lse = fattn.fwd(q, k, v, causal=True)     # q,k,v: [B,H,N,D] cuda tensors
"""
import ctypes
import math
import os

import torch

__all__ = ["fwd", "fwd_host", "bwd", "bwd_host", "bwd_workspace_bytes", "fwd_unfused", "fwd_unfused_static", "unfused_workspace_bytes",
           "UNFUSED_STATIC_BYTES", "plan", "get_device_status", "selftest_wait_timeout",
           "status_string", "library_path", "load", "FattnError", "FattnLibraryMissing",
           "DTYPE_CODES", "STATUS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfattn.so")

DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
STATUS = {0: "FATTN_OK", 1: "FATTN_ERR_INVALID_ARG", 2: "FATTN_ERR_UNSUPPORTED",
          3: "FATTN_ERR_MISALIGNED", 4: "FATTN_ERR_CUDA", 5: "FATTN_ERR_TIMEOUT",
          6: "FATTN_ERR_NO_DEVICE", 7: "FATTN_ERR_INTERNAL"}
UNFUSED_STATIC_BYTES = 64 << 20  # FATTN_UNFUSED_STATIC_BYTES
PLAN_FIELDS = ("path", "grid_x", "grid_y", "threads", "smem_bytes", "tasks", "kv_tiles",
               "rows_per_task", "keys_per_kv_tile")


class FattnError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s returned %s (%d)" % (where, STATUS.get(code, "?"), code))


class FattnLibraryMissing(RuntimeError):
    pass


_lib = None


def library_path():
    return _LIB_PATH


def load():
    """Load libfattn.so (once).  Raises FattnLibraryMissing if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise FattnLibraryMissing(
            "libfattn.so is not built at %s; run `python -m tiled_attention_forward_gb300.build`"
            % _LIB_PATH)
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, f32, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    lib.fattn_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, ci, ci, vp]
    lib.fattn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, ci, ci, vp]
    lib.fattn_fwd_f32_rowwise.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, ci, vp]
    lib.fattn_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                   i64, i64, i64, i64, f32, ci, ci, vp]
    lib.fattn_fwd_unfused.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, ci,
                                      ci, vp]
    lib.fattn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, f32,
                              ci, ci, vp]
    lib.fattn_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                  i64, f32, ci, ci, vp]
    lib.fattn_bwd_host.argtypes = [vp] * 19 + [i64, i64, i64, i64, i64, f32, ci, ci, vp]
    lib.fattn_bwd_workspace_bytes.argtypes = [i64, i64, i64]
    lib.fattn_bwd_workspace_bytes.restype = i64
    lib.fattn_fwd_unfused_static.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, ci, ci, vp]
    lib.fattn_unfused_workspace_bytes.argtypes = [i64, i64, i64]
    lib.fattn_unfused_workspace_bytes.restype = i64
    lib.fattn_plan.argtypes = [i64, i64, i64, i64, ci, ci, ci, ctypes.POINTER(i64)]
    lib.fattn_plan_head_group.argtypes = [i64, i64, i64, i64, i64, ctypes.POINTER(i64)]
    lib.fattn_get_device_status.argtypes = [vp]
    lib.fattn_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.fattn_status_string.argtypes = [ci]
    lib.fattn_status_string.restype = ctypes.c_char_p
    lib.fattn_version.argtypes = []
    for f in ("fattn_fwd", "fattn_fwd_gqa", "fattn_fwd_host", "fattn_fwd_unfused", "fattn_bwd", "fattn_bwd_gqa", "fattn_bwd_host",
              "fattn_fwd_unfused_static", "fattn_plan", "fattn_plan_head_group",
              "fattn_get_device_status",
              "fattn_selftest_wait_timeout", "fattn_version"):
        getattr(lib, f).restype = ci
    _lib = lib
    return lib


def status_string(code):
    return load().fattn_status_string(int(code)).decode()


def _check(code, where):
    if code != 0:
        raise FattnError(code, where)


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _default_scale(D):
    # 1/sqrt(D) rounded once to fp32, the value the library multiplies by.
    return float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32).item())


def _check_qkv(q, k, v, allow_gqa=False):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    if v.shape != k.shape:
        raise ValueError("k and v must have the same shape")
    if allow_gqa:
        B, H, N, D = q.shape
        if k.shape[0] != B or k.shape[2] != N or k.shape[3] != D:
            raise ValueError("k, v must be [B, Hkv, N, D] with q's B, N and D")
    elif k.shape != q.shape:
        raise ValueError("q, k, v must have the same shape")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must have the same dtype")
    if q.dtype not in DTYPE_CODES:
        raise ValueError("dtype must be float32, float16 or bfloat16")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous row-major [B, H, N, D]")


def fwd(q, k, v, causal=False, scale=None, out=None, lse=None, return_lse=True, stream=None):
    """Attention forward on CUDA tensors.

    q: [B, H, N, D]; k, v: [B, Hkv, N, D] with H a multiple of Hkv
    (grouped-query attention when Hkv < H); contiguous CUDA tensors of one
    dtype (float32, float16 or bfloat16), D in {64, 128}.  Returns (o, lse): o has q's dtype
    and shape; lse is float32 [B, H, N] (natural-log log-sum-exp of the
    scaled scores), or None when return_lse is False.  ``out`` / ``lse`` may
    be given to write into existing tensors.  Enqueued on ``stream`` (default:
    torch's current stream); no synchronisation.
    """
    _check_qkv(q, k, v, allow_gqa=True)
    if not q.is_cuda:
        raise ValueError("fwd needs CUDA tensors; see fwd_host for host buffers")
    B, H, N, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = _default_scale(D)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    lse_ptr = lse.data_ptr() if (return_lse and lse is not None) else None
    lib = load()
    with torch.cuda.device(q.device):
        if Hkv == H:
            rc = lib.fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                               B, H, N, D, float(scale), int(bool(causal)), DTYPE_CODES[q.dtype],
                               _stream_handle(stream))
        else:
            rc = lib.fattn_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   lse_ptr, B, H, Hkv, N, D, float(scale), int(bool(causal)),
                                   DTYPE_CODES[q.dtype], _stream_handle(stream))
    _check(rc, "fattn_fwd" if Hkv == H else "fattn_fwd_gqa")
    return out, (lse if return_lse else None)


def fwd_f32_rowwise(q, k, v, causal=False, scale=None, out=None, lse=None, return_lse=True,
                    stream=None):
    """fp32 forward through the one-query-row-per-thread CUDA-core kernel
    (fattn_fwd_f32_rowwise).  q, k, v: contiguous float32 CUDA tensors of one
    shape [B, H, N, D]; otherwise as fwd."""
    _check_qkv(q, k, v)
    if not q.is_cuda or q.dtype != torch.float32:
        raise ValueError("fwd_f32_rowwise needs float32 CUDA tensors")
    B, H, N, D = q.shape
    if scale is None:
        scale = _default_scale(D)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    lse_ptr = lse.data_ptr() if (return_lse and lse is not None) else None
    lib = load()
    with torch.cuda.device(q.device):
        rc = lib.fattn_fwd_f32_rowwise(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       lse_ptr, B, H, N, D, float(scale), int(bool(causal)),
                                       _stream_handle(stream))
    _check(rc, "fattn_fwd_f32_rowwise")
    return out, (lse if return_lse else None)


def fwd_host(q_host, k_host, v_host, q_dev, k_dev, v_dev, o_dev, o_host, lse_dev=None,
             lse_host=None, causal=False, scale=None, stream=None):
    """End-to-end forward from host tensors: host->device copies, the kernels and
    the device->host copies of O (and LSE) are enqueued by the library, in up
    to four groups of heads so that copies overlap the kernels (two internal
    copy streams, joined to ``stream`` with events).  Host tensors should be
    pinned; the caller synchronises ``stream``."""
    _check_qkv(q_host, k_host, v_host)
    B, H, N, D = q_host.shape
    if scale is None:
        scale = _default_scale(D)
    lib = load()
    with torch.cuda.device(q_dev.device):
        rc = lib.fattn_fwd_host(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(),
                                o_host.data_ptr(),
                                lse_host.data_ptr() if lse_host is not None else None,
                                q_dev.data_ptr(), k_dev.data_ptr(), v_dev.data_ptr(),
                                o_dev.data_ptr(),
                                lse_dev.data_ptr() if lse_dev is not None else None,
                                B, H, N, D, float(scale), int(bool(causal)),
                                DTYPE_CODES[q_host.dtype], _stream_handle(stream))
    _check(rc, "fattn_fwd_host")


def bwd_workspace_bytes(B, H, N):
    """Bytes of workspace bwd needs (fp32 per-row statistics, rows padded to 128)."""
    return int(load().fattn_bwd_workspace_bytes(int(B), int(H), int(N)))


def bwd(q, k, v, o, lse, dout, causal=False, scale=None, dq=None, dk=None, dv=None,
        workspace=None, stream=None):
    """Attention backward on CUDA tensors: gradients of sum(dout * O) where
    (o, lse) is what ``fwd`` returned for (q, k, v).  bfloat16 / float16;
    q, o, dout [B, H, N, D]; k, v [B, Hkv, N, D] with H a multiple of Hkv
    (grouped-query attention when Hkv < H: dk, dv are summed over each
    group); lse float32 [B, H, N].  Returns (dq, dk, dv) in the input dtype
    with q's and k's shapes.  ``workspace`` (a CUDA uint8 tensor of at least
    ``bwd_workspace_bytes(B, H, N)`` bytes) is allocated here when None."""
    _check_qkv(q, k, v, allow_gqa=True)
    for t in (o, dout):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("o and dout must be contiguous with q's shape and dtype")
    if lse.dtype != torch.float32 or tuple(lse.shape) != tuple(q.shape[:3]) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B, H, N]")
    if not q.is_cuda:
        raise ValueError("bwd needs CUDA tensors")
    B, H, N, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = _default_scale(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(max(bwd_workspace_bytes(B, H, N), 16), dtype=torch.uint8,
                                device=q.device)
    lib = load()
    with torch.cuda.device(q.device):
        rc = lib.fattn_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), B, H, Hkv, N, D,
                               float(scale), int(bool(causal)), DTYPE_CODES[q.dtype],
                               _stream_handle(stream))
    _check(rc, "fattn_bwd_gqa")
    return dq, dk, dv


def bwd_host(hosts, devs, grads_host, grads_dev, workspace, causal=False, scale=None, stream=None):
    """End-to-end backward from host tensors (multi-head, bfloat16 / float16).

    hosts = (q, k, v, o, dout, lse) pinned host tensors; devs = the matching
    device buffers; grads_host / grads_dev = (dq, dk, dv) host / device
    buffers; workspace as for ``bwd``.  Copies in, the backward and copies
    out are enqueued by the library in groups of heads that overlap; the
    caller synchronises ``stream``."""
    q = hosts[0]
    B, H, N, D = q.shape
    if scale is None:
        scale = _default_scale(D)
    ptrs = [t.data_ptr() for t in hosts] + [t.data_ptr() for t in grads_host] + \
        [t.data_ptr() for t in devs] + [t.data_ptr() for t in grads_dev] + [workspace.data_ptr()]
    lib = load()
    with torch.cuda.device(devs[0].device):
        rc = lib.fattn_bwd_host(*ptrs, workspace.numel() * workspace.element_size(), B, H, N, D,
                                float(scale), int(bool(causal)), DTYPE_CODES[q.dtype],
                                _stream_handle(stream))
    _check(rc, "fattn_bwd_host")


def unfused_workspace_bytes(B, H, N):
    """Bytes of workspace fwd_unfused needs (S fp32 then P 16-bit, rows padded to 8)."""
    return int(load().fattn_unfused_workspace_bytes(int(B), int(H), int(N)))


def fwd_unfused(q, k, v, causal=False, scale=None, out=None, lse=None, workspace=None,
                return_lse=True, stream=None):
    """The materialising comparator: S = scale Q K^T and P = softmax(S) are
    written to ``workspace`` (a CUDA uint8 tensor of at least
    ``unfused_workspace_bytes(B, H, N)`` bytes; allocated here when None) and
    O = P V is computed from P.  bfloat16 / float16 only, q, k, v of one shape.
    Returns (o, lse) like ``fwd``."""
    _check_qkv(q, k, v)
    if not q.is_cuda:
        raise ValueError("fwd_unfused needs CUDA tensors")
    B, H, N, D = q.shape
    if scale is None:
        scale = _default_scale(D)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = unfused_workspace_bytes(B, H, N)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    lse_ptr = lse.data_ptr() if (return_lse and lse is not None) else None
    lib = load()
    with torch.cuda.device(q.device):
        rc = lib.fattn_fwd_unfused(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   lse_ptr, workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), B, H, N, D,
                                   float(scale), int(bool(causal)), DTYPE_CODES[q.dtype],
                                   _stream_handle(stream))
    _check(rc, "fattn_fwd_unfused")
    return out, (lse if return_lse else None)


def fwd_unfused_static(q, k, v, causal=False, scale=None, out=None, lse=None, return_lse=True,
                       stream=None):
    """``fwd_unfused`` with the library's fixed per-device workspace of
    UNFUSED_STATIC_BYTES (no workspace argument, nothing allocated by the
    library).  Calls on one device must not overlap in time (one stream)."""
    _check_qkv(q, k, v)
    if not q.is_cuda:
        raise ValueError("fwd_unfused_static needs CUDA tensors")
    B, H, N, D = q.shape
    if scale is None:
        scale = _default_scale(D)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    lse_ptr = lse.data_ptr() if (return_lse and lse is not None) else None
    lib = load()
    with torch.cuda.device(q.device):
        rc = lib.fattn_fwd_unfused_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                          lse_ptr, B, H, N, D, float(scale), int(bool(causal)),
                                          DTYPE_CODES[q.dtype], _stream_handle(stream))
    _check(rc, "fattn_fwd_unfused_static")
    return out, (lse if return_lse else None)


def plan(B, H, N, D, causal=False, dtype=torch.bfloat16, num_sms=0):
    """Launch plan (host only when num_sms > 0) as a dict; see fattn_plan."""
    out = (ctypes.c_int64 * 9)()
    code = DTYPE_CODES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    rc = load().fattn_plan(B, H, N, D, int(bool(causal)), code, int(num_sms), out)
    _check(rc, "fattn_plan")
    return dict(zip(PLAN_FIELDS, list(out)))


def plan_head_group(B, H, N, D, Hkv=None):
    """Query heads per group of the causal task order (host only); see
    fattn_plan_head_group."""
    out = ctypes.c_int64(0)
    rc = load().fattn_plan_head_group(B, H, H if Hkv is None else Hkv, N, D, ctypes.byref(out))
    _check(rc, "fattn_plan_head_group")
    return out.value


def get_device_status(stream=None):
    """Synchronise the stream and return (and clear) the device error word."""
    return load().fattn_get_device_status(_stream_handle(stream))


def selftest_wait_timeout(timeout_ns, stream=None):
    rc = load().fattn_selftest_wait_timeout(int(timeout_ns), _stream_handle(stream))
    _check(rc, "fattn_selftest_wait_timeout")
