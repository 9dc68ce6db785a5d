"""fp64 CPU oracle for exact scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this
package.  The product path (the CUDA library and its Python binding) never
imports, links or calls it, and it shares no code with that path.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64); this module only
marshals numpy float64 arrays through ctypes.  See ``attn_oracle.h`` for the
definition each entry point follows and the passages it cites.
"""
import ctypes

import numpy as np

from . import build as _build


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check4(q, k, v):
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B,H,N,D] shape")
    return q.shape


class OracleLib:
    """ctypes view of one compiled copy of attn_oracle.c."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.attn_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                        ctypes.c_double, ci, ci]
        lib.attn_oracle_rows.argtypes = [dp, dp, dp, i64, i64, i64, i64,
                                         ctypes.c_double, ci, i64p, i64p, i64, dp, dp, ci]
        lib.attn_oracle_probs.argtypes = [dp, dp, i64, i64, i64, i64, i64,
                                          ctypes.c_double, ci, dp]
        lib.attn_oracle_online_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                               ctypes.c_double, ci, i64, i64, ci]
        lib.attn_oracle_fwd_gqa.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, i64,
                                            ctypes.c_double, ci, ci]
        lib.attn_oracle_rows_gqa.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64,
                                             ctypes.c_double, ci, i64p, i64p, i64, dp, dp, ci]
        lib.attn_oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                        ctypes.c_double, ci, ci]
        lib.attn_oracle_bwd_gqa.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, i64,
                                            ctypes.c_double, ci, ci]
        lib.attn_oracle_bwd_stats.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64,
                                              ctypes.c_double, ci, i64p, i64, dp, dp, ci]
        lib.attn_oracle_bwd_dq_rows.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64,
                                                ctypes.c_double, ci, i64p, i64, dp, dp,
                                                i64p, i64p, i64, dp, ci]
        lib.attn_oracle_bwd_dkdv_rows.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64,
                                                  ctypes.c_double, ci, i64p, i64, dp, dp,
                                                  i64p, i64p, i64, dp, dp, ci]
        lib.attn_oracle_default_threads.argtypes = []
        for f in ("attn_oracle_fwd", "attn_oracle_rows", "attn_oracle_probs",
                  "attn_oracle_online_fwd", "attn_oracle_fwd_gqa", "attn_oracle_rows_gqa",
                  "attn_oracle_bwd", "attn_oracle_bwd_gqa", "attn_oracle_bwd_stats", "attn_oracle_bwd_dq_rows",
                  "attn_oracle_bwd_dkdv_rows", "attn_oracle_default_threads"):
            getattr(lib, f).restype = ci
        self._lib = lib
        self.path = path

    def default_threads(self) -> int:
        return self._lib.attn_oracle_default_threads()

    def attention(self, q, k, v, scale, causal=False, nthreads=0):
        """Full forward from the definition.  Returns (o [B,H,N,D], lse [B,H,N]) fp64."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, D = _check4(q, k, v)
        o = np.empty((B, H, N, D), np.float64)
        lse = np.empty((B, H, N), np.float64)
        rc = self._lib.attn_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                       B, H, N, D, float(scale), int(bool(causal)),
                                       int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_fwd failed: %d" % rc)
        return o, lse

    def attention_gqa(self, q, k, v, scale, causal=False, nthreads=0):
        """Grouped-query forward: q [B,H,N,D], k and v [B,Hkv,N,D], H % Hkv == 0."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        if q.ndim != 4 or k.shape != v.shape or k.ndim != 4:
            raise ValueError("q [B,H,N,D], k and v [B,Hkv,N,D]")
        B, H, N, D = q.shape
        if k.shape[0] != B or k.shape[2] != N or k.shape[3] != D:
            raise ValueError("k/v must match q in B, N and D")
        Hkv = k.shape[1]
        o = np.empty((B, H, N, D), np.float64)
        lse = np.empty((B, H, N), np.float64)
        rc = self._lib.attn_oracle_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                           B, H, Hkv, N, D, float(scale), int(bool(causal)),
                                           int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_fwd_gqa failed: %d" % rc)
        return o, lse

    def attention_rows_gqa(self, q, k, v, scale, causal, bh_idx, row_idx, nthreads=0):
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, D = q.shape
        Hkv = k.shape[1]
        bh = np.ascontiguousarray(np.asarray(bh_idx, dtype=np.int64))
        ri = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int64))
        R = bh.shape[0]
        o = np.empty((R, D), np.float64)
        lse = np.empty((R,), np.float64)
        i64p = ctypes.POINTER(ctypes.c_int64)
        rc = self._lib.attn_oracle_rows_gqa(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, N, D,
                                            float(scale), int(bool(causal)),
                                            bh.ctypes.data_as(i64p), ri.ctypes.data_as(i64p), R,
                                            _ptr(o), _ptr(lse), int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_rows_gqa failed: %d" % rc)
        return o, lse

    def attention_rows(self, q, k, v, scale, causal, bh_idx, row_idx, nthreads=0):
        """Selected rows (bh_idx[r] = b*H+h, row_idx[r]).  Returns (o [R,D], lse [R])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, D = _check4(q, k, v)
        bh = np.ascontiguousarray(np.asarray(bh_idx, dtype=np.int64))
        ri = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int64))
        if bh.shape != ri.shape or bh.ndim != 1:
            raise ValueError("bh_idx and row_idx must be 1-D of equal length")
        R = bh.shape[0]
        o = np.empty((R, D), np.float64)
        lse = np.empty((R,), np.float64)
        i64p = ctypes.POINTER(ctypes.c_int64)
        rc = self._lib.attn_oracle_rows(_ptr(q), _ptr(k), _ptr(v), B, H, N, D,
                                        float(scale), int(bool(causal)),
                                        bh.ctypes.data_as(i64p), ri.ctypes.data_as(i64p), R,
                                        _ptr(o), _ptr(lse), int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_rows failed: %d" % rc)
        return o, lse

    def probabilities(self, q, k, scale, causal=False, bh=0):
        """Attention probabilities P [N,N] of head bh (0 where not visible)."""
        q, k = _f64(q), _f64(k)
        if q.ndim != 4 or q.shape != k.shape:
            raise ValueError("q, k must share one [B,H,N,D] shape")
        B, H, N, D = q.shape
        p = np.empty((N, N), np.float64)
        rc = self._lib.attn_oracle_probs(_ptr(q), _ptr(k), B, H, N, D, int(bh),
                                         float(scale), int(bool(causal)), _ptr(p))
        if rc != 0:
            raise RuntimeError("attn_oracle_probs failed: %d" % rc)
        return p

    def attention_online(self, q, k, v, scale, causal=False, Br=128, Bc=32, nthreads=0):
        """The tiled online-softmax method restated in fp64 (pins the tiling algebra)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, D = _check4(q, k, v)
        o = np.full((B, H, N, D), np.nan, np.float64)
        lse = np.full((B, H, N), np.nan, np.float64)
        rc = self._lib.attn_oracle_online_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                              B, H, N, D, float(scale), int(bool(causal)),
                                              int(Br), int(Bc), int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_online_fwd failed: %d" % rc)
        return o, lse

    def backward(self, q, k, v, dout, scale, causal=False, nthreads=0):
        """Gradients of sum(dout * O) from the definition.  Returns (dq, dk, dv) fp64."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
        B, H, N, D = _check4(q, k, v)
        if do.shape != q.shape:
            raise ValueError("dout must have q's shape")
        dq, dk, dv = (np.full((B, H, N, D), np.nan, np.float64) for _ in range(3))
        rc = self._lib.attn_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk),
                                       _ptr(dv), B, H, N, D, float(scale), int(bool(causal)),
                                       int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_bwd failed: %d" % rc)
        return dq, dk, dv

    def backward_gqa(self, q, k, v, dout, scale, causal=False, nthreads=0):
        """Grouped-query backward: q, dout [B,H,N,D]; k, v [B,Hkv,N,D].
        Returns (dq [B,H,N,D], dk, dv [B,Hkv,N,D]) fp64."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
        B, H, N, D = q.shape
        Hkv = k.shape[1]
        if k.shape != (B, Hkv, N, D) or v.shape != k.shape or do.shape != q.shape:
            raise ValueError("q, dout [B,H,N,D]; k, v [B,Hkv,N,D]")
        dq = np.full((B, H, N, D), np.nan, np.float64)
        dk = np.full((B, Hkv, N, D), np.nan, np.float64)
        dv = np.full((B, Hkv, N, D), np.nan, np.float64)
        rc = self._lib.attn_oracle_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk),
                                           _ptr(dv), B, H, Hkv, N, D, float(scale),
                                           int(bool(causal)), int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_bwd_gqa failed: %d" % rc)
        return dq, dk, dv

    def backward_rows(self, q, k, v, dout, scale, causal, bh_rows, rows, bh_keys, keys,
                      nthreads=0):
        """Selected rows of dQ (heads bh_rows, query rows `rows`) and of dK, dV
        (heads bh_keys, keys `keys`).  Returns (dq [R,D], dk [K,D], dv [K,D])."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
        B, H, N, D = _check4(q, k, v)
        if do.shape != q.shape:
            raise ValueError("dout must have q's shape")
        bh_rows = np.asarray(bh_rows, np.int64).ravel()
        bh_keys = np.asarray(bh_keys, np.int64).ravel()
        rows = np.ascontiguousarray(np.asarray(rows, np.int64).ravel())
        keys = np.ascontiguousarray(np.asarray(keys, np.int64).ravel())
        if bh_rows.shape != rows.shape or bh_keys.shape != keys.shape:
            raise ValueError("head and index lists must have equal lengths")
        heads = np.ascontiguousarray(np.unique(np.concatenate([bh_rows, bh_keys])))
        slot_rows = np.ascontiguousarray(np.searchsorted(heads, bh_rows).astype(np.int64))
        slot_keys = np.ascontiguousarray(np.searchsorted(heads, bh_keys).astype(np.int64))
        nh = heads.shape[0]
        lse = np.empty((nh, N), np.float64)
        delta = np.empty((nh, N), np.float64)
        i64p = ctypes.POINTER(ctypes.c_int64)
        ip = lambda a: a.ctypes.data_as(i64p)
        common = (_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, H, N, D, float(scale),
                  int(bool(causal)), ip(heads), nh)
        rc = self._lib.attn_oracle_bwd_stats(*common, _ptr(lse), _ptr(delta), int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_bwd_stats failed: %d" % rc)
        dq = np.empty((rows.shape[0], D), np.float64)
        dk = np.empty((keys.shape[0], D), np.float64)
        dv = np.empty((keys.shape[0], D), np.float64)
        rc = self._lib.attn_oracle_bwd_dq_rows(*common, _ptr(lse), _ptr(delta), ip(slot_rows),
                                               ip(rows), rows.shape[0], _ptr(dq), int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_bwd_dq_rows failed: %d" % rc)
        rc = self._lib.attn_oracle_bwd_dkdv_rows(*common, _ptr(lse), _ptr(delta), ip(slot_keys),
                                                 ip(keys), keys.shape[0], _ptr(dk), _ptr(dv),
                                                 int(nthreads))
        if rc != 0:
            raise RuntimeError("attn_oracle_bwd_dkdv_rows failed: %d" % rc)
        return dq, dk, dv


_default = None


def _get():
    global _default
    if _default is None:
        _default = OracleLib(_build.build())
    return _default


def default_threads():
    return _get().default_threads()


def attention(q, k, v, scale, causal=False, nthreads=0):
    return _get().attention(q, k, v, scale, causal, nthreads)


def attention_rows(q, k, v, scale, causal, bh_idx, row_idx, nthreads=0):
    return _get().attention_rows(q, k, v, scale, causal, bh_idx, row_idx, nthreads)


def probabilities(q, k, scale, causal=False, bh=0):
    return _get().probabilities(q, k, scale, causal, bh)


def attention_gqa(q, k, v, scale, causal=False, nthreads=0):
    return _get().attention_gqa(q, k, v, scale, causal, nthreads)


def attention_rows_gqa(q, k, v, scale, causal, bh_idx, row_idx, nthreads=0):
    return _get().attention_rows_gqa(q, k, v, scale, causal, bh_idx, row_idx, nthreads)


def attention_online(q, k, v, scale, causal=False, Br=128, Bc=32, nthreads=0):
    return _get().attention_online(q, k, v, scale, causal, Br, Bc, nthreads)


def backward(q, k, v, dout, scale, causal=False, nthreads=0):
    return _get().backward(q, k, v, dout, scale, causal, nthreads)


def backward_gqa(q, k, v, dout, scale, causal=False, nthreads=0):
    return _get().backward_gqa(q, k, v, dout, scale, causal, nthreads)


def backward_rows(q, k, v, dout, scale, causal, bh_rows, rows, bh_keys, keys, nthreads=0):
    return _get().backward_rows(q, k, v, dout, scale, causal, bh_rows, rows, bh_keys, keys,
                                nthreads)


def lib_path() -> str:
    return _build.LIB


__all__ = ["OracleLib", "attention", "attention_rows", "probabilities",
           "attention_online", "attention_gqa", "attention_rows_gqa", "backward", "backward_gqa",
           "backward_rows", "default_threads",
           "lib_path"]
