"""Python face of the decode-step oracle (oracle/oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the bench's
CPU-baseline leg, never by the library.  The C code is plain double-precision
loops; this module only marshals numpy arrays into it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with plain -O2 (no fast-math, no vector intrinsics), OpenMP
    for its (row, output) and (row, head) loops."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", "-fopenmp",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        D = ctypes.c_double
        L.orc_half_to_double.argtypes = [ctypes.c_uint16]
        L.orc_half_to_double.restype = D
        L.orc_double_to_half.argtypes = [D]
        L.orc_double_to_half.restype = ctypes.c_uint16
        L.orc_gemv_q8.argtypes = [P, I64, I64, P, I, I64, P, I64]
        L.orc_q8_dequant.argtypes = [P, I64, I64, P]
        L.orc_gemv_f16w.argtypes = [P, I64, I64, P, I, I64, P, I64]
        L.orc_matmul.argtypes = [P, I64, I64, P, I, I64, P, I64]
        L.orc_rope_vec.argtypes = [P, I, I, D, D]
        L.orc_rope_vec.restype = None
        L.orc_rope_kv_store.argtypes = [P, I64, P, I64, P, I64, P, P, P, I,
                                        I, I, I, I, I, D, P, I64, P, P, I64, I]
        L.orc_rope_kv_store_f32.argtypes = L.orc_rope_kv_store.argtypes
        L.orc_rope_kv_store_q8.argtypes = [P, I64, P, I64, P, I64, P, P, P, I,
                                           I, I, I, I, I, D, P, I64, P, P, P, P, I64, I]
        L.orc_q8_encode_block.argtypes = [P, P, P]
        L.orc_q8_encode_block.restype = None
        L.orc_attn_split_q8.argtypes = [P, I64, I, I, I, I, P, P, P, P, I64, I, P, P, I, I, P, P]
        L.orc_attn_full_q8.argtypes = [P, I64, I, I, I, I, P, P, P, P, I64, I, P, P, P, I64, P]
        L.orc_attn_split.argtypes = [P, I64, I, I, I, I, P, P, I64, I, P, P, I, I, P, P]
        L.orc_attn_split_f32.argtypes = L.orc_attn_split.argtypes
        L.orc_attn_merge.argtypes = [P, P, I, I, I, I, P, I64, P]
        L.orc_attn_full.argtypes = [P, I64, I, I, I, I, P, P, I64, I, P, P, P, I64, P]
        L.orc_attn_full_f32.argtypes = L.orc_attn_full.argtypes
        L.orc_plan_groups.argtypes = [I, I, P]
        L.orc_set_threads.argtypes = [I]
        L.orc_set_threads.restype = I
        L.orc_set_threads(1)
        for f in ("orc_gemv_q8", "orc_gemv_f16w", "orc_q8_dequant", "orc_matmul", "orc_rope_kv_store",
                  "orc_rope_kv_store_f32", "orc_rope_kv_store_q8", "orc_attn_split", "orc_attn_split_f32",
                  "orc_attn_split_q8", "orc_attn_merge", "orc_attn_full", "orc_attn_full_f32", "orc_attn_full_q8",
                  "orc_plan_groups"):
            getattr(L, f).restype = I
        _lib = L
    return _lib


def set_threads(n: int) -> int:
    """Threads of the oracle's parallel (row, output) and (row, head) loops from now on; returns the
    number in effect.  Results do not depend on it."""
    return int(lib().orc_set_threads(int(n)))


def _np(a, dtype) -> np.ndarray:
    """A C-contiguous numpy array of `dtype` (torch CPU tensors are accepted)."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, a.dtype))
    return a


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError("oracle %s rejected its arguments (rc=%d)" % (what, rc))


def half_to_double(h: int) -> float:
    return lib().orc_half_to_double(h)


def double_to_half(x: float) -> int:
    return lib().orc_double_to_half(x)


def gemv_q8(blocks, x) -> np.ndarray:
    """y[r][o] (float64) of Q8_0 blocks uint8 [n_out][n_in/32][34] against x float32 [rows][n_in]."""
    b = _np(blocks, np.uint8)
    xx = _np(x, np.float32)
    n_out, nb = b.shape[0], b.shape[1]
    n_in = nb * 32
    rows = xx.shape[0]
    assert xx.shape[1] == n_in
    y = np.zeros((rows, n_out), np.float64)
    _check(lib().orc_gemv_q8(_p(b), n_out, n_in, _p(xx), rows, n_in, _p(y), n_out), "gemv_q8")
    return y


def gemv_f16w(w, x) -> np.ndarray:
    """y[r][o] (float64) of an f16 weight matrix [n_out][n_in] (float16 values or their uint16
    bits) against x float32 [rows][n_in]."""
    if hasattr(w, "detach"):
        w = w.detach().cpu().numpy()
    ww = np.ascontiguousarray(w)
    if ww.dtype == np.float16:
        ww = ww.view(np.uint16)
    if ww.dtype != np.uint16:
        raise TypeError("expected float16 values or uint16 bits, got %s" % ww.dtype)
    xx = _np(x, np.float32)
    n_out, n_in = ww.shape
    rows = xx.shape[0]
    assert xx.shape[1] == n_in
    y = np.zeros((rows, n_out), np.float64)
    _check(lib().orc_gemv_f16w(_p(ww), n_out, n_in, _p(xx), rows, n_in, _p(y), n_out), "gemv_f16w")
    return y


def q8_dequant(blocks) -> np.ndarray:
    b = _np(blocks, np.uint8)
    n_out, n_in = b.shape[0], b.shape[1] * 32
    w = np.zeros((n_out, n_in), np.float64)
    _check(lib().orc_q8_dequant(_p(b), n_out, n_in, _p(w)), "q8_dequant")
    return w


def matmul(w, x) -> np.ndarray:
    ww = _np(w, np.float64)
    xx = _np(x, np.float32)
    n_out, n_in = ww.shape
    rows = xx.shape[0]
    y = np.zeros((rows, n_out), np.float64)
    _check(lib().orc_matmul(_p(ww), n_out, n_in, _p(xx), rows, n_in, _p(y), n_out), "matmul")
    return y


def rope_vec(x, rot_dim: int, neox: bool, theta: float, pos: float) -> np.ndarray:
    v = np.array(x, dtype=np.float64, copy=True)
    lib().orc_rope_vec(_p(v), rot_dim, 1 if neox else 0, float(theta), float(pos))
    return v


class Q8Plane:
    """A q8_0 mirror plane: int8 codes [reg][n_kv][cap][D] and f16 scale bits [reg][n_kv][cap][D/32]."""

    def __init__(self, codes: np.ndarray, scales: np.ndarray):
        assert codes.dtype == np.int8 and scales.dtype == np.uint16
        assert codes.flags.c_contiguous and scales.flags.c_contiguous
        assert codes.shape[:3] == scales.shape[:3] and codes.shape[3] == 32 * scales.shape[3]
        self.codes, self.scales = codes, scales
        self.shape = codes.shape

    def values(self) -> np.ndarray:
        """Decoded values (float64): scale * code."""
        d = self.scales.view(np.float16).astype(np.float64)
        return self.codes.astype(np.float64) * np.repeat(d, 32, axis=3)


def q8_encode_block(x) -> tuple:
    """The q8_0 mirror's encoding of 32 float32 values: (codes int8[32], scale bits uint16)."""
    xx = _np(np.asarray(x, np.float32), np.float32)
    assert xx.shape == (32,)
    q = np.zeros(32, np.int8)
    d = np.zeros(1, np.uint16)
    lib().orc_q8_encode_block(_p(xx), _p(q), _p(d))
    return q, int(d[0])


def rope_kv_store(q, k, v, pos, kcache, vcache, *, n_q, n_kv, head_dim, rot_dim, theta,
                  neox=True, bias=None, row_region=None):
    """Returns q' (float64 [rows][n_q*D]); writes kcache/vcache in place: uint16 [reg][n_kv][cap][D]
    (the f16 mirror) or float32 (the f32 mirror)."""
    qq = _np(q, np.float32).reshape(q.shape[0], -1)
    kk = _np(k, np.float32).reshape(k.shape[0], -1)
    vv = _np(v, np.float32).reshape(v.shape[0], -1)
    pp = _np(pos, np.int32)
    bb = None if bias is None else _np(bias, np.float32)
    rr = None if row_region is None else _np(row_region, np.int32)
    if isinstance(kcache, Q8Plane):
        rows = qq.shape[0]
        cap = kcache.shape[2]
        region_stride = kcache.shape[1] * cap * head_dim
        qo = np.zeros((rows, n_q * head_dim), np.float64)
        _check(lib().orc_rope_kv_store_q8(_p(qq), qq.shape[1], _p(kk), kk.shape[1], _p(vv), vv.shape[1],
                                          _p(bb), _p(pp), _p(rr), rows, n_q, n_kv, head_dim, rot_dim,
                                          1 if neox else 0, float(theta), _p(qo), n_q * head_dim,
                                          _p(kcache.codes), _p(kcache.scales), _p(vcache.codes), _p(vcache.scales),
                                          region_stride, cap), "rope_kv_store_q8")
        return qo
    assert kcache.dtype in (np.uint16, np.float32) and vcache.dtype == kcache.dtype
    assert kcache.flags.c_contiguous and vcache.flags.c_contiguous
    rows = qq.shape[0]
    cap = kcache.shape[2]
    region_stride = kcache.shape[1] * cap * head_dim
    qo = np.zeros((rows, n_q * head_dim), np.float64)
    fn = lib().orc_rope_kv_store_f32 if kcache.dtype == np.float32 else lib().orc_rope_kv_store
    _check(fn(_p(qq), qq.shape[1], _p(kk), kk.shape[1], _p(vv), vv.shape[1],
                                   _p(bb), _p(pp), _p(rr), rows, n_q, n_kv, head_dim, rot_dim,
                                   1 if neox else 0, float(theta), _p(qo), n_q * head_dim,
                                   _p(kcache), _p(vcache), region_stride, cap), "rope_kv_store")
    return qo


def attn_split(q, kcache, vcache, seqlen, *, n_q, n_kv, head_dim, chunk, n_splits, row_region=None):
    """Per-piece (o, lse): float64 [rows][n_q][n_splits][D] and [rows][n_q][n_splits]."""
    qq = np.ascontiguousarray(np.asarray(q, dtype=np.float64)).reshape(-1, n_q * head_dim)
    sl = _np(seqlen, np.int32)
    rr = None if row_region is None else _np(row_region, np.int32)
    rows = qq.shape[0]
    cap = kcache.shape[2]
    region_stride = kcache.shape[1] * cap * head_dim
    po = np.zeros((rows, n_q, n_splits, head_dim), np.float64)
    pl = np.zeros((rows, n_q, n_splits), np.float64)
    if isinstance(kcache, Q8Plane):
        _check(lib().orc_attn_split_q8(_p(qq), n_q * head_dim, rows, n_q, n_kv, head_dim,
                                       _p(kcache.codes), _p(kcache.scales), _p(vcache.codes), _p(vcache.scales),
                                       region_stride, cap, _p(rr), _p(sl), chunk, n_splits, _p(po), _p(pl)),
               "attn_split_q8")
        return po, pl
    fn = lib().orc_attn_split_f32 if np.asarray(kcache).dtype == np.float32 else lib().orc_attn_split
    _check(fn(_p(qq), n_q * head_dim, rows, n_q, n_kv, head_dim,
                                _p(np.ascontiguousarray(kcache)), _p(np.ascontiguousarray(vcache)),
                                region_stride, cap, _p(rr), _p(sl), chunk, n_splits,
                                _p(po), _p(pl)), "attn_split")
    return po, pl


def attn_merge(part_o, part_lse):
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    rows, n_q, n_splits, D = po.shape
    out = np.zeros((rows, n_q * D), np.float64)
    lse = np.zeros((rows, n_q), np.float64)
    _check(lib().orc_attn_merge(_p(po), _p(pl), rows, n_q, n_splits, D, _p(out), n_q * D, _p(lse)),
           "attn_merge")
    return out, lse


def attn_full(q, kcache, vcache, seqlen, *, n_q, n_kv, head_dim, row_region=None):
    qq = np.ascontiguousarray(np.asarray(q, dtype=np.float64)).reshape(-1, n_q * head_dim)
    sl = _np(seqlen, np.int32)
    rr = None if row_region is None else _np(row_region, np.int32)
    rows = qq.shape[0]
    cap = kcache.shape[2]
    region_stride = kcache.shape[1] * cap * head_dim
    out = np.zeros((rows, n_q * head_dim), np.float64)
    lse = np.zeros((rows, n_q), np.float64)
    if isinstance(kcache, Q8Plane):
        _check(lib().orc_attn_full_q8(_p(qq), n_q * head_dim, rows, n_q, n_kv, head_dim,
                                      _p(kcache.codes), _p(kcache.scales), _p(vcache.codes), _p(vcache.scales),
                                      region_stride, cap, _p(rr), _p(sl), _p(out), n_q * head_dim, _p(lse)),
               "attn_full_q8")
        return out, lse
    fn = lib().orc_attn_full_f32 if np.asarray(kcache).dtype == np.float32 else lib().orc_attn_full
    _check(fn(_p(qq), n_q * head_dim, rows, n_q, n_kv, head_dim,
                               _p(np.ascontiguousarray(kcache)), _p(np.ascontiguousarray(vcache)),
                               region_stride, cap, _p(rr), _p(sl), _p(out), n_q * head_dim, _p(lse)),
           "attn_full")
    return out, lse


def attention(q, kcache, vcache, seqlen, *, n_q, n_kv, head_dim, chunk, n_splits, row_region=None):
    """Split-KV attention followed by the merge: (out [rows][n_q*D], lse [rows][n_q])."""
    po, pl = attn_split(q, kcache, vcache, seqlen, n_q=n_q, n_kv=n_kv, head_dim=head_dim,
                        chunk=chunk, n_splits=n_splits, row_region=row_region)
    return attn_merge(po, pl)


def plan_groups(n: int, max_rows: int = 8):
    sizes = np.zeros(max(1, (n + max_rows - 1) // max_rows), np.int32)
    g = lib().orc_plan_groups(n, max_rows, _p(sizes))
    if g < 0:
        raise ValueError("plan_groups rejected n=%d" % n)
    return [int(s) for s in sizes[:g]]


def layer_step(blocks: dict, x, kcache, vcache, pos, *, n_q, n_kv, head_dim, theta, chunk, n_splits,
               regions=None, x_ffn=None, h=None):
    """One decode layer step in the oracle, the same sequence the library runs:
    QKV GEMV -> rope + KV store -> split attention + merge -> O GEMV, and the
    gate/up and down GEMVs on their own activation rows.  Caches are updated in
    place (uint16 f16 planes).  Returns a dict of float64 results."""
    D = head_dim
    qkv = gemv_q8(blocks["wqkv"], x)
    qd, kd = n_q * D, n_kv * D
    q = qkv[:, :qd].astype(np.float32)
    k = qkv[:, qd:qd + kd].astype(np.float32)
    v = qkv[:, qd + kd:].astype(np.float32)
    pos = np.asarray(pos, np.int32)
    qr = rope_kv_store(q, k, v, pos, kcache, vcache, n_q=n_q, n_kv=n_kv, head_dim=D, rot_dim=D,
                       theta=theta, row_region=None if regions is None else np.asarray(regions, np.int32))
    out, lse = attention(qr, kcache, vcache, pos + 1, n_q=n_q, n_kv=n_kv, head_dim=D, chunk=chunk,
                         n_splits=n_splits, row_region=None if regions is None else np.asarray(regions, np.int32))
    res = {"qkv": qkv, "q": qr, "attn": out, "lse": lse,
           "y_o": gemv_q8(blocks["wo"], out.astype(np.float32))}
    if "wgu" in blocks and x_ffn is not None:
        res["gu"] = gemv_q8(blocks["wgu"], x_ffn)
        res["y_down"] = gemv_q8(blocks["wdown"], h)
    return res
