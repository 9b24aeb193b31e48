"""GB300 decode-step library: Python binding of libdl_gb300.so.

Argument marshalling only.  Every step of the decode path runs in the library's
CUDA kernels; torch supplies device memory (tensors) and the current stream.
There is no fallback: if the shared library is missing or a call fails, an
exception is raised.

The functions carry the C names of include/dl.h (dl_gemv_q8, dl_rope_kv_store,
dl_decode_attn, dl_attn_merge, ...) and take torch tensors where the C call
takes device pointers.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdl_gb300.so")

DL_OK = 0
DL_E_ARG = -1
DL_E_SHAPE = -2
DL_E_ALIGN = -3
DL_E_WORKSPACE = -4
DL_E_CUDA = -5
DL_E_RANGE = -6
DL_STATUS_POS_RANGE = 0x1
DL_STATUS_REGION_RANGE = 0x2
DL_STATUS_SEQLEN_RANGE = 0x4
DL_STATUS_SYNC_TIMEOUT = 0x8
DL_MAX_ROWS = 8

_ERRNAMES = {DL_E_ARG: "DL_E_ARG", DL_E_SHAPE: "DL_E_SHAPE", DL_E_ALIGN: "DL_E_ALIGN",
             DL_E_WORKSPACE: "DL_E_WORKSPACE", DL_E_CUDA: "DL_E_CUDA", DL_E_RANGE: "DL_E_RANGE"}


class DLError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("%s (%d): %s" % (_ERRNAMES.get(code, "DL_E_?"), code, msg))
        self.code = code


class dl_q8_weight(ctypes.Structure):
    _fields_ = [("qs", ctypes.c_void_p), ("d", ctypes.c_void_p),
                ("n_out", ctypes.c_int64), ("n_in", ctypes.c_int64)]


class dl_f16_weight(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("n_out", ctypes.c_int64), ("n_in", ctypes.c_int64)]


class dl_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("region_stride", ctypes.c_int64),
                ("n_regions", ctypes.c_int), ("n_kv", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("capacity", ctypes.c_int), ("elem_bytes", ctypes.c_int),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


class dl_rope(ctypes.Structure):
    _fields_ = [("cos_sin", ctypes.c_void_p), ("max_pos", ctypes.c_int), ("rot_dim", ctypes.c_int),
                ("neox", ctypes.c_int)]


_R = DL_MAX_ROWS


class dl_attn_plan(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int), ("n_q", ctypes.c_int), ("n_kv", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("chunk", ctypes.c_int), ("max_splits", ctypes.c_int),
                ("n_sessions", ctypes.c_int), ("n_work", ctypes.c_int), ("sm_count", ctypes.c_int),
                ("cluster", ctypes.c_int),
                ("row_region", ctypes.c_int * _R), ("row_keys_max", ctypes.c_int * _R),
                ("sess_rows", ctypes.c_int * _R), ("sess_begin", ctypes.c_int * (_R + 1)),
                ("sess_splits", ctypes.c_int * _R), ("sess_item0", ctypes.c_int * (_R + 1)),
                ("workspace_bytes", ctypes.c_size_t)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libdl_gb300.so is not built (run __graft_entry__.build() or "
                               "python row_decode_step_gb300/_build.py)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "dl_last_error": ([], ctypes.c_char_p),
            "dl_version": ([], I),
            "dl_status_read": ([P, P], I),
            "dl_l2_prefetch_next": ([I, P, P], I),
            "dl_q8_packed_size": ([I64, I64, P, P], I),
            "dl_q8_pack": ([P, I64, I64, P, P, P], I),
            "dl_gemv_q8": ([P, P, I, I64, P, I64, P], I),
            "dl_gemv_q8_ex": ([P, P, I, I64, P, I64, I, P], I),
            "dl_gemv_q8_chain": ([P, P, P, P, P, I, I, P, P, I, P], I),
            "dl_f16w_packed_size": ([I64, I64, P], I),
            "dl_f16w_pack": ([P, I64, I64, P, P], I),
            "dl_gemv_f16w": ([P, P, I, I64, P, I64, P], I),
            "dl_gemv_f16w_ex": ([P, P, I, I64, P, I64, I, P], I),
            "dl_rope_table_bytes": ([I, I, P], I),
            "dl_rope_table_build": ([ctypes.c_double, I, I, P], I),
            "dl_rope_kv_store": ([P, I64, P, I64, P, I64, P, P, P, I, I, P, P, P, P], I),
            "dl_plan_groups": ([I, I, P], I),
            "dl_attn_plan_build": ([I, P, P, I, I, I, I, I, P], I),
            "dl_decode_attn": ([P, I64, P, P, P, P, SZ, P, P], I),
            "dl_decode_attn_ex": ([P, I64, P, P, P, P, SZ, P, I, P], I),
            "dl_decode_attn_rope": ([P, I64, P, I64, P, I64, P, P, P, P, P, P, P, SZ, P, I, P], I),
            "dl_attn_plan_build_cluster": ([I, P, P, I, I, I, I, I, P], I),
            "dl_decode_attn_cluster": ([P, I64, P, P, P, P, P, I64, P, P, I, P], I),
            "dl_decode_attn_merged": ([P, I64, P, P, P, P, P, SZ, P, I64, P, P, I, P], I),
            "dl_attn_merge": ([P, P, P, P, I64, P, P], I),
            "dl_layer_step_workspace_size": ([P, P, P], I),
            "dl_layer_step": ([P, P, P, P, P, P, P, P, P, SZ, P, I, P], I),
            "dl_decode_attention_noalloc_max_bytes": ([], SZ),
            "dl_decode_attention_noalloc": ([P, I64, P, P, P, P, I64, P, P, P], I),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(rc: int):
    if rc != DL_OK:
        raise DLError(rc, lib().dl_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


# ------------------------------------------------------------------ weights

class PackedQ8:
    """A Q8_0 weight in the library's device form (two planes kept alive here)."""

    def __init__(self, qs: torch.Tensor, d: torch.Tensor, n_out: int, n_in: int):
        self.qs, self.d, self.n_out, self.n_in = qs, d, int(n_out), int(n_in)
        self.c = dl_q8_weight(qs.data_ptr(), d.data_ptr(), self.n_out, self.n_in)

    @property
    def nbytes_q8_0(self) -> int:
        """Bytes of the same matrix in the 34-bytes-per-32 interchange form."""
        return self.n_out * self.n_in // 32 * 34


def dl_q8_packed_size(n_out: int, n_in: int):
    qb, db = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().dl_q8_packed_size(n_out, n_in, ctypes.byref(qb), ctypes.byref(db)))
    return qb.value, db.value


def dl_q8_pack(blocks: torch.Tensor, n_out: int, n_in: int, stream=None) -> PackedQ8:
    """Pack interchange Q8_0 blocks (uint8 CUDA tensor, n_out*n_in/32*34 bytes)."""
    _dev(blocks, torch.uint8, "blocks")
    if not blocks.is_contiguous() or blocks.numel() != n_out * (n_in // 32) * 34:
        raise ValueError("blocks must be contiguous [n_out][n_in/32][34]")
    qb, db = dl_q8_packed_size(n_out, n_in)
    qs = torch.empty(qb, dtype=torch.uint8, device=blocks.device)
    d = torch.empty(db, dtype=torch.uint8, device=blocks.device)
    _check(lib().dl_q8_pack(_ptr(blocks), n_out, n_in, _ptr(qs), _ptr(d), _stream(stream)))
    return PackedQ8(qs, d, n_out, n_in)


class PackedF16W:
    """An f16 weight in the library's device form (the plane kept alive here)."""

    def __init__(self, w: torch.Tensor, n_out: int, n_in: int):
        self.w, self.n_out, self.n_in = w, int(n_out), int(n_in)
        self.c = dl_f16_weight(w.data_ptr(), self.n_out, self.n_in)

    @property
    def nbytes_f16(self) -> int:
        """Bytes of the matrix as f16 values."""
        return self.n_out * self.n_in * 2


def dl_f16w_packed_size(n_out: int, n_in: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().dl_f16w_packed_size(n_out, n_in, ctypes.byref(b)))
    return b.value


def dl_f16w_pack(w: torch.Tensor, stream=None) -> PackedF16W:
    """Pack a row-major f16 weight matrix (float16 CUDA tensor [n_out][n_in])."""
    _dev(w, torch.float16, "w")
    if w.dim() != 2 or not w.is_contiguous():
        raise ValueError("w must be a contiguous [n_out][n_in] float16 tensor")
    n_out, n_in = w.shape
    packed = torch.empty(dl_f16w_packed_size(n_out, n_in), dtype=torch.uint8, device=w.device)
    _check(lib().dl_f16w_pack(_ptr(w), n_out, n_in, _ptr(packed), _stream(stream)))
    return PackedF16W(packed, n_out, n_in)


GEMV_PATH_AUTO, GEMV_PATH_CUDA_CORE, GEMV_PATH_TENSOR = 0, 1, 2


def dl_gemv_q8(W: PackedQ8, x: torch.Tensor, y: Optional[torch.Tensor] = None, stream=None,
               path: int = GEMV_PATH_AUTO) -> torch.Tensor:
    """y[r] = W x[r] for every row of x (f32 [rows][>= n_in], rows may exceed eight).
    `path` selects the inner product (dl_gemv_q8_ex); the default is the library's choice."""
    _dev(x, torch.float32, "x")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit inner stride")
    rows = x.shape[0]
    if y is None:
        y = torch.empty(rows, W.n_out, dtype=torch.float32, device=x.device)
    _dev(y, torch.float32, "y")
    if path == GEMV_PATH_AUTO:
        _check(lib().dl_gemv_q8(ctypes.byref(W.c), _ptr(x), rows, x.stride(0), _ptr(y), y.stride(0),
                                _stream(stream)))
    else:
        _check(lib().dl_gemv_q8_ex(ctypes.byref(W.c), _ptr(x), rows, x.stride(0), _ptr(y), y.stride(0),
                                   path, _stream(stream)))
    return y


def dl_gemv_f16w(W: PackedF16W, x: torch.Tensor, y: Optional[torch.Tensor] = None, stream=None,
                 path: int = GEMV_PATH_AUTO) -> torch.Tensor:
    """y[r] = W x[r] for every row of x with f16 weights (f32 [rows][>= n_in], rows may exceed eight)."""
    _dev(x, torch.float32, "x")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit inner stride")
    rows = x.shape[0]
    if y is None:
        y = torch.empty(rows, W.n_out, dtype=torch.float32, device=x.device)
    _dev(y, torch.float32, "y")
    if path == GEMV_PATH_AUTO:
        _check(lib().dl_gemv_f16w(ctypes.byref(W.c), _ptr(x), rows, x.stride(0), _ptr(y), y.stride(0),
                                  _stream(stream)))
    else:
        _check(lib().dl_gemv_f16w_ex(ctypes.byref(W.c), _ptr(x), rows, x.stride(0), _ptr(y), y.stride(0),
                                     path, _stream(stream)))
    return y


def dl_gemv_q8_chain(Ws: Sequence[PackedQ8], xs: Sequence[torch.Tensor], ys: Sequence[torch.Tensor],
                     sync: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None,
                     path: int = GEMV_PATH_AUTO) -> None:
    """Phases y_p = W_p x_p in one persistent launch, in order (x_{p+1} may be y_p); `sync` is a
    zeroed int32 CUDA tensor of at least 4 elements, reused call after call."""
    n = len(Ws)
    assert len(xs) == n and len(ys) == n and n >= 1
    rows = xs[0].shape[0]
    for t in list(xs) + list(ys):
        _dev(t, torch.float32, "x/y")
        if t.dim() != 2 or t.stride(1) != 1 or t.shape[0] != rows:
            raise ValueError("x and y must be 2-D rows with unit inner stride, the same row count")
    _dev(sync, torch.int32, "sync")
    Warr = (ctypes.c_void_p * n)(*[ctypes.cast(ctypes.pointer(W.c), ctypes.c_void_p) for W in Ws])
    xarr = (ctypes.c_void_p * n)(*[t.data_ptr() for t in xs])
    yarr = (ctypes.c_void_p * n)(*[t.data_ptr() for t in ys])
    xst = (ctypes.c_int64 * n)(*[t.stride(0) for t in xs])
    yst = (ctypes.c_int64 * n)(*[t.stride(0) for t in ys])
    _check(lib().dl_gemv_q8_chain(Warr, xarr, xst, yarr, yst, n, rows, _ptr(sync), _ptr(status), path,
                                  _stream(stream)))


# ------------------------------------------------------------------ KV cache

class KVCache:
    """A K/V mirror [n_regions][n_kv][capacity][head_dim]: float16 (the default) or float32."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor):
        assert k.shape == v.shape and k.dim() == 4
        dt = torch.float32 if k.dtype == torch.float32 else torch.float16
        _dev(k, dt, "k")
        _dev(v, dt, "v")
        self.k, self.v = k, v
        n_reg, n_kv, cap, D = k.shape
        self.c = dl_kv_cache(k.data_ptr(), v.data_ptr(), k.stride(0), n_reg, n_kv, D, cap,
                             4 if dt == torch.float32 else 2, None, None)

    @classmethod
    def q8(cls, k_codes: torch.Tensor, k_scale: torch.Tensor, v_codes: torch.Tensor, v_scale: torch.Tensor):
        """The q8_0 mirror: int8 codes [n_regions][n_kv][capacity][head_dim] and float16 scales
        [n_regions][n_kv][capacity][head_dim / 32]."""
        assert k_codes.shape == v_codes.shape and k_codes.dim() == 4
        assert k_scale.shape == v_scale.shape and tuple(k_scale.shape) == tuple(k_codes.shape[:3]) + (
            k_codes.shape[3] // 32,)
        for t, n in ((k_codes, "k_codes"), (v_codes, "v_codes")):
            _dev(t, torch.int8, n)
        for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
            _dev(t, torch.float16, n)
        self = cls.__new__(cls)
        self.k, self.v, self.k_scale, self.v_scale = k_codes, v_codes, k_scale, v_scale
        n_reg, n_kv, cap, D = k_codes.shape
        self.c = dl_kv_cache(k_codes.data_ptr(), v_codes.data_ptr(), k_codes.stride(0), n_reg, n_kv, D, cap, 1,
                             k_scale.data_ptr(), v_scale.data_ptr())
        return self

    @classmethod
    def empty(cls, n_regions, n_kv, capacity, head_dim, device="cuda", dtype=torch.float16):
        shape = (n_regions, n_kv, capacity, head_dim)
        return cls(torch.empty(shape, dtype=dtype, device=device), torch.empty(shape, dtype=dtype, device=device))


class Rope:
    def __init__(self, table: torch.Tensor, max_pos: int, rot_dim: int, neox: bool = True):
        self.table = table
        self.c = dl_rope(table.data_ptr(), max_pos, rot_dim, 1 if neox else 0)


def dl_rope_table_build(theta: float, rot_dim: int, max_pos: int) -> torch.Tensor:
    """Host f32 table [max_pos][rot_dim/2][2] of (cos, sin), built in double precision."""
    t = torch.empty(max_pos, rot_dim // 2, 2, dtype=torch.float32)
    _check(lib().dl_rope_table_build(float(theta), rot_dim, max_pos, _ptr(t)))
    return t


def make_rope(theta: float, rot_dim: int, max_pos: int, neox: bool = True, device="cuda") -> Rope:
    return Rope(dl_rope_table_build(theta, rot_dim, max_pos).to(device), max_pos, rot_dim, neox)


def dl_rope_kv_store(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, pos: torch.Tensor,
                     rope: Rope, kv: KVCache, n_q: int, bias: Optional[torch.Tensor] = None,
                     row_region: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev(t, torch.float32, n)
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("%s must be 2-D rows with unit inner stride" % n)
    _dev(pos, torch.int32, "pos")
    if bias is not None:
        _dev(bias, torch.float32, "bias")
    if row_region is not None:
        _dev(row_region, torch.int32, "row_region")
    if status is not None:
        _dev(status, torch.int32, "status")
    _check(lib().dl_rope_kv_store(_ptr(q), q.stride(0), _ptr(k), k.stride(0), _ptr(v), v.stride(0),
                                  _ptr(bias), _ptr(pos), _ptr(row_region), q.shape[0], n_q,
                                  ctypes.byref(rope.c), ctypes.byref(kv.c), _ptr(status), _stream(stream)))


# ------------------------------------------------------------------ planning and attention

def dl_plan_groups(n: int, max_rows: int = DL_MAX_ROWS):
    sizes = (ctypes.c_int * max(1, -(-n // max_rows)))()
    g = lib().dl_plan_groups(n, max_rows, sizes)
    if g < 0:
        _check(g)
    return [sizes[i] for i in range(g)]


def dl_attn_plan_build(seqlen: Sequence[int], n_q: int, n_kv: int, head_dim: int,
                       regions: Optional[Sequence[int]] = None, sm_count: int = 0,
                       force_chunk: int = 0) -> dl_attn_plan:
    rows = len(seqlen)
    sl = (ctypes.c_int32 * rows)(*[int(s) for s in seqlen])
    rg = None if regions is None else (ctypes.c_int32 * rows)(*[int(r) for r in regions])
    plan = dl_attn_plan()
    _check(lib().dl_attn_plan_build(rows, sl, rg, n_q, n_kv, head_dim, sm_count, force_chunk,
                                    ctypes.byref(plan)))
    return plan


def workspace_for(plan: dl_attn_plan, device="cuda") -> torch.Tensor:
    """A workspace for the plan, zeroed (the last-piece merge's counters start at zero)."""
    return torch.zeros(max(16, plan.workspace_bytes), dtype=torch.uint8, device=device)


ATTN_PATH_AUTO, ATTN_PATH_CUDA_CORE, ATTN_PATH_TENSOR = 0, 1, 2


def dl_decode_attn(q: torch.Tensor, kv: KVCache, seqlen: torch.Tensor, plan: dl_attn_plan,
                   workspace: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None,
                   path: int = ATTN_PATH_AUTO) -> None:
    _dev(q, torch.float32, "q")
    _dev(seqlen, torch.int32, "seqlen")
    _dev(workspace, torch.uint8, "workspace")
    if path == ATTN_PATH_AUTO:
        _check(lib().dl_decode_attn(_ptr(q), q.stride(0), ctypes.byref(kv.c), _ptr(seqlen), ctypes.byref(plan),
                                    _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream)))
    else:
        _check(lib().dl_decode_attn_ex(_ptr(q), q.stride(0), ctypes.byref(kv.c), _ptr(seqlen),
                                       ctypes.byref(plan), _ptr(workspace), workspace.numel(), _ptr(status),
                                       path, _stream(stream)))


def dl_decode_attn_rope(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, pos: torch.Tensor, rope: "Rope",
                        kv: KVCache, seqlen: torch.Tensor, plan: dl_attn_plan, workspace: torch.Tensor,
                        bias: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                        stream=None, path: int = ATTN_PATH_AUTO) -> None:
    """dl_rope_kv_store followed by dl_decode_attn_ex in one launch; q stays as projected."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev(t, torch.float32, n)
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("%s must be 2-D rows with unit inner stride" % n)
    _dev(pos, torch.int32, "pos")
    _dev(seqlen, torch.int32, "seqlen")
    _dev(workspace, torch.uint8, "workspace")
    if bias is not None:
        _dev(bias, torch.float32, "bias")
    if status is not None:
        _dev(status, torch.int32, "status")
    _check(lib().dl_decode_attn_rope(_ptr(q), q.stride(0), _ptr(k), k.stride(0), _ptr(v), v.stride(0),
                                     _ptr(bias), _ptr(pos), ctypes.byref(rope.c), ctypes.byref(kv.c),
                                     _ptr(seqlen), ctypes.byref(plan), _ptr(workspace), workspace.numel(),
                                     _ptr(status), path, _stream(stream)))


class dl_attn_rope_in(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("k_stride", ctypes.c_int64), ("v", ctypes.c_void_p),
                ("v_stride", ctypes.c_int64), ("bias", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("rope", ctypes.c_void_p)]


def dl_attn_plan_build_cluster(seqlen: Sequence[int], n_q: int, n_kv: int, head_dim: int,
                               regions: Optional[Sequence[int]] = None, sm_count: int = 0,
                               max_cluster: int = 0) -> dl_attn_plan:
    rows = len(seqlen)
    sl = (ctypes.c_int32 * rows)(*[int(s) for s in seqlen])
    rg = None if regions is None else (ctypes.c_int32 * rows)(*[int(r) for r in regions])
    plan = dl_attn_plan()
    _check(lib().dl_attn_plan_build_cluster(rows, sl, rg, n_q, n_kv, head_dim, sm_count, max_cluster,
                                            ctypes.byref(plan)))
    return plan


def dl_decode_attn_cluster(q: torch.Tensor, kv: KVCache, seqlen: torch.Tensor, plan: dl_attn_plan,
                           out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                           k: Optional[torch.Tensor] = None, v: Optional[torch.Tensor] = None,
                           pos: Optional[torch.Tensor] = None, rope: Optional["Rope"] = None,
                           bias: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                           stream=None, path: int = ATTN_PATH_AUTO) -> None:
    """Attention with the merge inside the launch (a plan from dl_attn_plan_build_cluster); with
    k, v, pos and rope given, the rope and store happen in the launch too."""
    _dev(q, torch.float32, "q")
    _dev(seqlen, torch.int32, "seqlen")
    _dev(out, torch.float32, "out")
    if lse is not None:
        _dev(lse, torch.float32, "lse")
    rin = None
    if k is not None:
        for t, n in ((k, "k"), (v, "v")):
            _dev(t, torch.float32, n)
        _dev(pos, torch.int32, "pos")
        if bias is not None:
            _dev(bias, torch.float32, "bias")
        rin = dl_attn_rope_in(_ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(bias), _ptr(pos),
                              ctypes.cast(ctypes.pointer(rope.c), ctypes.c_void_p))
    _check(lib().dl_decode_attn_cluster(_ptr(q), q.stride(0), None if rin is None else ctypes.byref(rin),
                                        ctypes.byref(kv.c), _ptr(seqlen), ctypes.byref(plan), _ptr(out),
                                        out.stride(0), _ptr(lse), _ptr(status), path, _stream(stream)))


def _rope_in(k, v, pos, rope, bias):
    if k is None:
        return None
    for t, n in ((k, "k"), (v, "v")):
        _dev(t, torch.float32, n)
    _dev(pos, torch.int32, "pos")
    if bias is not None:
        _dev(bias, torch.float32, "bias")
    return dl_attn_rope_in(_ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(bias), _ptr(pos),
                           ctypes.cast(ctypes.pointer(rope.c), ctypes.c_void_p))


def dl_decode_attn_merged(q: torch.Tensor, kv: KVCache, seqlen: torch.Tensor, plan: dl_attn_plan,
                          workspace: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                          k: Optional[torch.Tensor] = None, v: Optional[torch.Tensor] = None,
                          pos: Optional[torch.Tensor] = None, rope: Optional["Rope"] = None,
                          bias: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                          stream=None, path: int = ATTN_PATH_AUTO) -> None:
    """Attention whose last piece per (session, KV head) merges the partials (one launch; a
    workspace from workspace_for, zeroed once); with k, v, pos and rope given, the rope and
    store happen in the launch too."""
    _dev(q, torch.float32, "q")
    _dev(seqlen, torch.int32, "seqlen")
    _dev(workspace, torch.uint8, "workspace")
    _dev(out, torch.float32, "out")
    if lse is not None:
        _dev(lse, torch.float32, "lse")
    rin = _rope_in(k, v, pos, rope, bias)
    _check(lib().dl_decode_attn_merged(_ptr(q), q.stride(0), None if rin is None else ctypes.byref(rin),
                                       ctypes.byref(kv.c), _ptr(seqlen), ctypes.byref(plan), _ptr(workspace),
                                       workspace.numel(), _ptr(out), out.stride(0), _ptr(lse), _ptr(status), path,
                                       _stream(stream)))


def dl_attn_merge(workspace: torch.Tensor, plan: dl_attn_plan, seqlen: torch.Tensor,
                  out: torch.Tensor, lse: Optional[torch.Tensor] = None, stream=None) -> None:
    _dev(out, torch.float32, "out")
    _check(lib().dl_attn_merge(_ptr(workspace), ctypes.byref(plan), _ptr(seqlen), _ptr(out), out.stride(0),
                               _ptr(lse), _stream(stream)))


def dl_l2_prefetch_next(ranges) -> None:
    """Byte ranges the next launching call of this thread asks L2 to fetch for a later kernel:
    each a device tensor (its elements) or a (device pointer, bytes) pair."""
    ptrs, sizes = [], []
    for r in ranges:
        if isinstance(r, torch.Tensor):
            if not r.is_cuda or not r.is_contiguous():
                raise ValueError("dl_l2_prefetch_next: ranges must be contiguous device tensors")
            ptrs.append(r.data_ptr())
            sizes.append(r.numel() * r.element_size())
        else:
            ptrs.append(int(r[0]))
            sizes.append(int(r[1]))
    n = len(ptrs)
    _check(lib().dl_l2_prefetch_next(n, (ctypes.c_void_p * max(1, n))(*ptrs),
                                     (ctypes.c_size_t * max(1, n))(*sizes)))


def dl_status_read(status: torch.Tensor) -> int:
    v = ctypes.c_int32()
    _check(lib().dl_status_read(_ptr(status), ctypes.byref(v)))
    return v.value


def decode_attention(q, kv, seqlen, plan, workspace, out=None, lse=None, status=None, stream=None, path=0):
    """dl_decode_attn followed by dl_attn_merge; returns (out, lse)."""
    rows = plan.rows
    if out is None:
        out = torch.empty(rows, plan.n_q * plan.head_dim, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(rows, plan.n_q, dtype=torch.float32, device=q.device)
    dl_decode_attn(q, kv, seqlen, plan, workspace, status=status, stream=stream, path=path)
    dl_attn_merge(workspace, plan, seqlen, out, lse, stream=stream)
    return out, lse


# ------------------------------------------------------------------ whole layer step

class dl_layer_weights(ctypes.Structure):
    _fields_ = [("qkv", dl_q8_weight), ("o", dl_q8_weight), ("gu", dl_q8_weight), ("down", dl_q8_weight)]


class dl_layer_bufs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("x_stride", ctypes.c_int64),
                ("qkv", ctypes.c_void_p), ("qkv_stride", ctypes.c_int64),
                ("attn", ctypes.c_void_p), ("attn_stride", ctypes.c_int64),
                ("lse", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("o_stride", ctypes.c_int64),
                ("x_ffn", ctypes.c_void_p), ("x_ffn_stride", ctypes.c_int64),
                ("gu", ctypes.c_void_p), ("gu_stride", ctypes.c_int64),
                ("x_down", ctypes.c_void_p), ("x_down_stride", ctypes.c_int64),
                ("down", ctypes.c_void_p), ("down_stride", ctypes.c_int64)]


def _q8c(W: Optional[PackedQ8]) -> dl_q8_weight:
    return dl_q8_weight(None, None, 0, 0) if W is None else W.c


def layer_weights_c(wqkv: PackedQ8, wo: PackedQ8, wgu: Optional[PackedQ8] = None,
                    wdown: Optional[PackedQ8] = None) -> dl_layer_weights:
    return dl_layer_weights(_q8c(wqkv), _q8c(wo), _q8c(wgu), _q8c(wdown))


def dl_layer_step_workspace_size(Wc: dl_layer_weights, plan: dl_attn_plan) -> int:
    b = ctypes.c_size_t()
    _check(lib().dl_layer_step_workspace_size(ctypes.byref(Wc), ctypes.byref(plan), ctypes.byref(b)))
    return b.value


def _rows2d(t: Optional[torch.Tensor], name: str):
    if t is None:
        return None, 0
    _dev(t, torch.float32, name)
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("%s must be 2-D rows with unit inner stride" % name)
    return t.data_ptr(), t.stride(0)


def dl_layer_step(Wc: dl_layer_weights, x: torch.Tensor, qkv: torch.Tensor, attn: torch.Tensor,
                  lse: Optional[torch.Tensor], o: torch.Tensor, x_ffn: Optional[torch.Tensor],
                  gu: Optional[torch.Tensor], x_down: Optional[torch.Tensor], down: Optional[torch.Tensor],
                  pos: torch.Tensor, rope: Rope, kv: KVCache, seqlen: torch.Tensor, plan: dl_attn_plan,
                  workspace: torch.Tensor, bias: Optional[torch.Tensor] = None,
                  status: Optional[torch.Tensor] = None, stream=None, path: int = GEMV_PATH_AUTO) -> None:
    """One command's whole layer step in one launch (weights from layer_weights_c; the workspace
    zeroed once, dl_layer_step_workspace_size bytes)."""
    B = dl_layer_bufs()
    B.x, B.x_stride = _rows2d(x, "x")
    B.qkv, B.qkv_stride = _rows2d(qkv, "qkv")
    B.attn, B.attn_stride = _rows2d(attn, "attn")
    if lse is not None:
        _dev(lse, torch.float32, "lse")
        B.lse = lse.data_ptr()
    B.o, B.o_stride = _rows2d(o, "o")
    B.x_ffn, B.x_ffn_stride = _rows2d(x_ffn, "x_ffn")
    B.gu, B.gu_stride = _rows2d(gu, "gu")
    B.x_down, B.x_down_stride = _rows2d(x_down, "x_down")
    B.down, B.down_stride = _rows2d(down, "down")
    _dev(pos, torch.int32, "pos")
    _dev(seqlen, torch.int32, "seqlen")
    _dev(workspace, torch.uint8, "workspace")
    if bias is not None:
        _dev(bias, torch.float32, "bias")
    if status is not None:
        _dev(status, torch.int32, "status")
    _check(lib().dl_layer_step(ctypes.byref(Wc), ctypes.byref(B), _ptr(bias), _ptr(pos), ctypes.byref(rope.c),
                               ctypes.byref(kv.c), _ptr(seqlen), ctypes.byref(plan), _ptr(workspace),
                               workspace.numel(), _ptr(status), path, _stream(stream)))


def device_sm_count(device=None) -> int:
    return torch.cuda.get_device_properties(device if device is not None else torch.cuda.current_device()).multi_processor_count

