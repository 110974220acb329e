"""Multi-Segment Attention (MSA) on one B300 -- thin Python binding of libmsa.so.

The library (C ABI declared in include/msa.h) does all the work: the host planner and
the sm_103a kernels.  This module only marshals arguments: numpy arrays for the layout,
torch CUDA tensors for device memory and the current torch stream for ordering.  There
is no fallback: if libmsa.so cannot be loaded every call raises.

Paper: "Multi-Segment Attention: Enabling Efficient KV-Cache Management for Faster Large
Language Model Serving" (Eq. 1; section 4.1; abstract).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# MSA_LIBRARY=debug selects the MSA_DEBUG build (device-side bounds checks; build.py --debug)
LIB_PATH = os.path.join(_PKG, "libmsa_debug.so" if os.environ.get("MSA_LIBRARY") == "debug" else "libmsa.so")

MSA_PREFILL, MSA_DECODE = 0, 1
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported", -3: "position overlap",
          -4: "block out of range", -5: "workspace", -6: "cuda", -7: "timeout", -8: "mode"}


class MSAError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({code})")
        self.code = code


class _Opts(ctypes.Structure):
    _fields_ = [("num_heads_q", ctypes.c_int32), ("num_heads_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("decode_split_blocks", ctypes.c_int32), ("decode_min_ctas", ctypes.c_int32),
                ("prefill_ctas", ctypes.c_int32), ("chunk_queries_only", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2)]


class _Stats(ctypes.Structure):
    _fields_ = [("useful_flops", ctypes.c_int64), ("kv_tokens", ctypes.c_int64),
                ("algorithmic_bytes", ctypes.c_int64), ("num_kv_tiles", ctypes.c_int32),
                ("num_q_tiles", ctypes.c_int32), ("num_work_items", ctypes.c_int32),
                ("num_tile_pairs", ctypes.c_int32), ("num_partial_pairs", ctypes.c_int32),
                ("num_splits", ctypes.c_int32), ("num_prefill_ctas", ctypes.c_int32),
                ("num_split_items", ctypes.c_int32)]


class _EvictOpts(ctypes.Structure):
    _fields_ = [("k5", ctypes.c_double), ("k_const", ctypes.c_double), ("beta", ctypes.c_double),
                ("alpha", ctypes.c_double), ("tau0", ctypes.c_double), ("lambda0", ctypes.c_double),
                ("window", ctypes.c_int32), ("period", ctypes.c_int32), ("policy", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_I32P = ctypes.POINTER(ctypes.c_int32)

EXPORTS = {
    # name: (restype, argtypes)
    "msa_plan_create": (_I32, [ctypes.POINTER(_Opts), _I32, _I32, _P, _I32, _P, _I32, _P, _P, _I32, _P, _P,
                               ctypes.POINTER(_P)]),
    "msa_plan_destroy": (None, [_P]),
    "msa_plan_device_bytes": (_SZ, [_P]),
    "msa_plan_upload": (_I32, [_P, _P, _SZ, _P]),
    "msa_workspace_bytes": (_SZ, [_P]),
    "msa_workspace_init": (_I32, [_P, _SZ, _P]),
    "msa_plan_export": (_I32, [_P, _P, _SZ, ctypes.POINTER(_SZ)]),
    "msa_plan_export_splits": (_I32, [_P, _P, _SZ, ctypes.POINTER(_SZ)]),
    "msa_plan_export_schedule": (_I32, [_P, _P, _SZ, ctypes.POINTER(_SZ)]),
    "msa_plan_get_stats": (_I32, [_P, ctypes.POINTER(_Stats)]),
    "msa_chunk_sizes": (_I32, [_I32, _I32, _I32, _P, _I32, _I32P]),
    "msa_prefill": (_I32, [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _SZ, _P]),
    "msa_decode": (_I32, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _SZ, _P]),
    "msa_decode_no_alloc": (_I32, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P]),
    "msa_get_status_no_alloc": (_I32, [_P]),
    "msa_merge_lse": (_I32, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P]),
    "msa_gather": (_I32, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "msa_append_plan": (_I32, [_P, _I32, _P, _I32, _P, _I32, _P, _P, _I32, _P, _P, _I32P]),
    "msa_kv_append": (_I32, [_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P]),
    "msa_get_status": (_I32, [_P, _P]),
    "msa_set_wait_limit": (None, [ctypes.c_int64]),
    "msa_set_test_drop": (None, [_I32, _I32, _I32]),
    "msa_evict_create": (_I32, [ctypes.POINTER(_EvictOpts), ctypes.POINTER(_P)]),
    "msa_evict_destroy": (None, [_P]),
    "msa_evict_insert": (_I32, [_P, _I32, _I32, ctypes.c_double]),
    "msa_evict_access": (_I32, [_P, _I32, ctypes.c_double]),
    "msa_evict_remove": (_I32, [_P, _I32]),
    "msa_evict_victim": (_I32, [_P, ctypes.c_double, _I32P]),
    "msa_evict_score": (_I32, [_P, _I32, ctypes.c_double, ctypes.POINTER(ctypes.c_double)]),
    "msa_evict_get_lambda": (_I32, [_P, ctypes.POINTER(ctypes.c_double)]),
    "msa_evict_size": (_I32, [_P]),
    "msa_evict_check": (_I32, [_P, ctypes.c_double]),
    "msa_status_string": (ctypes.c_char_p, [_I32]),
    "msa_version": (_I32, []),
}


def lib():
    """Load libmsa.so (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmsa.so is not built ({LIB_PATH}); run "
                               "`python -m segmented_kv_attention_msa_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(code: int, what: str):
    if code != 0:
        raise MSAError(int(code), what)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def chunk_sizes(R: int, min_chunk: int, max_chunk: int) -> list:
    """Adaptive chunk tiler of the library (see msa_chunk_sizes in include/msa.h)."""
    n = ctypes.c_int32(0)
    _check(lib().msa_chunk_sizes(R, min_chunk, max_chunk, None, 0, ctypes.byref(n)), "msa_chunk_sizes")
    out = np.zeros(max(1, n.value), np.int32)
    _check(lib().msa_chunk_sizes(R, min_chunk, max_chunk, _ptr(out), len(out), ctypes.byref(n)),
           "msa_chunk_sizes")
    return [int(x) for x in out[:n.value]]


class Plan:
    """Host plan (validated layout, tiles, work list) plus its device image."""

    def __init__(self, mode: str, num_heads_q: int, num_heads_kv: int, head_dim: int,
                 segments, block_table, block_pos, block_fill, cu_q, q_pos=None,
                 decode_split_blocks: int = 0, decode_min_ctas: int = 0, prefill_ctas: int = 0,
                 chunk_queries_only: bool = False):
        self.mode = mode
        m = MSA_PREFILL if mode == "prefill" else MSA_DECODE
        opts = _Opts(num_heads_q, num_heads_kv, head_dim, 16, decode_split_blocks, decode_min_ctas,
                     prefill_ctas, 1 if chunk_queries_only else 0)
        self._keep = [np.ascontiguousarray(np.asarray(x, np.int32)) for x in
                      (segments, block_table, block_pos, block_fill, cu_q,
                       q_pos if q_pos is not None else np.zeros(0, np.int32))]
        seg, bt, bp, bf, cq, qp = self._keep
        num_seqs = len(cq) - 1
        h = ctypes.c_void_p(0)
        _check(lib().msa_plan_create(ctypes.byref(opts), m, num_seqs, _ptr(seg), len(seg.reshape(-1, 3)),
                                     _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0, _ptr(bp), _ptr(bf),
                                     len(bp), _ptr(cq), _ptr(qp) if qp.size else None, ctypes.byref(h)),
               "msa_plan_create")
        self._h = h
        self.num_heads_q, self.num_heads_kv, self.head_dim = num_heads_q, num_heads_kv, head_dim
        self.num_seqs = num_seqs
        self.total_q = int(cq[-1])
        self.num_pool_blocks = int(bp.shape[0])
        self.dev = None
        self.ws = None

    @classmethod
    def from_layout(cls, layout, **kw) -> "Plan":
        return cls(layout.mode, layout.num_heads_q, layout.num_heads_kv, layout.head_dim,
                   layout.segments, layout.block_table, layout.block_pos, layout.block_fill,
                   layout.cu_q, layout.q_pos if layout.mode == "prefill" else None, **kw)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.msa_plan_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    @property
    def device_bytes(self) -> int:
        return int(lib().msa_plan_device_bytes(self._h))

    @property
    def workspace_bytes(self) -> int:
        return int(lib().msa_workspace_bytes(self._h))

    def export(self) -> np.ndarray:
        n = ctypes.c_size_t(0)
        _check(lib().msa_plan_export(self._h, None, 0, ctypes.byref(n)), "msa_plan_export")
        out = np.zeros(n.value, np.int32)
        _check(lib().msa_plan_export(self._h, _ptr(out), n.value, ctypes.byref(n)), "msa_plan_export")
        return out

    def export_splits(self) -> np.ndarray:
        n = ctypes.c_size_t(0)
        _check(lib().msa_plan_export_splits(self._h, None, 0, ctypes.byref(n)), "msa_plan_export_splits")
        out = np.zeros(max(1, n.value), np.int32)
        _check(lib().msa_plan_export_splits(self._h, _ptr(out), n.value, ctypes.byref(n)),
               "msa_plan_export_splits")
        return out[:n.value].reshape(-1, 3)

    def export_schedule(self) -> np.ndarray:
        """Prefill pieces, one row each: (cta, qt, g, h0, j0, n, nparts, slot0, slot)."""
        n = ctypes.c_size_t(0)
        _check(lib().msa_plan_export_schedule(self._h, None, 0, ctypes.byref(n)), "msa_plan_export_schedule")
        out = np.zeros(max(1, n.value), np.int32)
        _check(lib().msa_plan_export_schedule(self._h, _ptr(out), n.value, ctypes.byref(n)),
               "msa_plan_export_schedule")
        return out[:n.value].reshape(-1, 9)

    def stats(self) -> dict:
        s = _Stats()
        _check(lib().msa_plan_get_stats(self._h, ctypes.byref(s)), "msa_plan_get_stats")
        return {f: int(getattr(s, f)) for f, _ in _Stats._fields_}

    def upload(self, device="cuda", stream=None):
        """Allocate the device image and workspace (torch) and fill them (library calls)."""
        import torch
        nb = max(256, self.device_bytes)
        self.dev = torch.empty(nb, dtype=torch.uint8, device=device)
        _check(lib().msa_plan_upload(self._h, _dptr(self.dev), nb, _stream(stream)), "msa_plan_upload")
        wb = max(256, self.workspace_bytes)
        self.ws = torch.empty(wb, dtype=torch.uint8, device=device)
        _check(lib().msa_workspace_init(_dptr(self.ws), wb, _stream(stream)), "msa_workspace_init")
        return self


def _expect(t, shape, name, dtype=None, min_first=False):
    """Raise ValueError unless tensor `t` has `shape` (with min_first: a first dimension of
    at least shape[0]) and, if given, `dtype`.  The C ABI takes raw pointers and cannot
    check sizes, so this is where a too-small tensor is caught before a kernel reads or
    writes past its end."""
    s = tuple(t.shape)
    ok = len(s) == len(shape) and s[1:] == tuple(shape[1:]) and (
        s[0] >= shape[0] if min_first else s[0] == shape[0])
    if not ok:
        need = ("at least " if min_first else "") + str(tuple(shape))
        raise ValueError(f"{name} has shape {s}; the plan needs {need}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}; the plan needs {dtype}")


def _check_pool(plan: "Plan", k_pool, v_pool):
    shape = (plan.num_pool_blocks, plan.num_heads_kv, 16, plan.head_dim)
    _expect(k_pool, shape, "k_pool", min_first=True)
    _expect(v_pool, tuple(k_pool.shape), "v_pool")


def _check_outputs(plan: "Plan", rows: int, out, lse):
    import torch
    _expect(out, (rows, plan.num_heads_q, plan.head_dim), "out", torch.bfloat16)
    _expect(lse, (rows, plan.num_heads_q), "lse", torch.float32)
    if not lse.is_contiguous():
        raise ValueError("lse must be contiguous")


def check_prefill_args(plan: "Plan", q, k_chunk, v_chunk, k_pool, v_pool, out=None, lse=None):
    """Shapes and dtypes of a prefill call against its plan (no device access)."""
    import torch
    if plan.mode != "prefill":
        raise ValueError("prefill needs a prefill plan")
    T, Hq, Hkv, d = plan.total_q, plan.num_heads_q, plan.num_heads_kv, plan.head_dim
    _expect(q, (T, Hq, d), "q", torch.bfloat16)
    _expect(k_chunk, (T, Hkv, d), "k_chunk", torch.bfloat16)
    _expect(v_chunk, (T, Hkv, d), "v_chunk", torch.bfloat16)
    _check_pool(plan, k_pool, v_pool)
    if out is not None or lse is not None:
        _check_outputs(plan, T, out if out is not None else q, lse if lse is not None else
                       torch.empty(T, Hq, dtype=torch.float32, device="meta"))


def check_decode_args(plan: "Plan", q, k_pool, v_pool, out=None, lse=None):
    """Shapes and dtypes of a decode call against its plan (no device access)."""
    import torch
    if plan.mode != "decode":
        raise ValueError("decode needs a decode plan")
    B, Hq, d = plan.num_seqs, plan.num_heads_q, plan.head_dim
    _expect(q, (B, Hq, d), "q", torch.bfloat16)
    _check_pool(plan, k_pool, v_pool)
    if out is not None or lse is not None:
        _check_outputs(plan, B, out if out is not None else q, lse if lse is not None else
                       torch.empty(B, Hq, dtype=torch.float32, device="meta"))


def _bf16(t, name):
    import torch
    if t is None:
        return None
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    return t


def prefill(plan: Plan, q, k_chunk, v_chunk, k_pool, v_pool, out=None, lse=None,
            scale: Optional[float] = None, stream=None):
    """MSA prefill; returns (out bf16 [Tq, Hq, d], lse fp32 [Tq, Hq])."""
    import torch
    for t, n in ((q, "q"), (k_chunk, "k_chunk"), (v_chunk, "v_chunk"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _bf16(t, n)
    check_prefill_args(plan, q, k_chunk, v_chunk, k_pool, v_pool, out, lse)
    if out is not None:
        _bf16(out, "out")
    if plan.dev is None:
        plan.upload(q.device, stream)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(plan.head_dim) if scale is None else float(scale)
    _check(lib().msa_prefill(plan.handle, _dptr(plan.dev), _dptr(q), _dptr(k_chunk), _dptr(v_chunk),
                             _dptr(k_pool), _dptr(v_pool), _dptr(out), _dptr(lse), scale,
                             _dptr(plan.ws), plan.ws.numel(), _stream(stream)), "msa_prefill")
    return out, lse


def decode(plan: Plan, q, k_pool, v_pool, out=None, lse=None, scale: Optional[float] = None, stream=None):
    """MSA decode (split-KV + LSE merge); returns (out bf16 [B, Hq, d], lse fp32 [B, Hq])."""
    import torch
    for t, n in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _bf16(t, n)
    check_decode_args(plan, q, k_pool, v_pool, out, lse)
    if out is not None:
        _bf16(out, "out")
    if plan.dev is None:
        plan.upload(q.device, stream)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    scale = 1.0 / math.sqrt(plan.head_dim) if scale is None else float(scale)
    _check(lib().msa_decode(plan.handle, _dptr(plan.dev), _dptr(q), _dptr(k_pool), _dptr(v_pool),
                            _dptr(out), _dptr(lse), scale, _dptr(plan.ws), plan.ws.numel(), _stream(stream)),
           "msa_decode")
    return out, lse


def merge_lse(o_a, lse_a, o_b, lse_b, out=None, lse=None, stream=None):
    """Merge two partial results (fp32 O [rows, H, d], fp32 LSE [rows, H]) -> bf16 O, fp32 LSE."""
    import torch
    rows, heads, d = o_a.shape
    for t in (o_a, lse_a, o_b, lse_b):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("merge_lse inputs must be contiguous fp32 CUDA tensors")
    _expect(o_b, (rows, heads, d), "o_b")
    _expect(lse_a, (rows, heads), "lse_a")
    _expect(lse_b, (rows, heads), "lse_b")
    if out is not None:
        _bf16(out, "out")
        _expect(out, (rows, heads, d), "out")
    if lse is not None:
        _expect(lse, (rows, heads), "lse", torch.float32)
    if out is None:
        out = torch.empty(rows, heads, d, dtype=torch.bfloat16, device=o_a.device)
    if lse is None:
        lse = torch.empty(rows, heads, dtype=torch.float32, device=o_a.device)
    _check(lib().msa_merge_lse(_dptr(o_a), _dptr(lse_a), _dptr(o_b), _dptr(lse_b), _dptr(out), _dptr(lse),
                               rows, heads, d, _stream(stream)), "msa_merge_lse")
    return out, lse


def gather(plan: Plan, k_chunk, v_chunk, k_pool, v_pool, out=None, stream=None):
    """KV context of every sequence in canonical (position) order: (K, V, pos).

    `out` = (k, v, pos) writes into caller buffers instead: bf16 [>= n, Hkv, d] twice and
    int32 [>= n], n = the plan's KV tokens; the first n rows are returned."""
    import torch
    _check_pool(plan, k_pool, v_pool)
    if plan.mode == "prefill" and plan.total_q > 0:
        for t, name in ((k_chunk, "k_chunk"), (v_chunk, "v_chunk")):
            _bf16(t, name)
            _expect(t, (plan.total_q, plan.num_heads_kv, plan.head_dim), name)
    n = plan.stats()["kv_tokens"]
    dev = k_pool.device
    if plan.dev is None:
        plan.upload(dev, stream)
    if out is not None:
        k, v, pos = out
        for t, name in ((k, "out k"), (v, "out v")):
            _bf16(t, name)
            if t.dim() != 3 or t.shape[0] < max(1, n) or tuple(t.shape[1:]) != (plan.num_heads_kv, plan.head_dim):
                raise ValueError(f"{name}: expected [>= {max(1, n)}, {plan.num_heads_kv}, {plan.head_dim}], "
                                 f"got {tuple(t.shape)}")
        if (pos.dtype != torch.int32 or not pos.is_cuda or not pos.is_contiguous() or pos.dim() != 1
                or pos.shape[0] < max(1, n)):
            raise ValueError(f"out pos: expected contiguous int32 CUDA [>= {max(1, n)}]")
    else:
        k = torch.empty(max(1, n), plan.num_heads_kv, plan.head_dim, dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        pos = torch.empty(max(1, n), dtype=torch.int32, device=dev)
    _check(lib().msa_gather(plan.handle, _dptr(plan.dev), _dptr(k_chunk), _dptr(v_chunk), _dptr(k_pool),
                            _dptr(v_pool), _dptr(k), _dptr(v), _dptr(pos),
                            min(k.shape[0], v.shape[0], pos.shape[0]), _stream(stream)),
           "msa_gather")
    return k[:n], v[:n], pos[:n]


def append_plan(q_pos, free_blocks, block_pos, block_fill, seq_blocks=()):
    """Placement of one sequence's chunk rows in the pool (see msa_append_plan in
    include/msa.h).  block_pos / block_fill (int32 numpy arrays) are updated in place.
    Returns (dst_slot int32 [n], new_blocks int32 [n_new])."""
    q = np.ascontiguousarray(np.asarray(q_pos, np.int32))
    fb = np.ascontiguousarray(np.asarray(free_blocks, np.int32))
    sb = np.ascontiguousarray(np.asarray(seq_blocks, np.int32))
    for a in (block_pos, block_fill):
        if a.dtype != np.int32 or not a.flags.c_contiguous:
            raise ValueError("block_pos and block_fill must be contiguous int32 arrays (updated in place)")
    dst = np.zeros(max(1, len(q)), np.int32)
    new = np.zeros(max(1, len(fb)), np.int32)
    n_new = ctypes.c_int32(0)
    _check(lib().msa_append_plan(_ptr(q), len(q), _ptr(fb), len(fb), _ptr(sb) if sb.size else None, len(sb),
                                 _ptr(block_pos), _ptr(block_fill), len(block_pos), _ptr(dst), _ptr(new),
                                 ctypes.byref(n_new)),
           "msa_append_plan")
    return dst[:len(q)], new[:n_new.value]


def kv_append(dst_slot, k_chunk, v_chunk, k_pool, v_pool, stream=None):
    """Copy chunk rows of K and V into their pool slots (device, bit-exact)."""
    import torch
    for t, n in ((k_chunk, "k_chunk"), (v_chunk, "v_chunk"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _bf16(t, n)
    if dst_slot.dtype != torch.int32 or not dst_slot.is_cuda or not dst_slot.is_contiguous():
        raise ValueError("dst_slot must be a contiguous int32 CUDA tensor")
    n, hkv, d = k_chunk.shape
    _expect(v_chunk, (n, hkv, d), "v_chunk")
    _expect(k_pool, (k_pool.shape[0], hkv, 16, d) if k_pool.dim() == 4 else (0, hkv, 16, d), "k_pool")
    _expect(v_pool, tuple(k_pool.shape), "v_pool")
    _expect(dst_slot, (n,), "dst_slot")
    _check(lib().msa_kv_append(_dptr(dst_slot), _dptr(k_chunk), _dptr(v_chunk), _dptr(k_pool), _dptr(v_pool),
                               n, hkv, d, k_pool.shape[0], _stream(stream)), "msa_kv_append")


def get_status(plan: Plan, stream=None) -> int:
    """Synchronise, read and clear the device status word of the plan's workspace."""
    return int(lib().msa_get_status(_dptr(plan.ws), _stream(stream)))


def set_wait_limit(ns: int):
    lib().msa_set_wait_limit(int(ns))


def set_test_drop(kernel: str = None, cta: int = -1, index: int = -1):
    """Test hook of the give-up path (msa_set_test_drop): later prefill or decode launches
    leave out one copy so that the wait for it runs out.  No argument turns it off."""
    k = {"prefill": 0, "decode": 1}.get(kernel, -1)
    lib().msa_set_test_drop(k, int(cta), int(index))



EVICT_POLICIES = {"cost": 0, "cost_scan": 1, "lru": 2, "prefix": 3}


class EvictionPolicy:
    """Host-side KV-block eviction policy of the library (msa_evict_* in include/msa.h):
    the cost-aware score (Eq. 5 recompute cost times a piecewise exponential reuse
    estimate, lambda from Eq. 10), or the LRU / prefix-only baselines."""

    def __init__(self, policy: str = "cost", k5: float = 3.07463e-6, k_const: float = 3.49e-5,
                 beta: float = 16.0, alpha: float = 64.0, tau0: float = 0.0, lambda0: float = 1.0,
                 window: int = 64, period: int = 16):
        opts = _EvictOpts(k5, k_const, beta, alpha, tau0, lambda0, window, period, EVICT_POLICIES[policy], 0)
        h = ctypes.c_void_p(0)
        _check(lib().msa_evict_create(ctypes.byref(opts), ctypes.byref(h)), "msa_evict_create")
        self._h = h
        self.policy = policy

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.msa_evict_destroy(h)
            self._h = None

    def insert(self, block: int, pos_block: int, now: float):
        _check(lib().msa_evict_insert(self._h, int(block), int(pos_block), float(now)), "msa_evict_insert")

    def access(self, block: int, now: float):
        _check(lib().msa_evict_access(self._h, int(block), float(now)), "msa_evict_access")

    def remove(self, block: int):
        _check(lib().msa_evict_remove(self._h, int(block)), "msa_evict_remove")

    def victim(self, now: float) -> int:
        b = ctypes.c_int32(-1)
        _check(lib().msa_evict_victim(self._h, float(now), ctypes.byref(b)), "msa_evict_victim")
        return int(b.value)

    def score(self, block: int, now: float) -> float:
        v = ctypes.c_double(0.0)
        _check(lib().msa_evict_score(self._h, int(block), float(now), ctypes.byref(v)), "msa_evict_score")
        return float(v.value)

    @property
    def lam(self) -> float:
        v = ctypes.c_double(0.0)
        _check(lib().msa_evict_get_lambda(self._h, ctypes.byref(v)), "msa_evict_get_lambda")
        return float(v.value)

    def __len__(self) -> int:
        return int(lib().msa_evict_size(self._h))

    def check(self, now: float = 0.0) -> bool:
        return lib().msa_evict_check(self._h, float(now)) == 0
