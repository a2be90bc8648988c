"""CPU oracle of the HSDP fully_shard data path with dim-0 ragged shards.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product library
(``hsdp_sharded_parameter_gb300``) never imports it, and the two share no
code: the arithmetic lives in ``hsdp_oracle.c`` (plain single-threaded C
loops); this module only marshals numpy arrays into it.

Data convention: f32 data are ``np.float32`` arrays, bf16 data are
``np.uint16`` arrays holding the raw bits. Every buffer is a flat contiguous
array. Per-(rank, param) lists are indexed ``w * P + p``.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms and the pages' worked examples, exact-arithmetic brute force,
library round-to-nearest-even, error bounds); none is parity-unpinned.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
AVG, SUM = 0, 1
OK, EINVAL, ENOTIMPL, ENOMEM = 0, 1, 2, 3

_NP = {F32: np.float32, BF16: np.uint16}
_DT = {"f32": F32, "bf16": BF16, F32: F32, BF16: BF16}
_OP = {"avg": AVG, "sum": SUM, AVG: AVG, SUM: SUM}

_lib = None
_threaded = False


class OracleError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"oracle {what} failed with status {code}")
        self.code = code


def use_threaded(threaded=True):
    """Switches this process to the -fopenmp build of the same source (the
    labelled multi-core CPU baseline; same bytes as the oracle) or back."""
    global _lib, _threaded
    if bool(threaded) != _threaded:
        _lib, _threaded = None, bool(threaded)


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        path = _build.library_path(_threaded)
        if not os.path.exists(path):
            _build.build(threaded=_threaded)
        L = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.hor_plan.argtypes = [i32, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
        L.hor_plan_bucketed.argtypes = [i32, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
        L.hor_effective_shard_size.argtypes = [i32, i32]
        L.hor_slice_numel.argtypes = [i64, i32]
        L.hor_slice_numel.restype = i64
        L.hor_group_ranks.argtypes = [i32, i32, i32, vp, vp]
        L.hor_comm_calls.argtypes = [i32, i32, vp, vp]
        L.hor_ag_copy_in.argtypes = [vp, i32, vp, i32, i64, vp]
        L.hor_ag_gather.argtypes = [vp, i32, i64, vp]
        L.hor_ag_copy_out.argtypes = [vp, i32, i64, vp, vp]
        L.hor_rs_copy_in.argtypes = [vp, i32, i64, vp, vp]
        L.hor_rs_ar_reduce.argtypes = [vp, i32, i64, vp, i64, vp]
        L.hor_rs_reduce.argtypes = [vp, i32, i64, vp, i32, i64, vp]
        L.hor_ar_reduce.argtypes = [vp, i32, i64, vp]
        L.hor_apply_grads.argtypes = [vp, vp, i32, i32, i32, vp]
        L.hor_locate_fused_many.argtypes = [vp, i64, vp, vp, vp, vp]
        L.hor_locate_gathered_many.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp]
        L.hor_fold_nested_many.argtypes = [i32, i32, i64, vp, vp]
        L.hor_f32_to_bf16_many.argtypes = [i64, vp, vp]
        L.hor_div_many.argtypes = [i64, vp, ctypes.c_float, vp]
        L.hor_f32_to_bf16.argtypes = [ctypes.c_float]
        L.hor_f32_to_bf16.restype = ctypes.c_uint16
        L.hor_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.hor_bf16_to_f32.restype = ctypes.c_float
        _lib = L
    return _lib


class _CLayout(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int), ("W", ctypes.c_int), ("S", ctypes.c_int),
                ("D", ctypes.c_int), ("d0", ctypes.c_void_p), ("inner", ctypes.c_void_p),
                ("dss", ctypes.c_void_p), ("off", ctypes.c_void_p),
                ("len", ctypes.c_void_p), ("o", ctypes.c_void_p)]


def _ptr(a):
    return a.ctypes.data


def _ptrs(arrays):
    arr = (ctypes.c_void_p * max(1, len(arrays)))()
    for i, a in enumerate(arrays):
        assert a.flags["C_CONTIGUOUS"]
        arr[i] = a.ctypes.data
    return arr


def _check(code, what):
    if code != OK:
        raise OracleError(code, what)


class Layout:
    """The oracle's plan: chunk rows, shard ranges and slice offsets."""

    def __init__(self, d0, inner, rank_size, shard_size, enable_param_shard=1, shard_dim=0,
                 bucket=None):
        L = lib()
        self.bucket = None if bucket is None else np.ascontiguousarray(bucket, dtype=np.int32)
        self.d0 = np.ascontiguousarray(d0, dtype=np.int64)
        self.inner = np.ascontiguousarray(inner, dtype=np.int64)
        self.P = len(self.d0)
        self.W = int(rank_size)
        self.S = int(L.hor_effective_shard_size(shard_size, enable_param_shard))
        S = max(self.S, 1)
        self.dss = np.zeros(max(self.P, 1), np.int64)
        self.off = np.zeros((max(self.P, 1), S), np.int64)
        self.len = np.zeros((max(self.P, 1), S), np.int64)
        self.o = np.zeros(self.P + 1, np.int64)
        code = L.hor_plan_bucketed(self.P, _ptr(self.d0), _ptr(self.inner),
                                   None if self.bucket is None else _ptr(self.bucket), self.W,
                                   shard_size, enable_param_shard, shard_dim, _ptr(self.dss),
                                   _ptr(self.off), _ptr(self.len), _ptr(self.o))
        _check(code, "plan")
        self.dss = self.dss[: self.P]
        self.off = self.off[: self.P]
        self.len = self.len[: self.P]
        self.D = self.W // self.S
        self.sum_padded = int(self.o[-1])
        self._c = _CLayout(self.P, self.W, self.S, self.D, _ptr(self.d0), _ptr(self.inner),
                           _ptr(self.dss), _ptr(self.off), _ptr(self.len), _ptr(self.o))

    @property
    def c(self):
        return ctypes.byref(self._c)

    def slice(self, dt):
        return int(lib().hor_slice_numel(self.sum_padded, _DT[dt]))

    def numel(self, p):
        return int(self.d0[p] * self.inner[p])

    def shard_numel(self, p, s):
        return int(self.len[p, s] * self.inner[p])

    def group_ranks(self, w):
        sg = np.zeros(self.S, np.int32)
        rg = np.zeros(self.D, np.int32)
        lib().hor_group_ranks(self.W, self.S, w, _ptr(sg), _ptr(rg))
        return sg, rg

    def comm_calls(self):
        rs, ar = ctypes.c_int(), ctypes.c_int()
        lib().hor_comm_calls(self.S, self.D, ctypes.byref(rs), ctypes.byref(ar))
        return rs.value, ar.value


def _alloc(n, dt, fill=None):
    a = np.zeros(n, _NP[dt])
    if fill is not None:
        a.view(np.uint8)[:] = fill
    return a


def ag_copy_in(L, shards, src_dt, dst_dt, ag_out=None):
    src_dt, dst_dt = _DT[src_dt], _DT[dst_dt]
    sl = L.slice(dst_dt)
    if ag_out is None:
        ag_out = [_alloc(L.S * sl, dst_dt, 0xFF) for _ in range(L.W)]
    _check(lib().hor_ag_copy_in(L.c, src_dt, _ptrs(shards), dst_dt, sl, _ptrs(ag_out)), "ag_copy_in")
    return ag_out


def ag_gather(L, ag_out, dt):
    dt = _DT[dt]
    _check(lib().hor_ag_gather(L.c, dt, L.slice(dt), _ptrs(ag_out)), "ag_gather")
    return ag_out


def ag_copy_out(L, ag_out, dt, full=None):
    dt = _DT[dt]
    if full is None:
        full = [_alloc(L.numel(p), dt, 0xFF) for _ in range(L.W) for p in range(L.P)]
    _check(lib().hor_ag_copy_out(L.c, dt, L.slice(dt), _ptrs(ag_out), _ptrs(full)), "ag_copy_out")
    return full


def rs_copy_in(L, grads, dt, rs_in=None):
    dt = _DT[dt]
    sl = L.slice(dt)
    if rs_in is None:
        rs_in = [_alloc(L.S * sl, dt, 0xFF) for _ in range(L.W)]
    _check(lib().hor_rs_copy_in(L.c, dt, sl, _ptrs(grads), _ptrs(rs_in)), "rs_copy_in")
    return rs_in


def rs_ar_reduce(L, rs_in, dt, fused=None):
    """Fused ReduceScatter-sum + AllReduce-sum of the reduce-scatter inputs."""
    dt = _DT[dt]
    sf = L.slice(F32)
    if fused is None:
        fused = [_alloc(sf, F32, 0xFF) for _ in range(L.W)]
    _check(lib().hor_rs_ar_reduce(L.c, dt, L.slice(dt), _ptrs(rs_in), sf, _ptrs(fused)),
           "rs_ar_reduce")
    return fused


def fused_from_grads(L, grads, dt):
    """The whole fused gradient sync from unpadded gradients: copy-in, then
    the fused reduction (the product's single-pass kernel computes this)."""
    return rs_ar_reduce(L, rs_copy_in(L, grads, dt), dt)


def rs_reduce(L, rs_in, dt, op, out=None):
    dt = _DT[dt]
    sf = L.slice(F32)
    if out is None:
        out = [_alloc(sf, F32, 0xFF) for _ in range(L.W)]
    _check(lib().hor_rs_reduce(L.c, dt, L.slice(dt), _ptrs(rs_in), _OP[op], sf, _ptrs(out)),
           "rs_reduce")
    return out


def ar_reduce(L, buf, op):
    _check(lib().hor_ar_reduce(L.c, _OP[op], L.slice(F32), _ptrs(buf)), "ar_reduce")
    return buf


def apply_grads(L, fused, op, dt, accumulate=False, shard_grads=None):
    dt = _DT[dt]
    if shard_grads is None:
        shard_grads = [_alloc(L.shard_numel(p, w % L.S), dt, 0xFF)
                       for w in range(L.W) for p in range(L.P)]
    _check(lib().hor_apply_grads(L.c, _ptrs(fused), _OP[op], dt, int(bool(accumulate)),
                                 _ptrs(shard_grads)), "apply_grads")
    return shard_grads


def locate_fused(L, s, j):
    s = np.ascontiguousarray(s, np.int32)
    j = np.ascontiguousarray(j, np.int64)
    p = np.zeros(len(s), np.int32)
    e = np.zeros(len(s), np.int64)
    lib().hor_locate_fused_many(L.c, len(s), _ptr(s), _ptr(j), _ptr(p), _ptr(e))
    return p, e


def locate_gathered(L, dt, p, e):
    p = np.ascontiguousarray(p, np.int32)
    e = np.ascontiguousarray(e, np.int64)
    shard = np.zeros(len(p), np.int32)
    k = np.zeros(len(p), np.int64)
    idx = np.zeros(len(p), np.int64)
    lib().hor_locate_gathered_many(L.c, L.slice(_DT[dt]), len(p), _ptr(p), _ptr(e),
                                   _ptr(shard), _ptr(k), _ptr(idx))
    return shard, k, idx


def fold_nested(S, D, vals):
    vals = np.ascontiguousarray(vals, np.float32)
    n = vals.shape[0]
    assert vals.shape[1] == S * D
    out = np.zeros(n, np.float32)
    lib().hor_fold_nested_many(S, D, n, _ptr(vals), _ptr(out))
    return out


def f32_to_bf16(x):
    x = np.ascontiguousarray(x, np.float32)
    out = np.zeros(x.shape, np.uint16)
    lib().hor_f32_to_bf16_many(x.size, _ptr(x), _ptr(out))
    return out


def bf16_to_f32(h):
    h = np.ascontiguousarray(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def div(x, d):
    x = np.ascontiguousarray(x, np.float32)
    out = np.zeros(x.shape, np.float32)
    lib().hor_div_many(x.size, _ptr(x), float(d), _ptr(out))
    return out
