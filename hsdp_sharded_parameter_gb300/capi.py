"""Thin Python binding of the C-ABI library (include/hsdp_fsdp.h).

Argument marshalling only: every step of the data path runs in the
library's CUDA kernels. Functions keep the C names; ``Plan`` and
``Binding`` own the C handles. Tensors are passed as device pointers
(``data_ptr()``); streams as ``torch.cuda.Stream`` or raw handles.

The library must have been built (``python -m hsdp_sharded_parameter_gb300.build``
or ``__graft_entry__.build()``): there is no fallback of any kind, a missing
library raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from .build import library_path

FSDP_OK, FSDP_ERR_INVALID_ARG, FSDP_ERR_NOT_IMPLEMENTED, FSDP_ERR_CUDA, FSDP_ERR_NOMEM = range(5)
FSDP_F32, FSDP_BF16 = 0, 1
FSDP_AVG, FSDP_SUM = 0, 1
FSDP_STATUS_PRODUCER_WAIT, FSDP_STATUS_CONSUMER_WAIT, FSDP_STATUS_ORDER = 1, 2, 4
(FSDP_ROLE_SHARDS, FSDP_ROLE_AG_OUTPUT, FSDP_ROLE_FULL_PARAMS, FSDP_ROLE_GRADS,
 FSDP_ROLE_RS_INPUT, FSDP_ROLE_FUSED, FSDP_ROLE_SHARD_GRADS) = range(7)

ROLES = {"shards": FSDP_ROLE_SHARDS, "ag_output": FSDP_ROLE_AG_OUTPUT,
         "full_params": FSDP_ROLE_FULL_PARAMS, "grads": FSDP_ROLE_GRADS,
         "rs_input": FSDP_ROLE_RS_INPUT, "fused": FSDP_ROLE_FUSED,
         "shard_grads": FSDP_ROLE_SHARD_GRADS}
DTYPES = {"f32": FSDP_F32, "bf16": FSDP_BF16}
# roles that take one buffer per (rank, parameter); the others one per rank
PER_PARAM_ROLES = {FSDP_ROLE_SHARDS, FSDP_ROLE_FULL_PARAMS, FSDP_ROLE_GRADS, FSDP_ROLE_SHARD_GRADS}
OPS = {"avg": FSDP_AVG, "sum": FSDP_SUM}

_lib = None


class FsdpError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"[status {code}] {msg}")
        self.code = code


def header_symbols():
    """Names of the functions include/hsdp_fsdp.h declares."""
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                       "hsdp_fsdp.h")
    text = open(hdr).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fsdp_[a-z0-9_]+)\s*\(", text)))


def lib():
    """The loaded C-ABI library. Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing "
                               "(run __graft_entry__.build())")
        L = ctypes.CDLL(path)
        i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        P = ctypes.POINTER
        L.fsdp_last_error.restype = ctypes.c_char_p
        L.fsdp_launch_count.restype = ctypes.c_uint64
        L.fsdp_plan_create.argtypes = [i32, vp, vp, i32, i32, i32, i32, P(vp)]
        L.fsdp_plan_create_bucketed.argtypes = [i32, vp, vp, vp, i32, i32, i32, i32, P(vp)]
        L.fsdp_plan_destroy.argtypes = [vp]
        L.fsdp_plan_upload.argtypes = [vp]
        L.fsdp_plan_set_grid_limit.argtypes = [vp, i32]
        L.fsdp_plan_set_wait_limit.argtypes = [vp, ctypes.c_uint64]
        L.fsdp_plan_inject_stall.argtypes = [vp, i32]
        L.fsdp_plan_status.argtypes = [vp, vp, P(i32)]
        L.fsdp_plan_check_tables.argtypes = [vp]
        L.fsdp_plan_info.argtypes = [vp, P(i32), P(i32), P(i32), P(i32), P(i64)]
        L.fsdp_slice_numel.argtypes = [vp, i32, P(i64)]
        L.fsdp_sharded_size.argtypes = [vp, i32, i32, P(i64), P(i64)]
        L.fsdp_padded_sharded_param_size.argtypes = [vp, i32, P(i64)]
        L.fsdp_offsets.argtypes = [vp, vp]
        L.fsdp_group_ranks.argtypes = [vp, i32, vp, vp]
        L.fsdp_comm_calls.argtypes = [vp, P(i32), P(i32)]
        L.fsdp_bind.argtypes = [vp, i32, i32, vp, vp, P(vp)]
        L.fsdp_binding_destroy.argtypes = [vp]
        L.fsdp_ag_copy_in.argtypes = [vp, vp, vp, i32, vp]
        L.fsdp_ag_gather.argtypes = [vp, vp, vp]
        L.fsdp_ag_copy_out.argtypes = [vp, vp, vp, vp]
        L.fsdp_rs_copy_in.argtypes = [vp, vp, vp, vp]
        L.fsdp_rs_ar_reduce.argtypes = [vp, vp, vp, vp]
        L.fsdp_apply_grads.argtypes = [vp, vp, i32, i32, vp, vp]
        L.fsdp_rs_reduce.argtypes = [vp, vp, i32, vp, vp]
        L.fsdp_rs_ar_reduce_apply.argtypes = [vp, vp, vp, i32, i32, vp, vp]
        L.fsdp_ar_reduce.argtypes = [vp, vp, i32, vp]
        L.fsdp_rs_ar_reduce_noalloc.argtypes = [vp, i32, vp, vp, vp]
        L.fsdp_ag_unshard.argtypes = [vp, vp, vp, vp]
        _lib = L
    return _lib


def _check(code):
    if code != FSDP_OK:
        raise FsdpError(code, lib().fsdp_last_error().decode())


def _stream(stream):
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return 0
    return getattr(stream, "cuda_stream", stream)


def fsdp_launch_count():
    return int(lib().fsdp_launch_count())


class Plan:
    """Owns an fsdp_plan_t. Host-only until ``upload()``."""

    def __init__(self, dim0, inner, rank_size, shard_size, enable_param_shard=1, shard_dim=0,
                 bucket=None):
        import numpy as np

        self._d0 = np.ascontiguousarray(dim0, dtype=np.int64)
        self._inner = np.ascontiguousarray(inner, dtype=np.int64)
        self._bucket = None if bucket is None else np.ascontiguousarray(bucket, dtype=np.int32)
        h = ctypes.c_void_p()
        _check(lib().fsdp_plan_create_bucketed(
            len(self._d0), self._d0.ctypes.data, self._inner.ctypes.data,
            None if self._bucket is None else self._bucket.ctypes.data,
            rank_size, shard_size, enable_param_shard, shard_dim, ctypes.byref(h)))
        self.handle = h
        W, S, D, P = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        sp = ctypes.c_int64()
        _check(lib().fsdp_plan_info(h, ctypes.byref(W), ctypes.byref(S), ctypes.byref(D),
                                    ctypes.byref(P), ctypes.byref(sp)))
        self.W, self.S, self.D, self.P, self.sum_padded = W.value, S.value, D.value, P.value, sp.value

    def close(self):
        if getattr(self, "handle", None):
            lib().fsdp_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def upload(self):
        _check(lib().fsdp_plan_upload(self.handle))
        return self

    def check_tables(self):
        """Host-side bounds and coverage check of the plan's work tables
        (no GPU needed); raises FsdpError naming the first violation."""
        _check(lib().fsdp_plan_check_tables(self.handle))
        return self

    def set_grid_limit(self, max_blocks):
        _check(lib().fsdp_plan_set_grid_limit(self.handle, int(max_blocks)))
        return self

    def set_wait_limit(self, nanoseconds):
        _check(lib().fsdp_plan_set_wait_limit(self.handle, int(nanoseconds)))
        return self

    def inject_stall(self, on=True):
        _check(lib().fsdp_plan_inject_stall(self.handle, int(bool(on))))
        return self

    def status(self, stream=None):
        """The plan's status word after the calls enqueued on `stream` (the
        stream is synchronised; the word is cleared): 0, or the
        FSDP_STATUS_* bits of waits that ran out."""
        v = ctypes.c_int(0)
        _check(lib().fsdp_plan_status(self.handle, _stream(stream), ctypes.byref(v)))
        return v.value

    def slice_numel(self, dt):
        out = ctypes.c_int64()
        _check(lib().fsdp_slice_numel(self.handle, DTYPES.get(dt, dt), ctypes.byref(out)))
        return out.value

    def sharded_size(self, p, s):
        a, n = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().fsdp_sharded_size(self.handle, p, s, ctypes.byref(a), ctypes.byref(n)))
        return a.value, n.value

    def padded_sharded_param_size(self, p):
        c = ctypes.c_int64()
        _check(lib().fsdp_padded_sharded_param_size(self.handle, p, ctypes.byref(c)))
        return c.value

    def offsets(self):
        import numpy as np

        o = np.zeros(self.P + 1, np.int64)
        _check(lib().fsdp_offsets(self.handle, o.ctypes.data))
        return o

    def group_ranks(self, w):
        import numpy as np

        sg = np.zeros(self.S, np.int32)
        rg = np.zeros(self.D, np.int32)
        _check(lib().fsdp_group_ranks(self.handle, w, sg.ctypes.data, rg.ctypes.data))
        return sg, rg

    def comm_calls(self):
        rs, ar = ctypes.c_int(), ctypes.c_int()
        _check(lib().fsdp_comm_calls(self.handle, ctypes.byref(rs), ctypes.byref(ar)))
        return rs.value, ar.value

    # sizes the caller allocates
    def shard_numel(self, p, s):
        _, n = self.sharded_size(p, s)
        return n * int(self._inner[p])

    def numel(self, p):
        return int(self._d0[p] * self._inner[p])

    def bind(self, role, dt, tensors, check_sizes=True):
        return Binding(self, role, dt, tensors, check_sizes)


def _torch_dtype(dt):
    import torch

    return {FSDP_F32: torch.float32, FSDP_BF16: torch.bfloat16}.get(DTYPES.get(dt, dt))


def _check_tensors(what, tensors, count, dt, numel_of=None):
    """Host-side checks before a pointer array goes to the library, which
    reads exactly `count` entries: the count, then (when dt is given) each
    tensor's dtype, device and contiguity, and (numel_of(i)) its size."""
    if len(tensors) != count:
        raise FsdpError(FSDP_ERR_INVALID_ARG, f"{what}: {len(tensors)} tensors given, the plan needs {count}")
    if dt is None:
        return
    want = _torch_dtype(dt)
    for i, t in enumerate(tensors):
        if t.dtype != want or not t.is_cuda or not t.is_contiguous():
            raise FsdpError(FSDP_ERR_INVALID_ARG,
                            f"{what}: tensor {i} is {t.dtype} on {t.device}"
                            f"{'' if t.is_contiguous() else ', not contiguous'}; expected contiguous {want} on a GPU")
        if numel_of is not None and t.numel() < numel_of(i):
            raise FsdpError(FSDP_ERR_INVALID_ARG,
                            f"{what}: tensor {i} holds {t.numel()} elements, needs {numel_of(i)}")


class Binding:
    """Owns an fsdp_binding_t: a device table of the tensors' pointers.
    Keeps the tensors alive while the binding lives. The number of tensors
    is always checked (the library reads W*P or W pointers); with
    check_sizes (the default) their dtypes and sizes are checked too, the
    sizes again by the library."""

    def __init__(self, plan, role, dt, tensors, check_sizes=True):
        r = ROLES.get(role, role)
        _check_tensors(f"bind {role}", tensors, plan.W * plan.P if r in PER_PARAM_ROLES else plan.W,
                       dt if check_sizes else None)
        n = len(tensors)
        ptrs = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in tensors])
        numels = (ctypes.c_int64 * max(n, 1))(*[t.numel() for t in tensors])
        h = ctypes.c_void_p()
        _check(lib().fsdp_bind(plan.handle, ROLES.get(role, role), DTYPES.get(dt, dt), ptrs,
                               numels if check_sizes else None, ctypes.byref(h)))
        self.handle = h
        self.plan = plan
        self.tensors = list(tensors)

    def close(self):
        if getattr(self, "handle", None):
            lib().fsdp_binding_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fsdp_ag_copy_in(plan, shards, ag_out, fuse_gather=False, stream=None):
    _check(lib().fsdp_ag_copy_in(plan.handle, shards.handle, ag_out.handle, int(bool(fuse_gather)),
                                 _stream(stream)))


def fsdp_ag_gather(plan, ag_out, stream=None):
    _check(lib().fsdp_ag_gather(plan.handle, ag_out.handle, _stream(stream)))


def fsdp_ag_copy_out(plan, ag_out, full_params, stream=None):
    _check(lib().fsdp_ag_copy_out(plan.handle, ag_out.handle, full_params.handle, _stream(stream)))


def fsdp_ag_unshard(plan, shards, full_params, stream=None):
    _check(lib().fsdp_ag_unshard(plan.handle, shards.handle, full_params.handle, _stream(stream)))


def fsdp_rs_copy_in(plan, grads, rs_in, stream=None):
    _check(lib().fsdp_rs_copy_in(plan.handle, grads.handle, rs_in.handle, _stream(stream)))


def fsdp_rs_ar_reduce(plan, grads, fused, stream=None):
    _check(lib().fsdp_rs_ar_reduce(plan.handle, grads.handle, fused.handle, _stream(stream)))


def fsdp_apply_grads(plan, fused, op, shard_grads, accumulate=False, stream=None):
    _check(lib().fsdp_apply_grads(plan.handle, fused.handle, OPS.get(op, op), int(bool(accumulate)),
                                  shard_grads.handle, _stream(stream)))


def fsdp_rs_ar_reduce_apply(plan, grads, fused, op, shard_grads, accumulate=False, stream=None):
    _check(lib().fsdp_rs_ar_reduce_apply(plan.handle, grads.handle, fused.handle, OPS.get(op, op),
                                         int(bool(accumulate)), shard_grads.handle, _stream(stream)))


def fsdp_rs_reduce(plan, rs_in, op, fused, stream=None):
    _check(lib().fsdp_rs_reduce(plan.handle, rs_in.handle, OPS.get(op, op), fused.handle,
                                _stream(stream)))


def fsdp_ar_reduce(plan, fused, op, stream=None):
    _check(lib().fsdp_ar_reduce(plan.handle, fused.handle, OPS.get(op, op), _stream(stream)))


def fsdp_rs_ar_reduce_noalloc(plan, grad_dt, grads, fused, stream=None):
    """The fused gradient sync without any device allocation by the library
    (for callers that cannot allocate device memory): ``plan`` needs no
    upload, ``grads`` (W*P tensors) and ``fused`` (W fp32 tensors) are passed
    as pointer arrays on every call. The library cannot see the tensors'
    sizes here, so their count, dtype and size are checked before the call."""
    P = plan.P
    # both counts first (the library reads both arrays), then each tensor
    _check_tensors("rs_ar_reduce_noalloc grads", grads, plan.W * P, None)
    _check_tensors("rs_ar_reduce_noalloc fused", fused, plan.W, None)
    _check_tensors("rs_ar_reduce_noalloc grads", grads, plan.W * P, grad_dt, lambda i: plan.numel(i % P))
    sf = plan.slice_numel("f32")
    _check_tensors("rs_ar_reduce_noalloc fused", fused, plan.W, "f32", lambda i: sf)
    g = (ctypes.c_void_p * max(len(grads), 1))(*[t.data_ptr() for t in grads])
    f = (ctypes.c_void_p * max(len(fused), 1))(*[t.data_ptr() for t in fused])
    _check(lib().fsdp_rs_ar_reduce_noalloc(plan.handle, DTYPES.get(grad_dt, grad_dt), g, f,
                                           _stream(stream)))
