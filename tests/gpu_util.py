"""Helpers of the GPU parity tests: guarded allocation, host copies, fills and
the comparison of every output of the C-ABI path with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from hsdp_sharded_parameter_gb300 import capi as C
from hsdp_sharded_parameter_gb300 import workloads as WL
from hsdp_sharded_parameter_gb300.runtime import TORCH_DT, HsdpUnit

GUARD = 4096
CANARY = 0xA5
DIRTY = 0xFF  # every output is pre-filled with this byte (a NaN pattern)

OUTPUT_ROLES = {"ag_output", "full_params", "fused", "shard_grads", "rs_input"}


class GuardedAlloc:
    """Allocates every buffer inside a larger byte buffer with a 4 KiB canary
    band on both sides. ``offsets`` maps a role to a byte offset added to the
    buffer start (element aligned, to exercise unaligned paths)."""

    def __init__(self, offsets=None):
        self.offsets = offsets or {}
        self.bufs = []

    def __call__(self, numel, dt, dev, role=None):
        es = 4 if dt == "f32" else 2
        nbytes = int(numel) * es
        off = self.offsets.get(role, 0)
        raw = torch.full((nbytes + 2 * GUARD + 16,), CANARY, dtype=torch.uint8, device=dev)
        start = GUARD + off
        raw[start:start + nbytes] = DIRTY
        t = raw[start:start + nbytes].view(TORCH_DT[dt])
        self.bufs.append((raw, start, nbytes))
        return t

    def check_guards(self):
        for raw, start, nbytes in self.bufs:
            assert bool((raw[:start] == CANARY).all()), "canary before a buffer was overwritten"
            assert bool((raw[start + nbytes:] == CANARY).all()), "canary after a buffer was overwritten"


def to_np(t):
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def dirty(tensors):
    for t in tensors:
        if t.numel():
            t.view(torch.uint8).fill_(DIRTY)


def fill_(tensors, seed, std, dt):
    """Fill device tensors in place with the seeded generator's values."""
    WL.torch_fill_(tensors, seed, std, dt)


def fill_special_(tensors, seed, dt):
    """Values that stress the arithmetic: subnormals, signed zeros, huge
    magnitudes that overflow when summed, exact rounding ties."""
    rng = np.random.default_rng(seed)
    for t in tensors:
        n = t.numel()
        if n == 0:
            continue
        choice = rng.integers(0, 6, n)
        x = rng.standard_normal(n).astype(np.float32)
        x[choice == 1] = np.float32(1e-39) * rng.standard_normal((choice == 1).sum()).astype(np.float32)
        x[choice == 2] = np.where(rng.random((choice == 2).sum()) < 0.5, 0.0, -0.0).astype(np.float32)
        x[choice == 3] = np.float32(3.0e38) * np.sign(rng.standard_normal((choice == 3).sum())).astype(np.float32)
        x[choice == 4] = (1.0 + 2.0 ** -8) * rng.integers(-4, 5, (choice == 4).sum()).astype(np.float32)
        if dt == "bf16":
            b = (x.view(np.uint32) >> 16).astype(np.uint16)
            t.copy_(torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(t.device))
        else:
            t.copy_(torch.from_numpy(x).to(t.device))


def same_bits(a, b):
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def same_values(a, b, dt):
    """Bit equality, except that NaN matches any NaN (the bit pattern of a
    NaN produced by arithmetic differs between CPU and GPU)."""
    if a.shape != b.shape:
        return False
    fa = O.bf16_to_f32(a) if dt == "bf16" else a
    fb = O.bf16_to_f32(b) if dt == "bf16" else b
    na, nb = np.isnan(fa), np.isnan(fb)
    return np.array_equal(na, nb) and np.array_equal(a[~na].view(np.uint8), b[~nb].view(np.uint8))


def make(S, D, d0, inner, param_dt="bf16", grad_dt="bf16", ag_dt=None, offsets=None, **plan_kw):
    """A unit over guarded buffers and the oracle's layout of the same plan
    (plan_kw: enable_param_shard, bucket)."""
    plan = C.Plan(d0, inner, S * D, S, **plan_kw).upload()
    L = O.Layout(d0, inner, S * D, S, **plan_kw)
    alloc = GuardedAlloc(offsets)
    unit = HsdpUnit(plan, param_dt, grad_dt, ag_dt, with_unfused=True, alloc=alloc)
    return plan, L, unit, alloc


def check_every_step(L, unit, alloc, seed=0, special=False, ops=("avg", "sum")):
    """Runs every C-ABI call on the unit and compares every output buffer,
    byte for byte (padding and untouched regions included), with the oracle
    run on the same inputs. Returns the number of buffers compared."""
    pdt, gdt, adt = unit.param_dt, unit.grad_dt, unit.ag_dt
    if special:
        fill_special_(unit.shards, seed + 1, pdt)
        fill_special_(unit.grads, seed + 2, gdt)
    else:
        fill_(unit.shards, seed + 1, 1.0, pdt)
        fill_(unit.grads, seed + 2, 1.0, gdt)
    shards = [to_np(t) for t in unit.shards]
    grads = [to_np(t) for t in unit.grads]
    n = 0
    cmp = same_values if special else (lambda a, b, dt: same_bits(a, b))

    # forward, unfused: copy-in (own slices only), gather, copy-out
    dirty(unit.ag_out)
    unit.ag_copy_in(fuse_gather=False)
    ref_ag = O.ag_copy_in(L, shards, pdt, adt)
    torch.cuda.synchronize()
    for g, r in zip(unit.ag_out, ref_ag):
        assert cmp(to_np(g), r, adt), "ag_copy_in"
        n += 1
    unit.ag_gather()
    O.ag_gather(L, ref_ag, adt)
    torch.cuda.synchronize()
    for g, r in zip(unit.ag_out, ref_ag):
        assert cmp(to_np(g), r, adt), "ag_gather"
        n += 1
    dirty(unit.full)
    unit.ag_copy_out()
    ref_full = O.ag_copy_out(L, ref_ag, adt)
    torch.cuda.synchronize()
    for g, r in zip(unit.full, ref_full):
        assert cmp(to_np(g), r, adt), "ag_copy_out"
        n += 1
    # forward in one pass, straight from the shards
    dirty(unit.full)
    unit.unshard_direct()
    torch.cuda.synchronize()
    for g, r in zip(unit.full, ref_full):
        assert cmp(to_np(g), r, adt), "ag_unshard"
        n += 1
    # forward, fused copy-in + gather on a dirty buffer
    dirty(unit.ag_out)
    unit.ag_copy_in(fuse_gather=True)
    torch.cuda.synchronize()
    for g, r in zip(unit.ag_out, ref_ag):
        assert cmp(to_np(g), r, adt), "ag_copy_in fused with gather"
        n += 1

    # backward, fused
    dirty(unit.fused)
    unit.rs_ar_reduce()
    ref_rs_in = O.rs_copy_in(L, grads, gdt)
    ref_fused = O.rs_ar_reduce(L, ref_rs_in, gdt)
    torch.cuda.synchronize()
    for g, r in zip(unit.fused, ref_fused):
        assert cmp(to_np(g), r, "f32"), "rs_ar_reduce"
        n += 1
    for op in ops:
        dirty(unit.shard_grads)
        unit.apply_grads(op)
        ref = O.apply_grads(L, ref_fused, op, gdt)
        torch.cuda.synchronize()
        for g, r in zip(unit.shard_grads, ref):
            assert cmp(to_np(g), r, gdt), f"apply_grads {op}"
            n += 1
    # accumulation on top of the last result
    before = [to_np(t) for t in unit.shard_grads]
    unit.apply_grads("avg", accumulate=True)
    ref = O.apply_grads(L, ref_fused, "avg", gdt, accumulate=True, shard_grads=[b.copy() for b in before])
    torch.cuda.synchronize()
    for g, r in zip(unit.shard_grads, ref):
        assert cmp(to_np(g), r, gdt), "apply_grads accumulate"
        n += 1

    # backward in one pass: the fused reduce with the apply folded in (the
    # same fused regions and shard gradients), fresh and accumulating
    for op in ops:
        dirty(unit.fused)
        dirty(unit.shard_grads)
        unit.reduce_grads_one_pass(op)
        ref = O.apply_grads(L, ref_fused, op, gdt)
        torch.cuda.synchronize()
        for g, r in zip(unit.fused, ref_fused):
            assert cmp(to_np(g), r, "f32"), f"rs_ar_reduce_apply fused {op}"
            n += 1
        for g, r in zip(unit.shard_grads, ref):
            assert cmp(to_np(g), r, gdt), f"rs_ar_reduce_apply shard grads {op}"
            n += 1
    before = [to_np(t) for t in unit.shard_grads]
    unit.reduce_grads_one_pass("sum", accumulate=True)
    ref = O.apply_grads(L, ref_fused, "sum", gdt, accumulate=True, shard_grads=[b.copy() for b in before])
    torch.cuda.synchronize()
    for g, r in zip(unit.shard_grads, ref):
        assert cmp(to_np(g), r, gdt), "rs_ar_reduce_apply accumulate"
        n += 1

    # backward, unfused: RS copy-in, RS, AR, apply
    dirty(unit.rs_in)
    C.fsdp_rs_copy_in(unit.plan, unit.b_grads, unit.b_rs_in)
    torch.cuda.synchronize()
    for g, r in zip(unit.rs_in, ref_rs_in):
        assert cmp(to_np(g), r, gdt), "rs_copy_in"
        n += 1
    for op in ops:
        dirty(unit.fused)
        C.fsdp_rs_reduce(unit.plan, unit.b_rs_in, op, unit.b_fused)
        ref_buf = O.rs_reduce(L, ref_rs_in, gdt, op)
        torch.cuda.synchronize()
        for g, r in zip(unit.fused, ref_buf):
            assert cmp(to_np(g), r, "f32"), f"rs_reduce {op}"
            n += 1
        C.fsdp_ar_reduce(unit.plan, unit.b_fused, op)
        O.ar_reduce(L, ref_buf, op)
        torch.cuda.synchronize()
        for g, r in zip(unit.fused, ref_buf):
            assert cmp(to_np(g), r, "f32"), f"ar_reduce {op}"
            n += 1
    torch.cuda.synchronize()
    alloc.check_guards()
    return n
