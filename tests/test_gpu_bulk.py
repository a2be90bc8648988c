"""GPU parity of the fused gradient sync on a capped grid, where one block per
SM splits into a producer warp issuing TMA bulk loads into a shared-memory
ring and eight warps folding from it, and the failure detection of its
bounded waits (the plan's status word).

Every fused region and every shard gradient is compared byte for byte with
the CPU oracle; guard bands around every buffer must stay untouched."""
import time

import numpy as np
import pytest
import torch

import oracle as O
from hsdp_sharded_parameter_gb300 import capi as C

from gpu_util import GuardedAlloc, dirty, fill_, make, same_bits, to_np

pytestmark = pytest.mark.gpu


class SkewedAlloc(GuardedAlloc):
    """Each gradient tensor starts at its own element offset (0 .. 7 elements
    past a 16-byte boundary), so the sources of one run are shifted
    differently against each other and against the fused rows."""

    def __init__(self):
        super().__init__()
        self.k = 0

    def __call__(self, numel, dt, dev, role=None):
        es = 4 if dt == "f32" else 2
        if role == "grads":
            self.offsets = {"grads": es * (self.k % (16 // es))}
            self.k += 1
        else:
            self.offsets = {}
        return super().__call__(numel, dt, dev, role)


def check_sync(plan, L, unit, alloc, cap, seed, ops=("avg", "sum")):
    """Fused reduce, then the one-pass sync (each op, then accumulating), on
    a grid capped at `cap` blocks, against the oracle."""
    gdt = unit.grad_dt
    fill_(unit.grads, seed, 1.0, gdt)
    grads = [to_np(t) for t in unit.grads]
    ref_fused = O.rs_ar_reduce(L, O.rs_copy_in(L, grads, gdt), gdt)
    plan.set_grid_limit(cap)
    dirty(unit.fused)
    unit.rs_ar_reduce()
    torch.cuda.synchronize()
    for g, r in zip(unit.fused, ref_fused):
        assert same_bits(to_np(g), r), ("rs_ar_reduce", cap)
    for op in ops:
        dirty(unit.fused)
        dirty(unit.shard_grads)
        unit.reduce_grads_one_pass(op)
        ref = O.apply_grads(L, ref_fused, op, gdt)
        torch.cuda.synchronize()
        for g, r in zip(unit.fused, ref_fused):
            assert same_bits(to_np(g), r), ("one pass, fused", op, cap)
        for g, r in zip(unit.shard_grads, ref):
            assert same_bits(to_np(g), r), ("one pass, shard grads", op, cap)
    before = [to_np(t) for t in unit.shard_grads]
    unit.reduce_grads_one_pass("avg", accumulate=True)
    ref = O.apply_grads(L, ref_fused, "avg", gdt, accumulate=True, shard_grads=[b.copy() for b in before])
    torch.cuda.synchronize()
    for g, r in zip(unit.shard_grads, ref):
        assert same_bits(to_np(g), r), ("one pass, accumulate", cap)
    assert plan.status() == 0
    plan.set_grid_limit(0)
    alloc.check_guards()


# (W, S): the compiled shapes of the bulk-fed reduce, the generic one, and a
# 24-source mesh with a two-stage ring. Ragged parameters: zero-length
# shards, padding rows, runs shifted against the fused rows (odd-sized
# vectors), runs much longer than a chunk.
SHAPES = [(16, 8), (8, 4), (8, 8), (8, 1), (12, 3), (24, 8)]


@pytest.mark.parametrize("cap", [1, 5, 64])
@pytest.mark.parametrize("W,S", SHAPES)
def test_capped_sync_matches_oracle(W, S, cap):
    plan, L, unit, alloc = make(S, W // S, [1500, 7, 4099, 33, 3], [17, 16, 1, 64, 5], "bf16", "bf16")
    check_sync(plan, L, unit, alloc, cap, seed=W * 10 + S + cap)


@pytest.mark.parametrize("grad_dt", ["bf16", "f32"])
def test_capped_sync_skewed_sources(grad_dt):
    # every source of a run at its own 16-byte phase
    d0, inner, S, D = [900, 5, 2049, 11], [9, 64, 1, 3], 4, 2
    plan = C.Plan(d0, inner, S * D, S).upload()
    L = O.Layout(d0, inner, S * D, S)
    alloc = SkewedAlloc()
    from hsdp_sharded_parameter_gb300.runtime import HsdpUnit
    unit = HsdpUnit(plan, grad_dt, grad_dt, alloc=alloc)
    check_sync(plan, L, unit, alloc, 7, seed=31)


def test_capped_sync_tiny_fp32_workload():
    # the tiny fsdp workload: fp32 gradients, four ranks in one shard group
    plan, L, unit, alloc = make(4, 1, [7, 16, 5, 3], [8, 8, 1, 4], "f32", "f32")
    check_sync(plan, L, unit, alloc, 3, seed=5)


def test_capped_sync_unaligned_fused_rows():
    # fused rows off the 16-byte grid: every granule element by element
    plan, L, unit, alloc = make(4, 2, [300, 7, 129], [16, 1, 64], "bf16", "bf16",
                                offsets={"fused": 4, "shard_grads": 2})
    check_sync(plan, L, unit, alloc, 6, seed=9)


def test_capped_sync_many_runs():
    # more than 1024 runs: the producer's lookups use the tile -> run map
    rng = np.random.default_rng(12)
    d0 = [int(x) for x in rng.integers(0, 9, 900)]
    inner = [int(x) for x in rng.choice([1, 8, 40, 300], 900)]
    plan, L, unit, alloc = make(2, 2, d0, inner, "bf16", "bf16")
    check_sync(plan, L, unit, alloc, 9, seed=12, ops=("avg",))


def test_capped_sync_32_sources_falls_back():
    # 32 bf16 sources leave no room for two stages: the per-warp cp.async
    # reduce takes the call, with the same bytes
    plan, L, unit, alloc = make(16, 2, [70, 3, 129], [5, 16, 1], "bf16", "bf16")
    check_sync(plan, L, unit, alloc, 4, seed=32, ops=("avg",))


def test_wait_limit_reports_through_status():
    # The test hook withholds block 0's first chunk: its consumers' wait runs
    # out after the 20 ms limit, the block records it in the plan's status
    # word and leaves; the call returns, the context stays usable, and the
    # next call without the hook gives the oracle's bytes and a clear status.
    plan, L, unit, alloc = make(4, 2, [300, 7, 129], [16, 1, 64], "bf16", "bf16")
    gdt = unit.grad_dt
    fill_(unit.grads, 41, 1.0, gdt)
    grads = [to_np(t) for t in unit.grads]
    ref_fused = O.rs_ar_reduce(L, O.rs_copy_in(L, grads, gdt), gdt)
    plan.set_grid_limit(4).set_wait_limit(20_000_000)
    assert plan.status() == 0
    for one_pass in (False, True):
        plan.inject_stall(True)
        t0 = time.monotonic()
        if one_pass:
            unit.reduce_grads_one_pass("avg")
        else:
            unit.rs_ar_reduce()
        st = plan.status()
        elapsed = time.monotonic() - t0
        assert st & C.FSDP_STATUS_CONSUMER_WAIT, st
        assert elapsed < 20.0
        assert plan.status() == 0  # reading clears it
        plan.inject_stall(False)
        dirty(unit.fused)
        dirty(unit.shard_grads)
        if one_pass:
            unit.reduce_grads_one_pass("avg")
        else:
            unit.rs_ar_reduce()
        assert plan.status() == 0
        for g, r in zip(unit.fused, ref_fused):
            assert same_bits(to_np(g), r)
        if one_pass:
            for g, r in zip(unit.shard_grads, O.apply_grads(L, ref_fused, "avg", gdt)):
                assert same_bits(to_np(g), r)
    plan.set_grid_limit(0)
    alloc.check_guards()
