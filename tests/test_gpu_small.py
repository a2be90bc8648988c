"""GPU parity on small plans: every output buffer of every C-ABI call equals
the CPU oracle byte for byte, padding and untouched regions included; guard
bands around every buffer stay intact."""
import numpy as np
import pytest
import torch

import oracle as O
from hsdp_sharded_parameter_gb300 import capi as C
from hsdp_sharded_parameter_gb300 import workloads as WL
from hsdp_sharded_parameter_gb300.runtime import HsdpUnit

from gpu_util import GuardedAlloc, check_every_step, make, to_np, fill_

pytestmark = pytest.mark.gpu


def test_tiny_workload_every_step():
    wl = WL.WORKLOADS["tiny_fsdp"]
    plan, L, unit, alloc = make(4, 1, wl.d0, wl.inner, "f32", "f32")
    assert check_every_step(L, unit, alloc, seed=wl.seed_params) > 30


def test_tiny_workload_with_bf16_gather_cast():
    # all-gather copy-in with cast f32 -> bf16 ("Hyper通信掩盖方案" PR #758 §二.1)
    wl = WL.WORKLOADS["tiny_fsdp"]
    plan, L, unit, alloc = make(4, 1, wl.d0, wl.inner, "f32", "f32", ag_dt="bf16")
    check_every_step(L, unit, alloc, seed=7)


def random_plan(seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 10))
    D = int(rng.integers(1, 5))
    P = int(rng.integers(1, 9))
    d0 = [int(x) for x in rng.integers(0, 41, P)]
    inner = [int(x) for x in rng.choice([1, 1, 2, 3, 5, 8, 16, 17, 64], P)]
    pdt, gdt, adt = [("bf16", "bf16", "bf16"), ("f32", "f32", "f32"), ("f32", "bf16", "bf16"),
                     ("f32", "f32", "bf16")][int(rng.integers(0, 4))]
    return S, D, d0, inner, pdt, gdt, adt


@pytest.mark.parametrize("seed", range(40))
def test_random_plans(seed):
    S, D, d0, inner, pdt, gdt, adt = random_plan(seed)
    plan, L, unit, alloc = make(S, D, d0, inner, pdt, gdt, adt)
    check_every_step(L, unit, alloc, seed=seed)


@pytest.mark.parametrize("seed", range(6))
def test_long_ragged_runs_span_many_tiles(seed):
    # runs of several warp tiles with ragged heads and tails, shifted sources
    rng = np.random.default_rng(100 + seed)
    S = int(rng.integers(2, 9))
    D = int(rng.integers(1, 3))
    d0 = [int(x) for x in rng.integers(1, 3000, 5)] + [S - 1, 1]
    inner = [int(x) for x in rng.choice([1, 3, 7, 128, 33], len(d0))]
    plan, L, unit, alloc = make(S, D, d0, inner, "bf16", "bf16")
    check_every_step(L, unit, alloc, seed=seed, ops=("avg",))


@pytest.mark.parametrize("S,D,dts", [
    (8, 5, ("bf16", "bf16", "bf16")),   # 40 ranks: more sources than the staged reduce holds
    (33, 1, ("f32", "f32", "f32")),     # 33-member shard group
    (2, 13, ("f32", "f32", "f32")),     # fp32 sources past the staged shared-memory limit
    (16, 2, ("bf16", "bf16", "bf16")),  # 32 sources: the largest staged case
])
def test_wide_meshes(S, D, dts):
    plan, L, unit, alloc = make(S, D, [70, 3, 129], [5, 16, 1], *dts)
    check_every_step(L, unit, alloc, seed=S * 100 + D, ops=("avg",))


@pytest.mark.parametrize("W,S", [(16, 8), (8, 4), (8, 8), (8, 1), (16, 16), (16, 4), (4, 4), (4, 2),
                                 (4, 1), (2, 2), (2, 1), (12, 3)])
def test_every_compiled_mesh_shape(W, S):
    # the bf16 fused reduce is compiled per mesh shape (the last case takes
    # the generic kernel); shards longer than a 256-element step, some
    # aligned with their sources and some shifted (odd-sized vectors move
    # every later offset), so each shape's fast paths run, including the
    # fan-out to several replicas
    plan, L, unit, alloc = make(S, W // S, [1500, 7, 4099, 33], [17, 16, 1, 64], "bf16", "bf16")
    check_every_step(L, unit, alloc, seed=W * 100 + S, ops=("avg", "sum"))


@pytest.mark.parametrize("offsets", [
    # sources shifted against 16-byte boundaries, destinations aligned: funnel-shift path
    {"shards": 2, "grads": 6, "ag_output": 0},
    # every buffer off 16-byte alignment: element-wise path everywhere
    {"shards": 2, "grads": 2, "ag_output": 2, "full_params": 4, "fused": 4, "shard_grads": 2,
     "rs_input": 6},
])
def test_unaligned_pointers(offsets):
    plan, L, unit, alloc = make(4, 2, [13, 40, 7, 1, 300], [5, 1, 16, 3, 9], "bf16", "bf16",
                                offsets=offsets)
    check_every_step(L, unit, alloc, seed=3)


@pytest.mark.parametrize("S,D", [(4, 2), (8, 1), (2, 4)])
@pytest.mark.parametrize("offsets", [None, {"shards": 16, "ag_output": 16, "full_params": 16}, {"shards": 2}])
def test_plans_with_no_shifted_run(S, D, offsets):
    # every inner size a multiple of 8 elements puts every run's source on
    # its destination's 16-byte phase: with 16-byte aligned buffers the bf16
    # copy-in and copy-out take their build without the realigning path
    # (uneven dim 0: padding rows, ragged tails, runs over many tiles); a
    # shard buffer 2 bytes off the grid sends them back to the general build
    plan, L, unit, alloc = make(S, D, [1000, 7, 3, 513, 64], [8, 24, 16, 8, 40], "bf16", "bf16", offsets=offsets)
    check_every_step(L, unit, alloc, seed=S * 10 + D)


@pytest.mark.parametrize("dts", [("bf16", "bf16", "bf16"), ("f32", "f32", "f32"), ("f32", "bf16", "bf16")])
def test_special_values(dts):
    # subnormals (kept: no flush to zero), signed zeros, overflow to infinity,
    # Inf - Inf = NaN, rounding ties
    plan, L, unit, alloc = make(2, 2, [33, 8, 150], [9, 1, 4], *dts)
    check_every_step(L, unit, alloc, seed=11, special=True)


def test_fused_and_unfused_paths_agree_bitwise():
    # "Hyper通信掩盖方案" PR #758 §二.4 fix 1 / §三: fused and unfused AVG agree.
    wl = WL.WORKLOADS["hsdp_2x4_llama"]
    d0 = [a // 64 for a in wl.d0]
    inner = [max(1, i // 64) for i in wl.inner]
    plan, L, unit, alloc = make(4, 2, d0, inner, "bf16", "bf16")
    fill_(unit.grads, 5, 0.02, "bf16")
    unit.reduce_grads("avg")
    a = [to_np(t).copy() for t in unit.shard_grads]
    unit.reduce_grads_unfused("avg")
    b = [to_np(t) for t in unit.shard_grads]
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_each_call_launches_exactly_one_kernel():
    plan, L, unit, alloc = make(4, 2, [7, 16], [8, 1], "bf16", "bf16")
    c0 = C.fsdp_launch_count()
    unit.step()
    torch.cuda.synchronize()
    assert C.fsdp_launch_count() - c0 == 4  # copy-in(+gather), copy-out, rs_ar_reduce, apply
    c0 = C.fsdp_launch_count()
    unit.unshard(fuse_gather=False)
    unit.reduce_grads_unfused()
    torch.cuda.synchronize()
    assert C.fsdp_launch_count() - c0 == 7
    c0 = C.fsdp_launch_count()
    unit.reduce_grads_one_pass()  # the fused reduce with the apply folded in
    torch.cuda.synchronize()
    assert C.fsdp_launch_count() - c0 == 1
    # a mesh too wide for the staged reduce: the two calls it stands for
    plan, L, unit, alloc = make(8, 5, [7, 16], [8, 1], "bf16", "bf16")
    c0 = C.fsdp_launch_count()
    unit.reduce_grads_one_pass()
    torch.cuda.synchronize()
    assert C.fsdp_launch_count() - c0 == 2


def test_empty_and_degenerate_plans():
    # all parameters empty: the slices are 0 elements and nothing launches
    plan = C.Plan([0, 0], [4, 1], 4, 2).upload()
    assert plan.slice_numel("f32") == 0
    unit = HsdpUnit(plan, "bf16", "bf16")
    c0 = C.fsdp_launch_count()
    unit.step()
    torch.cuda.synchronize()
    assert C.fsdp_launch_count() == c0
    # S = D = 1: no communication, the gradient is kept
    plan, L, unit, alloc = make(1, 1, [5, 3], [3, 2], "f32", "f32")
    check_every_step(L, unit, alloc, seed=2)


def test_bad_bindings_are_refused():
    plan = C.Plan([7, 16], [8, 1], 4, 2).upload()
    ok = [torch.empty(plan.shard_numel(p, w % 2), dtype=torch.bfloat16, device="cuda")
          for w in range(4) for p in range(2)]
    with pytest.raises(C.FsdpError) as e:  # too small
        plan.bind("shards", "bf16", [torch.empty(1, dtype=torch.bfloat16, device="cuda")] * 8)
    assert e.value.code == C.FSDP_ERR_INVALID_ARG
    raw = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(C.FsdpError):  # f32 buffer at an odd address
        plan.bind("fused", "f32", [raw[1:].view(torch.uint8)] * 4, check_sizes=False)
    with pytest.raises(C.FsdpError):  # fused buffers are fp32
        plan.bind("fused", "bf16", ok[:4], check_sizes=False)
    b = plan.bind("shards", "bf16", ok)
    with pytest.raises(C.FsdpError) as e:  # wrong role for the call
        C.fsdp_rs_ar_reduce(plan, b, b)
    assert "expected a GRADS binding" in str(e.value)


@pytest.mark.parametrize("seed", range(8))
def test_bucketed_plans(seed):
    # several buckets in one fused buffer ("Hyper通信掩盖方案" PR #758 §二.1,
    # AllReduceParamGroup): every call covers all buckets, gaps stay zero
    S, D, d0, inner, pdt, gdt, adt = random_plan(1000 + seed)
    rng = np.random.default_rng(seed)
    bucket = sorted(int(x) for x in rng.integers(0, 4, len(d0)))
    plan, L, unit, alloc = make(S, D, d0, inner, pdt, gdt, adt, bucket=bucket)
    check_every_step(L, unit, alloc, seed=seed)


def test_many_small_parameters():
    # thousands of tiny runs per table (the lookup's multi-round search,
    # zero-length shards, one-row parameters), every output byte checked
    rng = np.random.default_rng(77)
    P = 1500
    d0 = [int(x) for x in rng.integers(0, 10, P)]
    inner = [int(x) for x in rng.choice([1, 3, 8], P)]
    plan, L, unit, alloc = make(4, 1, d0, inner, "bf16", "bf16")
    check_every_step(L, unit, alloc, seed=78, ops=("avg",))


@pytest.mark.parametrize("cap", [1, 3, 7])
@pytest.mark.parametrize("case", ["ragged", "fanout", "many_runs"])
def test_grid_limits_give_the_same_bytes(case, cap):
    # a grid capped to a few blocks (fsdp_plan_set_grid_limit) makes every
    # warp stride over many tiles: long forward run lookups (search and
    # tile map), the staged reduce's ring and the fan-out images over many
    # steps; every output must still equal the oracle byte for byte
    rng = np.random.default_rng(cap)
    if case == "ragged":
        S, D = 4, 2
        d0 = [int(x) for x in rng.integers(1, 900, 6)] + [3, 1]
        inner = [int(x) for x in rng.choice([1, 3, 64, 129], len(d0))]
    elif case == "fanout":  # (8,1): 8 replicas, fan-out of the fused reduce and the AllReduce
        S, D = 1, 8
        d0, inner = [700, 5, 333], [17, 64, 1]
    else:  # more than 1024 runs per table: the tile -> run map
        S, D = 2, 2
        d0 = [int(x) for x in rng.integers(0, 6, 700)]
        inner = [int(x) for x in rng.choice([1, 8, 40], 700)]
    plan, L, unit, alloc = make(S, D, d0, inner, "bf16", "bf16")
    plan.set_grid_limit(cap)
    check_every_step(L, unit, alloc, seed=10 * cap + len(case), ops=("avg",))


@pytest.mark.parametrize("offsets", [None, {"shard_grads": 2, "fused": 4}])
@pytest.mark.parametrize("S,D", [(4, 2), (8, 1)])
def test_shifted_apply_plans(S, D, offsets):
    # a one-element first parameter moves every later o_p off the 16-byte
    # grid of the fp32 fused rows, so almost all of the apply's data is
    # shifted (the apply's realigning path, and with unaligned buffers its
    # element-wise path); every byte against the oracle
    plan, L, unit, alloc = make(S, D, [1, 3000, 777, 5, 2049], [1, 33, 8, 1, 16], "bf16", "bf16", offsets=offsets)
    check_every_step(L, unit, alloc, seed=S * 10 + D, ops=("avg", "sum"))
