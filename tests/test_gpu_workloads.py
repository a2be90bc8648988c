"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (fused copy-in + gather, copy-out, fused RS+AR, apply AVG).

Every output byte of the step is compared with the CPU oracle: every
gathered buffer, every full parameter, every fp32 fused region and every
applied shard gradient, data and padding (``full_parity``: the oracle runs
on parameter groups and column blocks of the plan, each a plan of its own,
spread over the host cores)."""
import gc

import pytest
import torch

import full_parity as FP
import oracle as O
from hsdp_sharded_parameter_gb300 import capi as C
from hsdp_sharded_parameter_gb300 import workloads as WL
from hsdp_sharded_parameter_gb300.runtime import HsdpUnit

from gpu_util import dirty, fill_

pytestmark = pytest.mark.gpu


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def build(key, with_unfused=False):
    wl = WL.WORKLOADS[key]
    plan = C.Plan(wl.d0, wl.inner, wl.rank_size, wl.shard_size).upload()
    L = O.Layout(wl.d0, wl.inner, wl.rank_size, wl.shard_size)
    unit = HsdpUnit(plan, wl.param_dtype, wl.grad_dtype, with_unfused=with_unfused)
    fill_(unit.shards, wl.seed_params, wl.param_std, wl.param_dtype)
    fill_(unit.grads, wl.seed_grads, wl.grad_std, wl.grad_dtype)
    for bufs in [unit.ag_out, unit.full, unit.fused, unit.shard_grads]:
        dirty(bufs)
    return wl, plan, L, unit


def free(*objs):
    for o in objs:
        if hasattr(o, "close"):
            o.close()
    gc.collect()
    torch.cuda.empty_cache()


# The per-test gather of sampled positions is slow for thousands of params;
# keep the pure-TP workload's random sample smaller.
@pytest.mark.parametrize("key", ["hsdp_2x4_llama", "ragged_fsdp", "pure_tp_compat", "large_hsdp"])
def test_workload_full_size(key):
    wl, plan, L, unit = build(key)
    unit.step(op="avg", fuse_gather=True)
    torch.cuda.synchronize()
    assert FP.check_unit(L, unit, "avg") >= 1
    free(unit, plan)


@pytest.mark.parametrize("key", ["ragged_fsdp", "large_hsdp"])
def test_direct_unshard_full_size(key):
    # all three forward steps in one pass give the oracle's full parameters
    wl, plan, L, unit = build(key)
    unit.unshard_direct()
    torch.cuda.synchronize()
    FP.check_unit(L, unit, forward=True, gathered=False, backward=False)
    free(unit, plan)


@pytest.mark.parametrize("key", ["hsdp_2x4_llama", "ragged_fsdp", "pure_tp_compat", "large_hsdp"])
def test_one_pass_sync_full_size(key):
    # the fused reduce with the apply folded in gives the oracle's fused
    # regions and shard gradients, every byte
    wl, plan, L, unit = build(key)
    unit.reduce_grads_one_pass("avg")
    torch.cuda.synchronize()
    FP.check_unit(L, unit, "avg", forward=False)
    free(unit, plan)


@pytest.mark.parametrize("key,cap", [("hsdp_2x4_llama", 56), ("large_hsdp", 48), ("ragged_fsdp", 64)])
def test_capped_one_pass_sync_full_size(key, cap):
    # the gradient sync as the benchmark's pipeline runs it beside backward
    # compute: on a grid capped at `cap` blocks (the TMA-bulk-fed kernel),
    # every byte of the fused regions and shard gradients against the oracle
    wl, plan, L, unit = build(key)
    plan.set_grid_limit(cap)
    unit.reduce_grads_one_pass("avg")
    torch.cuda.synchronize()
    plan.set_grid_limit(0)
    assert plan.status() == 0
    FP.check_unit(L, unit, "avg", forward=False)
    free(unit, plan)


def test_pure_tp_sum_op():
    # the DTensor-managed (pure TP) default is SUM ("Hyper通信掩盖方案" PR #758 §二.3)
    wl, plan, L, unit = build("pure_tp_compat")
    assert plan.comm_calls() == (0, 8)
    unit.reduce_grads("sum")
    torch.cuda.synchronize()
    FP.check_unit(L, unit, "sum", forward=False)
    free(unit, plan)


def test_offsets_beyond_32_bits():
    # Maximum sizes: a 600001 x 4096 bf16 parameter (2.46e9 elements, 4.9 GB
    # per full tensor) on a (2,2) mesh, ragged over the shard group, followed
    # by small parameters whose runs sit past 2^31 elements and 2^32 bytes in
    # the gathered buffer, the RS input and the fp32 fused region (an inner-1
    # parameter of odd size shifts every later run off the 16-byte grid).
    shapes = [(600001, 4096), (5,), (9, 4096), (3,)]
    d0 = [s[0] for s in shapes]
    inner = [s[1] if len(s) > 1 else 1 for s in shapes]
    plan = C.Plan(d0, inner, 4, 2).upload()
    L = O.Layout(d0, inner, 4, 2)
    assert 2 * L.slice("bf16") > 2**31 and L.slice("f32") * 4 > 2**32
    unit = HsdpUnit(plan, "bf16", "bf16", with_unfused=True)
    fill_(unit.shards, 6001, 1.0, "bf16")
    fill_(unit.grads, 6002, 1.0, "bf16")
    for bufs in [unit.ag_out, unit.full, unit.fused, unit.shard_grads, unit.rs_in]:
        dirty(bufs)
    unit.step(op="avg", fuse_gather=True)
    torch.cuda.synchronize()
    FP.check_unit(L, unit, "avg")
    # the unfused path and the direct unshard give the same bits
    fused = [t.clone() for t in unit.shard_grads]
    dirty(unit.shard_grads)
    unit.reduce_grads_unfused("avg")
    torch.cuda.synchronize()
    for a, b in zip(fused, unit.shard_grads):
        assert torch.equal(bits(a), bits(b))
    del fused
    full = [t.clone() for t in unit.full]
    dirty(unit.full)
    unit.unshard_direct()
    torch.cuda.synchronize()
    for a, b in zip(full, unit.full):
        assert torch.equal(bits(a), bits(b))
    del full
    free(unit, plan)


def test_fused_equals_unfused_at_full_size():
    # "Hyper通信掩盖方案" PR #758 §三: comm_fusion on/off give bitwise-equal
    # gradients on the HSDP (2,4) mesh.
    wl, plan, L, unit = build("hsdp_2x4_llama", with_unfused=True)
    unit.reduce_grads("avg")
    torch.cuda.synchronize()
    fused = [t.clone() for t in unit.shard_grads]
    dirty(unit.shard_grads)
    unit.reduce_grads_unfused("avg")
    torch.cuda.synchronize()
    for a, b in zip(fused, unit.shard_grads):
        assert torch.equal(bits(a), bits(b))
    del fused
    free(unit, plan)
