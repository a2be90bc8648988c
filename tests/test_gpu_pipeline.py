"""The pipelined backward over a stack of layers (the 4-step schedule of the
"Hyper通信掩盖方案" PR #758 write-up §二.2) and CUDA-graph replay of a step.

The pipeline's applied shard gradients are compared byte for byte with the
CPU oracle: the fused path (and its one-pass form, the apply folded into
the fused reduce) with the oracle's RS copy-in + fused reduce + apply (AVG
divides by W once), the unfused path with the oracle's unfused
steps (ReduceScatter with AVG over the shard group, AllReduce with AVG over
the replicas, apply SUM). Both run with the sync kernels on the whole GPU
and with their grid capped to a few SMs (one block per SM of many warps)."""
import numpy as np
import pytest
import torch

import oracle as O
from hsdp_sharded_parameter_gb300 import capi as C
from hsdp_sharded_parameter_gb300 import workloads as WL
from hsdp_sharded_parameter_gb300.runtime import BackwardPipeline, HsdpUnit

from gpu_util import to_np

pytestmark = pytest.mark.gpu

# (dim0 list, inner list, rank_size, shard_size): an HSDP layer, a pure-FSDP
# layer (dp_size 1, applied right after its ReduceScatter) and a ragged
# HSDP layer
LAYERS = [([300, 64, 7], [128, 1, 33], 8, 4),
          ([1000, 5], [64, 3], 4, 4),
          ([129, 40, 1], [256, 2, 9], 8, 2)]


def build_stack():
    units, truth = [], []
    for i, (d0, inner, W, S) in enumerate(LAYERS):
        # only the sync's buffers (no forward buffers), as the benchmark's stacks
        u = HsdpUnit(C.Plan(d0, inner, W, S).upload(), "bf16", "bf16", with_unfused=True, backward_only=True)
        WL.torch_fill_(u.grads, 50 + i, 1.0, "bf16")
        truth.append([g.clone() for g in u.grads])
        units.append(u)
    return units, truth


def oracle_shard_grads(layer, grads, op, fused):
    d0, inner, W, S = layer
    L = O.Layout(d0, inner, W, S)
    g = [to_np(t) for t in grads]
    if fused:
        return O.apply_grads(L, O.fused_from_grads(L, g, "bf16"), op, "bf16")
    buf = O.rs_reduce(L, O.rs_copy_in(L, g, "bf16"), "bf16", op)
    if L.D > 1:
        buf = O.ar_reduce(L, buf, op)
    return O.apply_grads(L, buf, "sum", "bf16")


@pytest.mark.parametrize("comm_blocks", [0, 6])
@pytest.mark.parametrize("fused", [False, True, "one_pass"])
@pytest.mark.parametrize("op", ["avg", "sum"])
def test_pipelined_backward_matches_oracle(fused, op, comm_blocks):
    units, truth = build_stack()
    for u in units:  # the pipeline must wait for gradients it has not seen yet
        for g in u.grads:
            g.view(torch.uint8).fill_(0xFF)
        for s in u.shard_grads:
            s.view(torch.uint8).fill_(0xFF)
    a = torch.randn(2048, 2048, device="cuda", dtype=torch.bfloat16)

    def backward_compute(L):
        for _ in range(4):  # stand-in backward work on the compute stream
            torch.mm(a, a)
        for g, v in zip(units[L].grads, truth[L]):  # "produce" the gradients
            g.copy_(v)

    one_pass = fused == "one_pass"
    fused = bool(fused)
    pipe = BackwardPipeline(units, op=op, fused=fused, comm_blocks=comm_blocks, one_pass=one_pass)
    done = pipe.run(backward_compute)
    BackwardPipeline.finish(done, timeout_s=60)
    pipe.check_status()
    for L, u in enumerate(units):
        exp = oracle_shard_grads(LAYERS[L], truth[L], op, fused)
        for i, (s, e) in enumerate(zip(u.shard_grads, exp)):
            assert np.array_equal(to_np(s), e), (L, i, fused, op, comm_blocks)
    steps = pipe.log
    # every layer's gradients are computed before its ReduceScatter is issued
    for L in range(len(units)):
        assert steps.index(("compute", L)) < steps.index(("rs", L))
    if not fused:
        # pure-FSDP layer 1 is applied right after waiting on its ReduceScatter
        assert steps.index(("wait_rs", 1)) < steps.index(("apply", 1)) < steps.index(("rs", 0))
        # HSDP layers: the AllReduce of layer L+1 is issued after layer L's ReduceScatter
        assert steps.index(("rs", 1)) < steps.index(("ar", 2))
        assert ("ar", 1) not in steps
    for u in units:
        u.close()


def test_graph_replay_matches_eager_step():
    wl = WL.WORKLOADS["tiny_fsdp"]
    plan = C.Plan(wl.d0, wl.inner, wl.rank_size, wl.shard_size).upload()
    unit = HsdpUnit(plan, "f32", "f32")
    WL.torch_fill_(unit.shards, 1, 1.0, "f32")
    WL.torch_fill_(unit.grads, 2, 1.0, "f32")
    unit.step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in unit.full + unit.shard_grads]
    graph = unit.capture_step()
    for t in unit.full + unit.shard_grads:
        t.fill_(float("nan"))
    c0 = C.fsdp_launch_count()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert C.fsdp_launch_count() == c0  # replays do not go through the C ABI
    for a, b in zip(eager, unit.full + unit.shard_grads):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
