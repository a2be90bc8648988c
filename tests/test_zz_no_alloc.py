"""The allocation-free fused gradient sync (fsdp_rs_ar_reduce_noalloc).

It serves callers that cannot allocate device memory: a framework whose own
caching allocator owns the whole device (a library allocating on the side
breaks its accounting), or a job running so close to the memory limit that
an allocation in the middle of a step could fail. It keeps its work tables
in a fixed array inside the library instead of allocating them.

Checked through the C ABI against the regular fsdp_rs_ar_reduce on the same
inputs, bit for bit (the tolerance of every parity test here), on two calls
in a row: the second call reuses the shared array after the first left its
tables there, and writes over an output buffer that was dirtied in between.
This file is collected last so that a run stopping at the first failure
has already run every other test."""
import pytest
import torch

from hsdp_sharded_parameter_gb300 import capi as C
from hsdp_sharded_parameter_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

CASES = [
    # ragged HSDP mesh (2 replicas x 4 shards): empty shards, padding rows,
    # sources shifted against the fused region
    ([7, 16, 5, 3, 37, 1, 0, 130], [8, 8, 1, 4, 3, 17, 5, 1], 8, 4, "bf16"),
    # the tiny fp32 workload (4 ranks, shard group of 4)
    ([7, 16, 5, 3], [8, 8, 1, 4], 4, 4, "f32"),
    # AllReduce only (shard size 1) with many small parameters
    ([64] * 40 + [1024] * 3, [3] * 40 + [1] * 3, 8, 1, "bf16"),
]


def bits(t):
    return t.view(torch.int32)


@pytest.mark.parametrize("d0,inner,W,S,dt", CASES)
def test_noalloc_matches_fused_sync_on_two_calls(d0, inner, W, S, dt):
    dev = torch.device("cuda", 0)
    ref_plan = C.Plan(d0, inner, W, S).upload()
    host_plan = C.Plan(d0, inner, W, S)  # never uploaded: no device tables
    P = len(d0)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    grads = [torch.empty(d0[p] * inner[p], dtype=tdt, device=dev) for _ in range(W) for p in range(P)]
    sf = ref_plan.slice_numel("f32")
    ref = [torch.empty(sf, dtype=torch.float32, device=dev) for _ in range(W)]
    out = [torch.empty(sf, dtype=torch.float32, device=dev) for _ in range(W)]
    b_grads = ref_plan.bind("grads", dt, grads)
    b_ref = ref_plan.bind("fused", "f32", ref)
    for call, seed in enumerate([11, 12]):
        WL.torch_fill_(grads, seed, 1.0, dt)
        for t in ref + out:
            t.view(torch.uint8).fill_(0xFF)
        C.fsdp_rs_ar_reduce(ref_plan, b_grads, b_ref)
        C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, grads, out)
        torch.cuda.synchronize()
        for w in range(W):
            assert torch.equal(bits(out[w]), bits(ref[w])), (call, w)


def test_noalloc_refuses_a_plan_too_large_for_its_array():
    # 40,000 parameters of 1 row over 8 ranks: the pointer table alone is
    # 8 * 40,000 * 8 bytes = 2.56 MB, beyond the fixed array
    P = 40_000
    plan = C.Plan([1] * P, [1] * P, 8, 8)
    g = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    f = torch.zeros(plan.slice_numel("f32"), dtype=torch.float32, device="cuda")
    with pytest.raises(C.FsdpError) as e:
        C.fsdp_rs_ar_reduce_noalloc(plan, "bf16", [g] * (8 * P), [f] * 8)
    assert e.value.code == C.FSDP_ERR_INVALID_ARG and "bytes of work tables" in str(e.value)
