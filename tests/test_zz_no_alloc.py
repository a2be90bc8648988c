"""The allocation-free fused gradient sync (fsdp_rs_ar_reduce_noalloc).

It serves callers that cannot allocate device memory: a framework whose own
caching allocator owns the whole device (a library allocating on the side
breaks its accounting), or a job running so close to the memory limit that
an allocation in the middle of a step could fail. It keeps its work tables
in a fixed array inside the library instead of allocating them.

Checked through the C ABI, bit for bit (the tolerance of every parity test
here), against the CPU oracle and against the regular fsdp_rs_ar_reduce on
the same inputs, on two calls in a row: the second call reuses the shared
array after the first left its tables there, and writes over an output
buffer that was dirtied in between. Also checked: a call leaves the device's
free memory unchanged, a grid cap applies, a plan with more than a thousand
runs (where the regular path carries a tile -> run map) computes the same
bits, a call during stream capture is refused, and so are short pointer
lists and undersized tensors. This file is collected last so that a run
stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle as O
from hsdp_sharded_parameter_gb300 import capi as C
from hsdp_sharded_parameter_gb300 import workloads as WL

from gpu_util import to_np

pytestmark = pytest.mark.gpu

CASES = {
    # ragged HSDP mesh (2 replicas x 4 shards): empty shards, padding rows,
    # sources shifted against the fused region
    "ragged_2x4": ([7, 16, 5, 3, 37, 1, 0, 130], [8, 8, 1, 4, 3, 17, 5, 1], 8, 4, "bf16"),
    # the tiny fp32 workload (4 ranks, shard group of 4)
    "tiny_f32": ([7, 16, 5, 3], [8, 8, 1, 4], 4, 4, "f32"),
    # AllReduce only (shard size 1) with many small parameters
    "ar_only": ([64] * 40 + [1024] * 3, [3] * 40 + [1] * 3, 8, 1, "bf16"),
    # 1500 parameters over a (2,2) mesh: more than 1024 runs per table
    "many_runs": ([3 + (i % 5) for i in range(1500)], [1 + (i % 7) for i in range(1500)], 4, 2, "bf16"),
}


def bits(t):
    return t.view(torch.int32)


def setup(key):
    d0, inner, W, S, dt = CASES[key]
    dev = torch.device("cuda", 0)
    ref_plan = C.Plan(d0, inner, W, S).upload()
    host_plan = C.Plan(d0, inner, W, S)  # never uploaded: no device tables
    P = len(d0)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    grads = [torch.empty(d0[p] * inner[p], dtype=tdt, device=dev) for _ in range(W) for p in range(P)]
    sf = ref_plan.slice_numel("f32")
    ref = [torch.empty(sf, dtype=torch.float32, device=dev) for _ in range(W)]
    out = [torch.empty(sf, dtype=torch.float32, device=dev) for _ in range(W)]
    L = O.Layout(d0, inner, W, S)
    return dt, ref_plan, host_plan, grads, ref, out, L


@pytest.mark.parametrize("grid", [0, 3])
@pytest.mark.parametrize("key", list(CASES))
def test_noalloc_matches_oracle_and_fused_sync_on_two_calls(key, grid):
    dt, ref_plan, host_plan, grads, ref, out, L = setup(key)
    if grid:
        # a cap of 3 blocks: every warp strides over many tiles
        host_plan.set_grid_limit(grid)
    b_grads = ref_plan.bind("grads", dt, grads)
    b_ref = ref_plan.bind("fused", "f32", ref)
    for call, seed in enumerate([11, 12]):
        WL.torch_fill_(grads, seed, 1.0, dt)
        for t in ref + out:
            t.view(torch.uint8).fill_(0xFF)
        C.fsdp_rs_ar_reduce(ref_plan, b_grads, b_ref)
        C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, grads, out)
        torch.cuda.synchronize()
        exp = O.fused_from_grads(L, [to_np(g) for g in grads], dt)
        for w in range(L.W):
            got = to_np(out[w])
            assert np.array_equal(got.view(np.uint32), exp[w].view(np.uint32)), (call, w, "oracle")
            assert torch.equal(bits(out[w]), bits(ref[w])), (call, w, "fsdp_rs_ar_reduce")


def test_noalloc_call_allocates_no_device_memory():
    dt, ref_plan, _, grads, _, out, L = setup("many_runs")
    WL.torch_fill_(grads, 21, 1.0, dt)
    # a first call on this device loads the library's array and kernel
    C.fsdp_rs_ar_reduce_noalloc(C.Plan([4], [2], 4, 2), dt,
                                [torch.zeros(8, dtype=torch.bfloat16, device="cuda")] * 4,
                                [torch.zeros(C.Plan([4], [2], 4, 2).slice_numel("f32"),
                                             dtype=torch.float32, device="cuda")] * 4)
    C.fsdp_rs_ar_reduce_noalloc(C.Plan(*CASES["many_runs"][:4]), dt, grads, out)
    torch.cuda.synchronize()
    fresh = C.Plan(*CASES["many_runs"][:4])  # a plan no call has seen yet
    free0, _ = torch.cuda.mem_get_info()
    n0 = C.fsdp_launch_count()
    C.fsdp_rs_ar_reduce_noalloc(fresh, dt, grads, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert C.fsdp_launch_count() - n0 == 1
    exp = O.fused_from_grads(L, [to_np(g) for g in grads], dt)
    for w in range(L.W):
        assert np.array_equal(to_np(out[w]).view(np.uint32), exp[w].view(np.uint32)), w


def test_noalloc_is_refused_during_stream_capture():
    dt, _, host_plan, grads, _, out, _ = setup("ragged_2x4")
    WL.torch_fill_(grads, 31, 1.0, dt)
    C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, grads, out)  # set-up before any capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    x = torch.zeros(16, device="cuda")
    g = torch.cuda.CUDAGraph()
    n0 = C.fsdp_launch_count()
    with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
        x.add_(1.0)
        with pytest.raises(C.FsdpError) as e:
            C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, grads, out, stream=side)
    assert e.value.code == C.FSDP_ERR_INVALID_ARG and "captured" in str(e.value)
    assert C.fsdp_launch_count() == n0
    g.replay()
    torch.cuda.synchronize()
    assert float(x[0]) == 1.0
    # the stream works as before once the capture has ended
    C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, grads, out, stream=side)
    torch.cuda.synchronize()


def test_noalloc_refuses_short_lists_and_undersized_tensors():
    dt, _, host_plan, grads, _, out, _ = setup("ragged_2x4")
    with pytest.raises(C.FsdpError, match="tensors given"):
        C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, grads[:-1], out)
    with pytest.raises(C.FsdpError, match="tensors given"):
        C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, grads, out[:3])
    small = list(grads)
    small[5] = torch.empty(small[5].numel() - 1, dtype=small[5].dtype, device="cuda")
    with pytest.raises(C.FsdpError, match="needs"):
        C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, small, out)
    with pytest.raises(C.FsdpError, match="needs"):
        C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, grads, [out[0][:-1]] + out[1:])
    with pytest.raises(C.FsdpError, match="expected"):
        C.fsdp_rs_ar_reduce_noalloc(host_plan, dt, [g.float() for g in grads], out)


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
