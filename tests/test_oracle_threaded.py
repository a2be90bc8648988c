"""The labelled multi-core CPU baseline is a separate -fopenmp build of the
oracle's source: its pragmas only split loops over ranks, parameters and
shard rows whose iterations write disjoint outputs. Every step must give
the single-threaded oracle's bytes exactly."""
import os

import numpy as np
import pytest

import oracle as O
from oracle import build as OB
from hsdp_sharded_parameter_gb300 import workloads as WL


def every_output(L, shards, grads, dt):
    ag = O.ag_gather(L, O.ag_copy_in(L, shards, dt, dt), dt)
    full = O.ag_copy_out(L, ag, dt)
    rs_in = O.rs_copy_in(L, grads, dt)
    fused = O.rs_ar_reduce(L, rs_in, dt)
    avg = O.apply_grads(L, fused, "avg", dt)
    acc = O.apply_grads(L, fused, "sum", dt, accumulate=True, shard_grads=[a.copy() for a in avg])
    unf = O.rs_reduce(L, rs_in, dt, "avg")
    unf = O.ar_reduce(L, unf, "avg")
    return ag + full + rs_in + fused + avg + acc + unf


PLANS = [([7, 16, 5, 3], [8, 8, 1, 4], 4, 4, "f32"),
         ([300, 64, 7, 0, 1, 129], [128, 1, 33, 5, 17, 3], 8, 4, "bf16"),
         ([1000, 5, 77], [64, 3, 9], 8, 1, "bf16"),
         ([61, 12289, 4099], [3, 1, 2], 16, 8, "bf16")]


@pytest.mark.parametrize("d0,inner,W,S,dt", PLANS)
def test_threaded_build_gives_the_oracles_bytes(d0, inner, W, S, dt):
    try:
        OB.build(threaded=True)
    except Exception as e:  # a host compiler without OpenMP
        pytest.skip(f"no -fopenmp build: {e}")
    os.environ.setdefault("OMP_NUM_THREADS", "4")
    O.use_threaded(False)
    L = O.Layout(d0, inner, W, S)
    shards = WL.np_tensors([L.shard_numel(p, w % S) for w in range(W) for p in range(L.P)], 31, 1.0, dt)
    grads = WL.np_tensors([L.numel(p) for _ in range(W) for p in range(L.P)], 32, 1.0, dt)
    ref = every_output(L, shards, grads, dt)
    try:
        O.use_threaded(True)
        Lt = O.Layout(d0, inner, W, S)
        got = every_output(Lt, shards, grads, dt)
    finally:
        O.use_threaded(False)
    assert len(ref) == len(got)
    for i, (a, b) in enumerate(zip(ref, got)):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), i
