"""The full-size parity checker (tests/full_parity.py) on the CPU: fed the
oracle's own whole-plan outputs it passes, with the plan cut into parameter
groups and column blocks; a single planted byte in any output buffer kind,
in data or padding, makes it fail."""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import full_parity as FP
import oracle as O
from hsdp_sharded_parameter_gb300 import workloads as WL

D0 = [7, 16, 5, 3, 37, 1, 0, 130, 300, 9]
INNER = [8, 8, 1, 4, 3, 17, 5, 1, 64, 40]
W, S = 8, 4


def as_torch(a):
    t = torch.from_numpy(np.ascontiguousarray(a).copy())
    return t.view(torch.bfloat16) if a.dtype == np.uint16 else t


def oracle_unit(op="avg"):
    L = O.Layout(D0, INNER, W, S)
    shards = WL.np_tensors([L.shard_numel(p, w % S) for w in range(W) for p in range(L.P)], 5, 1.0, "bf16")
    grads = WL.np_tensors([L.numel(p) for _ in range(W) for p in range(L.P)], 6, 1.0, "bf16")
    ag = O.ag_gather(L, O.ag_copy_in(L, shards, "bf16", "bf16"), "bf16")
    full = O.ag_copy_out(L, ag, "bf16")
    fused = O.fused_from_grads(L, grads, "bf16")
    sg = O.apply_grads(L, fused, op, "bf16")
    unit = SimpleNamespace(param_dt="bf16", ag_dt="bf16", grad_dt="bf16",
                           shards=[as_torch(a) for a in shards], ag_out=[as_torch(a) for a in ag],
                           full=[as_torch(a) for a in full], grads=[as_torch(a) for a in grads],
                           fused=[as_torch(a) for a in fused], shard_grads=[as_torch(a) for a in sg])
    return L, unit


@pytest.mark.parametrize("op", ["avg", "sum"])
def test_checker_passes_the_oracles_own_outputs(op):
    L, unit = oracle_unit(op)
    budget = 3000
    ps = FP.pieces(L, budget)
    assert any(c0 is not None for _, c0, _ in ps), "no column block"
    assert any(len(g) > 1 for g, _, _ in ps), "no parameter group"
    # the pieces cover every parameter's columns exactly once
    for p in range(L.P):
        cover = sorted((c0 or 0, c1 if c1 is not None else int(L.inner[p])) for g, c0, c1 in ps if p in g)
        assert cover[0][0] == 0 and cover[-1][1] == L.inner[p]
        assert all(a[1] == b[0] for a, b in zip(cover, cover[1:]))
    assert FP.check_unit(L, unit, op, budget=budget) == len(ps)


P = len(D0)


@pytest.mark.parametrize("kind,i,where", [
    ("full", 1 * P + 8, "data"),          # rank 1's full copy of the column-cut parameter
    ("full", 0 * P + 3, "data"),
    ("ag_out", 5, "pad"),                 # a padding row of a gathered slice
    ("ag_out", 2, "tail"),                # the slice tail past the last parameter
    ("fused", 7, "pad"),                  # rank 7 = shard 3: parameter 0's padding row
    ("fused", 1, "tail"),
    ("fused", 6, "data"),
    ("shard_grads", 3 * P + 8, "data"),
    ("shard_grads", 2 * P + 4, "data"),
])
def test_checker_finds_a_planted_byte(kind, i, where):
    L, unit = oracle_unit()
    t = getattr(unit, kind)[i]
    es = t.element_size()
    sl = t.numel() // (S if kind == "ag_out" else 1)  # one slice row
    if where == "data":
        pos = (t.numel() // 2) * es
    elif where == "tail":
        assert L.sum_padded < sl
        pos = (sl - 1) * es
    else:
        # parameter 0 (dim 0 = 7 over 4 shards) has one padding row in shard 3
        assert L.len[0, 3] < L.dss[0]
        row = 3 if kind == "ag_out" else 0
        assert kind == "ag_out" or i % S == 3
        pos = (row * sl + int(L.o[0]) + int(L.len[0, 3]) * int(L.inner[0])) * es
    assert t.numel() > 0
    t.view(torch.uint8)[pos] ^= 0x01
    with pytest.raises(AssertionError):
        FP.check_unit(L, unit, "avg", budget=3000)
