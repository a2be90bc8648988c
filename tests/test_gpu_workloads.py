"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (fused copy-in + gather, copy-out, fused RS+AR, apply AVG).

The forward path is checked completely with the oracle's layout: every
gathered buffer and every full parameter, data and padding. The gradient
sync is checked on sampled outputs the oracle computes one by one (random
positions plus every run boundary and its neighbours), and completely for the
properties that hold at any size (padding is +0, replicas agree)."""
import gc

import numpy as np
import pytest
import torch

import oracle as O
from hsdp_sharded_parameter_gb300 import capi as C
from hsdp_sharded_parameter_gb300 import workloads as WL
from hsdp_sharded_parameter_gb300.runtime import HsdpUnit

from gpu_util import dirty, fill_, to_np

pytestmark = pytest.mark.gpu

N_RANDOM = 200_000


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def data_mask(L, s, length, device):
    """Device bool mask over a slice row of shard s: True on actual shard
    elements, from the oracle's layout."""
    m = torch.zeros(length, dtype=torch.bool, device=device)
    for p in range(L.P):
        n = L.shard_numel(p, s)
        if n:
            m[L.o[p]:L.o[p] + n] = True
    return m


def check_forward(L, unit):
    S, P, W = L.S, L.P, L.W
    sl = L.slice(unit.ag_dt)
    dev = unit.device
    masks = [data_mask(L, s, sl, dev) for s in range(S)]
    for w in range(W):
        d = w // S
        for sp in range(S):
            row = unit.ag_out[w][sp * sl:(sp + 1) * sl]
            # padding rows and the slice tail are zero
            assert int(bits(row)[~masks[sp]].count_nonzero()) == 0, ("ag padding", w, sp)
            # actual rows hold shard sp of the shard-group member (d, sp)
            for p in range(P):
                n = L.shard_numel(p, sp)
                if n:
                    src = unit.shards[(d * S + sp) * P + p]
                    assert torch.equal(bits(row[L.o[p]:L.o[p] + n]), bits(src)), ("ag data", w, sp, p)
        for p in range(P):
            parts = [unit.shards[(d * S + sp) * P + p] for sp in range(S)]
            # [RAGGED §6.4]: after the gather only the logical parameter is exposed
            assert torch.equal(bits(unit.full[w * P + p]), bits(torch.cat(parts))), ("full", w, p)


def sample_rows(L, rng, sf):
    """(s, j) samples over the fused region: random positions plus, for every
    run of every shard row, its first and last element and both neighbours."""
    s = rng.integers(0, L.S, N_RANDOM)
    j = rng.integers(0, max(sf, 1), N_RANDOM)
    bs, bj = [], []
    for sh in range(L.S):
        for p in range(L.P):
            n = L.shard_numel(p, sh)
            for x in (L.o[p] - 1, L.o[p], L.o[p] + 1, L.o[p] + n - 1, L.o[p] + n, L.o[p] + n + 1):
                if 0 <= x < sf:
                    bs.append(sh)
                    bj.append(x)
        for x in (sf - 1, L.sum_padded, L.sum_padded - 1):
            if 0 <= x < sf:
                bs.append(sh)
                bj.append(x)
    return np.concatenate([s, bs]).astype(np.int32), np.concatenate([j, bj]).astype(np.int64)


def gather_grads(L, unit, p_idx, e_idx):
    """Gradient values g_{w,p}[e] for every rank w at the sampled (p, e)
    (padding samples get 0), as fp32 on the host, shape (n, W)."""
    n = len(p_idx)
    vals = np.zeros((n, L.W), np.float32)
    dev = unit.device
    for p in np.unique(p_idx[p_idx >= 0]):
        sel = np.nonzero(p_idx == p)[0]
        idx = torch.from_numpy(e_idx[sel]).to(dev)
        cols = torch.stack([unit.grads[w * L.P + p][idx] for w in range(L.W)], dim=1)
        vals[sel] = cols.float().cpu().numpy()
    return vals


def check_backward(L, unit, rng, op="avg"):
    S, D, P, W = L.S, L.D, L.P, L.W
    sf = L.slice("f32")
    dev = unit.device
    # properties over every element: padding is +0, replicas agree
    for s in range(S):
        mask = data_mask(L, s, sf, dev)
        for d in range(D):
            f = unit.fused[d * S + s]
            assert int(bits(f)[~mask].count_nonzero()) == 0, ("fused padding", d, s)
            if d:
                assert torch.equal(bits(f), bits(unit.fused[s])), ("replicas differ", d, s)
    # sampled values: the oracle folds the gathered gradients
    s_idx, j_idx = sample_rows(L, rng, sf)
    p_idx, e_idx = O.locate_fused(L, s_idx, j_idx)
    exp = O.fold_nested(S, D, gather_grads(L, unit, p_idx, e_idx))
    exp[p_idx < 0] = 0.0
    for d in range(D):
        got = np.zeros(len(s_idx), np.float32)
        for s in range(S):
            sel = np.nonzero(s_idx == s)[0]
            got[sel] = unit.fused[d * S + s][torch.from_numpy(j_idx[sel]).to(dev)].cpu().numpy()
        assert np.array_equal(got.view(np.uint32), exp.view(np.uint32)), ("fused values", d)
    # applied gradients at the sampled data positions
    keep = p_idx >= 0
    div = W if op == "avg" else 1
    q = O.div(exp[keep], div)
    exp_g = O.f32_to_bf16(q) if unit.grad_dt == "bf16" else q
    ks = j_idx[keep] - L.o[p_idx[keep]]
    sk, pk = s_idx[keep], p_idx[keep]
    groups = {}
    for i, key in enumerate(zip(sk.tolist(), pk.tolist())):
        groups.setdefault(key, []).append(i)
    for d in range(D):
        got = np.zeros(len(ks), exp_g.dtype)
        for (s, p), rows in groups.items():
            rows = np.asarray(rows)
            idx = torch.from_numpy(ks[rows]).to(dev)
            got[rows] = to_np(unit.shard_grads[(d * S + s) * P + p][idx])
        assert np.array_equal(got.view(np.uint8), exp_g.view(np.uint8)), ("applied grads", d)
    return len(s_idx)


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
    rng = np.random.default_rng(wl.index)
    unit.step(op="avg", fuse_gather=True)
    torch.cuda.synchronize()
    check_forward(L, unit)
    n = check_backward(L, unit, rng, "avg")
    assert n >= N_RANDOM
    free(unit, plan)


@pytest.mark.parametrize("key", ["ragged_fsdp", "large_hsdp"])
def test_direct_unshard_full_size(key):
    # all three forward steps in one pass must give the same full parameters
    wl, plan, L, unit = build(key)
    unit.unshard_direct()
    torch.cuda.synchronize()
    S, P = L.S, L.P
    for w in range(L.W):
        d = w // S
        for p in range(P):
            parts = [unit.shards[(d * S + sp) * P + p] for sp in range(S)]
            assert torch.equal(bits(unit.full[w * P + p]), bits(torch.cat(parts))), (w, p)
    free(unit, plan)


def test_pure_tp_sum_op():
    # the DTensor-managed (pure TP) default is SUM ("Hyper通信掩盖方案" PR #758 §二.3)
    wl, plan, L, unit = build("pure_tp_compat")
    assert plan.comm_calls() == (0, 8)
    unit.reduce_grads("sum")
    torch.cuda.synchronize()
    check_backward(L, unit, np.random.default_rng(9), "sum")
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
    check_forward(L, unit)
    check_backward(L, unit, np.random.default_rng(6003), "avg")
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
