"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something the pages or the mathematics
fix: the pages' worked examples and size relations, hand-derived tables,
closed-form invariants of the chunking, exact integer arithmetic (brute force
on the dense, unsharded tensors), library round-to-nearest-even, the textbook
error bound of recursive summation, and hand-worked rounding cases. A
plausible slip in the oracle (a dropped term, a wrong offset, sign or index,
transposed ranks) fails at least one of them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from hsdp_sharded_parameter_gb300 import workloads as WL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_to_bf16_torch(x):
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def cut_shards(L, fulls, dt):
    """Shards of per-(rank, param) full tensors by plain row slicing."""
    out = []
    for w in range(L.W):
        s = w % L.S
        for p in range(L.P):
            rows = fulls[w * L.P + p].reshape(L.d0[p], L.inner[p])
            a, n = L.off[p, s], L.len[p, s]
            out.append(np.ascontiguousarray(rows[a:a + n].reshape(-1)))
    return out


# --------------------------------------------------------------------------
# Planning
# --------------------------------------------------------------------------

def read_plan_fixture():
    rows, extra = [], {}
    with open(os.path.join(GOLDEN, "tiny_fsdp_plan.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if "|" in line:
                a, b, c = (x.split() for x in line.split("|"))
                rows.append((list(map(int, a)), [tuple(map(int, t.split(","))) for t in b],
                             list(map(int, c))))
            else:
                k, v = line.split()
                extra[k] = int(v)
    return rows, extra


def test_plan_matches_hand_derived_tiny_table():
    rows, extra = read_plan_fixture()
    wl = WL.WORKLOADS["tiny_fsdp"]
    L = O.Layout(wl.d0, wl.inner, wl.rank_size, wl.shard_size)
    assert L.P == len(rows) == 4
    for p, ((d0, inner, chunk), shards, (pad, off)) in enumerate(rows):
        assert (L.d0[p], L.inner[p], L.dss[p]) == (d0, inner, chunk)
        assert [(int(L.off[p, s]), int(L.len[p, s])) for s in range(4)] == shards
        assert L.dss[p] * L.inner[p] == pad
        assert L.o[p] == off
    assert L.sum_padded == extra["sum_padded"]
    assert L.slice("f32") == extra["slice_f32"]
    assert L.slice("bf16") == extra["slice_bf16"]


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 7, 8, 9, 16])
def test_chunking_invariants(S):
    """Closed-form facts of fixed-size chunking that any correct plan obeys:
    the shards tile [0, d0) in rank order; every non-empty shard but the
    last has exactly `chunk` rows; chunk is the smallest size with
    S * chunk >= d0; empty shards only trail; offsets are prefix sums."""
    d0 = list(range(0, 41)) + [4099, 11003]
    inner = [1 + (i * 7) % 17 for i in range(len(d0))]
    L = O.Layout(d0, inner, S * 2, S)
    for p in range(L.P):
        c = int(L.dss[p])
        assert S * c >= d0[p] and (c == 0 or S * (c - 1) < d0[p])
        pos, seen_short = 0, False
        for s in range(S):
            a, n = int(L.off[p, s]), int(L.len[p, s])
            assert a == pos
            assert 0 <= n <= c
            if seen_short:
                assert n == 0
            if n < c:
                seen_short = True
            pos += n
        assert pos == d0[p]
    assert list(L.o) == list(np.concatenate([[0], np.cumsum(L.dss * L.inner)]))


def test_uniform_params_have_no_padding_rows():
    # issue 319 §9.2, last boundary: an evenly divisible parameter gets no padding.
    for key in ["hsdp_2x4_llama", "large_hsdp"]:
        wl = WL.WORKLOADS[key]
        L = O.Layout(wl.d0, wl.inner, wl.rank_size, wl.shard_size)
        assert all(L.dss * L.S == L.d0)
        assert (L.len == L.dss[:, None]).all()
        assert L.sum_padded * L.S == wl.numel_per_rank


def test_dp_size_and_comm_calls_from_the_rfc_examples():
    # FullyShard RFC §2.2.5 item 5: HSDP rank_size=8, shard_size=4 -> dp_size=2,
    # RS(4) + AR(2); pure-TP compat rank_size=8, shard_size=1 -> dp_size=8, AR(8) only.
    L = O.Layout([8], [1], 8, 4)
    assert (L.S, L.D) == (4, 2)
    assert L.comm_calls() == (4, 2)
    L = O.Layout([8], [1], 8, 1)
    assert (L.S, L.D) == (1, 8)
    assert L.comm_calls() == (0, 8)
    # §5.2 item 1: 1D FSDP is RS only; item 5: enable_param_shard=False never issues RS.
    assert O.Layout([8], [1], 8, 8).comm_calls() == (8, 0)
    L = O.Layout([8], [1], 8, 4, enable_param_shard=0)
    assert (L.S, L.D) == (1, 8) and L.comm_calls() == (0, 8)
    # §2.2.2 case 3: neither sharded nor replicated -> no communication.
    assert O.Layout([8], [1], 1, 1).comm_calls() == (0, 0)
    # The large workload: rank_size 16, shard 8 -> dp 2.
    assert O.Layout([8], [1], 16, 8).D == 2


def test_group_ranks_partition_the_mesh():
    W, S = 8, 4
    L = O.Layout([8], [1], W, S)
    shard_groups, rep_groups = set(), set()
    for w in range(W):
        sg, rg = L.group_ranks(w)
        assert w in sg and w in rg
        assert len(sg) == S and len(rg) == W // S
        assert len(set(sg) & set(rg)) == 1
        shard_groups.add(tuple(sg))
        rep_groups.add(tuple(rg))
    assert sorted(x for g in shard_groups for x in g) == list(range(W))
    assert sorted(x for g in rep_groups for x in g) == list(range(W))
    # Reading (replicate index outer): rank 5 of a (2,4) mesh is (d=1, s=1).
    sg, rg = L.group_ranks(5)
    assert list(sg) == [4, 5, 6, 7] and list(rg) == [1, 5]


def test_non_dim0_and_invalid_plans_are_rejected():
    # issue 319 §3.2 non-goal 1: uneven sharding on an axis other than dim 0 is unsupported.
    with pytest.raises(O.OracleError) as e:
        O.Layout([7], [8], 4, 4, shard_dim=1)
    assert e.value.code == O.ENOTIMPL
    with pytest.raises(O.OracleError) as e:
        O.Layout([7], [8], 6, 4)  # rank_size not a multiple of shard_size
    assert e.value.code == O.EINVAL


def test_workload_sizes():
    sizes = {k: WL.WORKLOADS[k].numel_per_rank for k in WL.ORDER}
    assert sizes == {"tiny_fsdp": 201, "hsdp_2x4_llama": 202_383_360,
                     "ragged_fsdp": 557_261_111, "pure_tp_compat": 50_552_832,
                     "large_hsdp": 855_654_400}
    pads = {}
    for k in WL.ORDER:
        wl = WL.WORKLOADS[k]
        pads[k] = O.Layout(wl.d0, wl.inner, wl.rank_size, wl.shard_size).sum_padded
    assert pads == {"tiny_fsdp": 54, "hsdp_2x4_llama": 50_595_840, "ragged_fsdp": 69_697_873,
                    "pure_tp_compat": 50_552_832, "large_hsdp": 106_956_800}
    rag = WL.WORKLOADS["ragged_fsdp"]
    L = O.Layout(rag.d0, rag.inner, 8, 8)
    assert int((L.len == 0).any(axis=1).sum()) == 7
    assert sorted(rag.inner).count(1) == 20 and rag.inner.count(128) == 20
    assert rag.inner.count(4096) == 24


def test_splitmix64_known_values():
    g = WL.splitmix64(3)
    assert [next(g) % 12289 + 1 for _ in range(3)] == [7777, 1639, 2844]
    assert WL.WORKLOADS["ragged_fsdp"].d0[9:12] == [7777, 1639, 2844]


# --------------------------------------------------------------------------
# Rounding
# --------------------------------------------------------------------------

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, 200_000, dtype=np.uint64).astype(np.uint32)
    # exact ties (rest == 0x8000) with odd and even kept bits, and neighbours
    ties = (rng.integers(0, 2**16, 5000, dtype=np.uint32) << 16) | 0x8000
    near = np.concatenate([ties - 1, ties + 1])
    special = np.array([0, 0x80000000, 0x00000001, 0x807FFFFF, 0x7F7FFFFF, 0xFF7FFFFF,
                        0x7F7F8000, 0x7F800000, 0xFF800000, 0x3F808000, 0x3F818000],
                       dtype=np.uint32)
    x = np.concatenate([bits, ties, near, special]).astype(np.uint32).view(np.float32)
    finite = np.isfinite(x) | np.isinf(x)
    got = O.f32_to_bf16(x)
    ref = f32_to_bf16_torch(x)
    assert np.array_equal(got[finite], ref[finite])
    nan = ~finite
    assert nan.any()
    back = O.bf16_to_f32(got[nan])
    assert np.isnan(back).all()
    assert np.array_equal(np.signbit(back), np.signbit(x[nan]))


def test_bf16_widening_is_exact():
    h = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    f = O.bf16_to_f32(h)
    ok = ~np.isnan(f)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(f[ok].view(np.uint32), ref[ok].view(np.uint32))


# --------------------------------------------------------------------------
# Forward path: copy-in, all-gather, copy-out
# --------------------------------------------------------------------------

RANDOM_PLANS = [
    # (S, D, d0 list, inner list)
    (4, 1, [7, 16, 5, 3], [8, 8, 1, 4]),
    (3, 2, [0, 1, 2, 10, 11, 40], [5, 1, 17, 3, 1, 2]),
    (5, 1, [4, 3, 9, 1], [1, 7, 2, 9]),
    (1, 4, [6, 9], [3, 1]),
    (2, 2, [13, 1, 0, 2], [1, 16, 4, 3]),
    (9, 1, [8, 25, 17], [3, 1, 6]),
    (1, 1, [5, 3], [2, 7]),
]


def make_plan(S, D, d0, inner, **kw):
    return O.Layout(d0, inner, S * D, S, **kw)


@pytest.mark.parametrize("S,D,d0,inner", RANDOM_PLANS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_allgather_round_trip_restores_the_parameter(S, D, d0, inner, dt):
    # Hyper通信掩盖方案 PR #758 write-up §四.1 (send = own slice) and issue 319 §6.4
    # (only the logical shape is exposed after the all-gather): unpacking the
    # gathered buffer must give back, bit for bit, the parameter that was sharded.
    L = make_plan(S, D, d0, inner)
    sizes = [L.numel(p) for _ in range(L.W) for p in range(L.P)]
    full = WL.np_tensors(sizes, 11, 1.0, dt)
    # every replica group holds the same parameter in HSDP; keep them distinct to
    # catch reads from the wrong replica
    shards = cut_shards(L, full, dt)
    ag = O.ag_copy_in(L, shards, dt, dt)
    O.ag_gather(L, ag, dt)
    out = O.ag_copy_out(L, ag, dt)
    for w in range(L.W):
        d = w // S
        for p in range(L.P):
            # row r of the result comes from the shard-group member holding it,
            # which is replica d's copy
            src_rows = np.concatenate([
                full[(d * S + s) * L.P + p].reshape(L.d0[p], L.inner[p])[L.off[p, s]:L.off[p, s] + L.len[p, s]]
                for s in range(S)]).reshape(-1) if L.d0[p] else np.zeros(0, full[0].dtype)
            assert np.array_equal(out[w * L.P + p].view(np.uint8), src_rows.view(np.uint8))


def test_allgather_with_cast_rounds_once():
    L = make_plan(4, 1, [7, 16, 5, 3], [8, 8, 1, 4])
    sizes = [L.numel(p) for _ in range(L.W) for p in range(L.P)]
    full = WL.np_tensors(sizes, 5, 1.0, "f32")
    # make all ranks hold the same parameter so the gathered result is that parameter
    for w in range(1, L.W):
        for p in range(L.P):
            full[w * L.P + p] = full[p]
    shards = cut_shards(L, full, "f32")
    ag = O.ag_copy_in(L, shards, "f32", "bf16")
    O.ag_gather(L, ag, "bf16")
    out = O.ag_copy_out(L, ag, "bf16")
    for w in range(L.W):
        for p in range(L.P):
            assert np.array_equal(out[w * L.P + p], f32_to_bf16_torch(full[p]))


@pytest.mark.parametrize("S,D,d0,inner", RANDOM_PLANS)
def test_copy_in_padding_is_zero_even_on_a_dirty_buffer(S, D, d0, inner):
    # issue 319 §9.2: padding starts at 0 and is still 0 when the buffer is reused.
    L = make_plan(S, D, d0, inner)
    shard_sizes = [L.shard_numel(p, w % S) for w in range(L.W) for p in range(L.P)]
    sl = L.slice("bf16")
    for attempt in range(2):
        shards = WL.np_tensors(shard_sizes, 21 + attempt, 1.0, "bf16")
        ag = [np.full(S * sl, 0xFFFF, np.uint16) for _ in range(L.W)]
        O.ag_copy_in(L, shards, "bf16", "bf16", ag_out=ag)
        for w in range(L.W):
            s = w % S
            row = ag[w][s * sl:(s + 1) * sl]
            data = np.zeros(sl, bool)
            for p in range(L.P):
                n = L.shard_numel(p, s)
                data[L.o[p]:L.o[p] + n] = True
                assert np.array_equal(row[L.o[p]:L.o[p] + n], shards[w * L.P + p])
            assert (row[~data] == 0).all()
            # slices of other shard ranks are left alone by copy-in
            others = np.delete(ag[w], np.arange(s * sl, (s + 1) * sl))
            assert (others == 0xFFFF).all()


# --------------------------------------------------------------------------
# Backward path: copy-in, fused reduction, apply
# --------------------------------------------------------------------------

def int_grads(L, seed, dt, lo=-8, hi=8):
    """Small integer gradients: every fp32 partial sum is exact, so the
    expected result is plain integer arithmetic, independent of order."""
    rng = np.random.default_rng(seed)
    ints = [rng.integers(lo, hi + 1, L.numel(p)).astype(np.int64)
            for _ in range(L.W) for p in range(L.P)]
    if dt == "f32":
        vals = [a.astype(np.float32) for a in ints]
    else:
        vals = [(a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16) for a in ints]
    return ints, vals


def rational_to_f32(fr):
    # A small-integer numerator over a small denominator is either exact in
    # binary64 or a repeating binary fraction that is never a binary32 tie,
    # so rounding through binary64 equals rounding once.
    return np.float32(np.float64(fr.numerator) / np.float64(fr.denominator))


@pytest.mark.parametrize("S,D,d0,inner", RANDOM_PLANS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["avg", "sum"])
def test_sharded_grads_equal_dense_sum(S, D, d0, inner, dt, op):
    # issue 319 §9.1 (Level0): gradients equal the non-distributed result.
    # Brute force on the dense tensors with no padding logic at all: the grad
    # shard of rank (d, s) for param p is rows [off, off+len) of
    # sum over all ranks of the full gradient, divided by W for AVG.
    L = make_plan(S, D, d0, inner)
    ints, grads = int_grads(L, 3 + S * 10 + D, dt)
    fused = O.fused_from_grads(L, grads, dt)
    out = O.apply_grads(L, fused, op, dt)
    for w in range(L.W):
        s = w % S
        for p in range(L.P):
            dense = sum(ints[v * L.P + p] for v in range(L.W)).reshape(L.d0[p], L.inner[p])
            rows = dense[L.off[p, s]:L.off[p, s] + L.len[p, s]].reshape(-1)
            div = L.W if op == "avg" else 1
            exp = np.array([rational_to_f32(Fraction(int(v), div)) for v in rows], np.float32)
            if dt == "bf16":
                exp = f32_to_bf16_torch(exp)
            assert np.array_equal(out[w * L.P + p], exp), (w, p)


@pytest.mark.parametrize("S,D,d0,inner", RANDOM_PLANS)
def test_fused_buffer_layout_and_zero_padding(S, D, d0, inner):
    # Hyper通信掩盖方案 PR #758 §二.1: RS outputs sit in views of one 512B-aligned
    # fused buffer; issue 319 §6.4/§9.2: the padding tail of every param is 0.
    L = make_plan(S, D, d0, inner)
    ints, grads = int_grads(L, 99, "f32")
    fused = O.fused_from_grads(L, grads, "f32")
    sf = L.slice("f32")
    assert sf * 4 % 512 == 0 and sf >= L.sum_padded
    for w in range(L.W):
        s = w % S
        assert len(fused[w]) == sf
        data = np.zeros(sf, bool)
        for p in range(L.P):
            n = L.shard_numel(p, s)
            data[L.o[p]:L.o[p] + n] = True
            dense = sum(ints[v * L.P + p] for v in range(L.W)).reshape(-1)
            first = L.off[p, s] * L.inner[p]
            assert np.array_equal(fused[w][L.o[p]:L.o[p] + n], dense[first:first + n].astype(np.float32))
        z = fused[w][~data]
        assert (z == 0).all() and not np.signbit(z).any()
    # replicas of a shard rank hold identical regions
    for w in range(L.W):
        for v in range(L.W):
            if w % S == v % S:
                assert np.array_equal(fused[w], fused[v])


def test_summation_order_hand_worked():
    with open(os.path.join(GOLDEN, "nested_order.json")) as f:
        g = json.load(f)
    L = O.Layout([g["shape"][0]], [1], g["rank_size"], g["shard_size"])
    grads = [np.array(v, np.float32) for v in g["grads"]]
    fused = O.fused_from_grads(L, grads, "f32")
    assert [float(f[0]) for f in fused] == g["fused_first_element"]
    for op, key in [("avg", "shard_grad_avg"), ("sum", "shard_grad_sum")]:
        out = O.apply_grads(L, fused, op, "f32")
        assert [list(map(float, a)) for a in out] == g[key]


def test_fold_matches_textbook_error_bound():
    # |fl(sum) - sum| <= gamma_(n-1) * sum|x| for any order of n-1 additions.
    rng = np.random.default_rng(5)
    for S, D in [(4, 1), (4, 2), (8, 2), (1, 8), (3, 3)]:
        W = S * D
        vals = rng.standard_normal((20000, W)).astype(np.float32)
        got = O.fold_nested(S, D, vals).astype(np.float64)
        exact = vals.astype(np.float64).sum(axis=1)
        u = 2.0 ** -24
        gamma = (W - 1) * u / (1 - (W - 1) * u)
        bound = gamma * np.abs(vals.astype(np.float64)).sum(axis=1)
        assert (np.abs(got - exact) <= bound).all()


@pytest.mark.parametrize("S,D", [(4, 2), (2, 4), (8, 2), (4, 1), (1, 8), (2, 2)])
def test_fused_and_unfused_avg_are_bitwise_equal(S, D):
    # Hyper通信掩盖方案 PR #758 write-up §二.4 fix 1 and §三: the unfused path
    # (RS AVG over the shard group, AR AVG over replicas) equals the fused path
    # (SUM, SUM, then one divide) bit for bit. Power-of-two mesh sizes, as in
    # every workload; for other sizes the two placements of the divide can
    # differ in the last bit (a stated reading).
    L = make_plan(S, D, [13, 8, 5, 31], [3, 16, 1, 2])
    sizes = [L.numel(p) for _ in range(L.W) for p in range(L.P)]
    for dt in ["f32", "bf16"]:
        grads = WL.np_tensors(sizes, 31, 1.0, dt)
        rs_in = O.rs_copy_in(L, grads, dt)
        fused = O.apply_grads(L, O.rs_ar_reduce(L, rs_in, dt), "avg", dt)
        buf = O.rs_reduce(L, rs_in, dt, "avg")
        O.ar_reduce(L, buf, "avg")
        unfused = O.apply_grads(L, buf, "sum", dt)
        for a, b in zip(fused, unfused):
            assert np.array_equal(a, b)
        # Negative control: the pre-fix unfused path skipped the replicate-dim
        # divide, so its gradients come out D times too large.
        bad = O.rs_reduce(L, rs_in, dt, "avg")
        O.ar_reduce(L, bad, "sum")
        good = O.rs_reduce(L, rs_in, dt, "avg")
        O.ar_reduce(L, good, "avg")
        for a, b in zip(bad, good):
            nz = b != 0
            assert np.array_equal(a[nz], b[nz] * np.float32(D))
            if D > 1:
                assert not np.array_equal(a[nz], b[nz])


def test_special_cases_reduce_to_textbook_operations():
    rng = np.random.default_rng(1)
    # S = D = 1: no communication, the gradient is kept (RFC §2.2.2 case 3).
    L = make_plan(1, 1, [7, 3], [4, 5])
    g = [rng.standard_normal(L.numel(p)).astype(np.float32) for p in range(2)]
    out = O.apply_grads(L, O.fused_from_grads(L, g, "f32"), "avg", "f32")
    assert all(np.array_equal(a, b) for a, b in zip(out, g))
    # S = 1 (AllReduce only, pure-TP compat): a plain left-to-right sum over ranks.
    L = make_plan(1, 8, [9], [3])
    g = [rng.standard_normal(27).astype(np.float32) for _ in range(8)]
    fused = O.fused_from_grads(L, g, "f32")
    acc = g[0].copy()
    for v in g[1:]:
        acc = (acc + v).astype(np.float32)
    assert np.array_equal(fused[0][:27], acc)
    # D = 1 (1D FSDP, ReduceScatter only): shard s is the sum of rows of shard s.
    L = make_plan(4, 1, [7], [8])
    g = [rng.standard_normal(56).astype(np.float32) for _ in range(4)]
    fused = O.fused_from_grads(L, g, "f32")
    acc = g[0].copy()
    for v in g[1:]:
        acc = (acc + v).astype(np.float32)
    for s in range(4):
        n = L.shard_numel(0, s)
        assert np.array_equal(fused[s][:n], acc[L.off[0, s] * 8: L.off[0, s] * 8 + n])


def test_grad_accumulation_adds_then_rounds_once():
    # RFC §5.2 item 9 (requires_grad_sync False/True): accumulated gradients
    # equal old + new, exact here because all values are small integers.
    L = make_plan(2, 2, [6, 3], [4, 1])
    ints, grads = int_grads(L, 17, "bf16")
    fused = O.fused_from_grads(L, grads, "bf16")
    old_ints = [np.arange(L.shard_numel(p, w % 2)) % 5 for w in range(4) for p in range(2)]
    old = [(a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16) for a in old_ints]
    out = O.apply_grads(L, fused, "sum", "bf16", accumulate=True, shard_grads=[a.copy() for a in old])
    for w in range(4):
        s = w % 2
        for p in range(2):
            dense = sum(ints[v * 2 + p] for v in range(4)).reshape(L.d0[p], -1)
            rows = dense[L.off[p, s]:L.off[p, s] + L.len[p, s]].reshape(-1)
            exp = f32_to_bf16_torch((rows + old_ints[w * 2 + p]).astype(np.float32))
            assert np.array_equal(out[w * 2 + p], exp)


# --------------------------------------------------------------------------
# Element locators (used for sampled checks at full size)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("S,D,d0,inner", RANDOM_PLANS)
def test_locators_agree_with_whole_buffer_steps(S, D, d0, inner):
    L = make_plan(S, D, d0, inner)
    sizes = [L.numel(p) for _ in range(L.W) for p in range(L.P)]
    grads = WL.np_tensors(sizes, 8, 1.0, "bf16")
    fused = O.fused_from_grads(L, grads, "bf16")
    sf = L.slice("f32")
    s_idx = np.repeat(np.arange(S), sf)
    j_idx = np.tile(np.arange(sf), S)
    p, e = O.locate_fused(L, s_idx, j_idx)
    vals = np.zeros((len(s_idx), L.W), np.float32)
    for i in range(len(s_idx)):
        if p[i] >= 0:
            for v in range(L.W):
                vals[i, v] = O.bf16_to_f32(grads[v * L.P + p[i]][e[i]: e[i] + 1])[0]
    got = O.fold_nested(S, D, vals)
    for w in range(L.W):
        s = w % S
        assert np.array_equal(got[s * sf:(s + 1) * sf], fused[w])
    # gathered-buffer locator against the forward steps
    shards = cut_shards(L, grads, "bf16")
    ag = O.ag_gather(L, O.ag_copy_in(L, shards, "bf16", "bf16"), "bf16")
    for w in range(L.W):
        for q in range(L.P):
            n = L.numel(q)
            if n == 0:
                continue
            sh, k, idx = O.locate_gathered(L, "bf16", np.full(n, q), np.arange(n))
            d = w // S
            src = np.array([shards[(d * S + sh[i]) * L.P + q][k[i]] for i in range(n)], np.uint16)
            assert np.array_equal(ag[w][idx], src)


# --------------------------------------------------------------------------
# Several buckets in one fused buffer
# --------------------------------------------------------------------------

def test_bucketed_plan_matches_hand_derived_table():
    rows, extra = [], {}
    with open(os.path.join(GOLDEN, "bucketed_plan.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0].isdigit():
                rows.append(tuple(map(int, parts)))
            else:
                extra[parts[0]] = int(parts[1])
    L = O.Layout([7, 5, 3], [8, 1, 4], 4, 4, bucket=[0, 0, 1])
    assert [(p, b, int(L.o[p])) for p, b, _ in rows] == rows
    assert L.sum_padded == extra["end"]
    assert L.slice("f32") == extra["slice_f32"] and L.slice("bf16") == extra["slice_bf16"]


def test_bucket_bases_are_512_byte_aligned_in_both_dtypes():
    rng = np.random.default_rng(4)
    d0 = [int(x) for x in rng.integers(0, 300, 20)]
    inner = [int(x) for x in rng.choice([1, 3, 7, 64], 20)]
    bucket = sorted(int(x) for x in rng.integers(0, 6, 20))
    L = O.Layout(d0, inner, 8, 4, bucket=bucket)
    for p in range(1, 20):
        if bucket[p] != bucket[p - 1]:
            assert L.o[p] % 256 == 0  # 512 B in bf16, 1024 B in fp32
            assert L.o[p] - (L.o[p - 1] + L.dss[p - 1] * L.inner[p - 1]) < 256
        else:
            assert L.o[p] == L.o[p - 1] + L.dss[p - 1] * L.inner[p - 1]
    with pytest.raises(O.OracleError):
        O.Layout([4, 4], [1, 1], 4, 4, bucket=[1, 0])  # buckets must follow registration order


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_bucketed_sharded_grads_equal_dense_sum(dt):
    # one fused sync over several buckets gives each parameter exactly what a
    # single-bucket plan gives it (the gaps between buckets stay +0)
    d0, inner, bucket = [13, 8, 5, 31, 2], [3, 16, 1, 2, 9], [0, 0, 1, 2, 2]
    Lb = O.Layout(d0, inner, 8, 4, bucket=bucket)
    L1 = O.Layout(d0, inner, 8, 4)
    ints, grads = int_grads(L1, 77, dt)
    fb = O.fused_from_grads(Lb, grads, dt)
    out_b = O.apply_grads(Lb, fb, "avg", dt)
    out_1 = O.apply_grads(L1, O.fused_from_grads(L1, grads, dt), "avg", dt)
    assert all(np.array_equal(a, b) for a, b in zip(out_b, out_1))
    for w in range(8):
        data = np.zeros(Lb.slice("f32"), bool)
        for p in range(Lb.P):
            data[Lb.o[p]:Lb.o[p] + Lb.shard_numel(p, w % 4)] = True
        assert (fb[w][~data] == 0).all()
    # the forward path round-trips through bucketed slices as well
    shards = cut_shards(Lb, grads, dt)
    full = O.ag_copy_out(Lb, O.ag_gather(Lb, O.ag_copy_in(Lb, shards, dt, dt), dt), dt)
    for w in range(8):
        d = w // 4
        for p in range(Lb.P):
            rows = np.concatenate([shards[(d * 4 + s) * Lb.P + p] for s in range(4)])
            assert np.array_equal(full[w * Lb.P + p], rows)
