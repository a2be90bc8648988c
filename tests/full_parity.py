"""Element-by-element parity of a whole HSDP unit with the CPU oracle, at
sizes too large for one oracle call (tens of GB per buffer kind).

Every output element of the data path depends on the inputs of one
parameter only, and within a parameter every column (a fixed index into the
non-dim-0 dims) is laid out, gathered, reduced and applied independently of
the others: the chunk rows, shard ranges and padding rows are the same for
any number of columns ("FSDP dim-0 uneven-sharding RFC" §6.4). So the oracle
is run on pieces of the plan, each a plan of its own:

  * a group of consecutive small parameters (their padded regions are
    contiguous in every slice, at the whole plan's offsets minus the group's
    first offset), or
  * a block of columns of one large parameter (same rows, fewer columns).

Each piece gets host copies of its inputs from the GPU, the oracle's whole
steps (copy-in, gather, copy-out; RS copy-in + fused reduce, apply), and
every output byte of the piece is compared with the GPU's bytes at the
place the oracle's layout of the whole plan gives it. The slice tails past
the last parameter (the oracle writes +0 there) are compared with zeros.
Together the pieces and the tails cover every byte of every output buffer.
Pieces run on a thread pool: the oracle's C calls, the device-to-host copies
and numpy's comparisons release the GIL, and each oracle call stays the
plain single-threaded loop.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle as O

from gpu_util import to_np

# elements over all ranks per piece (~128 MB of bf16 gradients)
PIECE_ELEMS = 64 * 1024 * 1024


def pieces(L, budget=None):
    """(params, c0, c1): a group of whole parameters (c0 = c1 = None) or
    columns [c0, c1) of one parameter."""
    budget = budget or PIECE_ELEMS
    out, group, size = [], [], 0
    for p in range(L.P):
        n = L.numel(p) * L.W
        if n > budget and L.inner[p] > 1:
            if group:
                out.append((group, None, None))
                group, size = [], 0
            ic = max(1, budget // max(1, int(L.d0[p]) * L.W))
            for c0 in range(0, int(L.inner[p]), ic):
                out.append(([p], c0, min(int(L.inner[p]), c0 + ic)))
            continue
        if group and size + n > budget:
            out.append((group, None, None))
            group, size = [], 0
        group.append(p)
        size += n
    if group:
        out.append((group, None, None))
    return out


def _sub_layout(L, ps, c0, c1):
    width = [int(L.inner[q]) if c0 is None else c1 - c0 for q in ps]
    Ls = O.Layout([int(L.d0[q]) for q in ps], width, L.W, L.S)
    # the piece is sharded exactly like its parameters in the whole plan
    for i, q in enumerate(ps):
        assert Ls.dss[i] == L.dss[q] and np.array_equal(Ls.off[i], L.off[q]) and np.array_equal(Ls.len[i], L.len[q])
    if c0 is None:
        assert np.array_equal(Ls.o, L.o[ps[0]:ps[-1] + 2] - L.o[ps[0]])
    return Ls, width


def _cols(t, rows, inner, c0, c1):
    """Host copy of columns [c0, c1) of a (rows, inner) device tensor."""
    if c0 is None:
        return to_np(t)
    return to_np(t.view(int(rows), int(inner))[:, c0:c1].contiguous())


def _host_inputs(L, ps, c0, c1, tensors, rows_of):
    """Per (w, q in ps) host copies of a per-(rank, param) input, in the
    oracle's order (w major)."""
    out = []
    for w in range(L.W):
        if c0 is None:
            parts = [tensors[w * L.P + q] for q in ps]
            sizes = [int(t.numel()) for t in parts]
            flat = to_np(torch.cat(parts)) if sum(sizes) else to_np(parts[0][:0])
            out.extend(np.split(flat, np.cumsum(sizes)[:-1]))
        else:
            q = ps[0]
            out.append(_cols(tensors[w * L.P + q], rows_of(w, q), L.inner[q], c0, c1))
    return out


def _same(got, exp, what):
    g = np.ascontiguousarray(got).view(np.uint8)
    e = np.ascontiguousarray(exp).view(np.uint8)
    if g.shape != e.shape or not np.array_equal(g, e):
        bad = -1 if g.shape != e.shape else int(np.argmax(g != e))
        raise AssertionError(f"{what}: {g.size} bytes, first difference at byte {bad}")


def _region(L, Ls, ps, c0, c1, t_row, row_len, s_row):
    """The piece's part of one slice row: from the GPU row t_row (a device
    tensor of the whole plan's row) and the oracle row s_row (host, the
    piece's row). Returns (got, expected) host arrays."""
    if c0 is None:
        a, b = int(L.o[ps[0]]), int(L.o[ps[-1] + 1])
        return to_np(t_row[a:b]), s_row[:Ls.sum_padded]
    q = ps[0]
    dss, inner = int(L.dss[q]), int(L.inner[q])
    a = int(L.o[q])
    got = to_np(t_row[a:a + dss * inner].view(dss, inner)[:, c0:c1].contiguous())
    return got, s_row[:dss * (c1 - c0)].reshape(dss, c1 - c0)


def check_forward_piece(L, unit, piece, gathered=True):
    ps, c0, c1 = piece
    Ls, _ = _sub_layout(L, ps, c0, c1)
    pdt, adt = unit.param_dt, unit.ag_dt
    S, W, P = L.S, L.W, L.P
    shards = _host_inputs(L, ps, c0, c1, unit.shards, lambda w, q: L.len[q, w % S])
    ag = O.ag_gather(Ls, O.ag_copy_in(Ls, shards, pdt, adt), adt)
    full = O.ag_copy_out(Ls, ag, adt)
    if gathered:
        sl, sls = L.slice(adt), Ls.slice(adt)
        for w in range(W):
            for s in range(S):
                got, exp = _region(L, Ls, ps, c0, c1, unit.ag_out[w][s * sl:(s + 1) * sl], sl,
                                   ag[w][s * sls:(s + 1) * sls])
                _same(got, exp, f"ag_output rank {w} slice {s} params {ps[0]}..{ps[-1]} cols {c0}:{c1}")
    for w in range(W):
        for i, q in enumerate(ps):
            got = _cols(unit.full[w * P + q], L.d0[q], L.inner[q], c0, c1)
            _same(got, full[w * len(ps) + i].reshape(got.shape), f"full param {q} rank {w} cols {c0}:{c1}")


def check_backward_piece(L, unit, piece, op):
    ps, c0, c1 = piece
    Ls, _ = _sub_layout(L, ps, c0, c1)
    gdt = unit.grad_dt
    S, W, P = L.S, L.W, L.P
    grads = _host_inputs(L, ps, c0, c1, unit.grads, lambda w, q: L.d0[q])
    fused = O.fused_from_grads(Ls, grads, gdt)
    sf = L.slice("f32")
    for w in range(W):
        got, exp = _region(L, Ls, ps, c0, c1, unit.fused[w], sf, fused[w])
        _same(got, exp, f"fused rank {w} params {ps[0]}..{ps[-1]} cols {c0}:{c1}")
    sg = O.apply_grads(Ls, fused, op, gdt)
    for w in range(W):
        for i, q in enumerate(ps):
            got = _cols(unit.shard_grads[w * P + q], L.len[q, w % S], L.inner[q], c0, c1)
            _same(got, sg[w * len(ps) + i].reshape(got.shape), f"shard grads param {q} rank {w} cols {c0}:{c1}")


def check_tails(L, unit, forward=True, backward=True):
    """Past the last parameter every slice row and fused region is +0."""
    S, end = L.S, L.sum_padded
    if forward:
        sl = L.slice(unit.ag_dt)
        for w in range(L.W):
            rows = unit.ag_out[w].view(S, sl)[:, end:]
            assert int(rows.view(torch.int16 if unit.ag_dt == "bf16" else torch.int32).count_nonzero()) == 0, \
                ("ag_output tail", w)
    if backward:
        for w in range(L.W):
            assert int(unit.fused[w][end:].view(torch.int32).count_nonzero()) == 0, ("fused tail", w)


def run(fn, items, threads=None):
    threads = threads or max(1, min(12, (os.cpu_count() or 2) - 2))
    with ThreadPoolExecutor(threads) as ex:
        for f in [ex.submit(fn, it) for it in items]:
            f.result()


def check_unit(L, unit, op="avg", forward=True, gathered=True, backward=True, budget=None):
    """Compares every output byte of the unit's last step with the oracle.
    Returns the number of pieces the oracle ran."""
    if torch.cuda.is_available():
        torch.cuda.synchronize()
    O.lib()  # load the oracle once, before the threads
    ps = pieces(L, budget)
    if forward:
        run(lambda pc: check_forward_piece(L, unit, pc, gathered), ps)
    if backward:
        run(lambda pc: check_backward_piece(L, unit, pc, op), ps)
    check_tails(L, unit, forward and gathered, backward)
    return len(ps)
