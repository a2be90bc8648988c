"""Buffers and call sequence of one HSDP unit (all W virtual ranks on one GPU).

``HsdpUnit`` allocates, with PyTorch, every per-rank buffer the data path
uses (the caller owns device memory, as the C ABI requires), binds them once,
and issues the C-ABI calls in the order of the pages' forward and backward:

* unshard (forward pre-hook): all-gather copy-in (optionally fused with the
  all-gather), all-gather, copy-out ("Hyper通信掩盖方案" PR #758 write-up
  §二.1, §四.1);
* reduce_grads (post-backward): the fused reduce-scatter + all-reduce into
  the fp32 fused buffer, then applying the gradients to the actual shards
  (§二.1 AllReduceParamGroup, §二.3 wait_and_apply_grads);
* reduce_grads_unfused: reduce-scatter copy-in, ReduceScatter, AllReduce,
  apply (the unfused reference path of §二.4).

No arithmetic happens here; every step is one kernel of the library.
"""
from __future__ import annotations

import torch

from . import capi as C

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _empty(numel, dtype, device, role=None):
    return torch.empty(int(numel), dtype=TORCH_DT[dtype], device=device)


class HsdpUnit:
    def __init__(self, plan: C.Plan, param_dt="bf16", grad_dt="bf16", ag_dt=None, device="cuda",
                 with_unfused=False, alloc=None, backward_only=False):
        """backward_only: allocate only the gradient sync's buffers (grads,
        fused regions, shard gradients; the RS input with with_unfused);
        the forward calls are then unavailable."""
        self.plan = plan
        self.param_dt, self.grad_dt = param_dt, grad_dt
        self.ag_dt = ag_dt or param_dt
        self.device = torch.device(device)
        alloc = alloc or _empty
        W, S, P = plan.W, plan.S, plan.P
        sl_ag = plan.slice_numel(self.ag_dt)
        sl_f = plan.slice_numel("f32")
        dev = self.device
        self.backward_only = bool(backward_only)
        if self.backward_only:
            self.shards, self.ag_out, self.full = [], [], []
        else:
            self.shards = [alloc(plan.shard_numel(p, w % S), param_dt, dev, "shards") for w in range(W)
                           for p in range(P)]
            self.ag_out = [alloc(S * sl_ag, self.ag_dt, dev, "ag_output") for _ in range(W)]
            self.full = [alloc(plan.numel(p), self.ag_dt, dev, "full_params") for _ in range(W) for p in range(P)]
        self.grads = [alloc(plan.numel(p), grad_dt, dev, "grads") for _ in range(W) for p in range(P)]
        self.fused = [alloc(sl_f, "f32", dev, "fused") for _ in range(W)]
        self.shard_grads = [alloc(plan.shard_numel(p, w % S), grad_dt, dev, "shard_grads") for w in range(W) for p in range(P)]
        self.b_shards = self.b_ag = self.b_full = None
        if not self.backward_only:
            self.b_shards = plan.bind("shards", param_dt, self.shards)
            self.b_ag = plan.bind("ag_output", self.ag_dt, self.ag_out)
            self.b_full = plan.bind("full_params", self.ag_dt, self.full)
        self.b_grads = plan.bind("grads", grad_dt, self.grads)
        self.b_fused = plan.bind("fused", "f32", self.fused)
        self.b_shard_grads = plan.bind("shard_grads", grad_dt, self.shard_grads)
        self.rs_in = None
        if with_unfused:
            sl_g = plan.slice_numel(grad_dt)
            self.rs_in = [alloc(S * sl_g, grad_dt, dev, "rs_input") for _ in range(W)]
            self.b_rs_in = plan.bind("rs_input", grad_dt, self.rs_in)

    # ---------------------------------------------------------- forward
    def ag_copy_in(self, fuse_gather=True, stream=None):
        C.fsdp_ag_copy_in(self.plan, self.b_shards, self.b_ag, fuse_gather, stream)

    def ag_gather(self, stream=None):
        C.fsdp_ag_gather(self.plan, self.b_ag, stream)

    def ag_copy_out(self, stream=None):
        C.fsdp_ag_copy_out(self.plan, self.b_ag, self.b_full, stream)

    def unshard_direct(self, stream=None):
        """All three forward steps in one kernel, no gathered buffer."""
        C.fsdp_ag_unshard(self.plan, self.b_shards, self.b_full, stream)

    def unshard(self, fuse_gather=True, stream=None):
        self.ag_copy_in(fuse_gather, stream)
        if not fuse_gather:
            self.ag_gather(stream)
        self.ag_copy_out(stream)

    # --------------------------------------------------------- backward
    def rs_ar_reduce(self, stream=None):
        C.fsdp_rs_ar_reduce(self.plan, self.b_grads, self.b_fused, stream)

    def apply_grads(self, op="avg", accumulate=False, stream=None):
        C.fsdp_apply_grads(self.plan, self.b_fused, op, self.b_shard_grads, accumulate, stream)

    def reduce_grads(self, op="avg", accumulate=False, stream=None):
        self.rs_ar_reduce(stream)
        self.apply_grads(op, accumulate, stream)

    def reduce_grads_one_pass(self, op="avg", accumulate=False, stream=None):
        """reduce_grads with the apply folded into the fused reduce (the same
        bits in the fused buffer and the shard gradients, one pass)."""
        C.fsdp_rs_ar_reduce_apply(self.plan, self.b_grads, self.b_fused, op, self.b_shard_grads, accumulate,
                                  stream)

    def reduce_grads_unfused(self, op="avg", stream=None):
        assert self.rs_in is not None, "built without the unfused path"
        C.fsdp_rs_copy_in(self.plan, self.b_grads, self.b_rs_in, stream)
        C.fsdp_rs_reduce(self.plan, self.b_rs_in, op, self.b_fused, stream)
        C.fsdp_ar_reduce(self.plan, self.b_fused, op, stream)
        # the collectives already scaled (AVG): apply only unpads and rounds
        C.fsdp_apply_grads(self.plan, self.b_fused, "sum", self.b_shard_grads, False, stream)

    def step(self, op="avg", fuse_gather=True, stream=None):
        """One pass of the whole hot path: unshard, then gradient sync."""
        self.unshard(fuse_gather, stream)
        self.reduce_grads(op, stream=stream)

    # unfused halves, for the pipelined backward
    def rs(self, op="avg", stream=None):
        """Shard-domain ReduceScatter: copy-in, then the shard-group sum."""
        C.fsdp_rs_copy_in(self.plan, self.b_grads, self.b_rs_in, stream)
        C.fsdp_rs_reduce(self.plan, self.b_rs_in, op, self.b_fused, stream)

    def ar(self, op="avg", stream=None):
        """Replicate-domain AllReduce of the fused buffer, in place."""
        C.fsdp_ar_reduce(self.plan, self.b_fused, op, stream)

    def capture_step(self, op="avg", fuse_gather=True, warmup=2):
        """Records one step into a CUDA graph (after `warmup` eager steps on a
        side stream, which also fixes every launch's grid) and returns it;
        graph.replay() then issues the whole step with one launch."""
        side = torch.cuda.Stream(device=self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            for _ in range(warmup):
                self.step(op, fuse_gather)
        torch.cuda.current_stream(self.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.step(op, fuse_gather)
        return graph

    def close(self):
        for b in [self.b_shards, self.b_ag, self.b_full, self.b_grads, self.b_fused, self.b_shard_grads]:
            if b is not None:
                b.close()
        if self.rs_in is not None:
            self.b_rs_in.close()


class BackwardPipeline:
    """Gradient sync of a stack of HSDP units (one per layer) overlapped with
    the backward computation, in the order of the pages' backward hook
    ("Hyper通信掩盖方案" PR #758 write-up §二.2, the 4-step pipeline), on
    three streams: the compute stream (the caller's current stream), a
    shard-domain stream for ReduceScatter, a replicate-domain stream for the
    fused AllReduce. Layers are visited last to first. After layer L's
    gradients are produced:

      step 1: the compute stream waits for layer L+1's ReduceScatter;
      step 2: pure-FSDP layers (dp_size 1) apply their RS result at once;
      step 3: layer L's ReduceScatter is issued on the shard stream;
      step 4: layer L+1's fused AllReduce is issued on the replicate stream.

    At the end (the root's delay_apply_reduce_grads) the compute stream
    waits for the last ReduceScatter and every AllReduce and applies the
    remaining layers. With fused=True each layer's RS + AR run as the single
    fused kernel on the shard stream and are applied at the end. No call
    blocks the host; finish() waits on the host with a time limit."""

    def __init__(self, units, op="avg", fused=False, comm_blocks=0, sync_priority=-1, one_pass=False):
        """comm_blocks > 0 caps the thread blocks of every sync kernel the
        pipeline issues on its sync streams while backward compute may still
        run beside it (fsdp_plan_set_grid_limit; the reduces then run one
        block per SM), leaving the other SMs to the backward compute; the
        compute should leave those SMs free (torch's cuBLAS SM carveout does
        that for GEMMs). The syncs issued after the last layer's backward
        (layer 0's ReduceScatter or fused sync, the root's AllReduce) and
        the applies on the compute stream have nothing to share the GPU
        with and run uncapped. one_pass (fused only): each layer's sync is the fused reduce
        with the apply folded in (fsdp_rs_ar_reduce_apply) on the shard
        stream, so nothing is left to apply at the root (same bits).
        sync_priority is the sync streams' priority:
        -1 (high, the default) places their blocks as soon as SMs free up;
        0 (the compute stream's) lets compute blocks go first."""
        self.units = list(units)
        self.op = op
        self.fused = fused
        self.comm_blocks = comm_blocks
        self.one_pass = bool(one_pass) and bool(fused)
        dev = self.units[0].device if self.units else torch.device("cuda")
        self.rs_stream = torch.cuda.Stream(device=dev, priority=sync_priority)
        self.ar_stream = torch.cuda.Stream(device=dev, priority=sync_priority)
        self.log = []  # (step, layer) in issue order

    def _apply(self, L, stream=None):
        u = self.units[L]
        # unfused results are already scaled by the collectives (AVG);
        # the fused buffer holds the raw sum
        op = self.op if self.fused else "sum"
        # apply runs on the compute stream: the whole GPU, not the sync cap
        u.plan.set_grid_limit(0)
        C.fsdp_apply_grads(u.plan, u.b_fused, op, u.b_shard_grads, False, stream)
        u.plan.set_grid_limit(self.comm_blocks)
        self.log.append(("apply", L))

    def run(self, backward_compute):
        """backward_compute(L) issues layer L's backward on the current
        stream (it produces units[L].grads). Returns the event that marks
        the end of the whole sync on the compute stream."""
        for u in self.units:
            u.plan.set_grid_limit(self.comm_blocks)
        try:
            return self._run(backward_compute)
        finally:
            for u in self.units:
                u.plan.set_grid_limit(0)

    def _run(self, backward_compute):
        comp = torch.cuda.current_stream()
        n = len(self.units)
        ev_rs = [None] * n
        ev_ar = []
        pending_apply = []
        for L in reversed(range(n)):
            backward_compute(L)
            self.log.append(("compute", L))
            ev_grad = comp.record_event()
            prev = L + 1 if L + 1 < n else None
            if prev is not None and not self.fused:
                comp.wait_event(ev_rs[prev])                       # step 1
                self.log.append(("wait_rs", prev))
                if self.units[prev].plan.D == 1:                   # step 2
                    self._apply(prev, comp)
            self.rs_stream.wait_event(ev_grad)                     # step 3
            if L == 0:  # no backward compute left beside it
                self.units[L].plan.set_grid_limit(0)
            with torch.cuda.stream(self.rs_stream):
                if self.one_pass:
                    self.units[L].reduce_grads_one_pass(self.op)
                elif self.fused:
                    self.units[L].rs_ar_reduce()
                else:
                    self.units[L].rs(self.op)
            self.log.append(("rs", L))
            ev_rs[L] = self.rs_stream.record_event()
            if self.one_pass:
                self.log.append(("apply", L))
            elif self.fused:
                pending_apply.append(L)
            elif prev is not None and self.units[prev].plan.D > 1:  # step 4
                self.ar_stream.wait_event(ev_rs[prev])
                with torch.cuda.stream(self.ar_stream):
                    self.units[prev].ar(self.op)
                self.log.append(("ar", prev))
                ev_ar.append(self.ar_stream.record_event())
                pending_apply.append(prev)
        # root: the last layer visited (0) and every pending AllReduce
        if n:
            comp.wait_event(ev_rs[0])
            self.log.append(("wait_rs", 0))
            if not self.fused:
                if self.units[0].plan.D == 1:
                    self._apply(0, comp)
                else:
                    self.ar_stream.wait_event(ev_rs[0])
                    with torch.cuda.stream(self.ar_stream):
                        self.units[0].ar(self.op)
                    self.log.append(("ar", 0))
                    ev_ar.append(self.ar_stream.record_event())
                    pending_apply.append(0)
        for ev in ev_ar:
            comp.wait_event(ev)
        for L in pending_apply:
            self._apply(L, comp)
        return comp.record_event()

    def check_status(self):
        """Reads (and clears) every layer's plan status word after the sync
        has finished; raises if a wait inside a capped-grid sync kernel ran
        out (its layer's results are then undefined)."""
        bad = {L: st for L, st in ((L, u.plan.status()) for L, u in enumerate(self.units)) if st}
        if bad:
            raise RuntimeError(f"gradient sync: a wait inside the kernel ran out (layer: status bits) {bad}")

    @staticmethod
    def finish(event, timeout_s=60.0, poll_s=0.001):
        """Waits on the host for `event` for at most timeout_s seconds;
        raises TimeoutError instead of blocking forever."""
        import time

        deadline = time.monotonic() + timeout_s
        while not event.query():
            if time.monotonic() > deadline:
                raise TimeoutError(f"gradient sync not finished after {timeout_s} s")
            time.sleep(poll_s)
