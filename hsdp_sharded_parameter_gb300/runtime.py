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
                 with_unfused=False, alloc=None):
        self.plan = plan
        self.param_dt, self.grad_dt = param_dt, grad_dt
        self.ag_dt = ag_dt or param_dt
        self.device = torch.device(device)
        alloc = alloc or _empty
        W, S, P = plan.W, plan.S, plan.P
        sl_ag = plan.slice_numel(self.ag_dt)
        sl_f = plan.slice_numel("f32")
        dev = self.device
        self.shards = [alloc(plan.shard_numel(p, w % S), param_dt, dev, "shards") for w in range(W) for p in range(P)]
        self.ag_out = [alloc(S * sl_ag, self.ag_dt, dev, "ag_output") for _ in range(W)]
        self.full = [alloc(plan.numel(p), self.ag_dt, dev, "full_params") for _ in range(W) for p in range(P)]
        self.grads = [alloc(plan.numel(p), grad_dt, dev, "grads") for _ in range(W) for p in range(P)]
        self.fused = [alloc(sl_f, "f32", dev, "fused") for _ in range(W)]
        self.shard_grads = [alloc(plan.shard_numel(p, w % S), grad_dt, dev, "shard_grads") for w in range(W) for p in range(P)]
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

    def close(self):
        for b in [self.b_shards, self.b_ag, self.b_full, self.b_grads, self.b_fused, self.b_shard_grads]:
            b.close()
        if self.rs_in is not None:
            self.b_rs_in.close()
