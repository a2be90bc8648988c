"""Seeded synthetic workloads: shapes, mesh sizes and random tensors.

This module holds none of the method's arithmetic (no chunking, no offsets,
no sums): it only names the workloads and draws seeded random values. Shard
sizes are passed in by the caller, computed by whichever side (the library's
plan or the test oracle's) is under test. Both the product tests and the
oracle tests draw their inputs from here.

Workloads (parameter shapes in registration order):

* ``tiny_fsdp``: rank_size 4, shard_size 4; fp32 params (7,8) (16,8) (5,)
  (3,4), N(0,1) params and grads. Dim 0 is ragged, some shards are empty.
* ``hsdp_2x4_llama``: rank_size 8, shard_size 4 (mesh (2,4)); one Llama-style
  decoder layer with hidden 4096, FFN 11008: q,k,v,o 4096x4096, gate,up
  11008x4096, down 4096x11008, two RMSNorm (4096,). bf16 N(0, 0.02).
* ``ragged_fsdp``: rank_size 8, shard_size 8; 64 bf16 params whose dim 0 is
  [4099, 11003, 1..7] then 55 SplitMix64 draws ``r % 12289 + 1`` and whose
  dim 1 is ``{1,128,4096}[r % 3]`` (1 means a vector), SplitMix64 seeded with
  3. Grads and params N(0,1).
* ``pure_tp_compat``: rank_size 8, shard_size 1 (AllReduce only); 2000 bf16
  params: 88 x (128,4096), 800 x (4096,), 1112 x (1024,). Grads N(0, 1e-3),
  params N(0, 0.02).
* ``large_hsdp``: rank_size 16, shard_size 8 (mesh (2,8)); one 70B-class GQA
  decoder layer, hidden 8192, FFN 28672, 64 q / 8 kv heads: q,o 8192x8192,
  k,v 1024x8192, gate,up 28672x8192, down 8192x28672, two norms (8192,).
  bf16 N(0, 0.02).

Seeds: workload k (1-based, in the order above) draws params from seed
1000k+1 and grads from seed 1000k+2; every virtual rank draws its own values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MASK64 = (1 << 64) - 1


def splitmix64(seed: int):
    """SplitMix64 (Steele, Lea, Flood 2014): a Weyl-sequence state advanced
    by the golden-ratio constant, finalised by two xor-shift-multiply rounds
    and a last xor-shift. Yields 64-bit unsigned integers."""
    state = seed & MASK64
    while True:
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        yield z ^ (z >> 31)


def _ragged_shapes():
    g = splitmix64(3)
    d0 = [4099, 11003, 1, 2, 3, 4, 5, 6, 7]
    d0 += [next(g) % 12289 + 1 for _ in range(55)]
    d1 = [(1, 128, 4096)[next(g) % 3] for _ in range(64)]
    return tuple((a,) if b == 1 else (a, b) for a, b in zip(d0, d1))


def _llama_layer(h, kv, ffn):
    return ((h, h), (kv, h), (kv, h), (h, h), (ffn, h), (ffn, h), (h, ffn), (h,), (h,))


@dataclass(frozen=True)
class Workload:
    key: str
    title: str
    rank_size: int
    shard_size: int
    shapes: tuple
    param_dtype: str
    grad_dtype: str
    param_std: float
    grad_std: float
    index: int
    names: tuple = field(default=())

    @property
    def seed_params(self):
        return 1000 * self.index + 1

    @property
    def seed_grads(self):
        return 1000 * self.index + 2

    @property
    def n_params(self):
        return len(self.shapes)

    @property
    def d0(self):
        return [s[0] for s in self.shapes]

    @property
    def inner(self):
        return [int(np.prod(s[1:], dtype=np.int64)) if len(s) > 1 else 1 for s in self.shapes]

    @property
    def numel_per_rank(self):
        return int(sum(a * b for a, b in zip(self.d0, self.inner)))

    def describe(self):
        return (f"{self.title}: rank_size={self.rank_size}, shard_size={self.shard_size}, "
                f"{self.n_params} {self.param_dtype} params, {self.numel_per_rank} elements per rank")


_LLAMA_NAMES = ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj",
                "input_norm", "post_attn_norm")

WORKLOADS = {
    w.key: w
    for w in [
        Workload("tiny_fsdp", "Tiny FSDP (4 ranks, shard 4, fp32, ragged dim 0)", 4, 4,
                 ((7, 8), (16, 8), (5,), (3, 4)), "f32", "f32", 1.0, 1.0, 1),
        Workload("hsdp_2x4_llama", "HSDP (2,4) mesh, Llama decoder layer h4096/ffn11008", 8, 4,
                 _llama_layer(4096, 4096, 11008), "bf16", "bf16", 0.02, 0.02, 2, _LLAMA_NAMES),
        Workload("ragged_fsdp", "Ragged-heavy FSDP (8 ranks, shard 8, 64 params)", 8, 8,
                 _ragged_shapes(), "bf16", "bf16", 1.0, 1.0, 3),
        Workload("pure_tp_compat", "Pure-TP compat (8 ranks, shard 1, AllReduce only, 2000 params)",
                 8, 1, ((128, 4096),) * 88 + ((4096,),) * 800 + ((1024,),) * 1112,
                 "bf16", "bf16", 0.02, 1e-3, 4),
        Workload("large_hsdp", "Large HSDP (2,8) mesh, 70B-class GQA layer h8192/ffn28672", 16, 8,
                 _llama_layer(8192, 1024, 28672), "bf16", "bf16", 0.02, 0.02, 5, _LLAMA_NAMES),
    ]
}

ORDER = ["tiny_fsdp", "hsdp_2x4_llama", "ragged_fsdp", "pure_tp_compat", "large_hsdp"]


# --------------------------------------------------------------------------
# Random tensors (numpy on the host, torch on a device)
# --------------------------------------------------------------------------

def _np_draw(rng, n, std, dtype):
    x = rng.standard_normal(n, dtype=np.float32) * np.float32(std)
    if dtype == "f32":
        return x
    # bf16 inputs: keep the upper 16 bits of the binary32 draw (truncation).
    # Inputs only need to be bf16 values; how they were drawn is immaterial.
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def np_tensors(sizes, seed, std, dtype):
    """One flat numpy array per entry of ``sizes`` (element counts), drawn in
    order from one seeded PCG64 stream. f32 -> float32, bf16 -> uint16 bits."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [_np_draw(rng, int(n), std, dtype) for n in sizes]


def torch_fill_(tensors, seed, std, dtype):
    """Fill existing flat device tensors in order from one seeded generator
    on their device: N(0, std^2) drawn in fp32, then stored in the tensors'
    dtype (bf16 by PyTorch's round-to-nearest conversion)."""
    import torch

    if not tensors:
        return tensors
    gen = torch.Generator(device=tensors[0].device)
    gen.manual_seed(seed)
    for t in tensors:
        n = t.numel()
        if n:
            x = torch.randn(n, generator=gen, device=t.device, dtype=torch.float32)
            t.copy_(x.mul_(std))
            del x
    return tensors


def torch_tensors(sizes, seed, std, dtype, device):
    """One flat torch tensor per entry of ``sizes``, each a separate
    allocation on ``device``, drawn in order from one seeded generator."""
    import torch

    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    out = [torch.empty(int(n), dtype=tdt, device=device) for n in sizes]
    return torch_fill_(out, seed, std, dtype)


def grad_sizes(wl):
    """Element counts of the full per-(rank, param) gradients, index w*P + p."""
    return [a * b for _ in range(wl.rank_size) for a, b in zip(wl.d0, wl.inner)]
