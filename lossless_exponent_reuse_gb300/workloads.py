"""Seeded synthetic weight sequences for the five workloads.

This module only makes inputs: bf16 weights w_0, w_1, ... of the shapes and
value distributions of sharded MoE training, handed out as flat uint16 bit
patterns.  It holds none of the compression method's arithmetic, and both
the CUDA path and the CPU oracle consume the same bytes it produces.

Update rule (input generation, not the method):
    w_{t+1} = bf16_rne( fp32(w_t) + fp32(step) * z ),  z ~ N(0, 1)
with z drawn from a ``torch.Generator`` seeded by (seed, workload, t).
A "forced" iteration flips bit 7 of every value (the exponent's lowest
bit), so every exponent changes; values drawn from N(0, 0.02) stay finite.

The shapes follow the models named in "CIERA: Cross-Iteration Exponent Reuse
for Lossless Allgather in Sharded MoE Training" (Section 2 setup and Section
4.1: OLMoE-1B-7B with 64 experts per layer, fine-grained MoE variants); the
paper's datasets and trained weights are not used: random weights of those
shapes stand in for them.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import List, Optional, Sequence, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Tensor:
    name: str
    shape: Tuple[int, ...]
    mean: float = 0.0
    sigma: float = 0.02

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload.

    ``tensors`` lists the tensors of each layer; every layer has the same
    tensors.  ``steps`` gives the update step of iterations 1.. (iteration 0
    is the initial draw); ``forced`` names iterations whose exponents are all
    flipped instead of stepped.
    """
    name: str
    tensors: Tuple[Tensor, ...]
    layers: int
    ranks: int
    block: int
    iterations: int
    steps: Tuple[float, ...]
    forced: Tuple[int, ...] = ()
    seed: int = 1234
    # clustered variant: probability that a block of ``block`` values is
    # perturbed at all in an iteration (None = every value perturbed)
    p_block: Optional[float] = None

    @property
    def layer_numel(self) -> int:
        return sum(t.numel for t in self.tensors)

    @property
    def numel(self) -> int:
        return self.layer_numel * self.layers

    def step_of(self, t: int) -> float:
        """Update step used to go from iteration t-1 to iteration t (t >= 1)."""
        return self.steps[(t - 1) % len(self.steps)]


def _experts(n: int, d_model: int, d_ff: int, sigma: float) -> Tuple[Tensor, ...]:
    out = []
    for e in range(n):
        out.append(Tensor(f"expert{e}.gate", (d_ff, d_model), sigma=sigma))
        out.append(Tensor(f"expert{e}.up", (d_ff, d_model), sigma=sigma))
        out.append(Tensor(f"expert{e}.down", (d_model, d_ff), sigma=sigma))
    return tuple(out)


def _olmoe_layer_tensors() -> Tuple[Tensor, ...]:
    attn = tuple(Tensor(f"attn.{p}", (2048, 2048)) for p in ("q", "k", "v", "o"))
    router = (Tensor("router", (64, 2048)),)
    norms = (Tensor("input_norm", (2048,), mean=1.0, sigma=0.01),
             Tensor("post_attn_norm", (2048,), mean=1.0, sigma=0.01))
    return attn + router + norms + _experts(64, 2048, 1024, 0.02)


def workload(cfg: int, variant: str = "") -> Workload:
    """The five workloads (1-based), plus labelled variants.

    1  one 256x512 matrix, N(0,0.02), 4 ranks, block 256, 3 iterations, step 1e-4
    2  one OLMoE MoE layer: 64 experts x {gate,up 2048x1024, down 1024x2048},
       16 ranks, block 4096, 10 iterations, step 1e-5
    3  same layer, warm-up regime: steps 1e-3 and 3e-3, then one iteration with
       every exponent forced to change
    4  16 OLMoE-1B-7B-shaped layers (attention, router, two norms, 64 experts),
       8 ranks, block 4096, 5 iterations, step 3e-5
    5  fine-grained MoE layer: 128 experts x {gate,up 4096x1536, down
       1536x4096}, N(0,0.015), 32 ranks, block 4096, 5 iterations per step,
       steps 2.2e-6 / 2.35e-5 / 3.9e-4
    variant "clustered<p>" (cfg 2 or 5): each block is perturbed with
    probability p and left untouched otherwise.
    variant "experts<k>" (cfg 2, 3 or 5): the same layer cut to its first k
    experts (a smaller case of the same kernels, e.g. for profiling).
    """
    if cfg == 1:
        w = Workload("cfg1_matrix_256x512", (Tensor("w", (256, 512)),), 1, 4, 256, 3,
                     (1e-4,))
    elif cfg == 2:
        w = Workload("cfg2_olmoe_moe_layer", _experts(64, 2048, 1024, 0.02), 1, 16, 4096, 10,
                     (1e-5,))
    elif cfg == 3:
        w = Workload("cfg3_olmoe_moe_layer_warmup", _experts(64, 2048, 1024, 0.02), 1, 16,
                     4096, 4, (1e-3, 3e-3), forced=(3,))
    elif cfg == 4:
        w = Workload("cfg4_olmoe_1b7b_stack", _olmoe_layer_tensors(), 16, 8, 4096, 5, (3e-5,))
    elif cfg == 5:
        w = Workload("cfg5_finegrained_moe_layer", _experts(128, 1536, 4096, 0.015), 1, 32,
                     4096, 16, (2.2e-6,) * 5 + (2.35e-5,) * 5 + (3.9e-4,) * 5)
    else:
        raise ValueError(f"no workload {cfg}")
    for v in filter(None, variant.split(",")):
        if v.startswith("clustered"):
            p = float(v[len("clustered"):])
            w = dataclasses.replace(w, name=f"{w.name}_clustered{p:g}", p_block=p)
        elif v.startswith("experts") and cfg in (2, 3, 5):
            k = int(v[len("experts"):])
            w = dataclasses.replace(w, name=f"{w.name}_experts{k}", tensors=w.tensors[:3 * k])
        else:
            raise ValueError(f"unknown variant {v!r}")
    return w


def small(name: str, shapes: Sequence[Tuple[int, ...]], ranks: int, block: int,
          iterations: int = 3, step: float = 1e-4, sigma: float = 0.02, seed: int = 7,
          forced: Tuple[int, ...] = (), p_block: Optional[float] = None) -> Workload:
    """A small ad-hoc workload for tests (ragged sizes, odd blocks, ...)."""
    ts = tuple(Tensor(f"t{i}", tuple(s), sigma=sigma) for i, s in enumerate(shapes))
    return Workload(name, ts, 1, ranks, block, iterations, (step,), forced=forced, seed=seed,
                    p_block=p_block)


def _seed(*parts) -> int:
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _normal(n: int, mean: float, sigma: float, gen: torch.Generator, device) -> torch.Tensor:
    z = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    return z * sigma + mean


def initial_layer(wl: Workload, layer: int, device="cpu") -> torch.Tensor:
    """Iteration-0 weights of one layer: flat uint16 bit patterns (bucket order)."""
    parts = []
    for i, t in enumerate(wl.tensors):
        g = torch.Generator(device=device)
        g.manual_seed(_seed(wl.seed, wl.name, "init", layer, i))
        parts.append(_normal(t.numel, t.mean, t.sigma, g, device).to(torch.bfloat16))
    return torch.cat(parts).view(torch.uint16) if parts else torch.empty(0, dtype=torch.uint16)


def step_layer(wl: Workload, w: torch.Tensor, layer: int, t: int) -> torch.Tensor:
    """Weights of iteration t (t >= 1) from those of iteration t-1 (uint16 bits)."""
    assert w.dtype == torch.uint16
    if t in wl.forced:
        return (w.view(torch.int16) ^ 0x0080).view(torch.uint16)
    device = w.device
    g = torch.Generator(device=device)
    g.manual_seed(_seed(wl.seed, wl.name, "step", layer, t))
    z = torch.randn(w.numel(), generator=g, device=device, dtype=torch.float32)
    if wl.p_block is not None:
        nb = (w.numel() + wl.block - 1) // wl.block
        keep = (torch.rand(nb, generator=g, device=device) < wl.p_block).to(torch.float32)
        z = z * keep.repeat_interleave(wl.block)[: w.numel()]
    x = w.view(torch.bfloat16).to(torch.float32) + wl.step_of(t) * z
    return x.to(torch.bfloat16).view(torch.uint16)


def layer_offsets(wl: Workload) -> List[Tuple[str, int, int]]:
    """(name, offset, numel) of each tensor inside one layer's flat buffer."""
    out, off = [], 0
    for t in wl.tensors:
        out.append((t.name, off, t.numel))
        off += t.numel
    return out


def sequence(wl: Workload, iterations: int, layer: int = 0, device="cpu"):
    """Yield w_0 .. w_{iterations-1} of one layer (flat uint16 tensors)."""
    w = initial_layer(wl, layer, device)
    yield w
    for t in range(1, iterations):
        w = step_layer(wl, w, layer, t)
        yield w
