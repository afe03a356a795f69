"""Seeded synthetic gradient buckets shaped like the LoCo paper's workloads.

This module only draws random numbers into flat buffers; it holds none of
the compression arithmetic.  Both the CUDA path and the CPU oracle are fed
from it (the oracle through host copies of the same bytes).

The paper trains LLaMA-family and Mixtral-style MoE models under FSDP, whose
communication hook hands over a flattened gradient bucket ("LoCo: Low-Bit
Communication Adaptor for Large-scale Model Training", §2 related work on
FSDP hooks, §3.3).  No datasets or weights exist here, so each model is
represented by its parameter shapes only, filled with seeded noise:

* LLM buckets: per tensor sigma = 10**U(-5, -2), values N(0, sigma^2).
* MoE layer: Student-t (nu = 3) noise times 1e-3; chosen experts all zero.
* Flat buckets: N(0, 1e-3^2), optionally with Bernoulli(p) outliers x100.

Seed convention: rank w at step k uses ``seed_for(base, k, w) = base + 1000*k + w``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

CHUNK = 1 << 26  # elements generated per torch call (bounds temporaries)


def seed_for(base: int, step: int, rank: int) -> int:
    return base + 1000 * step + rank


# --------------------------------------------------------------------------
# Parameter layouts (name, numel), in flattening order.
# --------------------------------------------------------------------------

def llama_layout(vocab: int, hidden: int, ffn: int, layers: int, kv_dim: int):
    out = [("embed", vocab * hidden)]
    for i in range(layers):
        out += [
            (f"l{i}.q", hidden * hidden),
            (f"l{i}.k", kv_dim * hidden),
            (f"l{i}.v", kv_dim * hidden),
            (f"l{i}.o", hidden * hidden),
            (f"l{i}.gate", ffn * hidden),
            (f"l{i}.up", ffn * hidden),
            (f"l{i}.down", hidden * ffn),
            (f"l{i}.attn_norm", hidden),
            (f"l{i}.mlp_norm", hidden),
        ]
    out += [("final_norm", hidden), ("head", vocab * hidden)]
    return out


def llama2_7b_layout():
    """Llama-2-7B: 32 layers, hidden 4096, ffn 11008, vocab 32000 (6,738,415,616 params)."""
    return llama_layout(32000, 4096, 11008, 32, 4096)


def tinyllama_layout():
    """TinyLlama-1.1B: 22 layers, hidden 2048, ffn 5632, GQA kv dim 256 (1,100,048,384 params)."""
    return llama_layout(32000, 2048, 5632, 22, 256)


def mixtral_moe_layer_layout(experts: int = 8, hidden: int = 4096, ffn: int = 14336):
    """One Mixtral-8x7B MoE layer: per expert w1, w3 (ffn x hidden) and w2 (hidden x ffn)."""
    out = []
    for e in range(experts):
        out += [(f"e{e}.w1", ffn * hidden), (f"e{e}.w3", ffn * hidden), (f"e{e}.w2", hidden * ffn)]
    return out


def layout_numel(layout) -> int:
    return sum(n for _, n in layout)


# --------------------------------------------------------------------------
# Generators.  `out` is a flat contiguous tensor (fp32 or bf16) on any device.
# --------------------------------------------------------------------------

def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _fill_normal(dst: torch.Tensor, sigma: float, gen: torch.Generator):
    n = dst.numel()
    for s in range(0, n, CHUNK):
        e = min(s + CHUNK, n)
        z = torch.randn(e - s, generator=gen, device=dst.device, dtype=torch.float32)
        z.mul_(sigma)
        dst[s:e].copy_(z)


def fill_llm_grads(out: torch.Tensor, layout, seed: int):
    """Per-tensor N(0, sigma^2) with sigma = 10**U(-5,-2) drawn per tensor."""
    assert out.numel() == layout_numel(layout)
    sig_rng = np.random.default_rng(seed)
    sigmas = 10.0 ** sig_rng.uniform(-5.0, -2.0, size=len(layout))
    gen = _gen(out.device, seed)
    off = 0
    for (name, n), sigma in zip(layout, sigmas):
        _fill_normal(out[off:off + n], float(sigma), gen)
        off += n
    return out


def fill_moe_grads(out: torch.Tensor, layout, seed: int, zero_experts=(3, 7), scale: float = 1e-3,
                   nu: int = 3):
    """Student-t(nu) * scale (t = Z / sqrt(chi2_nu / nu)); tensors of zero_experts all zero."""
    assert out.numel() == layout_numel(layout)
    gen = _gen(out.device, seed)
    off = 0
    for name, n in layout:
        dst = out[off:off + n]
        expert = int(name.split(".")[0][1:])
        if expert in zero_experts:
            dst.zero_()
        else:
            for s in range(0, n, CHUNK):
                e = min(s + CHUNK, n)
                z = torch.randn(e - s, generator=gen, device=out.device, dtype=torch.float32)
                chi2 = torch.zeros_like(z)
                for _ in range(nu):
                    c = torch.randn(e - s, generator=gen, device=out.device, dtype=torch.float32)
                    chi2.addcmul_(c, c)
                z.div_(torch.sqrt(chi2 / nu)).mul_(scale)
                dst[s:e].copy_(z)
        off += n
    return out


def fill_flat_normal(out: torch.Tensor, seed: int, sigma: float = 1e-3, outlier_p: float = 0.0,
                     outlier_mult: float = 100.0):
    """N(0, sigma^2); with outlier_p > 0 a Bernoulli(outlier_p) mask of entries is multiplied."""
    gen = _gen(out.device, seed)
    n = out.numel()
    for s in range(0, n, CHUNK):
        e = min(s + CHUNK, n)
        z = torch.randn(e - s, generator=gen, device=out.device, dtype=torch.float32)
        z.mul_(sigma)
        if outlier_p > 0:
            u = torch.rand(e - s, generator=gen, device=out.device, dtype=torch.float32)
            z = torch.where(u < outlier_p, z * outlier_mult, z)
        out[s:e].copy_(z)
    return out


def fill_uniform(out: torch.Tensor, seed: int, lo: float, hi: float):
    gen = _gen(out.device, seed)
    n = out.numel()
    for s in range(0, n, CHUNK):
        e = min(s + CHUNK, n)
        z = torch.rand(e - s, generator=gen, device=out.device, dtype=torch.float32)
        out[s:e].copy_(z * (hi - lo) + lo)
    return out


# --------------------------------------------------------------------------
# The five workloads (sizes and settings), by name.
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    grad_dtype: torch.dtype
    bits: int
    block: int
    W: int
    steps: int
    kind: str          # "flat", "llm", "moe", "flat_outliers"
    layout: tuple = ()

    def fill(self, out: torch.Tensor, seed: int):
        if self.kind == "flat":
            return fill_flat_normal(out, seed)
        if self.kind == "flat_outliers":
            return fill_flat_normal(out, seed, outlier_p=1e-3)
        if self.kind == "llm":
            return fill_llm_grads(out, self.layout, seed)
        if self.kind == "moe":
            return fill_moe_grads(out, self.layout, seed)
        raise ValueError(self.kind)


FLAT_1M = Workload("flat-fp32-1M", 1 << 20, torch.float32, 4, 256, 4, 8, "flat")
TINYLLAMA = Workload("tinyllama-1.1b-bf16", layout_numel(tinyllama_layout()), torch.bfloat16,
                     8, 128, 8, 4, "llm", tuple(tinyllama_layout()))
LLAMA2_7B = Workload("llama2-7b-bf16", layout_numel(llama2_7b_layout()), torch.bfloat16,
                     4, 256, 8, 1, "llm", tuple(llama2_7b_layout()))
MIXTRAL_MOE = Workload("mixtral-8x7b-moe-layer-bf16", layout_numel(mixtral_moe_layer_layout()),
                       torch.bfloat16, 4, 128, 8, 4, "moe", tuple(mixtral_moe_layer_layout()))


def sweep_workload(n: int, dtype: torch.dtype, bits: int, block: int, W: int) -> Workload:
    return Workload(f"flat-sweep-{n}", n, dtype, bits, block, W, 1, "flat_outliers")


WORKLOADS = {w.name: w for w in (FLAT_1M, TINYLLAMA, LLAMA2_7B, MIXTRAL_MOE)}
