"""Seeded synthetic inputs for the Averis linear layer (shared by tests and bench).

This module only draws random numbers and rounds them to bf16; it holds none
of the method's arithmetic.  Both the CPU oracle's tests and the CUDA path's
tests take their inputs from here, so neither side imports the other.

The pages train Qwen3 models on DCLM ("均值偏置的诅咒与祝福" summary, section
复现评估 / reproduction); neither the data nor the weights are available, so
these generators plant the structure the method targets instead: a coherent
rank-one column mean (the "mean bias" of the analysis sections) plus
Gaussian noise plus sparse spikes.

Recipe (identical for the NumPy and the torch backends, different streams):
  X = 1 mu^T + N(0, 1);   mu_j ~ 8 * N(0, 1);
      then a Bernoulli(1e-3) subset of entries is multiplied by ``spike``
      (x50 for the small and quantize-sweep shapes, x30 for the Qwen3 shapes)
  W ~ N(0, 0.02^2)
  D = 1 nu^T + N(0, (1e-3)^2);   nu_j ~ 1e-2 * N(0, 1)
Every tensor is drawn in float32 and rounded to bf16 (round to nearest even).
NumPy uses Generator(PCG64(seed)); the torch backend uses a seeded
torch.Generator on the target device (used by the benchmark for sizes the
CPU would take minutes to draw).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# ------------------------------------------------------------ shapes ----

#: Single linear fwd+bwd, b=2 s=128 -> l=256, m=n=256.
SMALL = dict(l=256, m=256, n=256, spike=50.0)

#: Qwen3-0.6B-shaped linears at l=8192 (b=4, s=2048): (name, m, n).
QWEN3_06B_LINEARS = (
    ("qkv", 1024, 4096),
    ("o_proj", 2048, 1024),
    ("gate_up", 1024, 6144),
    ("down", 3072, 1024),
)
QWEN3_L = 8192
QWEN3_SPIKE = 30.0

#: Quantize-only sweep: l x m.
QUANT_SWEEP_L = (4096, 16384, 65536)
QUANT_SWEEP_M = (1024, 2048, 4096, 8192)

#: 28-layer stack of the Qwen3 linears at l=16384.
STACK_LAYERS = 28
STACK_L = 16384

#: MoE: hidden 2048, 64 experts, top-8, expert FFN 768, 16384 tokens, Zipf(1.1).
MOE = dict(hidden=2048, experts=64, top_k=8, ffn=768, tokens=16384, zipf=1.1)


# ---------------------------------------------------------- bf16 ----

def bf16_bits(a32: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of float32 values, round to nearest even."""
    a32 = np.ascontiguousarray(a32, dtype=np.float32)
    u = a32.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """float32 values of uint16 bf16 bit patterns (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(a32: np.ndarray) -> np.ndarray:
    """float32 array holding the bf16-rounded values."""
    return bf16_to_f32(bf16_bits(a32))


# ------------------------------------------------------ NumPy backend ----

def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def activation(g: np.random.Generator, l: int, m: int, *, mean_scale=8.0,
               spike=50.0, spike_frac=1e-3) -> np.ndarray:
    """bf16-valued float32 [l, m]: planted rank-one mean + N(0,1) + spikes."""
    mu = (mean_scale * g.standard_normal(m)).astype(np.float32)
    x = g.standard_normal((l, m), dtype=np.float32) + mu[None, :]
    mask = g.random((l, m), dtype=np.float32) < spike_frac
    x = np.where(mask, x * np.float32(spike), x)
    return bf16_round(x)


def weight(g: np.random.Generator, m: int, n: int, *, std=0.02) -> np.ndarray:
    """bf16-valued float32 [m, n] ~ N(0, std^2)."""
    return bf16_round(np.float32(std) * g.standard_normal((m, n), dtype=np.float32))


def output_grad(g: np.random.Generator, l: int, n: int, *, mean_scale=1e-2, noise=1e-3) -> np.ndarray:
    """bf16-valued float32 [l, n]: planted mean nu ~ 1e-2 N(0,1) + N(0, 1e-3^2)."""
    nu = (mean_scale * g.standard_normal(n)).astype(np.float32)
    d = np.float32(noise) * g.standard_normal((l, n), dtype=np.float32) + nu[None, :]
    return bf16_round(d)


@dataclass
class LinearCase:
    x: np.ndarray   # [l, m] float32 holding bf16 values
    w: np.ndarray   # [m, n]
    d: np.ndarray   # [l, n]


def linear_case(seed: int, l: int, m: int, n: int, *, spike=50.0) -> LinearCase:
    g = rng(seed)
    return LinearCase(activation(g, l, m, spike=spike), weight(g, m, n), output_grad(g, l, n))


def moe_routing(seed: int, tokens: int, experts: int, top_k: int, zipf: float) -> np.ndarray:
    """Rows per expert when each token picks ``top_k`` distinct experts with
    probability proportional to rank^(-zipf) (expert e has rank e + 1):
    Gumbel-top-k sampling with NumPy PCG64.  Returns int64 [experts] counts
    (they sum to tokens * top_k); expert-grouped rows are their prefix sums."""
    g = rng(seed)
    logp = -zipf * np.log(np.arange(1, experts + 1, dtype=np.float64))
    keys = logp[None, :] + g.gumbel(size=(tokens, experts))
    picks = np.argpartition(-keys, top_k - 1, axis=1)[:, :top_k]
    return np.bincount(picks.ravel(), minlength=experts).astype(np.int64)


# ------------------------------------------------------ torch backend ----

def torch_linear_case(seed: int, l: int, m: int, n: int, *, spike=50.0, device="cuda"):
    """Same recipe drawn with a seeded torch.Generator on ``device``; bf16 tensors."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    f32 = torch.float32
    mu = 8.0 * torch.randn(m, generator=gen, device=device, dtype=f32)
    x = torch.randn(l, m, generator=gen, device=device, dtype=f32) + mu[None, :]
    mask = torch.rand(l, m, generator=gen, device=device, dtype=f32) < 1e-3
    x = torch.where(mask, x * spike, x).to(torch.bfloat16)
    del mask
    w = (0.02 * torch.randn(m, n, generator=gen, device=device, dtype=f32)).to(torch.bfloat16)
    nu = 1e-2 * torch.randn(n, generator=gen, device=device, dtype=f32)
    d = (1e-3 * torch.randn(l, n, generator=gen, device=device, dtype=f32) + nu[None, :]).to(torch.bfloat16)
    return x, w, d


def torch_activation(seed: int, l: int, m: int, *, spike=50.0, device="cuda"):
    """bf16 [l, m] activation on ``device`` (quantize sweep)."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    mu = 8.0 * torch.randn(m, generator=gen, device=device)
    out = torch.empty(l, m, device=device, dtype=torch.bfloat16)
    step = max(1, (1 << 26) // m)          # bound the float32 temporaries
    for r0 in range(0, l, step):
        r1 = min(l, r0 + step)
        x = torch.randn(r1 - r0, m, generator=gen, device=device) + mu[None, :]
        mask = torch.rand(r1 - r0, m, generator=gen, device=device) < 1e-3
        out[r0:r1] = torch.where(mask, x * spike, x).to(torch.bfloat16)
    return out
