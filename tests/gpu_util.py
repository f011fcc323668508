"""Helpers shared by the GPU parity tests (marshalling only)."""

from __future__ import annotations

import numpy as np

import workloads


def to_dev_bf16(a32: np.ndarray, device="cuda"):
    """float32 array of bf16 values -> contiguous CUDA bf16 tensor (bit exact)."""
    import torch

    bits = workloads.bf16_bits(a32)
    return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16).contiguous()


def rel_fro(got: np.ndarray, want: np.ndarray) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def mu_close(mu_gpu: np.ndarray, x: np.ndarray, mu_ref: np.ndarray):
    """|mu_gpu - mu_ref| <= 1e-6 * max(|mu_ref|, mean |x|) per column (the binding tolerance for mu)."""
    scale = np.maximum(np.abs(mu_ref), np.abs(x).mean(axis=0))
    err = np.abs(np.asarray(mu_gpu, np.float64) - mu_ref)
    return bool(np.all(err <= 1e-6 * scale + 1e-30)), float(np.max(err / (scale + 1e-30)))
