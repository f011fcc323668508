"""Helpers shared by the GPU parity tests (marshalling and tolerances only)."""

from __future__ import annotations

import numpy as np

import workloads

#: binding tolerance of the column mean: 1e-6 relative to |mu_j| ...
MU_REL = 1e-6
#: ... with an absolute floor of MU_REL * 2^-2 * mean_i |x_ij|, which only matters for
#: columns whose mean is below a quarter of their mean magnitude.  A pure relative bound
#: is unattainable for mu_j near 0.  The floor is the error bound of the library's sum:
#: each thread adds groups of up to 8 bf16 values pairwise in binary32 (at most
#: 3 u sum|x| of error per group, u = 2^-24) and accumulates the group sums with
#: compensation, so |mu_gpu - mu| <= u |mu| + 3 u mean|x| + O(u^2) < 1e-6 (|mu| + 2^-2 mean|x|).
MU_FLOOR = 2.0 ** -2


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


def _mu_check(mu_gpu, mu_ref, absmean):
    mu_gpu = np.asarray(mu_gpu, np.float64)
    mu_ref = np.asarray(mu_ref, np.float64)
    err = np.abs(mu_gpu - mu_ref)
    ok = bool(np.all(err <= MU_REL * np.abs(mu_ref) + MU_REL * MU_FLOOR * absmean))
    nz = np.abs(mu_ref) > 0
    worst = float(np.max(err[nz] / np.abs(mu_ref[nz]))) if nz.any() else float(err.max(initial=0.0))
    return ok, worst


def mu_close(mu_gpu: np.ndarray, x: np.ndarray, mu_ref: np.ndarray):
    """(ok, worst relative error on |mu|): |mu_gpu - mu_ref| <= 1e-6 |mu_ref| per column,
    floored as MU_FLOOR states."""
    return _mu_check(mu_gpu, mu_ref, np.abs(np.asarray(x, np.float64)).mean(axis=0))


def mu_close_chunked(mu_gpu: np.ndarray, x: np.ndarray, chunk: int = 4096):
    """mu_close against the float64 column mean of a large x, summed in row chunks."""
    s = np.zeros(x.shape[1])
    a = np.zeros(x.shape[1])
    for r0 in range(0, x.shape[0], chunk):
        xb = np.asarray(x[r0:r0 + chunk], np.float64)
        s += xb.sum(axis=0)
        a += np.abs(xb).sum(axis=0)
    return _mu_check(mu_gpu, s / x.shape[0], a / x.shape[0])
