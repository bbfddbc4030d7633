"""Shared helpers of the GPU parity tests (run on the GPU machine only)."""
import numpy as np
import torch

import oracle
from expert_slot_cache_device_gb300 import workload as wl
from expert_slot_cache_device_gb300.cache import ExpertSlotCache

ATOL = 2e-2   # max |y_gpu - y_oracle| on bf16 outputs
RTOL_L2 = 1e-2  # ||y_gpu - y_oracle||_2 / ||y_oracle||_2


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def x_dev(x_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x_bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


def oracle_ffn(cache: ExpertSlotCache, layer: int, ids: np.ndarray, w: np.ndarray, x_bits: np.ndarray,
               tokens=None, threads: int = 0) -> np.ndarray:
    """Oracle y for the given tokens (default all), reading expert bytes from the host banks."""
    cfg = cache.cfg
    ids = np.asarray(ids)
    tokens = range(ids.shape[0]) if tokens is None else list(tokens)
    pairs = [cache.expert_host_ptrs(layer, int(ids[t, j])) for t in tokens for j in range(ids.shape[1])]
    return oracle.expert_ffn(cfg.fmt, cfg.H, cfg.I, pairs, x_bits[list(tokens)], w[list(tokens)], threads=threads)


def assert_ffn_close(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = ""):
    err = np.abs(y_gpu - y_ref)
    l2 = np.linalg.norm(y_gpu - y_ref) / max(np.linalg.norm(y_ref), 1e-30)
    assert np.isfinite(y_gpu).all(), what
    assert err.max() <= ATOL, f"{what}: max abs err {err.max():.3e} (|y| max {np.abs(y_ref).max():.3f})"
    assert l2 <= RTOL_L2, f"{what}: rel L2 err {l2:.3e}"
    return float(err.max()), float(l2)
