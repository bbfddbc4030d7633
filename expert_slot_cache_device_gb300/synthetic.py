"""Caches over seeded synthetic banks (tests and benchmarks).

Builds page-locked host banks with the value distributions of ``workload`` and wraps them in
an :class:`ExpertSlotCache`; the cache itself takes any caller banks. Nothing here computes
any part of the decode step.
"""
from __future__ import annotations

from typing import Sequence

import torch

from . import workload as wl
from .cache import ExpertSlotCache


def synthetic_host_banks(cfg: wl.Config, host_layers: Sequence[int] = (0,), alias_all: bool = False,
                         fill: bool = True, device: str = "cuda", gen: str = "device"):
    """host_sources[b][l] for the banks of ``cfg``: one page-locked [E, bytes_b] tensor per
    filled layer (default layer 0 only, as the copy benchmark drives a single layer), None for
    the others; ``alias_all`` gives every layer one shared tensor (long multi-layer traces)."""
    layers = [0] if alias_all else list(host_layers)
    sources = []
    for b, g in enumerate(wl.bank_schema(cfg)):
        made = {}
        for l in layers:
            t = torch.empty((cfg.E, g.bytes), dtype=torch.uint8, pin_memory=True)
            if fill and gen == "device":
                wl.fill_bank_device(cfg, b, t, device=device)
            elif fill:
                wl.fill_bank(cfg, b, t.numpy())
            made[l] = t
        if alias_all:
            sources.append([made[0]] * cfg.L)
        else:
            sources.append([made.get(l) for l in range(cfg.L)])
    return sources


def synthetic_cache(cfg: wl.Config, max_pairs: int, host_layers: Sequence[int] = (0,), alias_all: bool = False,
                    fill: bool = True, device: str = "cuda", stream=None, gen: str = "device") -> ExpertSlotCache:
    """An :class:`ExpertSlotCache` over synthetic banks of ``cfg`` (``cache.cfg`` = cfg)."""
    sources = synthetic_host_banks(cfg, host_layers, alias_all, fill, device, gen)
    cache = ExpertSlotCache(cfg.fmt, cfg.E, cfg.L, cfg.S, cfg.H, cfg.I, wl.bank_schema(cfg), sources, max_pairs,
                            device=device, stream=stream)
    cache.cfg = cfg
    return cache


def release_memory() -> None:
    """Return cached device memory and cached page-locked host blocks to the system (between
    workloads of one benchmark run, so their banks are not all held at once)."""
    import gc

    gc.collect()
    if torch.cuda.is_available():
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    if hasattr(torch._C, "_host_emptyCache"):
        torch._C._host_emptyCache()
