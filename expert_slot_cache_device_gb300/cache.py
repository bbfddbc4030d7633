"""Python-side owner of one expert slot cache: PyTorch provides the page-locked host
banks, the device slot banks and the workspace; every step runs in libftmoe through
the C-ABI binding (``ftmoe``). Nothing here computes any part of the decode step.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

from . import ftmoe as F
from . import workload as wl


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


class ExpertSlotCache:
    """A cache over the banks of ``cfg`` (one workload geometry).

    host_layers: which layers get their own host bank (default: layer 0 only, as the
    copy benchmark drives a single layer); ``alias_all`` makes every layer point at
    one shared host bank (used for long multi-layer traces).
    """

    def __init__(self, cfg: wl.Config, max_pairs: int, host_layers: Sequence[int] = (0,), alias_all: bool = False,
                 fill: bool = True, device: str = "cuda", stream=None, gen: str = "device"):
        F.lib()
        self.cfg = cfg
        self.schema = wl.bank_schema(cfg)
        self.nb = len(self.schema)
        self.device = torch.device(device)
        self.max_pairs = max_pairs
        E, L, S = cfg.E, cfg.L, cfg.S
        # host banks: one pinned tensor per (bank, filled layer)
        self.host: List[dict] = [dict() for _ in range(self.nb)]
        layers = [0] if alias_all else list(host_layers)
        for b, g in enumerate(self.schema):
            for l in layers:
                t = torch.empty((E, g.bytes), dtype=torch.uint8, pin_memory=True)
                if fill and gen == "device":
                    wl.fill_bank_device(cfg, b, t, device=str(self.device))
                elif fill:
                    wl.fill_bank(cfg, b, t.numpy())
                self.host[b][l] = t
        self.host_ptrs = []
        for b in range(self.nb):
            if alias_all:
                ptrs = [self.host[b][0].data_ptr()] * L
            else:
                ptrs = [self.host[b][l].data_ptr() if l in self.host[b] else 0 for l in range(L)]
            self.host_ptrs.append(ptrs)
        self.slots = [torch.empty((S, g.bytes), dtype=torch.uint8, device=self.device) for g in self.schema]
        fmt = F.FORMATS[cfg.fmt]
        self.ws_bytes = F.ftmoe_cache_workspace_bytes(fmt, self.nb, E, L, S, cfg.H, cfg.I, max_pairs)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        specs = [dict(name=g.name, dtype=F.DTYPES[g.dtype], rows=g.rows, row_bytes=g.row_bytes,
                      host_src=self.host_ptrs[b], dev_slots=self.slots[b].data_ptr())
                 for b, g in enumerate(self.schema)]
        self._specs, self._keep = F.make_bank_specs(specs)
        self.handle = F.ftmoe_cache_create(self._specs, self.nb, fmt, E, L, S, cfg.H, cfg.I, max_pairs,
                                           self.workspace.data_ptr(), self.ws_bytes, _stream(stream))

    def close(self):
        if getattr(self, "handle", None):
            F.ftmoe_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ steps
    def ensure(self, layer: int, d_ids: torch.Tensor, d_slots: torch.Tensor, stream=None):
        bs, k = d_ids.shape
        F.ftmoe_ensure_experts(self.handle, layer, d_ids.data_ptr(), bs, k, d_slots.data_ptr(), _stream(stream))

    def copy_missing(self, stream=None):
        F.ftmoe_copy_missing(self.handle, _stream(stream))

    def ffn(self, d_x: torch.Tensor, d_slots: torch.Tensor, d_w: torch.Tensor, d_y: torch.Tensor, stream=None):
        bs, k = d_slots.shape
        F.ftmoe_expert_ffn(self.handle, d_x.data_ptr(), bs, d_slots.data_ptr(), d_w.data_ptr(), k, d_y.data_ptr(),
                           _stream(stream))

    def set_copy_mode(self, mode: int):
        F.ftmoe_set_copy_mode(self.handle, mode)

    def set_ffn_kernels(self, kind: int):
        """FFN kernel family of a bf16 cache: F.FFN_AUTO, F.FFN_ROWS or F.FFN_MMA."""
        F.ftmoe_set_ffn_kernels(self.handle, kind)

    def prefetch_layer(self, layer: int, stream=None):
        F.ftmoe_prefetch_layer(self.handle, layer, _stream(stream))

    def prefill_layers(self, layers, d_ids, d_x, d_w, d_y, compute_stream, copy_stream):
        """Double-buffered prefill: lists of per-step device tensors (ids [bs, k] int32,
        x [bs, H] bf16 bits, w [bs, k] fp32, y [bs, H] bf16 bits)."""
        bs, k = d_ids[0].shape
        F.ftmoe_prefill_layers(self.handle, list(layers), [t.data_ptr() for t in d_ids], bs, k,
                               [t.data_ptr() for t in d_x], [t.data_ptr() for t in d_w],
                               [t.data_ptr() for t in d_y], _stream(compute_stream), _stream(copy_stream))

    # ------------------------------------------------------------------ state
    def get_state(self, stream=None):
        S = self.cfg.S
        owner = np.empty(S, np.int32)
        stamp = np.empty(S, np.uint32)
        clock = np.zeros(1, np.uint32)
        F.ftmoe_cache_get_state(self.handle, owner.ctypes.data, stamp.ctypes.data, clock.ctypes.data, _stream(stream))
        return owner, stamp, int(clock[0])

    def set_state(self, owner, stamp, clock: int, stream=None):
        owner = np.ascontiguousarray(owner, np.int32)
        stamp = np.ascontiguousarray(stamp, np.uint32)
        F.ftmoe_cache_set_state(self.handle, owner.ctypes.data, stamp.ctypes.data, int(clock), _stream(stream))

    def miss_list(self, stream=None):
        cap = max(1, min(self.cfg.E, self.cfg.S))
        ids = np.empty(cap, np.int32)
        slots = np.empty(cap, np.int32)
        m = np.zeros(1, np.int32)
        F.ftmoe_get_miss_list(self.handle, ids.ctypes.data, slots.ctypes.data, m.ctypes.data, _stream(stream))
        return ids[: m[0]].copy(), slots[: m[0]].copy()

    def counters(self, reset: bool = False, stream=None):
        """(ensure calls, distinct ids looked up, fetched misses) since creation or reset."""
        return F.ftmoe_get_counters(self.handle, reset, _stream(stream))

    def status(self, stream=None) -> int:
        st = np.zeros(1, np.int32)
        F.ftmoe_get_device_status(self.handle, st.ctypes.data, _stream(stream))
        return int(st[0])

    # ------------------------------------------------------------------ views
    def host_expert_bytes(self, b: int, layer: int, e: int) -> np.ndarray:
        key = 0 if len(self.host[b]) == 1 and layer not in self.host[b] else layer
        return self.host[b][key][e].numpy()

    def expert_host_ptrs(self, layer: int, e: int) -> List[int]:
        """Host addresses of expert e's bytes in every bank of `layer` (for the oracle)."""
        return [self.host_ptrs[b][layer] + e * g.bytes for b, g in enumerate(self.schema)]

    @property
    def bytes_per_expert(self) -> int:
        return sum(g.bytes for g in self.schema)
