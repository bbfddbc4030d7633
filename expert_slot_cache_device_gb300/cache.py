"""Python-side owner of one expert slot cache over the caller's banks.

The caller supplies the page-locked host banks (per bank, one tensor per layer, entries may
alias or be None for layers that are never driven) and, optionally, the device slot banks;
PyTorch provides whatever device memory the caller did not (slot banks, workspace). Every
step of the decode path runs in libftmoe through the C-ABI binding (``ftmoe``); nothing here
computes any part of it. Synthetic banks for tests and benchmarks are built by
``synthetic.synthetic_cache``.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Union

import numpy as np
import torch

from . import ftmoe as F


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


@dataclasses.dataclass(frozen=True)
class Bank:
    """Per-expert geometry of one bank, as declared to the library: one expert occupies
    ``rows * row_bytes`` bytes. ``dtype`` is a key of ``ftmoe.DTYPES`` (informative; the
    FFN formats check each bank's per-expert bytes against their schema)."""
    name: str
    dtype: str
    rows: int
    row_bytes: int

    @property
    def bytes(self) -> int:
        return self.rows * self.row_bytes


def _as_bank(g) -> Bank:
    return g if isinstance(g, Bank) else Bank(g.name, g.dtype, int(g.rows), int(g.row_bytes))


def check_banks(fmt: Union[str, int], E: int, L: int, S: int, banks: Sequence, host_sources: Sequence[Sequence],
                slot_banks: Optional[Sequence] = None) -> List[Bank]:
    """Host-side validation of caller banks before they reach the library: per bank, L host
    entries, each None or a contiguous uint8 tensor holding E experts of the bank's bytes
    (shape [E, bytes] or any shape with E * bytes elements) on the host; slot banks, when
    given, contiguous uint8 device tensors with S * bytes elements. Raises ValueError."""
    if isinstance(fmt, str):
        if fmt not in F.FORMATS:
            raise ValueError(f"unknown format {fmt!r}")
    elif fmt not in F.FORMATS.values():
        raise ValueError(f"unknown format code {fmt}")
    banks = [_as_bank(g) for g in banks]
    if not 1 <= len(banks) <= F.MAX_BANKS:
        raise ValueError(f"{len(banks)} banks (1..{F.MAX_BANKS})")
    if len(host_sources) != len(banks):
        raise ValueError(f"host_sources has {len(host_sources)} entries for {len(banks)} banks")
    for b, (g, src) in enumerate(zip(banks, host_sources)):
        if g.dtype not in F.DTYPES:
            raise ValueError(f"bank {g.name}: unknown dtype {g.dtype!r}")
        if g.rows <= 0 or g.row_bytes <= 0:
            raise ValueError(f"bank {g.name}: rows and row_bytes must be positive")
        if len(src) != L:
            raise ValueError(f"bank {g.name}: {len(src)} host entries for {L} layers")
        for l, t in enumerate(src):
            if t is None:
                continue
            if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8:
                raise ValueError(f"bank {g.name} layer {l}: host source must be a uint8 tensor")
            if t.device.type != "cpu" or not t.is_contiguous():
                raise ValueError(f"bank {g.name} layer {l}: host source must be a contiguous host tensor")
            if t.numel() != E * g.bytes:
                raise ValueError(f"bank {g.name} layer {l}: {t.numel()} bytes, expected E * {g.bytes}")
    if slot_banks is not None:
        if len(slot_banks) != len(banks):
            raise ValueError(f"slot_banks has {len(slot_banks)} entries for {len(banks)} banks")
        for g, t in zip(banks, slot_banks):
            if t.dtype != torch.uint8 or not t.is_contiguous() or t.numel() != S * g.bytes:
                raise ValueError(f"slot bank {g.name}: needs a contiguous uint8 tensor of S * {g.bytes} bytes")
    return banks


class ExpertSlotCache:
    """A cache over caller-owned banks.

    fmt           "bf16" | "nvfp4" | "mxfp4" | "fp8" | "q4_0" | "raw" (or an FTMOE_FMT_* code)
    banks         per-bank geometry (``Bank`` or any object with name, dtype, rows, row_bytes),
                  in the schema order of the format
    host_sources  host_sources[b][l]: page-locked uint8 tensor of layer l's E experts of
                  bank b (pin_memory, cudaHostRegister'ed memory), or None for a layer whose
                  bank is not filled; entries may alias (the same tensor for several layers)
    slot_banks    optional device uint8 tensors [S, bytes_b]; allocated here when omitted
    max_pairs     routed pairs (bs * topk) of the largest FFN call (0: no FFN scratch)
    """

    def __init__(self, fmt: Union[str, int], E: int, L: int, S: int, H: int, I: int, banks: Sequence,
                 host_sources: Sequence[Sequence[Optional[torch.Tensor]]], max_pairs: int,
                 slot_banks: Optional[Sequence[torch.Tensor]] = None, device: str = "cuda", stream=None):
        F.lib()
        self.schema = check_banks(fmt, E, L, S, banks, host_sources, slot_banks)
        self.fmt = fmt if isinstance(fmt, str) else {v: k for k, v in F.FORMATS.items()}[fmt]
        self.E, self.L, self.S, self.H, self.I = E, L, S, H, I
        self.nb = len(self.schema)
        self.device = torch.device(device)
        self.max_pairs = max_pairs
        self.cfg = None  # set by the synthetic builder (workload geometry of test caches)
        # host[b]: layer -> tensor for the distinct tensors of bank b (first layer naming each)
        self.host: List[dict] = []
        self.host_ptrs: List[List[int]] = []
        for src in host_sources:
            seen, d = {}, {}
            for l, t in enumerate(src):
                if t is not None and t.data_ptr() not in seen:
                    seen[t.data_ptr()] = l
                    d[l] = t
            self.host.append(d)
            self.host_ptrs.append([t.data_ptr() if t is not None else 0 for t in src])
        self._host_sources = [list(src) for src in host_sources]  # keep the caller's tensors alive
        if slot_banks is None:
            slot_banks = [torch.empty((S, g.bytes), dtype=torch.uint8, device=self.device) for g in self.schema]
        self.slots = [t.view(S, g.bytes) for t, g in zip(slot_banks, self.schema)]
        code = F.FORMATS[self.fmt]
        self.ws_bytes = F.ftmoe_cache_workspace_bytes(code, self.nb, E, L, S, H, I, max_pairs)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        specs = [dict(name=g.name, dtype=F.DTYPES[g.dtype], rows=g.rows, row_bytes=g.row_bytes,
                      host_src=self.host_ptrs[b], dev_slots=self.slots[b].data_ptr())
                 for b, g in enumerate(self.schema)]
        self._specs, self._keep = F.make_bank_specs(specs)
        self.handle = F.ftmoe_cache_create(self._specs, self.nb, code, E, L, S, H, I, max_pairs,
                                           self.workspace.data_ptr(), self.ws_bytes, _stream(stream))

    def close(self, release: bool = False):
        """Destroy the library handle; ``release`` also drops the references this object holds
        to the host banks, slot banks and workspace (so their memory can be freed)."""
        if getattr(self, "handle", None):
            F.ftmoe_cache_destroy(self.handle)
            self.handle = None
        if release:
            self.host, self.host_ptrs, self._host_sources = [], [], []
            self.slots, self.workspace = [], None

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
        S = self.S
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
        cap = max(1, min(self.E, self.S))
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
    def host_tensor(self, b: int, layer: int) -> torch.Tensor:
        """Layer `layer`'s host bank b viewed as [E, bytes_b]."""
        t = self._host_sources[b][layer]
        if t is None:
            raise ValueError(f"bank {b} of layer {layer} is not filled")
        return t.view(self.E, self.schema[b].bytes)

    def host_expert_bytes(self, b: int, layer: int, e: int) -> np.ndarray:
        return self.host_tensor(b, layer)[e].numpy()

    def expert_host_ptrs(self, layer: int, e: int) -> List[int]:
        """Host addresses of expert e's bytes in every bank of `layer` (for the oracle)."""
        return [self.host_ptrs[b][layer] + e * g.bytes for b, g in enumerate(self.schema)]

    @property
    def bytes_per_expert(self) -> int:
        return sum(g.bytes for g in self.schema)
