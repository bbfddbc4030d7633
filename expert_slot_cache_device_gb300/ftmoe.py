"""Thin ctypes binding of libftmoe (see include/ftmoe.h for every contract).

Functions keep the C names and only marshal arguments: device pointers and streams
are plain integers (``tensor.data_ptr()``, ``torch.cuda.Stream.cuda_stream``). Every
non-zero status raises :class:`FtmoeError` with the library's message. Loading fails
loudly when the compiled library is missing; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
# FTMOE_CHECKED=1 loads the bounds-checked debug build (build.build(check=True)) instead
LIB_PATH = os.path.join(_HERE, "libftmoe_check.so" if os.environ.get("FTMOE_CHECKED") == "1" else "libftmoe.so")

OK = 0
ERR_INVALID_ARG, ERR_CAPACITY, ERR_ID_RANGE, ERR_CUDA, ERR_FORMAT, ERR_STATE = -1, -2, -3, -4, -5, -6
ERR_NAMES = {0: "OK", -1: "INVALID_ARG", -2: "CAPACITY", -3: "ID_RANGE", -4: "CUDA", -5: "FORMAT", -6: "STATE"}
FMT_RAW, FMT_BF16, FMT_NVFP4, FMT_MXFP4, FMT_FP8, FMT_Q4_0 = 0, 1, 2, 3, 4, 5
FORMATS = {"raw": FMT_RAW, "bf16": FMT_BF16, "nvfp4": FMT_NVFP4, "mxfp4": FMT_MXFP4, "fp8": FMT_FP8,
           "q4_0": FMT_Q4_0}
DT_U8, DT_BF16, DT_F16, DT_E4M3, DT_E8M0, DT_F32, DT_Q4_0 = 0, 1, 2, 3, 4, 5, 6
DTYPES = {"u8": DT_U8, "bf16": DT_BF16, "f16": DT_F16, "e4m3": DT_E4M3, "e8m0": DT_E8M0, "f32": DT_F32,
          "q4_0": DT_Q4_0}
COPY_FUSED, COPY_PER_BANK, COPY_ENGINE = 0, 1, 2
FFN_AUTO, FFN_ROWS, FFN_MMA, FFN_TC05 = 0, 1, 2, 3
DEBUG_WAIT_NS, DEBUG_FFN_SKIP_STAGE = 1, 2
MAX_BANKS = 8

EXPORTS = [
    "ftmoe_cache_workspace_bytes", "ftmoe_cache_create", "ftmoe_cache_destroy", "ftmoe_ensure_experts",
    "ftmoe_copy_missing", "ftmoe_expert_ffn", "ftmoe_set_copy_mode", "ftmoe_cache_get_state",
    "ftmoe_cache_set_state", "ftmoe_get_miss_list", "ftmoe_get_device_status", "ftmoe_h2d_stream_copy",
    "ftmoe_last_error", "ftmoe_expert_ffn_noalloc", "ftmoe_ensure_experts_hybrid", "ftmoe_hybrid_fetch_fraction",
    "ftmoe_expert_ffn_hybrid", "ftmoe_cpu_expert_ffn", "ftmoe_prefetch_layer", "ftmoe_prefill_layers",
    "ftmoe_measure_link", "ftmoe_measure_cpu_moe", "ftmoe_moe_backend_decision", "ftmoe_get_counters",
    "ftmoe_set_ffn_kernels", "ftmoe_ffn_kernels_for", "ftmoe_measure_cpu_read", "ftmoe_set_debug",
]
BACKEND_OFFLOAD, BACKEND_HYBRID = 0, 1
NOALLOC_SCRATCH_BYTES = 16 << 20


class FtmoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"ftmoe error {code} ({ERR_NAMES.get(code, '?')}): {msg}")
        self.code = code


class BankSpec(ctypes.Structure):
    _fields_ = [
        ("name", ctypes.c_char_p),
        ("dtype", ctypes.c_int32),
        ("rows", ctypes.c_int64),
        ("row_bytes", ctypes.c_int64),
        ("host_src", ctypes.POINTER(ctypes.c_void_p)),
        ("dev_slots", ctypes.c_void_p),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libftmoe.so (built by ``expert_slot_cache_device_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first (python -m expert_slot_cache_device_gb300.build)")
    L = ctypes.CDLL(LIB_PATH)
    i32, u32, P, sz = ctypes.c_int32, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_size_t
    sig = {
        "ftmoe_cache_workspace_bytes": [i32, i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)],
        "ftmoe_cache_create": [ctypes.POINTER(BankSpec), i32, i32, i32, i32, i32, i32, i32, i32, P, sz, P,
                               ctypes.POINTER(P)],
        "ftmoe_cache_destroy": [P],
        "ftmoe_ensure_experts": [P, i32, P, i32, i32, P, P],
        "ftmoe_copy_missing": [P, P],
        "ftmoe_expert_ffn": [P, P, i32, P, P, i32, P, P],
        "ftmoe_set_copy_mode": [P, i32],
        "ftmoe_set_ffn_kernels": [P, i32],
        "ftmoe_set_debug": [P, i32, ctypes.c_int64],
        "ftmoe_ffn_kernels_for": [P, i32, i32, P],
        "ftmoe_cache_get_state": [P, P, P, P, P],
        "ftmoe_cache_set_state": [P, P, P, u32, P],
        "ftmoe_get_miss_list": [P, P, P, P, P],
        "ftmoe_get_device_status": [P, P, P],
        "ftmoe_h2d_stream_copy": [P, P, sz, P],
        "ftmoe_expert_ffn_noalloc": [i32, ctypes.POINTER(P), i32, i32, i32, i32, P, i32, P, P, i32, P, P],
        "ftmoe_ensure_experts_hybrid": [P, i32, P, i32, i32, i32, ctypes.c_float, P, P, P],
        "ftmoe_hybrid_fetch_fraction": [ctypes.c_double, ctypes.c_double, P],
        "ftmoe_expert_ffn_hybrid": [P, P, i32, P, P, i32, P, P, P],
        "ftmoe_cpu_expert_ffn": [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, i32],
        "ftmoe_prefetch_layer": [P, i32, P],
        "ftmoe_prefill_layers": [P, i32, P, P, i32, i32, P, P, P, P, P],
        "ftmoe_measure_link": [P, P, sz, i32, P, P, P],
        "ftmoe_measure_cpu_moe": [i32, i32, i32, i32, P, P, i32, i32, i32, P],
        "ftmoe_measure_cpu_read": [P, sz, i32, i32, P],
        "ftmoe_moe_backend_decision": [i32, ctypes.c_double, ctypes.c_double, ctypes.c_double, P, P],
        "ftmoe_get_counters": [P, P, i32, P],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.ftmoe_last_error.argtypes = []
    L.ftmoe_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(rc: int) -> int:
    if rc != OK:
        raise FtmoeError(rc, lib().ftmoe_last_error().decode(errors="replace"))
    return rc


def ftmoe_last_error() -> str:
    return lib().ftmoe_last_error().decode(errors="replace")


def ftmoe_cache_workspace_bytes(fmt: int, num_banks: int, E: int, L: int, S: int, H: int, I: int,
                                max_pairs: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().ftmoe_cache_workspace_bytes(fmt, num_banks, E, L, S, H, I, max_pairs, ctypes.byref(out)))
    return out.value


def make_bank_specs(banks: Sequence[dict]):
    """ctypes array of ftmoe_bank_spec from dicts with keys name, dtype (code), rows,
    row_bytes, host_src (list of L integer host addresses, 0 = unfilled), dev_slots
    (integer device address). Returns (array, keepalive)."""
    arr = (BankSpec * len(banks))()
    keep = []
    for i, b in enumerate(banks):
        srcs = (ctypes.c_void_p * len(b["host_src"]))(*[v or None for v in b["host_src"]])
        name = b.get("name", "").encode()
        keep += [srcs, name]
        arr[i] = BankSpec(name, b["dtype"], b["rows"], b["row_bytes"], srcs, b["dev_slots"])
    return arr, keep


def ftmoe_cache_create(specs, num_banks: int, fmt: int, E: int, L: int, S: int, H: int, I: int, max_pairs: int,
                       d_workspace: int, workspace_bytes: int, stream: int) -> int:
    out = ctypes.c_void_p(0)
    _check(lib().ftmoe_cache_create(specs, num_banks, fmt, E, L, S, H, I, max_pairs, d_workspace, workspace_bytes,
                                    stream, ctypes.byref(out)))
    return out.value


def ftmoe_cache_destroy(cache: int) -> None:
    _check(lib().ftmoe_cache_destroy(cache))


def ftmoe_ensure_experts(cache: int, layer: int, d_topk_ids: int, bs: int, topk: int, d_slots_out: int,
                         stream: int) -> None:
    _check(lib().ftmoe_ensure_experts(cache, layer, d_topk_ids, bs, topk, d_slots_out, stream))


def ftmoe_copy_missing(cache: int, stream: int) -> None:
    _check(lib().ftmoe_copy_missing(cache, stream))


def ftmoe_expert_ffn(cache: int, d_x: int, bs: int, d_slots: int, d_weights: int, topk: int, d_y: int,
                     stream: int) -> None:
    _check(lib().ftmoe_expert_ffn(cache, d_x, bs, d_slots, d_weights, topk, d_y, stream))


def ftmoe_set_copy_mode(cache: int, mode: int) -> None:
    _check(lib().ftmoe_set_copy_mode(cache, mode))


def ftmoe_set_ffn_kernels(cache: int, kind: int) -> None:
    _check(lib().ftmoe_set_ffn_kernels(cache, kind))


def ftmoe_set_debug(cache: int, what: int, value: int) -> None:
    """Test settings (bounded-wait limit, a stage left unfilled); see include/ftmoe.h."""
    _check(lib().ftmoe_set_debug(cache, what, value))


def ftmoe_ffn_kernels_for(cache: int, bs: int, topk: int) -> int:
    kind = ctypes.c_int32(0)
    _check(lib().ftmoe_ffn_kernels_for(cache, bs, topk, ctypes.byref(kind)))
    return kind.value


def ftmoe_cache_get_state(cache: int, h_owner: int, h_stamp: int, h_clock: int, stream: int) -> None:
    _check(lib().ftmoe_cache_get_state(cache, h_owner, h_stamp, h_clock, stream))


def ftmoe_cache_set_state(cache: int, h_owner: int, h_stamp: int, clock: int, stream: int) -> None:
    _check(lib().ftmoe_cache_set_state(cache, h_owner, h_stamp, clock, stream))


def ftmoe_get_miss_list(cache: int, h_ids: int, h_slots: int, h_m: int, stream: int) -> None:
    _check(lib().ftmoe_get_miss_list(cache, h_ids, h_slots, h_m, stream))


def ftmoe_get_device_status(cache: int, h_status: int, stream: int) -> None:
    _check(lib().ftmoe_get_device_status(cache, h_status, stream))


def ftmoe_h2d_stream_copy(d_dst: int, h_src: int, nbytes: int, stream: int) -> None:
    _check(lib().ftmoe_h2d_stream_copy(d_dst, h_src, nbytes, stream))


def ftmoe_expert_ffn_noalloc(fmt: int, d_slot_banks, S: int, H: int, I: int, d_x: int, bs: int, d_slots: int,
                             d_weights: int, topk: int, d_y: int, stream: int) -> None:
    """Allocation-free expert FFN (fixed device scratch inside the library)."""
    banks = (ctypes.c_void_p * len(d_slot_banks))(*d_slot_banks)
    _check(lib().ftmoe_expert_ffn_noalloc(fmt, banks, len(d_slot_banks), S, H, I, d_x, bs, d_slots, d_weights,
                                          topk, d_y, stream))


def ftmoe_ensure_experts_hybrid(cache: int, layer: int, d_topk_ids: int, bs: int, topk: int, max_fetch: int,
                                fetch_fraction: float, d_slots_out: int, d_counts: int, stream: int) -> None:
    _check(lib().ftmoe_ensure_experts_hybrid(cache, layer, d_topk_ids, bs, topk, max_fetch, fetch_fraction,
                                             d_slots_out, d_counts, stream))


def ftmoe_hybrid_fetch_fraction(pcie_gbps: float, cpu_gbps: float) -> float:
    out = ctypes.c_float(0.0)
    _check(lib().ftmoe_hybrid_fetch_fraction(pcie_gbps, cpu_gbps, ctypes.byref(out)))
    return out.value


def ftmoe_expert_ffn_hybrid(cache: int, d_x: int, bs: int, d_slots: int, d_weights: int, topk: int, d_addend: int,
                            d_y: int, stream: int) -> None:
    _check(lib().ftmoe_expert_ffn_hybrid(cache, d_x, bs, d_slots, d_weights, topk, d_addend, d_y, stream))


def ftmoe_cpu_expert_ffn(fmt: int, H: int, I: int, bs: int, topk: int, h_topk_ids: int, h_slots: int,
                         h_layer_banks, bank_bytes, h_x: int, h_weights: int, h_y: int, threads: int = 0) -> None:
    """Host CPU executor of the hybrid path (all pointers are host addresses)."""
    banks = (ctypes.c_void_p * len(h_layer_banks))(*h_layer_banks)
    bb = (ctypes.c_int64 * len(bank_bytes))(*bank_bytes)
    _check(lib().ftmoe_cpu_expert_ffn(fmt, H, I, bs, topk, h_topk_ids, h_slots, banks, bb, h_x, h_weights, h_y,
                                      threads))


def ftmoe_prefetch_layer(cache: int, layer: int, stream: int) -> None:
    _check(lib().ftmoe_prefetch_layer(cache, layer, stream))


def ftmoe_prefill_layers(cache: int, layers: Sequence[int], d_topk_ids: Sequence[int], bs: int, topk: int,
                         d_x: Sequence[int], d_weights: Sequence[int], d_y: Sequence[int], compute_stream: int,
                         copy_stream: int) -> None:
    """Per-step device pointers are passed as host arrays of addresses."""
    n = len(layers)
    if not (len(d_topk_ids) == len(d_x) == len(d_weights) == len(d_y) == n):
        raise ValueError("one id, x, weight and y pointer per pipeline step")
    lay = (ctypes.c_int32 * n)(*layers)
    arr = lambda v: (ctypes.c_void_p * n)(*v)
    _check(lib().ftmoe_prefill_layers(cache, n, lay, arr(d_topk_ids), bs, topk, arr(d_x), arr(d_weights),
                                      arr(d_y), compute_stream, copy_stream))


def ftmoe_measure_link(h_src: int, d_dst: int, nbytes: int, reps: int, stream: int):
    """Returns (memcpy GB/s, SM read GB/s)."""
    a, b = ctypes.c_double(0), ctypes.c_double(0)
    _check(lib().ftmoe_measure_link(h_src, d_dst, nbytes, reps, stream, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def ftmoe_measure_cpu_moe(fmt: int, H: int, I: int, E: int, layer_banks: Sequence[int], bank_bytes: Sequence[int],
                          experts: int, threads: int, reps: int) -> float:
    nb = len(layer_banks)
    out = ctypes.c_double(0)
    _check(lib().ftmoe_measure_cpu_moe(fmt, H, I, E, (ctypes.c_void_p * nb)(*layer_banks),
                                       (ctypes.c_int64 * nb)(*bank_bytes), experts, threads, reps,
                                       ctypes.byref(out)))
    return out.value


def ftmoe_measure_cpu_read(h_buf: int, nbytes: int, threads: int, reps: int) -> float:
    """STREAM-style host memory read ceiling (GB/s) over the host buffer at h_buf."""
    out = ctypes.c_double(0)
    _check(lib().ftmoe_measure_cpu_read(h_buf, nbytes, threads, reps, ctypes.byref(out)))
    return out.value


def ftmoe_moe_backend_decision(fmt: int, link_gbps: float, cpu_gbps: float, threshold: float = 0.0):
    """Returns (backend, fetch_fraction)."""
    be, fr = ctypes.c_int32(0), ctypes.c_float(0)
    _check(lib().ftmoe_moe_backend_decision(fmt, link_gbps, cpu_gbps, threshold, ctypes.byref(be), ctypes.byref(fr)))
    return be.value, fr.value


def ftmoe_get_counters(cache: int, reset: bool, stream: int):
    """Returns (ensure calls, distinct ids looked up, fetched misses)."""
    out = (ctypes.c_uint64 * 3)()
    _check(lib().ftmoe_get_counters(cache, out, 1 if reset else 0, stream))
    return int(out[0]), int(out[1]), int(out[2])
