"""CPU oracle of the offloaded expert slot cache — TEST INFRASTRUCTURE ONLY.

Python wrapper (ctypes) around ``liboracle.so``, the plain C restatement of what the
cache's decode step computes (LRU ensure_experts, copy_missing, expert FFN in fp64).
Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
package; the product path never does. It shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRCS = ["lru.c", "copy.c", "ffn.c"]

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_ID_RANGE, ERR_STATE = 0, -1, -2, -3, -6
FMT = {"bf16": 0, "nvfp4": 1, "mxfp4": 2, "fp8": 3, "q4_0": 4}
NUM = {"e2m1": 0, "e4m3": 1, "e8m0": 2, "f16": 3, "bf16": 4}


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (C11, OpenMP); returns its path."""
    srcs = [os.path.join(_HERE, s) for s in _SRCS] + [os.path.join(_HERE, "oracle.h")]
    if not force and os.path.exists(_SO):
        if os.path.getmtime(_SO) >= max(os.path.getmtime(s) for s in srcs):
            return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp]
    cmd += [os.path.join(_HERE, s) for s in _SRCS] + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i32, u32, i64 = ctypes.c_int32, ctypes.c_uint32, ctypes.c_int64
        P = ctypes.c_void_p
        L.orc_ensure.argtypes = [i32, i32, i32, P, P, P, P, i32, P, i32, P, P, P, P]
        L.orc_ensure.restype = ctypes.c_int
        L.orc_ensure_hybrid.argtypes = [i32, i32, i32, P, P, P, P, i32, P, i32, i32, ctypes.c_float, P, P, P, P, P]
        L.orc_ensure_hybrid.restype = ctypes.c_int
        L.orc_rebuild_id2slot.argtypes = [i32, i32, i32, P, P]
        L.orc_rebuild_id2slot.restype = ctypes.c_int
        L.orc_copy_missing.argtypes = [i32, P, P, P, i32, P, P, i32]
        L.orc_copy_missing.restype = None
        L.orc_decode.argtypes = [i32, u32]
        L.orc_decode.restype = ctypes.c_double
        L.orc_weight.argtypes = [i32, i32, P, i32, i32, i64, i64]
        L.orc_weight.restype = ctypes.c_double
        L.orc_bias.argtypes = [i32, i32, P, i32, i32, i64]
        L.orc_bias.restype = ctypes.c_double
        L.orc_expert_ffn.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, i32]
        L.orc_expert_ffn.restype = ctypes.c_int
        L.orc_num_banks.argtypes = [i32]
        L.orc_num_banks.restype = i32
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ptr_array(arrs: Sequence) -> np.ndarray:
    """uint64 array of data pointers (numpy arrays or raw integer addresses)."""
    return np.array([a if isinstance(a, int) else a.ctypes.data for a in arrs], dtype=np.uint64)


class Cache:
    """Oracle LRU state: owner[S], stamp[S], id2slot[L*E], clock."""

    def __init__(self, E: int, L: int, S: int, owner=None, stamp=None, clock: int = 0):
        self.E, self.L, self.S = E, L, S
        self.owner = np.full(S, -1, np.int32) if owner is None else np.array(owner, np.int32)
        self.stamp = np.zeros(S, np.uint32) if stamp is None else np.array(stamp, np.uint32)
        self.clock = np.array([clock], dtype=np.uint32)
        self.id2slot = np.full(E * L, -1, np.int32)
        rc = lib().orc_rebuild_id2slot(E, L, S, _p(self.owner), _p(self.id2slot))
        if rc != OK:
            raise ValueError("inconsistent owner table")

    def ensure(self, layer: int, topk_ids: np.ndarray):
        """Returns (rc, slots[n], miss_ids[m], miss_slots[m])."""
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32).reshape(-1)
        n = ids.size
        slots = np.empty(max(n, 1), np.int32)
        cap = max(min(self.E, n), 1)
        mid = np.empty(cap, np.int32)
        msl = np.empty(cap, np.int32)
        m = np.zeros(1, np.int32)
        rc = lib().orc_ensure(self.E, self.L, self.S, _p(self.owner), _p(self.stamp), _p(self.id2slot),
                              _p(self.clock), layer, _p(ids) if n else 0, n, _p(slots), _p(mid), _p(msl), _p(m))
        k = int(m[0])
        return rc, slots[:n].reshape(np.shape(topk_ids)), mid[:k].copy(), msl[:k].copy()

    def ensure_hybrid(self, layer: int, topk_ids: np.ndarray, max_fetch: int, fetch_fraction: float = 0.0):
        """Returns (rc, slots, miss_ids, miss_slots, (num_indices, num_missing_full))."""
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32).reshape(-1)
        n = ids.size
        slots = np.empty(max(n, 1), np.int32)
        cap = max(min(self.E, n), 1)
        mid = np.empty(cap, np.int32)
        msl = np.empty(cap, np.int32)
        m = np.zeros(1, np.int32)
        counts = np.zeros(2, np.int32)
        rc = lib().orc_ensure_hybrid(self.E, self.L, self.S, _p(self.owner), _p(self.stamp), _p(self.id2slot),
                                     _p(self.clock), layer, _p(ids) if n else 0, n, int(max_fetch),
                                     float(fetch_fraction), _p(slots), _p(mid), _p(msl), _p(m), _p(counts))
        k = int(m[0])
        return (rc, slots[:n].reshape(np.shape(topk_ids)), mid[:k].copy(), msl[:k].copy(),
                (int(counts[0]), int(counts[1])))


def copy_missing(bank_bytes: Sequence[int], host_layer: Sequence, slots: Sequence, E: int,
                 miss_ids: np.ndarray, miss_slots: np.ndarray) -> None:
    bb = np.array(bank_bytes, dtype=np.int64)
    hp = _ptr_array(host_layer)
    sp = _ptr_array(slots)
    mi = np.ascontiguousarray(miss_ids, np.int32)
    ms = np.ascontiguousarray(miss_slots, np.int32)
    lib().orc_copy_missing(len(bb), _p(bb), _p(hp), _p(sp), E, _p(mi) if mi.size else 0,
                           _p(ms) if ms.size else 0, int(mi.size))


def decode(kind: str, bits) -> np.ndarray:
    L = lib()
    b = np.atleast_1d(np.asarray(bits, dtype=np.uint64))
    return np.array([L.orc_decode(NUM[kind], int(v)) for v in b], dtype=np.float64)


def weight(fmt: str, which: int, expert_banks: Sequence[np.ndarray], H: int, I: int, n: int, k: int) -> float:
    ptrs = _ptr_array(expert_banks)
    return lib().orc_weight(FMT[fmt], which, _p(ptrs), H, I, n, k)


def bias(fmt: str, which: int, expert_banks: Sequence[np.ndarray], H: int, I: int, n: int) -> float:
    ptrs = _ptr_array(expert_banks)
    return lib().orc_bias(FMT[fmt], which, _p(ptrs), H, I, n)


def expert_ffn(fmt: str, H: int, I: int, pair_banks: List[Sequence], x_bf16: np.ndarray,
               w: np.ndarray, threads: int = 0) -> np.ndarray:
    """y [bs, H] fp64. ``pair_banks[t * k + j]`` lists the expert's byte buffers per bank
    (numpy arrays or integer host addresses) for routed position (t, j)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    wt = np.ascontiguousarray(w, dtype=np.float32)
    bs, k = wt.shape
    nb = lib().orc_num_banks(FMT[fmt])
    assert len(pair_banks) == bs * k and all(len(p) == nb for p in pair_banks)
    ptrs = _ptr_array([a for p in pair_banks for a in p])
    y = np.zeros((bs, H), dtype=np.float64)
    rc = lib().orc_expert_ffn(FMT[fmt], H, I, bs, k, nb, _p(ptrs), _p(x), _p(wt), _p(y), threads)
    if rc != OK:
        raise ValueError(f"orc_expert_ffn rc={rc}")
    return y
