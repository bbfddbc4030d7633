"""Seeded synthetic workloads for the offloaded expert slot cache.

This module only *generates inputs*: expert bank bytes, routed top-k ids, router
probabilities, activations and the prepared cache state of the copy benchmark.
It holds none of the cache's, the copy's or the FFN's arithmetic, so both the
CUDA path and the CPU oracle can consume what it makes without sharing code.

Workloads follow the cache-copy benchmark of the FreeToken benchmark guide
("FreeToken MoE 离线推理基准完全指南", section 4: synthetic tensors, bank layout
per format schema, a prepared state where every slot belongs to another layer,
``misses = round(active_unique * miss_rate)`` with
``active_unique = min(E, bs * topk)``).
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional, Sequence

import numpy as np

# --------------------------------------------------------------------------------------
# Workload geometries
# --------------------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Config:
    key: str          # short key used by tests and the bench ("c1".."c5")
    name: str         # descriptive workload name with its sizes
    index: int        # position in the workload list (seeds depend on it)
    fmt: str          # "bf16" | "nvfp4" | "mxfp4"
    E: int            # experts per layer
    topk: int
    H: int            # hidden size
    I: int            # moe intermediate size
    L: int            # layers sharing the flat id space
    S: int            # GPU slots
    bs_list: tuple
    mr_list: tuple
    ids: str          # "top2_logits" | "uniform" | "zipf"
    zipf_a: float
    seed: int
    steps: int = 0            # decode steps of the multi-step trace (0 = single call)
    down_rows_literal: bool = False  # tiny layer declares its down bank as [E, I, H]

    @property
    def bytes_per_expert(self) -> int:
        return sum(b.bytes for b in bank_schema(self))


CONFIGS: Dict[str, Config] = {
    "c1": Config("c1", "tiny_bf16_E8_k2_H256_I128_S4", 0, "bf16", 8, 2, 256, 128, 2, 4,
                 (1,), (1.0,), "top2_logits", 0.0, 0, down_rows_literal=True),
    "c2": Config("c2", "bf16_E128_k8_H2048_I768_L48_S256", 1, "bf16", 128, 8, 2048, 768, 48, 256,
                 (1, 4, 16), (0.0, 0.25, 0.5, 1.0), "uniform", 0.0, 0),
    "c3": Config("c3", "nvfp4_E256_k8_H7168_I2048_L58_S512", 2, "nvfp4", 256, 8, 7168, 2048, 58, 512,
                 (1, 8, 32), (0.1, 0.3, 1.0), "uniform", 0.0, 0),
    "c4": Config("c4", "mxfp4_E128_k4_H2880_I2880_L36_S192", 3, "mxfp4", 128, 4, 2880, 2880, 36, 192,
                 (1, 16, 64), (0.05, 0.5), "zipf", 1.1, 0),
    "c5": Config("c5", "bf16_trace_E256_k8_H4096_I1536_L61_S1024", 4, "bf16", 256, 8, 4096, 1536, 61,
                 1024, (1,), (), "zipf", 1.2, 7, steps=512),
    # GGUF Q4_0 layer: the nvfp4 layer's shape with the Q4_0 bank schema
    "c7": Config("c7", "q4_0_E256_k8_H7168_I2048_L58_S512", 6, "q4_0", 256, 8, 7168, 2048, 58, 512,
                 (1, 8, 32), (0.1, 0.3, 1.0), "uniform", 0.0, 0),
    # block-FP8 layer: the nvfp4 layer's shape with the block-FP8 bank schema
    "c6": Config("c6", "fp8_E256_k8_H7168_I2048_L58_S512", 5, "fp8", 256, 8, 7168, 2048, 58, 512,
                 (1, 8, 32), (0.1, 0.3, 1.0), "uniform", 0.0, 0),
}


def scaled(cfg: Config, **kw) -> Config:
    """A copy of ``cfg`` with some geometry replaced (used for small parity cases)."""
    return dataclasses.replace(cfg, **kw)


# --------------------------------------------------------------------------------------
# Bank schemas (per-expert geometry of every bank, per format)
# --------------------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class BankGeom:
    name: str
    dtype: str        # "bf16" | "u8" | "e4m3" | "f16" | "e8m0"
    rows: int
    row_bytes: int

    @property
    def bytes(self) -> int:
        return self.rows * self.row_bytes


def bank_schema(cfg: Config) -> List[BankGeom]:
    """Per-expert bank geometry, in the schema order of the benchmark guide section 4.2."""
    H, I = cfg.H, cfg.I
    if cfg.fmt == "raw":
        # copy-only cache: one byte bank of H bytes per expert (tiny LRU/copy tests)
        return [BankGeom("rows", "u8", 1, H)]
    if cfg.fmt == "bf16":
        down = BankGeom("down", "bf16", I, 2 * H) if cfg.down_rows_literal else BankGeom("down", "bf16", H, 2 * I)
        return [BankGeom("gate_up", "bf16", 2 * I, 2 * H), down]
    if cfg.fmt == "nvfp4":
        return [
            BankGeom("gate_up_codes", "u8", 2 * I, H // 2),
            BankGeom("gate_up_scales", "e4m3", 2 * I, H // 16),
            BankGeom("gate_up_global", "f16", 2 * I, 2),
            BankGeom("down_codes", "u8", H, I // 2),
            BankGeom("down_scales", "e4m3", H, I // 16),
            BankGeom("down_global", "f16", H, 2),
        ]
    if cfg.fmt == "mxfp4":
        return [
            BankGeom("gate_up_blocks", "u8", H // 2, 2 * I),
            BankGeom("gate_up_scales", "e8m0", H // 32, 2 * I),
            BankGeom("gate_up_bias", "bf16", 2 * I, 2),
            BankGeom("down_blocks", "u8", I // 2, H),
            BankGeom("down_scales", "e8m0", I // 32, H),
            BankGeom("down_bias", "bf16", H, 2),
        ]
    if cfg.fmt == "fp8":
        # block FP8: e4m3 weights [N, K] and one binary32 scale per 128 x 128 block
        return [
            BankGeom("gate_up_weight", "e4m3", 2 * I, H),
            BankGeom("gate_up_scale", "f32", (2 * I + 127) // 128, 4 * ((H + 127) // 128)),
            BankGeom("down_weight", "e4m3", H, I),
            BankGeom("down_scale", "f32", (H + 127) // 128, 4 * ((I + 127) // 128)),
        ]
    if cfg.fmt == "q4_0":
        # GGUF Q4_0: rows of K/32 blocks, 18 bytes each (binary16 scale + 16 nibble bytes)
        return [
            BankGeom("gate_up_q4_0", "q4_0", 2 * I, (H // 32) * 18),
            BankGeom("down_q4_0", "q4_0", H, (I // 32) * 18),
        ]
    raise ValueError(f"unknown format {cfg.fmt!r}")


# --------------------------------------------------------------------------------------
# Value generation helpers
# --------------------------------------------------------------------------------------


def _rng(*words: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(w) & 0xFFFFFFFF for w in words]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bfloat16 bit patterns (finite inputs)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even, saturating float32 -> OCP e4m3fn bytes (uses torch's cast)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


_SEED_BANK = 0xBA4C
FP8_Q_STD = 112.0  # standard deviation of the synthetic block-FP8 codes (before e4m3 rounding)
Q4_D = 0.02 / np.sqrt(21.5)  # Q4_0 block scale: (q - 8) over uniform nibbles has mean square 21.5


def _gen_bank_expert(cfg: Config, b: int, geom: BankGeom, e: int) -> np.ndarray:
    """Bytes of bank ``b`` for expert ``e`` (flat uint8 of ``geom.bytes``)."""
    rng = _rng(cfg.seed, cfg.index, _SEED_BANK, b, e)
    name = geom.name
    if geom.dtype == "u8":
        return rng.integers(0, 256, size=geom.bytes, dtype=np.uint8)
    if geom.dtype == "bf16":
        n = geom.bytes // 2
        std = 0.02
        vals = rng.standard_normal(n, dtype=np.float32) * np.float32(std)
        return f32_to_bf16_bits(vals).view(np.uint8)
    if geom.dtype == "e4m3" and name.endswith("_weight"):
        # block-FP8 weights: N(0, 1) * 112, so a block's largest |value| reaches the top
        # of the e4m3 range (448) the way a max-scaled quantisation does
        vals = rng.standard_normal(geom.bytes, dtype=np.float32) * np.float32(FP8_Q_STD)
        return f32_to_e4m3_bits(vals)
    if geom.dtype == "e4m3":
        vals = np.abs(rng.standard_normal(geom.bytes, dtype=np.float32))
        return f32_to_e4m3_bits(vals)
    if geom.dtype == "f32":
        # block scales: w = q * s has standard deviation ~0.02 * (0.5 + U)
        u = rng.random(geom.bytes // 4)
        return ((0.5 + u) * (0.02 / FP8_Q_STD)).astype(np.float32).view(np.uint8)
    if geom.dtype == "f16":
        # Per-output-row global of nvfp4; sized so the row dot product is O(1):
        # 8.5625 is the mean square of the 16 e2m1 code values, K the reduction length.
        K = cfg.H if name.startswith("gate_up") else cfg.I
        u = rng.random(geom.bytes // 2)
        g = (0.5 + u) / np.sqrt(8.5625 * K)
        return g.astype(np.float16).view(np.uint8)
    if geom.dtype == "e8m0":
        return rng.integers(117, 121, size=geom.bytes, dtype=np.uint8)
    if geom.dtype == "q4_0":
        # uniform nibbles (q - 8 has mean square 21.5); d = (0.5 + U) * Q4_D, so w has a
        # standard deviation near 0.02
        blocks = rng.integers(0, 256, size=(geom.bytes // 18, 18), dtype=np.uint8)
        d = ((0.5 + rng.random(blocks.shape[0])) * Q4_D).astype(np.float16)
        blocks[:, 0:2] = d.view(np.uint8).reshape(-1, 2)
        return blocks.reshape(-1)
    raise ValueError(geom.dtype)


def fill_bank(cfg: Config, b: int, out: np.ndarray, experts: Optional[Sequence[int]] = None,
              threads: int = 8) -> None:
    """Write bank ``b`` of ``cfg`` into ``out`` (uint8, shape [E, bytes_b] or [n, bytes_b]).

    ``experts`` selects which experts' bytes go into the rows of ``out`` (default: all E),
    so tiny parity cases and sampled oracle checks can generate a subset.
    """
    geom = bank_schema(cfg)[b]
    ids = list(range(cfg.E)) if experts is None else list(experts)
    assert out.dtype == np.uint8 and out.shape == (len(ids), geom.bytes), (out.shape, geom)

    def one(i: int) -> None:
        out[i, :] = _gen_bank_expert(cfg, b, geom, ids[i])

    if threads <= 1 or len(ids) <= 1:
        for i in range(len(ids)):
            one(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(len(ids))))


def fill_bank_device(cfg: Config, b: int, out, experts: Optional[Sequence[int]] = None,
                     device: str = "cuda") -> None:
    """Like :func:`fill_bank` but draws the values with torch's seeded Philox generator on
    ``device`` and copies them into ``out`` (a torch uint8 tensor [n, bytes_b], normally
    page-locked host memory). Same value distributions, different (but seeded) draws;
    used for the multi-GiB banks, which the numpy path generates too slowly."""
    import torch

    geom = bank_schema(cfg)[b]
    ids = list(range(cfg.E)) if experts is None else list(experts)
    assert tuple(out.shape) == (len(ids), geom.bytes) and out.dtype == torch.uint8
    gen = torch.Generator(device=device)
    for i, e in enumerate(ids):
        seed = int(np.random.SeedSequence([cfg.seed, cfg.index, _SEED_BANK, b, e, 0xD]).generate_state(1,
                                                                                                      np.uint64)[0])
        gen.manual_seed(seed)
        n = geom.bytes
        if geom.dtype == "u8":
            t = torch.randint(0, 256, (n,), dtype=torch.uint8, device=device, generator=gen)
        elif geom.dtype == "bf16":
            t = (torch.randn(n // 2, device=device, generator=gen) * 0.02).to(torch.bfloat16).view(torch.uint8)
        elif geom.dtype == "e4m3" and geom.name.endswith("_weight"):
            v = (torch.randn(n, device=device, generator=gen) * FP8_Q_STD).clamp(-448.0, 448.0)
            t = v.to(torch.float8_e4m3fn).view(torch.uint8)
        elif geom.dtype == "e4m3":
            v = torch.randn(n, device=device, generator=gen).abs().clamp(max=448.0)
            t = v.to(torch.float8_e4m3fn).view(torch.uint8)
        elif geom.dtype == "f32":
            u = torch.rand(n // 4, device=device, generator=gen, dtype=torch.float64)
            t = ((0.5 + u) * (0.02 / FP8_Q_STD)).to(torch.float32).view(torch.uint8)
        elif geom.dtype == "f16":
            K = cfg.H if geom.name.startswith("gate_up") else cfg.I
            u = torch.rand(n // 2, device=device, generator=gen, dtype=torch.float64)
            t = ((0.5 + u) / np.sqrt(8.5625 * K)).to(torch.float16).view(torch.uint8)
        elif geom.dtype == "e8m0":
            t = torch.randint(117, 121, (n,), dtype=torch.uint8, device=device, generator=gen)
        elif geom.dtype == "q4_0":
            blocks = torch.randint(0, 256, (n // 18, 18), dtype=torch.uint8, device=device, generator=gen)
            u = torch.rand(n // 18, device=device, generator=gen, dtype=torch.float64)
            d = ((0.5 + u) * Q4_D).to(torch.float16).view(torch.uint8).view(-1, 2)
            blocks[:, 0:2] = d
            t = blocks.reshape(-1)
        else:
            raise ValueError(geom.dtype)
        out[i].copy_(t, non_blocking=True)
    torch.cuda.synchronize()


def make_banks(cfg: Config, experts: Optional[Sequence[int]] = None) -> List[np.ndarray]:
    """All banks of one layer as numpy arrays (small configurations only)."""
    ids = list(range(cfg.E)) if experts is None else list(experts)
    out = []
    for b, g in enumerate(bank_schema(cfg)):
        a = np.empty((len(ids), g.bytes), dtype=np.uint8)
        fill_bank(cfg, b, a, ids)
        out.append(a)
    return out


# --------------------------------------------------------------------------------------
# Routing inputs and the prepared benchmark state
# --------------------------------------------------------------------------------------


@dataclasses.dataclass
class Route:
    topk_ids: np.ndarray   # [bs, k] int32, local expert ids
    weights: np.ndarray    # [bs, k] float32 router probabilities
    x: np.ndarray          # [bs, H] uint16 bf16 bit patterns
    active: int            # number of distinct ids
    misses: int            # planned misses for the prepared state
    hits: np.ndarray       # local ids installed as hits by the prepared state (ascending)
    owner: np.ndarray      # [S] int32 prepared owner table (flat ids, -1 empty)
    stamp: np.ndarray      # [S] uint32 prepared stamps
    clock: int             # prepared clock


def zipf_p(E: int, a: float) -> np.ndarray:
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-a)
    return p / p.sum()


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=-1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=-1, keepdims=True)


def _activations(rng: np.random.Generator, bs: int, H: int) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal((bs, H), dtype=np.float32))


def planned_misses(active: int, miss_rate: float) -> int:
    """Python ``round`` (half to even) of active * miss_rate, as the copy benchmark states."""
    return int(round(active * miss_rate))


def _lay_out_ids(rng: np.random.Generator, active_set: np.ndarray, bs: int, k: int,
                 p_active: Optional[np.ndarray]) -> np.ndarray:
    """Place the active set into a [bs, k] id matrix: distinct ids per row, every active
    id at least once; surplus positions redrawn from the active set."""
    a = len(active_set)
    perm = rng.permutation(active_set)
    ids = np.full((bs, k), -1, dtype=np.int64)
    flat = ids.reshape(-1)
    flat[:a] = perm
    for r in range(bs):
        row = ids[r]
        have = set(int(v) for v in row if v >= 0)
        need = k - len(have)
        if need == 0:
            continue
        pool = np.array([v for v in active_set if int(v) not in have], dtype=np.int64)
        if p_active is None:
            pick = rng.choice(pool, size=need, replace=False)
        else:
            pp = np.array([p_active[int(np.where(active_set == v)[0][0])] for v in pool])
            pick = rng.choice(pool, size=need, replace=False, p=pp / pp.sum())
        row[row < 0] = pick
    return ids.astype(np.int32)


def make_route(cfg: Config, bs: int, miss_rate: float, layer: int = 0) -> Route:
    """Routed inputs plus the prepared state for one (bs, miss_rate) point."""
    E, k, S = cfg.E, cfg.topk, cfg.S
    rng = _rng(cfg.seed, cfg.index, bs, int(round(miss_rate * 1000)))
    if cfg.ids == "top2_logits":
        logits = rng.standard_normal((bs, E))
        order = np.argsort(-logits, axis=1, kind="stable")
        topk_ids = order[:, :k].astype(np.int32)
        probs = _softmax_rows(logits)
        weights = np.take_along_axis(probs, topk_ids.astype(np.int64), axis=1).astype(np.float32)
        active = len(np.unique(topk_ids))
    else:
        active = min(E, bs * k)
        if cfg.ids == "uniform":
            p = None
            active_set = np.sort(rng.choice(E, size=active, replace=False))
        else:
            p = zipf_p(E, cfg.zipf_a)
            active_set = np.sort(rng.choice(E, size=active, replace=False, p=p))
        p_active = None if p is None else p[active_set]
        topk_ids = _lay_out_ids(rng, active_set, bs, k, p_active)
        weights = _softmax_rows(rng.standard_normal((bs, k))).astype(np.float32)
    x = _activations(rng, bs, cfg.H)
    m = planned_misses(active, miss_rate)
    uniq = np.unique(topk_ids)
    h = active - m
    hits = np.sort(rng.choice(uniq, size=h, replace=False)) if h > 0 else np.zeros(0, np.int64)
    owner, stamp, clock = prepared_state(cfg, hits, layer)
    return Route(topk_ids, weights, x, active, m, hits.astype(np.int32), owner, stamp, clock)


def prepared_state(cfg: Config, hits: Sequence[int], layer: int = 0):
    """The copy benchmark's prepared state: every slot is owned by another layer
    (slot s holds flat id ``(layer + 1) * E + s``), except that the planned hits of the
    driven layer sit in slots ``0..len(hits)-1`` in ascending id. Stamps and clock are 0."""
    E, S, L = cfg.E, cfg.S, cfg.L
    base = (layer + 1) * E
    if base + S > L * E:
        raise ValueError("prepared state needs L >= layer + 1 + ceil(S / E)")
    owner = (base + np.arange(S)).astype(np.int32)
    for i, e in enumerate(sorted(int(v) for v in hits)):
        owner[i] = layer * E + e
    stamp = np.zeros(S, dtype=np.uint32)
    return owner, stamp, 0


def empty_state(cfg: Config):
    return np.full(cfg.S, -1, dtype=np.int32), np.zeros(cfg.S, dtype=np.uint32), 0


def trace_call(cfg: Config, step: int, layer: int):
    """Ids, router probabilities and activations of one (step, layer) call of the
    multi-step decode trace (bs = 1; k distinct zipf-distributed ids per call)."""
    rng = _rng(cfg.seed, cfg.index, 0x7ACE, step, layer)
    p = zipf_p(cfg.E, cfg.zipf_a)
    ids = rng.choice(cfg.E, size=cfg.topk, replace=False, p=p).astype(np.int32)[None, :]
    weights = _softmax_rows(rng.standard_normal((1, cfg.topk))).astype(np.float32)
    x = _activations(rng, 1, cfg.H)
    return ids, weights, x


def random_trace_ids(seed: int, calls: int, E: int, L: int, bs: int, k: int, zipf_a: float = 0.0):
    """(layer, ids[bs, k]) for ``calls`` random ensure calls (tiny LRU trace tests).
    Ids within a row are distinct; rows may repeat ids across tokens."""
    rng = _rng(seed, 0x1D5, calls, E, L)
    p = zipf_p(E, zipf_a) if zipf_a > 0 else None
    out = []
    for _ in range(calls):
        layer = int(rng.integers(0, L))
        ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(bs)]).astype(np.int32)
        out.append((layer, ids))
    return out
