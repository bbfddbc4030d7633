"""GPU parity of the CUDA path against the CPU oracle (GB300 only).

Every test calls the library through its C-ABI binding and compares with the oracle:
slot tables, miss lists, copied bytes and status codes bit-exactly; FFN outputs
within max-abs 2e-2 and relative L2 1e-2 (bf16 output against the fp64 oracle).
"""
import numpy as np
import pytest
import torch

import oracle
from expert_slot_cache_device_gb300 import ftmoe as F
from expert_slot_cache_device_gb300 import workload as wl
from expert_slot_cache_device_gb300.synthetic import synthetic_cache
from gpu_helpers import assert_ffn_close, bf16_to_f64, oracle_ffn, to_dev, x_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_slot_cache_device_gb300 import build

    build.build()
    oracle.build()


def raw_cfg(E, L, S, nbytes=64, seed=0):
    return wl.Config("raw", "raw", 9, "raw", E, 1, nbytes, 0, L, S, (1,), (1.0,), "uniform", 0.0, seed)


# ------------------------------------------------------------------ ensure + copy


@pytest.mark.parametrize("seed", range(8))
def test_ensure_copy_random_traces(seed):
    rng = np.random.default_rng(100 + seed)
    E = int(rng.integers(2, 40))
    L = int(rng.integers(1, 4))
    k = int(rng.integers(1, min(E, 8) + 1))
    S = int(rng.integers(k, k + 24))
    bs = int(rng.integers(1, 4))
    nbytes = int(rng.choice([16, 48, 64, 4096, 40000]))
    cfg = raw_cfg(E, L, S, nbytes, seed)
    cache = synthetic_cache(cfg, 0, host_layers=range(L))
    orc = oracle.Cache(E, L, S)
    d_slots = torch.empty((bs, k), dtype=torch.int32, device="cuda")
    errors = 0
    for layer, ids in wl.random_trace_ids(seed, 200, E, L, bs, k, [0.0, 1.2][seed % 2]):
        rc, slots, mids, msl = orc.ensure(layer, ids)
        cache.ensure(layer, to_dev(ids), d_slots)
        cache.copy_missing()
        st = cache.status()
        if rc != oracle.OK:
            errors += 1
            assert st == rc
            assert (d_slots.cpu().numpy() == -1).all()
        else:
            assert st == F.OK
            assert np.array_equal(d_slots.cpu().numpy(), slots)
        gi, gs = cache.miss_list()
        assert np.array_equal(gi, mids) and np.array_equal(gs, msl)
        owner, stamp, clock = cache.get_state()
        assert np.array_equal(owner, orc.owner) and np.array_equal(stamp, orc.stamp)
        assert clock == int(orc.clock[0])
        for f, s in zip(mids.tolist(), msl.tolist()):
            want = cache.host[0][f // E][f % E]
            assert torch.equal(cache.slots[0][s].cpu(), want)
    assert errors < 200
    cache.close()


def test_ensure_error_paths():
    cfg = raw_cfg(8, 2, 3)
    cache = synthetic_cache(cfg, 0, host_layers=[0, 1])
    d_slots = torch.empty((1, 4), dtype=torch.int32, device="cuda")
    before = cache.get_state()
    cache.ensure(0, to_dev(np.array([[0, 1, 9, 2]], np.int32)), d_slots)
    assert cache.status() == F.ERR_ID_RANGE
    assert (d_slots.cpu() == -1).all()
    after = cache.get_state()
    assert all(np.array_equal(a, b) for a, b in zip(before[:2], after[:2])) and before[2] == after[2]
    cache.ensure(0, to_dev(np.array([[0, 1, 2, 3]], np.int32)), d_slots)
    assert cache.status() == F.ERR_CAPACITY
    assert cache.get_state()[2] == 0
    # the sticky status keeps the first error until read
    cache.ensure(0, to_dev(np.array([[0, 1, 9, 2]], np.int32)), d_slots)
    cache.ensure(0, to_dev(np.array([[0, 1, 2, 3]], np.int32)), d_slots)
    assert cache.status() == F.ERR_ID_RANGE and cache.status() == F.OK
    # host-detected errors
    with pytest.raises(F.FtmoeError) as ei:
        cache.ensure(2, to_dev(np.array([[0]], np.int32)), d_slots[:, :1])
    assert ei.value.code == F.ERR_INVALID_ARG
    with pytest.raises(F.FtmoeError) as ei:
        cache.set_state(np.array([5, 5, -1], np.int32), np.zeros(3, np.uint32), 0)
    assert ei.value.code == F.ERR_STATE
    # a layer without host banks cannot be driven
    c2 = synthetic_cache(cfg, 0, host_layers=[0])
    with pytest.raises(F.FtmoeError) as ei:
        c2.ensure(1, to_dev(np.array([[0]], np.int32)), d_slots[:, :1])
    assert ei.value.code == F.ERR_INVALID_ARG
    with pytest.raises(F.FtmoeError) as ei:
        F.ftmoe_copy_missing(c2.handle, 0)
    assert ei.value.code == F.ERR_STATE
    cache.close()
    c2.close()


def test_clock_exhausted():
    cfg = raw_cfg(4, 1, 2)
    cache = synthetic_cache(cfg, 0)
    cache.set_state(np.array([0, -1], np.int32), np.array([5, 0], np.uint32), 0xFFFFFFFF)
    d = torch.empty((1, 1), dtype=torch.int32, device="cuda")
    cache.ensure(0, to_dev(np.array([[0]], np.int32)), d)
    assert cache.status() == F.ERR_STATE
    assert cache.get_state()[2] == 0xFFFFFFFF
    cache.close()


def test_large_E_and_S():
    """Sizes beyond one CTA's thread count (E, S > 1024) and many ids per call."""
    E, L, S = 3000, 2, 2500
    cfg = raw_cfg(E, L, S, 32)
    cache = synthetic_cache(cfg, 0, host_layers=[0, 1])
    orc = oracle.Cache(E, L, S)
    rng = np.random.default_rng(5)
    d_slots = torch.empty((64, 32), dtype=torch.int32, device="cuda")
    for call in range(12):
        layer = call % 2
        ids = np.stack([rng.choice(E, 32, replace=False) for _ in range(64)]).astype(np.int32)
        rc, slots, mids, msl = orc.ensure(layer, ids)
        cache.ensure(layer, to_dev(ids), d_slots)
        assert cache.status() == rc
        if rc == oracle.OK:
            assert np.array_equal(d_slots.cpu().numpy(), slots)
        gi, gs = cache.miss_list()
        assert np.array_equal(gi, mids) and np.array_equal(gs, msl)
    owner, stamp, clock = cache.get_state()
    assert np.array_equal(owner, orc.owner) and np.array_equal(stamp, orc.stamp)
    cache.close()


def test_link_probe_copy():
    for n in (16, 48, 1000, 32768 * 3 + 16, 5 * 2 ** 20 + 7):
        src = torch.randint(0, 256, (n,), dtype=torch.uint8).pin_memory()
        dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
        F.ftmoe_h2d_stream_copy(dst.data_ptr(), src.data_ptr(), n, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert torch.equal(dst.cpu(), src)


# ------------------------------------------------------------------ workload points


def install_hits(cache, r):
    """The prepared state's resident experts (slots 0..h-1) get their bytes."""
    for i, e in enumerate(sorted(int(v) for v in r.hits)):
        for b in range(cache.nb):
            cache.slots[b][i].copy_(cache.host[b][0][e])


def _run_point(cache, cfg, bs, mr, modes=(F.COPY_FUSED, F.COPY_PER_BANK, F.COPY_ENGINE), ffn_tokens=None):
    r = wl.make_route(cfg, bs, mr)
    orc = oracle.Cache(cfg.E, cfg.L, cfg.S, r.owner, r.stamp, r.clock)
    rc, slots, mids, msl = orc.ensure(0, r.topk_ids)
    assert rc == oracle.OK and mids.size == r.misses
    d_ids = to_dev(r.topk_ids)
    d_slots = torch.empty_like(d_ids)
    snapshots = []
    install_hits(cache, r)
    for mode in modes:
        cache.set_state(r.owner, r.stamp, r.clock)
        for b in range(cache.nb):
            cache.slots[b][msl.tolist()] = 0  # make stale bytes visible
        cache.set_copy_mode(mode)
        cache.ensure(0, d_ids, d_slots)
        cache.copy_missing()
        assert cache.status() == F.OK
        assert np.array_equal(d_slots.cpu().numpy(), slots)
        gi, gs = cache.miss_list()
        assert np.array_equal(gi, mids) and np.array_equal(gs, msl)
        owner, stamp, clock = cache.get_state()
        assert np.array_equal(owner, orc.owner) and np.array_equal(stamp, orc.stamp) and clock == 1
        for b in range(cache.nb):
            for f, s in zip(mids.tolist(), msl.tolist()):
                assert torch.equal(cache.slots[b][s].cpu(), cache.host[b][0][f % cfg.E]), (mode, b, f, s)
        snapshots.append([cache.slots[b][msl.tolist()].clone() for b in range(cache.nb)])
    for snap in snapshots[1:]:
        assert all(torch.equal(a, b) for a, b in zip(snap, snapshots[0]))
    cache.set_copy_mode(F.COPY_FUSED)
    # FFN over the resolved slots
    d_w = to_dev(r.weights)
    d_x = x_dev(r.x)
    d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
    cache.ffn(d_x, d_slots, d_w, d_y)
    assert cache.status() == F.OK
    y = bf16_to_f64(d_y)
    toks = list(range(bs)) if ffn_tokens is None or ffn_tokens >= bs else \
        sorted(np.random.default_rng(bs).choice(bs, ffn_tokens, replace=False).tolist())
    ref = oracle_ffn(cache, 0, r.topk_ids, r.weights, r.x, toks)
    return assert_ffn_close(y[toks], ref, f"{cfg.key} bs={bs} mr={mr}")


@pytest.mark.parametrize("key", ["c1", "c2", "c3", "c4", "c6", "c7"])
def test_workload_points(key):
    cfg = wl.CONFIGS[key]
    max_pairs = max(cfg.bs_list) * cfg.topk
    cache = synthetic_cache(cfg, max_pairs)
    # every token of every point against the oracle: hot experts run several passes of
    # tokens, and a fault confined to one pass's token lanes must not escape a sample
    for bs in cfg.bs_list:
        for mr in cfg.mr_list:
            _run_point(cache, cfg, bs, mr, ffn_tokens=None)
    cache.close()


@pytest.mark.parametrize("key,bs,mr", [("c2", 16, 1.0), ("c2", 64, 0.5), ("c5", 1, 1.0)])
def test_bf16_tc05_full_size(key, bs, mr):
    """The tcgen05 bf16 pipeline on full-size bf16 layers (every token against the oracle):
    one routed token per expert at bs 16, hot experts over several passes of 16 tokens at
    bs 64, and the decode-trace layer shape (H 4096, I 1536) at bs 1."""
    cfg = wl.CONFIGS[key]
    if key == "c5":  # the trace layer's geometry with a single layer's banks and a small pool
        cfg = wl.scaled(cfg, E=16, S=16, L=2, steps=0, bs_list=(1,), mr_list=(1.0,), ids="uniform")
    cache = synthetic_cache(cfg, bs * cfg.topk)
    cache.set_ffn_kernels(F.FFN_TC05)
    r = wl.make_route(cfg, bs, mr) if key != "c5" else None
    if r is None:
        rng = np.random.default_rng(5)
        ids = np.stack([rng.choice(cfg.E, cfg.topk, replace=False) for _ in range(bs)]).astype(np.int32)
        w = rng.random((bs, cfg.topk)).astype(np.float32)
        w /= w.sum(axis=1, keepdims=True)
        x = wl.f32_to_bf16_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))
    else:
        ids, w, x = r.topk_ids, r.weights, r.x
    slot_of = _install_all(cache, cfg, np.random.default_rng(9)) if cfg.E <= cfg.S else None
    if slot_of is None:  # install only the routed experts, in ascending slots
        used = sorted(set(int(v) for v in ids.reshape(-1)))
        slot_of = {e: i for i, e in enumerate(used)}
        for b in range(cache.nb):
            for e, sl in slot_of.items():
                cache.slots[b][sl].copy_(cache.host[b][0][e])
    slots = np.vectorize(slot_of.get)(ids).astype(np.int32)
    d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
    cache.ffn(x_dev(x), to_dev(slots), to_dev(w), d_y)
    assert cache.status() == F.OK
    assert F.ftmoe_ffn_kernels_for(cache.handle, bs, cfg.topk) == F.FFN_TC05
    ref = oracle_ffn(cache, 0, ids, w, x)
    assert_ffn_close(bf16_to_f64(d_y), ref, f"tc05 {key} bs={bs}")
    cache.close()


# ------------------------------------------------------------------ FFN on small geometries


SCALED = [
    ("bf16", dict(E=12, H=264, I=72, L=2, S=12)),
    ("bf16", dict(E=6, H=1024, I=256, L=2, S=6)),
    ("nvfp4", dict(E=10, H=320, I=96, L=2, S=10)),
    ("nvfp4", dict(E=5, H=2048, I=512, L=2, S=5)),
    ("nvfp4", dict(E=5, H=768, I=256, L=2, S=5)),   # gate_up rows whole in one stage
    ("mxfp4", dict(E=9, H=160, I=96, L=2, S=9)),
    ("mxfp4", dict(E=5, H=576, I=320, L=2, S=5)),
    ("fp8", dict(E=6, H=512, I=512, L=2, S=6)),
    ("fp8", dict(E=5, H=1024, I=1536, L=2, S=5)),
    ("q4_0", dict(E=6, H=512, I=256, L=2, S=6)),
    ("q4_0", dict(E=5, H=1024, I=768, L=2, S=5)),
    ("q4_0", dict(E=5, H=768, I=512, L=2, S=5)),    # gate_up rows whole in one stage
]


@pytest.mark.parametrize("fmt,geo", SCALED)
def test_ffn_small_geometries(fmt, geo):
    """Several tiles with ragged tails, hot experts with more tokens than one pass
    holds, duplicate experts in a row, and a token routed to a single expert."""
    base = {"bf16": "c2", "nvfp4": "c3", "mxfp4": "c4", "fp8": "c6", "q4_0": "c7"}[fmt]
    cfg = wl.scaled(wl.CONFIGS[base], topk=3, **geo)
    bs = 11
    cache = synthetic_cache(cfg, bs * cfg.topk)
    rng = np.random.default_rng(geo["H"])
    ids = rng.integers(0, cfg.E, (bs, cfg.topk)).astype(np.int32)
    ids[:, 0] = 0            # expert 0 gets every token (> one pass of tokens)
    ids[3] = [2, 2, 2]       # duplicates within a row
    w = rng.random((bs, cfg.topk)).astype(np.float32)
    x = wl.f32_to_bf16_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))
    # install the experts by plain copies of the host bytes (FFN tested on its own)
    perm = rng.permutation(cfg.S)
    slot_of = {e: int(perm[e]) for e in range(cfg.E)}
    for b in range(cache.nb):
        for e in range(cfg.E):
            cache.slots[b][slot_of[e]].copy_(cache.host[b][0][e])
    slots = np.vectorize(slot_of.get)(ids).astype(np.int32)
    d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
    cache.ffn(x_dev(x), to_dev(slots), to_dev(w), d_y)
    assert cache.status() == F.OK
    ref = oracle_ffn(cache, 0, ids, w, x)
    assert_ffn_close(bf16_to_f64(d_y), ref, f"{fmt} {geo}")
    # bitwise reproducible
    d_y2 = torch.empty_like(d_y)
    cache.ffn(x_dev(x), to_dev(slots), to_dev(w), d_y2)
    assert torch.equal(d_y, d_y2)
    # a bad slot writes nothing and sets the status
    bad = slots.copy()
    bad[1, 1] = cfg.S
    d_y3 = torch.full_like(d_y, 7.0)
    cache.ffn(x_dev(x), to_dev(bad), to_dev(w), d_y3)
    assert cache.status() == F.ERR_INVALID_ARG
    assert (d_y3.float() == 7.0).all()
    cache.close()


FOLD = [
    ("bf16", F.FFN_ROWS, dict(E=6, H=1024, I=256, L=2, S=6), 3),
    ("bf16", F.FFN_MMA, dict(E=6, H=1024, I=256, L=2, S=6), 3),
    ("bf16", F.FFN_MMA, dict(E=20, H=512, I=768, L=2, S=20), 30),   # 90 pairs, several passes
    ("bf16", F.FFN_TC05, dict(E=6, H=1024, I=256, L=2, S=6), 3),
    ("bf16", F.FFN_TC05, dict(E=4, H=512, I=768, L=2, S=4), 30),    # passes of 16 tokens and a ragged one
    ("nvfp4", F.FFN_AUTO, dict(E=5, H=2048, I=512, L=2, S=5), 4),
    ("q4_0", F.FFN_AUTO, dict(E=6, H=512, I=256, L=2, S=6), 4),
    ("mxfp4", F.FFN_AUTO, dict(E=5, H=576, I=320, L=2, S=5), 4),
    ("mxfp4", F.FFN_AUTO, dict(E=9, H=2880, I=2880, L=2, S=9), 1),  # mxfp4 layer shape at one token
    ("fp8", F.FFN_AUTO, dict(E=5, H=1024, I=1536, L=2, S=5), 4),
]


@pytest.mark.parametrize("fmt,kind,geo,bs", FOLD)
def test_ffn_combine_edge_cases(fmt, kind, geo, bs):
    """The weighted combine in every pipelined kernel family at small and larger calls: a
    token with every position computed elsewhere (y = its addend, rounded once), a token
    routed three times to one expert, the other positions on the GPU, against the oracle plus
    the addend; two calls in a row give identical bits."""
    base = {"bf16": "c2", "nvfp4": "c3", "mxfp4": "c4", "fp8": "c6", "q4_0": "c7"}[fmt]
    cfg = wl.scaled(wl.CONFIGS[base], topk=3, **geo)
    cache = synthetic_cache(cfg, bs * cfg.topk)
    if kind != F.FFN_AUTO:
        cache.set_ffn_kernels(kind)
    rng = np.random.default_rng(geo["E"] * 131 + bs)
    ids = np.stack([rng.choice(cfg.E, cfg.topk, replace=False) for _ in range(bs)]).astype(np.int32)
    if bs > 1:
        ids[1] = [ids[1, 0]] * cfg.topk  # the same expert three times
    w = rng.random((bs, cfg.topk)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)  # router probabilities: |y| stays O(1), as the tolerance assumes
    x = wl.f32_to_bf16_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))
    slot_of = _install_all(cache, cfg, rng)
    slots = np.vectorize(slot_of.get)(ids).astype(np.int32)
    if bs > 2:
        slots[2] = -1  # every position of token 2 elsewhere
        slots[0, 1] = -1
    add = (rng.standard_normal((bs, cfg.H)) * 0.1).astype(np.float32)
    outs = []
    for _ in range(2):
        d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
        d_add = to_dev(add)
        d_x, d_s, d_w = x_dev(x), to_dev(slots), to_dev(w)
        F.ftmoe_expert_ffn_hybrid(cache.handle, d_x.data_ptr(), bs, d_s.data_ptr(), d_w.data_ptr(), cfg.topk,
                                  d_add.data_ptr(), d_y.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert cache.status() == F.OK
        outs.append(d_y.clone())
    assert torch.equal(outs[0], outs[1])
    w_gpu = np.where(slots >= 0, w, 0.0).astype(np.float32)
    ref = oracle_ffn(cache, 0, ids, w_gpu, x) + add.astype(np.float64)
    y = bf16_to_f64(outs[0])
    assert_ffn_close(y, ref, f"{fmt} kind={kind} {geo} bs={bs}")
    if bs > 2:  # the addend alone, rounded once
        want = torch.from_numpy(add[2]).to(torch.bfloat16).float().numpy()
        assert np.array_equal(outs[0][2].float().cpu().numpy(), want)
    cache.close()


def _install_all(cache, cfg, rng):
    perm = rng.permutation(cfg.S)
    slot_of = {e: int(perm[e]) for e in range(cfg.E)}
    for b in range(cache.nb):
        for e in range(cfg.E):
            cache.slots[b][slot_of[e]].copy_(cache.host[b][0][e])
    return slot_of


@pytest.mark.parametrize("geo", [dict(E=6, H=1024, I=256, L=2, S=6), dict(E=5, H=512, I=768, L=2, S=7)])
def test_bf16_ffn_kernel_families(geo):
    """Every bf16 FFN kernel family (CUDA-core rows pipeline, mma.sync pipeline, tcgen05
    pipeline) and the automatic choice against the oracle on one routed batch: a hot expert
    over two passes of eight tokens, duplicates within a row, several 64-row tiles per
    matrix."""
    cfg = wl.scaled(wl.CONFIGS["c2"], topk=4, **geo)
    bs = 13
    cache = synthetic_cache(cfg, bs * cfg.topk)
    rng = np.random.default_rng(geo["I"])
    ids = rng.integers(0, cfg.E, (bs, cfg.topk)).astype(np.int32)
    ids[:, 0] = 1
    ids[4] = [3, 3, 3, 3]
    w = rng.random((bs, cfg.topk)).astype(np.float32)
    x = wl.f32_to_bf16_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))
    slot_of = _install_all(cache, cfg, rng)
    slots = np.vectorize(slot_of.get)(ids).astype(np.int32)
    ref = oracle_ffn(cache, 0, ids, w, x)
    for kind in (F.FFN_TC05, F.FFN_ROWS, F.FFN_MMA, F.FFN_AUTO):
        cache.set_ffn_kernels(kind)
        d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
        cache.ffn(x_dev(x), to_dev(slots), to_dev(w), d_y)
        assert cache.status() == F.OK
        assert_ffn_close(bf16_to_f64(d_y), ref, f"bf16 kernels={kind} {geo}")
    with pytest.raises(F.FtmoeError) as ei:
        cache.set_ffn_kernels(7)
    assert ei.value.code == F.ERR_INVALID_ARG
    cache.close()


def test_ffn_kernel_selector_formats():
    """ROWS / MMA only on bf16 caches; MMA only where the shape has the tensor-core pipeline;
    the AUTO choice as reported by ftmoe_ffn_kernels_for."""
    c2 = synthetic_cache(wl.scaled(wl.CONFIGS["c2"], E=16, L=1, S=16), 128)
    kinds = {bs: F.ftmoe_ffn_kernels_for(c2.handle, bs, 8) for bs in (1, 2, 3, 4, 8)}
    # E = 16: ROWS for 4 <= 8 bs < 32 routed pairs (about one per expert), tcgen05 otherwise
    assert kinds == {1: F.FFN_ROWS, 2: F.FFN_ROWS, 3: F.FFN_ROWS, 4: F.FFN_TC05, 8: F.FFN_TC05}, kinds
    c2.set_ffn_kernels(F.FFN_MMA)
    assert F.ftmoe_ffn_kernels_for(c2.handle, 2, 8) == F.FFN_MMA
    c2.set_ffn_kernels(F.FFN_TC05)
    assert F.ftmoe_ffn_kernels_for(c2.handle, 2, 8) == F.FFN_TC05
    c2.set_ffn_kernels(F.FFN_ROWS)
    assert F.ftmoe_ffn_kernels_for(c2.handle, 8, 8) == F.FFN_ROWS
    c2.close()
    c1 = synthetic_cache(wl.CONFIGS["c1"], 8)  # I = 128: no tensor-core pipeline
    assert F.ftmoe_ffn_kernels_for(c1.handle, 8, 1) == F.FFN_ROWS
    c1.set_ffn_kernels(F.FFN_ROWS)
    c1.set_ffn_kernels(F.FFN_AUTO)
    for kind in (F.FFN_MMA, F.FFN_TC05):
        with pytest.raises(F.FtmoeError) as ei:
            c1.set_ffn_kernels(kind)
        assert ei.value.code == F.ERR_FORMAT
    c1.close()
    nv = synthetic_cache(wl.scaled(wl.CONFIGS["c3"], E=4, H=512, I=256, L=1, S=4), 8)
    nv.set_ffn_kernels(F.FFN_AUTO)
    for kind in (F.FFN_ROWS, F.FFN_MMA, F.FFN_TC05):
        with pytest.raises(F.FtmoeError) as ei:
            nv.set_ffn_kernels(kind)
        assert ei.value.code == F.ERR_FORMAT
    nv.close()


# ------------------------------------------------------------------ multi-step trace


def test_multistep_trace():
    """Every (step, layer) call of the 512-step, 61-layer decode trace: slot tables and
    miss lists bit-exact after every call; every newly filled slot of every call compared
    byte for byte with the expert's bytes in a device copy of the shared host bank (made
    by torch, independent of the library), and on every 8th step also slot by slot; the
    FFN on a sample of calls."""
    cfg = wl.CONFIGS["c5"]
    cache = synthetic_cache(cfg, cfg.topk, alias_all=True)
    dev_bank = [cache.host[b][0].cuda() for b in range(cache.nb)]
    orc = oracle.Cache(cfg.E, cfg.L, cfg.S)
    d_slots = torch.empty((1, cfg.topk), dtype=torch.int32, device="cuda")
    d_y = torch.empty((1, cfg.H), dtype=torch.bfloat16, device="cuda")
    rng = np.random.default_rng(77)
    sample = set(map(tuple, np.stack([rng.integers(0, cfg.steps, 24), rng.integers(0, cfg.L, 24)], 1).tolist()))
    total_miss = total_unique = 0
    for step in range(cfg.steps):
        for layer in range(cfg.L):
            ids, w, x = wl.trace_call(cfg, step, layer)
            rc, slots, mids, msl = orc.ensure(layer, ids)
            assert rc == oracle.OK
            total_unique += np.unique(ids).size
            d_ids = to_dev(ids)
            cache.ensure(layer, d_ids, d_slots)
            cache.copy_missing()
            cache.ffn(x_dev(x), d_slots, to_dev(w), d_y)
            gi, gs = cache.miss_list()
            assert np.array_equal(gi, mids) and np.array_equal(gs, msl), (step, layer)
            assert np.array_equal(d_slots.cpu().numpy(), slots), (step, layer)
            total_miss += mids.size
            if mids.size:  # all newly filled slots of this call in one gather per bank
                d_ms = to_dev(msl.astype(np.int64))
                d_me = to_dev((mids % cfg.E).astype(np.int64))
                for b in range(cache.nb):
                    assert torch.equal(cache.slots[b].index_select(0, d_ms), dev_bank[b].index_select(0, d_me)), \
                        (step, layer, b)
            if step % 8 == 0:
                for b in range(cache.nb):
                    for f, s in zip(mids.tolist(), msl.tolist()):
                        assert torch.equal(cache.slots[b][s], dev_bank[b][f % cfg.E]), (step, layer, b)
            if (step, layer) in sample:
                ref = oracle_ffn(cache, layer, ids, w, x)
                assert_ffn_close(bf16_to_f64(d_y), ref, f"trace step {step} layer {layer}")
        if step % 64 == 63:
            owner, stamp, clock = cache.get_state()
            assert np.array_equal(owner, orc.owner) and np.array_equal(stamp, orc.stamp)
            assert clock == int(orc.clock[0])
    assert cache.status() == F.OK
    assert total_miss > 0
    # the cumulative counters agree with the oracle's trace
    assert cache.counters() == (cfg.steps * cfg.L, total_unique, total_miss)
    cache.close()
