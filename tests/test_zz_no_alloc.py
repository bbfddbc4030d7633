"""The allocation-free FFN entry point (GPU).

ftmoe_expert_ffn_noalloc serves callers that cannot call cudaMalloc — code running
inside a runtime that already owns all device memory, or on a path that must not pay
for an allocation's device synchronisation. Its scratch is a fixed array inside the
library, so this test checks, through the C-ABI, two calls in a row (with different
inputs, so stale scratch from the first call would show) against the CPU oracle and
against ftmoe_expert_ffn for the same slot banks, within the FFN tolerance of the other
tests; positions with slot -1 (computed elsewhere) against ftmoe_expert_ffn_hybrid and
the oracle with those positions left out; that a slot outside [-1, S) leaves the output
untouched; and that an over-sized call is refused. This file is collected last.
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ATOL, RTOL_L2 = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import oracle
    from expert_slot_cache_device_gb300 import build

    build.build()
    oracle.build()


def _close(a, ref: np.ndarray, what: str):
    x = a.float().cpu().numpy().astype(np.float64) if isinstance(a, torch.Tensor) else a
    err = np.abs(x - ref).max()
    l2 = np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30)
    assert np.isfinite(x).all() and err <= ATOL and l2 <= RTOL_L2, (what, err, l2)


def _oracle(cache, ids, w, x_bits):
    """The CPU oracle's y for routed local ids (positions with weight 0 add nothing)."""
    import oracle

    cfg = cache.cfg
    pairs = [cache.expert_host_ptrs(0, int(e)) for e in ids.reshape(-1)]
    return oracle.expert_ffn(cfg.fmt, cfg.H, cfg.I, pairs, x_bits, w)


CASES = [("c2", {}, 16), ("c3", dict(E=6, H=1024, I=256, S=6, topk=4), 5), ("c4", dict(E=6, H=576, I=320, S=6), 7)]


def _setup(key, geo, bs):
    from expert_slot_cache_device_gb300 import workload as wl
    from expert_slot_cache_device_gb300.synthetic import synthetic_cache

    cfg = wl.scaled(wl.CONFIGS[key], **geo)
    cache = synthetic_cache(cfg, bs * cfg.topk)
    rng = np.random.default_rng(11)
    perm = rng.permutation(cfg.S)
    n_fill = min(cfg.S, cfg.E)
    for b in range(cache.nb):
        for e in range(n_fill):
            cache.slots[b][int(perm[e])].copy_(cache.host_tensor(b, 0)[e])
    return cfg, cache, rng, perm, n_fill


def _inputs(cfg, rng, bs, n_fill, call):
    from expert_slot_cache_device_gb300 import workload as wl

    ids = np.stack([rng.choice(n_fill, cfg.topk, replace=False) for _ in range(bs)]).astype(np.int32)
    w = rng.random((bs, cfg.topk)).astype(np.float32)
    x_bits = wl.f32_to_bf16_bits(np.random.default_rng(100 + call).standard_normal((bs, cfg.H)).astype(np.float32))
    return ids, w, x_bits


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _x_dev(x_bits):
    return torch.from_numpy(x_bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("key,geo,bs", CASES)
def test_noalloc_matches_oracle_two_calls(key, geo, bs):
    from expert_slot_cache_device_gb300 import ftmoe as F

    cfg, cache, rng, perm, n_fill = _setup(key, geo, bs)
    stream = torch.cuda.current_stream().cuda_stream
    banks = [t.data_ptr() for t in cache.slots]
    for call in range(2):
        ids, w, x_bits = _inputs(cfg, rng, bs, n_fill, call)
        slots, d_w, d_x = _dev(perm[ids].astype(np.int32)), _dev(w), _x_dev(x_bits)
        y_ref = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
        y = torch.full((bs, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        F.ftmoe_expert_ffn(cache.handle, d_x.data_ptr(), bs, slots.data_ptr(), d_w.data_ptr(), cfg.topk,
                           y_ref.data_ptr(), stream)
        F.ftmoe_expert_ffn_noalloc(F.FORMATS[cfg.fmt], banks, cfg.S, cfg.H, cfg.I, d_x.data_ptr(), bs,
                                   slots.data_ptr(), d_w.data_ptr(), cfg.topk, y.data_ptr(), stream)
        torch.cuda.synchronize()
        ref = _oracle(cache, ids, w, x_bits)
        _close(y, ref, f"{key} call {call} vs oracle")
        _close(y, y_ref.float().cpu().numpy().astype(np.float64), f"{key} call {call} vs ftmoe_expert_ffn")
    cache.close()


@pytest.mark.parametrize("key,geo,bs", CASES[:2])
def test_noalloc_cpu_positions_and_bad_slot(key, geo, bs):
    """Slot -1 positions add nothing (as in ftmoe_expert_ffn_hybrid without an addend);
    a slot >= S leaves y as it was."""
    from expert_slot_cache_device_gb300 import ftmoe as F

    cfg, cache, rng, perm, n_fill = _setup(key, geo, bs)
    stream = torch.cuda.current_stream().cuda_stream
    banks = [t.data_ptr() for t in cache.slots]
    ids, w, x_bits = _inputs(cfg, rng, bs, n_fill, 5)
    slots = perm[ids].astype(np.int32)
    cpu = rng.random(slots.shape) < 0.3
    cpu[0, :] = True  # one token with every position elsewhere: y = 0
    slots[cpu] = -1
    d_slots, d_w, d_x = _dev(slots), _dev(w), _x_dev(x_bits)
    y = torch.full((bs, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_hyb = torch.empty_like(y)
    F.ftmoe_expert_ffn_noalloc(F.FORMATS[cfg.fmt], banks, cfg.S, cfg.H, cfg.I, d_x.data_ptr(), bs,
                               d_slots.data_ptr(), d_w.data_ptr(), cfg.topk, y.data_ptr(), stream)
    F.ftmoe_expert_ffn_hybrid(cache.handle, d_x.data_ptr(), bs, d_slots.data_ptr(), d_w.data_ptr(), cfg.topk, 0,
                              y_hyb.data_ptr(), stream)
    torch.cuda.synchronize()
    w_gpu = np.where(cpu, 0.0, w).astype(np.float32)
    ref = _oracle(cache, ids, w_gpu, x_bits)
    _close(y, ref, f"{key} slot -1 vs oracle")
    _close(y, y_hyb.float().cpu().numpy().astype(np.float64), f"{key} slot -1 vs ftmoe_expert_ffn_hybrid")
    assert (y[0].float() == 0).all()
    # a slot outside [-1, S): nothing is written
    bad = slots.copy()
    bad[bs - 1, 0] = cfg.S
    y_bad = torch.full((bs, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    F.ftmoe_expert_ffn_noalloc(F.FORMATS[cfg.fmt], banks, cfg.S, cfg.H, cfg.I, d_x.data_ptr(), bs,
                               _dev(bad).data_ptr(), d_w.data_ptr(), cfg.topk, y_bad.data_ptr(), stream)
    torch.cuda.synchronize()
    assert torch.isnan(y_bad.float()).all()
    # and the next good call is correct again (the fixed scratch carries nothing over)
    F.ftmoe_expert_ffn_noalloc(F.FORMATS[cfg.fmt], banks, cfg.S, cfg.H, cfg.I, d_x.data_ptr(), bs,
                               d_slots.data_ptr(), d_w.data_ptr(), cfg.topk, y_bad.data_ptr(), stream)
    torch.cuda.synchronize()
    _close(y_bad, ref, f"{key} after a bad call")
    cache.close()


def test_noalloc_rejects_oversized_calls():
    from expert_slot_cache_device_gb300 import ftmoe as F

    H, I, topk = 4096, 1536, 8
    bs = F.NOALLOC_SCRATCH_BYTES // (topk * (H + I) * 4) + 1
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_expert_ffn_noalloc(F.FMT_BF16, [1 << 30, 1 << 31], 16, H, I, 1 << 32, bs, 1 << 33, 1 << 34, topk,
                                   1 << 35, 0)
    assert e.value.code == F.ERR_INVALID_ARG and "too large" in F.ftmoe_last_error()
    # sizes whose byte counts would wrap a 64-bit product are refused the same way
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_expert_ffn_noalloc(F.FMT_BF16, [1 << 30, 1 << 31], 16, 1 << 30, 1 << 30, 1 << 32, 60000,
                                   1 << 33, 1 << 34, 30000, 1 << 35, 0)
    assert e.value.code == F.ERR_INVALID_ARG
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_expert_ffn_noalloc(F.FMT_BF16, [1 << 30, 1 << 31], 16, 64, 64, 1 << 32, 70000,
                                   1 << 33, 1 << 34, 1, 1 << 35, 0)
    assert e.value.code == F.ERR_INVALID_ARG and "65535" in F.ftmoe_last_error()
