"""Hybrid decode path on the GPU against the oracle (GB300 only).

FreeToken benchmark guide, section 5.4: ensure_experts_hybrid fetches at most a capped
number of misses (the first ones in ascending flat id), rewrites the others to slot -1
and counts fetched / uncapped misses; the CPU executor computes the -1 positions and
its output is added to the GPU FFN before the final bf16 round.
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


@pytest.mark.parametrize("seed", range(4))
def test_hybrid_ensure_random_traces(seed):
    rng = np.random.default_rng(300 + seed)
    E, L, k = int(rng.integers(8, 40)), int(rng.integers(1, 4)), int(rng.integers(2, 6))
    S = int(rng.integers(k, k + 16))
    cfg = wl.Config("raw", "raw", 9, "raw", E, 1, 64, 0, L, S, (1,), (1.0,), "uniform", 0.0, seed)
    cache = synthetic_cache(cfg, 0, host_layers=range(L))
    orc = oracle.Cache(E, L, S)
    d_slots = torch.empty((2, k), dtype=torch.int32, device="cuda")
    d_counts = torch.zeros(2, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    for layer, ids in wl.random_trace_ids(seed + 5, 150, E, L, 2, k, 1.1):
        max_fetch = int(rng.integers(-1, 5))
        frac = float(rng.choice([0.0, 0.25, 0.5, 0.8]))
        rc, slots, mids, msl, counts = orc.ensure_hybrid(layer, ids, max_fetch, frac)
        d_ids = to_dev(ids)
        F.ftmoe_ensure_experts_hybrid(cache.handle, layer, d_ids.data_ptr(), 2, k, max_fetch, frac,
                                      d_slots.data_ptr(), d_counts.data_ptr(), st)
        cache.copy_missing()
        assert cache.status() == rc
        assert tuple(d_counts.cpu().tolist()) == counts
        if rc == oracle.OK:
            assert np.array_equal(d_slots.cpu().numpy(), slots)
        gi, gs = cache.miss_list()
        assert np.array_equal(gi, mids) and np.array_equal(gs, msl)
        owner, stamp, clock = cache.get_state()
        assert np.array_equal(owner, orc.owner) and np.array_equal(stamp, orc.stamp) and clock == int(orc.clock[0])
        for f, s in zip(mids.tolist(), msl.tolist()):
            assert torch.equal(cache.slots[0][s].cpu(), cache.host[0][f // E][f % E])
    cache.close()


CASES = [("c2", dict(), 16, 0.5, 24), ("c3", dict(E=64, S=96), 8, 1.0, 20), ("c4", dict(E=48, S=64), 16, 0.5, 5),
         ("c4", dict(E=48, S=64), 64, 0.5, -1)]


@pytest.mark.parametrize("key,geo,bs,mr,max_fetch", CASES)
def test_hybrid_step_matches_oracle(key, geo, bs, mr, max_fetch):
    cfg = wl.scaled(wl.CONFIGS[key], **geo)
    cache = synthetic_cache(cfg, bs * cfg.topk)
    r = wl.make_route(cfg, bs, mr)
    for i, e in enumerate(sorted(int(v) for v in r.hits)):
        for b in range(cache.nb):
            cache.slots[b][i].copy_(cache.host[b][0][e])
    cache.set_state(r.owner, r.stamp, r.clock)
    orc = oracle.Cache(cfg.E, cfg.L, cfg.S, r.owner, r.stamp, r.clock)
    frac = 0.3 if max_fetch < 0 else 0.0
    rc, slots, mids, msl, counts = orc.ensure_hybrid(0, r.topk_ids, max_fetch, frac)
    assert rc == oracle.OK and counts[1] == r.misses
    st = torch.cuda.current_stream().cuda_stream
    d_ids = to_dev(r.topk_ids)
    d_slots = torch.empty_like(d_ids)
    d_counts = torch.zeros(2, dtype=torch.int32, device="cuda")
    F.ftmoe_ensure_experts_hybrid(cache.handle, 0, d_ids.data_ptr(), bs, cfg.topk, max_fetch, frac,
                                  d_slots.data_ptr(), d_counts.data_ptr(), st)
    cache.copy_missing()
    h_slots = d_slots.cpu().numpy()
    assert np.array_equal(h_slots, slots) and tuple(d_counts.cpu().tolist()) == counts
    # CPU executor for the -1 positions, GPU FFN for the rest, summed before the bf16 round
    y_cpu = np.empty((bs, cfg.H), np.float32)
    F.ftmoe_cpu_expert_ffn(F.FORMATS[cfg.fmt], cfg.H, cfg.I, bs, cfg.topk, r.topk_ids.ctypes.data,
                           h_slots.ctypes.data, [cache.host_ptrs[b][0] for b in range(cache.nb)],
                           [g.bytes for g in cache.schema], r.x.ctypes.data, r.weights.ctypes.data, y_cpu.ctypes.data,
                           0)
    # keep every device tensor referenced until the kernels have run (a temporary's
    # memory could be handed to the next allocation before the FFN reads it)
    d_add = torch.from_numpy(y_cpu).cuda()
    d_x = x_dev(r.x)
    d_w = to_dev(r.weights)
    d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
    F.ftmoe_expert_ffn_hybrid(cache.handle, d_x.data_ptr(), bs, d_slots.data_ptr(), d_w.data_ptr(), cfg.topk,
                              d_add.data_ptr(), d_y.data_ptr(), st)
    assert cache.status() == F.OK
    ref = oracle_ffn(cache, 0, r.topk_ids, r.weights, r.x)
    assert_ffn_close(bf16_to_f64(d_y), ref, f"hybrid {key} bs={bs}")
    cache.close()
