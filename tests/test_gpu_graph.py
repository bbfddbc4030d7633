"""Decode calls captured in a CUDA graph (stream capture through the C-ABI binding) replay
exactly like the same calls issued one by one: slot tables, miss lists, copied slot bytes
and FFN outputs bit-identical, on both bf16 FFN kernel families (GB300 only).

The graph is what a serving loop replays once per token: the routed ids, router weights
and activations are device buffers that the caller rewrites before each replay.
"""
import numpy as np
import pytest
import torch

from expert_slot_cache_device_gb300 import ftmoe as F
from expert_slot_cache_device_gb300 import workload as wl
from expert_slot_cache_device_gb300.synthetic import synthetic_cache
from gpu_helpers import to_dev, x_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_slot_cache_device_gb300 import build

    build.build()


def _calls(cfg, bs, steps, seed):
    rng = np.random.default_rng(seed)
    calls = []
    for _ in range(steps):
        for layer in range(cfg.L):
            ids = np.stack([rng.choice(cfg.E, cfg.topk, replace=False) for _ in range(bs)]).astype(np.int32)
            w = rng.random((bs, cfg.topk)).astype(np.float32)
            x = wl.f32_to_bf16_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))
            calls.append((layer, to_dev(ids), to_dev(w), x_dev(x)))
    return calls


@pytest.mark.parametrize("bs", [2, 4])
def test_decode_calls_replay_from_a_graph(bs):
    # E = 16, topk 8: bs 2 routes 16 pairs (CUDA-core FFN), bs 4 routes 32 (tcgen05 FFN)
    cfg = wl.scaled(wl.CONFIGS["c2"], E=16, L=3, S=24)
    cache = synthetic_cache(cfg, bs * cfg.topk, host_layers=range(cfg.L))
    expect = F.FFN_ROWS if bs == 2 else F.FFN_TC05
    assert F.ftmoe_ffn_kernels_for(cache.handle, bs, cfg.topk) == expect
    calls = _calls(cfg, bs, steps=2, seed=bs)
    d_slots = [torch.empty((bs, cfg.topk), dtype=torch.int32, device="cuda") for _ in calls]
    d_y = [torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda") for _ in calls]
    owner0 = np.full(cfg.S, -1, np.int32)
    stamp0 = np.zeros(cfg.S, np.uint32)

    def run(stream):
        for i, (layer, ids, w, x) in enumerate(calls):
            cache.ensure(layer, ids, d_slots[i], stream=stream)
            cache.copy_missing(stream=stream)
            cache.ffn(x, d_slots[i], w, d_y[i], stream=stream)

    def reset():
        cache.set_state(owner0, stamp0, 0)
        for s in cache.slots:
            s.zero_()
        for y, sl in zip(d_y, d_slots):
            y.zero_()
            sl.fill_(-7)
        torch.cuda.synchronize()

    reset()
    run(None)
    torch.cuda.synchronize()
    assert cache.status() == F.OK
    ref_y = [y.clone() for y in d_y]
    ref_sl = [s.clone() for s in d_slots]
    ref_bytes = [s.clone() for s in cache.slots]
    ref_state = cache.get_state()
    ref_miss = cache.miss_list()

    reset()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        run(side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):  # the same graph, replayed twice from the same starting state
        reset()
        g.replay()
        torch.cuda.synchronize()
        assert cache.status() == F.OK
        for a, b in zip(d_y, ref_y):
            assert torch.equal(a, b)
        for a, b in zip(d_slots, ref_sl):
            assert torch.equal(a, b)
        for a, b in zip(cache.slots, ref_bytes):
            assert torch.equal(a, b)
        owner, stamp, clock = cache.get_state()
        assert np.array_equal(owner, ref_state[0]) and np.array_equal(stamp, ref_state[1])
        assert clock == ref_state[2] == len(calls)
        ids, slots = cache.miss_list()
        assert np.array_equal(ids, ref_miss[0]) and np.array_equal(slots, ref_miss[1])
    del g
    cache.close()
