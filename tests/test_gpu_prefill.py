"""GPU parity of the whole-layer double-buffered prefill pipeline (ftmoe_prefill_layers).

Architecture deep-dive, section 五: prefill streams each layer's experts into the global LRU
cache through a double buffer, the copy of the next layer overlapping the current layer's
expert FFN. Checked against the oracle replaying the same LRU calls one after another
(prefetch = ensure of all E experts, then the routed ensure): the final slot tables are
bit-exact, every step's output is within the FFN tolerance of the fp64 oracle and
bit-identical to the same single calls made one after another on one stream.
"""
import numpy as np
import pytest
import torch

import oracle
from expert_slot_cache_device_gb300 import ftmoe as F
from expert_slot_cache_device_gb300 import workload as wl
from expert_slot_cache_device_gb300.synthetic import synthetic_cache
from gpu_helpers import assert_ffn_close, bf16_to_f64, oracle_ffn, to_dev, x_dev

pytestmark = pytest.mark.gpu

CASES = {
    "bf16": wl.scaled(wl.CONFIGS["c2"], E=16, topk=4, H=256, I=128, L=4, S=32),
    "nvfp4": wl.scaled(wl.CONFIGS["c3"], E=8, topk=4, H=512, I=256, L=3, S=16),
    "mxfp4": wl.scaled(wl.CONFIGS["c4"], E=8, topk=4, H=256, I=256, L=3, S=16),
    "fp8": wl.scaled(wl.CONFIGS["c6"], E=8, topk=4, H=512, I=512, L=3, S=16),
    "q4_0": wl.scaled(wl.CONFIGS["c7"], E=8, topk=4, H=512, I=256, L=3, S=16),
}


def make_cache(cfg, bs):
    cache = synthetic_cache(cfg, max_pairs=bs * cfg.topk, host_layers=range(cfg.L))
    # make every layer's bank different: layer l holds layer 0's experts rolled by l
    for b in range(cache.nb):
        base = cache.host[b][0].clone()
        for l in range(1, cfg.L):
            cache.host[b][l].copy_(torch.roll(base, shifts=l, dims=0))
    return cache


def step_inputs(cfg, bs, steps, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(steps):
        ids = np.stack([rng.permutation(cfg.E)[:cfg.topk] for _ in range(bs)]).astype(np.int32)
        logits = rng.standard_normal((bs, cfg.topk))
        w = (np.exp(logits) / np.exp(logits).sum(1, keepdims=True)).astype(np.float32)
        x = wl.f32_to_bf16_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))
        out.append((ids, w, x))
    return out


@pytest.mark.parametrize("fmt", list(CASES))
@pytest.mark.parametrize("mode", ["engine", "fused"])
def test_prefill_pipeline_matches_oracle_and_sequential(fmt, mode):
    cfg = CASES[fmt]
    bs, steps = 6, 5
    layers = [i % cfg.L for i in range(steps)]
    inputs = step_inputs(cfg, bs, steps, seed=11)
    cache = make_cache(cfg, bs)
    cache.set_copy_mode(F.COPY_ENGINE if mode == "engine" else F.COPY_FUSED)
    d_ids = [to_dev(ids) for ids, _, _ in inputs]
    d_w = [to_dev(w) for _, w, _ in inputs]
    d_x = [x_dev(x) for _, _, x in inputs]
    d_y = [torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    cache.prefill_layers(layers, d_ids, d_x, d_w, d_y, compute, copy)
    torch.cuda.synchronize()
    assert cache.status() == 0
    owner, stamp, clock = cache.get_state()

    # oracle: the same LRU calls one after another
    orc_cache = oracle.Cache(cfg.E, cfg.L, cfg.S)
    for i, layer in enumerate(layers):
        rc, *_ = orc_cache.ensure(layer, np.arange(cfg.E, dtype=np.int32)[None, :])
        assert rc == oracle.OK
        rc, slots, mids, _ = orc_cache.ensure(layer, inputs[i][0])
        assert rc == oracle.OK and mids.size == 0
    assert owner.tolist() == orc_cache.owner.tolist()
    assert stamp.tolist() == orc_cache.stamp.tolist()
    assert clock == int(orc_cache.clock[0])

    # the same single calls one after another on one stream (same kernels, same inputs)
    ref = make_cache(cfg, bs)
    ref.set_copy_mode(F.COPY_FUSED)
    d_slots = torch.empty((bs, cfg.topk), dtype=torch.int32, device="cuda")
    for i, layer in enumerate(layers):
        ref.prefetch_layer(layer)
        ref.ensure(layer, d_ids[i], d_slots)
        y_seq = torch.empty_like(d_y[i])
        ref.ffn(d_x[i], d_slots, d_w[i], y_seq)
        torch.cuda.synchronize()
        assert torch.equal(y_seq.view(torch.int16), d_y[i].view(torch.int16)), f"step {i}"
        y_ref = oracle_ffn(cache, layer, inputs[i][0], inputs[i][1], inputs[i][2])
        assert_ffn_close(bf16_to_f64(d_y[i]), y_ref, f"{fmt} {mode} step {i} layer {layer}")
    ref.close()
    cache.close()


def test_prefill_rejects_single_buffer():
    cfg = wl.scaled(CASES["bf16"], S=24)  # S < 2E
    bs = 2
    cache = make_cache(cfg, bs)
    ids = [to_dev(np.zeros((bs, cfg.topk), np.int32) + np.arange(cfg.topk, dtype=np.int32))]
    x = [torch.zeros((bs, cfg.H), dtype=torch.bfloat16, device="cuda")]
    w = [torch.ones((bs, cfg.topk), dtype=torch.float32, device="cuda")]
    y = [torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")]
    with pytest.raises(F.FtmoeError) as e:
        cache.prefill_layers([0], ids, x, w, y, torch.cuda.current_stream(), torch.cuda.current_stream())
    assert e.value.code == F.ERR_INVALID_ARG
    cache.close()
