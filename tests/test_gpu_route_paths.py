"""The routing kernel groups a call's pairs by slot either with one warp (calls of at most 32
routed pairs: a bitonic network over register keys, runs by ballot, pass offsets by a warp
scan) or with the whole block (larger calls). Both must give the same tables, so a token's
output carries the same bits whichever path routed its call: the first tokens of a 5-token
call (40 pairs, block path) against 4-token and 1-token calls (32 and 8 pairs, one warp) over
the same slots, with experts shared between tokens, a token routed to one expert twice and
positions computed elsewhere (slot -1). A bad slot in a one-warp call leaves y untouched and
records FTMOE_ERR_INVALID_ARG, and the next call is exact again (GB300 only).
"""
import numpy as np
import pytest
import torch

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


GEOS = {
    "bf16": ("c2", dict(E=24, H=1024, I=512, L=1, S=24)),
    "nvfp4": ("c3", dict(E=24, H=2048, I=768, L=1, S=24)),
    "q4_0": ("c7", dict(E=24, H=2048, I=512, L=1, S=24)),
}


def _ffn(cache, x, slots, w, bs):
    cfg = cache.cfg
    d_y = torch.full((bs, cfg.H), 7.0, dtype=torch.bfloat16, device="cuda")
    F.ftmoe_expert_ffn_hybrid(cache.handle, x.data_ptr(), bs, slots.data_ptr(), w.data_ptr(), cfg.topk, 0,
                              d_y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return d_y


@pytest.mark.parametrize("fmt", sorted(GEOS))
def test_one_warp_and_block_routing_agree(fmt):
    base, geo = GEOS[fmt]
    cfg = wl.scaled(wl.CONFIGS[base], topk=8, **geo)
    cache = synthetic_cache(cfg, 5 * cfg.topk)
    if fmt == "bf16":
        cache.set_ffn_kernels(F.FFN_ROWS)  # the CUDA-core pipeline (nvfp4 and Q4_0 have no other)
    rng = np.random.default_rng(17)
    perm = rng.permutation(cfg.S)
    for b in range(cache.nb):
        for e in range(cfg.E):
            cache.slots[b][int(perm[e])].copy_(cache.host[b][0][e])
    ids = np.stack([rng.choice(cfg.E, cfg.topk, replace=False) for _ in range(5)]).astype(np.int32)
    ids[3, :3] = ids[0, :3]  # experts shared between tokens
    ids[1, 6] = ids[1, 2]    # one token routed to one expert twice
    slots = perm[ids].astype(np.int32)
    slots[2, 4] = -1         # positions computed elsewhere
    slots[0, 7] = -1
    d_s = to_dev(slots)
    w = rng.random((5, cfg.topk)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    x = wl.f32_to_bf16_bits(rng.standard_normal((5, cfg.H)).astype(np.float32))
    d_x, d_w = x_dev(x), to_dev(w)
    y5 = _ffn(cache, d_x, d_s, d_w, 5)                                                      # 40 pairs
    y4 = _ffn(cache, d_x[:4].contiguous(), d_s[:4].contiguous(), d_w[:4].contiguous(), 4)   # 32 pairs
    y1 = _ffn(cache, d_x[1:2].contiguous(), d_s[1:2].contiguous(), d_w[1:2].contiguous(), 1)  # 8 pairs
    torch.cuda.synchronize()
    assert cache.status() == F.OK
    assert torch.equal(y4, y5[:4]), f"{fmt}: the 4-token call differs from the 5-token call"
    assert torch.equal(y1[0], y5[1]), f"{fmt}: the 1-token call differs from the 5-token call"
    w_gpu = np.where(slots >= 0, w, 0.0).astype(np.float32)
    assert_ffn_close(bf16_to_f64(y4), oracle_ffn(cache, 0, ids[:4], w_gpu[:4], x[:4]), f"{fmt} 4 tokens")

    bad = slots[:2].copy()
    bad[1, 5] = cfg.S
    y_bad = _ffn(cache, d_x[:2].contiguous(), to_dev(bad), d_w[:2].contiguous(), 2)
    torch.cuda.synchronize()
    assert cache.status() == F.ERR_INVALID_ARG  # (reading the status clears it)
    assert bool((y_bad.float() == 7.0).all())
    y2 = _ffn(cache, d_x[:2].contiguous(), d_s[:2].contiguous(), d_w[:2].contiguous(), 2)
    torch.cuda.synchronize()
    assert cache.status() == F.OK
    assert torch.equal(y2, y5[:2])
    cache.close()
