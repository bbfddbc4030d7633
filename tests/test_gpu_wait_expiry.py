"""The bounded-wait error path of the FFN pipeline (GPU), made to run out on purpose without any
fault: a test setting leaves one shared-memory stage of the CUDA-core pipeline unfilled (no copy
is issued for it, nothing arrives), with a 1 ms wait limit. The call must return, record
FTMOE_ERR_STATE in the status word, and the next call on the same cache must be correct."""
import time

import numpy as np
import pytest
import torch

from gpu_helpers import assert_ffn_close, bf16_to_f64, oracle_ffn, to_dev, x_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import oracle
    from expert_slot_cache_device_gb300 import build

    build.build()
    oracle.build()


@pytest.mark.parametrize("key,geo", [("c2", dict(E=6, H=1024, I=256, L=2, S=6)),
                                     ("c3", dict(E=5, H=2048, I=512, L=2, S=5))])
def test_wait_runs_out_and_the_next_call_is_correct(key, geo):
    from expert_slot_cache_device_gb300 import ftmoe as F
    from expert_slot_cache_device_gb300 import workload as wl
    from expert_slot_cache_device_gb300.synthetic import synthetic_cache

    cfg = wl.scaled(wl.CONFIGS[key], topk=3, **geo)
    bs = 4
    cache = synthetic_cache(cfg, bs * cfg.topk)
    if cfg.fmt == "bf16":
        cache.set_ffn_kernels(F.FFN_ROWS)  # the CUDA-core pipeline carries the test setting
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(cfg.E, cfg.topk, replace=False) for _ in range(bs)]).astype(np.int32)
    w = rng.random((bs, cfg.topk)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    x = wl.f32_to_bf16_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))
    perm = rng.permutation(cfg.S)
    for b in range(cache.nb):
        for e in range(cfg.E):
            cache.slots[b][int(perm[e])].copy_(cache.host_tensor(b, 0)[e])
    slots = perm[ids].astype(np.int32)
    d_x, d_s, d_w = x_dev(x), to_dev(slots), to_dev(w)
    d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
    assert cache.status() == F.OK

    F.ftmoe_set_debug(cache.handle, F.DEBUG_WAIT_NS, 1_000_000)  # 1 ms
    F.ftmoe_set_debug(cache.handle, F.DEBUG_FFN_SKIP_STAGE, 1)
    t0 = time.perf_counter()
    cache.ffn(d_x, d_s, d_w, d_y)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0  # the waits ran out after about 1 ms each
    assert cache.status() == F.ERR_STATE

    F.ftmoe_set_debug(cache.handle, F.DEBUG_FFN_SKIP_STAGE, 0)
    F.ftmoe_set_debug(cache.handle, F.DEBUG_WAIT_NS, 0)
    cache.ffn(d_x, d_s, d_w, d_y)
    torch.cuda.synchronize()
    assert cache.status() == F.OK
    ref = oracle_ffn(cache, 0, ids, w, x)
    assert_ffn_close(bf16_to_f64(d_y), ref, f"{key} after an expired wait")
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_set_debug(cache.handle, 99, 0)
    assert e.value.code == F.ERR_INVALID_ARG
    cache.close()
