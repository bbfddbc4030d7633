"""The allocation-free FFN entry point against the regular one (GPU).

ftmoe_expert_ffn_noalloc serves callers that cannot call cudaMalloc — code running
inside a runtime that already owns all device memory, or on a path that must not pay
for an allocation's device synchronisation. Its scratch is a fixed array inside the
library, so this test checks, through the C-ABI, that two calls in a row (with
different inputs, so stale scratch from the first call would show) give what
ftmoe_expert_ffn gives for the same slot banks, within the FFN tolerance of the
other tests, and that an over-sized call is refused. This file is collected last.
"""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ATOL, RTOL_L2 = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_slot_cache_device_gb300 import build

    build.build()


def _close(a: torch.Tensor, b: torch.Tensor):
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    err = np.abs(x - y).max()
    l2 = np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30)
    assert np.isfinite(x).all() and err <= ATOL and l2 <= RTOL_L2, (err, l2)


CASES = [("c2", {}, 16), ("c3", dict(E=6, H=1024, I=256, S=6, topk=4), 5), ("c4", dict(E=6, H=576, I=320, S=6), 7)]


@pytest.mark.parametrize("key,geo,bs", CASES)
def test_noalloc_matches_regular_ffn_two_calls(key, geo, bs):
    from expert_slot_cache_device_gb300 import ftmoe as F
    from expert_slot_cache_device_gb300 import workload as wl
    from expert_slot_cache_device_gb300.cache import ExpertSlotCache

    cfg = wl.scaled(wl.CONFIGS[key], **geo)
    cache = ExpertSlotCache(cfg, bs * cfg.topk)
    rng = np.random.default_rng(11)
    perm = rng.permutation(cfg.S)
    n_fill = min(cfg.S, cfg.E)
    for b in range(cache.nb):
        for e in range(n_fill):
            cache.slots[b][int(perm[e])].copy_(cache.host[b][0][e])
    stream = torch.cuda.current_stream().cuda_stream
    banks = [t.data_ptr() for t in cache.slots]
    for call in range(2):
        ids = np.stack([rng.choice(n_fill, cfg.topk, replace=False) for _ in range(bs)])
        slots = torch.from_numpy(perm[ids].astype(np.int32)).cuda()
        w = torch.from_numpy(rng.random((bs, cfg.topk)).astype(np.float32)).cuda()
        x = torch.randn((bs, cfg.H), generator=torch.Generator().manual_seed(call)).to(torch.bfloat16).cuda()
        y_ref = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
        y = torch.full((bs, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        F.ftmoe_expert_ffn(cache.handle, x.data_ptr(), bs, slots.data_ptr(), w.data_ptr(), cfg.topk,
                           y_ref.data_ptr(), stream)
        F.ftmoe_expert_ffn_noalloc(F.FORMATS[cfg.fmt], banks, cfg.S, cfg.H, cfg.I, x.data_ptr(), bs,
                                   slots.data_ptr(), w.data_ptr(), cfg.topk, y.data_ptr(), stream)
        torch.cuda.synchronize()
        _close(y, y_ref)
    cache.close()


def test_noalloc_rejects_oversized_calls():
    from expert_slot_cache_device_gb300 import ftmoe as F

    H, I, topk = 4096, 1536, 8
    bs = F.NOALLOC_SCRATCH_BYTES // (topk * (H + I) * 4) + 1
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_expert_ffn_noalloc(F.FMT_BF16, [1 << 30, 1 << 31], 16, H, I, 1 << 32, bs, 1 << 33, 1 << 34, topk,
                                   1 << 35, 0)
    assert e.value.code == F.ERR_INVALID_ARG and "too large" in F.ftmoe_last_error()
