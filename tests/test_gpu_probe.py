"""GPU check of the link probe and the backend decision on measured numbers (benchmark
guide, section 5.2: measure the pinned -> device gather bandwidth and the CPU MoE
bandwidth, then pick offload or hybrid)."""
import pytest
import torch

from expert_slot_cache_device_gb300 import ftmoe as F
from expert_slot_cache_device_gb300 import workload as wl
from expert_slot_cache_device_gb300.synthetic import synthetic_cache

pytestmark = pytest.mark.gpu


def test_link_probe_and_decision():
    n = 64 << 20
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    src.fill_(3)
    dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
    mc, sm = F.ftmoe_measure_link(src.data_ptr(), dst.data_ptr(), n, 3, torch.cuda.current_stream().cuda_stream)
    assert 1.0 < mc < 2000.0 and 1.0 < sm < 2000.0
    assert bool((dst == 3).all())  # the probe really moved the bytes

    cfg = wl.scaled(wl.CONFIGS["c2"], E=16, H=256, I=128, L=2, S=16)
    cache = synthetic_cache(cfg, max_pairs=8)
    ptrs = [cache.host_ptrs[b][0] for b in range(cache.nb)]
    cpu = F.ftmoe_measure_cpu_moe(F.FMT_BF16, cfg.H, cfg.I, cfg.E, ptrs, [g.bytes for g in cache.schema], 8, 0, 2)
    be, fr = F.ftmoe_moe_backend_decision(F.FMT_BF16, max(mc, sm), cpu)
    if cpu > 2.0 * max(mc, sm):
        assert be == F.BACKEND_HYBRID and abs(fr - max(mc, sm) / cpu) < 1e-5
    else:
        assert be == F.BACKEND_OFFLOAD and fr == 1.0
    cache.close()
