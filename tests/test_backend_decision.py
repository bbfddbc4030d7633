"""The offload / hybrid backend decision and the CPU MoE probe (CPU only).

Benchmark guide, section 5.2: hybrid is recommended for a (workload, format) when the CPU
MoE bandwidth exceeds a threshold (2x by default) times the pinned -> device gather
bandwidth, offload otherwise; a format without a CPU MoE weight path always offloads.
Section 5.4: a hybrid step fetches pcie / cpu of its misses.
"""
import numpy as np
import pytest

from expert_slot_cache_device_gb300 import build as B
from expert_slot_cache_device_gb300 import ftmoe as F
from expert_slot_cache_device_gb300 import workload as wl


@pytest.fixture(scope="module")
def lib():
    B.build()
    return F.lib()


CASES = [
    # fmt, link, cpu, threshold -> backend, fraction
    (F.FMT_BF16, 200.0, 500.0, 0.0, F.BACKEND_HYBRID, 0.4),
    (F.FMT_BF16, 200.0, 400.0, 0.0, F.BACKEND_OFFLOAD, 1.0),   # exactly 2x is not above 2x
    (F.FMT_BF16, 200.0, 399.0, 0.0, F.BACKEND_OFFLOAD, 1.0),
    (F.FMT_NVFP4, 25.0, 100.0, 0.0, F.BACKEND_HYBRID, 0.25),
    (F.FMT_MXFP4, 100.0, 350.0, 3.0, F.BACKEND_HYBRID, 100.0 / 350.0),
    (F.FMT_MXFP4, 100.0, 250.0, 3.0, F.BACKEND_OFFLOAD, 1.0),
    (F.FMT_BF16, 211.0, 32.7, 0.0, F.BACKEND_OFFLOAD, 1.0),    # the measured Grace-GB300 machine
    (F.FMT_RAW, 10.0, 1000.0, 0.0, F.BACKEND_OFFLOAD, 1.0),    # no CPU MoE path
    (F.FMT_BF16, 0.0, 1000.0, 0.0, F.BACKEND_OFFLOAD, 1.0),    # no link profile
]


@pytest.mark.parametrize("fmt,link,cpu,thr,want,frac", CASES)
def test_backend_decision(lib, fmt, link, cpu, thr, want, frac):
    be, fr = F.ftmoe_moe_backend_decision(fmt, link, cpu, thr)
    assert be == want
    assert abs(fr - frac) < 1e-6


def test_cpu_moe_probe_runs_and_scales(lib):
    cfg = wl.scaled(wl.CONFIGS["c1"], E=8, H=256, I=128)
    banks = [np.empty((cfg.E, g.bytes), np.uint8) for g in wl.bank_schema(cfg)]
    for b, arr in enumerate(banks):
        wl.fill_bank(cfg, b, arr)
    ptrs = [a.ctypes.data for a in banks]
    sizes = [a.shape[1] for a in banks]
    gbps = F.ftmoe_measure_cpu_moe(F.FMT_BF16, cfg.H, cfg.I, cfg.E, ptrs, sizes, 8, 1, 2)
    assert 0.0 < gbps < 1e4
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_measure_cpu_moe(F.FMT_RAW, cfg.H, cfg.I, cfg.E, ptrs, sizes, 8, 1, 1)
    assert e.value.code == F.ERR_FORMAT
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_measure_cpu_moe(F.FMT_BF16, cfg.H, cfg.I, cfg.E, ptrs, sizes, 0, 1, 1)
    assert e.value.code == F.ERR_INVALID_ARG


def test_link_probe_rejects_bad_arguments(lib):
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_measure_link(0, 0, 16, 1, 0)
    assert e.value.code == F.ERR_INVALID_ARG
