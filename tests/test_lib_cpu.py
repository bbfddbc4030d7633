"""CPU-side checks of the C-ABI library (no GPU): it builds, loads, exports every
entry point the header declares, and rejects bad arguments on the host."""
import os
import re

import pytest

from expert_slot_cache_device_gb300 import build as B
from expert_slot_cache_device_gb300 import ftmoe as F
from expert_slot_cache_device_gb300 import workload as wl

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ftmoe.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return F.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ftmoe_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(F.EXPORTS)


def test_workspace_bytes_and_host_checks(lib):
    for key, cfg in wl.CONFIGS.items():
        nb = len(wl.bank_schema(cfg))
        n = F.ftmoe_cache_workspace_bytes(F.FORMATS[cfg.fmt], nb, cfg.E, cfg.L, cfg.S, cfg.H, cfg.I,
                                          max(cfg.bs_list) * cfg.topk)
        assert n > cfg.E * cfg.L * 4 + cfg.S * 8
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_cache_workspace_bytes(F.FMT_BF16, 3, 8, 2, 4, 256, 128, 2)
    assert e.value.code == F.ERR_FORMAT
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_cache_workspace_bytes(F.FMT_NVFP4, 6, 8, 2, 4, 100, 128, 2)
    assert e.value.code == F.ERR_FORMAT
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_cache_workspace_bytes(F.FMT_RAW, 1, 0, 2, 4, 0, 0, 0)
    assert e.value.code == F.ERR_INVALID_ARG
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_cache_workspace_bytes(F.FMT_RAW, 1, 8, 2, 9000, 0, 0, 0)
    assert e.value.code == F.ERR_INVALID_ARG
    # the FFN kernel selector and its query check their handle before anything else
    for call in (lambda: F.ftmoe_set_ffn_kernels(0, F.FFN_MMA), lambda: F.ftmoe_ffn_kernels_for(0, 4, 8)):
        with pytest.raises(F.FtmoeError) as e:
            call()
        assert e.value.code == F.ERR_INVALID_ARG


def test_create_rejects_schema_mismatch_before_any_cuda_call(lib):
    cfg = wl.CONFIGS["c1"]
    schema = wl.bank_schema(cfg)
    specs = [dict(name=g.name, dtype=F.DTYPES[g.dtype], rows=g.rows, row_bytes=g.row_bytes + (16 if b else 0),
                  host_src=[1 << 20] * cfg.L, dev_slots=1 << 30) for b, g in enumerate(schema)]
    arr, keep = F.make_bank_specs(specs)
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_cache_create(arr, 2, F.FMT_BF16, cfg.E, cfg.L, cfg.S, cfg.H, cfg.I, 2, 1 << 32, 1 << 30, 0)
    assert e.value.code == F.ERR_FORMAT
    specs[1]["row_bytes"] -= 16
    specs[1]["dtype"] = F.DT_U8
    arr, keep = F.make_bank_specs(specs)
    with pytest.raises(F.FtmoeError) as e:
        F.ftmoe_cache_create(arr, 2, F.FMT_BF16, cfg.E, cfg.L, cfg.S, cfg.H, cfg.I, 2, 1 << 32, 1 << 30, 0)
    assert e.value.code == F.ERR_FORMAT
    with pytest.raises(F.FtmoeError) as e:  # workspace too small
        F.ftmoe_cache_create(arr, 2, F.FMT_BF16, cfg.E, cfg.L, cfg.S, cfg.H, cfg.I, 2, 1 << 32, 64, 0)
    assert e.value.code == F.ERR_INVALID_ARG
    with pytest.raises(F.FtmoeError) as e:  # misaligned workspace
        F.ftmoe_cache_create(arr, 2, F.FMT_BF16, cfg.E, cfg.L, cfg.S, cfg.H, cfg.I, 2, (1 << 32) + 8, 1 << 30, 0)
    assert e.value.code == F.ERR_INVALID_ARG


def test_null_handles(lib):
    for call in (lambda: F.ftmoe_copy_missing(None, 0), lambda: F.ftmoe_set_copy_mode(None, 0),
                 lambda: F.ftmoe_ensure_experts(None, 0, 0, 1, 1, 0, 0)):
        with pytest.raises(F.FtmoeError) as e:
            call()
        assert e.value.code == F.ERR_INVALID_ARG
    F.ftmoe_cache_destroy(None)


def test_binding_constants_match_the_header():
    """Every integer constant of the header that the binding names has the same value there."""
    text = open(HEADER).read()
    defs = {}
    for name, val in re.findall(r"^#define FTMOE_([A-Z0-9_]+)\s+\(?(-?\d+)u?\)?", text, flags=re.M):
        defs[name] = int(val)
    noalloc = re.search(r"^#define FTMOE_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text, flags=re.M)
    defs["NOALLOC_SCRATCH_BYTES"] = int(noalloc.group(1)) << int(noalloc.group(2))
    checked = 0
    for name, val in defs.items():
        if hasattr(F, name):
            assert getattr(F, name) == val, name
            checked += 1
    for family in ("ERR_", "FMT_", "DT_", "COPY_", "FFN_", "BACKEND_", "DEBUG_"):
        names = [n for n in defs if n.startswith(family)]
        assert names and all(hasattr(F, n) for n in names), family
    assert checked >= 30


def test_bounds_checked_build_exports_every_symbol():
    """The debug build with device-side index checks (-DFTMOE_CHECK) compiles and exports the
    same entry points as the release library."""
    import ctypes

    path = B.build(check=True)
    assert path.endswith("libftmoe_check.so")
    lib_check = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(lib_check, n), n
