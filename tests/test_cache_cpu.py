"""Host-side checks of the cache owner over caller banks (no GPU): the validation that runs
before any bank reaches the library."""
import pytest
import torch

from expert_slot_cache_device_gb300 import workload as wl
from expert_slot_cache_device_gb300.cache import Bank, check_banks


def _banks(cfg, layers):
    schema = wl.bank_schema(cfg)
    return schema, [[torch.zeros((cfg.E, g.bytes), dtype=torch.uint8) if l in layers else None
                     for l in range(cfg.L)] for g in schema]


def test_caller_banks_accepted():
    cfg = wl.CONFIGS["c1"]
    schema, src = _banks(cfg, {0})
    got = check_banks("bf16", cfg.E, cfg.L, cfg.S, schema, src)
    assert [g.bytes for g in got] == [g.bytes for g in schema]
    # any geometry object works, entries may alias, a flat tensor of E * bytes is fine
    flat = [torch.zeros(cfg.E * g.bytes, dtype=torch.uint8) for g in schema]
    alias = [[flat[b]] * cfg.L for b in range(len(schema))]
    banks = [Bank(g.name, g.dtype, g.rows, g.row_bytes) for g in schema]
    check_banks(1, cfg.E, cfg.L, cfg.S, banks, alias)
    slots = [torch.zeros((cfg.S, g.bytes), dtype=torch.uint8) for g in schema]
    check_banks("bf16", cfg.E, cfg.L, cfg.S, banks, alias, slots)


@pytest.mark.parametrize("bad", ["format", "dtype", "layers", "bytes", "tensor_dtype", "noncontig", "banks",
                                 "slot_bytes"])
def test_caller_banks_rejected(bad):
    cfg = wl.CONFIGS["c1"]
    schema, src = _banks(cfg, {0, 1})
    fmt, slots = "bf16", None
    banks = [Bank(g.name, g.dtype, g.rows, g.row_bytes) for g in schema]
    if bad == "format":
        fmt = "bf32"
    elif bad == "dtype":
        banks[0] = Bank("gate_up", "int7", 1, banks[0].bytes)
    elif bad == "layers":
        src[0] = src[0][:1]
    elif bad == "bytes":
        src[1][0] = torch.zeros((cfg.E, schema[1].bytes - 16), dtype=torch.uint8)
    elif bad == "tensor_dtype":
        src[0][1] = torch.zeros((cfg.E, schema[0].bytes // 2), dtype=torch.int16)
    elif bad == "noncontig":
        src[0][0] = torch.zeros((schema[0].bytes, cfg.E), dtype=torch.uint8).t()
    elif bad == "banks":
        src = src[:1]
    elif bad == "slot_bytes":
        slots = [torch.zeros((cfg.S, g.bytes), dtype=torch.uint8) for g in schema]
        slots[1] = slots[1][:-1]
    with pytest.raises(ValueError):
        check_banks(fmt, cfg.E, cfg.L, cfg.S, banks, src, slots)
