"""Pins of the oracle's copy_missing and of the bank schemas (CPU only).

FreeToken MoE offline benchmark guide, section 4.2: the cache only moves rows, so a
miss must land byte-identical in its slot of every bank; section 4.4:
copy_MiB = misses * bytes per expert. The per-expert byte counts of every workload
are pinned against a table written from the workload shapes.
"""
import numpy as np

from conftest import golden_lines
from expert_slot_cache_device_gb300 import workload as wl


def test_bytes_per_expert_table():
    for ln in golden_lines("bytes_per_expert.txt"):
        key, *vals = ln.split()
        cfg = wl.CONFIGS[key]
        assert [g.bytes for g in wl.bank_schema(cfg)] == [int(v) for v in vals]
    assert wl.CONFIGS["c1"].bytes_per_expert == 196608
    # the tiny workload keeps its literal down shape [E, 128, 256]
    down = wl.bank_schema(wl.CONFIGS["c1"])[1]
    assert (down.rows, down.row_bytes // 2) == (128, 256)


def test_copy_moves_rows_unchanged(orc):
    cfg = wl.scaled(wl.CONFIGS["c3"], E=6, H=64, I=32, S=4, L=3)
    banks = wl.make_banks(cfg)
    bb = [g.bytes for g in wl.bank_schema(cfg)]
    rng = np.random.default_rng(0)
    slots = [rng.integers(0, 256, (cfg.S, n), dtype=np.uint8) for n in bb]
    before = [s.copy() for s in slots]
    c = orc.Cache(cfg.E, cfg.L, cfg.S)
    layer = 1
    rc, _, mids, msl = c.ensure(layer, np.array([[4, 1, 5]], np.int32))
    assert rc == orc.OK and mids.tolist() == [layer * cfg.E + e for e in (1, 4, 5)]
    orc.copy_missing(bb, banks, slots, cfg.E, mids, msl)
    moved = 0
    for b in range(len(bb)):
        for s in range(cfg.S):
            if s in msl.tolist():
                e = int(mids[msl.tolist().index(s)]) % cfg.E
                assert np.array_equal(slots[b][s], banks[b][e])
                moved += slots[b][s].nbytes
            else:
                assert np.array_equal(slots[b][s], before[b][s])
    assert moved == mids.size * sum(bb)
    assert moved / 2 ** 20 == mids.size * cfg.bytes_per_expert / 2 ** 20
