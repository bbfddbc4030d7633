"""Pins of the oracle's hybrid ensure_experts (CPU only).

FreeToken MoE offline benchmark guide, section 5.4: the hybrid ensure assigns slots to
at most hybrid_max_fetch missing experts per step, rewrites the overflow to -1 for the
CPU executor, and counts num_indices (fetched) and num_missing_full (uncapped); with a
bandwidth profile the fetch share follows pcie_bw : (cpu_bw - pcie_bw), i.e. a fraction
pcie_bw / cpu_bw of the misses; without one the cap is 1. Readings: the fetched misses
are the first ones in ascending flat id; the fraction rule rounds half to even in
binary32.
"""
import numpy as np
import pytest

from expert_slot_cache_device_gb300 import workload as wl
from test_oracle_lru import BruteLRU


class BruteHybrid(BruteLRU):
    def ensure_capped(self, layer, ids, cap):
        ids = [int(v) for v in np.asarray(ids).reshape(-1)]
        wanted = sorted(set(layer * self.E + i for i in ids))
        missing = [f for f in wanted if self.where(f) < 0]
        keep = set(missing[cap:])  # overflow: left to the CPU, cache untouched
        st, slots, mids, ms = self.ensure_subset(layer, ids, keep)
        return st, slots, mids, ms, (len(missing) - len(keep), len(missing))

    def ensure_subset(self, layer, ids, skip):
        now = self.clock + 1
        used_now = set()
        wanted = sorted(set(layer * self.E + i for i in ids))
        missing = []
        for f in wanted:
            s = self.where(f)
            if s >= 0:
                used_now.add(s)
            elif f not in skip:
                missing.append(f)
        if len(missing) > self.S - len(used_now):
            return "ERR_CAPACITY", None, None, None
        self.clock = now
        for s in used_now:
            self.last_use[s] = now
        mslots = []
        for f in missing:
            best = None
            for s in range(self.S):
                if s in used_now:
                    continue
                if best is None or self.last_use[s] < self.last_use[best]:
                    best = s
            used_now.add(best)
            self.owner[best] = f
            self.last_use[best] = now
            mslots.append(best)
        slots = [self.where(layer * self.E + i) for i in ids]
        return "OK", slots, missing, mslots


@pytest.mark.parametrize("seed", range(8))
def test_hybrid_matches_brute_force(orc, seed):
    rng = np.random.default_rng(40 + seed)
    E, L = int(rng.integers(4, 12)), int(rng.integers(1, 4))
    k = int(rng.integers(1, min(E, 4) + 1))
    S = int(rng.integers(k, k + 6))
    bs = int(rng.integers(1, 3))
    o = orc.Cache(E, L, S)
    b = BruteHybrid(E, L, S)
    for call, (layer, ids) in enumerate(wl.random_trace_ids(seed + 77, 200, E, L, bs, k, 1.1)):
        cap = int(rng.integers(0, 4))
        rc, slots, mids, msl, counts = o.ensure_hybrid(layer, ids, cap)
        st, bslots, bm, bms, bcounts = b.ensure_capped(layer, ids, cap)
        if st == "OK":
            assert rc == orc.OK
            assert slots.reshape(-1).tolist() == bslots
            assert mids.tolist() == bm and msl.tolist() == bms
            assert counts == bcounts
            assert o.owner.tolist() == b.owner and o.stamp.tolist() == b.last_use
            # overflow positions are -1, fetched and resident positions have slots
            for i, s in zip(np.asarray(ids).reshape(-1), slots.reshape(-1)):
                assert (s == -1) == (o.id2slot[layer * E + int(i)] < 0)
        else:
            assert rc == orc.ERR_CAPACITY and counts == (0, 0)


def test_fetch_fraction_rule(orc):
    """cap = round_half_even(float32(misses) * fraction); fraction <= 0 means no profile (cap 1)."""
    cases = [(10, 0.25, 2), (6, 0.25, 2), (7, 0.5, 4), (5, 0.5, 2), (8, 1.0, 8), (8, 2.0, 8), (3, 0.1, 0),
             (9, 0.0, 1), (9, -1.0, 1)]
    for misses, frac, want in cases:
        E, L, S = 16, 2, 16
        o = orc.Cache(E, L, S)
        ids = np.arange(misses, dtype=np.int32)[None, :]
        rc, slots, mids, msl, counts = o.ensure_hybrid(0, ids, -1, frac)
        assert rc == orc.OK
        assert counts == (min(want, misses), misses), (misses, frac)
        assert mids.tolist() == list(range(min(want, misses)))  # the first ids ascending
        assert (slots.reshape(-1) >= 0).sum() == min(want, misses)


def test_split_formula_closed_form():
    """Fetched : CPU-computed = pcie : (cpu - pcie) <=> fetched = misses * pcie / cpu."""
    for m, p, c in [(64, 200.0, 400.0), (10, 100.0, 500.0), (7, 50.0, 175.0)]:
        f = m * p / c
        assert abs(f / (m - f) - p / (c - p)) < 1e-12


def test_cap_zero_fetches_nothing_and_counts(orc):
    cfg = wl.CONFIGS["c2"]
    r = wl.make_route(cfg, 4, 0.5)
    o = orc.Cache(cfg.E, cfg.L, cfg.S, r.owner, r.stamp, r.clock)
    before = o.owner.copy()
    rc, slots, mids, msl, counts = o.ensure_hybrid(0, r.topk_ids, 0)
    assert rc == orc.OK and mids.size == 0 and counts == (0, r.misses)
    assert np.array_equal(o.owner, before) and int(o.clock[0]) == 1
    assert (slots == -1).sum() == sum(1 for v in r.topk_ids.reshape(-1) if int(v) not in set(r.hits.tolist()))
