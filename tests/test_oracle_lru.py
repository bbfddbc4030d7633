"""Pins of the oracle's LRU ensure_experts (CPU only).

The oracle's LRU is checked against things other than itself:
  * a brute-force LRU written differently (one miss at a time, a full linear scan for
    the least recently used untouched slot, lowest slot first on equal recency);
  * a hand-worked trace and the worked tiny case of the cache-copy benchmark
    (FreeToken MoE offline benchmark guide, section 4.3: flat id = layer * E + expert,
    prepared state in which every slot belongs to another layer);
  * the closed-form miss count round(min(E, bs * topk) * miss_rate) on the prepared
    state of every workload point (same section);
  * invariants: owner and id2slot stay inverse, hits never move, capacity errors leave
    the state untouched.
"""
import numpy as np
import pytest

from conftest import golden_lines
from expert_slot_cache_device_gb300 import workload as wl


class BruteLRU:
    """Recency cache over S slots, one eviction decision at a time."""

    def __init__(self, E, L, S, owner=None, stamp=None, clock=0):
        self.E, self.L, self.S = E, L, S
        self.owner = [-1] * S if owner is None else [int(v) for v in owner]
        self.last_use = [0] * S if stamp is None else [int(v) for v in stamp]
        self.clock = clock

    def where(self, f):
        for s in range(self.S):
            if self.owner[s] == f:
                return s
        return -1

    def ensure(self, layer, ids):
        ids = [int(v) for v in np.asarray(ids).reshape(-1)]
        if any(i < 0 or i >= self.E for i in ids):
            return "ERR_ID_RANGE", None, None, None
        now = self.clock + 1
        used_now = set()
        wanted = sorted(set(layer * self.E + i for i in ids))
        missing = []
        for f in wanted:
            s = self.where(f)
            if s >= 0:
                used_now.add(s)
            else:
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


def check_inverse(c):
    for s in range(c.S):
        f = int(c.owner[s])
        if f >= 0:
            assert c.id2slot[f] == s
    for f in range(c.E * c.L):
        s = int(c.id2slot[f])
        if s >= 0:
            assert c.owner[s] == f


@pytest.mark.parametrize("seed", range(12))
def test_oracle_matches_brute_force_lru(orc, seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(2, 9))
    L = int(rng.integers(1, 4))
    k = int(rng.integers(1, min(E, 4) + 1))
    S = int(rng.integers(k, k + 5))
    bs = int(rng.integers(1, 3))
    zipf = [0.0, 1.1, 2.0][seed % 3]
    trace = wl.random_trace_ids(seed, 300, E, L, bs, k, zipf)
    o = orc.Cache(E, L, S)
    b = BruteLRU(E, L, S)
    errors = 0
    for layer, ids in trace:
        before = (o.owner.copy(), o.stamp.copy(), int(o.clock[0]))
        rc, slots, mids, msl = o.ensure(layer, ids)
        st, bslots, bmiss, bms = b.ensure(layer, ids)
        if st == "OK":
            assert rc == orc.OK
            assert slots.reshape(-1).tolist() == bslots
            assert mids.tolist() == bmiss and msl.tolist() == bms
            assert o.owner.tolist() == b.owner
            assert o.stamp.tolist() == b.last_use
            assert int(o.clock[0]) == b.clock
        else:
            errors += 1
            assert rc == orc.ERR_CAPACITY
            assert (slots == -1).all() and mids.size == 0
            assert np.array_equal(o.owner, before[0]) and np.array_equal(o.stamp, before[1])
            assert int(o.clock[0]) == before[2]
        check_inverse(o)
    assert errors < len(trace)


def test_oracle_every_tie_pattern_small(orc):
    """Exhaustive: all stamp patterns over 4 slots with values in {0,1,2} and every id set
    of a 4-expert layer; the victim order must be ascending (stamp, slot)."""
    import itertools

    E, L, S = 4, 2, 4
    for stamps in itertools.product(range(3), repeat=S):
        for mask in range(1, 16):
            ids = [e for e in range(E) if mask >> e & 1]
            owner = [E + s for s in range(S)]
            o = orc.Cache(E, L, S, owner, stamps, clock=2)
            b = BruteLRU(E, L, S, owner, stamps, clock=2)
            rc, slots, mids, msl = o.ensure(0, np.array(ids, np.int32))
            st, bslots, bmiss, bms = b.ensure(0, ids)
            assert st == "OK" and rc == orc.OK
            assert msl.tolist() == bms
            want = sorted(range(S), key=lambda s: (stamps[s], s))[: len(ids)]
            assert msl.tolist() == want


def test_hand_worked_trace(orc):
    o = orc.Cache(4, 2, 3)
    for ln in golden_lines("lru_trace_hand.txt"):
        parts = [p.strip() for p in ln.split("|")]
        layer = int(parts[0])
        ids = np.array([int(v) for v in parts[1].split()], np.int32)
        before = (o.owner.copy(), o.stamp.copy(), int(o.clock[0]))
        rc, slots, mids, msl = o.ensure(layer, ids)
        if parts[2] == "ERR_CAPACITY":
            assert rc == orc.ERR_CAPACITY
            assert np.array_equal(o.owner, before[0]) and np.array_equal(o.stamp, before[1])
            assert int(o.clock[0]) == before[2]
            continue
        assert rc == orc.OK
        assert slots.tolist() == [int(v) for v in parts[2].split()]
        exp_m = [] if parts[3] == "-" else [int(v) for v in parts[3].split()]
        exp_s = [] if parts[4] == "-" else [int(v) for v in parts[4].split()]
        assert mids.tolist() == exp_m and msl.tolist() == exp_s
        assert o.owner.tolist() == [int(v) for v in parts[5].split()]
        assert o.stamp.tolist() == [int(v) for v in parts[6].split()]


def test_worked_tiny_case(orc):
    g = {}
    for ln in golden_lines("c1_worked.txt"):
        key, *vals = ln.split()
        g[key] = vals
    cfg = wl.CONFIGS["c1"]
    r = wl.make_route(cfg, 1, 1.0)
    a, b = sorted(np.unique(r.topk_ids).tolist())
    sub = {"a": a, "b": b}
    val = lambda v: sub[v] if v in sub else int(v)
    assert r.owner.tolist() == [val(v) for v in g["owner_before"]]
    assert r.stamp.tolist() == [val(v) for v in g["stamp_before"]]
    o = orc.Cache(cfg.E, cfg.L, cfg.S, r.owner, r.stamp, r.clock)
    rc, slots, mids, msl = o.ensure(int(g["layer"][0]), r.topk_ids)
    assert rc == orc.OK
    assert mids.tolist() == [val(v) for v in g["misses"]]
    assert msl.tolist() == [val(v) for v in g["miss_slots"]]
    assert o.owner.tolist() == [val(v) for v in g["owner_after"]]
    assert o.stamp.tolist() == [val(v) for v in g["stamp_after"]]
    assert int(o.clock[0]) == int(g["clock_after"][0])


def test_miss_counts_closed_form(orc):
    """Every benchmark point: the prepared state realises exactly the planned misses,
    and those equal the table written from round(min(E, bs*k) * miss_rate)."""
    rows = [ln.split() for ln in golden_lines("miss_counts.txt")]
    assert len(rows) == 1 + 12 + 9 + 6
    for key, E, k, bs, mr, active, misses in rows:
        cfg = wl.CONFIGS[key]
        assert (cfg.E, cfg.topk) == (int(E), int(k))
        r = wl.make_route(cfg, int(bs), float(mr))
        assert r.active == int(active) == len(np.unique(r.topk_ids))
        assert r.misses == int(misses)
        o = orc.Cache(cfg.E, cfg.L, cfg.S, r.owner, r.stamp, r.clock)
        rc, slots, mids, msl = o.ensure(0, r.topk_ids)
        assert rc == orc.OK
        assert mids.size == int(misses)
        # the driven layer hits exactly the planned hits, nothing else
        assert len(set(slots.reshape(-1).tolist()) & set(range(len(r.hits)))) == len(r.hits)
        if float(mr) == 1.0:
            assert msl.tolist() == list(range(int(misses)))  # stamps all 0: lowest slots first


def test_prepared_state_never_hits(orc):
    """A prepared state with every slot owned by another layer gives zero hits."""
    for key in ("c1", "c2", "c3", "c4"):
        cfg = wl.CONFIGS[key]
        owner, stamp, clock = wl.prepared_state(cfg, [])
        assert all(int(f) // cfg.E != 0 for f in owner)
        r = wl.make_route(cfg, cfg.bs_list[-1], cfg.mr_list[-1])
        o = orc.Cache(cfg.E, cfg.L, cfg.S, owner, stamp, clock)
        rc, slots, mids, msl = o.ensure(0, r.topk_ids)
        assert rc == orc.OK and mids.size == len(np.unique(r.topk_ids))


def test_error_paths(orc):
    o = orc.Cache(4, 2, 2)
    rc, slots, mids, _ = o.ensure(0, np.array([0, 4], np.int32))
    assert rc == orc.ERR_ID_RANGE and (slots == -1).all() and mids.size == 0
    rc, *_ = o.ensure(0, np.array([-1], np.int32))
    assert rc == orc.ERR_ID_RANGE
    rc, *_ = o.ensure(2, np.array([0], np.int32))
    assert rc == orc.ERR_INVALID_ARG
    rc, *_ = o.ensure(0, np.array([0, 1, 2], np.int32))
    assert rc == orc.ERR_CAPACITY
    assert int(o.clock[0]) == 0 and (o.owner == -1).all()
    o2 = orc.Cache(4, 2, 2, clock=0xFFFFFFFF)
    rc, *_ = o2.ensure(0, np.array([0], np.int32))
    assert rc == orc.ERR_STATE
    with pytest.raises(ValueError):
        orc.Cache(4, 2, 2, owner=[3, 3])
    # an empty call only ticks the clock
    rc, slots, mids, _ = o.ensure(1, np.zeros(0, np.int32))
    assert rc == orc.OK and mids.size == 0 and int(o.clock[0]) == 1


def test_layers_do_not_alias(orc):
    """Same local expert in two layers are different flat ids (no hit across layers)."""
    o = orc.Cache(4, 3, 3)
    rc, _, m0, s0 = o.ensure(0, np.array([1], np.int32))
    rc, _, m1, s1 = o.ensure(2, np.array([1], np.int32))
    assert m0.tolist() == [1] and m1.tolist() == [9] and s0.tolist() != s1.tolist()
    rc, slots, m2, _ = o.ensure(0, np.array([1], np.int32))
    assert m2.size == 0 and slots.tolist() == s0.tolist()
