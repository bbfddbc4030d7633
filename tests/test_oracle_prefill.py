"""Pins of the whole-layer double-buffered prefill schedule on the oracle's LRU (CPU only).

Architecture deep-dive, section 五: the global LRU expert cache streams prefill layer by
layer through a double buffer, copies overlapping compute. The schedule built on it is
prefetch(layer) = ensure of all E experts, then the routed ensure of the same layer. With
S = 2E the plain LRU rules fix what must happen, checked here against closed forms:
- the routed ensure after a prefetch never misses;
- a prefetch never evicts the layer that is still computing (the previous step's), so the
  two layers in flight always occupy disjoint slots;
- from the third step on, a prefetch takes exactly the slots of the step before last (the
  double buffer), in ascending slot order for a prefetch into a cold cache.
"""
import numpy as np
import pytest


def schedule(orc, E, L, S, steps, k, seed):
    rng = np.random.default_rng(seed)
    o = orc.Cache(E, L, S)
    layers = [int(v) for v in rng.integers(0, L, steps)]
    # consecutive steps run different layers, as a model's layers do
    for i in range(1, steps):
        if layers[i] == layers[i - 1]:
            layers[i] = (layers[i] + 1) % L
    held, log = [], []
    for i, layer in enumerate(layers):
        rc, slots, mids, msl = o.ensure(layer, np.arange(E, dtype=np.int32)[None, :])
        assert rc == orc.OK
        ids = np.stack([rng.permutation(E)[:k] for _ in range(3)]).astype(np.int32)
        rc2, rslots, rmids, _ = o.ensure(layer, ids)
        assert rc2 == orc.OK
        log.append((layer, slots.reshape(-1).copy(), mids.copy(), msl.copy(), rmids.size, rslots))
        held.append(set(int(s) for s in slots.reshape(-1)))
    return layers, held, log


@pytest.mark.parametrize("seed", range(4))
def test_prefill_double_buffer_closed_forms(orc, seed):
    E, L, k = 8, 5, 3
    S = 2 * E
    layers, held, log = schedule(orc, E, L, S, 12, k, seed)
    for i, (layer, slots, mids, msl, rmiss, rslots) in enumerate(log):
        assert rmiss == 0, "routed ensure after a prefetch must hit"
        assert len(held[i]) == E
        if i >= 1:
            assert held[i].isdisjoint(held[i - 1]), "prefetch evicted the layer still computing"
        if i >= 2 and layers[i] != layers[i - 2]:
            assert held[i] == held[i - 2], "the prefetch reuses the step-before-last's slots"
    # cold start: the first prefetch fills slots 0..E-1 in ascending expert order
    assert log[0][1].tolist() == list(range(E))
    assert log[0][2].tolist() == [log[0][0] * E + e for e in range(E)]


def test_prefill_needs_two_layers_of_slots(orc):
    """With S < 2E the next prefetch must evict some of the computing layer's experts."""
    E, L = 8, 3
    o = orc.Cache(E, L, 2 * E - 1)
    rc, s0, _, _ = o.ensure(0, np.arange(E, dtype=np.int32)[None, :])
    rc, s1, _, _ = o.ensure(1, np.arange(E, dtype=np.int32)[None, :])
    assert rc == orc.OK
    assert set(s0.reshape(-1).tolist()) & set(s1.reshape(-1).tolist())
