"""A cache over the caller's own banks (GPU): plain page-locked tensors and caller-owned slot
banks, no workload configuration, one decode step of two layers checked against the oracle."""
import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import oracle
    from expert_slot_cache_device_gb300 import build

    build.build()
    oracle.build()


def test_cache_over_caller_banks():
    import oracle
    from expert_slot_cache_device_gb300 import ftmoe as F
    from expert_slot_cache_device_gb300.cache import Bank, ExpertSlotCache

    E, L, S, H, I, k, bs = 6, 3, 5, 256, 128, 2, 3
    g = torch.Generator().manual_seed(3)
    # bf16 banks drawn here, one per layer, caller-owned slot banks
    banks = [Bank("gate_up", "bf16", 2 * I, 2 * H), Bank("down", "bf16", H, 2 * I)]
    host = [[(torch.randn(E * b.bytes // 2, generator=g) * 0.05).to(torch.bfloat16).view(torch.uint8).pin_memory()
             for _ in range(L)] for b in banks]
    slots = [torch.zeros((S, b.bytes), dtype=torch.uint8, device="cuda") for b in banks]
    cache = ExpertSlotCache("bf16", E, L, S, H, I, banks, host, max_pairs=bs * k, slot_banks=slots)
    assert cache.slots[0].data_ptr() == slots[0].data_ptr()
    orc = oracle.Cache(E, L, S)
    rng = np.random.default_rng(5)
    for layer in (2, 0):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(bs)]).astype(np.int32)
        w = rng.random((bs, k)).astype(np.float32)
        x = torch.randn((bs, H), generator=g).to(torch.bfloat16)
        d_ids = torch.from_numpy(ids).cuda()
        d_slots = torch.empty((bs, k), dtype=torch.int32, device="cuda")
        d_y = torch.empty((bs, H), dtype=torch.bfloat16, device="cuda")
        cache.ensure(layer, d_ids, d_slots)
        cache.copy_missing()
        cache.ffn(x.cuda(), d_slots, torch.from_numpy(w).cuda(), d_y)
        torch.cuda.synchronize()
        assert cache.status() == F.OK
        rc, want_slots, mids, msl = orc.ensure(layer, ids)
        assert rc == oracle.OK and np.array_equal(d_slots.cpu().numpy(), want_slots)
        for b in range(2):
            for f, s in zip(mids.tolist(), msl.tolist()):
                assert torch.equal(slots[b][s].cpu(), cache.host_tensor(b, layer)[f % E])
        pairs = [cache.expert_host_ptrs(layer, int(e)) for e in ids.reshape(-1)]
        x_bits = x.view(torch.int16).numpy().view(np.uint16)
        ref = oracle.expert_ffn("bf16", H, I, pairs, x_bits, w)
        y = d_y.float().cpu().numpy().astype(np.float64)
        assert np.abs(y - ref).max() <= 2e-2 and np.linalg.norm(y - ref) / np.linalg.norm(ref) <= 1e-2
    cache.close()
