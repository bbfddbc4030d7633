"""The hybrid path's CPU expert executor (host code of libftmoe) against the oracle.

FreeToken benchmark guide, section 5.4: misses beyond the fetch cap get slot -1 and are
computed by a CPU executor from the host banks. This runs on the CPU only: for every
format, the executor's fp32 partial output over the -1 positions must match the fp64
oracle FFN restricted to those positions. On an Arm host with the BF16 extension (the Grace
host of the GPU machines) the executor's dot products run on BFDOT, elsewhere on fp32 loops;
the same tolerance holds for both.
"""
import numpy as np
import pytest

from expert_slot_cache_device_gb300 import build as B
from expert_slot_cache_device_gb300 import ftmoe as F
from expert_slot_cache_device_gb300 import workload as wl

CASES = [("bf16", dict(E=6, H=264, I=72)), ("nvfp4", dict(E=5, H=320, I=96)), ("mxfp4", dict(E=5, H=160, I=96)),
         ("mxfp4", dict(E=4, H=576, I=320))]


@pytest.fixture(scope="module")
def lib():
    B.build()
    return F.lib()


@pytest.mark.parametrize("fmt,geo", CASES)
def test_cpu_executor_matches_oracle(lib, orc, fmt, geo):
    base = {"bf16": "c2", "nvfp4": "c3", "mxfp4": "c4"}[fmt]
    cfg = wl.scaled(wl.CONFIGS[base], topk=3, L=2, S=4, **geo)
    banks = wl.make_banks(cfg)
    rng = np.random.default_rng(geo["H"])
    bs = 5
    ids = np.stack([rng.choice(cfg.E, cfg.topk, replace=False) for _ in range(bs)]).astype(np.int32)
    slots = rng.integers(0, cfg.S, ids.shape).astype(np.int32)
    cpu_mask = rng.random(ids.shape) < 0.6
    cpu_mask[0, :] = True
    slots[cpu_mask] = -1
    w = rng.random(ids.shape).astype(np.float32)
    x = wl.f32_to_bf16_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))
    y = np.empty((bs, cfg.H), np.float32)
    F.ftmoe_cpu_expert_ffn(F.FORMATS[fmt], cfg.H, cfg.I, bs, cfg.topk, ids.ctypes.data, slots.ctypes.data,
                           [b.ctypes.data for b in banks], [b.shape[1] for b in banks], x.ctypes.data, w.ctypes.data,
                           y.ctypes.data, 4)
    w_cpu = np.where(cpu_mask, w, 0.0).astype(np.float32)
    pairs = [[b[int(e)] for b in banks] for e in ids.reshape(-1)]
    ref = orc.expert_ffn(fmt, cfg.H, cfg.I, pairs, x, w_cpu)
    err = np.abs(y - ref).max()
    l2 = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert err <= 1e-4 and l2 <= 1e-5, (err, l2)  # fp32 accumulation against fp64


def test_cpu_executor_no_cpu_pairs_gives_zero(lib):
    cfg = wl.scaled(wl.CONFIGS["c2"], E=2, H=64, I=32, topk=1)
    banks = wl.make_banks(cfg)
    ids = np.zeros((2, 1), np.int32)
    slots = np.zeros((2, 1), np.int32)
    x = np.zeros((2, 64), np.uint16)
    w = np.ones((2, 1), np.float32)
    y = np.full((2, 64), 7.0, np.float32)
    F.ftmoe_cpu_expert_ffn(F.FMT_BF16, 64, 32, 2, 1, ids.ctypes.data, slots.ctypes.data,
                           [b.ctypes.data for b in banks], [b.shape[1] for b in banks], x.ctypes.data, w.ctypes.data,
                           y.ctypes.data, 2)
    assert (y == 0).all()


def test_fetch_fraction_helper(lib):
    assert F.ftmoe_hybrid_fetch_fraction(200.0, 800.0) == pytest.approx(0.25)
    assert F.ftmoe_hybrid_fetch_fraction(200.0, 150.0) == 1.0
    assert F.ftmoe_hybrid_fetch_fraction(0.0, 800.0) == 0.0
    with pytest.raises(F.FtmoeError):
        F.ftmoe_cpu_expert_ffn(9, 64, 32, 1, 1, 0, 0, [0, 0], [1, 1], 0, 0, 0, 1)


def test_cpu_read_ceiling_probe(lib):
    """The STREAM-style host read probe runs on the host cores: a positive rate for a real
    buffer, host-side argument errors otherwise."""
    buf = np.arange(1 << 22, dtype=np.uint8)
    gbps = F.ftmoe_measure_cpu_read(buf.ctypes.data, buf.nbytes, 2, 2)
    assert 0.1 < gbps < 1e5
    for args in ((0, buf.nbytes, 1, 1), (buf.ctypes.data, 32, 1, 1), (buf.ctypes.data, buf.nbytes, 1, 0)):
        with pytest.raises(F.FtmoeError) as e:
            F.ftmoe_measure_cpu_read(*args)
        assert e.value.code == F.ERR_INVALID_ARG


def test_cpu_executor_concurrent_calls(lib):
    """The executor's worker pool is shared: calls from several host threads at once (ctypes
    releases the GIL), with different formats and worker counts, queue on it and each returns
    exactly what the same call returns alone."""
    import threading

    jobs = []
    for i, (fmt, geo) in enumerate(CASES * 2):
        base = {"bf16": "c2", "nvfp4": "c3", "mxfp4": "c4"}[fmt]
        cfg = wl.scaled(wl.CONFIGS[base], topk=2, L=2, S=4, **geo)
        banks = wl.make_banks(cfg)
        rng = np.random.default_rng(100 + i)
        bs = 3
        ids = np.stack([rng.choice(cfg.E, cfg.topk, replace=False) for _ in range(bs)]).astype(np.int32)
        slots = np.full(ids.shape, -1, np.int32)
        w = rng.random(ids.shape).astype(np.float32)
        x = wl.f32_to_bf16_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))
        jobs.append((fmt, cfg, banks, ids, slots, w, x, 1 + (3 * i) % 7))

    def run(job, out):
        fmt, cfg, banks, ids, slots, w, x, threads = job
        F.ftmoe_cpu_expert_ffn(F.FORMATS[fmt], cfg.H, cfg.I, ids.shape[0], cfg.topk, ids.ctypes.data,
                               slots.ctypes.data, [b.ctypes.data for b in banks], [b.shape[1] for b in banks],
                               x.ctypes.data, w.ctypes.data, out.ctypes.data, threads)

    alone = []
    for job in jobs:
        y = np.empty((job[3].shape[0], job[1].H), np.float32)
        run(job, y)
        alone.append(y)
    for _ in range(3):
        outs = [np.full_like(y, np.nan) for y in alone]
        ts = [threading.Thread(target=run, args=(job, out)) for job, out in zip(jobs, outs)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        for y, y0 in zip(outs, alone):
            assert np.array_equal(y, y0)


@pytest.mark.filterwarnings("ignore::DeprecationWarning")  # Python warns about fork in a threaded process
def test_cpu_executor_after_fork(lib):
    """A process forked after the executor has run (its worker pool started) runs the executor
    itself with a pool of its own and gets the parent's result."""
    import os

    fmt, geo = CASES[0]
    cfg = wl.scaled(wl.CONFIGS["c2"], topk=2, L=2, S=4, **geo)
    banks = wl.make_banks(cfg)
    rng = np.random.default_rng(5)
    ids = np.stack([rng.choice(cfg.E, cfg.topk, replace=False) for _ in range(3)]).astype(np.int32)
    slots = np.full(ids.shape, -1, np.int32)
    w = rng.random(ids.shape).astype(np.float32)
    x = wl.f32_to_bf16_bits(rng.standard_normal((3, cfg.H)).astype(np.float32))

    def run():
        y = np.empty((3, cfg.H), np.float32)
        F.ftmoe_cpu_expert_ffn(F.FMT_BF16, cfg.H, cfg.I, 3, cfg.topk, ids.ctypes.data, slots.ctypes.data,
                               [b.ctypes.data for b in banks], [b.shape[1] for b in banks], x.ctypes.data,
                               w.ctypes.data, y.ctypes.data, 4)
        return y

    y0 = run()  # starts the parent's workers
    pid = os.fork()
    if pid == 0:  # child: exit status 0 only if the call returns the parent's bits
        code = 1
        try:
            code = 0 if np.array_equal(run(), y0) else 2
        finally:
            os._exit(code)
    import time

    deadline = time.monotonic() + 60
    while True:
        done, status = os.waitpid(pid, os.WNOHANG)
        if done:
            break
        if time.monotonic() > deadline:
            os.kill(pid, 9)
            os.waitpid(pid, 0)
            raise AssertionError("the forked executor call did not return")
        time.sleep(0.05)
    assert os.WIFEXITED(status) and os.WEXITSTATUS(status) == 0
    assert np.array_equal(run(), y0)
