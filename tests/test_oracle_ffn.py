"""Pins of the oracle's expert FFN (CPU only).

The FFN is checked against closed forms, not against a second copy of itself:
  * sparse experts whose gate, up and down matrices hold one non-zero per output
    row at a chosen column (a permutation-like map); the FFN then reduces to
    y = sum_j w_j * c[n] * silu(a x[p]) * b x[q] evaluated element by element, so a
    transposed operand, a swapped gate/up half, a wrong nibble, scale block or
    global row fails;
  * the byte layout of each format, placed by an encoder written in this test
    (bytes in, value out), at random positions;
  * linearity of the combine in the router weights.
The readings of the layouts are those of the oracle's header (gate rows first, low
nibble = even k, nvfp4 scale per 16 along k, mxfp4 blocks transposed [K/2, N], block
FP8 one binary32 scale per 128 x 128 block, Q4_0 18-byte blocks of 32 with element j and
j + 16 in the low and high nibble of byte j).
"""
import math

import numpy as np
import pytest
import torch

from expert_slot_cache_device_gb300 import workload as wl

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def e4m3_val(b):
    return float(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).double())


def bf16_val(bits):
    return float(torch.tensor([np.int16(np.uint16(bits))], dtype=torch.int16).view(torch.bfloat16).double())


def f16_val(bits):
    return float(np.array([bits], np.uint16).view(np.float16)[0])


class ExpertBuilder:
    """Empty expert banks of one format plus an encoder that places single weights."""

    def __init__(self, fmt, H, I):
        self.fmt, self.H, self.I = fmt, H, I
        cfg = wl.Config("t", "t", 0, fmt, 1, 1, H, I, 1, 1, (1,), (1.0,), "uniform", 0.0, 0)
        self.banks = [np.zeros(g.bytes, np.uint8) for g in wl.bank_schema(cfg)]
        if fmt == "q4_0":  # zero weights: nibble 8 (q - 8 = 0) everywhere, scale 0 until used
            for bk in self.banks:
                blk = bk.reshape(-1, 18)
                blk[:, 2:] = 0x88

    def NK(self, which):
        return (2 * self.I, self.H) if which == 0 else (self.H, self.I)

    def place(self, which, n, k, rng):
        """Put a random non-zero weight at (n, k); returns its value."""
        N, K = self.NK(which)
        if self.fmt == "bf16":
            v = np.float32(rng.choice([0.5, -0.75, 1.25, 2.0, -1.5, 0.375]))
            bits = int(wl.f32_to_bf16_bits(np.array([v]))[0])
            self.banks[which].view(np.uint16)[n * K + k] = bits
            return bf16_val(bits)
        if self.fmt == "q4_0":
            # nibble at (n, k) of the row's 18-byte block; the block's binary16 scale is chosen
            # on its first use and shared by the block's 32 weights
            blk = self.banks[which].reshape(-1, 18)[n * (K // 32) + k // 32]
            j = k % 32
            q = int(rng.choice([0, 1, 3, 5, 7, 9, 10, 12, 15]))  # never 8 (that is zero)
            if j < 16:
                blk[2 + j] = (blk[2 + j] & 0xF0) | q
            else:
                blk[2 + j - 16] = (blk[2 + j - 16] & 0x0F) | (q << 4)
            d = blk[0:2].view(np.float16)
            if d[0] == 0:
                d[0] = np.float16(rng.choice([0.25, 0.0625, 1.5, 0.001953125, 3.0]))
            return (q - 8) * float(d[0])
        if self.fmt == "fp8":
            # e4m3 code at (n, k) of the row-major weight; the 128 x 128 block's binary32
            # scale is chosen on its first use and shared by every weight in the block
            wq, sc = self.banks[2 * which: 2 * which + 2]
            b = int(rng.choice([c for c in range(1, 127) if c != 0x7F] + [c | 0x80 for c in (1, 9, 56, 100, 126)]))
            wq[n * K + k] = b
            scv = sc.view(np.float32)
            j = (n // 128) * ((K + 127) // 128) + k // 128
            if scv[j] == 0.0:
                scv[j] = np.float32(rng.choice([0.125, 0.75, 1.5, 2.0 ** -9, 3.0]))
            return e4m3_val(b) * float(scv[j])
        code = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15]))
        if self.fmt == "nvfp4":
            codes, scales, glob = self.banks[3 * which: 3 * which + 3]
            byte = n * (K // 2) + k // 2
            codes[byte] = (codes[byte] & 0xF0) | code if k % 2 == 0 else (codes[byte] & 0x0F) | (code << 4)
            sb = int(rng.choice([0x30, 0x38, 0x3C, 0x40, 0x28, 0x44]))
            scales[n * (K // 16) + k // 16] = sb
            gbits = int(np.array([rng.uniform(0.25, 2.0)], np.float16).view(np.uint16)[0])
            glob.view(np.uint16)[n] = gbits
            return E2M1[code] * e4m3_val(sb) * f16_val(gbits)
        blocks, scales, _ = self.banks[3 * which: 3 * which + 3]
        byte = (k // 2) * N + n
        blocks[byte] = (blocks[byte] & 0xF0) | code if k % 2 == 0 else (blocks[byte] & 0x0F) | (code << 4)
        sb = int(rng.integers(124, 131))
        scales[(k // 32) * N + n] = sb
        return E2M1[code] * 2.0 ** (sb - 127)

    def set_bias(self, which, n, rng):
        if self.fmt != "mxfp4":
            return 0.0
        bits = int(wl.f32_to_bf16_bits(np.array([rng.normal(0, 0.5)], np.float32))[0])
        self.banks[3 * which + 2].view(np.uint16)[n] = bits
        return bf16_val(bits)


FMT_GEOMS = [("bf16", 64, 32), ("bf16", 48, 80), ("nvfp4", 64, 32), ("nvfp4", 96, 64), ("mxfp4", 64, 32),
             ("mxfp4", 96, 64), ("fp8", 256, 128), ("fp8", 128, 256), ("q4_0", 64, 32), ("q4_0", 96, 160)]


@pytest.mark.parametrize("fmt,H,I", FMT_GEOMS)
def test_single_weight_layout(orc, fmt, H, I):
    rng = np.random.default_rng(hash((fmt, H, I)) & 0xFFFF)
    for which in (0, 1):
        for _ in range(20):
            eb = ExpertBuilder(fmt, H, I)
            N, K = eb.NK(which)
            n, k = int(rng.integers(N)), int(rng.integers(K))
            v = eb.place(which, n, k, rng)
            assert orc.weight(fmt, which, eb.banks, H, I, n, k) == v
            for dn, dk in ((0, 1), (0, -1), (1, 0), (-1, 0), (0, 16), (0, 2)):
                n2, k2 = n + dn, k + dk
                if 0 <= n2 < N and 0 <= k2 < K:
                    assert orc.weight(fmt, which, eb.banks, H, I, n2, k2) == 0.0
            # the other matrix stays empty
            N2, K2 = eb.NK(1 - which)
            assert orc.weight(fmt, 1 - which, eb.banks, H, I, n % N2, k % K2) == 0.0


def silu(z):
    # z * sigmoid(z); for z < 0 the sigmoid is e^z / (1 + e^z), which neither overflows
    # nor cancels
    if z >= 0:
        return z / (1.0 + math.exp(-z))
    ez = math.exp(z)
    return z * ez / (1.0 + ez)


@pytest.mark.parametrize("fmt,H,I", FMT_GEOMS)
def test_ffn_sparse_closed_form(orc, fmt, H, I):
    rng = np.random.default_rng(7 + H + I)
    bs, k = 3, 2
    experts = []
    for _ in range(bs * k):
        eb = ExpertBuilder(fmt, H, I)
        p = rng.permutation(H)[:I] if I <= H else rng.integers(0, H, I)
        q = rng.permutation(H)[:I] if I <= H else rng.integers(0, H, I)
        r = rng.integers(0, I, H)
        a = [eb.place(0, i, int(p[i]), rng) for i in range(I)]
        b = [eb.place(0, I + i, int(q[i]), rng) for i in range(I)]
        c = [eb.place(1, n, int(r[n]), rng) for n in range(H)]
        ba = [eb.set_bias(0, i, rng) for i in range(I)]
        bb = [eb.set_bias(0, I + i, rng) for i in range(I)]
        bc = [eb.set_bias(1, n, rng) for n in range(H)]
        experts.append((eb.banks, p, q, r, a, b, c, ba, bb, bc))
    xbits = wl.f32_to_bf16_bits(rng.standard_normal((bs, H)).astype(np.float32))
    xv = torch.from_numpy(xbits.view(np.int16)).view(torch.bfloat16).double().numpy()
    w = rng.random((bs, k)).astype(np.float32)
    y = orc.expert_ffn(fmt, H, I, [e[0] for e in experts], xbits, w)
    for t in range(bs):
        want = np.zeros(H)
        mag = np.zeros(H)  # sum of |terms|: the rounding-order difference scales with it
        for j in range(k):
            _, p, q, r, a, b, c, ba, bb, bc = experts[t * k + j]
            h = [silu(a[i] * xv[t, p[i]] + ba[i]) * (b[i] * xv[t, q[i]] + bb[i]) for i in range(I)]
            o = np.array([c[n] * h[r[n]] + bc[n] for n in range(H)])
            want += float(w[t, j]) * o
            mag += abs(float(w[t, j])) * np.abs(o)
        err = np.abs(y[t] - want)
        assert (err <= 1e-12 + 1e-13 * mag).all(), (err.max(), mag.max())


def test_ffn_linear_in_router_weights(orc):
    cfg = wl.scaled(wl.CONFIGS["c3"], E=4, H=128, I=64)
    banks = wl.make_banks(cfg)
    rng = np.random.default_rng(3)
    ids = [[0, 2], [1, 2], [3, 3]]
    pair = [[bk[e] for bk in banks] for row in ids for e in row]
    x = wl.f32_to_bf16_bits(rng.standard_normal((3, cfg.H)).astype(np.float32))
    # dyadic weights: their sums are exact in fp32, so only fp64 rounding remains
    w1 = (rng.integers(1, 64, (3, 2)) / 64.0).astype(np.float32)
    w2 = (rng.integers(1, 64, (3, 2)) / 64.0).astype(np.float32)
    y1 = orc.expert_ffn("nvfp4", cfg.H, cfg.I, pair, x, w1)
    y2 = orc.expert_ffn("nvfp4", cfg.H, cfg.I, pair, x, w2)
    y12 = orc.expert_ffn("nvfp4", cfg.H, cfg.I, pair, x, (w1.astype(np.float64) + w2).astype(np.float32))
    np.testing.assert_allclose(y12, y1 + y2, rtol=1e-12, atol=1e-14)
    # a duplicated expert with weights (a, b) equals a single one with a + b
    wd = np.array([[0.25, 0.5]], np.float32)
    yd = orc.expert_ffn("nvfp4", cfg.H, cfg.I, pair[4:6], x[2:3], wd)
    ys = orc.expert_ffn("nvfp4", cfg.H, cfg.I, pair[4:5], x[2:3], np.array([[0.75]], np.float32))
    np.testing.assert_allclose(yd, ys, rtol=1e-12, atol=1e-12)


def test_workload_output_magnitudes(orc):
    """The synthetic value distributions keep outputs O(1) (so the absolute
    tolerance measures arithmetic error, not the bf16 rounding of large outputs)."""
    for key in ("c2", "c3", "c4"):
        cfg = wl.CONFIGS[key]
        sub = wl.scaled(cfg)
        banks = wl.make_banks(sub, experts=[0, 1])
        rng = np.random.default_rng(5)
        x = wl.f32_to_bf16_bits(rng.standard_normal((1, cfg.H)).astype(np.float32))
        pair = [[bk[0] for bk in banks], [bk[1] for bk in banks]]
        y = orc.expert_ffn(cfg.fmt, cfg.H, cfg.I, pair, x, np.array([[0.6, 0.4]], np.float32))
        rms = float(np.sqrt(np.mean(y ** 2)))
        assert 0.05 < rms < 4.0, (key, rms)
