"""Pins of the oracle's number-format decoders (CPU only).

Each decoder is checked over its whole code space against an independent source:
the OCP MX v1.0 E2M1 table (golden fixture), torch's float8_e4m3fn / float8_e8m0fnu
casts, numpy's IEEE binary16 and torch's bfloat16.
"""
import math

import numpy as np
import torch

from conftest import golden_lines


def test_e2m1_table(orc):
    rows = [ln.split() for ln in golden_lines("e2m1_values.txt")]
    codes = [int(c) for c, _ in rows]
    want = [float(v) for _, v in rows]
    got = orc.decode("e2m1", codes)
    assert codes == list(range(16))
    for c, g, w in zip(codes, got, want):
        assert g == w and math.copysign(1.0, g) == math.copysign(1.0, w), (c, g, w)


def test_e4m3_all_bytes(orc):
    got = orc.decode("e4m3", np.arange(256))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.flatnonzero(nan).tolist() == [0x7F, 0xFF]
    assert np.array_equal(got[~nan], ref[~nan])
    # spec landmarks: max normal, min normal, min subnormal, one
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e8m0_all_bytes(orc):
    got = orc.decode("e8m0", np.arange(256))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert got[127] == 1.0 and got[118] == 2.0 ** -9


def test_f16_all_codes(orc):
    codes = np.arange(65536, dtype=np.uint32)
    got = orc.decode("f16", codes)
    ref = codes.astype(np.uint16).view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_all_codes(orc):
    codes = np.arange(65536, dtype=np.uint32)
    got = orc.decode("bf16", codes)
    ref = torch.from_numpy(codes.astype(np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
