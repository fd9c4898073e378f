"""Pins of the oracle's number formats against things other than the oracle:
the published E2M1 table, torch's float8_e4m3fn decode and RNE cast, and
hand-worked closed-form cases."""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_e2m1():
    out = {}
    for line in open(os.path.join(GOLDEN, "e2m1_values.txt")):
        line = line.split("#")[0].strip()
        if line:
            c, v = line.split()
            out[int(c)] = float(v)
    return out


def test_e2m1_matches_published_table():
    table = _golden_e2m1()
    assert len(table) == 16
    for code, v in table.items():
        got = oracle.e2m1_value(code)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (code, got, v)


def _torch_e4m3(codes):
    return torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_all_codes_match_torch():
    ref = _torch_e4m3(list(range(256)))
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # S.1111.111
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_round_fixed_points():
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(v):
            assert oracle.e4m3_round(v) & 0x7F == 0x7F
        else:
            assert oracle.e4m3_round(v) == c, c


def test_e4m3_round_midpoints_tie_to_even_and_match_torch():
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]  # non-negative finite, increasing
    mids, want = [], []
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        m = (lo + hi) / 2
        mids.append(m)
        want.append(c if c % 2 == 0 else c + 1)
        # just off the midpoint goes to the nearer neighbour
        assert oracle.e4m3_round(np.nextafter(m, 0)) == c
        assert oracle.e4m3_round(np.nextafter(m, 1e9)) == c + 1
    got = [oracle.e4m3_round(m) for m in mids]
    assert got == want
    tref = torch.tensor(mids, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    assert got == tref
    assert [oracle.e4m3_round(-m) for m in mids] == [w | 0x80 for w in want]


def test_e4m3_round_random_float32_match_torch():
    rng = np.random.default_rng(7)
    mag = np.exp2(rng.uniform(-13, 9.2, size=20000)).astype(np.float32)
    x = (mag * rng.choice([-1, 1], size=mag.size)).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_round(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_round_saturates_instead_of_overflowing():
    for x in (448.0, 449.0, 463.9, 464.0, 464.1, 1e6, math.inf):
        assert oracle.e4m3_round(x) == 0x7E
        assert oracle.e4m3_round(-x) == 0xFE
    assert math.isnan(oracle.e4m3_value(oracle.e4m3_round(math.nan)))


def test_dequant_table_exhaustive_matches_independent_round():
    """All 256 scales x 16 codes: exact FP64 product, then torch's RNE cast
    to E4M3 after clamping to +-448 (saturating), decoded again."""
    tab = oracle.dequant_table()
    e2m1 = np.array([_golden_e2m1()[c] for c in range(16)])
    scale = _torch_e4m3(list(range(256)))
    prod = scale[:, None] * e2m1[None, :]
    nan = np.isnan(prod)
    ref = torch.from_numpy(np.clip(np.nan_to_num(prod), -448, 448).astype(np.float32)).to(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    assert np.array_equal(np.isnan(tab), nan)
    assert np.array_equal(tab[~nan], ref[~nan])
    # 2,048 distinct (scale, magnitude) entries, the size of a byte-per-entry
    # table over 256 scales x 8 magnitudes
    assert tab[:, :8].size == 2048


def test_dequant_hand_cases():
    # scale 0x38 = 1.0: the E2M1 values themselves
    for c, v in _golden_e2m1().items():
        assert oracle.dequant_value(c, 0x38) == v
    # scale 0x39 = 1.125; 1.5 * 1.125 = 1.6875 lies halfway between 1.625 (odd
    # mantissa) and 1.75 (even) -> 1.75
    assert oracle.dequant_value(3, 0x39) == 1.75
    # 3 * 1.125 = 3.375 -> halfway between 3.25 and 3.5 -> 3.5 (even)
    assert oracle.dequant_value(5, 0x39) == 3.5
    # 6 * 448 saturates to 448
    assert oracle.dequant_value(7, 0x7E) == 448.0
    # 0.5 * 2^-9 = 2^-10 is halfway between 0 and 2^-9 -> 0
    assert oracle.dequant_value(1, 0x01) == 0.0
    # 1.5 * 2^-9 -> halfway between 2^-9 and 2^-8 -> 2^-8 (even code 2)
    assert oracle.dequant_value(3, 0x01) == 2.0 ** -8
