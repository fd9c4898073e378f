"""Pins of the oracle's NVFP4 quantiser (the KV-insert step).

[vLLM-zh] "QKV GEMM + norm + RoPE + KV insert fusion": the epilogue quantises the FP32
K, V and index keys to NVFP4 and writes them into the caches. NVFP4 here: per 16
elements one E4M3 scale = amax / 6 rounded to nearest (ties to even, saturating), and
per element the E2M1 value nearest x / scale (ties to the even code, saturating at 6).

The pins below come from the two formats' definitions, closed forms and a brute-force
nearest-value search written independently of the oracle (numpy over every candidate
value), not from the oracle's own code.
"""
import numpy as np
import pytest
import torch

import oracle

# E2M1 magnitudes, codes 0..7, from the format (bias 1, one mantissa bit)
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
# E4M3 values of the non-negative finite codes 0..126, decoded by torch's own float8 type
E4M3 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_grid_is_increasing_and_ends_at_448():
    assert E4M3[0] == 0.0 and E4M3[1] == 2.0 ** -9 and E4M3[126] == 448.0
    assert np.all(np.diff(E4M3) > 0)


def test_e2m1_round_on_grid_and_at_midpoints():
    for c, m in enumerate(E2M1):
        assert oracle.e2m1_round(m) == c
        if c:
            assert oracle.e2m1_round(-m) == 8 | c
    # the midpoint between codes lo and lo + 1 goes to the even one of the two; just
    # above it to lo + 1, just below it to lo
    for lo in range(7):
        y = 0.5 * (E2M1[lo] + E2M1[lo + 1])
        even = lo if lo % 2 == 0 else lo + 1
        assert oracle.e2m1_round(y) == even, y
        assert oracle.e2m1_round(-y) == 8 | even, -y
        assert oracle.e2m1_round(y * (1 + 1e-12)) == lo + 1, y
        assert oracle.e2m1_round(y * (1 - 1e-12)) == lo, y
    for y in (6.0, 6.5, 7.0, 100.0, 1e30):
        assert oracle.e2m1_round(y) == 7 and oracle.e2m1_round(-y) == 15


def _group(amax, rest=0.0):
    x = np.full(16, rest, np.float32)
    x[5] = amax
    return x


def test_scale_of_exact_multiples():
    """amax = 6 v(c) exactly gives scale code c, for every positive finite E4M3 code."""
    rows = np.stack([np.tile(_group(np.float32(6.0 * E4M3[c])), 8) for c in range(1, 127)])
    assert np.all(rows.astype(np.float64)[:, 5] == 6.0 * E4M3[1:127])  # exact in FP32
    _, scales = oracle.nvfp4_quantize_rows(rows)
    assert np.all(scales == np.arange(1, 127, dtype=np.uint8)[:, None])


def test_scale_ties_go_to_even_code():
    """amax / 6 exactly halfway between two E4M3 values picks the even code."""
    cs = np.arange(0, 126)
    amax = 3.0 * (E4M3[cs] + E4M3[cs + 1])
    assert np.all(amax.astype(np.float32).astype(np.float64) == amax)
    rows = np.stack([np.tile(_group(np.float32(a)), 8) for a in amax])
    _, scales = oracle.nvfp4_quantize_rows(rows)
    want = np.where(cs % 2 == 0, cs, cs + 1)
    assert np.array_equal(scales[:, 0], want.astype(np.uint8))


def test_saturation_and_zero_groups():
    x = np.zeros(128, np.float32)
    x[:16] = _group(1e6, rest=-3e5)          # amax / 6 > 448: scale 448, codes saturate at 6
    x[16:32] = 0.0                           # amax 0: scale 0, codes 0
    x[32:48] = _group(1e-4, rest=-1e-4)      # amax / 6 < 2^-10: scale rounds to 0, codes 0
    x[48:64] = _group(6.0 * 2.0 ** -10)      # amax / 6 = 2^-10 exactly: a tie, to the even code 0
    codes, scales = oracle.nvfp4_quantize_rows(x[None])
    assert scales[0, 0] == 0x7E
    assert codes[0, 2] >> 4 == 7 and codes[0, 0] == (15 | (15 << 4))   # +6 at element 5; -6 elsewhere
    assert scales[0, 1] == 0 and not codes[0, 8:16].any()
    assert scales[0, 2] == 0 and not codes[0, 16:24].any()
    assert scales[0, 3] == 0 and not codes[0, 24:32].any()


def test_round_trip_of_representable_rows():
    """x = e2m1(c) * v(s) with one element at +-6 v(s) quantises back to (c, s)."""
    rng = np.random.default_rng(7)
    for _ in range(20):
        s = rng.integers(1, 127, size=8)
        c = rng.integers(0, 16, size=(8, 16))
        c[np.arange(8), rng.integers(0, 16, size=8)] = rng.choice([7, 15], size=8)
        mag = E2M1[c & 7] * np.where(c & 8, -1.0, 1.0)
        x = (mag * E4M3[s][:, None]).astype(np.float32)
        assert np.all(x.astype(np.float64) == mag * E4M3[s][:, None])
        codes, scales = oracle.nvfp4_quantize_rows(x.reshape(1, 128))
        assert np.array_equal(scales[0], s.astype(np.uint8))
        want = (c.reshape(128)[0::2] | (c.reshape(128)[1::2] << 4)).astype(np.uint8)
        # a zero element comes back as +0 or -0 with the sign of x (-0.0 for code 8)
        assert np.array_equal(codes[0], want)


def _nearest(grid, y):
    """Index of the grid value nearest y (y >= 0), ties to the even index; brute force."""
    d = np.abs(grid[None, :] - y[:, None])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = cand & (np.arange(grid.size)[None, :] % 2 == 0)
    return np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))


def test_brute_force_nearest_on_random_rows():
    rng = np.random.default_rng(11)
    sig = np.exp(rng.uniform(-12, 8, size=(64, 8, 1)))
    x = (rng.standard_normal((64, 8, 16)) * sig).astype(np.float32)
    x[0, 0] = 0.0
    codes, scales = oracle.nvfp4_quantize_rows(x.reshape(64, 128))
    amax = np.abs(x.astype(np.float64)).max(axis=2).reshape(-1)
    want_s = _nearest(E4M3, np.minimum(amax / 6.0, 448.0))
    assert np.array_equal(scales.reshape(-1), want_s.astype(np.uint8))
    sv = E4M3[want_s].reshape(64, 8, 1)
    y = np.where(sv > 0, np.abs(x.astype(np.float64)) / np.where(sv > 0, sv, 1.0), 0.0)
    mag = _nearest(E2M1, np.minimum(y, 6.0).reshape(-1)).reshape(64, 8, 16)
    sign = np.where(np.signbit(x) & (sv > 0), 8, 0)
    c = (mag | sign).reshape(64, 128)
    assert np.array_equal(codes, (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8))


def _caches(P, fill=0xA5):
    return {"k_data": np.full((P, 4, 128, 64), fill, np.uint8), "k_scale": np.full((P, 4, 128, 8), fill, np.uint8),
            "v_data": np.full((P, 4, 128, 64), fill, np.uint8), "v_scale": np.full((P, 4, 128, 8), fill, np.uint8),
            "ki_data": np.full((P, 128, 64), fill, np.uint8), "ki_scale": np.full((P, 128, 8), fill, np.uint8)}


def test_kv_insert_places_rows_and_leaves_the_rest():
    rng = np.random.default_rng(3)
    P, T = 3, 6
    slots = np.array([2 * 128 + 5, -1, 0, 128 + 127, 2 * 128 + 6, 7], np.int64)
    k = rng.standard_normal((T, 4, 128)).astype(np.float32)
    v = rng.standard_normal((T, 4, 128)).astype(np.float32)
    ki = rng.standard_normal((T, 128)).astype(np.float32)
    c = _caches(P)
    assert oracle.kv_insert(slots, k, v, ki, c, P) == 0
    ref = _caches(P)
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        pg, s = divmod(int(sl), 128)
        ref["k_data"][pg, :, s], ref["k_scale"][pg, :, s] = oracle.nvfp4_quantize_rows(k[t])
        ref["v_data"][pg, :, s], ref["v_scale"][pg, :, s] = oracle.nvfp4_quantize_rows(v[t])
        ref["ki_data"][pg, s], ref["ki_scale"][pg, s] = oracle.nvfp4_quantize_rows(ki[t])
    for n in c:
        assert np.array_equal(c[n], ref[n]), n
    # a NULL source leaves its cache untouched
    c2 = _caches(P)
    assert oracle.kv_insert(slots, None, v, None, c2, P) == 0
    assert np.all(c2["k_data"] == 0xA5) and np.all(c2["ki_scale"] == 0xA5)
    assert np.array_equal(c2["v_data"], ref["v_data"])


def test_kv_insert_reports_a_page_out_of_range():
    P = 2
    slots = np.array([5, P * 128 + 1, 130], np.int64)
    x = np.ones((3, 4, 128), np.float32)
    c = _caches(P)
    assert oracle.kv_insert(slots, x, x, x[:, 0], c, P) == -1
    # the valid tokens are written: amax 1 gives 1/6 = 1.333 * 2^-3, E4M3 exponent field 4,
    # mantissa 2.67 -> 3
    assert np.all(c["k_scale"][0, :, 5] == (4 << 3) | 3) and np.all(c["ki_scale"][1, 2] == (4 << 3) | 3)
    # scale value 1.375 * 2^-3 = 0.171875, so 1 / scale = 5.82 > 5 (midpoint of 4 and 6): code 7
    assert np.all(c["k_data"][0, :, 5] == 0x77)


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
