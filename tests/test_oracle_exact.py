"""Pins of the oracle's exact-score mode (the exact-score indexer).

[vLLM-zh] "Rubin MSA kernels": dequantising NVFP4 to FP16 keeps the product of the E2M1
value and its E4M3 scale exact, so the index scores are free of the E4M3 re-rounding an
FP8 MMA implies. In this mode the oracle scores the index keys with those exact values;
everything else (pooling, selection, attention on FP8 K/V) is unchanged. The pins use the
published E2M1 table and torch's E4M3 decoding, not the oracle's own code."""
import numpy as np
import pytest
import torch

import oracle
from tests import _wl


@pytest.fixture(scope="module")
def ragged():
    return _wl.small([700, 130, 2000, 1, 4500, 3000], [3, 8, 1, 1, 5, 2], needles=2, seed=21)


def test_exact_dequant_is_the_plain_product_for_every_scale_and_code():
    e2m1, e4m3 = _wl.e2m1_table(), _wl.e4m3_values()
    for s in range(256):
        for c in range(16):
            got, want = oracle.dequant_value_exact(c, s), e2m1[c] * e4m3[s]
            assert (np.isnan(got) and np.isnan(want)) or got == want, (s, c)


def test_exact_and_rounded_agree_exactly_when_the_product_is_representable():
    """A power-of-two scale (mantissa 0) times an E2M1 value is an E4M3 value while it
    stays in range, so both modes give the same number; other scales can differ."""
    for e in range(2, 14):
        s = e << 3
        for c in range(16):
            assert oracle.dequant_value_exact(c, s) == oracle.dequant_value(c, s), (s, c)
    # 1.5 x 1.875 = 2.8125 needs 5 significant bits: E4M3 rounds it to 2.75
    assert oracle.dequant_value_exact(3, 0x3F) == 2.8125 and oracle.dequant_value(3, 0x3F) == 2.75


def _brute_scores_exact(wl, b):
    N, R, r0 = _wl.geom(wl, b)
    kidx = torch.from_numpy(_wl.keys_of(wl, b, "ki", exact=True))
    q = torch.from_numpy(_wl.e4m3_values()[wl.q_idx[r0:r0 + R].astype(np.int64)])
    s = torch.einsum("rgd,td->rgt", q, kidx).numpy()
    pos = N - R + np.arange(R)
    s[np.broadcast_to(np.arange(N)[None, None, :] > pos[:, None, None], s.shape)] = -np.inf
    return s


def test_exact_token_scores_equal_bruteforce_exactly(ragged):
    # products of an E4M3 query value and an exact key value have at most 10 significant
    # bits and lie within 2^-19 .. 2^21: 128 of them sum exactly in FP64 in any order
    for b in range(ragged.num_reqs):
        got = oracle.token_scores(ragged, b, exact=True)
        assert np.array_equal(got, _brute_scores_exact(ragged, b)), b


def test_exact_block_scores_are_the_pooled_exact_scores_and_differ_from_rounded(ragged):
    differ = 0
    for b in range(ragged.num_reqs):
        S = oracle.block_scores(ragged, b, exact=True)
        s = oracle.token_scores(ragged, b, exact=True)
        N, R, r0 = _wl.geom(ragged, b)
        nb = (N + 127) // 128
        pooled = np.array([[s[:, g, c * 128:min(N, c * 128 + 128)].max() for c in range(nb)] for g in range(4)])
        assert np.array_equal(S, pooled), b
        # re-rounding moves each key value by at most 2^-4 of itself, so a score by at
        # most 2^-4 sum_j |q_j k_j|
        sr = oracle.token_scores(ragged, b)
        q = np.abs(_wl.e4m3_values()[ragged.q_idx[r0:r0 + R].astype(np.int64)])
        bound = np.einsum("rgd,td->rgt", q, np.abs(_wl.keys_of(ragged, b, "ki", exact=True))) * 2.0 ** -4
        fin = np.isfinite(s)
        assert np.array_equal(fin, np.isfinite(sr))
        assert np.all(np.abs(s[fin] - sr[fin]) <= bound[fin]), b
        differ += int(np.sum(S != oracle.block_scores(ragged, b)))
    assert differ > 0
