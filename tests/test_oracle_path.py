"""Pins of the oracle's path (scores, block max pool, top-k, attention) against
brute force written independently with numpy/torch, textbook special cases and
invariants the MSA pages state."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import _wl


# ragged contexts (not multiples of 128), rows straddling a block boundary
# (130 tokens with 8 rows: positions 122..129 span blocks 0 and 1)
@pytest.fixture(scope="module")
def ragged():
    return _wl.small([700, 130, 2000, 1], [3, 8, 1, 1], needles=2, seed=21)


def brute_scores(wl, b):
    N, R, r0 = _wl.geom(wl, b)
    kidx = torch.from_numpy(_wl.keys_of(wl, b, "ki"))
    q = torch.from_numpy(_wl.e4m3_values()[wl.q_idx[r0:r0 + R].astype(np.int64)])
    s = torch.einsum("rgd,td->rgt", q, kidx).numpy()
    pos = N - R + np.arange(R)
    s[np.broadcast_to(np.arange(N)[None, None, :] > pos[:, None, None], s.shape)] = -np.inf
    return s


def test_token_scores_equal_bruteforce_exactly(ragged):
    # every product of two E4M3 values is exact and 128 of them sum exactly in FP64,
    # so any summation order gives the same bits
    for b in range(ragged.num_reqs):
        got = oracle.token_scores(ragged, b)
        ref = brute_scores(ragged, b)
        assert got.shape == ref.shape
        assert np.array_equal(got, ref), b


def test_block_maxpool_equals_bruteforce(ragged):
    for b in range(ragged.num_reqs):
        s = brute_scores(ragged, b)
        N = s.shape[2]
        nb = (N + 127) // 128
        pad = np.full((s.shape[0], 4, nb * 128), -np.inf)
        pad[:, :, :N] = s
        ref = pad.reshape(s.shape[0], 4, nb, 128).max(axis=(0, 3))
        assert np.array_equal(oracle.block_scores(ragged, b), ref)
        assert np.array_equal(oracle.block_maxpool(s), ref)


def check_selection(S, ids, top_k=16):
    nb = len(S)
    sel = [int(i) for i in ids if i >= 0]
    assert list(ids[len(sel):]) == [-1] * (top_k - len(sel))
    assert sel == sorted(sel) and len(set(sel)) == len(sel)
    if nb <= top_k:
        assert sel == list(range(nb))
        return
    assert len(sel) == top_k and nb - 1 in sel
    others = [c for c in sel if c != nb - 1]
    rest = [c for c in range(nb - 1) if c not in others]
    for c in others:
        for d in rest:
            assert S[c] > S[d] or (S[c] == S[d] and c < d), (c, d)


def test_select_invariants_random_with_ties():
    rng = np.random.default_rng(3)
    for trial in range(300):
        nb = int(rng.integers(1, 80))
        S = rng.integers(-5, 5, size=nb).astype(np.float64)  # many ties
        if trial % 3 == 0:
            S = rng.normal(size=nb)
        ids = oracle.select(S)
        check_selection(S, ids)


def test_select_keeps_recent_block_and_prefers_lower_id_on_ties():
    S = np.zeros(40)
    S[-1] = -1e6
    ids = oracle.select(S)
    assert list(ids) == list(range(15)) + [39]
    S = np.arange(40, dtype=np.float64)[::-1].copy()  # block 0 best
    assert list(oracle.select(S)) == list(range(15)) + [39]
    assert list(oracle.select(np.ones(5))) == [0, 1, 2, 3, 4] + [-1] * 11


def test_needle_blocks_are_selected():
    for wl in (_wl.small([4096], [1], needles=4, seed=0),
               _wl.small([9000, 20000, 5000], [1, 8, 2], needles=5, seed=4)):
        r = oracle.decode(wl)
        for i, b in enumerate(r["reqs"]):
            for g in range(4):
                for c in wl.needles[b][g]:
                    assert c in r["ids"][i, g], (b, g, c)


def dense_reference(wl, b):
    """Plain softmax attention over every visible key (torch SDPA, FP64)."""
    N, R, r0 = _wl.geom(wl, b)
    K = torch.from_numpy(_wl.keys_of(wl, b, "k"))   # [N, 4, 128]
    V = torch.from_numpy(_wl.keys_of(wl, b, "v"))
    q = torch.from_numpy(_wl.e4m3_values()[wl.q[r0:r0 + R].astype(np.int64)])  # [R, 32, 128]
    Kh = K.repeat_interleave(8, dim=1).permute(1, 0, 2)[None]   # [1, 32, N, 128]
    Vh = V.repeat_interleave(8, dim=1).permute(1, 0, 2)[None]
    Q = q.permute(1, 0, 2)[None]                                 # [1, 32, R, 128]
    pos = N - R + torch.arange(R)
    mask = torch.arange(N)[None, :] <= pos[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(Q, Kh, Vh, attn_mask=mask, scale=wl.sm_scale)
    logits = (Q @ Kh.transpose(-1, -2)) * wl.sm_scale
    logits = logits.masked_fill(~mask, -math.inf)
    lse = torch.logsumexp(logits, dim=-1)
    return out[0].permute(1, 0, 2).numpy(), lse[0].permute(1, 0).numpy()


def test_all_blocks_selected_equals_dense_attention():
    # top-k covering every block reduces MSA to plain attention
    wl = _wl.small([4096, 700, 130], [1, 3, 8], needles=2, seed=9, top_k=32)
    r = oracle.decode(wl)
    for i, b in enumerate(r["reqs"]):
        N, R, r0 = _wl.geom(wl, b)
        nb = (N + 127) // 128
        assert list(r["ids"][i, 0, :nb]) == list(range(nb))
        out, lse = dense_reference(wl, b)
        np.testing.assert_allclose(r["out"][r0:r0 + R], out, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(r["lse"][r0:r0 + R], lse, rtol=1e-12, atol=1e-13)


def test_single_key_gives_its_value():
    wl = _wl.small([1], [1], seed=13)
    r = oracle.decode(wl)
    v = _wl.keys_of(wl, 0, "v")[0]       # [4, 128]
    k = _wl.keys_of(wl, 0, "k")[0]
    q = _wl.e4m3_values()[wl.q[0].astype(np.int64)]
    for h in range(32):
        assert np.array_equal(r["out"][0, h], v[h // 8])
        assert r["lse"][0, h] == pytest.approx(float(q[h] @ k[h // 8]) * wl.sm_scale, rel=1e-15)


def test_lse_merge_of_disjoint_block_sets_equals_whole(ragged):
    wl = _wl.small([6000, 3000], [4, 1], needles=3, seed=17)
    r = oracle.decode(wl)
    for i, b in enumerate(r["reqs"]):
        N, R, r0 = _wl.geom(wl, b)
        ids = r["ids"][i]
        a = np.where(np.arange(16)[None, :] % 2 == 0, ids, -1)
        c = np.where(np.arange(16)[None, :] % 2 == 1, ids, -1)
        oa, la = oracle.attend(wl, b, a)
        oc, lc = oracle.attend(wl, b, c)
        m = np.maximum(la, lc)
        wa, wc = np.exp(la - m), np.exp(lc - m)
        merged = (wa[..., None] * oa + wc[..., None] * oc) / (wa + wc)[..., None]
        np.testing.assert_allclose(merged, r["out"][r0:r0 + R], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(m + np.log(wa + wc), r["lse"][r0:r0 + R], rtol=1e-12)


def test_block_table_permutation_leaves_results_unchanged(ragged):
    w2 = _wl.permuted_pages(ragged)
    a, b = oracle.decode(ragged), oracle.decode(w2)
    for k in ("ids", "S", "out", "lse"):
        assert np.array_equal(a[k], b[k]), k


def test_shared_prefix_equals_copied_prefix():
    wl = _wl.small([2300, 4000, 2100], [2, 1, 4], shared=3, seed=31)
    assert wl.num_pages == 3 + (18 - 3) + (32 - 3) + (17 - 3)
    w2 = _wl.unshared_copy(wl)
    a, b = oracle.decode(wl), oracle.decode(w2)
    for k in ("ids", "S", "out", "lse"):
        assert np.array_equal(a[k], b[k]), k


def test_decode_composes_the_steps(ragged):
    r = oracle.decode(ragged)
    for i, b in enumerate(r["reqs"]):
        S = oracle.block_scores(ragged, b)
        nb = S.shape[1]
        assert np.array_equal(r["S"][i][:, :nb], S)
        for g in range(4):
            assert np.array_equal(r["ids"][i, g], oracle.select(S[g]))
        out, lse = oracle.attend(ragged, b, r["ids"][i])
        N, R, r0 = _wl.geom(ragged, b)
        assert np.array_equal(out, r["out"][r0:r0 + R])


def test_key_cap_is_2048_per_query():
    wl = _wl.small([40000], [2], needles=4, seed=5)
    r = oracle.decode(wl)
    per_group = (r["ids"][0] >= 0).sum(axis=1) * 128
    assert np.all(per_group == 2048)
