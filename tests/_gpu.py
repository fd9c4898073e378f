"""Helpers for the GPU parity tests: run libmsa through the C ABI and compare
with the oracle using the path's acceptance rules."""
import numpy as np
import torch

import oracle
from block_sparse_attention_nvfp4_gb300 import DecodeBatch, KVCache, MSADecoder

OUT_ATOL, OUT_RTOL = 2e-2, 2e-2      # |gpu - oracle| <= 2e-2 + 2e-2 |oracle|
TIE_REL = 1e-4                        # selection may differ only at a near-tie boundary


def decoder(wl, **kw):
    return MSADecoder(KVCache.from_host(wl), DecodeBatch.from_host(wl), sm_scale=wl.sm_scale, **kw)


def assert_out_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    excess = np.abs(got - ref) - (OUT_ATOL + OUT_RTOL * np.abs(ref))
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, f"{what}: worst at {i}: got {got[i]} ref {ref[i]}"


def selection_matches(gpu_ids, ref_ids, S_ref, nb):
    """True when the GPU's ids equal the oracle's, or differ only at a near-tie:
    the oracle's 16th and 17th block scores (the 15th/16th best non-recent blocks)
    differ but lie within TIE_REL relative of each other, and every swapped block
    lies inside that band. An exact tie (equal scores) is never waived: the lower
    block id must win, as the oracle's rule says."""
    g = sorted(int(x) for x in gpu_ids if x >= 0)
    r = sorted(int(x) for x in ref_ids if x >= 0)
    if g == r:
        return True
    if nb <= 16:
        return False
    others = np.sort(S_ref[: nb - 1])[::-1]
    s15, s16 = others[14], others[15]
    if s15 == s16:
        return False
    band = TIE_REL * max(abs(s15), abs(s16))
    if abs(s15 - s16) > band:
        return False
    swapped = set(g) ^ set(r)
    return all(abs(S_ref[c] - s15) <= 2 * band or abs(S_ref[c] - s16) <= 2 * band for c in swapped)


def assert_topk_exact_on_own_scores(ids, block_scores, nb, what=""):
    """The top-k given the GPU's own FP32 block scores is exact: the ids equal the
    oracle's selection (full sort, ties to the lower id) run on those same scores."""
    want = oracle.select(np.asarray(block_scores[:nb], dtype=np.float32).astype(np.float64))
    assert np.array_equal(np.asarray(ids), want), (what, ids, want)


def check_decode(wl, reqs=None, dec=None):
    """Run msa_decode and compare ids (exact up to near-ties) and outputs with the
    oracle for the listed requests. Returns the decoder."""
    dec = dec or decoder(wl)
    out, ids = dec.decode()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    ref = oracle.decode(wl, reqs)
    gids = ids.cpu().numpy()
    o = out.float().cpu().numpy()
    lse = dec.lse.cpu().numpy()
    n_waived = 0
    for i, b in enumerate(ref["reqs"]):
        b = int(b)
        N = int(wl.context_lens[b])
        nb = (N + 127) // 128
        r0, r1 = int(wl.q_indptr[b]), int(wl.q_indptr[b + 1])
        if r1 == r0:  # no query rows: nothing is selected or attended
            assert np.all(gids[b] == -1), b
            continue
        exact = True
        for g in range(4):
            same = np.array_equal(gids[b, g], ref["ids"][i, g])
            if not same:
                assert selection_matches(gids[b, g], ref["ids"][i, g], ref["S"][i, g], nb), (b, g, gids[b, g],
                                                                                              ref["ids"][i, g])
                exact = False
                n_waived += 1
        if exact:
            ro, rl = ref["out"][r0:r1], ref["lse"][r0:r1]
        else:  # a legitimately different selection: compare with the oracle on the GPU's blocks
            ro, rl = oracle.attend(wl, b, gids[b])
        assert_out_close(o[r0:r1], ro, f"request {b} out")
        np.testing.assert_allclose(lse[r0:r1], rl, atol=1e-3, rtol=1e-4, err_msg=f"request {b} lse")
    return dec, n_waived
