"""GPU parity of the exact-score selection (msa_select_blocks_exact, through the C ABI)
against the oracle's exact mode.

[vLLM-zh, Rubin MSA kernels]: dequantising NVFP4 to FP16 keeps the E2M1 value times its
scale exact, so the index scores carry no E4M3 re-rounding. The kernel multiplies FP16
operands (exact products) and sums 128 of them in FP32: block scores within the FP32
summation bound 8e-6 sum_j |q_j k_j| of the token that attains them, block ids equal to the
oracle's except at a near-tie (the rule of the fused selection)."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_nvfp4_gb300 import synth
from tests import _gpu, _wl

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _block_bound(wl, b):
    """Per (group, block): 8e-6 x the largest sum_j |q_j k_j| over the block's tokens and rows."""
    N, R, r0 = _wl.geom(wl, b)
    q = np.abs(_wl.e4m3_values()[wl.q_idx[r0:r0 + R].astype(np.int64)])
    k = np.abs(_wl.keys_of(wl, b, "ki", exact=True))
    A = np.einsum("rgd,td->gt", q, k) if R == 1 else np.einsum("rgd,td->rgt", q, k).max(axis=0)
    nb = (N + 127) // 128
    pad = np.full((4, nb * 128), 0.0)
    pad[:, :N] = A
    return 8e-6 * pad.reshape(4, nb, 128).max(axis=2) + 1e-6


def test_exact_selection_matches_oracle():
    wl = _wl.small([9000, 40000, 130, 2047, 700, 1], [2, 8, 8, 1, 3, 1], needles=3, seed=6)
    dec = _gpu.decoder(wl, with_block_scores=True)
    ids = dec.select_blocks_exact().cpu().numpy()
    bs = dec.block_scores.cpu().numpy()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    ids_r = dec.select_blocks().cpu().numpy()
    bs_r = dec.block_scores.cpu().numpy()
    torch.cuda.synchronize()
    differ = 0
    for b in range(wl.num_reqs):
        N, R, r0 = _wl.geom(wl, b)
        nb = (N + 127) // 128
        Sr = oracle.block_scores(wl, b, exact=True)
        got = bs[b, :, :nb].astype(np.float64)
        fin = np.isfinite(Sr)
        assert np.array_equal(np.isfinite(got), fin) and np.all(np.isneginf(bs[b, :, nb:])), b
        assert np.all(np.abs(got[fin] - Sr[fin]) <= _block_bound(wl, b)[fin]), b
        for g in range(4):
            assert _gpu.selection_matches(ids[b, g], oracle.select(Sr[g]), Sr[g], nb), (b, g)
        differ += int(np.sum(bs[b, :, :nb] != bs_r[b, :, :nb]))
    assert differ > 0, "the exact and the E4M3 selections gave identical block scores"


def test_exact_selection_full_size():
    """The benchmark's shape (16 x 131,072 tokens x 8 rows); every request checked against
    the oracle's exact mode, and the top-k exact on the GPU's own block scores."""
    wl = synth.make_workload(synth.preset("spec8_128k"))
    dec = _gpu.decoder(wl, with_block_scores=True)
    ids = dec.select_blocks_exact().cpu().numpy()
    bs = dec.block_scores.cpu().numpy()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    for b in range(wl.num_reqs):
        nb = (int(wl.context_lens[b]) + 127) // 128
        Sr = oracle.block_scores(wl, b, exact=True)
        np.testing.assert_allclose(bs[b, :, :nb], Sr, rtol=1e-5, atol=1e-4)
        for g in range(4):
            assert _gpu.selection_matches(ids[b, g], oracle.select(Sr[g]), Sr[g], nb), (b, g)
            _gpu.assert_topk_exact_on_own_scores(ids[b, g], bs[b, g], nb, (b, g))
    for b in range(wl.num_reqs):
        nb = (int(wl.context_lens[b]) + 127) // 128
        for g in range(4):
            row = ids[b, g]
            assert np.all(np.diff(row) > 0) and row[-1] == nb - 1 and row[0] >= 0, (b, g)
