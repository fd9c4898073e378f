"""GPU top-k under exact ties and survivor overflow, through the C ABI.

[vLLM-zh "How MiniMax sparse attention works"; MSA-fig §1 "TopK"] the selection is
the most recent block plus the 15 best others; the oracle breaks equal scores
toward the lower block id. Random data almost never ties, so these cases build
ties on purpose: many logical blocks of a request map, through the block table, to
a few physical pages. Blocks on the same page get bit-identical block scores on
both sides (same keys, same queries, exact maxima), so the lower-id rule decides
the selection, and long runs of equal keys push the kernels' threshold filters
past the sort of their survivors into the merge of two sorted halves and the
chunked merge of every candidate above the threshold. Each case names the branch it
must reach; a host model of the filters (tests/_topk_sim.py) computes the branch
from the GPU's own block scores, so the claim is checked on every run. Ids must equal the oracle's exactly (no near-tie waiver applies to an
exact tie)."""
import copy

import numpy as np
import pytest
import torch

import oracle
from tests import _gpu, _topk_sim, _wl

gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def aliased(n_pages, nb, run, rows=2, tail=0, max_pages=None, seed=40, zero_index_scales=False):
    """One request of nb blocks whose logical block c lives on physical page
    (c // run) % n_pages of a small seeded cache (every slot of every page
    written). tail > 0 leaves the last page partial."""
    base = _wl.small([n_pages * 128], [rows], seed=seed)
    wl = copy.copy(base)
    mp = max_pages or nb
    bt = np.zeros((1, mp), np.int32)
    bt[0, :nb] = base.block_table[0, (np.arange(nb) // run) % n_pages]
    wl.block_table = bt
    wl.max_pages_per_req = mp
    wl.context_lens = np.array([nb * 128 - tail], np.int32)
    if zero_index_scales:
        wl.ki_scale = np.zeros_like(base.ki_scale)
    return wl


def branches(bs, nb):
    """Every (warp, group) branch of the top-k kernel's filter on these block scores."""
    return {br for g in range(4) for _, br in _topk_sim.topk_kernel(bs[g], nb)}


# (pages, blocks, run, max_pages or None, branch that at least one group must reach). Up to
# 1,025 blocks: the direct form's rank counting (<= 32 survivors) or its exact insertion merge;
# longer rows: quad_best15's survivor sort (<= 32), two sorted halves (33..64) or chunked merge
# (> 64), each warp's quarter streamed twice. The last case's block-table rows hold 10,300
# entries, far more than the request uses.
CASES = [
    (8, 300, 1, None, "direct/rank"),
    (4, 300, 8, None, "direct/insertion"),
    (3, 1100, 1, None, "sort/stream"),
    (8, 1100, 8, None, "two_sorts/stream"),
    (8, 3000, 1, 10300, "chunked/stream"),
]


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("pages,nb,run,max_pages,branch", CASES)
def test_topk_ties_and_overflow(pages, nb, run, max_pages, branch):
    wl = aliased(pages, nb, run, max_pages=max_pages, tail=37)
    dec = _gpu.decoder(wl, with_block_scores=True)
    ids = dec.select_blocks().cpu().numpy()
    bs = dec.block_scores.cpu().numpy()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    got = branches(bs[0], nb)
    assert branch in got, got
    ref = oracle.decode(wl)
    S = ref["S"][0][:, :nb]
    np.testing.assert_allclose(bs[0, :, :nb], S, rtol=1e-5, atol=1e-4)
    for g in range(4):
        _gpu.assert_topk_exact_on_own_scores(ids[0, g], bs[0, g], nb, (branch, g))
        # the page with the best score has many aliases: an exact tie at the boundary
        others = np.sort(S[g, :nb - 1])[::-1]
        assert others[14] == others[15], "the case must put an exact tie at the 15/16 boundary"
        assert np.array_equal(ids[0, g], ref["ids"][0, g]), (g, ids[0, g], ref["ids"][0, g])
    # and the whole decode on the same blocks
    _gpu.check_decode(wl)


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("nb,max_pages", [(300, None), (1100, None), (1100, 10300)])
def test_zero_index_scales_tie_every_block(nb, max_pages):
    """An index cache whose scales are all zero scores every token 0: every block
    ties, so the selection is the 15 lowest ids plus the recent block."""
    wl = aliased(4, nb, 1, max_pages=max_pages, zero_index_scales=True)
    dec = _gpu.decoder(wl, with_block_scores=True)
    ids = dec.select_blocks().cpu().numpy()
    bs = dec.block_scores.cpu().numpy()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    assert np.all(bs[0, :, :nb] == 0)
    want = np.array(list(range(15)) + [nb - 1], np.int32)
    for g in range(4):
        assert np.array_equal(ids[0, g], want), (g, ids[0, g])
    _gpu.check_decode(wl)


def test_branch_coverage_of_the_cases():
    """The parametrised cases reach every branch of the top-k kernel's two forms (CASES) and
    of the attention kernel's fused top-k, register and streamed (FUSED), CASES each with an
    exact tie at the 15/16 boundary (checked on the host model over the oracle's block
    scores, so this runs quickly and states the coverage claim next to the cases)."""
    all_branches = {f"{b}/{p}" for b in ("sort", "two_sorts", "chunked") for p in ("regs", "stream")}
    seen = set()
    for pages, nb, run, max_pages, branch in CASES:
        wl = aliased(pages, nb, run, max_pages=max_pages, tail=37)
        S = oracle.decode(wl)["S"][0][:, :nb].astype(np.float32)
        got = branches(S, nb)
        assert branch in got, (pages, nb, run, got)
        seen |= got
        for g in range(4):
            others = np.sort(S[g, :nb - 1])[::-1]
            assert others[14] == others[15], (pages, nb, run, g)
    assert seen >= {"direct/rank", "direct/insertion", "sort/stream", "two_sorts/stream", "chunked/stream"}, sorted(seen)
    seen = set()
    for nreq, pages, nb, run, branch in FUSED:
        # the page scores of the aliased request (every block but the last fully visible)
        ps = oracle.decode(aliased(pages, pages + 1, 1, rows=1, seed=41))["S"][0][:, :pages].astype(np.float32)
        bs = ps[:, (np.arange(nb) // run) % pages]
        splits = _topk_sim.attention_splits(nreq, 152)  # GB300's SM count
        got = {br for g in range(4) for br in _topk_sim.fused_branches(bs[g], nb, splits)}
        assert branch in got, (pages, nb, run, got)
        seen |= got
    assert seen >= all_branches, sorted(seen)


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("pattern", ["sort", "rank", "insertion"])
def test_maxpool_topk_ties_from_given_scores(pattern):
    """msa_block_maxpool_topk (one warp per group) on token scores built with ties:
    every token of a block carries the block's value, values repeat in runs."""
    nb = 1100
    run = {"sort": 1, "rank": 9, "insertion": 8}[pattern]
    n_vals = {"sort": 3, "rank": 3, "insertion": 4}[pattern]
    wl = aliased(4, nb, 1, rows=1)
    dec = _gpu.decoder(wl, with_block_scores=True)
    rng = np.random.default_rng(7)
    vals = rng.standard_normal((4, n_vals)).astype(np.float32)
    blockv = vals[:, (np.arange(nb) // run) % n_vals]                 # [4, nb]
    stride = wl.max_pages_per_req * 128
    S32 = np.full((1, 4, stride), np.nan, np.float32)
    S32[0, :, :nb * 128] = np.repeat(blockv, 128, axis=1)
    ids = dec.maxpool_topk(torch.from_numpy(S32).cuda()).cpu().numpy()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    got = [_topk_sim.warp(blockv[g], nb)[1] for g in range(4)]
    assert pattern in got, got
    for g in range(4):
        assert np.array_equal(ids[0, g], oracle.select(blockv[g].astype(np.float64))), g


@pytest.mark.gpu
@gpu
def test_signed_zero_scores_tie():
    """-0.0 and +0.0 are equal scores: the lower block id wins between them, as in
    the oracle's comparison (both the one-warp and the fused forms)."""
    nb = 300
    wl = aliased(4, nb, 1, rows=1)
    dec = _gpu.decoder(wl, with_block_scores=True)
    blockv = np.zeros((4, nb), np.float32)
    blockv[:, 1::2] = -0.0                     # odd blocks -0.0, even blocks +0.0
    blockv[1, 5:40:3] = 1.0
    blockv[2, :] = -blockv[2, :]               # signs swapped
    stride = wl.max_pages_per_req * 128
    S32 = np.full((1, 4, stride), np.nan, np.float32)
    S32[0, :, :nb * 128] = np.repeat(blockv, 128, axis=1)
    ids = dec.maxpool_topk(torch.from_numpy(S32).cuda()).cpu().numpy()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    for g in range(4):
        want = oracle.select(blockv[g].astype(np.float64))
        assert np.array_equal(ids[0, g], want), (g, ids[0, g], want)
    assert np.array_equal(ids[0, 0], np.array(list(range(15)) + [nb - 1], np.int32))


# msa_decode ranks inside its attention kernel (1) requests of over 1,025 blocks when each
# (request, group) is split over 4 or more CTAs: each CTA of the (request, group)'s cluster
# ranks a share of the candidates (quad_best15) and the cluster merges the shares' 15 best
# exactly (one request: 8 CTAs per (request, group)); (2) requests of at most 1,025 blocks
# when each (request, group) is one CTA (20 or more requests on 152 SMs): that CTA ranks all
# of its group's candidates.
# (requests, pages, blocks, run, branch one warp of one CTA must reach)
FUSED = [
    (1, 3, 3000, 1, "sort/regs"),             # 8 CTAs x ~375 candidates, ~94 per warp
    (1, 8, 3000, 1, "two_sorts/regs"),
    (1, 4, 8193, 8, "chunked/regs"),          # 256 candidates per warp
    (1, 3, 10000, 1, "sort/stream"),          # ~312 per warp: read twice
    (1, 8, 10000, 8, "two_sorts/stream"),
    (1, 4, 10000, 1, "chunked/stream"),
    (20, 3, 1000, 1, "sort/regs"),            # one CTA per (request, group), ~250 per warp
    (20, 8, 600, 2, "two_sorts/regs"),
    (20, 8, 1000, 1, "chunked/regs"),
]


def _aliased_batch(nreq, pages, nb, run, rows=1, seed=41):
    one = aliased(pages, nb, run, rows=rows, seed=seed, tail=37)
    wl = copy.copy(one)
    wl.num_reqs = nreq
    wl.context_lens = np.repeat(one.context_lens, nreq)
    wl.block_table = np.repeat(one.block_table, nreq, axis=0)
    wl.q_indptr = np.arange(nreq + 1, dtype=np.int32) * rows
    wl.total_rows = nreq * rows
    wl.q = np.tile(one.q, (nreq, 1, 1))
    wl.q_idx = np.tile(one.q_idx, (nreq, 1, 1))
    return wl


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("nreq,pages,nb,run,branch", FUSED)
def test_decode_with_the_topk_inside_the_attention(nreq, pages, nb, run, branch):
    wl = _aliased_batch(nreq, pages, nb, run)
    splits = _topk_sim.attention_splits(nreq, torch.cuda.get_device_properties(0).multi_processor_count)
    dec = _gpu.decoder(wl, with_block_scores=True)
    dec.select_blocks()                     # the same scan: the block scores the attention ranks
    bs = dec.block_scores.cpu().numpy()
    torch.cuda.synchronize()
    got = {br for b in range(min(nreq, 2)) for g in range(4) for br in _topk_sim.fused_branches(bs[b, g], nb, splits)}
    assert branch in got, (splits, got)
    _gpu.check_decode(wl, dec=_gpu.decoder(wl))
