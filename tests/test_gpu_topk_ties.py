"""GPU top-k under exact ties and survivor overflow, through the C ABI.

[vLLM-zh "How MiniMax sparse attention works"; MSA-fig §1 "TopK"] the selection is
the most recent block plus the 15 best others; the oracle breaks equal scores
toward the lower block id. Random data almost never ties, so these cases build
ties on purpose: many logical blocks of a request map, through the block table, to
a few physical pages. Blocks on the same page get bit-identical block scores on
both sides (same keys, same queries, exact maxima), so the lower-id rule decides
the selection, and long runs of equal keys push the kernels' threshold filters
past their register/shared-memory ranking into their exact fallbacks. Each case
names the branch it must reach; a host model of the filters (tests/_topk_sim.py)
computes the branch from the GPU's own block scores, so the claim is checked on
every run. Ids must equal the oracle's exactly (no near-tie waiver applies to an
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


def branches(form, bs, nb):
    model = {"direct": _topk_sim.direct, "staged": _topk_sim.staged, "warp": _topk_sim.warp}[form]
    return [model(bs[g], nb) for g in range(4)]


# (pages, blocks, run, max_pages or None, form, branch that at least one group must reach)
CASES = [
    (8, 300, 1, None, "direct", "rank"),          # <= 32 survivors, ranked by counting
    (4, 300, 8, None, "direct", "insertion"),     # > 32 survivors: exact insertion merge
    (3, 1100, 1, None, "staged", "sort"),         # staged rows, <= 32 survivors
    (4, 1100, 64, None, "staged", "rank"),        # 33..64 survivors
    (8, 3000, 8, None, "staged", "insertion"),    # > 64 survivors
    (8, 3000, 1, 10300, "warp", "sort"),          # rows too long to stage: one warp per group
    (3, 1100, 9, 10300, "warp", "rank"),          # 33..48 survivors
    (4, 3000, 8, 10300, "warp", "insertion"),     # > 48 survivors
]


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("pages,nb,run,max_pages,form,branch", CASES)
def test_fused_topk_ties_and_overflow(pages, nb, run, max_pages, form, branch):
    wl = aliased(pages, nb, run, max_pages=max_pages, tail=37)
    assert _topk_sim.kernel_form(nb, wl.max_pages_per_req) == form
    dec = _gpu.decoder(wl, with_block_scores=True)
    ids = dec.select_blocks().cpu().numpy()
    bs = dec.block_scores.cpu().numpy()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    got = branches(form, bs[0], nb)
    assert branch in [b for _, b in got], got
    ref = oracle.decode(wl)
    S = ref["S"][0][:, :nb]
    np.testing.assert_allclose(bs[0, :, :nb], S, rtol=1e-5, atol=1e-4)
    for g in range(4):
        _gpu.assert_topk_exact_on_own_scores(ids[0, g], bs[0, g], nb, (form, g))
        # the page with the best score has many aliases: an exact tie at the boundary
        others = np.sort(S[g, :nb - 1])[::-1]
        assert others[14] == others[15], "the case must put an exact tie at the 15/16 boundary"
        assert np.array_equal(ids[0, g], ref["ids"][0, g]), (g, ids[0, g], ref["ids"][0, g])
    # and the whole decode on the same blocks
    _gpu.check_decode(wl)


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("nb,max_pages,form", [(300, None, "direct"), (1100, None, "staged"),
                                               (1100, 10300, "warp")])
def test_zero_index_scales_tie_every_block(nb, max_pages, form):
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
    """The parametrised cases above reach every ranking branch of every kernel form
    (checked on the host model over the oracle's block scores, so this runs quickly
    and states the coverage claim next to the cases)."""
    seen = set()
    for pages, nb, run, max_pages, form, branch in CASES:
        wl = aliased(pages, nb, run, max_pages=max_pages, tail=37)
        S = oracle.decode(wl)["S"][0][:, :nb].astype(np.float32)
        seen |= {(form, b) for _, b in branches(form, S, nb)}
    for form, brs in (("direct", ("rank", "insertion")), ("staged", ("sort", "rank", "insertion")),
                      ("warp", ("sort", "rank", "insertion"))):
        for b in brs:
            assert (form, b) in seen, (form, b, sorted(seen))


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


# msa_decode ranks requests of over 1,025 blocks inside its attention kernel when each
# (request, group) is split over 4 or more CTAs: each CTA of the (request, group)'s cluster
# ranks a share of the candidates and the cluster merges the shares' 15 best exactly.
# (requests, pages, blocks, run, ranking branch one CTA must reach)
FUSED = [
    (1, 8, 3000, 8, "rank/direct"),            # 8 CTAs x ~375 candidates
    (1, 4, 3000, 64, "insertion/direct"),      # long runs of one page in a CTA's share
    (1, 8, 10000, 1, "rank/strided"),          # 8 CTAs x 1,250 candidates
    (1, 128, 10000, 1, "insertion/strided"),   # each thread's share holds one page: 15 pages survive
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
