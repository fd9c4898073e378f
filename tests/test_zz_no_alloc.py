"""The allocation-free selection entry point (msa_select_blocks_noalloc).

It serves callers that cannot allocate device memory (plugin interfaces that
own the allocator, decode loops that must not call cudaMalloc), keeping its
scratch in a fixed buffer inside libmsa. This file runs last so that a failure
here leaves every other test already run; it also passes on its own in a fresh
process (it builds and loads everything it needs)."""
import copy

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_nvfp4_gb300 import _lib
from tests import _gpu, _wl

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("ctx,rows,seed", [
    ([700, 130, 2000, 1, 4500, 3000], [3, 8, 1, 1, 5, 2], 21),
    ([131072] * 2, [8, 8], 2),
])
def test_noalloc_select_matches_workspace_select_twice(ctx, rows, seed):
    wl = _wl.small(ctx, rows, needles=3, seed=seed)
    dec = _gpu.decoder(wl, with_block_scores=True)
    ref_ids = dec.select_blocks().clone()
    ref_scores = dec.block_scores.clone()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    for _ in range(2):  # two calls in a row: the shared buffer must come back clean
        ids = torch.full_like(ref_ids, -7)
        scores = torch.full_like(ref_scores, float("nan"))
        _lib.msa_select_blocks_noalloc(dec.args, ids, scores)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids)
        np.testing.assert_array_equal(scores.cpu().numpy(), ref_scores.cpu().numpy())
        assert _lib.msa_select_blocks_noalloc_get_error() == 0


def test_noalloc_rejects_batches_beyond_its_buffer():
    wl = _wl.small([3000], [1], seed=3)
    dec = _gpu.decoder(wl)
    a = _lib.make_args(dec.cache, dec.batch, wl.sm_scale)
    a.max_pages_per_req = 1 << 20          # 256 + 16 x 1 x 2^20 B = 16 MiB of block scores > 8 MiB
    ids = torch.empty((1, 4, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.MSAError) as e:
        _lib.msa_select_blocks_noalloc(a, ids, None)
    assert e.value.code == -4
    assert _lib.load().msa_select_blocks_noalloc(None, None, None, None) == -1


def test_noalloc_reports_a_bad_page_then_clears():
    """A block-table entry past the cache: the kernels skip that page and flag it; the
    flags of the call are read from the library's buffer, and the next good call
    reports none."""
    wl = _wl.small([3000, 9000], [2, 4], needles=2, seed=52)
    bad = copy.copy(wl)
    bad.block_table = wl.block_table.copy()
    bad.block_table[1, 3] = wl.num_pages + 5
    dec = _gpu.decoder(bad)
    ids = torch.full((2, 4, 16), -7, dtype=torch.int32, device="cuda")
    _lib.msa_select_blocks_noalloc(dec.args, ids, None)
    flags = _lib.msa_select_blocks_noalloc_get_error()
    assert flags & _lib.FLAG_BAD_PAGE, hex(flags)
    good = _gpu.decoder(wl)
    _lib.msa_select_blocks_noalloc(good.args, ids, None)
    assert _lib.msa_select_blocks_noalloc_get_error() == 0
    ref = oracle.decode(wl)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
