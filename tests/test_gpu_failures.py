"""Device-side failure handling of the decode path, through the C ABI.

Corrupt values only the device can see (block-table entries, context lengths,
row offsets, block ids handed to the attention) are fed from the host. The
kernels' own checks must catch each one: set the matching MSA_FLAG_* bit (read
back with msa_get_error), skip the affected work without a trap, and leave every
other request's results equal to the oracle's. The pages describe no failure
handling; this is the library's contract (include/msa.h)."""
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


def _base():
    return _wl.small([3000, 9000, 700, 20000], [2, 8, 1, 3], needles=2, seed=51)


def _check_others(wl, dec, bad_reqs):
    """Requests not in bad_reqs: ids and outputs as the oracle's."""
    ids = dec.block_ids.cpu().numpy()
    out = dec.out.float().cpu().numpy()
    good = [b for b in range(wl.num_reqs) if b not in bad_reqs]
    ref = oracle.decode(wl, good)
    for i, b in enumerate(good):
        r0, r1 = int(wl.q_indptr[b]), int(wl.q_indptr[b + 1])
        assert np.array_equal(ids[b], ref["ids"][i]), b
        _gpu.assert_out_close(out[r0:r1], ref["out"][r0:r1], f"request {b}")


@pytest.mark.parametrize("bad_page", ["past_end", "negative"])
def test_bad_page_id_in_block_table(bad_page):
    wl = _base()
    wl.block_table = wl.block_table.copy()
    wl.block_table[1, 5] = wl.num_pages + 3 if bad_page == "past_end" else -2
    dec = _gpu.decoder(wl)
    dec.decode()
    torch.cuda.synchronize()
    flags = dec.errors()
    assert flags & _lib.FLAG_BAD_PAGE, hex(flags)
    assert not flags & _lib.FLAG_TIMEOUT
    _check_others(wl, dec, {1})
    # the flags were read and cleared: a clean call reports nothing
    wl2 = _base()
    dec2 = _gpu.decoder(wl2)
    dec2.decode()
    torch.cuda.synchronize()
    assert dec2.errors() == 0


def test_context_length_beyond_the_block_table():
    wl = _base()
    wl.context_lens = wl.context_lens.copy()
    wl.context_lens[2] = wl.max_pages_per_req * 128 + 1        # longer than its table row
    dec = _gpu.decoder(wl)
    dec.decode()
    torch.cuda.synchronize()
    flags = dec.errors()
    assert flags & _lib.FLAG_BAD_LENGTH, hex(flags)
    assert np.all(dec.block_ids[2].cpu().numpy() == -1)    # nothing selected for it
    _check_others(wl, dec, {2})


def test_rows_beyond_the_declared_maximum():
    wl = _base()
    dec = _gpu.decoder(wl)
    # request 1 holds 8 rows; declare at most 4 per request to the kernels
    dec.args.max_rows_per_req = 4
    dec.args.total_rows = int(wl.total_rows)
    dec.ws = torch.zeros(_lib.msa_workspace_size(dec.args), dtype=torch.uint8, device="cuda")
    dec._decode_ptrs = None
    dec.decode()
    torch.cuda.synchronize()
    flags = dec.errors()
    assert flags & _lib.FLAG_BAD_LENGTH, hex(flags)
    _check_others(wl, dec, {1})


def test_attention_block_ids_outside_the_context():
    wl = _base()
    ref = oracle.decode(wl)
    ids = np.ascontiguousarray(ref["ids"]).copy()
    nb3 = (int(wl.context_lens[3]) + 127) // 128
    ids[3, 2, 4] = nb3 + 7                      # past the context: skipped, flagged
    dec = _gpu.decoder(wl)
    out = dec.sparse_attn(torch.from_numpy(ids).cuda()).float().cpu().numpy()
    torch.cuda.synchronize()
    flags = dec.errors()
    assert flags & _lib.FLAG_BAD_IDS, hex(flags)
    for b in range(wl.num_reqs):
        r0, r1 = int(wl.q_indptr[b]), int(wl.q_indptr[b + 1])
        if b == 3:
            # the bad id is skipped: the group attends over its other 15 blocks
            keep = ids[3].copy()
            keep[2, 4] = -1
            ro, _ = oracle.attend(wl, 3, keep)
        else:
            ro = ref["out"][r0:r1]
        _gpu.assert_out_close(out[r0:r1], ro, f"request {b}")


def test_bounded_wait_times_out_and_the_context_stays_usable():
    """The library's bounded wait, run on a barrier phase that never completes
    (msa_selftest_wait_timeout), gives up after its limit and reports MSA_FLAG_TIMEOUT
    through the workspace; the next decode on the same context is correct."""
    import time
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    _lib.msa_selftest_wait_timeout(ws)
    flags = _lib.msa_get_error(ws)
    dt = time.perf_counter() - t0
    assert flags == _lib.FLAG_TIMEOUT
    assert 0.9 < dt < 30.0, dt  # the limit is 1 s of the device timer
    assert _lib.msa_get_error(ws) == 0  # read and cleared
    wl = _base()
    dec = _gpu.decoder(wl)
    dec.decode()
    torch.cuda.synchronize()
    assert dec.errors() == 0
    _check_others(wl, dec, [])
