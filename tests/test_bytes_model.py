"""The byte model behind the roofline, pinned to the numbers the MSA pages print."""
import os

import pytest

from block_sparse_attention_nvfp4_gb300 import bytes_model as bm
from block_sparse_attention_nvfp4_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_byte_counts.txt")


@pytest.fixture(scope="module")
def page():
    out = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            out[k] = float(v)
    return out


def test_fp8_figures_of_the_pages(page):
    assert bm.index_bytes_per_token("fp8") == page["index_key_bytes_per_token_per_layer"]
    assert bm.dense_kv_bytes_per_token("fp8") == page["dense_kv_bytes_per_token_per_layer"]
    assert page["kv_heads"] == bm.HEADS and page["head_dim"] == bm.DIM and page["block_tokens"] == bm.BLOCK
    assert page["selected_blocks"] * page["block_tokens"] == page["max_keys_per_query"]
    # "about 12.5%" at long context: the index scan alone, 128 of 1,024 bytes
    assert bm.traffic_fraction(10**9, "fp8") == pytest.approx(page["long_context_traffic_fraction"], abs=1e-5)


def test_nvfp4_scaling_matches_the_pages_kv_sizes(page):
    ratio = page["nvfp4_kv_bytes_per_token"] / page["fp8_kv_bytes_per_token"]
    assert ratio == pytest.approx(1 - page["nvfp4_kv_saving"])
    assert bm.index_bytes_per_token("nvfp4") / bm.index_bytes_per_token("fp8") == ratio
    # both whole-model figures are whole multiples of the per-layer sizes (60 layers: our inference)
    assert page["fp8_kv_bytes_per_token"] / bm.dense_kv_bytes_per_token("fp8") == 60
    assert page["nvfp4_kv_bytes_per_token"] / bm.dense_kv_bytes_per_token("nvfp4") == 60


def test_long_context_fraction_closed_form():
    for n in (4096, 131072, 524288):
        sel = min(n, 2048)
        assert bm.traffic_fraction(n) == pytest.approx((72 * n + sel * 576) / (576 * n))
    assert bm.traffic_fraction(131072) == pytest.approx(0.125 + 2048 / 131072)


def test_step_bytes_of_the_128k_speculative_workload():
    s = synth.preset("spec8_128k")
    r = bm.step_bytes(s.context_lens, s.rows)
    assert r["index"] == 16 * 131072 * 72
    assert r["kv"] == 16 * 4 * 2048 * 144
    assert r["queries"] == 128 * (4096 + 512)
    assert abs(r["total"] - 171.6e6) < 0.1e6


def test_distinct_index_bytes_count_each_shared_page_once():
    """A shared prefix of 4 pages over 3 requests: the logical count has every request's
    pages, the distinct count the 4 prefix pages once; without sharing the two agree. A
    request with no rows reads nothing."""
    import numpy as np
    from tests import _wl

    ctx, rows = [1000, 2048, 600], [1, 2, 1]
    wl = _wl.small(ctx, rows, shared=4, seed=3)
    r = np.diff(wl.q_indptr)
    got = bm.distinct_index_bytes(wl.context_lens, r, wl.block_table)
    pages = [(n + 127) // 128 for n in ctx]                  # 8, 16, 5
    assert got["logical_pages"] == sum(pages)
    assert got["distinct_pages"] == sum(pages) - 2 * 4       # the prefix, once instead of 3 times
    assert got["logical"] == sum(ctx) * 72
    assert got["distinct"] == (sum(ctx) - 2 * 4 * 128) * 72  # the prefix pages are full in every request
    own = _wl.small(ctx, rows, shared=0, seed=3)
    got = bm.distinct_index_bytes(own.context_lens, np.diff(own.q_indptr), own.block_table)
    assert got["distinct"] == got["logical"] == sum(ctx) * 72
    got = bm.distinct_index_bytes(wl.context_lens, np.array([0, 2, 1]), wl.block_table)
    assert got["logical"] == (2048 + 600) * 72 and got["distinct"] == (2048 + 600 - 4 * 128) * 72
