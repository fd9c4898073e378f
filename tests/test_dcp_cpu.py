"""Indexer decode context parallelism (DCP) without a GPU
[vLLM-zh "NVFP4 indexer decode context parallelism": the context is split over the
GPUs, each sends its local top list per head, the owner merges them, and the
result is exact].

- The oracle's local lists and merge give the single-GPU selection (oracle.select,
  the C restatement of the top-k rule) for every world size, ties included: the
  exactness the pages claim, checked against an independent implementation.
- The partition covers every block once.
- The candidate key format (include/msa.h) decodes as documented: hand-built keys
  from IEEE-754 bit patterns.
- Two gloo ranks move their lists with the package's exchange (both the all-gather
  and the owner all-to-all) and the merge of what arrives is the selection.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from block_sparse_attention_nvfp4_gb300 import dcp

from . import _wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def tie_scores(rng, nb):
    """Block scores drawn from a handful of values (many exact ties, both zeros, -inf)."""
    pool = np.array([-np.inf, -3.5, -0.0, 0.0, 0.25, 1.0, 1.0, 2.5, 7.0])
    return pool[rng.integers(0, len(pool), nb)]


def merged(S, world):
    lists = [oracle.dcp_local_topk(S, r, world) for r in range(world)]
    return oracle.dcp_merge(lists, len(S))


@pytest.mark.parametrize("nb", [0, 1, 2, 15, 16, 17, 18, 31, 33, 64, 200, 4097])
def test_merge_of_local_lists_is_the_selection(nb):
    rng = np.random.default_rng(1000 + nb)
    for trial in range(3):
        S = tie_scores(rng, nb) if trial < 2 else rng.standard_normal(nb)
        want = oracle.select(S)
        for world in range(1, 9):
            got = merged(S, world)
            assert np.array_equal(got, want), (nb, world, trial, got, want)


def test_merge_on_workload_block_scores():
    wl = _wl.small([3000, 700, 129, 5000], [1, 2, 1, 3], needles=2, seed=5)
    for b in range(wl.num_reqs):
        S = oracle.block_scores(wl, b)
        for g in range(4):
            for world in (2, 3, 4, 8):
                assert np.array_equal(merged(S[g], world), oracle.select(S[g])), (b, g, world)


def test_local_lists_are_short_and_own_blocks_only():
    rng = np.random.default_rng(3)
    S = rng.standard_normal(300)
    for world in (1, 2, 5, 8):
        for r in range(world):
            lst = oracle.dcp_local_topk(S, r, world)
            assert len(lst) == min(15, len([c for c in range(299) if c % world == r]))
            assert all(c % world == r and c != 299 for _, c in lst)
            assert [s for s, _ in lst] == sorted((s for s, _ in lst), reverse=True)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 8])
def test_partition_covers_each_block_once(world):
    for nb in (0, 1, 5, 16, 17, 1000):
        seen = []
        for r in range(world):
            mine = list(dcp.owned_blocks(nb, r, world))
            assert mine == oracle.dcp_blocks(nb, r, world)
            seen += mine
        assert sorted(seen) == list(range(nb))


def test_owned_groups():
    assert [list(dcp.owned_groups(r, 4, "owner")) for r in range(4)] == [[0], [1], [2], [3]]
    assert [list(dcp.owned_groups(r, 2, "owner")) for r in range(2)] == [[0, 1], [2, 3]]
    assert list(dcp.owned_groups(1, 3, "gather")) == [0, 1, 2, 3]
    with pytest.raises(ValueError):
        dcp.owned_groups(0, 3, "owner")


def _key(score_bits_image, block_id):
    return (score_bits_image << 32) | (0xFFFFFFFF - block_id)


def test_key_format_decodes_as_documented():
    # IEEE-754 single: 1.0 = 0x3F800000, -2.0 = 0xC0000000, 0.5 = 0x3F000000;
    # image: non-negative u -> u | 0x80000000, negative u -> ~u (32 bits)
    k = np.array([_key(0xBF800000, 3),            # 1.0, block 3
                  _key(0x3FFFFFFF, 7),            # -2.0, block 7
                  _key(0x80000000, 0),            # +0.0 (and -0.0), block 0
                  _key(0xBF000000, 4096),         # 0.5, block 4096
                  0], dtype=np.uint64)
    s, ids, present = dcp.decode_keys(k.view(np.int64))
    assert list(present) == [True, True, True, True, False]
    assert list(ids) == [3, 7, 0, 4096, -1]
    assert s[0] == 1.0 and s[1] == -2.0 and s[2] == 0.0 and s[3] == 0.5 and np.isnan(s[4])
    # a larger key is a better block: higher score first, then the lower id
    better = [_key(0xBF800000, 2), _key(0xBF800000, 3), _key(0xBF000000, 0), _key(0x80000000, 9),
              _key(0x3FFFFFFF, 1)]
    assert better == sorted(better, reverse=True)


# ---------------------------------------------------------------- two gloo ranks

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _score_sets():
    """Per request, the four groups' block scores: tie-heavy draws and a workload's."""
    rng = np.random.default_rng(77)
    sets = [np.stack([tie_scores(rng, nb) for _ in range(4)]) for nb in (3, 16, 17, 40, 300, 1025)]
    wl = _wl.small([2000, 130], [2, 1], needles=1, seed=9)
    sets += [oracle.block_scores(wl, b) for b in range(wl.num_reqs)]
    return sets


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sets = _score_sets()
        B = len(sets)
        # this rank's lists: scores (NaN = empty) and ids (-1 = empty), [4, B, 16]
        sc = torch.full((4, B, dcp.SLOTS), float("nan"), dtype=torch.float64)
        ids = torch.full((4, B, dcp.SLOTS), -1, dtype=torch.int64)
        for b, S in enumerate(sets):
            for g in range(4):
                for j, (s, c) in enumerate(oracle.dcp_local_topk(S[g], rank, world)):
                    sc[g, b, j], ids[g, b, j] = s, c
        res = {}
        for mode in ("gather", "owner"):
            got_s = dcp.exchange(sc, torch.empty(dcp.exchange_shape(B, world, mode), dtype=torch.float64), mode)
            got_i = dcp.exchange(ids, torch.empty(dcp.exchange_shape(B, world, mode), dtype=torch.int64), mode)
            groups = list(dcp.owned_groups(rank, world, mode))
            sel = {}
            for gl, g in enumerate(groups):
                for b, S in enumerate(sets):
                    lists = [[(float(got_s[w, gl, b, j]), int(got_i[w, gl, b, j])) for j in range(dcp.SLOTS)
                              if got_i[w, gl, b, j] >= 0] for w in range(world)]
                    sel[(g, b)] = oracle.dcp_merge(lists, S.shape[1]).tolist()
            res[mode] = sel
        out[rank] = res
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_exchange_and_merge_to_the_selection():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0
        res = dict(out)
    sets = _score_sets()
    want = {(g, b): oracle.select(S[g]).tolist() for b, S in enumerate(sets) for g in range(4)}
    for r in range(world):
        assert res[r]["gather"] == want  # every rank merges every group
        owned = {k: v for k, v in want.items() if k[0] in dcp.owned_groups(r, world, "owner")}
        assert res[r]["owner"] == owned  # the owner merges its own groups
