"""Indexer decode context parallelism (DCP) through the C ABI on one GPU, the ranks
run one after another, each with a cache holding only its own pages
[vLLM-zh "NVFP4 indexer decode context parallelism": each GPU scores its share of
the context for every head, sends a local top list per head, and the owner's merge
gives the exact final top-16].

For every rank: its candidate lists (msa_dcp_local_topk) equal the oracle's local
lists (dcp_local_topk) computed on the single-GPU selection's own FP32 block
scores; block-table entries at other ranks' blocks are -1 and the rank's cache
holds only its pages, so a read outside the rank's share would flag a bad page.
The merge of all ranks' lists (msa_dcp_merge_topk), after an all-gather layout and
after an owner all-to-all layout, equals msa_select_blocks' ids exactly, ties
included. A corrupt or empty exchange sets MSA_FLAG_BAD_IDS."""
import copy

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_nvfp4_gb300 import DecodeBatch, KVCache, _lib, dcp, synth
from tests import _gpu, _topk_sim, _wl
from tests.test_gpu_topk_ties import aliased

gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def rank_workload(wl, rank, world):
    """Rank `rank`'s view: the pages its blocks use, renumbered into a cache of its own;
    block-table entries of other ranks' blocks (and past the context) set to -1."""
    nbs = (np.asarray(wl.context_lens, np.int64) + 127) // 128
    bt = np.full_like(wl.block_table, -1)
    pages = {}
    for b in range(wl.num_reqs):
        for c in range(rank, int(nbs[b]), world):
            phys = int(wl.block_table[b, c])
            bt[b, c] = pages.setdefault(phys, len(pages))
    keep = np.array(sorted(pages, key=pages.get) or [0], np.int64)
    w = copy.copy(wl)
    w.block_table = bt
    w.num_pages = len(keep)
    for name in ("k_data", "k_scale", "v_data", "v_scale", "ki_data", "ki_scale"):
        setattr(w, name, np.ascontiguousarray(getattr(wl, name)[keep]))
    return w


class Ranks:
    """The lists of every rank of a world, and a merge workspace."""

    def __init__(self, wl, world):
        self.wl, self.world, self.keys = wl, world, []
        for r in range(world):
            wr = rank_workload(wl, r, world)
            # args hold raw pointers: the rank's tensors must outlive the call
            cache, batch = KVCache.from_host(wr), DecodeBatch.from_host(wr)
            args = _lib.make_args(cache, batch, wl.sm_scale)
            ws = torch.empty(_lib.msa_workspace_size(args), dtype=torch.uint8, device="cuda")
            _lib.msa_workspace_init(ws)
            k = torch.zeros((4, wl.num_reqs, dcp.SLOTS), dtype=torch.int64, device="cuda")
            _lib.msa_dcp_local_topk(args, r, world, k, ws)
            assert _lib.msa_get_error(ws) == 0, f"rank {r}"
            self.keys.append(k)
            del cache, batch
        self.batch = DecodeBatch.from_host(wl)
        self.cache = KVCache.from_host(wl)
        self.args = _lib.make_args(self.cache, self.batch, wl.sm_scale)
        self.ws = torch.empty(_lib.msa_workspace_size(self.args), dtype=torch.uint8, device="cuda")
        _lib.msa_workspace_init(self.ws)

    def merge_gather(self, all_keys=None):
        if all_keys is None:
            all_keys = torch.stack(self.keys).contiguous()
        ids = torch.full((self.wl.num_reqs, 4, 16), -7, dtype=torch.int32, device="cuda")
        _lib.msa_dcp_merge_topk(self.args, self.world, 0, 4, all_keys, ids, self.ws)
        return ids.cpu().numpy(), _lib.msa_get_error(self.ws)

    def merge_owner(self):
        ids = torch.full((self.wl.num_reqs, 4, 16), -7, dtype=torch.int32, device="cuda")
        for r in range(self.world):
            gs = dcp.owned_groups(r, self.world, "owner")
            recv = torch.stack([k[gs.start:gs.stop] for k in self.keys]).contiguous()
            _lib.msa_dcp_merge_topk(self.args, self.world, gs.start, len(gs), recv, ids, self.ws)
        return ids.cpu().numpy(), _lib.msa_get_error(self.ws)


def single_gpu(wl):
    dec = _gpu.decoder(wl, with_block_scores=True)
    ids = dec.select_blocks().cpu().numpy()
    bs = dec.block_scores.cpu().numpy()
    assert dec.errors() == 0
    return ids, bs


def check_lists(ranks, bs):
    """Each rank's lists equal the oracle's local lists on the same FP32 block scores.
    Returns the filter branch (tests/_topk_sim.dcp_local) of each list."""
    wl, world = ranks.wl, ranks.world
    branches = set()
    for r, k in enumerate(ranks.keys):
        s, ids, present = dcp.decode_keys(k.cpu().numpy())
        for b in range(wl.num_reqs):
            nb = (int(wl.context_lens[b]) + 127) // 128
            R = int(wl.q_indptr[b + 1] - wl.q_indptr[b])
            if R == 0:
                nb = 0
            for g in range(4):
                S = bs[b, g, :nb].astype(np.float64)
                want = oracle.dcp_local_topk(S, r, world)
                n = int(present[g, b].sum())
                assert n == len(want) and not present[g, b, n:].any(), (r, b, g, n, len(want))
                assert [int(x) for x in ids[g, b, :n]] == [c for _, c in want], (r, b, g)
                assert [float(x) for x in s[g, b, :n]] == [v for v, _ in want], (r, b, g)
                loc = [c for c in range(r, nb, world) if c != nb - 1]
                if loc:
                    branches.update(br for _, br in _topk_sim.dcp_local(bs[b, g, loc], len(loc)))
    return branches


WORKLOADS = {
    "mixed": lambda: _wl.small([3000, 700, 129, 5000, 20000, 1], [1, 2, 1, 3, 8, 1], needles=2, seed=21),
    "ragged_rows0": lambda: _wl.small([4096, 2048, 300], [2, 0, 1], needles=1, seed=22),
}


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("name", sorted(WORKLOADS))
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_dcp_equals_single_gpu_selection(name, world):
    wl = WORKLOADS[name]()
    ids, bs = single_gpu(wl)
    ranks = Ranks(wl, world)
    check_lists(ranks, bs)
    got, flags = ranks.merge_gather()
    assert flags == 0
    assert np.array_equal(got, ids)
    if 4 % world == 0:
        got, flags = ranks.merge_owner()
        assert flags == 0
        assert np.array_equal(got, ids)


# tie-heavy single requests (logical blocks aliased onto a few pages): each reaches the
# named filter branch of the rank-local list on at least one (rank, group)
TIES = [
    (8, 3000, 8, 1, "chunked/stream"),     # quarters of ~750 candidates: streamed, > 64 survivors
    (8, 5000, 16, 2, "chunked/stream"),    # quarters of ~625: streamed
    (8, 3000, 8, 4, "chunked/regs"),       # quarters of ~187: held in registers, > 64 survivors
    (4, 3000, 8, 4, "two_sorts/regs"),     # registers, 33..64 survivors
    (8, 1100, 1, 2, "two_sorts/regs"),
    (8, 300, 1, 4, "sort/regs"),
]


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("pages,nb,run,world,branch", TIES)
def test_dcp_ties(pages, nb, run, world, branch):
    wl = aliased(pages, nb, run, tail=37)
    ids, bs = single_gpu(wl)
    _gpu.assert_topk_exact_on_own_scores(ids[0, 0], bs[0, 0], nb, "single")
    ranks = Ranks(wl, world)
    assert branch in check_lists(ranks, bs)
    got, flags = ranks.merge_gather()
    assert flags == 0 and np.array_equal(got, ids)
    if 4 % world == 0:
        got, flags = ranks.merge_owner()
        assert flags == 0 and np.array_equal(got, ids)


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("preset,world", [("long_512k", 4), ("spec8_128k", 4), ("ragged64", 2)])
def test_dcp_on_workload_shapes(preset, world):
    wl = synth.make_workload(synth.preset(preset))
    ids, bs = single_gpu(wl)
    ranks = Ranks(wl, world)
    check_lists(ranks, bs)
    got, flags = ranks.merge_gather()
    assert flags == 0 and np.array_equal(got, ids)


@pytest.mark.gpu
@gpu
def test_dcp_merge_flags_a_corrupt_exchange():
    wl = _wl.small([5000, 3000], [1, 2], seed=23)
    ids, _ = single_gpu(wl)
    ranks = Ranks(wl, 2)
    all_keys = torch.stack(ranks.keys).contiguous()
    # a key of rank 1 that names one of rank 0's blocks: dropped and flagged
    bad = all_keys.clone()
    k = bad[1, 2, 0, 0].item() & ~0xFFFFFFFF
    bad[1, 2, 0, 0] = k | (0xFFFFFFFF - 4)
    got, flags = ranks.merge_gather(bad)
    assert flags & _lib.FLAG_BAD_IDS
    assert np.array_equal(got[1], ids[1])  # the other request is untouched by the bad key
    # the recent block as a candidate
    bad = all_keys.clone()
    nb0 = (int(wl.context_lens[0]) + 127) // 128
    owner = (nb0 - 1) % 2
    bad[owner, 0, 0, 0] = (bad[owner, 0, 0, 0].item() & ~0xFFFFFFFF) | (0xFFFFFFFF - (nb0 - 1))
    _, flags = ranks.merge_gather(bad)
    assert flags & _lib.FLAG_BAD_IDS
    # nothing arrived for request 1, group 3: only the recent block, then -1
    bad = all_keys.clone()
    bad[:, 3, 1, :] = 0
    got, flags = ranks.merge_gather(bad)
    assert flags & _lib.FLAG_BAD_IDS
    nb1 = (int(wl.context_lens[1]) + 127) // 128
    assert got[1, 3].tolist() == [nb1 - 1] + [-1] * 15
    # a clean merge afterwards reports nothing
    got, flags = ranks.merge_gather()
    assert flags == 0 and np.array_equal(got, ids)


@pytest.mark.gpu
@gpu
def test_dcp_rejects_bad_rank_arguments():
    wl = _wl.small([1000], [1], seed=24)
    batch, cache = DecodeBatch.from_host(wl), KVCache.from_host(wl)
    args = _lib.make_args(cache, batch, wl.sm_scale)
    ws = torch.zeros(_lib.msa_workspace_size(args), dtype=torch.uint8, device="cuda")
    k = torch.zeros((4, 1, 16), dtype=torch.int64, device="cuda")
    for rank, world in ((2, 2), (-1, 2), (0, 0), (0, 9)):
        with pytest.raises(_lib.MSAError):
            _lib.msa_dcp_local_topk(args, rank, world, k, ws)
    ids = torch.zeros((1, 4, 16), dtype=torch.int32, device="cuda")
    for world, g0, ng in ((0, 0, 4), (9, 0, 4), (2, 3, 2), (2, 0, 0)):
        with pytest.raises(_lib.MSAError):
            _lib.msa_dcp_merge_topk(args, world, g0, ng, k.view(1, 4, 1, 16), ids, ws)


@pytest.mark.gpu
@gpu
@pytest.mark.parametrize("mode", ["gather", "owner"])
def test_dcp_selector_through_nccl_single_rank(mode):
    """dcp.DCPSelector end to end (local step, NCCL exchange, merge) in a one-rank group:
    the ids equal msa_select_blocks'."""
    import socket
    import torch.distributed as dist
    if not dist.is_nccl_available():
        pytest.skip("NCCL not available")
    wl = WORKLOADS["mixed"]()
    ids, _ = single_gpu(wl)
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        sel = dcp.DCPSelector(KVCache.from_host(wl), DecodeBatch.from_host(wl), mode=mode, sm_scale=wl.sm_scale)
        got = sel.select().cpu().numpy()
        torch.cuda.synchronize()
        assert sel.errors() == 0
        assert np.array_equal(got, ids)
    finally:
        dist.destroy_process_group()
