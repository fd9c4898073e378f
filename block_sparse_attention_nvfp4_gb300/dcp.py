"""Indexer decode context parallelism (DCP) across GPUs, one process per GPU
[vLLM-zh "NVFP4 indexer decode context parallelism"].

Each rank holds its share of every request's index-key pages (logical block c on
rank c % world), scores that share for all four groups (msa_dcp_local_topk), and
the ranks exchange their 15-candidate lists per (group, request). The merge
(msa_dcp_merge_topk) gives the exact top-16 of the whole context: the ids
msa_select_blocks returns on one GPU holding every page.

Two exchanges:
  "gather"  every rank receives every rank's lists (one all-gather of
            4 * B * 16 keys per rank) and merges all four groups;
  "owner"   group g's lists go to the rank that owns g (an all-to-all; world
            divides 4, rank r owns groups r * 4 / world ...), which merges only
            its own groups, as when the attention heads are split over the ranks.

The compute runs in libmsa's kernels; torch.distributed moves the lists (NCCL
between GPUs). Keys travel as int64 (the uint64 bits).
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch
import torch.distributed as dist

from . import _lib

MAX_WORLD = 8
SLOTS = 16  # keys per (group, request) list


def owned_blocks(num_blocks: int, rank: int, world: int) -> range:
    """Logical blocks of a request of num_blocks blocks that rank `rank` scores."""
    return range(rank, num_blocks, world)


def owned_groups(rank: int, world: int, mode: str) -> range:
    """Groups whose selection rank `rank` merges."""
    if mode == "gather":
        return range(4)
    if mode != "owner" or 4 % world:
        raise ValueError(f"exchange {mode!r} with world {world}: 'owner' needs a world that divides 4")
    per = 4 // world
    return range(rank * per, (rank + 1) * per)


def exchange_shape(num_reqs: int, world: int, mode: str) -> tuple:
    """Shape of the received lists: [world, groups merged here, B, 16]."""
    return (world, len(owned_groups(0, world, mode)), num_reqs, SLOTS)


def exchange(keys: torch.Tensor, out: torch.Tensor, mode: str = "gather", group=None) -> torch.Tensor:
    """Move every rank's lists keys [4, B, 16] into out (exchange_shape): rank order
    along dim 0; "gather" keeps all four groups, "owner" this rank's groups only."""
    world = dist.get_world_size(group)
    B = keys.shape[1]
    if tuple(out.shape) != exchange_shape(B, world, mode) or not out.is_contiguous():
        raise ValueError(f"exchange buffer {tuple(out.shape)}, expected {exchange_shape(B, world, mode)}")
    if mode == "gather":
        dist.all_gather_into_tensor(out.view(world * 4, B, SLOTS), keys, group=group)
    else:
        owned_groups(0, world, mode)  # checks the world
        dist.all_to_all_single(out.view(4, B, SLOTS), keys, group=group)
    return out


def decode_keys(keys) -> tuple:
    """Host view of candidate keys (any shape, int64 or uint64 bits): (scores FP32,
    block ids int64, present bool). Key = order image of the score << 32 | ~id;
    0 = no candidate."""
    k = np.asarray(keys).astype(np.int64).view(np.uint64)
    hi = (k >> np.uint64(32)).astype(np.uint32)
    lo = (k & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    neg = (hi & np.uint32(0x80000000)) == 0
    bits = np.where(neg, ~hi, hi & np.uint32(0x7FFFFFFF)).astype(np.uint32)
    scores = bits.view(np.float32)
    ids = (np.uint32(0xFFFFFFFF) - lo).astype(np.int64)
    present = k != 0
    return np.where(present, scores, np.float32(np.nan)), np.where(present, ids, -1), present


class DCPSelector:
    """Block selection of one rank of a DCP group: this rank's index-key cache and the
    whole batch's metadata (the block table's entries at this rank's blocks name pages
    of this rank's cache). select() runs the local scan and lists, the exchange and the
    merge, and returns block_ids [B, 4, 16] (rows of the groups this rank merges)."""

    def __init__(self, cache, batch, group=None, mode: str = "gather", sm_scale: Optional[float] = None):
        self.group, self.mode = group, mode
        self.rank, self.world = dist.get_rank(group), dist.get_world_size(group)
        if not 1 <= self.world <= MAX_WORLD:
            raise ValueError(f"world {self.world} outside 1..{MAX_WORLD}")
        self.groups = owned_groups(self.rank, self.world, mode)
        self.cache, self.batch = cache, batch  # the args below hold raw pointers into them
        self.args = _lib.make_args(cache, batch, sm_scale if sm_scale is not None else 128 ** -0.5)
        dev = batch.q_idx.device
        self.ws = torch.empty(_lib.msa_workspace_size(self.args), dtype=torch.uint8, device=dev)
        _lib.msa_workspace_init(self.ws)
        B = batch.num_reqs
        self.keys = torch.zeros((4, B, SLOTS), dtype=torch.int64, device=dev)
        self.received = torch.zeros(exchange_shape(B, self.world, mode), dtype=torch.int64, device=dev)
        self.block_ids = torch.full((B, 4, 16), -1, dtype=torch.int32, device=dev)

    def local(self, stream=None) -> torch.Tensor:
        _lib.msa_dcp_local_topk(self.args, self.rank, self.world, self.keys, self.ws, stream)
        return self.keys

    def merge(self, stream=None) -> torch.Tensor:
        _lib.msa_dcp_merge_topk(self.args, self.world, self.groups.start, len(self.groups), self.received,
                                self.block_ids, self.ws, stream)
        return self.block_ids

    def select(self) -> torch.Tensor:
        self.local()
        exchange(self.keys, self.received, self.mode, self.group)
        return self.merge()

    def errors(self, stream=None) -> int:
        return _lib.msa_get_error(self.ws, stream)
