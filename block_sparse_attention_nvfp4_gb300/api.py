"""User-facing Python API over libmsa: device-resident NVFP4 KV cache, a decode
batch, and a decoder object that owns its workspace and outputs. All compute
runs in libmsa's kernels (see _lib)."""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

from . import _lib


@dataclasses.dataclass
class KVCache:
    """Paged NVFP4 caches on the GPU: K/V [P,4,128,64|8], index keys [P,128,64|8] (uint8)."""
    k_data: torch.Tensor
    k_scale: torch.Tensor
    v_data: torch.Tensor
    v_scale: torch.Tensor
    ki_data: torch.Tensor
    ki_scale: torch.Tensor

    @property
    def num_pages(self) -> int:
        return int(self.ki_data.shape[0])

    @staticmethod
    def from_host(wl, device="cuda") -> "KVCache":
        t = lambda a: torch.from_numpy(a).to(device)  # noqa: E731
        return KVCache(t(wl.k_data), t(wl.k_scale), t(wl.v_data), t(wl.v_scale), t(wl.ki_data), t(wl.ki_scale))

    @staticmethod
    def empty(num_pages: int, device="cuda") -> "KVCache":
        z = lambda *shape: torch.zeros(shape, dtype=torch.uint8, device=device)  # noqa: E731
        return KVCache(z(num_pages, 4, 128, 64), z(num_pages, 4, 128, 8), z(num_pages, 4, 128, 64),
                       z(num_pages, 4, 128, 8), z(num_pages, 128, 64), z(num_pages, 128, 8))

    def insert(self, slot_mapping: torch.Tensor, k: Optional[torch.Tensor], v: Optional[torch.Tensor],
               k_idx: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
        """Quantise T new tokens to NVFP4 into their slots (msa_kv_insert_nvfp4): slot_mapping
        int64 [T] (page * 128 + slot, negative = skip), k and v FP32 [T, 4, 128], k_idx FP32
        [T, 128], any of them None; ws a zero-filled workspace of >= 256 bytes (error flags)."""
        args = _lib.make_kv_insert_args(self, slot_mapping, k, v, k_idx)
        _lib.msa_kv_insert_nvfp4(args, ws, stream)


@dataclasses.dataclass
class DecodeBatch:
    """One decode step's per-request metadata and FP8 queries on the GPU."""
    context_lens: torch.Tensor   # int32 [B]
    q_indptr: torch.Tensor       # int32 [B+1]
    block_table: torch.Tensor    # int32 [B, max_pages]
    q: torch.Tensor              # uint8 [rows, 32, 128]
    q_idx: torch.Tensor          # uint8 [rows, 4, 128]
    total_rows: int
    max_rows_per_req: int

    @property
    def num_reqs(self) -> int:
        return int(self.context_lens.shape[0])

    @staticmethod
    def from_host(wl, device="cuda") -> "DecodeBatch":
        t = lambda a: torch.from_numpy(a).to(device)  # noqa: E731
        rows = wl.q_indptr[1:] - wl.q_indptr[:-1]
        return DecodeBatch(t(wl.context_lens), t(wl.q_indptr), t(wl.block_table), t(wl.q), t(wl.q_idx),
                           int(wl.total_rows), max(1, int(rows.max(initial=1))))


class MSADecoder:
    """Holds the workspace and outputs for a (cache, batch) shape and runs the
    decode path through the C ABI."""

    def __init__(self, cache: KVCache, batch: DecodeBatch, sm_scale: Optional[float] = None,
                 with_lse: bool = True, with_block_scores: bool = False):
        self.cache, self.batch = cache, batch
        self.sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(128)
        self.args = _lib.make_args(cache, batch, self.sm_scale)
        dev = batch.q.device
        self.ws = torch.empty(_lib.msa_workspace_size(self.args), dtype=torch.uint8, device=dev)
        _lib.msa_workspace_init(self.ws)
        B, P = batch.num_reqs, batch.block_table.shape[1]
        self.block_ids = torch.empty((B, 4, 16), dtype=torch.int32, device=dev)
        self.out = torch.empty((batch.total_rows, 32, 128), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((batch.total_rows, 32), dtype=torch.float32, device=dev) if with_lse else None
        self.block_scores = torch.empty((B, 4, P), dtype=torch.float32, device=dev) if with_block_scores else None

    def rebind(self, batch: DecodeBatch):
        """Point at another batch of the same shape (same tensors sizes)."""
        self.batch = batch
        self.args = _lib.make_args(self.cache, batch, self.sm_scale)

    def decode(self, stream=None):
        _lib.msa_decode(self.args, self.block_ids, self.out.view(torch.int16), self.lse, self.ws, stream)
        return self.out, self.block_ids

    def select_blocks(self, stream=None):
        _lib.msa_select_blocks(self.args, self.block_ids, self.block_scores, self.ws, stream)
        return self.block_ids

    def sparse_attn(self, block_ids: torch.Tensor, stream=None):
        _lib.msa_sparse_attn_decode(self.args, block_ids, self.out.view(torch.int16), self.lse, self.ws, stream)
        return self.out

    def index_scores(self, stream=None) -> torch.Tensor:
        stride = self.batch.block_table.shape[1] * 128
        s = torch.full((self.batch.total_rows, 4, stride), float("nan"), dtype=torch.float32,
                       device=self.batch.q.device)
        _lib.msa_index_scores(self.args, s, self.ws, stream)
        return s

    def maxpool_topk(self, scores: torch.Tensor, stream=None):
        _lib.msa_block_maxpool_topk(self.args, scores, self.block_ids, self.block_scores, self.ws, stream)
        return self.block_ids

    def errors(self, stream=None) -> int:
        return _lib.msa_get_error(self.ws, stream)


def dequant_rows(codes: torch.Tensor, scales: torch.Tensor, path: int = 0) -> torch.Tensor:
    out = torch.empty((codes.shape[0], 128), dtype=torch.uint8, device=codes.device)
    _lib.msa_dequant_rows(codes, scales, out, path)
    return out
