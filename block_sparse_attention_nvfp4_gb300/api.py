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
        fast = getattr(self, "_decode_ptrs", None)
        if fast is None or fast[0] is not self.args:
            # the outputs and the workspace never move: marshal their pointers once
            fast = (self.args, _lib._ptr(self.block_ids), _lib._ptr(self.out.view(torch.int16)), _lib._ptr(self.lse),
                    _lib._ptr(self.ws), self.ws.numel() * self.ws.element_size())
            self._decode_ptrs = fast
        _lib.msa_decode_ptrs(*fast, stream)
        return self.out, self.block_ids

    def host_io(self) -> "HostIO":
        """Pinned host staging for whole decode steps from host memory (see HostIO)."""
        return HostIO(self)

    def host_stream(self, depth: int = 2) -> "HostStream":
        """Decode steps from host memory with `depth` steps in flight (see HostStream)."""
        return HostStream(self, depth)

    def select_blocks(self, stream=None):
        _lib.msa_select_blocks(self.args, self.block_ids, self.block_scores, self.ws, stream)
        return self.block_ids

    def select_blocks_exact(self, stream=None):
        """Selection with exact index scores (msa_select_blocks_exact)."""
        _lib.msa_select_blocks_exact(self.args, self.block_ids, self.block_scores, self.ws, stream)
        return self.block_ids

    def sparse_attn(self, block_ids: torch.Tensor, stream=None):
        _lib.msa_sparse_attn_decode(self.args, block_ids, self.out.view(torch.int16), self.lse, self.ws, stream)
        return self.out

    def sparse_attn_small_rows(self, block_ids: torch.Tensor, stream=None):
        """The attention with warp-level MMAs (msa_sparse_attn_decode_small_rows; at most 2
        rows per request)."""
        _lib.msa_sparse_attn_decode_small_rows(self.args, block_ids, self.out.view(torch.int16), self.lse, self.ws,
                                               stream)
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


def _packed(specs, device, pin):
    """One uint8 buffer holding the listed (name, shape, dtype) tensors at 256-byte aligned
    offsets; returns (buffer, {name: view})."""
    off, places = 0, []
    for name, shape, dtype in specs:
        n = int(math.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        places.append((name, shape, dtype, off, n))
        off += (n + 255) // 256 * 256
    buf = torch.empty(max(off, 256), dtype=torch.uint8, device=device, pin_memory=pin)
    views = {name: buf[o:o + n].view(dtype).view(shape) for name, shape, dtype, o, n in places}
    return buf, views


class HostIO:
    """A decode step from host memory with one copy each way.

    The decoder's batch inputs (context_lens, q_indptr, block_table, q, q_idx) are moved into
    one device buffer and its outputs (out, block_ids, lse) into another; `inputs` and
    `outputs` are views of pinned host mirrors with the same layout. Fill `inputs`, call
    `step()`: one host-to-device copy, the three decode kernels, one device-to-host copy,
    all on `stream`, then a synchronize; `outputs` then hold the step's results."""

    IN = ("context_lens", "q_indptr", "block_table", "q", "q_idx")

    def __init__(self, dec: "MSADecoder"):
        b = dec.batch
        dev = b.q.device
        spec_in = [(n, tuple(getattr(b, n).shape), getattr(b, n).dtype) for n in self.IN]
        self.dev_in, dviews = _packed(spec_in, dev, False)
        self.host_in, self.inputs = _packed(spec_in, "cpu", True)
        for n in self.IN:
            dviews[n].copy_(getattr(b, n))
            self.inputs[n].copy_(getattr(b, n).cpu())
        dec.rebind(DecodeBatch(dviews["context_lens"], dviews["q_indptr"], dviews["block_table"], dviews["q"],
                               dviews["q_idx"], b.total_rows, b.max_rows_per_req))
        spec_out = [("out", tuple(dec.out.shape), dec.out.dtype), ("block_ids", tuple(dec.block_ids.shape), torch.int32)]
        if dec.lse is not None:
            spec_out.append(("lse", tuple(dec.lse.shape), torch.float32))
        self.dev_out, oviews = _packed(spec_out, dev, False)
        self.host_out, self.outputs = _packed(spec_out, "cpu", True)
        dec.out, dec.block_ids = oviews["out"], oviews["block_ids"]
        dec.lse = oviews.get("lse")
        dec._decode_ptrs = None  # the outputs moved: marshal again
        self.dec = dec
        self.h2d_bytes = self.host_in.numel()
        self.d2h_bytes = self.host_out.numel()

    def step(self, stream=None, graph: bool = True):
        """One step: host inputs -> device, decode, outputs -> host, then synchronize. With
        graph=True the step is captured once as a CUDA graph (the two copies and the three
        kernels, their programmatic-launch chaining kept as graph edges) and replayed: one
        launch per step instead of five. If capture is not possible the step runs eagerly
        (`graph_error` says why)."""
        s = stream if stream is not None else torch.cuda.current_stream()
        self.launch(s, graph)
        s.synchronize()
        return self.outputs

    def launch(self, stream, graph: bool = True):
        """Enqueue one step on `stream` without waiting for it (`step` without the
        synchronize): `outputs` hold its results once the stream has reached that point."""
        if graph and self.graph is None and self.graph_error is None:
            self._capture()
        with torch.cuda.stream(stream):
            if graph and self.graph is not None:
                self.graph.replay()
            else:
                self._enqueue(stream)

    graph = None
    graph_error = None

    def _enqueue(self, s):
        self.dev_in.copy_(self.host_in, non_blocking=True)
        self.dec.decode(s)
        self.host_out.copy_(self.dev_out, non_blocking=True)

    def _capture(self):
        torch.cuda.synchronize()
        with torch.cuda.stream(torch.cuda.Stream()):
            self._enqueue(torch.cuda.current_stream())  # attributes set, pointers marshalled
        torch.cuda.synchronize()
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._enqueue(torch.cuda.current_stream())
            torch.cuda.synchronize()
            self.graph = g
        except Exception as e:  # keep the eager path
            self.graph_error = repr(e)
            torch.cuda.synchronize()


class HostStream:
    """Decode steps from host memory with several in flight: `depth` slots, each its own
    decoder (sharing the cache), pinned input and output mirrors, device buffers and
    workspace (HostIO). Step i uses slot i % depth once that slot's previous step has been
    consumed. Its input copy runs on a copy stream, its three kernels on one compute stream
    shared by all slots (the steps' kernels never compete for SMs), its output copy on a
    second copy stream, ordered by events: the copies of one step overlap the kernels of
    the steps next to it.

    run(steps, fill, consume): for each step, `fill(i, inputs)` writes its inputs into the
    slot's pinned input views (None: keep what is there), and `consume(i, outputs)` is called
    with the slot's pinned output views once the step is complete (before the slot is
    reused, or at the end)."""

    def __init__(self, dec: "MSADecoder", depth: int = 2):
        if depth < 1:
            raise ValueError("depth must be at least 1")
        self.slots = [HostIO(MSADecoder(dec.cache, dec.batch, sm_scale=dec.sm_scale, with_lse=dec.lse is not None))
                      for _ in range(depth)]
        self.copy_in, self.compute, self.copy_out = (torch.cuda.Stream() for _ in range(3))
        self.in_done = [torch.cuda.Event() for _ in range(depth)]
        self.kernels_done = [torch.cuda.Event() for _ in range(depth)]
        self.done = [torch.cuda.Event() for _ in range(depth)]
        self.h2d_bytes = self.slots[0].h2d_bytes
        self.d2h_bytes = self.slots[0].d2h_bytes

    @property
    def depth(self) -> int:
        return len(self.slots)

    def _launch(self, k: int):
        io = self.slots[k]
        with torch.cuda.stream(self.copy_in):
            io.dev_in.copy_(io.host_in, non_blocking=True)
            self.in_done[k].record(self.copy_in)
        self.compute.wait_event(self.in_done[k])
        io.dec.decode(self.compute)
        self.kernels_done[k].record(self.compute)
        self.copy_out.wait_event(self.kernels_done[k])
        with torch.cuda.stream(self.copy_out):
            io.host_out.copy_(io.dev_out, non_blocking=True)
            self.done[k].record(self.copy_out)

    def run(self, steps: int, fill=None, consume=None):
        pending = [None] * self.depth  # the step each slot last ran, until consumed
        for i in range(steps):
            k = i % self.depth
            if pending[k] is not None:
                self.done[k].synchronize()
                if consume is not None:
                    consume(pending[k], self.slots[k].outputs)
                pending[k] = None
            if fill is not None:
                fill(i, self.slots[k].inputs)
            self._launch(k)
            pending[k] = i
        for j in range(steps, steps + self.depth):  # the last steps, in order
            k = j % self.depth
            if pending[k] is not None:
                self.done[k].synchronize()
                if consume is not None:
                    consume(pending[k], self.slots[k].outputs)
                pending[k] = None
