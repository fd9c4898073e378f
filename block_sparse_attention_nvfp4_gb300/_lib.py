"""ctypes binding of libmsa (include/msa.h): argument marshalling only.

Every step of the MSA decode path runs in libmsa's CUDA kernels; this module
turns torch CUDA tensors into the C ABI's plain device pointers and sizes, and
raises MSAError on any non-OK status. There is no fallback: if libmsa.so is
missing or was built for another GPU, calls fail loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

MSA_OK = 0
STATUS = {0: "MSA_OK", -1: "MSA_ERR_INVALID_ARG", -2: "MSA_ERR_UNSUPPORTED", -3: "MSA_ERR_CUDA",
          -4: "MSA_ERR_WORKSPACE", -5: "MSA_ERR_BAD_TABLE", -6: "MSA_ERR_TIMEOUT"}
FLAG_BAD_PAGE, FLAG_BAD_LENGTH, FLAG_TIMEOUT, FLAG_BAD_IDS, FLAG_BAD_SLOT = 0x1, 0x2, 0x4, 0x8, 0x10

# symbols include/msa.h declares (checked by the CPU tests)
EXPORTS = ("msa_status_string", "msa_workspace_size", "msa_workspace_init", "msa_get_error", "msa_index_scores",
           "msa_block_maxpool_topk", "msa_select_blocks", "msa_select_blocks_noalloc", "msa_sparse_attn_decode",
           "msa_decode", "msa_dequant_rows", "msa_kv_insert_nvfp4", "msa_select_blocks_exact",
           "msa_select_blocks_noalloc_get_error", "msa_dcp_local_topk", "msa_dcp_merge_topk",
           "msa_selftest_wait_timeout", "msa_sparse_attn_decode_small_rows")


class MSAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)} ({_status_text(code)})")


class Args(ctypes.Structure):
    """Mirror of msa_decode_args."""
    _fields_ = [("num_reqs", ctypes.c_int32), ("total_rows", ctypes.c_int32), ("max_rows_per_req", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("max_pages_per_req", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("q_per_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("top_k", ctypes.c_int32), ("sm_scale", ctypes.c_float),
                ("context_lens", ctypes.c_void_p), ("q_indptr", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p),
                ("k_data", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_data", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("ki_data", ctypes.c_void_p), ("ki_scale", ctypes.c_void_p)]


class KvInsertArgs(ctypes.Structure):
    """Mirror of msa_kv_insert_args."""
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("slot_mapping", ctypes.c_void_p),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_idx", ctypes.c_void_p),
                ("k_data", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_data", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("ki_data", ctypes.c_void_p), ("ki_scale", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libmsa.so (built by block_sparse_attention_nvfp4_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise OSError(f"libmsa.so not found at {path}; build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
            ap = ctypes.POINTER(Args)
            lib.msa_status_string.restype = ctypes.c_char_p
            lib.msa_status_string.argtypes = [ctypes.c_int]
            lib.msa_workspace_size.argtypes = [ap, ctypes.POINTER(sz)]
            lib.msa_workspace_init.argtypes = [vp, sz, vp]
            lib.msa_get_error.argtypes = [vp, sz, vp, ctypes.POINTER(ctypes.c_uint32)]
            lib.msa_index_scores.argtypes = [ap, vp, i64, vp, sz, vp]
            lib.msa_block_maxpool_topk.argtypes = [ap, vp, i64, vp, vp, vp, sz, vp]
            lib.msa_select_blocks.argtypes = [ap, vp, vp, vp, sz, vp]
            lib.msa_select_blocks_exact.argtypes = [ap, vp, vp, vp, sz, vp]
            lib.msa_select_blocks_noalloc.argtypes = [ap, vp, vp, vp]
            lib.msa_select_blocks_noalloc_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
            lib.msa_sparse_attn_decode.argtypes = [ap, vp, vp, vp, vp, sz, vp]
            lib.msa_sparse_attn_decode_small_rows.argtypes = [ap, vp, vp, vp, vp, sz, vp]
            lib.msa_decode.argtypes = [ap, vp, vp, vp, vp, sz, vp]
            lib.msa_dequant_rows.argtypes = [vp, vp, i64, vp, ctypes.c_int32, vp]
            lib.msa_kv_insert_nvfp4.argtypes = [ctypes.POINTER(KvInsertArgs), vp, sz, vp]
            i32 = ctypes.c_int32
            lib.msa_dcp_local_topk.argtypes = [ap, i32, i32, vp, vp, sz, vp]
            lib.msa_dcp_merge_topk.argtypes = [ap, i32, i32, i32, vp, vp, vp, sz, vp]
            lib.msa_selftest_wait_timeout.argtypes = [vp, sz, vp]
            for f in EXPORTS[1:]:
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _status_text(code: int) -> str:
    try:
        return load().msa_status_string(code).decode()
    except OSError:
        return "?"


def _check(code: int, what: str):
    if code != MSA_OK:
        raise MSAError(code, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "libmsa takes contiguous CUDA tensors"
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_args(cache, batch, sm_scale: float, top_k: int = 16) -> Args:
    """Build msa_decode_args from a KV cache and a decode batch (objects holding
    contiguous CUDA tensors; see api.KVCache / api.DecodeBatch)."""
    a = Args()
    a.num_reqs = int(batch.num_reqs)
    a.total_rows = int(batch.total_rows)
    a.max_rows_per_req = int(batch.max_rows_per_req)
    a.num_pages = int(cache.num_pages)
    a.max_pages_per_req = int(batch.block_table.shape[1])
    a.num_kv_heads, a.q_per_kv, a.head_dim, a.block_size, a.top_k = 4, 8, 128, 128, int(top_k)
    a.sm_scale = float(sm_scale)
    for name in ("context_lens", "q_indptr", "block_table", "q", "q_idx"):
        setattr(a, name, _ptr(getattr(batch, name)).value)
    for name in ("k_data", "k_scale", "v_data", "v_scale", "ki_data", "ki_scale"):
        setattr(a, name, _ptr(getattr(cache, name)).value)
    return a


def msa_workspace_size(args: Args) -> int:
    n = ctypes.c_size_t(0)
    _check(load().msa_workspace_size(ctypes.byref(args), ctypes.byref(n)), "msa_workspace_size")
    return int(n.value)


def msa_workspace_init(ws: torch.Tensor, stream=None):
    _check(load().msa_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "msa_workspace_init")


def msa_get_error(ws: torch.Tensor, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    load().msa_get_error(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream), ctypes.byref(flags))
    return int(flags.value)


def msa_index_scores(args: Args, scores: torch.Tensor, ws: torch.Tensor, stream=None):
    _check(load().msa_index_scores(ctypes.byref(args), _ptr(scores), scores.shape[-1], _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)), "msa_index_scores")


def msa_block_maxpool_topk(args: Args, scores: torch.Tensor, block_ids: torch.Tensor,
                           block_scores: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    _check(load().msa_block_maxpool_topk(ctypes.byref(args), _ptr(scores), scores.shape[-1], _ptr(block_ids),
                                         _ptr(block_scores), _ptr(ws), ws.numel() * ws.element_size(),
                                         _stream(stream)), "msa_block_maxpool_topk")


def msa_select_blocks(args: Args, block_ids: torch.Tensor, block_scores: Optional[torch.Tensor], ws: torch.Tensor,
                      stream=None):
    _check(load().msa_select_blocks(ctypes.byref(args), _ptr(block_ids), _ptr(block_scores), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)), "msa_select_blocks")


def msa_select_blocks_exact(args: Args, block_ids: torch.Tensor, block_scores: Optional[torch.Tensor],
                            ws: torch.Tensor, stream=None):
    _check(load().msa_select_blocks_exact(ctypes.byref(args), _ptr(block_ids), _ptr(block_scores), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(stream)), "msa_select_blocks_exact")


def msa_select_blocks_noalloc(args: Args, block_ids: torch.Tensor, block_scores: Optional[torch.Tensor],
                              stream=None):
    """msa_select_blocks without a caller workspace (scratch inside the library;
    see include/msa.h for the size limit and the sharing rules)."""
    _check(load().msa_select_blocks_noalloc(ctypes.byref(args), _ptr(block_ids), _ptr(block_scores),
                                            _stream(stream)), "msa_select_blocks_noalloc")


def msa_select_blocks_noalloc_get_error(stream=None) -> int:
    """Device error flags (MSA_FLAG_*) of the most recent msa_select_blocks_noalloc call
    (synchronises the stream)."""
    flags = ctypes.c_uint32(0)
    code = load().msa_select_blocks_noalloc_get_error(_stream(stream), ctypes.byref(flags))
    if code not in (MSA_OK, -5, -6):
        _check(code, "msa_select_blocks_noalloc_get_error")
    return int(flags.value)


def msa_dcp_local_topk(args: Args, rank: int, world: int, cand_keys: torch.Tensor, ws: torch.Tensor, stream=None):
    """cand_keys: int64 [4, B, 16] (the uint64 keys' bits)."""
    _check(load().msa_dcp_local_topk(ctypes.byref(args), rank, world, _ptr(cand_keys), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)), "msa_dcp_local_topk")


def msa_dcp_merge_topk(args: Args, world: int, group0: int, n_groups: int, all_keys: torch.Tensor,
                       block_ids: torch.Tensor, ws: torch.Tensor, stream=None):
    """all_keys: int64 [world, n_groups, B, 16]."""
    _check(load().msa_dcp_merge_topk(ctypes.byref(args), world, group0, n_groups, _ptr(all_keys), _ptr(block_ids),
                                     _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "msa_dcp_merge_topk")


def msa_selftest_wait_timeout(ws: torch.Tensor, stream=None):
    """Launch the bounded-wait diagnostic (include/msa.h); read the outcome with msa_get_error."""
    _check(load().msa_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "msa_selftest_wait_timeout")


def msa_sparse_attn_decode(args: Args, block_ids: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor],
                           ws: torch.Tensor, stream=None):
    _check(load().msa_sparse_attn_decode(ctypes.byref(args), _ptr(block_ids), _ptr(out), _ptr(lse), _ptr(ws),
                                         ws.numel() * ws.element_size(), _stream(stream)), "msa_sparse_attn_decode")


def msa_sparse_attn_decode_small_rows(args: Args, block_ids: torch.Tensor, out: torch.Tensor,
                                      lse: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    _check(load().msa_sparse_attn_decode_small_rows(ctypes.byref(args), _ptr(block_ids), _ptr(out), _ptr(lse),
                                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "msa_sparse_attn_decode_small_rows")


def msa_decode_ptrs(args: Args, ids_p, out_p, lse_p, ws_p, ws_bytes: int, stream=None):
    """msa_decode with already-marshalled device pointers (ctypes.c_void_p or None)."""
    _check(load().msa_decode(ctypes.byref(args), ids_p, out_p, lse_p, ws_p, ws_bytes, _stream(stream)), "msa_decode")


def msa_decode(args: Args, block_ids: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor],
               ws: torch.Tensor, stream=None):
    _check(load().msa_decode(ctypes.byref(args), _ptr(block_ids), _ptr(out), _ptr(lse), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "msa_decode")


def msa_dequant_rows(codes: torch.Tensor, scales: torch.Tensor, out: torch.Tensor, path: int, stream=None):
    _check(load().msa_dequant_rows(_ptr(codes), _ptr(scales), codes.shape[0], _ptr(out), int(path),
                                   _stream(stream)), "msa_dequant_rows")


def make_kv_insert_args(cache, slot_mapping: torch.Tensor, k: Optional[torch.Tensor], v: Optional[torch.Tensor],
                        k_idx: Optional[torch.Tensor]) -> KvInsertArgs:
    """msa_kv_insert_args for T new tokens: slot_mapping int64 [T]; k, v FP32 [T, 4, 128]; k_idx FP32
    [T, 128] (any may be None); cache as api.KVCache."""
    a = KvInsertArgs()
    a.num_tokens = int(slot_mapping.shape[0])
    a.num_pages = int(cache.num_pages)
    a.slot_mapping = _ptr(slot_mapping).value
    for name, t in (("k", k), ("v", v), ("k_idx", k_idx)):
        p = _ptr(t)
        setattr(a, name, p.value if p is not None else None)
    for name in ("k_data", "k_scale", "v_data", "v_scale", "ki_data", "ki_scale"):
        setattr(a, name, _ptr(getattr(cache, name)).value)
    return a


def msa_kv_insert_nvfp4(args: KvInsertArgs, ws: torch.Tensor, stream=None):
    _check(load().msa_kv_insert_nvfp4(ctypes.byref(args), _ptr(ws), ws.numel() * ws.element_size(),
                                      _stream(stream)), "msa_kv_insert_nvfp4")
