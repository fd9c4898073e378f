"""Oracle for the MSA decode path — TEST INFRASTRUCTURE ONLY.

Python access to ``msa_oracle.c``, a plain FP64 CPU restatement of what the
MiniMax Sparse Attention decode path computes (index scan -> block max pool ->
top-16 selection with the recent block kept -> exact softmax attention over the
selected blocks' dequantised K/V). Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may use it; the product path never
does, and the oracle imports nothing from the product package.

Inputs are duck-typed: any object with the workload attributes (``num_reqs``,
``num_pages``, ``max_pages_per_req``, ``context_lens``, ``q_indptr``,
``block_table``, ``q``, ``q_idx``, ``k_data``/``k_scale``, ``v_data``/``v_scale``,
``ki_data``/``ki_scale``, ``sm_scale``, ``top_k``) as numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB = os.path.join(_HERE, "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None

G, HQ, D, BLOCK = 4, 32, 128, 128


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, FP64, no FMA contraction so x86 and Arm agree)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"],
                   check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Args(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_pages_per_req", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("sm_scale", ctypes.c_double),
                ("context_lens", ctypes.c_void_p), ("q_indptr", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p),
                ("k_data", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_data", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("ki_data", ctypes.c_void_p), ("ki_scale", ctypes.c_void_p),
                ("exact_index_scores", ctypes.c_int32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            ap = ctypes.POINTER(_Args)
            lib.oracle_e2m1_value.restype = ctypes.c_double
            lib.oracle_e2m1_value.argtypes = [ctypes.c_int]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_value.argtypes = [ctypes.c_int]
            lib.oracle_e4m3_round.restype = ctypes.c_int
            lib.oracle_e4m3_round.argtypes = [ctypes.c_double]
            lib.oracle_dequant_value.restype = ctypes.c_double
            lib.oracle_dequant_value.argtypes = [ctypes.c_int, ctypes.c_int]
            lib.oracle_dequant_value_exact.restype = ctypes.c_double
            lib.oracle_dequant_value_exact.argtypes = [ctypes.c_int, ctypes.c_int]
            lib.oracle_dequant_table.argtypes = [dp]
            lib.oracle_token_scores.argtypes = [ap, ctypes.c_int, dp]
            lib.oracle_block_maxpool.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp]
            lib.oracle_block_scores.argtypes = [ap, ctypes.c_int, dp]
            lib.oracle_select.argtypes = [ctypes.c_int, ctypes.c_int, dp, ip]
            lib.oracle_attend.argtypes = [ap, ctypes.c_int, ip, dp, dp]
            lib.oracle_decode.argtypes = [ap, ctypes.c_int, ip, ip, dp, dp, dp]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            u8p = ctypes.POINTER(ctypes.c_uint8)
            fp = ctypes.POINTER(ctypes.c_float)
            lib.oracle_e2m1_round.restype = ctypes.c_int
            lib.oracle_e2m1_round.argtypes = [ctypes.c_double]
            lib.oracle_nvfp4_quantize_row.argtypes = [fp, ctypes.c_int, u8p, u8p]
            lib.oracle_kv_insert.restype = ctypes.c_int
            lib.oracle_kv_insert.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int64), fp, fp, fp,
                                             u8p, u8p, u8p, u8p, u8p, u8p]
            for f in ("oracle_token_scores", "oracle_block_maxpool", "oracle_block_scores", "oracle_select",
                      "oracle_attend", "oracle_decode"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


class _Bound:
    """Keeps the numpy arrays alive while the C struct points at them."""

    def __init__(self, wl, exact: bool = False):
        self.arrs = {
            "context_lens": _c(wl.context_lens, np.int32), "q_indptr": _c(wl.q_indptr, np.int32),
            "block_table": _c(wl.block_table, np.int32), "q": _c(wl.q, np.uint8), "q_idx": _c(wl.q_idx, np.uint8),
            "k_data": _c(wl.k_data, np.uint8), "k_scale": _c(wl.k_scale, np.uint8),
            "v_data": _c(wl.v_data, np.uint8), "v_scale": _c(wl.v_scale, np.uint8),
            "ki_data": _c(wl.ki_data, np.uint8), "ki_scale": _c(wl.ki_scale, np.uint8),
        }
        self.args = _Args(num_reqs=int(wl.num_reqs), num_pages=int(wl.num_pages),
                          max_pages_per_req=int(wl.max_pages_per_req), top_k=int(getattr(wl, "top_k", 16)),
                          sm_scale=float(wl.sm_scale), exact_index_scores=1 if exact else 0,
                          **{k: v.ctypes.data for k, v in self.arrs.items()})

    def ref(self):
        return ctypes.byref(self.args)


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# ---- formats -----------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return _load().oracle_e4m3_value(int(byte))


def e4m3_round(x: float) -> int:
    return _load().oracle_e4m3_round(float(x))


def dequant_value(code: int, scale: int) -> float:
    return _load().oracle_dequant_value(int(code), int(scale))


def dequant_value_exact(code: int, scale: int) -> float:
    """E2M1(code) x E4M3(scale), not re-rounded (the exact-score indexer's key values)."""
    return _load().oracle_dequant_value_exact(int(code), int(scale))


def dequant_table() -> np.ndarray:
    """[256 scales, 16 codes] FP64 values the FP8 MMA consumes."""
    out = np.empty(256 * 16, np.float64)
    _load().oracle_dequant_table(_dp(out))
    return out.reshape(256, 16)


# ---- the path ----------------------------------------------------------------

def _geom(wl, b):
    N = int(wl.context_lens[b])
    R = int(wl.q_indptr[b + 1] - wl.q_indptr[b])
    return N, R


def token_scores(wl, b: int, exact: bool = False) -> np.ndarray:
    """Index scores of request b: [R, 4, N] FP64, -inf where a key lies after the row.
    exact=True: index keys dequantised without the E4M3 re-rounding (exact-score indexer)."""
    N, R = _geom(wl, b)
    out = np.empty(R * G * N + 1, np.float64)
    bd = _Bound(wl, exact)
    _check(_load().oracle_token_scores(bd.ref(), b, _dp(out)), "token_scores")
    return out[:R * G * N].reshape(R, G, N)


def block_maxpool(token_s: np.ndarray) -> np.ndarray:
    """[R, 4, N] token scores -> [4, nb] block scores (max over rows and block tokens)."""
    R, g, N = token_s.shape
    s = np.ascontiguousarray(token_s, dtype=np.float64)
    nb = (N + BLOCK - 1) // BLOCK
    out = np.empty(G * nb + 1, np.float64)
    _check(_load().oracle_block_maxpool(R, N, _dp(s), _dp(out)), "block_maxpool")
    return out[:G * nb].reshape(G, nb)


def block_scores(wl, b: int, exact: bool = False) -> np.ndarray:
    N, R = _geom(wl, b)
    nb = (N + BLOCK - 1) // BLOCK
    out = np.empty(G * nb + 1, np.float64)
    bd = _Bound(wl, exact)
    _check(_load().oracle_block_scores(bd.ref(), b, _dp(out)), "block_scores")
    return out[:G * nb].reshape(G, nb)


def select(S_g: np.ndarray, top_k: int = 16) -> np.ndarray:
    """Top-k block ids of one group's block scores (recent block kept), ascending, -1 padded."""
    S = np.ascontiguousarray(S_g, dtype=np.float64)
    ids = np.empty(top_k, np.int32)
    _check(_load().oracle_select(len(S), top_k, _dp(S), _ip(ids)), "select")
    return ids


# ---------------------------------------------------------------- indexer DCP
# [vLLM-zh] "NVFP4 indexer decode context parallelism": the context is split over
# the GPUs, each scores its part for all four heads (groups) and sends a local top
# list per head; the owner merges the lists into the final top-16, and the result is
# exact. Reading (the pages do not say how the context is split): logical block c
# belongs to rank c % world. The recent block is kept by the merge, so a local list
# holds the rank's top_k - 1 best other blocks.

def dcp_blocks(nb: int, rank: int, world: int) -> list:
    """Logical blocks of a request of nb blocks that rank `rank` of `world` scores."""
    return [c for c in range(nb) if c % world == rank]


def dcp_local_topk(S_g: np.ndarray, rank: int, world: int, top_k: int = 16) -> list:
    """One group's local list on one rank: [(score, block id)] of the rank's blocks other
    than the recent one, best first (higher score, then lower id), at most top_k - 1."""
    nb = len(S_g)
    cands = [(float(S_g[c]), c) for c in dcp_blocks(nb, rank, world) if c != nb - 1]
    assert not any(np.isnan(s) for s, _ in cands)
    cands.sort(key=lambda sc: (-sc[0], sc[1]))
    return cands[:top_k - 1]


def dcp_merge(lists, nb: int, top_k: int = 16) -> np.ndarray:
    """The owner's merge of every rank's list for one group of a request of nb blocks:
    the recent block plus the top_k - 1 best candidates of all lists; every block when
    nb <= top_k. Ids ascending, -1 padded (the layout of select())."""
    if nb <= top_k:
        chosen = list(range(nb))
    else:
        pool = sorted((sc for lst in lists for sc in lst), key=lambda sc: (-sc[0], sc[1]))
        chosen = sorted([c for _, c in pool[:top_k - 1]] + [nb - 1])
    return np.array(chosen + [-1] * (top_k - len(chosen)), np.int32)


def attend(wl, b: int, ids: np.ndarray):
    """Attention of request b over block ids [4, top_k]: (out [R,32,128], lse [R,32])."""
    N, R = _geom(wl, b)
    total = int(wl.total_rows)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    out = np.zeros((total, HQ, D), np.float64)
    lse = np.zeros((total, HQ), np.float64)
    bd = _Bound(wl)
    _check(_load().oracle_attend(bd.ref(), b, _ip(ids), _dp(out), _dp(lse)), "attend")
    r0 = int(wl.q_indptr[b])
    return out[r0:r0 + R], lse[r0:r0 + R]


def decode(wl, reqs=None):
    """The whole path for the listed requests (all by default).

    Returns dict(ids [n,4,top_k] int32, S [n,4,max_pages] FP64 block scores,
    out [total_rows,32,128] FP64, lse [total_rows,32]) — rows of unlisted
    requests stay zero."""
    if reqs is None:
        reqs = range(int(wl.num_reqs))
    reqs = np.ascontiguousarray(np.asarray(list(reqs), dtype=np.int32))
    n = len(reqs)
    top_k = int(getattr(wl, "top_k", 16))
    ids = np.empty((n, G, top_k), np.int32)
    S = np.empty((n, G, int(wl.max_pages_per_req)), np.float64)
    out = np.zeros((int(wl.total_rows), HQ, D), np.float64)
    lse = np.zeros((int(wl.total_rows), HQ), np.float64)
    bd = _Bound(wl)
    _check(_load().oracle_decode(bd.ref(), n, _ip(reqs), _ip(ids), _dp(S), _dp(out), _dp(lse)), "decode")
    return {"reqs": reqs, "ids": ids, "S": S, "out": out, "lse": lse}


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_threads(n: int) -> int:
    """Threads of decode()'s loop over requests (scheduling only; results do not
    depend on it). Returns the count in effect."""
    return int(_load().oracle_set_threads(int(n)))


# ---------------------------------------------------------------- NVFP4 insertion
# [vLLM-zh] "QKV GEMM + norm + RoPE + KV insert fusion": new K, V and index keys
# arrive as FP32 and are quantised to NVFP4 into their caches.

def e2m1_round(y: float) -> int:
    """E2M1 code (sign in bit 3) of the magnitude nearest |y|, ties to even, saturating."""
    return int(_load().oracle_e2m1_round(float(y)))


def nvfp4_quantize_rows(x: np.ndarray):
    """FP32 rows [..., n] (n a multiple of 16) -> (codes [..., n/2] u8, scales [..., n/16] u8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.shape[-1]
    if n % 16:
        raise ValueError("row length must be a multiple of 16")
    flat = x.reshape(-1, n)
    codes = np.zeros((flat.shape[0], n // 2), np.uint8)
    scales = np.zeros((flat.shape[0], n // 16), np.uint8)
    lib = _load()
    u8p = ctypes.POINTER(ctypes.c_uint8)
    fp = ctypes.POINTER(ctypes.c_float)
    for i in range(flat.shape[0]):
        lib.oracle_nvfp4_quantize_row(flat[i].ctypes.data_as(fp), n, codes[i].ctypes.data_as(u8p),
                                      scales[i].ctypes.data_as(u8p))
    return codes.reshape(x.shape[:-1] + (n // 2,)), scales.reshape(x.shape[:-1] + (n // 16,))


def kv_insert(slot_mapping, k, v, ki, caches: dict, num_pages: int) -> int:
    """Quantise T new tokens into ``caches`` (numpy u8 arrays k_data, k_scale, v_data,
    v_scale, ki_data, ki_scale, updated in place). k, v: [T][4][128] FP32 or None;
    ki: [T][128] FP32 or None. Returns the oracle status (0, or -1 for a page out of range)."""
    lib = _load()
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = sm.shape[0]
    fp = ctypes.POINTER(ctypes.c_float)
    u8p = ctypes.POINTER(ctypes.c_uint8)

    def f(a):
        if a is None:
            return None, None
        a = np.ascontiguousarray(a, dtype=np.float32)
        return a, a.ctypes.data_as(fp)

    (ka, kp), (va, vp), (ia, ip_) = f(k), f(v), f(ki)
    for name in ("k_data", "k_scale", "v_data", "v_scale", "ki_data", "ki_scale"):
        if not (caches[name].flags.c_contiguous and caches[name].dtype == np.uint8):
            raise ValueError(name + " must be a contiguous uint8 array")
    ptr = {n: caches[n].ctypes.data_as(u8p) for n in caches}
    return int(lib.oracle_kv_insert(T, num_pages, sm.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), kp, vp, ip_,
                                    ptr["k_data"], ptr["k_scale"], ptr["v_data"], ptr["v_scale"], ptr["ki_data"],
                                    ptr["ki_scale"]))
