"""Seeded synthetic MSA decode workloads.

Builds the inputs of the MSA decode path — FP8 E4M3 queries and NVFP4 paged
K/V/index-key caches behind a shuffled block table — with the shapes and value
distributions of the workloads the MSA pages describe: 128-token pages, 4 KV
heads x head dim 128, 8 query heads per KV head, one shared index-key head,
speculative decode rows, contexts up to 512K tokens. Values are N(0,1) from a
counter-based generator (``synth.c``) so a workload is a pure function of its
spec and seed, identical on every machine and thread count. This module holds
no arithmetic of the path itself; it is shared by the tests, the CUDA path's
benchmark and the oracle checks purely as an input source.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libmsa_synth.so")
_lock = threading.Lock()
_lib = None

G = 4          # KV heads = GQA groups
HQ = 32        # query heads
D = 128        # head dim
BLOCK = 128    # tokens per KV block / page
TOP_K = 16     # blocks kept per group

# generator streams
_S_Q, _S_QIDX, _S_K, _S_V, _S_KI = 1, 2, 10, 20, 30


def build(force: bool = False) -> str:
    """Compile libmsa_synth.so next to its source (host C, OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u8p = ctypes.POINTER(ctypes.c_uint8)
            lib.synth_normal.restype = ctypes.c_double
            lib.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_normal_e4m3.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, u8p]
            lib.synth_e4m3_decode.argtypes = [u8p, ctypes.c_int64, ctypes.POINTER(ctypes.c_double)]
            lib.synth_e4m3_encode.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.c_int64, u8p]
            lib.synth_nvfp4_encode_rows.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.c_int64, u8p, u8p]
            lib.synth_fill_pages.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_int32), ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double),
                                             u8p, u8p]
            lib.synth_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 (ties to even, saturating at +-448) of float values."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint8)
    _load().synth_e4m3_encode(_ptr(x, ctypes.c_double), x.size, _ptr(out, ctypes.c_uint8))
    return out


def e4m3_decode(b) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint8))
    out = np.empty(b.shape, dtype=np.float64)
    _load().synth_e4m3_decode(_ptr(b, ctypes.c_uint8), b.size, _ptr(out, ctypes.c_double))
    return out


def nvfp4_encode_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4-encode rows of 128 values: (codes [n,64], scales [n,8])."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(-1, 128))
    codes = np.empty((x.shape[0], 64), np.uint8)
    scales = np.empty((x.shape[0], 8), np.uint8)
    _load().synth_nvfp4_encode_rows(_ptr(x, ctypes.c_double), x.shape[0], _ptr(codes, ctypes.c_uint8),
                                    _ptr(scales, ctypes.c_uint8))
    return codes, scales


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    lib = _load()
    return np.array([lib.synth_normal(seed, stream, i) for i in range(n)])


@dataclasses.dataclass
class Spec:
    """What a workload is: per-request context lengths and query rows, plus the
    value structure (needle blocks per group, log-normal key-group scales,
    shared prefix pages)."""
    name: str
    context_lens: Sequence[int]
    rows: Sequence[int]
    needles_per_group: int = 0
    lognormal_keys: bool = False
    shared_prefix_pages: int = 0
    seed: int = 0
    max_pages_per_req: Optional[int] = None


@dataclasses.dataclass
class Workload:
    spec: Spec
    num_reqs: int
    num_pages: int
    max_pages_per_req: int
    total_rows: int
    context_lens: np.ndarray     # int32 [B]
    q_indptr: np.ndarray         # int32 [B+1]
    block_table: np.ndarray      # int32 [B, max_pages_per_req]
    q: np.ndarray                # uint8 E4M3 [rows, 32, 128]
    q_idx: np.ndarray            # uint8 E4M3 [rows, 4, 128]
    k_data: np.ndarray           # uint8 [P, 4, 128, 64]
    k_scale: np.ndarray          # uint8 [P, 4, 128, 8]
    v_data: np.ndarray
    v_scale: np.ndarray
    ki_data: np.ndarray          # uint8 [P, 128, 64]
    ki_scale: np.ndarray         # uint8 [P, 128, 8]
    needles: list                # needles[b][g] = sorted logical block ids
    sm_scale: float = 1.0 / math.sqrt(D)
    top_k: int = TOP_K

    @property
    def nbytes_caches(self) -> int:
        return sum(a.nbytes for a in (self.k_data, self.k_scale, self.v_data, self.v_scale, self.ki_data, self.ki_scale))


def make_workload(spec: Spec) -> Workload:
    """Generate the workload described by ``spec`` (see the module docstring)."""
    lib = _load()
    rng = np.random.default_rng(spec.seed)
    ctx = np.asarray(spec.context_lens, dtype=np.int64)
    rows = np.asarray(spec.rows, dtype=np.int64)
    B = len(ctx)
    assert len(rows) == B
    assert np.all(rows >= 0) and np.all(rows <= ctx), "each request's rows must lie within its context"
    nb = (ctx + BLOCK - 1) // BLOCK
    shared = spec.shared_prefix_pages
    if shared:
        assert np.all(nb >= shared), "a shared prefix needs every request to cover it"
    max_pages = int(spec.max_pages_per_req or max(1, int(nb.max(initial=1))))
    assert max_pages >= int(nb.max(initial=0))
    # physical pages: `shared` pages used by every request, then each request's own
    num_pages = int(shared + (nb - shared).sum()) if B else 0
    num_pages = max(num_pages, 1)
    perm = rng.permutation(num_pages).astype(np.int32)
    block_table = np.zeros((B, max_pages), dtype=np.int32)
    owner_valid = np.zeros(num_pages, dtype=np.int32)   # valid slots per physical page
    nxt = shared
    for b in range(B):
        for c in range(int(nb[b])):
            if c < shared:
                phys = perm[c]
            else:
                phys = perm[nxt]
                nxt += 1
            block_table[b, c] = phys
            owner_valid[phys] = min(BLOCK, int(ctx[b]) - c * BLOCK)
    q_indptr = np.zeros(B + 1, dtype=np.int32)
    q_indptr[1:] = np.cumsum(rows)
    total_rows = int(q_indptr[-1])

    q = np.empty((total_rows, HQ, D), np.uint8)
    q_idx = np.empty((total_rows, G, D), np.uint8)
    lib.synth_normal_e4m3(spec.seed, _S_Q, q.size, _ptr(q, ctypes.c_uint8))
    lib.synth_normal_e4m3(spec.seed, _S_QIDX, q_idx.size, _ptr(q_idx, ctypes.c_uint8))

    # needles: +0.5 * q_idx[first row of the request][g] on every index key of the block
    needles = [[[] for _ in range(G)] for _ in range(B)]
    add_index = np.full(num_pages, -1, dtype=np.int32)
    add_vecs = []
    if spec.needles_per_group:
        qi_val = e4m3_decode(q_idx)
        for b in range(B):
            cand = int(nb[b]) - 1          # the most recent block is kept anyway
            if cand <= 0 or rows[b] == 0:
                continue
            for g in range(G):
                picks = np.sort(rng.choice(cand, size=min(spec.needles_per_group, cand), replace=False))
                needles[b][g] = [int(c) for c in picks]
                for c in picks:
                    phys = int(block_table[b, c])
                    if add_index[phys] < 0:
                        add_index[phys] = len(add_vecs)
                        add_vecs.append(np.zeros(D))
                    add_vecs[add_index[phys]] += 0.5 * qi_val[q_indptr[b], g]
    add_arr = np.ascontiguousarray(np.array(add_vecs if add_vecs else np.zeros((1, D)), dtype=np.float64))

    P = num_pages
    k_data = np.empty((P, G, BLOCK, 64), np.uint8)
    k_scale = np.empty((P, G, BLOCK, 8), np.uint8)
    v_data = np.empty((P, G, BLOCK, 64), np.uint8)
    v_scale = np.empty((P, G, BLOCK, 8), np.uint8)
    ki_data = np.empty((P, BLOCK, 64), np.uint8)
    ki_scale = np.empty((P, BLOCK, 8), np.uint8)
    valid_p = _ptr(owner_valid, ctypes.c_int32)
    lib.synth_fill_pages(spec.seed, _S_K, P, G, valid_p, int(spec.lognormal_keys), None, None,
                         _ptr(k_data, ctypes.c_uint8), _ptr(k_scale, ctypes.c_uint8))
    lib.synth_fill_pages(spec.seed, _S_V, P, G, valid_p, 0, None, None,
                         _ptr(v_data, ctypes.c_uint8), _ptr(v_scale, ctypes.c_uint8))
    lib.synth_fill_pages(spec.seed, _S_KI, P, 1, valid_p, int(spec.lognormal_keys),
                         _ptr(add_index, ctypes.c_int32), _ptr(add_arr, ctypes.c_double),
                         _ptr(ki_data, ctypes.c_uint8), _ptr(ki_scale, ctypes.c_uint8))
    return Workload(spec=spec, num_reqs=B, num_pages=P, max_pages_per_req=max_pages, total_rows=total_rows,
                    context_lens=ctx.astype(np.int32), q_indptr=q_indptr, block_table=block_table,
                    q=q, q_idx=q_idx, k_data=k_data, k_scale=k_scale, v_data=v_data, v_scale=v_scale,
                    ki_data=ki_data, ki_scale=ki_scale, needles=needles)


def ragged_serving_lengths(seed: int, n: int = 64, lo: int = 2048, hi: int = 262144):
    """Context lengths log-uniform in [lo, hi] rounded to the nearest multiple of
    128 (clamped), and query rows uniform in {1, 2, 4, 8}."""
    rng = np.random.default_rng(seed + 1000)
    raw = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    ctx = np.clip(np.rint(raw / BLOCK) * BLOCK, lo, hi).astype(int)
    rows = rng.choice([1, 2, 4, 8], size=n)
    return [int(c) for c in ctx], [int(r) for r in rows]


def preset(name: str) -> Spec:
    """The five workload shapes of the MSA decode path, named by what they are."""
    if name == "tiny_4k":
        return Spec(name, [4096], [1], needles_per_group=4, seed=0)
    if name == "batch32_64k":
        return Spec(name, [65536] * 32, [1] * 32, needles_per_group=8, seed=1)
    if name == "spec8_128k":
        return Spec(name, [131072] * 16, [8] * 16, needles_per_group=8, seed=2)
    if name == "long_512k":
        return Spec(name, [524288], [4], needles_per_group=16, lognormal_keys=True, seed=3)
    if name == "ragged64":
        ctx, rows = ragged_serving_lengths(4)
        return Spec(name, ctx, rows, shared_prefix_pages=16, seed=4)
    raise KeyError(name)


PRESETS = ("tiny_4k", "batch32_64k", "spec8_128k", "long_512k", "ragged64")
