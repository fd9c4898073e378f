"""Test helpers: small seeded workloads and an independent numpy/torch
dequantiser (built from the published E2M1 table and torch's E4M3 cast, not
from the oracle) for brute-force checks."""
import copy
import os

import numpy as np
import torch

from block_sparse_attention_nvfp4_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(ctx, rows, needles=0, seed=11, shared=0, lognormal=False, top_k=None, max_pages=None):
    spec = synth.Spec("test", list(ctx), list(rows), needles_per_group=needles, lognormal_keys=lognormal,
                      shared_prefix_pages=shared, seed=seed, max_pages_per_req=max_pages)
    wl = synth.make_workload(spec)
    if top_k is not None:
        wl.top_k = top_k
    return wl


def e2m1_table():
    vals = {}
    for line in open(os.path.join(GOLDEN, "e2m1_values.txt")):
        line = line.split("#")[0].strip()
        if line:
            c, v = line.split()
            vals[int(c)] = float(v)
    return np.array([vals[c] for c in range(16)])


def e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def ref_dequant_table():
    prod = e4m3_values()[:, None] * e2m1_table()[None, :]
    nan = np.isnan(prod)
    t = torch.from_numpy(np.clip(np.nan_to_num(prod), -448, 448).astype(np.float32)).to(torch.float8_e4m3fn)
    t = t.to(torch.float64).numpy()
    t[nan] = np.nan
    return t


_TAB = None


def dequant(codes, scales):
    """codes [..., 64] u8, scales [..., 8] u8 -> [..., 128] float64 FP8 values."""
    global _TAB
    if _TAB is None:
        _TAB = ref_dequant_table()
    codes = np.asarray(codes)
    lo, hi = codes & 15, codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (128,))
    s = np.repeat(np.asarray(scales), 16, axis=-1)
    return _TAB[s.astype(np.int64), c.astype(np.int64)]


def dequant_exact(codes, scales):
    """Like dequant, without the E4M3 re-rounding: E2M1 value x E4M3 scale, exact in FP64."""
    codes = np.asarray(codes)
    lo, hi = codes & 15, codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (128,))
    s = np.repeat(np.asarray(scales), 16, axis=-1)
    return e2m1_table()[c.astype(np.int64)] * e4m3_values()[s.astype(np.int64)]


def geom(wl, b):
    N = int(wl.context_lens[b])
    r0 = int(wl.q_indptr[b])
    R = int(wl.q_indptr[b + 1]) - r0
    return N, R, r0


def keys_of(wl, b, which, exact=False):
    """Dequantised keys of request b in logical order: index keys [N,128] or
    K/V [N,4,128]; exact=True (index keys): without the E4M3 re-rounding."""
    N, _, _ = geom(wl, b)
    t = np.arange(N)
    phys = wl.block_table[b, t // 128]
    slot = t % 128
    if which == "ki":
        return (dequant_exact if exact else dequant)(wl.ki_data[phys, slot], wl.ki_scale[phys, slot])
    data, scale = (wl.k_data, wl.k_scale) if which == "k" else (wl.v_data, wl.v_scale)
    return dequant(data[phys, :, slot], scale[phys, :, slot])


def permuted_pages(wl, seed=5):
    """Same logical content, physical pages shuffled again."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(wl.num_pages)
    w2 = copy.copy(wl)
    for name in ("k_data", "k_scale", "v_data", "v_scale", "ki_data", "ki_scale"):
        src = getattr(wl, name)
        dst = np.empty_like(src)
        dst[perm] = src
        setattr(w2, name, dst)
    bt = wl.block_table.copy()
    nb = (wl.context_lens + 127) // 128
    for b in range(wl.num_reqs):
        bt[b, :nb[b]] = perm[wl.block_table[b, :nb[b]]]
    w2.block_table = bt
    return w2


def unshared_copy(wl):
    """Give every request private copies of pages that several requests share."""
    nb = (wl.context_lens + 127) // 128
    pages = []
    bt = np.zeros_like(wl.block_table)
    for b in range(wl.num_reqs):
        for c in range(nb[b]):
            bt[b, c] = len(pages)
            pages.append(int(wl.block_table[b, c]))
    pages = np.array(pages)
    w2 = copy.copy(wl)
    for name in ("k_data", "k_scale", "v_data", "v_scale", "ki_data", "ki_scale"):
        setattr(w2, name, np.ascontiguousarray(getattr(wl, name)[pages]))
    w2.block_table = bt
    w2.num_pages = len(pages)
    return w2
