"""Algorithmic HBM bytes of one MSA decode step (the roofline's numerator).

Per the MSA pages, decode reads the index keys of the whole context (128 B per
token per layer in FP8) and then the full K/V of the selected blocks only; with
FP8 K/V of 4 KV heads x 128 that is 1,024 B per token for dense attention, so at
long context the step moves about 12.5% of dense attention's bytes. Stored as
NVFP4 (4-bit elements + one 1-byte scale per 16) every such figure scales by
4.5/8 = 0.5625 (34,560 vs 61,440 B per token for the whole model).
"""
from __future__ import annotations

import numpy as np

HEADS, DIM, BLOCK, TOPK = 4, 128, 128, 16
NVFP4_BYTES_PER_ROW = DIM // 2 + DIM // 16        # 64 code bytes + 8 scale bytes = 72
FP8_BYTES_PER_ROW = DIM                          # 128


def index_bytes_per_token(fmt: str = "nvfp4") -> int:
    """Index-key bytes per context token (one shared head)."""
    return NVFP4_BYTES_PER_ROW if fmt == "nvfp4" else FP8_BYTES_PER_ROW


def dense_kv_bytes_per_token(fmt: str = "nvfp4") -> int:
    """K+V bytes per token over the 4 KV heads."""
    return 2 * HEADS * index_bytes_per_token(fmt)


def traffic_fraction(n_ctx: int, fmt: str = "nvfp4") -> float:
    """Sparse decode bytes / dense attention bytes for one context of n tokens
    (index scan + selected K/V vs all K/V)."""
    sel_tokens = min(n_ctx, TOPK * BLOCK)
    sparse = n_ctx * index_bytes_per_token(fmt) + sel_tokens * dense_kv_bytes_per_token(fmt)
    return sparse / (n_ctx * dense_kv_bytes_per_token(fmt))


def step_bytes(context_lens, rows, block_ids=None, with_lse=True) -> dict:
    """Algorithmic bytes of one decode step over a batch.

    index: every context token's NVFP4 index key; kv: K+V of the valid tokens of
    the selected blocks (all blocks when a request has <= 16; with block_ids
    given, exactly those); queries: FP8 q (32x128) + q_idx (4x128) per row;
    outputs: BF16 out (32x128) per row (+ FP32 lse); meta: block table entries,
    lengths and block ids."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    active = rows > 0
    nb = (ctx + BLOCK - 1) // BLOCK
    index = int((ctx * NVFP4_BYTES_PER_ROW)[active].sum())
    kv_tok = 0
    for b in np.nonzero(active)[0]:
        if block_ids is not None:
            for g in range(HEADS):
                for c in block_ids[b, g]:
                    if c >= 0:
                        kv_tok += min(BLOCK, int(ctx[b]) - int(c) * BLOCK)
        else:
            n_sel = min(int(nb[b]), TOPK)
            # the recent (last, possibly partial) block is always kept
            full = (n_sel - 1) * BLOCK + (int(ctx[b]) - (int(nb[b]) - 1) * BLOCK)
            kv_tok += HEADS * full
    kv = kv_tok * 2 * NVFP4_BYTES_PER_ROW
    R = int(rows.sum())
    queries = R * (32 * DIM + HEADS * DIM)
    outputs = R * 32 * DIM * 2 + (R * 32 * 4 if with_lse else 0)
    meta = int(nb[active].sum()) * 4 + len(ctx) * 8 + 4 + len(ctx) * HEADS * TOPK * 4
    total = index + kv + queries + outputs + meta
    return {"index": index, "kv": kv, "queries": queries, "outputs": outputs, "meta": meta, "total": total}


def distinct_index_bytes(context_lens, rows, block_table) -> dict:
    """Index-key bytes of the active requests counted per logical block (what the scan
    reads, `logical`) and per distinct physical page (`distinct`: a page that several
    requests map, e.g. a common prompt prefix, counted once, with the most tokens any of them
    uses). The difference is what reading each shared page once would save."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    bt = np.asarray(block_table)
    tokens = {}
    logical = 0
    for b in np.nonzero(rows > 0)[0]:
        n = int(ctx[b])
        for c in range((n + BLOCK - 1) // BLOCK):
            t = min(BLOCK, n - c * BLOCK)
            logical += t
            p = int(bt[b, c])
            tokens[p] = max(tokens.get(p, 0), t)
    distinct = sum(tokens.values())
    return {"logical": logical * NVFP4_BYTES_PER_ROW, "distinct": distinct * NVFP4_BYTES_PER_ROW,
            "logical_pages": int(sum((ctx[rows > 0] + BLOCK - 1) // BLOCK)), "distinct_pages": len(tokens)}


def select_bytes(context_lens, rows) -> int:
    """Bytes the fused selection kernel must move: the index scan, the index
    queries, block-table entries and the block ids it writes."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    active = rows > 0
    nb = (ctx + BLOCK - 1) // BLOCK
    return int((ctx * NVFP4_BYTES_PER_ROW)[active].sum() + rows.sum() * HEADS * DIM + nb[active].sum() * 4
               + len(ctx) * (8 + HEADS * TOPK * 4))
