"""A host model of the threshold filter inside libmsa's top-k kernels.

The kernels select the recent block plus the 15 best others by ranking keys
(score's order-preserving integer image in the high word, the complemented block
id in the low word: higher score first, then lower id). They first find a
threshold T no larger than the 15th best key, keep the candidates with key >= T
(the survivors), and rank those; when too many survive they fall back to an exact
insertion merge over all candidates. Which ranking branch runs depends only on
how many survive, so the tests use this model on the GPU's own block scores to
state which branch each case reaches. It mirrors the candidate-to-lane layout
and the threshold rule of each kernel form; it is not used to check results
(the oracle's full sort does that).
"""
import numpy as np

L = 15  # top-k minus the recent block


def keys(scores, ids=None):
    """Ranking keys (uint64) of FP32 scores; NaN ranks below everything."""
    s = np.asarray(scores, dtype=np.float32)
    s = np.where(s == 0, np.float32(0), s)          # -0.0 ties with +0.0
    u = s.view(np.uint32).astype(np.uint64)
    hi = np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)
    hi = np.where(np.isnan(s), 0, hi).astype(np.uint64)
    if ids is None:
        ids = np.arange(len(s))
    lo = (0xFFFFFFFF - np.asarray(ids, dtype=np.uint64)) & 0xFFFFFFFF
    return (hi << np.uint64(32)) | lo


def _survivors(k, T):
    return int(np.sum(k >= T))


def direct(block_scores, nb):
    """group_topk_direct (requests of 17..1025 blocks): lane l of warp q holds
    candidates 256q + 8l .. +7; T = the largest lane maximum that at least 15 lane
    maxima reach. Returns (survivors, branch)."""
    nc = nb - 1
    k = keys(block_scores[:nc])
    lm = np.zeros(128, np.uint64)
    for q in range(4):
        for l in range(32):
            c0 = 256 * q + 8 * l
            seg = k[c0:min(c0 + 8, nc)]
            lm[32 * q + l] = seg.max() if len(seg) else 0
    T = max((m for m in lm if np.sum(lm >= m) >= L), default=np.uint64(0))
    n = _survivors(k, T)
    return n, ("insertion" if n > 32 else "rank")


def staged(block_scores, nb):
    """group_topk (scores staged in shared memory): warp q takes 16-byte chunks
    [q n4 / 4, (q + 1) n4 / 4), lane l the chunks a4 + l + 32 j; each warp publishes
    its 15 largest lane maxima; T = the largest published value that at least 15
    published values reach."""
    nc = nb - 1
    k = keys(block_scores[:nc])
    n4 = (nc + 3) // 4
    pub = []
    for q in range(4):
        a4, b4 = q * n4 // 4, (q + 1) * n4 // 4
        lm = np.zeros(32, np.uint64)
        for l in range(32):
            for c4 in range(a4 + l, b4, 32):
                seg = k[4 * c4:min(4 * c4 + 4, nc)]
                if len(seg):
                    lm[l] = max(lm[l], seg.max())
        pub.extend(sorted(lm, reverse=True)[:L])
    pub = np.array(pub, np.uint64)
    T = max((v for v in pub if np.sum(pub >= v) >= L), default=np.uint64(0))
    n = _survivors(k, T)
    return n, ("insertion" if n > 64 else "rank" if n > 32 else "sort")


def warp(block_scores, nb):
    """warp_topk (one warp; rows too long to stage, and the top-k from given token
    scores): lane l holds the candidates of 16-byte chunks l, l + 32, ...; T = the
    15th largest lane maximum."""
    nc = nb - 1
    k = keys(block_scores[:nc])
    lm = np.zeros(32, np.uint64)
    for l in range(32):
        for c4 in range(l, (nc + 3) // 4, 32):
            seg = k[4 * c4:min(4 * c4 + 4, nc)]
            if len(seg):
                lm[l] = max(lm[l], seg.max())
    T = np.sort(lm)[::-1][L - 1]
    n = _survivors(k, T)
    return n, ("insertion" if n > 48 else "rank" if n > 32 else "sort")


def kernel_form(nb, max_pages):
    """Which form the fused top-k kernel uses for a request of nb blocks in a batch
    whose block-table rows hold max_pages entries."""
    if nb <= 16:
        return "all"
    if nb - 1 <= 1024:
        return "direct"
    stride = (max_pages + 3) // 4 * 4
    return "staged" if 4 * stride * 4 <= 160 * 1024 else "warp"


def attention_splits(num_reqs, sm_count):
    """Splits per (request, group) of the attention (libmsa's launch plan): the fewest
    blocks per split, a power of two in [2, 16], that fit every (request, group) x split
    into one wave of sm_count CTAs."""
    pairs = 4 * num_reqs
    need = -(-16 * pairs // sm_count) if pairs else 16
    bps = 1
    while bps < need:
        bps *= 2
    bps = min(max(bps, 2), 16)
    return 16 // bps


def range_top15(block_scores, lo, hi):
    """The attention kernel's top-k of candidates [lo, hi) for one CTA of a cluster: 128
    threads; ranges of up to 1,024 candidates held 8 per thread (thread t: lo + 8t ..), longer
    ones strided (thread t: lo + t + 128 i); T = the largest per-thread maximum that at least
    15 per-thread maxima reach; more than 64 survivors take the exact insertion merge.
    Returns (survivors, branch)."""
    k = keys(block_scores[lo:hi], np.arange(lo, hi))
    n = hi - lo
    direct = n <= 1024
    lm = np.zeros(128, np.uint64)
    for t in range(128):
        seg = k[8 * t:8 * t + 8] if direct else k[t::128]
        lm[t] = seg.max() if len(seg) else 0
    T = max((m for m in lm if m != 0 and np.sum(lm >= m) >= L), default=np.uint64(0))
    n_surv = int(np.sum(k >= T))
    return n_surv, ("insertion" if n_surv > 64 else "rank") + ("/direct" if direct else "/strided")


def fused_branches(block_scores, nb, splits):
    """range_top15's branch on every CTA of a (request, group) cluster of `splits` CTAs."""
    nc = nb - 1
    return [range_top15(block_scores, s * nc // splits, (s + 1) * nc // splits)[1] for s in range(splits)]


def dcp_local(local_scores, nc):
    """warp_best15 of the DCP rank-local lists: four warps per group, warp q taking the
    candidates [q nc / 4, (q + 1) nc / 4) (the rank's blocks in order, recent block
    excluded), candidate c0 + i in lane i % 32; T = the 15th largest lane maximum of the
    warp. Returns the branch of each warp: "sort" (<= 32 survivors), "two_sorts" (33..64),
    "chunked" (> 64: the candidates merged 32 at a time)."""
    k = keys(local_scores[:nc])
    out = []
    for q in range(4):
        c0, c1 = q * nc // 4, (q + 1) * nc // 4
        if c1 <= c0:
            continue
        kq = k[c0:c1]
        lm = np.zeros(32, np.uint64)
        for i in range(len(kq)):
            lm[i % 32] = max(lm[i % 32], kq[i])
        T = np.sort(lm)[::-1][L - 1]
        n = int(np.sum((kq >= T) & (kq != 0)))
        out.append((n, "chunked" if n > 64 else "two_sorts" if n > 32 else "sort"))
    return out
