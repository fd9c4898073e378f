"""A host model of the threshold filter inside libmsa's top-k kernels.

The kernels select the recent block plus the 15 best others by ranking keys
(score's order-preserving integer image in the high word, the complemented block
id in the low word: higher score first, then lower id). Each warp ranks a range of
candidates: it finds a threshold T no larger than the range's 15th best key (the
15th largest of its lanes' maxima), keeps the candidates with key >= T (the
survivors) and sorts those, or, when more than 64 survive, merges every candidate
>= T into a running top 32. Which branch runs depends only on how many survive and
on the range's length, so the tests use this model on the GPU's own block scores to
state which branch each case reaches. It mirrors the candidate-to-lane layout and
the threshold rule of each kernel form; it is not used to check results (the
oracle's full sort does that).
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


def warp_best15(k):
    """warp_best15 over one warp's candidates (keys in candidate order; candidate i in lane
    i % 32): T = the 15th largest lane maximum; the candidates >= T survive. Returns
    (survivors, branch): "sort" (<= 32), "two_sorts" (33..64), "chunked" (> 64, merged 32 at
    a time), with "/regs" when the warp holds at most 256 candidates (read once into
    registers) and "/stream" otherwise (read twice)."""
    lm = np.zeros(32, np.uint64)
    for i in range(len(k)):
        lm[i % 32] = max(lm[i % 32], k[i])
    T = np.sort(lm)[::-1][L - 1]
    n = int(np.sum((k >= T) & (k != 0)))
    br = "chunked" if n > 64 else "two_sorts" if n > 32 else "sort"
    return n, br + ("/regs" if len(k) <= 256 else "/stream")


def quad(scores, lo, hi, ids=None):
    """quad_best15 over candidates lo .. hi-1 (four warps, warp q taking
    [lo + q n / 4, lo + (q + 1) n / 4), n = hi - lo): the (survivors, branch) of every warp
    with candidates. ids: the candidates' block ids (default: their index)."""
    if ids is None:
        ids = np.arange(len(scores))
    k = keys(np.asarray(scores)[lo:hi], np.asarray(ids)[lo:hi])
    n = hi - lo
    out = []
    for q in range(4):
        a, b = q * n // 4, (q + 1) * n // 4
        if b > a:
            out.append(warp_best15(k[a:b]))
    return out


def direct(block_scores, nb):
    """group_topk_direct (requests of 17..1025 blocks): lane l of warp q holds candidates
    256q + 8l .. +7; T = the largest lane maximum that at least 15 lane maxima reach.
    Returns (survivors, branch): "rank" (<= 32, ranked by counting) or "insertion" (the
    exact insertion merge)."""
    nc = nb - 1
    k = keys(block_scores[:nc])
    lm = np.zeros(128, np.uint64)
    for q in range(4):
        for l in range(32):
            c0 = 256 * q + 8 * l
            seg = k[c0:min(c0 + 8, nc)]
            lm[32 * q + l] = seg.max() if len(seg) else 0
    T = max((m for m in lm if np.sum(lm >= m) >= L), default=np.uint64(0))
    n = int(np.sum(k >= T))
    return n, ("insertion" if n > 32 else "rank")


def topk_kernel(block_scores, nb):
    """The top-k kernel (and the selection call): the (survivors, branch) list of the direct
    form for up to 1,024 candidates (branch prefixed "direct/"), else of quad over the
    nb - 1 candidates."""
    if nb - 1 <= 1024:
        n, br = direct(block_scores, nb)
        return [(n, "direct/" + br)]
    return quad(block_scores, 0, nb - 1)


def warp(block_scores, nb):
    """warp_topk (one warp: the top-k from given token scores): lane l holds the
    candidates of 16-byte chunks l, l + 32, ...; T = the 15th largest lane maximum.
    Returns (survivors, branch)."""
    nc = nb - 1
    k = keys(block_scores[:nc])
    lm = np.zeros(32, np.uint64)
    for l in range(32):
        for c4 in range(l, (nc + 3) // 4, 32):
            seg = k[4 * c4:min(4 * c4 + 4, nc)]
            if len(seg):
                lm[l] = max(lm[l], seg.max())
    T = np.sort(lm)[::-1][L - 1]
    n = int(np.sum(k >= T))
    return n, ("insertion" if n > 48 else "rank" if n > 32 else "sort")


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


def fused_branches(block_scores, nb, splits):
    """The attention kernel's fused top-k: CTA s of a (request, group) cluster of `splits`
    CTAs runs quad over candidates [s nc / splits, (s + 1) nc / splits); the branches of all
    warps of all CTAs."""
    nc = nb - 1
    return [br for s in range(splits) for _, br in quad(block_scores, s * nc // splits, (s + 1) * nc // splits)]


def dcp_local(local_scores, nc):
    """The DCP rank-local lists: quad over the rank's nc candidates (its blocks in order,
    recent block excluded). Returns (survivors, branch) of each warp."""
    return quad(local_scores, 0, nc)
