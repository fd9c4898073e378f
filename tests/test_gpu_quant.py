"""GPU parity of the NVFP4 KV-cache insertion (msa_kv_insert_nvfp4, through the C ABI)
against the oracle: every cache byte bit-exact. Codes and scales are integer results
that both sides decide in exact arithmetic (the oracle in FP64 from the definition,
the kernel by exact FP32 comparisons), so no tolerance applies.

[vLLM-zh "QKV GEMM + norm + RoPE + KV insert fusion"]: FP32 K, V and index keys are
quantised to NVFP4 and written into their caches."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_nvfp4_gb300 import KVCache, MSAError, _lib

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

E4M3 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
E2M1_MID = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
NAMES = ("k_data", "k_scale", "v_data", "v_scale", "ki_data", "ki_scale")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _rows(rng, n):
    """n FP32 rows of 128: normal values, each 16-element group at its own scale (2^-14 .. 2^9)."""
    sig = np.exp2(rng.uniform(-14, 9, size=(n, 8, 1)))
    return (rng.standard_normal((n, 8, 16)) * sig).astype(np.float32).reshape(n, 128)


def _adversarial(rng, rows):
    """Overwrite groups of `rows` with the cases where rounding is decided by a hair:
    amax / 6 exactly at and one FP32 ulp around every E4M3 midpoint; elements exactly at
    and 1..3 ulps around t x scale for every E2M1 midpoint t and every scale; zero, tiny,
    huge and negative-zero groups."""
    g = rows.reshape(-1, 16)
    n = g.shape[0]
    idx = rng.permutation(n)
    k = 0
    for c in range(0, 126):                              # scale ties and their neighbours
        for d in (-1, 0, 1):
            a = np.float32(3.0 * (E4M3[c] + E4M3[c + 1]))
            a = np.nextafter(a, np.float32(np.inf * d)) if d else a
            grp = rng.uniform(-1, 1, 16).astype(np.float32) * a
            grp[rng.integers(16)] = a * (1 if rng.random() < 0.5 else -1)
            g[idx[k]] = grp
            k += 1
    # element ties: for every scale s, elements at t x s and 1..3 FP32 ulps either side,
    # for every E2M1 midpoint t, in groups whose first element 6 s fixes the scale at s
    offs = np.arange(-3, 4)
    for sc in range(1, 127):
        s = E4M3[sc]
        vals = []
        for t in E2M1_MID:
            base = np.float32(t * s)
            for o in offs:
                v = base
                for _ in range(abs(o)):
                    v = np.nextafter(v, np.float32(np.inf if o > 0 else -np.inf))
                vals.append(v if rng.random() < 0.5 else -v)
        vals = np.array(vals, np.float32)
        for j in range(0, len(vals), 15):
            grp = np.zeros(16, np.float32)
            grp[0] = np.float32(6.0 * s)                 # amax = 6 s exactly, so the scale is s
            chunk = vals[j:j + 15]
            grp[1:1 + len(chunk)] = chunk
            g[idx[k]] = grp
            k += 1
    g[idx[k]] = 0.0
    g[idx[k + 1]] = np.float32(1e-4) * rng.uniform(-1, 1, 16).astype(np.float32)   # scale rounds to 0
    g[idx[k + 2]] = rng.uniform(-1, 1, 16).astype(np.float32) * np.float32(1e30)   # saturating scale
    g[idx[k + 3]] = -0.0
    g[idx[k + 3], 3] = 1.5
    return g.reshape(rows.shape)


def _host_caches(P, fill=0xA5):
    return {"k_data": np.full((P, 4, 128, 64), fill, np.uint8), "k_scale": np.full((P, 4, 128, 8), fill, np.uint8),
            "v_data": np.full((P, 4, 128, 64), fill, np.uint8), "v_scale": np.full((P, 4, 128, 8), fill, np.uint8),
            "ki_data": np.full((P, 128, 64), fill, np.uint8), "ki_scale": np.full((P, 128, 8), fill, np.uint8)}


def _dev(c):
    return KVCache(*(torch.from_numpy(c[n]).cuda() for n in NAMES))


def _ws():
    return torch.zeros(256, dtype=torch.uint8, device="cuda")


def _run(P, slots, k, v, ki):
    host = _host_caches(P)
    cache = _dev(host)
    ws = _ws()
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    cache.insert(torch.from_numpy(slots).cuda(), t(k), t(v), t(ki), ws)
    torch.cuda.synchronize()
    flags = _lib.msa_get_error(ws)
    ref = _host_caches(P)
    rc = oracle.kv_insert(slots, k, v, ki, ref, P)
    return cache, ref, flags, rc


def _assert_caches_equal(cache, ref):
    for n in NAMES:
        got = getattr(cache, n).cpu().numpy()
        bad = np.argwhere(got != ref[n])
        assert bad.size == 0, f"{n}: {len(bad)} bytes differ, first at {tuple(bad[0])}: " \
                              f"got {got[tuple(bad[0])]:#x} want {ref[n][tuple(bad[0])]:#x}"


def test_insert_matches_oracle_bit_exact_with_adversarial_groups():
    rng = np.random.default_rng(101)
    P, T = 5, 400
    slots = rng.permutation(P * 128)[:T].astype(np.int64)
    slots[rng.random(T) < 0.1] = -1
    k = _adversarial(rng, _rows(rng, T * 4)).reshape(T, 4, 128)
    v = _adversarial(rng, _rows(rng, T * 4)).reshape(T, 4, 128)
    ki = _adversarial(rng, _rows(rng, T))
    cache, ref, flags, rc = _run(P, slots, k, v, ki)
    assert flags == 0 and rc == 0
    _assert_caches_equal(cache, ref)


def test_null_sources_leave_their_caches_untouched():
    rng = np.random.default_rng(5)
    P, T = 2, 37
    slots = rng.permutation(P * 128)[:T].astype(np.int64)
    k = _rows(rng, T * 4).reshape(T, 4, 128)
    cache, ref, flags, rc = _run(P, slots, k, None, None)
    assert flags == 0 and rc == 0
    _assert_caches_equal(cache, ref)
    assert np.all(ref["v_data"] == 0xA5) and np.all(ref["ki_scale"] == 0xA5)


def test_slot_on_a_missing_page_is_flagged_and_skipped():
    rng = np.random.default_rng(9)
    P, T = 2, 20
    slots = rng.permutation(P * 128)[:T].astype(np.int64)
    slots[3] = P * 128 + 4          # page P does not exist
    slots[11] = 10 ** 12            # far outside
    k = _rows(rng, T * 4).reshape(T, 4, 128)
    ki = _rows(rng, T)
    cache, ref, flags, rc = _run(P, slots, k, k, ki)
    assert flags == _lib.FLAG_BAD_SLOT and rc == -1
    _assert_caches_equal(cache, ref)
    assert _lib.msa_get_error(_ws()) == 0


def test_host_validation():
    cache = KVCache.empty(1)
    slots = torch.zeros(4, dtype=torch.int64, device="cuda")
    k = torch.zeros(4, 4, 128, device="cuda")
    with pytest.raises(MSAError):                      # workspace too small
        cache.insert(slots, k, None, None, torch.zeros(16, dtype=torch.uint8, device="cuda"))
    bad = torch.zeros(4 * 4 * 128 + 1, device="cuda")[1:].view(4, 4, 128)  # 4-byte offset: misaligned
    with pytest.raises(MSAError):
        cache.insert(slots, bad, None, None, _ws())
    cache.insert(slots[:0], k[:0], None, None, _ws())  # no tokens: nothing to do


def test_full_size_insert_sampled_against_oracle():
    """The benchmarked shape (131,072 tokens into 1,024 pages, shuffled slots), on the
    device; 256 sampled tokens' rows compared with the oracle byte for byte."""
    T, P = 131072, 1024
    g = torch.Generator(device="cuda").manual_seed(17)
    k = torch.randn(T, 4, 128, device="cuda", generator=g) * 3.0
    v = torch.randn(T, 4, 128, device="cuda", generator=g)
    ki = torch.randn(T, 128, device="cuda", generator=g) * 0.1
    slots = torch.randperm(P * 128, device="cuda", generator=g)[:T].to(torch.int64)
    cache = KVCache.empty(P)
    ws = _ws()
    cache.insert(slots, k, v, ki, ws)
    torch.cuda.synchronize()
    assert _lib.msa_get_error(ws) == 0
    rng = np.random.default_rng(3)
    pick = rng.choice(T, 256, replace=False)
    pick_t = torch.from_numpy(pick).cuda()
    sl = slots.cpu().numpy()[pick]
    pg, s = sl // 128, sl % 128
    kc, ks = oracle.nvfp4_quantize_rows(k[pick_t].cpu().numpy())
    vc, vs = oracle.nvfp4_quantize_rows(v[pick_t].cpu().numpy())
    ic, is_ = oracle.nvfp4_quantize_rows(ki[pick_t].cpu().numpy())
    pgt, st = torch.from_numpy(pg).cuda(), torch.from_numpy(s).cuda()
    assert np.array_equal(cache.k_data[pgt, :, st].cpu().numpy(), kc)
    assert np.array_equal(cache.k_scale[pgt, :, st].cpu().numpy(), ks)
    assert np.array_equal(cache.v_data[pgt, :, st].cpu().numpy(), vc)
    assert np.array_equal(cache.v_scale[pgt, :, st].cpu().numpy(), vs)
    assert np.array_equal(cache.ki_data[pgt, st].cpu().numpy(), ic)
    assert np.array_equal(cache.ki_scale[pgt, st].cpu().numpy(), is_)
