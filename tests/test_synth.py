"""The seeded input generator: its encoders follow the NVFP4 / E4M3 formats, it
is deterministic across thread counts, and the workload presets have the shapes
of the MSA decode workloads."""
import hashlib
import os
import subprocess
import sys

import numpy as np
import torch

import oracle
from block_sparse_attention_nvfp4_gb300 import synth
from tests import _wl


def test_e4m3_encoder_matches_torch_cast():
    rng = np.random.default_rng(1)
    x = (np.exp2(rng.uniform(-14, 9.5, 50000)) * rng.choice([-1, 1], 50000)).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(synth.e4m3_encode(x.astype(np.float64)), ref)
    assert list(synth.e4m3_encode([500.0, -1e9, np.inf])) == [0x7E, 0xFE, 0x7E]


def test_nvfp4_encoder_scale_and_codes():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(4000, 128)) * np.exp(rng.normal(size=(4000, 8))).repeat(16, axis=1)
    codes, scales = synth.nvfp4_encode_rows(x)
    e2m1 = _wl.e2m1_table()
    sval = _wl.e4m3_values()[scales.astype(np.int64)]                 # [n, 8]
    amax = np.abs(x).reshape(-1, 8, 16).max(axis=2)
    want = np.array([[oracle.e4m3_round(a / 6) for a in row] for row in amax[:200]])
    assert np.array_equal(scales[:200], want)
    c = np.stack([codes & 15, codes >> 4], axis=-1).reshape(-1, 128)
    xq = e2m1[c] * np.repeat(sval, 16, axis=1)                        # exact reconstruction
    # each element is the nearest E2M1 grid point of x/scale (saturating at 6)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    y = np.abs(x) / np.repeat(sval, 16, axis=1)
    best = grid[np.abs(y[..., None] - grid).argmin(-1)]
    assert np.allclose(np.abs(xq) / np.repeat(sval, 16, axis=1), best)


def _digest(wl):
    h = hashlib.sha256()
    for a in (wl.q, wl.q_idx, wl.k_data, wl.k_scale, wl.v_data, wl.v_scale, wl.ki_data, wl.ki_scale, wl.block_table):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def test_generation_is_deterministic_and_thread_independent():
    wl = _wl.small([3000, 5000], [2, 1], needles=3, seed=77)
    d0 = _digest(wl)
    assert _digest(_wl.small([3000, 5000], [2, 1], needles=3, seed=77)) == d0
    code = ("import sys; sys.path.insert(0, %r); from tests import _wl, test_synth as t; "
            "print(t._digest(_wl.small([3000, 5000], [2, 1], needles=3, seed=77)))") % os.path.dirname(os.path.dirname(__file__))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    assert out.stdout.strip() == d0


def test_unwritten_slots_hold_garbage_and_valid_slots_are_nvfp4():
    wl = _wl.small([200], [1], seed=3)   # page 1 has 72 valid slots
    p1 = wl.block_table[0, 1]
    # valid slots: scales are non-negative E4M3 (amax/6 >= 0)
    assert np.all(wl.ki_scale[p1, :72] < 0x80)
    # unwritten slots are arbitrary bytes (NaN scales appear somewhere in a page)
    assert np.any(wl.k_scale[p1, :, 72:] >= 0x80)


def test_needles_raise_their_block_scores():
    wl = _wl.small([4096], [1], needles=4, seed=0)
    S = oracle.block_scores(wl, 0)
    for g in range(4):
        others = [c for c in range(31) if c not in wl.needles[0][g]]
        assert min(S[g][wl.needles[0][g]]) > max(S[g][others])


def test_presets_have_the_workload_shapes():
    s = synth.preset("spec8_128k")
    assert len(s.context_lens) == 16 and set(s.context_lens) == {131072} and set(s.rows) == {8}
    s = synth.preset("batch32_64k")
    assert len(s.context_lens) == 32 and set(s.context_lens) == {65536} and set(s.rows) == {1}
    s = synth.preset("long_512k")
    assert s.context_lens == [524288] and s.rows == [4] and s.lognormal_keys and s.needles_per_group == 16
    s = synth.preset("ragged64")
    ctx = np.array(s.context_lens)
    assert len(ctx) == 64 and np.all(ctx % 128 == 0) and ctx.min() >= 2048 and ctx.max() <= 262144
    assert set(s.rows) <= {1, 2, 4, 8} and s.shared_prefix_pages == 16
    s = synth.preset("tiny_4k")
    assert s.context_lens == [4096] and s.rows == [1] and s.needles_per_group == 4
