"""Benchmark of the MSA decode step (libmsa on GB300).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl libmsa|reference] [--workload NAME]

One step = one MSA decode pass (index scan -> block max pool -> top-16 ->
sparse attention) over a batch of synthetic inputs already resident in HBM;
the default workload is 16 requests x 131,072-token context x 8 speculative
query rows. Prints one JSON line (rank 0). Under torchrun with N>1 every rank
runs an independent replica on its own GPU (the decode of independent requests
needs no exchange); value = all ranks' query rows / the slowest rank's time.

--impl reference times the oracle (plain FP64 CPU restatement of the method) on
the host cores, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MSA decode query-rows/s at 128K ctx; achieved HBM GB/s vs ~8 TB/s roofline"
UNIT = "query-rows/s"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(kernel_tag: str, workload: str):
    """DRAM bytes per launch recorded by an ncu capture under profiles/, or None.
    The summary names the kernel source hash it was taken on; a different hash
    (the kernel changed since) gives None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "block_sparse_attention_nvfp4_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


class ClockSampler:
    """Samples SM clock and clock-event reasons of one GPU during a region
    (NVML through ctypes every few ms; nvidia-smi as a fallback). Read-only."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, uuid: str, period_s: float = 0.002):
        self.uuid, self.period = uuid, period_s
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self._stop = threading.Event()
        self._nvml = None
        self._h = None
        self._proc = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0:
                    self._nvml, self._h = nv, h
                    m = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                        self.max_mhz = int(m.value)
        except OSError:
            pass

    def _run(self):
        nv, h = self._nvml, self._h
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(int(mhz.value))
            if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(self.period)

    def __enter__(self):
        if self._nvml is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", self.uuid, "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE, text=True)
            except OSError:
                self._proc = None
        return self

    def __exit__(self, *exc):
        if self._nvml is not None:
            self._stop.set()
            self._t.join()
        elif self._proc is not None:
            self._proc.terminate()
            out = self._proc.communicate()[0]
            for line in out.splitlines():
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 3 and parts[0].isdigit():
                    self.samples.append(int(parts[0]))
                    self.max_mhz = int(parts[1])
                    self.reasons |= int(parts[2], 16)

    def summary(self):
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def spread(ms):
    """Median and spread of per-step times (ms) in microseconds."""
    a = np.sort(np.asarray(ms, dtype=np.float64)) * 1e3
    pick = lambda q: float(a[min(len(a) - 1, int(round(q * (len(a) - 1))))])  # noqa: E731
    return {"median_us": round(pick(0.5), 2), "p10_us": round(pick(0.1), 2), "p90_us": round(pick(0.9), 2),
            "min_us": round(float(a[0]), 2), "max_us": round(float(a[-1]), 2), "mean_us": round(float(a.mean()), 2)}


def reduce_over_ranks(local_seconds: float, local_units: float, dist=None):
    """Whole-job numbers: units summed over ranks, time = the slowest rank's."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return local_seconds, local_units
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def workload_config(name, spec, l2_note):
    rows = list(spec.rows)
    ctx = list(spec.context_lens)
    return {"workload": name,
            "description": f"{len(ctx)} requests, context {min(ctx)}..{max(ctx)} tokens, {min(rows)}..{max(rows)} "
                           "query rows per request (speculative rows causal among themselves); 4 KV heads x d=128, "
                           "8 FP8 query heads per KV head, 1 shared index-key head; NVFP4 K/V/index caches "
                           "(E2M1 + E4M3 scale per 16) in 128-token pages behind a shuffled block table; top-16 "
                           "blocks per group with the recent block kept",
            "requests": len(ctx), "context_tokens": max(ctx) if len(set(ctx)) == 1 else "mixed",
            "rows_per_request": rows[0] if len(set(rows)) == 1 else "mixed", "query_rows_per_step": int(sum(rows)),
            "needles_per_group": spec.needles_per_group, "seed": spec.seed, "l2": l2_note}


# ----------------------------------------------------------------------------- libmsa arm
def measure_kv_insert(l2_flush, stream, reps: int, tokens: int = 131072, pages: int = 1024):
    """The KV-insert step (msa_kv_insert_nvfp4) alone: `tokens` new tokens (a 128K-token
    prefill) quantised into `pages` pages through shuffled slots, inputs resident on the
    device (seeded normal FP32 K, V, index keys), L2 flushed before each launch. HBM-bound:
    algorithmic bytes per token = 9 rows x (512 B read + 72 B written) + the 8-byte slot."""
    import torch

    from block_sparse_attention_nvfp4_gb300 import KVCache, _lib

    g = torch.Generator(device="cuda").manual_seed(5)
    k = torch.randn(tokens, 4, 128, device="cuda", generator=g)
    v = torch.randn(tokens, 4, 128, device="cuda", generator=g)
    ki = torch.randn(tokens, 128, device="cuda", generator=g)
    slots = torch.randperm(pages * 128, device="cuda", generator=g)[:tokens].to(torch.int64)
    cache = KVCache.empty(pages)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        cache.insert(slots, k, v, ki, ws)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps):
        l2_flush()
        ev[i][0].record(stream)
        cache.insert(slots, k, v, ki, ws)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    flags = _lib.msa_get_error(ws)
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    nbytes = tokens * (9 * (512 + 72) + 8)
    peak, peak_kind = measured_peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    out = {"tokens": tokens, "rows": 9 * tokens, "us": round(us, 2), "algorithmic_bytes": nbytes,
           "achieved_gbs": round(gbs, 1), "peak_gbs": peak, "peak_source": peak_kind, "frac": round(gbs / peak, 4),
           "tokens_per_s": round(tokens / (us * 1e-6), 1), "launches": reps, "device_error_flags": flags,
           "traffic": profile_traffic("kv_insert_kernel", f"insert_{tokens}"),
           "data": "synthetic: seeded N(0,1) FP32 rows on the device, shuffled slots"}
    del k, v, ki, cache
    torch.cuda.empty_cache()
    return out


def time_calls(fn, l2_flush, stream, reps):
    """Per-call device times (ms) of fn() with the L2 flushed before each call (outside
    the events)."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps):
        l2_flush()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def measure_dcp(l2_flush, stream, reps, name="long_512k", world=4):
    """Indexer decode context parallelism emulated on one GPU: the rank-local half
    (msa_dcp_local_topk: the scan of one rank's share of the blocks and its candidate
    lists) for every rank of `world`, run one after another, and the merge of all ranks'
    lists (msa_dcp_merge_topk, all-gather layout), against the single-GPU selection of
    the same workload. Device times, L2 flushed before each call. The exchange between
    GPUs (an NCCL all-gather of the lists) is not run: one GPU."""
    import torch

    from block_sparse_attention_nvfp4_gb300 import DecodeBatch, KVCache, MSADecoder, _lib
    from block_sparse_attention_nvfp4_gb300 import synth

    wl = synth.make_workload(synth.preset(name))
    cache, batch = KVCache.from_host(wl), DecodeBatch.from_host(wl)
    dec = MSADecoder(cache, batch, sm_scale=wl.sm_scale)
    args = dec.args
    B = wl.num_reqs
    keys = [torch.zeros((4, B, 16), dtype=torch.int64, device="cuda") for _ in range(world)]
    ids = torch.full((B, 4, 16), -1, dtype=torch.int32, device="cuda")
    local_us = []
    for r in range(world):
        fn = (lambda rr: (lambda: _lib.msa_dcp_local_topk(args, rr, world, keys[rr], dec.ws)))(r)
        for _ in range(3):
            fn()
        local_us.append(spread(time_calls(fn, l2_flush, stream, reps))["mean_us"])
    all_keys = torch.stack(keys).contiguous()
    merge = lambda: _lib.msa_dcp_merge_topk(args, world, 0, 4, all_keys, ids, dec.ws)  # noqa: E731
    for _ in range(3):  # untimed first calls (module loading, first-touch costs)
        merge()
        dec.select_blocks()
    merge_us = spread(time_calls(merge, l2_flush, stream, reps))["mean_us"]
    single_us = spread(time_calls(dec.select_blocks, l2_flush, stream, reps))["mean_us"]
    torch.cuda.synchronize()
    same = bool(torch.equal(ids, dec.block_ids))
    flags = dec.errors()
    out = {"workload": name, "world": world, "rank_local_us": [round(x, 2) for x in local_us],
           "merge_us": round(merge_us, 2), "single_gpu_select_us": round(single_us, 2),
           "exchange_bytes_per_rank": 4 * B * 16 * 8, "ids_equal_single_gpu": same, "device_error_flags": flags,
           "what": "one GPU emulates the ranks one after another; the NCCL exchange is unmeasured (one GPU)"}
    del dec, cache, batch, wl
    torch.cuda.empty_cache()
    return out


def measure_preset(name, l2_flush, stream, reps, peak):
    """One workload shape's decode step, selection call and attention alone (device
    times, L2 flushed before each call, inputs resident), with its algorithmic bytes and
    the step's fraction of the measured copy rate."""
    import torch

    from block_sparse_attention_nvfp4_gb300 import DecodeBatch, KVCache, MSADecoder
    from block_sparse_attention_nvfp4_gb300 import bytes_model as bm
    from block_sparse_attention_nvfp4_gb300 import synth

    wl = synth.make_workload(synth.preset(name))
    dec = MSADecoder(KVCache.from_host(wl), DecodeBatch.from_host(wl), sm_scale=wl.sm_scale, with_lse=True)
    for _ in range(3):
        l2_flush()
        dec.decode()
    torch.cuda.synchronize()
    flags = dec.errors()
    ids = dec.block_ids.clone()
    dmsa = time_calls(dec.decode, l2_flush, stream, reps)
    smsa = time_calls(dec.select_blocks, l2_flush, stream, reps)
    amsa = time_calls(lambda: dec.sparse_attn(ids), l2_flush, stream, reps)
    rows = np.diff(wl.q_indptr)
    # groups of at most 16 query rows: the warp-MMA form of the attention, for comparison
    small = None
    if int(rows.max(initial=0)) <= 2:
        small = spread(time_calls(lambda: dec.sparse_attn_small_rows(ids), l2_flush, stream, reps))["mean_us"]
    sb = bm.step_bytes(wl.context_lens, rows, ids.cpu().numpy())
    d = spread(dmsa)
    step_s = d["mean_us"] * 1e-6
    out = {"decode": d, "select_us": spread(smsa)["mean_us"], "attention_us": spread(amsa)["mean_us"],
           "attention_small_rows_us": small,
           "query_rows": int(rows.sum()), "query_rows_per_s": round(float(rows.sum()) / step_s, 1),
           "step_bytes": sb["total"], "achieved_gbs": round(sb["total"] / step_s / 1e9, 1),
           "frac": round(sb["total"] / step_s / 1e9 / peak, 4), "reps": reps, "device_error_flags": flags}
    ib = bm.distinct_index_bytes(wl.context_lens, rows, wl.block_table)
    if ib["distinct"] < ib["logical"]:
        # pages shared by several requests: the step's bytes with each shared page's index keys
        # counted once (its K/V too are read from HBM once; the L2 serves the repeats)
        uniq = sb["total"] - ib["logical"] + ib["distinct"]
        out["shared_pages"] = {"index_bytes_logical": ib["logical"], "index_bytes_distinct": ib["distinct"],
                               "logical_pages": ib["logical_pages"], "distinct_pages": ib["distinct_pages"],
                               "step_bytes_distinct": uniq,
                               "frac_distinct": round(uniq / step_s / 1e9 / peak, 4)}
    del dec, wl
    torch.cuda.empty_cache()
    return out


def run_libmsa(args, rank, world, dist):
    import torch

    import oracle
    from block_sparse_attention_nvfp4_gb300 import DecodeBatch, KVCache, MSADecoder
    from block_sparse_attention_nvfp4_gb300 import bytes_model as bm
    from block_sparse_attention_nvfp4_gb300 import synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    spec = synth.preset(args.workload)
    wl = synth.make_workload(spec)
    cache, batch = KVCache.from_host(wl), DecodeBatch.from_host(wl)
    dec = MSADecoder(cache, batch, sm_scale=wl.sm_scale, with_lse=True)
    rows = int(wl.total_rows)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    flush_sink = torch.empty(1, dtype=torch.int64, device="cuda")

    def l2_flush():
        # write a buffer larger than L2 (129 MB), then read it back: the timed step starts
        # with none of its inputs cached and with clean lines in L2, so it does not also
        # pay for writing back the flush's own dirty lines
        flush.zero_()
        torch.sum(flush.view(torch.int64), dim=0, keepdim=True, out=flush_sink)

    for _ in range(args.warmup):
        l2_flush()
        dec.decode()
    torch.cuda.synchronize()
    assert dec.errors() == 0, "device error flags after warm-up"

    # ---- timed region: K decode steps, L2 flushed before each (flush outside the events)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    uuid = str(torch.cuda.get_device_properties(local).uuid)
    uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    sampler = ClockSampler(uuid)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with sampler:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            l2_flush()
            ev[i][0].record(stream)
            dec.decode()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dev_seconds = sum(step_ms) / 1e3
    t_max, units = reduce_over_ranks(dev_seconds, float(rows * args.steps), dist)
    value = units / t_max
    ms_per_step = statistics.mean(step_ms)
    ok_flags = dec.errors()

    # ---- the calls of the step alone, same flushing: the selection (the index-scan kernel
    # with its block max pool, then the top-k kernel it chains), the exact-score selection
    # and the sparse attention on the step's block ids
    kr = min(args.steps, 200)
    sel_ms = statistics.mean(time_calls(dec.select_blocks, l2_flush, stream, kr))
    ids_now = dec.block_ids.clone()
    selx_ms = statistics.mean(time_calls(dec.select_blocks_exact, l2_flush, stream, kr))
    dec.block_ids.copy_(ids_now)
    attn_ms = statistics.mean(time_calls(lambda: dec.sparse_attn(ids_now), l2_flush, stream, kr))

    kv_insert = measure_kv_insert(l2_flush, stream, reps=min(args.steps, 50))

    sel_bytes = bm.select_bytes(wl.context_lens, np.diff(wl.q_indptr))
    step_bytes = bm.step_bytes(wl.context_lens, np.diff(wl.q_indptr), ids_now.cpu().numpy())
    peak, peak_kind = measured_peaks()
    achieved = step_bytes["total"] / (ms_per_step * 1e-3) / 1e9
    sel_achieved = sel_bytes / (sel_ms * 1e-3) / 1e9
    traffic = [profile_traffic(k, args.workload) for k in ("select_kernel", "attn_kernel")]
    roofline = {"bound": "hbm",
                "kernel": "msa_decode = select_kernel (index scan + block max pool) -> topk_kernel -> attn_kernel, "
                          "chained by programmatic dependent launch",
                "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": (traffic[0] + traffic[1]) if None not in traffic else None,
                "algorithmic_bytes_per_launch": step_bytes["total"], "avg_launch_us": round(ms_per_step * 1e3, 2),
                "selection": {"kernel": "msa_select_blocks = select_kernel + topk_kernel (chained)",
                              "achieved": round(sel_achieved, 1), "frac": round(sel_achieved / peak, 4),
                              "traffic": traffic[0], "algorithmic_bytes_per_launch": sel_bytes,
                              "avg_launch_us": round(sel_ms * 1e3, 2)}}

    # ---- the other workload shapes (their parity is tested; here their device times)
    presets = {}
    if not args.no_presets:
        from block_sparse_attention_nvfp4_gb300 import synth as _synth
        for name in _synth.PRESETS:
            if name != args.workload:
                presets[name] = measure_preset(name, l2_flush, stream, min(args.steps, 30), peak)

    dcp = None
    if not args.no_presets and world == 1:
        dcp = measure_dcp(l2_flush, stream, min(args.steps, 30))

    # ---- end to end through the public API, every step's inputs copied in from pinned host
    # memory and its outputs copied back, inside the timed region.
    # (1) serial: MSADecoder.host_io().step() (the inputs packed into one buffer, one
    # host-to-device copy, the decode, one device-to-host copy of the packed outputs,
    # synchronize), the L2 flushed before every step outside the timed region;
    # (2) the headline: MSADecoder.host_stream(3).run(), three steps in flight (the copies of a
    # step overlap the kernels of the steps next to it; the kernels of all steps run in order on
    # one stream), timed over the whole run; no flush between steps: each step streams 171.6 MB
    # of inputs through the 129 MB L2.
    ke = min(args.steps, 50)
    io = dec.host_io()
    torch.cuda.synchronize()
    e2e_times = []
    for i in range(ke + 2):
        l2_flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        io.step()
        if i >= 2:
            e2e_times.append(time.perf_counter() - t0)
    assert torch.equal(io.outputs["block_ids"], ids_now.cpu()), "host-path ids differ from the device path's"
    serial = {"ms_per_step": round(1e3 * statistics.mean(e2e_times), 4),
              "value": round(rows * ke / sum(e2e_times), 1),
              "path": "MSADecoder.host_io().step(): 1 H2D copy, 3 kernels, 1 D2H copy, synchronize"
                      + (", replayed as one CUDA graph" if io.graph is not None else
                         f" (eager: graph capture failed: {io.graph_error})"),
              "l2": "flushed before every step, outside the timed region"}
    hs = dec.host_stream(3)
    seen = []
    touch = lambda i, out: seen.append(int(out["block_ids"][0, 0, 0]))  # noqa: E731  a host read of each result
    hs.run(2 * hs.depth, consume=touch)  # first calls: pointers marshalled, kernel attributes set
    torch.cuda.synchronize()
    seen.clear()
    t0 = time.perf_counter()
    hs.run(ke, consume=touch)
    t_pipe = time.perf_counter() - t0
    assert len(seen) == ke
    for slot in hs.slots:
        assert torch.equal(slot.outputs["block_ids"], ids_now.cpu()), "pipelined host-path ids differ"
    e2e_t, e2e_u = reduce_over_ranks(t_pipe, float(rows * ke), dist)
    e2e = {"value": round(e2e_u / e2e_t, 1), "unit": UNIT, "h2d_bytes_per_step": int(hs.h2d_bytes),
           "d2h_bytes_per_step": int(hs.d2h_bytes), "steps": ke,
           "ms_per_step": round(1e3 * t_pipe / ke, 4),
           "path": "MSADecoder.host_stream(3).run(): per step 1 H2D copy, 3 kernels, 1 D2H copy and a host read "
                   "of the result; three steps in flight (each slot its own buffers), copies on two copy streams, "
                   "the kernels of all steps on one compute stream",
           "l2": f"not flushed between steps ({step_bytes['total'] / 1e6:.1f} MB moved per step; L2 129 MB)",
           "serial": serial}

    # ---- CPU baseline: the oracle as it stands, rank 0 only, bounded sample, at all the
    # host's cores (OpenMP over requests) and at one core
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        reqs = list(range(min(wl.num_reqs, 16)))
        srows = int(sum(int(wl.q_indptr[b + 1] - wl.q_indptr[b]) for b in reqs))
        all_cores = oracle.num_threads()
        t0 = time.perf_counter()
        oracle.decode(wl, reqs)
        dt = time.perf_counter() - t0
        oracle.set_threads(1)
        one = reqs[:1]
        r1 = int(wl.q_indptr[one[0] + 1] - wl.q_indptr[one[0]])
        t1 = time.perf_counter()
        oracle.decode(wl, one)
        dt1 = time.perf_counter() - t1
        oracle.set_threads(all_cores)
        cpu = {"value": round(srows / dt, 3), "unit": UNIT, "cores": all_cores, "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"{len(reqs)} of {wl.num_reqs} requests of the same workload ({srows} query rows), "
                         f"one pass, {dt:.2f} s wall, OpenMP over requests",
               "one_core": {"value": round(r1 / dt1, 3), "unit": UNIT, "cores": 1,
                            "sample": f"1 request ({r1} query rows), {dt1:.2f} s wall"}}

    clocks = sampler.summary()
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)", "data": "synthetic",
            "config": dict(workload_config(args.workload, spec, "flushed before every timed step (512 MiB write, then read back)"),
                           l2_e2e=f"e2e: not flushed between steps ({step_bytes['total'] / 1e6:.1f} MB moved per "
                                  "step; L2 129 MB); e2e.serial: flushed before every step",
                           parallelism=f"replicas x{world}"),
            "step_time": spread(step_ms),
            "step_bytes": step_bytes, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 3 * args.steps,  # per step: index scan, top-k, sparse attention
            "kernels_us": {"decode": round(ms_per_step * 1e3, 2), "select": round(sel_ms * 1e3, 2),
                           "sparse_attention": round(attn_ms * 1e3, 2)},
            "select_exact": {"us": round(selx_ms * 1e3, 2),
                             "achieved_gbs": round(sel_bytes / (selx_ms * 1e-3) / 1e9, 1),
                             "frac": round(sel_bytes / (selx_ms * 1e-3) / 1e9 / peak, 4),
                             "traffic_scan": profile_traffic("select_kernel_exact", args.workload),
                             "what": "msa_select_blocks_exact: the same selection with exact index scores "
                                     "(FP16 tiles and MMAs), timed alone like the roofline call"},
            "kv_insert_nvfp4": kv_insert,
            "workloads": presets,
            "dcp_emulated": dcp,
            "clocks": clocks, "timed_wall_s": round(wall, 4), "device_error_flags": ok_flags,
            "impl": "libmsa"}
    return line


def run_dcp_only(args):
    """The emulated indexer-DCP timings alone (measure_dcp) for --workload at --dcp ranks."""
    import torch
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    sink = torch.empty(1, dtype=torch.int64, device="cuda")

    def l2_flush():
        flush.zero_()
        torch.sum(flush.view(torch.int64), dim=0, keepdim=True, out=sink)

    return measure_dcp(l2_flush, torch.cuda.current_stream(), max(args.steps, 1), name=args.workload,
                       world=args.dcp)


# ----------------------------------------------------------------------------- reference arm (oracle)
def run_reference(args):
    """The oracle as it stands, on the host cores (OpenMP over requests), on the same
    workload. A step is the whole batch when K + W such steps fit the time budget;
    otherwise each step is a bounded sample of it (an equal share of requests, so every
    core still has work), and the line says so."""
    import oracle
    from block_sparse_attention_nvfp4_gb300 import synth

    spec = synth.preset(args.workload)
    wl = synth.make_workload(spec)
    oracle.build()
    cores = oracle.num_threads()
    budget = 240.0
    steps_total = args.steps + args.warmup
    # probe: one pass over one request per core
    probe = list(range(min(wl.num_reqs, cores)))
    t0 = time.perf_counter()
    oracle.decode(wl, probe)
    per_wave = time.perf_counter() - t0                  # one request per core, all cores busy
    waves = math.ceil(wl.num_reqs / cores)
    if steps_total * waves * per_wave <= budget:
        per_step = list(range(wl.num_reqs))
        note = f"the whole batch per step ({wl.num_reqs} requests on {cores} threads)"
    else:
        n = max(1, min(wl.num_reqs, int(budget / (steps_total * per_wave)) * cores or 1))
        per_step = list(range(n))
        note = (f"{n} of {wl.num_reqs} requests per step (the whole batch would take "
                f"{waves * per_wave:.1f} s a step; budget {budget:.0f} s for {steps_total} steps)")
    rows_per_step = int(sum(int(wl.q_indptr[b + 1] - wl.q_indptr[b]) for b in per_step))
    for _ in range(args.warmup):
        oracle.decode(wl, per_step)
    total = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.decode(wl, per_step)
        total += time.perf_counter() - t0
    value = rows_per_step * args.steps / total
    return {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(args.workload, spec, "n/a (host)"), parallelism="host cores"),
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": min(cores, len(per_step)),
                             "cpu_model": cpu_model(), "kind": "oracle", "sample": note},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="libmsa", choices=["libmsa", "reference"])
    ap.add_argument("--workload", default="spec8_128k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-presets", action="store_true", help="skip the other workload shapes' figures")
    ap.add_argument("--dcp", type=int, default=0, metavar="WORLD",
                    help="only the emulated indexer-DCP timings of --workload at WORLD ranks (one JSON line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        tdist.init_process_group("nccl")
        dist = tdist
    if world == 1 and args.gpus != 1:
        raise SystemExit("--gpus N>1 runs under torchrun (one process per GPU)")
    import __graft_entry__
    __graft_entry__.build()
    if args.dcp:
        if rank == 0:
            print(json.dumps(run_dcp_only(args)), flush=True)
        return
    line = run_libmsa(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
