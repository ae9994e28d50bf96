"""Benchmark of the paged KV cache hot path on one GB300 (or N replicas).

One step = the whole decode hot path over one batch: the slot_mapping write of the
new K/V rows (kv_cache_write) followed by paged decode attention (split-KV
attention + LSE merge). Inputs are synthetic (synth/), resident in HBM; the KV
cache of the default workload (4.3 GB) is far larger than the 129 MB L2, so no L2
flush is needed between steps. Caches under 4x L2 (mha_tiny, swa) are flushed from
L2 before every timed step, outside the timed events (L2Flush).

Prints one JSON line (rank 0). Usage:
  python bench.py [--gpus N --steps K --warmup W] [--workload gqa_long|swa|mha_tiny]
  python bench.py --impl reference ...   # the fp64 CPU oracle as the reference arm
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time

if "--impl" in sys.argv and "reference" in sys.argv or "--cpu-baseline-child" in sys.argv:
    # The oracle timing runs single-threaded; pin BLAS before numpy loads.
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "paged-KV decode attention: achieved HBM GB/s (% of peak), seq-steps/s"


# Nominal HBM3e bandwidth of one GB300. The roofline's `peak` is the measured copy
# bandwidth (MEASURED_PEAKS.json); a copy moves half its bytes each way, and a
# read-only stream such as decode runs a little faster than that, so `frac` can pass
# 1.0. The fraction of this nominal figure is reported beside it.
NOMINAL_HBM_GBS = 7900.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def hbm_roofline(achieved: float, traffic, kernel: str, leg: dict) -> dict:
    """The HBM roofline object: achieved GB/s against the measured copy peak, and
    against the nominal bandwidth."""
    hbm, _, peak_kind = peaks()
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": traffic, "peak_kind": peak_kind,
            "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS,
            "kernel": kernel, **leg}


# ---------------------------------------------------------------- byte accounting
def q_len(wl: synth.Workload) -> int:
    return wl.q_hi if wl.kind == "spec_decode" else 1


def table_window(wl: synth.Workload) -> int:
    """Window the block table is built with: a speculative step keeps the blocks
    from the first new row's window start (W + q_len - 1)."""
    return wl.window + q_len(wl) - 1 if wl.window > 0 else 0


def decode_bytes(wl: synth.Workload, d: synth.Draw, out_bytes: int = 2) -> dict:
    """Algorithmic bytes of one decode step (keys visible to some query row, read
    once per kv head; no block overread)."""
    lens = d.seq_lens.astype(np.int64)
    span = table_window(wl)
    vis = np.minimum(lens, span) if span > 0 else lens
    row = wl.num_kv_heads * wl.head_dim * 2  # bytes of one token's K (or V) row
    kv = int(vis.sum()) * row * 2
    nblk = -(-lens // wl.block_size)
    live = nblk - (np.maximum(lens - span, 0) // wl.block_size if span > 0 else 0)
    qo = wl.batch * q_len(wl) * wl.num_heads * wl.head_dim * (2 + out_bytes)
    meta = int(live.sum()) * 4 + wl.batch * 4
    attn = kv + qo + meta
    new_rows = int(d.num_new.sum())
    write = new_rows * row * 2 * 2 + new_rows * 4  # read + write K and V rows, slots
    return {"attention": attn, "write": write, "step": attn + write, "kv": kv}


def mla_bytes(wl: synth.Workload, lens: np.ndarray, num_new: np.ndarray) -> dict:
    """Algorithmic bytes of one MLA step: each latent row (nope + rope) once, q and o of
    every query row, the table; the write reads and writes each new row once."""
    lens = np.asarray(lens, dtype=np.int64)
    Q, B, H = wl.q_hi, len(lens), wl.num_heads
    row = (wl.head_dim + wl.rope_dim) * 2
    T = int(np.asarray(num_new).sum())
    attn = int(lens.sum()) * row + B * Q * H * (wl.head_dim + wl.rope_dim) * 2 \
        + B * Q * H * wl.head_dim * 2 + int((-(-lens // wl.block_size)).sum()) * 4
    write = T * row * 2 + T * 4
    return {"attention": attn, "write": write, "step": attn + write}


def fp8_decode_bytes(wl: synth.Workload, lens: np.ndarray, num_new: np.ndarray) -> dict:
    """Algorithmic bytes of one decode step over the FP8 cache: codes (1 B per element)
    and one fp32 scale per (token, kv head) row of the visible keys, K and V; q and o;
    the table; the write reads bf16 rows and writes codes + scales."""
    lens = np.asarray(lens, dtype=np.int64)
    B, hkv, dh = len(lens), wl.num_kv_heads, wl.head_dim
    vis = np.minimum(lens, wl.window) if wl.window > 0 else lens
    kv = int(vis.sum()) * hkv * (dh + 4) * 2
    nblk = -(-lens // wl.block_size)
    live = nblk - (np.maximum(lens - wl.window, 0) // wl.block_size if wl.window > 0 else 0)
    attn = kv + B * wl.num_heads * dh * 4 + int(live.sum()) * 4 + B * 4
    new_rows = int(np.asarray(num_new).sum())
    write = new_rows * hkv * (dh * 2 + dh + 4) * 2 + new_rows * 4
    return {"attention": attn, "write": write, "step": attn + write, "kv": kv}


def prefill_row_flops(wl: synth.Workload, prior: int, r: int) -> int:
    """Algorithmic flops of query row r (0-based) of a sequence with `prior` cached
    positions: q.k and p.v over its prior + r + 1 visible keys, for every head."""
    return (prior + r + 1) * wl.num_heads * 4 * wl.head_dim


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        # Samples under load: the upper half of the observed clocks (the sampler
        # also sees the ramp before and after the timed region).
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sm)}


# ---------------------------------------------------------------- roofline leg
def timed_leg(fn, stream, min_s: float = 1.0, flush=None, max_calls: int = 200000):
    """Mean CUDA-event time of one fn() call over back-to-back calls that keep the GPU
    busy for at least min_s, so that the 100 ms clock sampler sees the load.

    With `flush` (an L2Flush), L2 is flushed before every call, outside
    that call's events. Returns a dict with the mean time in ms, the number of calls
    and the clocks sampled during the leg, with time x median SM clock (kcycles)."""
    import torch

    if BARE:  # profiling runs: no long leg (every launch is slow under a profiler)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b), {"call_us": a.elapsed_time(b) * 1e3, "calls": 1, "bare": True}

    def one_pass(n, with_flush):
        if not with_flush:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(n):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / n
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for i in range(n):
            flush(i)
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(x.elapsed_time(y) for x, y in evs)

    est = max(one_pass(5, flush is not None), 1e-4)
    per_call_wall = est
    if flush is not None:
        t = time.perf_counter()
        for i in range(5):
            flush(i)
        torch.cuda.synchronize()
        per_call_wall += (time.perf_counter() - t) * 1e3 / 5
    n = int(min(max_calls, max(20, math.ceil(min_s * 1e3 / per_call_wall))))
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    ms = one_pass(n, flush is not None)
    clocks = sampler.stop()
    leg = {"call_us": ms * 1e3, "calls": n, "leg_clocks": clocks,
           "l2": "flushed before every call (" + L2Flush.WHAT + ", not timed)" if flush is not None
                 else "not flushed: inputs larger than L2"}
    if clocks.get("sm_mhz"):
        leg["kcycles_per_call"] = ms * clocks["sm_mhz"]  # ms x MHz = thousands of cycles
    return ms, leg


_PROFILER_WARM = False
# --bare: the timed steps only, one call per leg, no activity profiler, no end-to-end
# leg, no other workloads, no CPU baseline (a short run to capture under ncu).
BARE = False


def kernel_breakdown(fn, calls: int = 10) -> dict:
    """Device time of each of our kernels over `calls` calls of fn, from CUDA activity
    records (torch.profiler, no replay or serialisation). A merge kernel launches as a
    programmatic dependent of the attention kernel and may start before it ends, so
    its `tail_us` (end of the merge minus end of the kernel launched before it) is the
    time it adds to the call."""
    if BARE:
        return {}
    try:
        import torch
        from torch.profiler import ProfilerActivity, profile

        global _PROFILER_WARM
        if not _PROFILER_WARM:  # the first profiled region of a process can come back empty
            with profile(activities=[ProfilerActivity.CUDA]):
                fn()
                torch.cuda.synchronize()
            _PROFILER_WARM = True
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            for _ in range(calls):
                fn()
            torch.cuda.synchronize()
        recs = []
        for e in prof.events():
            if e.device_type == torch.autograd.DeviceType.CUDA and "pkv::" in e.name:
                short = e.name.split("pkv::", 1)[1].split("(", 1)[0].split("<", 1)[0]
                recs.append((float(e.time_range.start), float(e.time_range.end), short))
        recs.sort()
        out = {}
        prev_end = None
        for start, end, name in recs:
            r = out.setdefault(name, {"launches": 0, "us": [], "tail_us": []})
            r["launches"] += 1
            r["us"].append(end - start)
            if "merge" in name and prev_end is not None:
                r["tail_us"].append(end - prev_end)
            if "merge" not in name:
                prev_end = end
        res = {}
        for name, r in out.items():
            res[name] = {"launches_per_call": r["launches"] / calls,
                         "mean_us": statistics.mean(r["us"])}
            if r["tail_us"]:
                res[name]["tail_us"] = statistics.mean(r["tail_us"])
        return res
    except Exception as exc:  # the profiler's CUDA activity tracing may be unavailable
        return {"error": str(exc)[:200]}


# ---------------------------------------------------------------- oracle timing
def host_info() -> dict:
    """The CPU the oracle is timed on: logical cores, the cores this process may use,
    and the CPU model (lscpu, else /proc/cpuinfo)."""
    info = {"machine": platform.machine(), "nproc": os.cpu_count()}
    try:
        info["usable_cores"] = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        info["usable_cores"] = os.cpu_count()
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            fields = {}
            for line in open("/proc/cpuinfo"):
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
            model = fields.get("model name") or " ".join(
                f"{k} {fields[k]}" for k in ("cpu implementer", "cpu part") if k in fields) or None
        except OSError:
            pass
    info["cpu_model"] = model
    return info


def time_oracle_all_cores(wl, d, max_seq: int, min_s: float = 10.0, max_reps: int = 5) -> dict:
    """The same oracle step (write, then decode of every sampled sequence) with the
    decode of each sequence as one task of a process pool over all usable cores; the
    write runs in this process, as it does in the one-thread leg."""
    from oracle import paged_ref as ref
    from oracle.pool import OraclePool, default_workers, task

    sub, sd, vals = oracle_sub_instance(wl, d, max_seq)
    post_k = ref.cache_write(vals["k_cache"], vals["k_new"], vals["slots"])
    post_v = ref.cache_write(vals["v_cache"], vals["v_new"], vals["slots"])
    fn = "paged_spec_decode" if wl.kind == "spec_decode" else "paged_decode"
    order = np.argsort(-sd.seq_lens, kind="stable")  # longest first: shorter tail
    tasks = [task(fn, shared_kwargs={"k_cache": "k", "v_cache": "v"}, q=vals["q"][b:b + 1],
                  block_table=vals["table"][b:b + 1], seq_lens=sd.seq_lens[b:b + 1],
                  block_size=wl.block_size, scale=wl.scale, window=wl.window)
             for b in order]
    step_bytes = decode_bytes(sub, sd)["step"]
    workers = default_workers()
    reps, el = 0, 0.0
    with OraclePool({"k": post_k, "v": post_v}, workers) as pool:
        while True:
            t = time.perf_counter()
            ref.cache_write(vals["k_cache"], vals["k_new"], vals["slots"])
            ref.cache_write(vals["v_cache"], vals["v_new"], vals["slots"])
            pool.map(tasks)
            el += time.perf_counter() - t
            reps += 1
            if el >= min_s or reps >= max_reps:
                break
    return {"value": step_bytes * reps / el / 1e9, "unit": "GB/s", "cores": workers,
            "kind": "oracle", "seq_steps_per_s": max_seq * reps / el,
            "sample": f"{max_seq} of {wl.batch} sequences x {reps} passes (write in one "
                      f"process, decode of each sequence a task of a {workers}-process pool, "
                      f"fp64, one BLAS thread each), {el:.1f} s"}


def oracle_sample_step(wl, d, vals, seqs):
    """One oracle pass (write + decode) over the sequences `seqs` of a sub-instance."""
    from oracle import paged_ref as ref

    post_k = ref.cache_write(vals["k_cache"], vals["k_new"], vals["slots"])
    post_v = ref.cache_write(vals["v_cache"], vals["v_new"], vals["slots"])
    fn = ref.paged_spec_decode if wl.kind == "spec_decode" else ref.paged_decode
    fn(vals["q"], post_k, post_v, vals["table"], d.seq_lens, wl.block_size, wl.scale, wl.window,
       batch_indices=seqs)


def oracle_sub_instance(wl: synth.Workload, d: synth.Draw, nseq: int):
    """The first nseq sequences of the workload as a self-contained CPU instance."""
    from oracle import block_pool_ref as bp

    sub = wl.scaled(batch=nseq)
    lens = d.seq_lens[:nseq]
    sd = synth.draw_explicit(sub, lens, d.num_new[:nseq]) if wl.layout == "pool" else synth.Draw(
        lens, d.num_new[:nseq], d.start_pos[:nseq], None, nseq * d.max_blocks_per_seq,
        d.max_blocks_per_seq)
    v = synth.values(sub, sd, "cpu")
    if wl.layout == "pool":
        table = bp.prepare_block_tables(bp.BlockPool(sd.num_blocks, sd.pool_order), lens,
                                        wl.block_size, table_window(wl), sd.max_blocks_per_seq)
    else:
        table = bp.block_table_arange(nseq, d.max_blocks_per_seq)
    slots = bp.slot_mapping(table, sd.start_pos, sd.num_new, wl.block_size)
    vals = {"k_cache": synth.bf16_bits(v["k_cache"]), "v_cache": synth.bf16_bits(v["v_cache"]),
            "k_new": synth.bf16_bits(v["k_new"]), "v_new": synth.bf16_bits(v["v_new"]),
            "q": v["q"].double().numpy(), "table": table, "slots": slots}
    return sub, sd, vals


def time_oracle(wl, d, budget_s: float, max_seq: int, min_s: float = 10.0, max_reps: int = 20):
    """Time oracle steps over a sub-batch of at most max_seq sequences (about budget_s
    per pass), repeating the pass until at least min_s of work has been timed."""
    sub, sd, vals = oracle_sub_instance(wl, d, max_seq)
    bytes_per_seq = [decode_bytes(sub.scaled(batch=1), synth.Draw(
        sd.seq_lens[i:i + 1], sd.num_new[i:i + 1], sd.start_pos[i:i + 1], None, 1, 1))["step"]
        for i in range(max_seq)]
    t = time.perf_counter()
    oracle_sample_step(sub, sd, vals, [0])
    one = time.perf_counter() - t
    nseq = int(max(1, min(max_seq, budget_s / max(one, 1e-3))))
    seqs = list(range(nseq))
    reps = 0
    t = time.perf_counter()
    while True:
        oracle_sample_step(sub, sd, vals, seqs)
        reps += 1
        el = time.perf_counter() - t
        if el >= min_s or reps >= max_reps:
            break
    nbytes = sum(bytes_per_seq[:nseq]) * reps
    return {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seq_steps_per_s": nseq * reps / el,
            "sample": f"{nseq} of {wl.batch} sequences x {reps} passes (write + decode, fp64, "
                      f"1 thread), {el:.1f} s"}


# ---------------------------------------------------------------- reference arm
def _decode_leg(wl, d, budget):
    """Oracle write + decode over a bounded sample of the workload's sequences."""
    sub, sd, vals = oracle_sub_instance(wl, d, min(8, wl.batch))
    t = time.perf_counter()
    oracle_sample_step(sub, sd, vals, [0])
    one = time.perf_counter() - t
    nseq = int(max(1, min(sub.batch, budget / max(one, 1e-3))))
    seqs = list(range(nseq))
    step_bytes = decode_bytes(sub.scaled(batch=nseq), synth.Draw(
        sd.seq_lens[:nseq], sd.num_new[:nseq], sd.start_pos[:nseq], None, 1, 1))["step"]
    return (METRIC, "GB/s", 1e9, lambda: oracle_sample_step(sub, sd, vals, seqs), step_bytes,
            f"{nseq} of {wl.batch} sequences per step")


def _mla_leg(wl, d, budget):
    """Oracle latent-row write + MLA decode (one or q_len rows per sequence) over a
    bounded sample of the workload's sequences."""
    from oracle import block_pool_ref as bp
    from oracle import paged_ref as ref

    nmax = min(8, wl.batch)
    sub = wl.scaled(batch=nmax)
    lens = d.seq_lens[:nmax]
    sd = synth.draw_explicit(sub, lens, d.num_new[:nmax])
    v = synth.values(sub, sd, "cpu")
    table = bp.prepare_block_tables(bp.BlockPool(sd.num_blocks, sd.pool_order), lens,
                                    wl.block_size, 0, sd.max_blocks_per_seq)
    slots = bp.slot_mapping(table, sd.start_pos, sd.num_new, wl.block_size)
    bits = {k: synth.bf16_bits(v[k]) for k in ("cache_nope", "cache_rope", "nope_new", "rope_new")}
    qn, qr = v["q_nope"].double().numpy(), v["q_rope"].double().numpy()
    fn = ref.mla_spec_decode if wl.q_hi > 1 else ref.mla_decode

    def step(seqs):
        rows = int(sd.num_new[:len(seqs)].sum())  # the sampled sequences' new rows
        pn = ref.cache_write(bits["cache_nope"], bits["nope_new"][:rows], slots[:rows])
        pr = ref.cache_write(bits["cache_rope"], bits["rope_new"][:rows], slots[:rows])
        fn(qn, qr, pn, pr, table, sd.seq_lens, wl.block_size, wl.scale, batch_indices=seqs)

    t = time.perf_counter()
    step([0])
    one = time.perf_counter() - t
    nseq = int(max(1, min(nmax, budget / max(one, 1e-3))))
    seqs = list(range(nseq))
    step_bytes = mla_bytes(wl, sd.seq_lens[:nseq], sd.num_new[:nseq])["step"]
    return ("MLA absorbed paged decode: achieved HBM GB/s and TFLOP/s", "GB/s", 1e9,
            lambda: step(seqs), step_bytes, f"{nseq} of {wl.batch} sequences per step")


def _prefill_leg(wl, d, budget):
    """Oracle K/V write + causal prefill of a bounded sample of query rows, spread over
    the first sequences of the workload (decode rows and prefill rows alike)."""
    from oracle import block_pool_ref as bp
    from oracle import paged_ref as ref

    nmax = min(6, wl.batch)  # sequences 0-3 are decode rows, 4-5 prefill rows
    sub = wl.scaled(batch=nmax)
    lens = d.seq_lens[:nmax]
    sd = synth.draw_explicit(sub, lens, d.num_new[:nmax])
    v = synth.values(sub, sd, "cpu")
    table = bp.prepare_block_tables(bp.BlockPool(sd.num_blocks, sd.pool_order), lens,
                                    wl.block_size, 0, sd.max_blocks_per_seq)
    slots = bp.slot_mapping(table, sd.start_pos, sd.num_new, wl.block_size)
    bits = {k: synth.bf16_bits(v[k]) for k in ("k_cache", "v_cache", "k_new", "v_new")}
    q = v["q"].double().numpy()
    cu = np.cumsum(sd.num_new).astype(np.int64)
    T = int(cu[-1])
    seq_of_row = np.searchsorted(cu, np.arange(T), side="right")
    prior = (sd.seq_lens - sd.num_new).astype(np.int64)
    starts = cu - sd.num_new

    def flops(rows):
        return sum(prefill_row_flops(wl, int(prior[seq_of_row[r]]), int(r - starts[seq_of_row[r]]))
                   for r in rows)

    def step(rows):
        pk = ref.cache_write(bits["k_cache"], bits["k_new"], slots)
        pv = ref.cache_write(bits["v_cache"], bits["v_new"], slots)
        ref.paged_prefill(q, cu, pk, pv, table, sd.seq_lens, wl.block_size, wl.scale, True, rows=rows)

    probe = [T - 1]
    t = time.perf_counter()
    step(probe)
    one = time.perf_counter() - t
    n = int(max(1, min(T, budget / max(one, 1e-3))))
    rows = sorted(set(np.linspace(0, T - 1, n).round().astype(int).tolist()))
    return ("causal paged prefill (mixed with decode rows): achieved TFLOP/s", "TFLOP/s", 1e12,
            lambda: step(rows), flops(rows),
            f"{len(rows)} of {T} query rows of the first {nmax} sequences per step")


def _fp8_leg(wl, d, budget):
    """Oracle quantising write of the new rows + dequantisation + decode over a bounded
    sample of the workload's sequences (the cache is quantised once beforehand)."""
    from oracle import fp8_ref
    from oracle import paged_ref as ref

    # At most two sequences: the oracle quantises and dequantises whole caches in fp64.
    sub, sd, vals = oracle_sub_instance(wl, d, min(2, wl.batch))
    nb, bs, hkv, dh = vals["k_cache"].shape
    every = np.arange(nb * bs)
    zc, zs = np.zeros((nb, bs, hkv, dh), np.uint8), np.zeros((nb, hkv, bs), np.float32)
    kc, ks = fp8_ref.cache_write_fp8(zc, zs, vals["k_cache"].reshape(nb * bs, hkv, dh), every)
    vc, vs = fp8_ref.cache_write_fp8(zc, zs, vals["v_cache"].reshape(nb * bs, hkv, dh), every)

    def step(seqs):
        k2, ks2 = fp8_ref.cache_write_fp8(kc, ks, vals["k_new"], vals["slots"])
        v2, vs2 = fp8_ref.cache_write_fp8(vc, vs, vals["v_new"], vals["slots"])
        ref.paged_decode(vals["q"], fp8_ref.dequantize_cache(k2, ks2), fp8_ref.dequantize_cache(v2, vs2),
                         vals["table"], sd.seq_lens, wl.block_size, wl.scale, wl.window,
                         batch_indices=seqs)

    t = time.perf_counter()
    step([0])
    one = time.perf_counter() - t
    nseq = int(max(1, min(sub.batch, budget / max(one, 1e-3))))
    seqs = list(range(nseq))
    step_bytes = fp8_decode_bytes(wl, sd.seq_lens[:nseq], sd.num_new[:nseq])["step"]
    return ("paged decode over an FP8 E4M3 cache: achieved HBM GB/s", "GB/s", 1e9,
            lambda: step(seqs), step_bytes, f"{nseq} of {wl.batch} sequences per step")


def _sized(total: int, budget: float, one_pass) -> int:
    """Rows of a bounded sample: all of them if one pass fits the budget, else a
    proportional share (at least 4096)."""
    t = time.perf_counter()
    one_pass(total)
    one = time.perf_counter() - t
    return total if one <= budget else max(min(total, 4096), int(total * budget / one))


def _scatter_leg(args, budget):
    """Oracle row copy through slot_mapping of K and V rows (the scatter workload)."""
    import torch

    from oracle import paged_ref as ref

    rows, hkv, d, bs = args.batch or 262144, 8, 128, 128
    nb = rows // bs
    g = torch.Generator()
    g.manual_seed(1005)
    k = synth.bf16_bits(torch.randn((rows, hkv, d), generator=g).to(torch.bfloat16))
    v = synth.bf16_bits(torch.randn((rows, hkv, d), generator=g).to(torch.bfloat16))
    kc = np.zeros((nb, bs, hkv, d), dtype=np.uint16)
    vc = np.zeros_like(kc)
    perm = np.random.default_rng(1005).permutation(nb * bs).astype(np.int32)

    def step(n):
        ref.cache_write(kc, k[:n], perm[:n])
        ref.cache_write(vc, v[:n], perm[:n])

    n = _sized(rows, budget, step)
    return ("kv_cache_write scatter: achieved HBM GB/s", "GB/s", 1e9, lambda: step(n),
            n * hkv * d * 2 * 2 * 2 + n * 4, f"{n} of {rows} rows per step")


def _mla_write_leg(args, budget):
    """Oracle RMSNorm + RoPE + write of latent rows (the mla_write workload)."""
    from oracle import mla_write_ref as mref

    T = args.batch or 262144
    nb = -(-T // 128) + 8
    v = synth.draw_mla_write(T, nb, 1007, device="cpu")
    bits = {k: synth.bf16_bits(v[k]) for k in ("cache_nope", "cache_rope", "latent", "gamma")}
    cos, sin = v["cos"].double().numpy(), v["sin"].double().numpy()
    slots = v["slots"].numpy()

    def step(n):
        mref.mla_rmsnorm_rope_write(bits["cache_nope"], bits["cache_rope"], bits["latent"][:n],
                                    bits["gamma"], cos[:n], sin[:n], slots[:n], 512, 1e-6)

    n = _sized(T, budget, step)
    return ("fused MLA RMSNorm+RoPE cache write: achieved HBM GB/s", "GB/s", 1e9,
            lambda: step(n), n * (1152 + 512 + 1152 + 4), f"{n} of {T} tokens per step")


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    extra = {"scatter": _scatter_leg, "mla_write": _mla_write_leg}
    if args.workload in extra and args.kv_dtype == "bf16":
        per_step_budget = max(0.05, args.ref_budget_s / max(1, args.steps + args.warmup))
        return _report_reference(args, args.workload, args.batch or 262144,
                                 *extra[args.workload](args, per_step_budget))
    if args.kv_dtype == "fp8" and args.workload in ("gqa_long", "swa"):
        wl = synth.WORKLOADS[args.workload]
        per_step_budget = max(0.05, args.ref_budget_s / max(1, args.steps + args.warmup))
        return _report_reference(args, wl.name, wl.batch, *_fp8_leg(wl, synth.draw(wl), per_step_budget))
    if args.workload not in synth.WORKLOADS or args.kv_dtype != "bf16":
        what = args.workload + ("" if args.kv_dtype == "bf16" else f" over an {args.kv_dtype} cache")
        print(json.dumps({"impl": "reference", "unavailable":
                          f"no oracle timing leg for the {what} workload; its oracle functions "
                          "are exercised by the tests"}), flush=True)
        return
    wl = synth.WORKLOADS[args.workload]
    d = synth.draw(wl)
    per_step_budget = max(0.05, args.ref_budget_s / max(1, args.steps + args.warmup))
    leg = {"mla_decode": _mla_leg, "prefill": _prefill_leg}.get(wl.kind, _decode_leg)
    _report_reference(args, wl.name, wl.batch, *leg(wl, d, per_step_budget))


def _report_reference(args, name, batch, metric, unit, scale, step, units, sample):
    """Time K oracle steps after W warm-ups and print the reference arm's line."""
    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t
    value = units * args.steps / el / scale
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "sample": sample, "batch": batch},
            "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline_child(args):
    """The oracle timed on this host: one thread over a sample of the sequences, then
    a process pool over all usable cores on (up to) every sequence of the workload."""
    wl = synth.WORKLOADS[args.workload]
    d = synth.draw(wl)
    line = time_oracle(wl, d, budget_s=15.0, max_seq=min(8, wl.batch))
    line["host"] = host_info()
    if not args.no_all_cores:
        try:
            line["all_cores"] = time_oracle_all_cores(wl, d, max_seq=min(wl.batch, 128))
        except Exception as exc:
            line["all_cores"] = {"value": None, "error": str(exc)[:300]}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks: the slowest replica sets the job's time."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step: float, world: int, ms_step: float) -> float:
    """Whole-job units per second: every replica does units_per_step per step, and a
    step takes ms_step milliseconds on the slowest replica."""
    return units_per_step * world / (ms_step * 1e-3)


# Caches below this size are L2-flushed between timed steps (4x the 129 MB L2).
class L2Flush:
    """Evicts a workload's inputs from L2 between timed calls, outside their events: a
    512 MB write (four times the 129 MB L2), then a 512 MB read of another buffer. The
    write alone would leave L2 full of dirty lines, whose write-back then competes with
    the timed kernel's reads (measured: +15 us on the swa call, +2 us on mha_tiny); the
    read writes them back first and leaves clean lines of an unrelated buffer."""

    WHAT = "512 MB write, then 512 MB read of another buffer"

    def __init__(self, dev):
        import torch
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.int64, device=dev)
        self.acc = torch.zeros((), dtype=torch.int64, device=dev)

    def __call__(self, i: int = 0):
        import torch
        self.w.fill_(i & 0xff)
        torch.sum(self.r, dim=(0,), out=self.acc)

L2_FLUSH_BELOW = 4 * 129e6


def traffic_from_profiles(kernel_key: str):
    """DRAM bytes per launch recorded from an ncu capture, if the kernel source is unchanged."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))[kernel_key]
        h = hashlib.sha256()
        for f in rec["sources"]:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if h.hexdigest() != rec["sha256"]:
            return None
        return rec["dram_bytes_per_launch"]
    except Exception:
        return None


def run_ours(args):
    import torch
    import torch.distributed as dist

    from paged_kv_cache_77_gb300 import api

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    api.set_decode_kernel({"auto": api.KERNEL_AUTO, "cuda_core": api.KERNEL_CUDA_CORE,
                           "tensor_core": api.KERNEL_TENSOR_CORE}[args.decode_kernel])
    line = run_workload(args, dev, world, rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_workload(args, dev, world: int = 1, rank: int = 0):
    """The line of one workload (every rank computes it; rank 0 prints it)."""
    if args.kv_dtype == "fp8":
        if args.workload not in ("gqa_long", "swa"):
            raise SystemExit("--kv-dtype fp8 applies to the gqa_long and swa workloads")
        return run_fp8(args, dev)
    other = {"scatter": run_scatter, "fork": run_fork, "mla_write": run_mla_write,
             "mla": run_mla, "mla_spec": run_mla, "mixed_prefill": run_prefill}
    if args.workload in other:
        return other[args.workload](args, dev)
    return run_decode(args, dev, world, rank)


# The other workloads, run briefly after the default one so that a single default run
# records every configuration: (label, workload, kv dtype).
PER_CONFIG = (("mha_tiny", "mha_tiny", "bf16"), ("swa", "swa", "bf16"),
              ("spec_decode", "spec_decode", "bf16"), ("mla", "mla", "bf16"),
              ("mla_spec", "mla_spec", "bf16"), ("mixed_prefill", "mixed_prefill", "bf16"),
              ("gqa_long_fp8", "gqa_long", "fp8"), ("scatter", "scatter", "bf16"),
              ("mla_write", "mla_write", "bf16"), ("fork", "fork", "bf16"))


def per_config(args, dev) -> dict:
    """Short runs of the other workloads (20 steps, 3 warm-ups, and a roofline leg of at
    least a second each): their metric, the call's time, the roofline fraction, the L2
    condition, the clocks and the per-kernel split."""
    import torch

    res = {}
    for label, name, kv in PER_CONFIG:
        sub = argparse.Namespace(**{**vars(args), "workload": name, "kv_dtype": kv, "batch": 0,
                                    "steps": min(args.steps, 20), "warmup": 3,
                                    "no_cpu_baseline": True, "no_per_config": True})
        try:
            line = run_workload(sub, dev)
        except Exception as exc:
            res[label] = {"error": str(exc)[:300]}
            continue
        finally:
            torch.cuda.empty_cache()
        r = line["roofline"]
        keep = ("bound", "achieved", "peak", "unit", "frac", "peak_kind", "frac_of_nominal",
                "traffic", "call_us", "calls", "l2", "kcycles_per_call", "kernels")
        res[label] = {"metric": line["metric"], "value": line["value"], "unit": line["unit"],
                      "ms_per_step": line["ms_per_step"], "config": line["config"]["workload"],
                      "roofline": {k: r[k] for k in keep if k in r},
                      "sm_mhz": (r.get("leg_clocks") or {}).get("sm_mhz"),
                      "clock_reasons": (r.get("leg_clocks") or {}).get("reasons")}
        if "tensor" in line:
            res[label]["tensor"] = line["tensor"]
    return res


def run_decode(args, dev, world: int = 1, rank: int = 0):
    import torch
    import torch.distributed as dist

    from paged_kv_cache_77_gb300 import api

    wl = synth.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.scaled(batch=args.batch)
    d = synth.draw(wl)
    v = synth.values(wl, d, dev)
    if wl.layout == "pool":
        pool = api.BlockPool(d.num_blocks, d.pool_order)
        table_np = pool.build_block_table(d.seq_lens, wl.block_size, table_window(wl),
                                          d.max_blocks_per_seq)
    else:
        table_np = api.build_block_table_arange(wl.batch, d.max_blocks_per_seq)
    slots_np = api.build_slot_mapping(table_np, d.start_pos, d.num_new, wl.block_size)
    table = torch.from_numpy(table_np).to(dev)
    slots = torch.from_numpy(slots_np).to(dev)
    seq_lens = torch.from_numpy(d.seq_lens).to(dev)
    spec = wl.kind == "spec_decode"
    out = torch.empty(tuple(v["q"].shape), dtype=torch.bfloat16, device=dev)
    if spec:
        ws = torch.empty(api.decode_spec_workspace_size(wl.batch, q_len(wl), wl.num_heads,
                                                        wl.num_kv_heads, wl.head_dim),
                         dtype=torch.uint8, device=dev)
    else:
        ws = torch.empty(api.decode_workspace_size(wl.batch, wl.num_heads, wl.num_kv_heads,
                                                   wl.head_dim), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def attend(q):
        if spec:
            api.paged_attention_decode_spec(q, v["k_cache"], v["v_cache"], table, seq_lens,
                                            wl.scale, wl.window, out=out, workspace=ws)
        else:
            api.paged_attention_decode(q, v["k_cache"], v["v_cache"], table, seq_lens, wl.scale,
                                       wl.window, out=out, workspace=ws)

    def step():
        api.kv_cache_write(v["k_cache"], v["v_cache"], v["k_new"], v["v_new"], slots)
        attend(v["q"])

    nbytes = decode_bytes(wl, d, out_bytes=2)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- device-resident timing: K steps, events around each decode call too
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # A cache smaller than 4x the 129 MB L2 would stay L2-resident from step to step:
    # then L2 is flushed before every step (outside the timed events)
    # and each step is timed by its own events.
    flush = L2Flush(dev) if nbytes["kv"] < L2_FLUSH_BELOW else None
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush(i)
        ev_step[i][0].record(stream)
        api.kv_cache_write(v["k_cache"], v["v_cache"], v["k_new"], v["v_new"], slots)
        attend(v["q"])
        ev_step[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    if flush is None:
        ms_total = t_start.elapsed_time(t_end)
    else:
        ms_total = sum(a.elapsed_time(b) for a, b in ev_step)
    ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    # The attention call's own time, for the roofline: back-to-back calls with no cache
    # write between them, for at least a second. (In the step loop the attention kernel
    # launches as a programmatic dependent of the write kernel and may start before the
    # event placed between them, so events around it there would miss part of its run.)
    dec_ms, leg = timed_leg(lambda: attend(v["q"]), stream, flush=flush)
    breakdown = kernel_breakdown(lambda: attend(v["q"]))
    l2_note = ("inputs larger than L2 (KV cache %.2f GB vs 129 MB L2)" % (nbytes["kv"] / 1e9)
               if flush is None else
               "L2 flushed before every timed step (" + L2Flush.WHAT + ", not timed); KV cache %.3f GB"
               % (nbytes["kv"] / 1e9))

    # ---- end to end through the public API with host buffers
    # The step's inputs (queries, new K/V rows, lengths, slots, block table) sit in one
    # pinned host staging buffer and cross to the device in one copy, into a device
    # buffer the calls read through views (each part starts on a 256-byte boundary);
    # the slots are rebuilt into their part every step. The output comes back in one
    # copy.
    parts = [("q", v["q"]), ("k_new", v["k_new"]), ("v_new", v["v_new"]),
             ("lens", torch.from_numpy(d.seq_lens)), ("slots", torch.from_numpy(slots_np)),
             ("table", torch.from_numpy(table_np))]
    offs, total = {}, 0
    for name, t in parts:
        offs[name] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, name, like):
        n = like.numel() * like.element_size()
        return buf[offs[name]:offs[name] + n].view(like.dtype).view(like.shape)

    for name, t in parts:
        view(stage_h, name, t).copy_(t.cpu())
    dq, dk, dv = (view(stage_d, n, v[n]) for n in ("q", "k_new", "v_new"))
    lens_d = view(stage_d, "lens", parts[3][1])
    slots_d = view(stage_d, "slots", parts[4][1])
    slots_h = view(stage_h, "slots", parts[4][1]).numpy()
    table_d = view(stage_d, "table", parts[5][1])
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for _, t in parts)
    d2h = out_host.numel() * out_host.element_size()

    def attend_e2e(q):
        if spec:
            api.paged_attention_decode_spec(q, v["k_cache"], v["v_cache"], table_d, lens_d,
                                            wl.scale, wl.window, out=out, workspace=ws)
        else:
            api.paged_attention_decode(q, v["k_cache"], v["v_cache"], table_d, lens_d, wl.scale,
                                       wl.window, out=out, workspace=ws)

    def e2e_step():
        if flush is not None:
            flush(1)
            torch.cuda.current_stream().synchronize()
        t = time.perf_counter()
        # The previous step's copy ended at its synchronize, so its part can be rewritten.
        api.build_slot_mapping(table_np, d.start_pos, d.num_new, wl.block_size, out=slots_h)
        stage_d.copy_(stage_h, non_blocking=True)
        api.kv_cache_write(v["k_cache"], v["v_cache"], dk, dv, slots_d)
        attend_e2e(dq)
        out_host.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return time.perf_counter() - t

    if BARE:
        e2e_s = float("nan")
    else:
        for _ in range(max(3, args.warmup)):
            e2e_step()
        e2e_steps = max(10, args.steps // 4)
        if world > 1:
            dist.barrier()
        e2e_s = sum(e2e_step() for _ in range(e2e_steps)) / e2e_steps
        e2e_s = max_over_ranks(e2e_s, dev)

    hbm, _, peak_kind = peaks()
    value = job_throughput(nbytes["step"], world, ms_step) / 1e9
    achieved = nbytes["attention"] / (dec_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "seq_steps_per_s": wl.batch * world / (ms_step * 1e-3),
        "pct_of_peak": value / world / hbm,
        "config": {"workload": f"{wl.name}: B={wl.batch} H={wl.num_heads} H_kv={wl.num_kv_heads} "
                               f"d={wl.head_dim} bs={wl.block_size} window={wl.window}"
                               + (f" q_len={q_len(wl)}" if spec else ""),
                   "seq_lens": f"U[{wl.len_lo},{wl.len_hi}] (sum {int(d.seq_lens.sum())})",
                   "step": "kv_cache_write + paged_attention_decode%s (attention + LSE merge)"
                           % ("_spec" if spec else ""),
                   "step_bytes": nbytes["step"],
                   "l2": l2_note,
                   "parallelism": f"replicas x{world}"},
        "roofline": {**hbm_roofline(
            achieved, traffic_from_profiles(f"decode:{wl.name}"),
            f"paged_attention_decode{'_spec' if spec else ''} (split-KV attention + merge), "
            f"{dec_ms * 1e3:.1f} us per call", leg),
            "decode_kernel": ["auto", "cuda_core", "tensor_core"][api.get_decode_kernel()],
            "kernels": breakdown},
        "e2e": {"value": nbytes["step"] * world / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_s * 1e3},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and wl.name == "gqa_long" and not args.batch \
            and not args.no_per_config:
        line["per_config"] = per_config(args, dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child",
                            "--workload", wl.name], capture_output=True, text=True,
                           env={**os.environ, "OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1",
                                "MKL_NUM_THREADS": "1", "CUDA_VISIBLE_DEVICES": ""})
        try:
            line["cpu_baseline"] = json.loads(r.stdout.strip().splitlines()[-1])
        except Exception:
            line["cpu_baseline"] = {"value": None, "error": r.stderr[-300:]}
    return line


def run_fp8(args, dev):
    """Decode step over an FP8 (E4M3) cache: quantising write of the new rows +
    paged_attention_decode_fp8. The cache is the workload's bf16 cache quantised once
    before timing. Bytes: codes (1 per element) + one fp32 scale per (token, kv
    head) row for K and V, read for the visible keys only."""
    import torch

    from paged_kv_cache_77_gb300 import api

    wl = synth.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.scaled(batch=args.batch)
    d = synth.draw(wl)
    v = synth.values(wl, d, dev)
    pool = api.BlockPool(d.num_blocks, d.pool_order)
    table_np = pool.build_block_table(d.seq_lens, wl.block_size, wl.window, d.max_blocks_per_seq)
    slots_np = api.build_slot_mapping(table_np, d.start_pos, d.num_new, wl.block_size)
    table = torch.from_numpy(table_np).to(dev)
    slots = torch.from_numpy(slots_np).to(dev)
    seq_lens = torch.from_numpy(d.seq_lens).to(dev)
    nb, bs, hkv, dh = v["k_cache"].shape
    kc = torch.empty((nb, bs, hkv, dh), dtype=torch.uint8, device=dev)
    vc = torch.empty_like(kc)
    ks = torch.empty((nb, hkv, bs), dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    every = torch.arange(nb * bs, dtype=torch.int32, device=dev)
    api.kv_cache_write_fp8(kc, vc, ks, vs, v["k_cache"].view(nb * bs, hkv, dh),
                           v["v_cache"].view(nb * bs, hkv, dh), every)
    del v["k_cache"], v["v_cache"]
    torch.cuda.synchronize()
    out = torch.empty((wl.batch, wl.num_heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(api.decode_workspace_size(wl.batch, wl.num_heads, hkv, dh), dtype=torch.uint8,
                     device=dev)
    lens = d.seq_lens.astype(np.int64)
    vis = np.minimum(lens, wl.window) if wl.window > 0 else lens
    fb = fp8_decode_bytes(wl, lens, d.num_new)
    kv, attn, write = fb["kv"], fb["attention"], fb["write"]
    bf16_kv = int(vis.sum()) * hkv * dh * 2 * 2
    stream = torch.cuda.current_stream(dev)

    def attend():
        api.paged_attention_decode_fp8(v["q"], kc, vc, ks, vs, table, seq_lens, wl.scale, wl.window,
                                       out=out, workspace=ws)

    def step():
        api.kv_cache_write_fp8(kc, vc, ks, vs, v["k_new"], v["v_new"], slots)
        attend()

    for _ in range(args.warmup):
        step()
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    # The attention call's own time: back-to-back calls for at least a second (in the
    # step loop it may start before an event placed after the write, as a programmatic
    # dependent of it).
    dec_ms, leg = timed_leg(attend, stream)
    breakdown = kernel_breakdown(attend)
    achieved = attn / (dec_ms * 1e-3) / 1e9
    return {
        "metric": "paged decode over an FP8 E4M3 cache: achieved HBM GB/s", "impl": "ours",
        "value": (attn + write) / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 cache, f16 tensor-core operands",
        "data": "synthetic", "seq_steps_per_s": wl.batch / (ms * 1e-3),
        "config": {"workload": f"{wl.name} (fp8 cache): B={wl.batch} H={wl.num_heads} "
                               f"H_kv={wl.num_kv_heads} d={wl.head_dim} window={wl.window}",
                   "kv_bytes": kv, "kv_bytes_if_bf16": bf16_kv,
                   "decode_us_per_call": dec_ms * 1e3,
                   "l2": "inputs larger than L2 (%.2f GB of codes and scales)" % (kv / 1e9)},
        "roofline": {**hbm_roofline(achieved, traffic_from_profiles(f"fp8:{wl.name}"),
                                    f"paged_attention_decode_fp8 (attention + merge), "
                                    f"{dec_ms * 1e3:.1f} us", leg), "kernels": breakdown},
        "gpu_launches": 3 * args.steps, "clocks": clocks}


def run_mla(args, dev):
    """Absorbed MLA decode step: latent row write (nope + rope) + mla_paged_decode, or
    with q_len > 1 rows per sequence (mla_spec) mla_paged_decode_spec."""
    import torch

    from paged_kv_cache_77_gb300 import api

    wl = synth.WORKLOADS[args.workload]
    Q = wl.q_hi
    if args.batch:
        wl = wl.scaled(batch=args.batch)
    d = synth.draw(wl)
    v = synth.values(wl, d, dev)
    pool = api.BlockPool(d.num_blocks, d.pool_order)
    table_np = pool.build_block_table(d.seq_lens, wl.block_size, 0, d.max_blocks_per_seq)
    slots = torch.from_numpy(api.build_slot_mapping(table_np, d.start_pos, d.num_new,
                                                    wl.block_size)).to(dev)
    table = torch.from_numpy(table_np).to(dev)
    seq_lens = torch.from_numpy(d.seq_lens).to(dev)
    rows_shape = (wl.batch, Q, wl.num_heads) if Q > 1 else (wl.batch, wl.num_heads)
    out = torch.empty(rows_shape + (wl.head_dim,), dtype=torch.bfloat16, device=dev)
    ws_bytes = (api.mla_decode_spec_workspace_size(wl.batch, Q, wl.num_heads) if Q > 1
                else api.mla_decode_workspace_size(wl.batch, wl.num_heads))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    lens = d.seq_lens.astype(np.int64)
    row = (wl.head_dim + wl.rope_dim) * 2
    mb = mla_bytes(wl, lens, d.num_new)
    attn_bytes, write_bytes = mb["attention"], mb["write"]
    # Positions seen by query row i of sequence b: len_b - Q + 1 + i (at least 0).
    seen = sum(int(np.maximum(lens - Q + 1 + i, 0).sum()) for i in range(Q))
    flops = seen * wl.num_heads * (2 * (wl.head_dim + wl.rope_dim) + 2 * wl.head_dim)

    def write():
        api.kv_cache_write(v["cache_nope"], v["cache_rope"], v["nope_new"], v["rope_new"], slots)

    def attend():
        if Q > 1:
            api.mla_paged_decode_spec(v["q_nope"], v["q_rope"], v["cache_nope"], v["cache_rope"],
                                      table, seq_lens, wl.scale, out=out, workspace=ws)
        else:
            api.mla_paged_decode(v["q_nope"], v["q_rope"], v["cache_nope"], v["cache_rope"], table,
                                 seq_lens, wl.scale, out=out, workspace=ws)

    for _ in range(args.warmup):
        write()
        attend()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        write()
        attend()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    # The attention call alone, back to back for at least a second (in the step loop it
    # launches as a programmatic dependent of the write and may start before an event
    # placed between them).
    dec_ms, leg = timed_leg(attend, stream)
    breakdown = kernel_breakdown(attend)
    hbm, tf, peak_kind = peaks()
    ach = attn_bytes / (dec_ms * 1e-3) / 1e9
    tfl = flops / (dec_ms * 1e-3) / 1e12
    return {
        "metric": "MLA absorbed paged decode: achieved HBM GB/s and TFLOP/s", "value":
        (attn_bytes + write_bytes) / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "seq_steps_per_s": wl.batch / (ms * 1e-3),
        "config": {"workload": f"{wl.name}: B={wl.batch} q_len={Q} H={wl.num_heads} latent "
                               f"{wl.head_dim} + rope {wl.rope_dim} bs {wl.block_size}",
                   "seq_lens": f"U[{wl.len_lo},{wl.len_hi}] (sum {int(lens.sum())})",
                   "l2": "inputs larger than L2 (latent cache %.2f GB)" % (int(lens.sum()) * row / 1e9)},
        "roofline": {**hbm_roofline(ach, traffic_from_profiles(f"mla:{wl.name}"),
                                    f"mla_paged_decode{'_spec' if Q > 1 else ''} (attention + "
                                    f"merge), {dec_ms * 1e3:.1f} us per call", leg),
                     "kernels": breakdown},
        "tensor": {"achieved_tflops": tfl, "peak_tflops": tf, "frac": tfl / tf,
                   "note": "algorithmic flops; each score product is split along K across a CTA pair, none is computed twice"
                           + ("; each query row reads the latent rows it sees, repeats are meant to hit L2" if Q > 1 else "")},
        "gpu_launches": 3 * args.steps, "clocks": clocks}


def run_prefill(args, dev):
    """Mixed chunked-prefill + decode step: write the new K/V rows through slot_mapping,
    then causal paged prefill over every new row (tensor-core bound)."""
    import torch

    from paged_kv_cache_77_gb300 import api

    wl = synth.WORKLOADS["mixed_prefill"]
    if args.batch:
        wl = wl.scaled(batch=args.batch)
    d = synth.draw(wl)
    v = synth.values(wl, d, dev)
    pool = api.BlockPool(d.num_blocks, d.pool_order)
    table_np = pool.build_block_table(d.seq_lens, wl.block_size, 0, d.max_blocks_per_seq)
    slots = torch.from_numpy(api.build_slot_mapping(table_np, d.start_pos, d.num_new,
                                                    wl.block_size)).to(dev)
    table = torch.from_numpy(table_np).to(dev)
    seq_lens = torch.from_numpy(d.seq_lens).to(dev)
    cu = torch.from_numpy(np.cumsum(d.num_new).astype(np.int32)).to(dev)
    T = int(d.num_new.sum())
    out = torch.empty((T, wl.num_heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(api.prefill_workspace_size(), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    q = d.num_new.astype(np.int64)
    c = (d.seq_lens - d.num_new).astype(np.int64)
    pairs = int((q * c + q * (q + 1) // 2).sum())  # visible (query row, key) pairs per head
    flops = pairs * wl.num_heads * 4 * wl.head_dim
    row = wl.num_kv_heads * wl.head_dim * 2
    write_bytes = T * row * 2 * 2 + T * 4

    def write():
        api.kv_cache_write(v["k_cache"], v["v_cache"], v["k_new"], v["v_new"], slots)

    def attend():
        api.paged_attention_prefill(v["q"], cu, v["k_cache"], v["v_cache"], table, seq_lens,
                                    wl.scale, causal=True, out=out, workspace=ws)

    for _ in range(args.warmup):
        write()
        attend()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        write()
        attend()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    pf_ms, leg = timed_leg(attend, stream)  # the prefill call alone, for at least a second
    breakdown = kernel_breakdown(attend)
    hbm, tf, peak_kind = peaks()
    tfl = flops / (pf_ms * 1e-3) / 1e12
    return {
        "metric": "causal paged prefill (mixed with decode rows): achieved TFLOP/s",
        "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": T / (ms * 1e-3),
        "config": {"workload": f"mixed_prefill: {wl.batch} seqs H={wl.num_heads} "
                               f"H_kv={wl.num_kv_heads} d={wl.head_dim}, {T} new rows, "
                               f"prior U[{wl.len_lo},{wl.len_hi}], q U[{wl.q_lo},{wl.q_hi}], "
                               f"{wl.forced_q1} decode rows",
                   "step": "kv_cache_write of the new rows + paged_attention_prefill",
                   "write_bytes": write_bytes, "flops": flops,
                   "l2": "inputs larger than L2 (KV cache read %.2f GB, q %.2f GB; tensor-bound)"
                         % (int(d.seq_lens.sum()) * row * 2 / 1e9, T * wl.num_heads * wl.head_dim * 2 / 1e9)},
        "roofline": {"bound": "tensor", "achieved": tfl, "peak": tf, "unit": "TFLOP/s",
                     "frac": tfl / tf, "traffic": traffic_from_profiles("prefill:mixed_prefill"),
                     "kernel": f"paged_attention_prefill (attention + merge), {pf_ms * 1e3:.1f} us",
                     "peak_kind": peak_kind + " bf16 dense burst", **leg, "kernels": breakdown},
        "gpu_launches": 3 * args.steps, "clocks": clocks}


def run_scatter(args, dev):
    """kv_cache_write alone at bandwidth scale: 262,144 rows of K and V (H_kv 8, d 128)
    scattered to a random permutation of the slots of a 2048-block cache."""
    import torch

    from paged_kv_cache_77_gb300 import api

    rows, hkv, d, bs = args.batch or 262144, 8, 128, 128
    nb = rows // bs
    g = torch.Generator(device=dev)
    g.manual_seed(1005)
    k = torch.randn((rows, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((rows, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    kc = torch.zeros((nb, bs, hkv, d), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    perm = np.random.default_rng(1005).permutation(nb * bs).astype(np.int32)
    slots = torch.from_numpy(perm).to(dev)
    nbytes = rows * hkv * d * 2 * 2 * 2 + rows * 4  # read + write of K and V rows, slots
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        api.kv_cache_write(kc, vc, k, v, slots)
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        api.kv_cache_write(kc, vc, k, v, slots)
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    gbs = nbytes / (ms * 1e-3) / 1e9
    leg_ms, leg = timed_leg(lambda: api.kv_cache_write(kc, vc, k, v, slots), stream)
    leg["kernels"] = kernel_breakdown(lambda: api.kv_cache_write(kc, vc, k, v, slots))
    return {
        "metric": "kv_cache_write scatter: achieved HBM GB/s", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"scatter: {rows} rows x (K+V) H_kv {hkv} d {d}, random slots",
                   "l2": "inputs larger than L2 (%.2f GB moved per step)" % (nbytes / 1e9)},
        "roofline": hbm_roofline(nbytes / (leg_ms * 1e-3) / 1e9, traffic_from_profiles("write:scatter"),
                                 f"kv_cache_write, {leg_ms * 1e3:.1f} us per call", leg),
        "gpu_launches": args.steps, "clocks": clocks}


def run_fork(args, dev):
    """Fork of 512 parent requests (prompt ~ U[1, 4096] tokens, H_kv 8, d 128, bs 128)
    into 4 children each through the library's allocator with shared full blocks:
    the timed step is the device copy of every incomplete last block in the K and
    the V cache (pkv_copy_blocks). Host costs of the allocator are reported beside."""
    import torch

    from paged_kv_cache_77_gb300 import api

    parents, kids, hkv, d, bs = args.batch or 512, 4, 8, 128, 128
    rng = np.random.default_rng(1006)
    prompts = rng.integers(1, 4097, size=parents)
    nb = int(sum(-(-int(n) // bs) for n in prompts)) + parents * kids + 1
    mgr = api.KVCacheManager([0], [nb], bs, 1 << 20, initial_orders=[rng.permutation(nb)])
    t_alloc = time.perf_counter()
    for i, n in enumerate(prompts):
        assert mgr.allocate_slots(i, 0, int(n))
    t_alloc = (time.perf_counter() - t_alloc) / parents
    pairs = []
    t_fork = time.perf_counter()
    for i, n in enumerate(prompts):
        pairs += mgr.fork(i, [parents + kids * i + c for c in range(kids)], int(n), True)[0]
    t_fork = (time.perf_counter() - t_fork) / parents
    t_dec = time.perf_counter()
    ndec = 0
    for i, n in enumerate(prompts[:64]):
        for step in range(32):
            mgr.allocate_slots(i, int(n) + step, 1)
            ndec += 1
    t_dec = (time.perf_counter() - t_dec) / ndec
    g = torch.Generator(device=dev)
    g.manual_seed(1006)
    kc = torch.randn((nb, bs, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn((nb, bs, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    src = torch.tensor([a for a, _ in pairs], dtype=torch.int32, device=dev)
    dst = torch.tensor([b for _, b in pairs], dtype=torch.int32, device=dev)
    block_bytes = bs * hkv * d * 2
    # K and V: each distinct source block read once (a parent's last block feeds all
    # of its children; the repeats come from L2), every destination written, ids.
    n_src = len({a for a, _ in pairs})
    nbytes = 2 * block_bytes * (n_src + len(pairs)) + 8 * len(pairs)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        api.copy_blocks(kc, src, dst)
        api.copy_blocks(vc, src, dst)
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        api.copy_blocks(kc, src, dst)
        api.copy_blocks(vc, src, dst)
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    gbs = nbytes / (ms * 1e-3) / 1e9

    def both():
        api.copy_blocks(kc, src, dst)
        api.copy_blocks(vc, src, dst)

    leg_ms, leg = timed_leg(both, stream)
    leg["kernels"] = kernel_breakdown(both)
    return {
        "metric": "fork block copy: achieved HBM GB/s", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"fork: {parents} parents x {kids} children, prompt U[1,4096], "
                               f"H_kv {hkv} d {d}, {len(pairs)} copied blocks per cache "
                               f"from {n_src} distinct sources",
                   "l2": "inputs larger than L2 (%.2f GB moved per step)" % (nbytes / 1e9),
                   "host_us_per_fork": t_fork * 1e6, "host_us_per_prefill_allocate": t_alloc * 1e6,
                   "host_us_per_decode_allocate": t_dec * 1e6},
        "roofline": hbm_roofline(nbytes / (leg_ms * 1e-3) / 1e9, None,
                                 f"copy_blocks on K and V, {leg_ms * 1e3:.1f} us per fork", leg),
        "gpu_launches": 2 * args.steps, "clocks": clocks}


def run_mla_write(args, dev):
    """Fused MLA cache write at bandwidth scale: 262,144 tokens of latent (512) + rope
    (64) rows, RMSNorm + RoPE, written to distinct random slots of a 2,056-block
    cache (pkv_mla_rmsnorm_rope_write, no k_nope / k_rope copies)."""
    import torch

    import synth
    from paged_kv_cache_77_gb300 import api

    T = args.batch or 262144
    nb = -(-T // 128) + 8
    v = synth.draw_mla_write(T, nb, 1007, device=dev)
    nbytes = T * (1152 + 512 + 1152 + 4)  # latent read, cos+sin read, rows written, slot
    stream = torch.cuda.current_stream(dev)

    def step():
        api.mla_rmsnorm_rope_write(v["cache_nope"], v["cache_rope"], v["latent"], v["gamma"],
                                   v["cos"], v["sin"], v["slots"], 1e-6)

    for _ in range(args.warmup):
        step()
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    gbs = nbytes / (ms * 1e-3) / 1e9
    leg_ms, leg = timed_leg(step, stream)
    leg["kernels"] = kernel_breakdown(step)
    return {
        "metric": "fused MLA RMSNorm+RoPE cache write: achieved HBM GB/s", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"mla_write: {T} tokens x (latent 512 + rope 64), random slots",
                   "l2": "inputs larger than L2 (%.2f GB moved per step)" % (nbytes / 1e9)},
        "roofline": hbm_roofline(nbytes / (leg_ms * 1e-3) / 1e9, None,
                                 f"mla_rmsnorm_rope_write, {leg_ms * 1e3:.1f} us per call", leg),
        "gpu_launches": args.steps, "clocks": clocks}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gqa_long",
                    choices=["gqa_long", "swa", "mha_tiny", "spec_decode", "scatter", "mla", "mla_spec",
                             "mixed_prefill",
                             "fork", "mla_write"])
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller cases for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="reference arm: seconds of oracle work over the whole run")
    ap.add_argument("--decode-kernel", default="auto", choices=["auto", "cuda_core", "tensor_core"])
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="fp8: decode workloads over an E4M3 cache with per-row scales")
    ap.add_argument("--cpu-baseline-child", action="store_true")
    ap.add_argument("--no-all-cores", action="store_true",
                    help="CPU baseline: skip the leg that runs the oracle on every core")
    ap.add_argument("--no-per-config", action="store_true",
                    help="default workload: skip the short runs of the other workloads")
    ap.add_argument("--bare", action="store_true",
                    help="only the timed steps (one call per roofline leg, no profiler, no e2e, "
                         "no other workloads, no CPU baseline): a short run to capture under ncu")
    args = ap.parse_args()
    if args.bare:
        global BARE
        BARE = True
        args.no_cpu_baseline = args.no_per_config = True
    if args.cpu_baseline_child:
        cpu_baseline_child(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
