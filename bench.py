"""Benchmark of one serving step of the paged-KV attention forward on GB300.

A step is one pass of the whole path over one synthetic batch:
pka_cache_write of the new tokens, then pka_paged_attn_forward (planner,
decode / prefill / extend kernels, split-KV and extend reductions).

Default workload (the headline): decode-only GQA, 256 requests with context
U[1024, 8192], 32 query / 4 KV heads, head dim 128, block 16. The metric is
the decode KV stream rate (algorithmic K+V bytes per step / step time). The
prefill, mixed and MLA workloads are timed after it and reported under
"workloads" (they are not the headline number).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 (started by torch.distributed.run, or by this script itself when
it was not) every rank runs its own batch (weak scaling, no collective on the
data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
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

from paged_kv_attention_07_gb300 import workloads as W  # noqa: E402

METRIC = "decode KV GB/s & tokens/s; prefill/extend TFLOPS; % of HBM / BF16 roofline"


# ---------------------------------------------------------------- work model
def algorithmic_work(spec: W.BatchSpec, kv_elem_bytes: int = 2) -> dict:
    """Bytes and flops a step must move/do, counted once (no re-reads).
    kv_elem_bytes: bytes per cache element (2 = bf16, 1 = the 8-bit cache)."""
    Hq, Hkv, d, dv = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.head_dim_v
    nd, ne = spec.num_decodes, spec.num_extends
    e = kv_elem_bytes
    row_bytes = (d * e) if spec.mla else Hkv * (d + dv) * e  # one key's K+V (latent: one row)
    dec_keys = sum(spec.seq_lens[:nd])
    dec_bytes = dec_keys * row_bytes
    dec_flops = dec_keys * Hq * 2 * (d + dv)
    pair_flops = Hq * 2 * (d + dv)  # per visible (query, key) pair
    ext_pairs = 0
    for r in range(nd, nd + ne):
        q, c = spec.qlen[r], spec.ctx[r]
        ext_pairs += q * c + q * (q + 1) // 2
    pre_pairs = sum(q * (q + 1) // 2 for q in spec.qlen[nd + ne:])
    # read (bf16 K/V rows) + write (cache elements)
    cw_bytes = spec.num_tokens * (Hkv * (d + (0 if spec.mla else dv)) * 2 + row_bytes)
    return {"dec_bytes": dec_bytes, "dec_flops": dec_flops, "ext_flops": ext_pairs * pair_flops,
            "pre_flops": pre_pairs * pair_flops, "cache_write_bytes": cw_bytes,
            "tokens": spec.num_tokens, "decode_tokens": nd}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def kernel_traffic(kernel_file: str, key: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since it was captured; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        ent = t[key]
        src = open(os.path.join(ROOT, "paged_kv_attention_07_gb300", "csrc", kernel_file), "rb").read()
        if hashlib.sha256(src).hexdigest()[:16] != ent["source_sha"]:
            return None
        return float(ent["bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [p for (t, p) in self.samples if t0 - 0.15 <= t <= t1 + 0.15] or [p for (_, p) in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- our arm
FP8_SCALES = (0.0125, 0.02)  # per-tensor K / V scales of the 8-bit cache workloads


def make_device_batch(spec, device, seed, unified=False, kv_scales=None):
    from paged_kv_attention_07_gb300.device_batch import DeviceBatch
    batch = W.make_batch(spec, values=False)
    return DeviceBatch(batch, device=device, values_on_device_seed=seed, unified=unified, kv_scales=kv_scales)


def time_steps(db, steps, warmup, flush_bytes=0, kernels=(), barrier=None):
    """Warm up, then time `steps` steps with CUDA events on the launching
    stream (L2 flushed between steps when flush_bytes > 0): that is the step
    time. Then `steps` more steps with the library's per-launch event timers
    on, for each kernel's own device time and the launch count (timers between
    the launches would hold back the overlap of one kernel's launch with its
    predecessor, so the step time is taken without them).
    Returns (ms per step, kernel stats, launches per timed pass, (t0, t1))."""
    import torch
    from paged_kv_attention_07_gb300 import pka
    stream = torch.cuda.current_stream()
    flush = torch.empty(flush_bytes // 4, dtype=torch.float32, device=db.device) if flush_bytes else None
    for _ in range(warmup):
        db.step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if barrier:
        barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(steps):
        if flush is not None:
            flush.fill_(float(i))
        ev[i][0].record(stream)
        db.step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if barrier:
        barrier()
    ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    all_k = list(pka.KERNELS)
    for k in all_k:
        pka.pka_kernel_timer(k, True)
    for i in range(steps):
        if flush is not None:
            flush.fill_(float(i))
        db.step()
    torch.cuda.synchronize()
    stats, launches = {}, 0
    for k in all_k:
        tot, n, timed = pka.pka_kernel_timer_read(k)
        launches += n
        if timed:
            stats[k] = {"avg_ms": tot / timed, "launches": n}
        pka.pka_kernel_timer(k, False)
    return ms, stats, launches, (t0, t1)


def e2e_steps(db, steps, warmup):
    """Same step through the public API with host-resident inputs: every step
    copies its inputs from pinned host memory to the device (one copy: the
    inputs sit in one staging arena, as a server keeps them), runs the step,
    and reads out and lse back (one copy). The arenas and output buffers are
    double-buffered and the copies run on their own streams, so step i's
    results go back and step i + 2's inputs come in while step i + 1 computes;
    every copy of every timed step is inside the timed region (events on the
    compute stream bracket the whole loop and wait for the last copy)."""
    import torch
    stream = torch.cuda.current_stream()
    arena0, outs0 = db.pack_io()
    arenas = [arena0, arena0.clone()]
    outs = [outs0, outs0.clone()]
    host_in = arena0.cpu().pin_memory()
    host_out = [torch.empty(outs0.shape, dtype=outs0.dtype).pin_memory() for _ in range(2)]
    h2d, d2h = host_in.numel(), outs0.numel()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def loop(n):
        ev_in = [None, None]       # inputs of buffer b landed
        ev_step = [None, None]     # the step that read buffer b finished
        ev_out = [None, None]      # buffer b's results left the device
        for i in range(min(2, n)):  # first two steps' inputs
            s_in.wait_stream(stream)
            with torch.cuda.stream(s_in):
                arenas[i].copy_(host_in, non_blocking=True)
                ev_in[i] = torch.cuda.Event()
                ev_in[i].record(s_in)
        for i in range(n):
            b = i & 1
            stream.wait_event(ev_in[b])
            if ev_out[b] is not None:
                stream.wait_event(ev_out[b])  # this output buffer was read back
            db.use_io(arenas[b], outs[b])
            db.step()
            ev_step[b] = torch.cuda.Event()
            ev_step[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_step[b])
                host_out[b].copy_(outs[b], non_blocking=True)
                ev_out[b] = torch.cuda.Event()
                ev_out[b].record(s_out)
            if i + 2 < n:  # step i + 2's inputs into this arena once step i is done with it
                with torch.cuda.stream(s_in):
                    s_in.wait_event(ev_step[b])
                    arenas[b].copy_(host_in, non_blocking=True)
                    ev_in[b] = torch.cuda.Event()
                    ev_in[b].record(s_in)
        for e in ev_out:
            if e is not None:
                stream.wait_event(e)

    loop(warmup)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    loop(steps)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


def roofline(bound, achieved, peak, unit, traffic):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic}


def secondary_workloads(device, steps, warmup, peaks, rank):
    """Prefill, mixed and MLA workloads, timed one after the other."""
    import torch
    res = {}
    # (name, spec, dominant kernel, bound, L2 flush bytes, committed ncu traffic entry)
    cases = [("decode_gqa_fp8", W.spec_decode_gqa(), "decode", "hbm", 0,
              ("decode_gqa_fp8.cu", "decode_gqa_fp8")),
             ("prefill_varlen", W.spec_prefill(), "prefill_extend", "tensor", 256 << 20,
              ("fa_fwd.cu", "fa_fwd_prefill_varlen")),
             ("mixed", W.spec_mixed(), "prefill_extend", "tensor", 0, ("fa_fwd.cu", "fa_fwd_mixed")),
             ("mixed_fp8", W.spec_mixed(), "prefill_extend", "tensor", 0, ("fa_fwd.cu", "fa_fwd_mixed_fp8")),
             ("mla_prefill_extend", W.spec_mla_prefill(), "prefill_extend", "tensor", 0,
              ("fa_fwd.cu", "fa_fwd_mla_prefill_extend")),
             ("mla_decode_bs64", W.spec_mla_decode(), "decode", "hbm", 0,
              ("decode_mla_tc.cu", "decode_mla_tc_mla_decode_bs64")),
             ("mla_decode_bs1", W.spec_mla_decode(block_size=1), "decode", "hbm", 0,
              ("decode_mla_tc.cu", "decode_mla_tc_mla_decode_bs1"))]
    for name, spec, dom, bound, flush, tkey in cases:
        traffic = kernel_traffic(*tkey) if tkey else None
        fp8 = name.endswith("_fp8")
        db = make_device_batch(spec, device, seed=1234 + rank, kv_scales=FP8_SCALES if fp8 else None)
        ms, stats, launches, _ = time_steps(db, steps, warmup, flush_bytes=flush)
        w = algorithmic_work(spec, 1 if fp8 else 2)
        ent = {"ms_per_step": round(ms, 4), "tokens_per_s": round(w["tokens"] / (ms * 1e-3), 1),
               "kernels": {k: round(v["avg_ms"], 4) for k, v in stats.items()}}
        if fp8:
            ent["cache"] = f"FP8 E4M3 codes, k_scale {FP8_SCALES[0]}, v_scale {FP8_SCALES[1]}"
        cd = stats.get("ctx_dequant", {}).get("avg_ms")
        if cd:  # the extends' context gathered out of the 8-bit cache: codes read, bf16 written
            ctx = sum(spec.ctx[spec.num_decodes:spec.num_decodes + spec.num_extends])
            gbytes = ctx * spec.num_kv_heads * (spec.head_dim + spec.head_dim_v) * 3
            ent["ctx_dequant"] = roofline("hbm", gbytes / (cd * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s", None)
        cw = stats.get("cache_write", {}).get("avg_ms")
        if cw:  # the step's cache write: its own bytes (read + write), its own roofline
            ent["cache_write"] = roofline("hbm", w["cache_write_bytes"] / (cw * 1e-3) / 1e9, peaks["hbm_gbs"],
                                          "GB/s", None)
        kms = stats.get(dom, {}).get("avg_ms")
        if bound == "tensor":
            flops = w["ext_flops"] + w["pre_flops"]
            ent["tflops_step"] = round(flops / (ms * 1e-3) / 1e12, 2)
            if kms:
                ent["roofline"] = roofline("tensor", flops / (kms * 1e-3) / 1e12, peaks["bf16_tflops"],
                                           "TFLOP/s", traffic)
            if w["dec_bytes"]:
                dk = stats.get("decode", {}).get("avg_ms")
                if dk:
                    ent["decode_kv_gbs"] = round(w["dec_bytes"] / (dk * 1e-3) / 1e9, 1)
        else:
            ent["kv_gbs_step"] = round(w["dec_bytes"] / (ms * 1e-3) / 1e9, 1)
            if kms:
                ent["roofline"] = roofline("hbm", w["dec_bytes"] / (kms * 1e-3) / 1e9, peaks["hbm_gbs"],
                                           "GB/s", traffic)
                ent["tflops_decode_kernel"] = round(w["dec_flops"] / (kms * 1e-3) / 1e12, 1)
        res[name] = ent
        del db
        torch.cuda.empty_cache()
    # single-path routing of the same mixed batch: the decodes go through the
    # prefill/extend kernel as one-token extends (num_decodes 0); compared with
    # the three-path step above
    spec = W.spec_mixed()
    db = make_device_batch(spec, device, seed=1234 + rank, unified=True)
    ms, stats, launches, _ = time_steps(db, steps, warmup)
    w = algorithmic_work(spec)
    ent = {"ms_per_step": round(ms, 4), "tokens_per_s": round(w["tokens"] / (ms * 1e-3), 1),
           "kernels": {k: round(v["avg_ms"], 4) for k, v in stats.items()},
           "three_path_ms_per_step": res.get("mixed", {}).get("ms_per_step")}
    kms = stats.get("prefill_extend", {}).get("avg_ms")
    if kms:
        flops = w["dec_flops"] + w["ext_flops"] + w["pre_flops"]
        ent["roofline"] = roofline("tensor", flops / (kms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s", None)
    res["mixed_unified"] = ent
    del db
    torch.cuda.empty_cache()
    # the mixed batch arriving in a shuffled request order: each step gathers
    # the rows into [decode : extend : prefill] order and the outputs back
    # (pka_batch_order + pka_gather_rows); roofline of the gather kernel
    import numpy as np
    from paged_kv_attention_07_gb300.device_batch import UnorderedBatch
    spec = W.spec_mixed()
    db = make_device_batch(spec, device, seed=1234 + rank)
    ub = UnorderedBatch(db, np.random.default_rng(5).permutation(spec.num_reqs))
    ms, stats, launches, _ = time_steps(ub, steps, warmup)
    ent = {"ms_per_step": round(ms, 4), "kernels": {k: round(v["avg_ms"], 4) for k, v in stats.items()},
           "gather_bytes_per_step": ub.gather_bytes}
    gk = stats.get("gather")
    if gk:
        gather_ms = gk["avg_ms"] * gk["launches"] / steps  # the step's 8 gathers together
        ent["gather_ms_per_step"] = round(gather_ms, 4)
        ent["roofline"] = roofline("hbm", ub.gather_bytes / (gather_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s",
                                   None)
    res["mixed_unordered"] = ent
    del ub, db
    torch.cuda.empty_cache()
    return res


class OracleStep:
    """One step of the oracle on a host batch: cache write of the new tokens
    into a cache that already holds the context (prepared once, untimed),
    then float64 attention of every row."""

    def __init__(self, batch):
        import oracle
        self.o = oracle
        self.batch = batch
        self.kc, self.vc = oracle.populate_cache(batch, "context")
        self.cores = oracle.default_threads()

    def __call__(self):
        b, s = self.batch, self.batch.spec
        self.o.cache_write(b.k_new, b.v_new, b.slot_mapping, self.kc, self.vc, s.block_size)
        return self.o.attention(b.q, self.kc, self.vc, b.block_table, b.query_start_loc, b.seq_lens,
                                s.scale, s.block_size, head_dim_v=s.head_dim_v, nthreads=self.cores)


def cpu_baseline(spec, max_reqs=64, min_seconds=10.0, max_repeats=200):
    """The float64 oracle on the host cores, on a bounded sample: the first
    `max_reqs` requests of the same workload, stepped repeatedly until about
    `min_seconds` of CPU work. Returns (GB/s, cores, sample, seconds)."""
    idx = list(range(min(max_reqs, spec.num_reqs)))
    sub = W.subset(spec, idx)
    step = OracleStep(W.make_batch(sub))
    cores = step.cores
    n = 0
    t0 = time.time()
    while n < max_repeats and (n == 0 or time.time() - t0 < min_seconds):
        step()
        n += 1
    dt = time.time() - t0
    w = algorithmic_work(sub)
    return (n * w["dec_bytes"] / dt / 1e9, cores,
            f"{len(idx)} of {spec.num_reqs} requests, {n} steps ({dt:.1f} s)", dt)


def max_over_ranks(ms: float, device=None) -> float:
    """Largest per-rank timed region (ms) over the process group (identity
    when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world: int, per_rank_bytes: float, ms: float) -> float:
    """Whole-job GB/s: every rank streams its own batch during the slowest rank's time."""
    return world * per_rank_bytes / (ms * 1e-3) / 1e9


def run_ours(args):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    peaks = load_peaks()
    if args.workload != "decode_gqa":
        return profile_workload(args, device)
    spec = W.spec_decode_gqa()
    db = make_device_batch(spec, device, seed=42 + rank)
    w = algorithmic_work(spec)

    def barrier():
        if world > 1:
            dist.barrier()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ms, stats, launches, (t0, t1) = time_steps(db, args.steps, args.warmup, kernels=("decode",),
                                               barrier=barrier)
    # keep the GPU busy long enough for the sampler to see the clocks under load
    extra_t0 = time.time()
    while args.clock_hold and time.time() - extra_t0 < 1.0:
        db.step()
    torch.cuda.synchronize()
    sampler.stop()
    clocks = sampler.summary(t0, max(t1, extra_t0 + 1.0))
    ms = max_over_ranks(ms, device)
    value = weak_scaling_value(world, w["dec_bytes"], ms)
    dec_ms = stats["decode"]["avg_ms"]
    achieved = w["dec_bytes"] / (dec_ms * 1e-3) / 1e9
    traffic = kernel_traffic("decode_gqa.cu", "decode_gqa")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, random block table)",
        "config": {"workload": "decode_gqa: 256 decode requests, ctx U[1024,8192], 32 q / 4 kv heads, "
                               "head_dim 128, block 16", "l2": "inputs larger than L2 (2.4 GB KV)",
                   "parallelism": f"replicas x{world}"},
        "decode_tokens_per_s": round(world * w["decode_tokens"] / (ms * 1e-3), 1),
        "roofline": roofline("hbm", achieved, peaks["hbm_gbs"], "GB/s", traffic),
        "roofline_peak_source": peaks["source"],
        "kernels_ms": {k: round(v["avg_ms"], 4) for k, v in stats.items()},
        "cache_write": (roofline("hbm", w["cache_write_bytes"] / (stats["cache_write"]["avg_ms"] * 1e-3) / 1e9,
                                 peaks["hbm_gbs"], "GB/s", None) if "cache_write" in stats else None),
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if args.e2e:
        e_ms, h2d, d2h = e2e_steps(db, max(3, args.steps // 2), 2)
        line["e2e"] = {"value": round(world * w["dec_bytes"] / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(e_ms, 5)}
    del db
    torch.cuda.empty_cache()
    if args.all_workloads:
        line["workloads"] = secondary_workloads(device, max(3, args.steps // 2), args.warmup, peaks, rank)
    if rank == 0 and world == 1 and args.cpu_baseline:
        v, cores, sample, _ = cpu_baseline(spec)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


WORKLOADS = {"decode_gqa": W.spec_decode_gqa, "decode_gqa_fp8": W.spec_decode_gqa,
             "prefill_varlen": W.spec_prefill, "mixed": W.spec_mixed, "mixed_fp8": W.spec_mixed,
             "mla_decode_bs64": W.spec_mla_decode, "mla_prefill_extend": W.spec_mla_prefill,
             # profiling cases: 64 heads (the warp-MMA MLA kernel), and the
             # non-absorbed prefill/extend at a size an ncu replay handles
             "mla_decode_h64": lambda: W.spec_mla_decode(heads=64),
             "mla_prefill_extend_small": lambda: W.spec_mla_prefill(n_ext=2, n_pre=1, heads=32),
             "mla_decode_bs1": lambda: W.spec_mla_decode(block_size=1),
             "mixed_unified": W.spec_mixed, "mixed_unordered": W.spec_mixed,
             # the public two-input merge alone, on fp32 partials of the mixed
             # batch's shape (every new token x 32 heads x 128 dims)
             "merge_attn_states": W.spec_mixed}


def profile_merge(args, device):
    """pka_merge_attn_states on two fp32 partial outputs with their LSEs, one
    row per (token, head) of the mixed batch: --steps timed calls."""
    import torch
    from paged_kv_attention_07_gb300 import pka
    spec = WORKLOADS["merge_attn_states"]()
    rows, dv = spec.num_tokens * spec.num_q_heads, spec.head_dim_v
    g = torch.Generator(device=device).manual_seed(7)
    a, b = (torch.randn(rows, dv, generator=g, device=device) for _ in range(2))
    la, lb = (torch.randn(rows, generator=g, device=device) * 4 for _ in range(2))
    out, lse = torch.empty_like(a), torch.empty_like(la)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        pka.pka_merge_attn_states(out, lse, a, la, b, lb)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for e0, e1 in ev:
        e0.record(stream)
        pka.pka_merge_attn_states(out, lse, a, la, b, lb)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / args.steps
    nbytes = rows * (3 * dv * 4 + 3 * 4)  # two partial rows and LSEs in, one row and LSE out
    print(json.dumps({"workload": "merge_attn_states", "rows": rows, "head_dim": dv, "io": "fp32",
                      "ms_per_call": ms, "gbs": round(nbytes / ms / 1e6, 1), "gpu_launches": args.steps}))


def profile_workload(args, device):
    """Run --steps steps of one workload and print its timing (for profilers)."""
    if args.workload == "merge_attn_states":
        return profile_merge(args, device)
    spec = WORKLOADS[args.workload]()
    db = make_device_batch(spec, device, seed=7, unified=args.workload == "mixed_unified",
                           kv_scales=FP8_SCALES if args.workload.endswith("_fp8") else None)
    if args.workload == "mixed_unordered":
        import numpy as np
        from paged_kv_attention_07_gb300.device_batch import UnorderedBatch
        db = UnorderedBatch(db, np.random.default_rng(5).permutation(spec.num_reqs))
    ms, stats, launches, _ = time_steps(db, args.steps, args.warmup)
    print(json.dumps({"workload": args.workload, "ms_per_step": ms,
                      "kernels_ms": {k: v["avg_ms"] for k, v in stats.items()}, "gpu_launches": launches}))


def run_reference(args):
    """The oracle (float64 C, host cores) as the reference arm, on a bounded
    sample of the same workload per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    spec = W.spec_decode_gqa()
    sub = W.subset(spec, list(range(16)))
    step = OracleStep(W.make_batch(sub))
    cores = step.cores
    for _ in range(args.warmup):
        step()
    t0 = time.time()
    for _ in range(args.steps):
        step()
    dt = (time.time() - t0) / args.steps
    wk = algorithmic_work(sub)
    value = wk["dec_bytes"] / dt / 1e9
    sample = f"16 of 256 requests per step ({dt:.2f} s per step)"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, random block table)",
            "config": {"workload": "decode_gqa: 256 decode requests, ctx U[1024,8192], 32 q / 4 kv heads, "
                                   "head_dim 128, block 16"},
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def launch_ranks(n: int, argv) -> int:
    """Run this script as n ranks under torch.distributed.run; returns its exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--primary-only", dest="all_workloads", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode_gqa",
                    help="run only this workload's steps (for profilers); the default is the headline")
    ap.add_argument("--profile", action="store_true",
                    help="short run for profilers: no clock hold, e2e, CPU baseline or secondary workloads")
    args = ap.parse_args()
    args.clock_hold = True
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not launched by torch.distributed.run: start the N ranks here (one
        # process per GPU, rendezvous on the loopback address)
        sys.exit(launch_ranks(args.gpus, sys.argv[1:]))
    if args.profile:
        args.e2e = args.all_workloads = args.cpu_baseline = args.clock_hold = False
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
