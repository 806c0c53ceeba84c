#!/usr/bin/env python
"""Benchmark of split-KV GQA decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--suite]

One step = one decode-attention call (the split-KV kernel, which merges every
segment of up to 8 pieces itself; a combine kernel follows only for longer
ones) over the largest decode configuration that fits one GPU, the mixed serving
batch: B=64, Hq=64, Hkv=8 (G=8), head_dim 128, sequence lengths log-uniform in
[1, 32768], paged bf16 cache with 16-token pages and a shuffled page table,
seeded N(0,1) inputs.  Inputs are resident in HBM; L2 is flushed before every
step (a write of a buffer larger than L2, then a read of another, so no dirty
lines are left to write back), outside the step's CUDA-event pair.  The value is
achieved GB/s of algorithmic bytes (K/V + Q + partials read + page table +
seq_lens); µs/call is reported beside it.  The same line carries "gates": the
long-context GQA-6 (ctx 4096 and 16384), paged-batch and very-long-sequence
configurations, measured the same way in the same run.

--impl reference times the fp64 CPU oracle on the host cores (bounded sample
per step).  --suite also measures every other workload (one JSON line each).
Under torchrun each rank runs an independent replica (no collective on the
data path); the value is the total over ranks divided by the slowest rank.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/call and achieved HBM GB/s vs GB300 peak (1 GPU)"
PREFILL_METRIC = "causal GQA prefill µs/call and achieved TFLOP/s vs GB300 bf16 peak (1 GPU)"
HEADLINE = "mixed_paged_b64_hq64_hkv8_d128_log1_32768_ps16"
# The other configurations with a bandwidth target (>= 70% of HBM), reported in
# the headline's line.
GATES = ["gqa6_contig_b1_hq24_hkv4_d256_ctx4096", "gqa6_contig_b1_hq24_hkv4_d256_ctx16384",
         "paged_b16_hq32_hkv8_d128_u256_8192_ps32", "long_contig_b1_hq32_hkv8_d128_ctx65536_outliers"]
GATE_FRAC = 0.70
# Published time per call of the pages' fa_split_gqa_kernel on the GQA-6 ctx-4096
# workload (RTX 5090, "perf(dspark): overlap KV staging with compute via
# cp.async", section "Why there was still headroom").
PAGES_US_PER_CALL = {"gqa6_contig_b1_hq24_hkv4_d256_ctx4096": 1110.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--suite", action="store_true", help="also measure every other workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gates", action="store_true", help="skip the gated configurations (profiling runs)")
    ap.add_argument("--cpu-child", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help=argparse.SUPPRESS)
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

# The sources each kind of workload runs (the ncu figures in profiles/ are tied to them).
KERNEL_SOURCES = {
    "decode": ("decode_attn.cu", "plan.cuh", "ptx.cuh", "split_kernel.cuh", "combine_kernel.cuh"),
    "prefill": ("prefill_host.cuh", "prefill_kernel.cuh", "prefill_tc.cuh", "tc05.cuh", "ptx.cuh"),
}


def kernel_source_hash(kind: str = "decode") -> str:
    csrc = os.path.join(ROOT, "gqa_split_kv_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash("prefill" if workload.startswith("prefill_") else "decode")
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == want:
            return int(parts[2])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        # the tool's start-up stalls the GPU for up to seconds: let it reach its
        # first sample before the timed region begins
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 15.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)
        time.sleep(0.15)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        mhz = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, dist=None, device="cpu"):
    """Each rank's timings (ms) -> the maximum over ranks of each, in order."""
    if dist is None:
        return [float(v) for v in values]
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_value(world: int, bytes_per_step: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput in GB/s: every rank moved bytes_per_step per step (weak
    scaling, one replica per GPU), and the slowest rank's time counts."""
    return world * bytes_per_step * steps / (total_ms / 1e3) / 1e9


# ------------------------------------------------------------ CPU baseline

def oracle_unit(oracle, wl, inp, b: int, g: int) -> int:
    """The oracle on one sample unit: every query row of KV head g of sequence b.
    Returns the unit's algorithmic bytes (its K/V rows and query rows); for a
    prefill workload the unit is one query head's chunk and the return is flops."""
    G = wl.Hq // wl.Hkv
    if wl.kind == "prefill":  # one query head over the whole chunk; returns flops
        oracle.prefill(inp, [(b, i, g * G) for i in range(wl.q_len)])
        L = int(inp["seq_lens"][b])
        return 4 * wl.D * sum(max(0, min(L, L - wl.q_len + 1 + i)) for i in range(wl.q_len))
    if wl.kv_dtype == "int8":
        oracle.decode_int8(inp, [(b, g * G + i) for i in range(G)])
        return 2 * (wl.D + 4) * int(inp["seq_lens"][b]) + G * wl.D * 2
    if wl.q_len == 1:
        oracle.decode_rows(inp, [(b, g * G + i) for i in range(G)])
    else:
        oracle.decode_multi(inp, [(b, g * G + i, j) for i in range(G) for j in range(wl.q_len)])
    return 2 * wl.D * 2 * int(inp["seq_lens"][b]) + G * wl.q_len * wl.D * 2


def cpu_child(workload: str, seconds: float):
    """Runs in a subprocess with the BLAS thread count fixed: times the oracle."""
    import numpy as np  # noqa: F401

    import oracle
    from gqa_split_kv_gb300.workloads import WORKLOADS, make_inputs

    wl = WORKLOADS[workload]
    inp = make_inputs(wl)
    # sample unit: all G query heads (x q_len query tokens) of one (sequence, KV head)
    groups = [(b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    done_bytes, n = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or n == 0:
        b, g = groups[n % len(groups)]
        done_bytes += oracle_unit(oracle, wl, inp, b, g)
        n += 1
    dt = time.perf_counter() - t0
    print(json.dumps({"gbs": done_bytes / dt / 1e9, "tflops": done_bytes / dt / 1e12, "units": n, "seconds": dt}))


def _cpu_child_run(workload: str, seconds: float, threads: int):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(threads)
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-child", workload, "--cpu-seconds",
                          str(seconds)], capture_output=True, text=True, env=env, cwd=ROOT)
    line = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    if res.returncode != 0 or not line:
        return None, res.stderr[-300:]
    return json.loads(line[-1]), ""


def run_cpu_baseline(workload: str, seconds: float) -> dict:
    """The oracle on the host cores (BLAS threads = cores), plus its single-thread rate
    on a shorter sample of the same units."""
    cores = os.cpu_count() or 1
    from gqa_split_kv_gb300.workloads import WORKLOADS
    pre = WORKLOADS[workload].kind == "prefill"
    unit, key = ("TFLOP/s", "tflops") if pre else ("GB/s", "gbs")
    d, err = _cpu_child_run(workload, seconds, cores)
    if d is None:
        return {"value": None, "unit": unit, "cores": cores, "kind": "oracle", "sample": f"failed: {err}"}
    d1, _ = _cpu_child_run(workload, max(1.0, seconds / 4), 1)
    what = ("one (sequence, query head) over the whole chunk" if pre else
            "one (sequence, KV head) with its G query heads over the full context")
    return {"value": round(d[key], 6 if pre else 4), "unit": unit, "cores": cores, "kind": "oracle",
            "sample": f"{d['units']} units of {what}, {d['seconds']:.1f} s, fp64 numpy oracle, BLAS threads = {cores}",
            "single_thread": None if d1 is None else {"value": round(d1[key], 6 if pre else 4), "units": d1["units"],
                                                        "seconds": round(d1["seconds"], 1)}}


# ------------------------------------------------------------ our arm

def measure(wl, inp, steps: int, warmup: int, flush_bytes: int, dist=None, sampler=None, e2e_steps: int = 0):
    import numpy as np
    import torch

    from gqa_split_kv_gb300 import binding
    from gqa_split_kv_gb300.accounting import traffic_bytes

    dev = torch.cuda.current_device()

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    kv8 = wl.kv_dtype == "int8"
    paged = wl.layout == "paged"
    q = to_dev(inp["q"])
    lens = torch.from_numpy(inp["seq_lens"]).cuda()
    table = torch.from_numpy(inp["page_table"]).cuda() if paged else None
    max_len = wl.max_ctx
    # host arrays of the cache: (K, V) or, for int8, (K, V, K scales, V scales)
    kv_names = ((("k_pool_i8", "v_pool_i8", "k_scale_pool", "v_scale_pool") if paged else
                 ("k_i8", "v_i8", "k_scale", "v_scale")) if kv8 else (("k_pool", "v_pool") if paged else ("k", "v")))
    if kv8:
        kv_dev = [torch.from_numpy(np.ascontiguousarray(inp[n])).cuda() for n in kv_names]
    else:
        kv_dev = [to_dev(inp[n]) for n in kv_names]
    kc, vc = kv_dev[0], kv_dev[1]
    S = binding.num_splits_multi(wl.B, wl.q_len, wl.Hq, wl.Hkv, max_len, wl.D)
    rows = (wl.B, wl.Hq) if wl.q_len == 1 else (wl.B, wl.Hq, wl.q_len)  # multi-query: q_len rows per head
    out = torch.empty(rows + (wl.D,), dtype=torch.bfloat16, device="cuda")
    pa = torch.empty(rows + (S, wl.D), dtype=torch.float32, device="cuda") if S > 1 else None
    pm = torch.empty(rows + (S, 2), dtype=torch.float32, device="cuda") if S > 1 else None
    ctr = torch.zeros(binding.counters_len(wl.B, wl.Hq, wl.Hkv, wl.q_len), dtype=torch.int64, device="cuda")
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device="cuda")
    flush_src = torch.empty(flush_bytes // 4, dtype=torch.float32, device="cuda").zero_()
    stream = torch.cuda.current_stream()

    def flush_l2():
        # write a buffer larger than L2, then read another: L2 ends up holding only
        # clean, unrelated lines, so the timed call pays no write-back of the flush
        flush.zero_()
        torch.sum(flush_src)

    attn_paged = binding.decode_attn_paged if wl.q_len == 1 else binding.decode_attn_multi_paged
    attn_contig = binding.decode_attn_contig if wl.q_len == 1 else binding.decode_attn_multi_contig

    def call(qq=q, kk=kc, vv=vc, ll=lens, oo=out):
        if kv8 and paged:
            binding.decode_attn_int8_paged(qq, kk, vv, kv_dev[2], kv_dev[3], table, ll, max_len, scale=wl.scale,
                                           splits=S, part_acc=pa, part_ml=pm, seg_counters=ctr, out=oo)
        elif kv8:
            binding.decode_attn_int8_contig(qq, kk, vv, kv_dev[2], kv_dev[3], ll, scale=wl.scale, splits=S,
                                            part_acc=pa, part_ml=pm, seg_counters=ctr, out=oo)
        elif paged:
            attn_paged(qq, kk, vv, table, ll, max_len, scale=wl.scale, splits=S, part_acc=pa, part_ml=pm,
                       seg_counters=ctr, out=oo)
        else:
            attn_contig(qq, kk, vv, ll, scale=wl.scale, splits=S, part_acc=pa, part_ml=pm, seg_counters=ctr,
                        out=oo)

    for _ in range(warmup):
        flush_l2()
        call()
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    for i in range(steps):
        flush_l2()
        ev0[i].record(stream)
        call()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    if sampler:
        clocks = sampler.stop()
    else:
        clocks = None
    if dist is not None:
        dist.barrier()
    times = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]  # ms
    assert binding.device_error() == 0
    tb = traffic_bytes(wl.B, wl.Hq, wl.Hkv, wl.D, inp["seq_lens"], S, wl.page_size if paged else None, wl.q_len,
                       wl.kv_dtype)
    # the split kernel, plus the combine kernel when a segment can have more than 8 pieces
    res = {"S": S, "times_ms": times, "bytes": tb, "clocks": clocks, "launches_per_step": 1 if S <= 8 else 2}

    if e2e_steps > 0:
        # end to end through the public call: pinned host inputs -> device, call, output -> host
        host = {"q": torch.from_numpy(np.ascontiguousarray(inp["q"]).view(np.int16)).pin_memory(),
                "lens": torch.from_numpy(inp["seq_lens"]).pin_memory()}
        kv_host = [torch.from_numpy(np.ascontiguousarray(inp[n])).pin_memory() for n in kv_names]
        # bf16 caches travel as their int16 bit patterns
        kv_dst = [t if kv8 else t.view(torch.int16) for t in kv_dev]
        kv_host = [h if kv8 else h.view(torch.int16) for h in kv_host]
        out_h = torch.empty(rows + (wl.D,), dtype=torch.int16).pin_memory()
        qi = q.view(torch.int16)
        h2d = sum(t.numel() * t.element_size() for t in [host["q"], host["lens"]] + kv_host)
        d2h = out_h.numel() * 2
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        for it in range(2):
            n = 3 if it == 0 else e2e_steps
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(n):
                qi.copy_(host["q"], non_blocking=True)
                for d, h in zip(kv_dst, kv_host):
                    d.copy_(h, non_blocking=True)
                lens.copy_(host["lens"], non_blocking=True)
                call()
                out_h.copy_(out.view(torch.int16), non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
        res["e2e_ms"] = e0.elapsed_time(e1) / e2e_steps
        res["h2d"] = h2d
        res["d2h"] = d2h
    del flush, flush_src
    return res


def measure_prefill(wl, inp, steps: int, warmup: int, flush_bytes: int, dist=None, sampler=None, e2e_steps: int = 0):
    """Causal prefill through the public call: device-timed steps (L2 flushed before
    each) and, optionally, end-to-end steps with the inputs copied in and the output out."""
    import numpy as np
    import torch

    from gqa_split_kv_gb300 import binding
    from gqa_split_kv_gb300.accounting import prefill_work

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    paged = wl.layout == "paged"
    names = ("k_pool", "v_pool") if paged else ("k", "v")
    q = to_dev(inp["q"])
    kc, vc = to_dev(inp[names[0]]), to_dev(inp[names[1]])
    lens = torch.from_numpy(inp["seq_lens"]).cuda()
    table = torch.from_numpy(inp["page_table"]).cuda() if paged else None
    out = torch.empty_like(q)
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device="cuda")
    flush_src = torch.empty(flush_bytes // 4, dtype=torch.float32, device="cuda").zero_()
    stream = torch.cuda.current_stream()

    def flush_l2():
        flush.zero_()
        torch.sum(flush_src)

    def call():
        if paged:
            binding.prefill_attn_paged(q, kc, vc, table, lens, wl.max_ctx, scale=wl.scale, out=out)
        else:
            binding.prefill_attn_contig(q, kc, vc, lens, scale=wl.scale, out=out)

    for _ in range(warmup):
        flush_l2()
        call()
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    for i in range(steps):
        flush_l2()
        ev0[i].record(stream)
        call()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    if dist is not None:
        dist.barrier()
    assert binding.device_error() == 0
    res = {"times_ms": [a.elapsed_time(b) for a, b in zip(ev0, ev1)], "clocks": clocks, "launches_per_step": 1,
           "work": prefill_work(wl.B, wl.Hq, wl.Hkv, wl.D, inp["seq_lens"], wl.q_len)}
    if e2e_steps > 0:
        hq = torch.from_numpy(np.ascontiguousarray(inp["q"]).view(np.int16)).pin_memory()
        hk = torch.from_numpy(np.ascontiguousarray(inp[names[0]]).view(np.int16)).pin_memory()
        hv = torch.from_numpy(np.ascontiguousarray(inp[names[1]]).view(np.int16)).pin_memory()
        hl = torch.from_numpy(inp["seq_lens"]).pin_memory()
        out_h = torch.empty(tuple(q.shape), dtype=torch.int16).pin_memory()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        for it in range(2):
            n = 3 if it == 0 else e2e_steps
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(n):
                q.view(torch.int16).copy_(hq, non_blocking=True)
                kc.view(torch.int16).copy_(hk, non_blocking=True)
                vc.view(torch.int16).copy_(hv, non_blocking=True)
                lens.copy_(hl, non_blocking=True)
                call()
                out_h.copy_(out.view(torch.int16), non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
        res["e2e_ms"] = e0.elapsed_time(e1) / e2e_steps
        res["h2d"] = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hl))
        res["d2h"] = out_h.numel() * 2
    del flush, flush_src
    return res


def prefill_line(wl, r, ws, K, W, total_ms, e2e_ms, peaks) -> dict:
    flops = r["work"]["flops"]
    per = sorted(r["times_ms"])
    achieved = flops / (total_ms / K / 1e3) / 1e12
    return {
        "metric": PREFILL_METRIC, "value": round(ws * flops * K / (total_ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": K, "warmup": W, "ms_per_step": round(total_ms / K, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "head_dim": wl.D, "ctx": wl.max_ctx,
                   "q_len": wl.q_len, "layout": wl.layout, "kind": "prefill", "accum": "fp32",
                   "l2": "flushed before every step (outside the timed pair)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "us_per_call": {"mean": round(1e3 * total_ms / K, 3), "median": round(1e3 * per[len(per) // 2], 3)},
        "work_per_call": r["work"],
        "roofline": {"bound": "tensor", "kernel": ("prefill_kernel (mma.sync bf16)" if wl.D == 32 else
                                                   "prefill_tc_kernel (tcgen05 bf16)") + ", events around the call",
                     "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "peak_source": f"{peaks['source']} cuBLAS bf16 burst", "traffic": ncu_traffic(wl.name)},
        "e2e": {"value": round(ws * flops / (e2e_ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": r["launches_per_step"] * K,
        "clocks": r["clocks"],
    }


def measure_gates(peaks, flush_bytes: int, steps: int, warmup: int) -> list:
    """The other gated configurations, each timed like the headline (L2 flushed
    before every call, CUDA events around it): median µs per call and the fraction
    of the measured HBM peak its algorithmic bytes reach."""
    from gqa_split_kv_gb300.workloads import WORKLOADS, make_inputs
    out = []
    for name in GATES:
        wl = WORKLOADS[name]
        r = measure(wl, make_inputs(wl), steps, warmup, flush_bytes)
        t = sorted(r["times_ms"])
        med = t[len(t) // 2]
        gbs = r["bytes"]["algorithmic"] / (med / 1e3) / 1e9
        out.append({"workload": name, "calls": steps, "us_per_call_median": round(1e3 * med, 3),
                    "us_per_call_p10": round(1e3 * t[len(t) // 10], 3), "achieved_gbs": round(gbs, 1),
                    "frac": round(gbs / peaks["hbm_gbs"], 4), "gate": GATE_FRAC,
                    "met": bool(gbs / peaks["hbm_gbs"] >= GATE_FRAC), "num_splits": r["S"]})
    return out


def ours(args):
    import torch

    from gqa_split_kv_gb300.workloads import WORKLOADS, make_inputs
    import gqa_split_kv_gb300

    ws, rank, local = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    else:
        torch.cuda.set_device(0)
    gqa_split_kv_gb300.load()
    peaks = measured_peaks()
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    flush_bytes = max(4 * l2, 256 << 20)
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl)
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    phys = vis[local] if local < len(vis) else str(local)
    sampler = ClockSampler(phys) if rank == 0 else None
    if wl.kind == "prefill":
        steps = min(args.steps, 200)  # a prefill call is ~1000x a decode call
        r = measure_prefill(wl, inp, steps, args.warmup, flush_bytes, dist=dist, sampler=sampler,
                            e2e_steps=max(3, min(steps, 20)))
        total_ms, e2e_ms = max_over_ranks([sum(r["times_ms"]), r["e2e_ms"]], dist, "cuda")
        line = prefill_line(wl, r, ws, steps, args.warmup, total_ms, e2e_ms, peaks)
        if rank == 0 and ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = run_cpu_baseline(wl.name, args.cpu_seconds)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    r = measure(wl, inp, args.steps, args.warmup, flush_bytes, dist=dist, sampler=sampler,
                e2e_steps=max(3, min(args.steps, 200)))
    total_ms, e2e_ms = max_over_ranks([sum(r["times_ms"]), r["e2e_ms"]], dist, "cuda")
    K = args.steps
    alg = r["bytes"]["algorithmic"]
    value = job_value(ws, alg, K, total_ms)
    per = sorted(r["times_ms"])
    us_med = 1e3 * per[len(per) // 2]
    achieved = alg / (total_ms / K / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (round(PAGES_US_PER_CALL[wl.name] / (1e3 * total_ms / K), 2)
                        if wl.name in PAGES_US_PER_CALL else None),
        "dtype": "bf16" if wl.kv_dtype == "bf16" else "f16 (int8 KV dequantized exactly)", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "head_dim": wl.D,
                   "ctx": wl.max_ctx, "q_len": wl.q_len, "layout": wl.layout, "kv_dtype": wl.kv_dtype,
                   "num_splits": r["S"], "accum": "fp32",
                   "l2": f"flushed before every step ({flush_bytes >> 20} MiB write + {flush_bytes >> 20} MiB read, "
                         "outside the timed pair)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "us_per_call": {"mean": round(1e3 * total_ms / K, 3), "median": round(us_med, 3),
                        "p10": round(1e3 * per[len(per) // 10], 3), "p90": round(1e3 * per[9 * len(per) // 10], 3)},
        "bytes_per_call": r["bytes"],
        "roofline": {"bound": "hbm", "kernel": "split_kernel (+ combine_kernel when S > 8), events around the call",
                     "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                     "traffic": ncu_traffic(wl.name)},
        "e2e": {"value": round(job_value(ws, alg, 1, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": r["launches_per_step"] * K,
        "clocks": r["clocks"],
    }
    if wl.name in PAGES_US_PER_CALL:
        line["vs_baseline_basis"] = "pages' fa_split_gqa_kernel 1.11 ms/call on RTX 5090, same workload (µs ratio)"
    if wl.name == HEADLINE and rank == 0 and not args.no_gates:
        line["gates"] = measure_gates(peaks, flush_bytes, max(20, min(args.steps, 200)), max(3, args.warmup))
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline(wl.name, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if args.suite and rank == 0:
        for name, other in WORKLOADS.items():
            if name == wl.name:
                continue
            oi = make_inputs(other)
            if other.kind == "prefill":
                rr = measure_prefill(other, oi, 20, 3, flush_bytes)
                t = sorted(rr["times_ms"])
                med = t[len(t) // 2]
                tf = rr["work"]["flops"] / (med / 1e3) / 1e12
                print(json.dumps({"suite": name, "us_per_call_median": round(1e3 * med, 3),
                                  "achieved_tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                                  "work": rr["work"]}), flush=True)
                del oi
                continue
            rr = measure(other, oi, 50, 5, flush_bytes)
            t = sorted(rr["times_ms"])
            med = t[len(t) // 2]
            a = rr["bytes"]["algorithmic"] / (med / 1e3) / 1e9
            print(json.dumps({"suite": name, "us_per_call_median": round(1e3 * med, 3),
                              "achieved_gbs": round(a, 1), "frac_of_peak": round(a / peaks["hbm_gbs"], 4),
                              "strict_gbs": round(rr["bytes"]["strict"] / (med / 1e3) / 1e9, 1),
                              "num_splits": rr["S"], "bytes": rr["bytes"]}), flush=True)
            del oi
    if dist is not None:
        dist.destroy_process_group()


def reference(args):
    """The reference arm: the fp64 CPU oracle, one bounded sample per step."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import numpy as np  # noqa: F401

    import oracle
    from gqa_split_kv_gb300.workloads import WORKLOADS, make_inputs

    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl)
    groups = [(b, g) for b in range(wl.B) for g in range(wl.Hkv)]

    def step(i):
        b, g = groups[i % len(groups)]
        return oracle_unit(oracle, wl, inp, b, g)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    nbytes = sum(step(i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    pre = wl.kind == "prefill"
    v = nbytes / dt / (1e12 if pre else 1e9)
    unit = "TFLOP/s" if pre else "GB/s"
    cores = os.cpu_count() or 1
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC if pre else METRIC, "value": round(v, 6), "unit": unit,
        "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "head_dim": wl.D, "ctx": wl.max_ctx,
                   "layout": wl.layout},
        "cpu_baseline": {"value": round(v, 6), "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": ("per step: one query head of one sequence over the whole chunk" if pre else
                                    "per step: all G query heads of one (sequence, KV head) over its full context")},
        "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.cpu_child:
        cpu_child(args.cpu_child, args.cpu_seconds)
        return
    if args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
