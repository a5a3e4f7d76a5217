"""Benchmark of the attention forward hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  1. prefill: llama7b_causal — B=1, Hq=Hkv=32, N=8192, d=128, causal, K drawn x2;
  2. decode:  decode_cache   — B=64, Hq=32, Hkv=8, d=128, cache capacity 8192,
              per-sequence length uniform in [512, 8192], split-KV + combine.
Inputs are resident in HBM when the timed region starts and larger than the
129 MB L2 (prefill Q/K/V/O 256 MB, decode caches 2.1 GB), so no L2 flush is
needed between steps.

The headline ``value`` is prefill TFLOP/s over the algorithmic work (4*d
FLOPs per visible (query, key) pair), timed with CUDA events around every
prefill launch on the launching stream; the ``decode`` object reports decode
GB/s over the algorithmic bytes (each cached K/V byte of a sequence's valid
range once per KV head, plus q, o and LSE).  ``e2e`` repeats each measurement
through the public API with the step's inputs copied from pinned host memory
and the result copied back inside the timed region.

``--impl reference`` times the fp64 CPU oracle on the host cores instead, on
a bounded sample of rows of the same prefill workload, in the same unit.
Multi-GPU (torchrun): replicas — every rank runs the same step on its own
GPU, no collective on the data path; value sums the ranks' work over the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from fa_workloads import (BERT_VARLEN, DECODE_CACHE, GQA_WINDOW, LLAMA7B_CAUSAL, TINY_MHA,  # noqa: E402
                          make_decode, make_prefill)

METRIC = "attention fwd TFLOP/s (prefill) & decode GB/s on 1 GB300, % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_NOTE = "inputs larger than L2 (prefill Q/K/V/O 256 MB, decode K/V cache 2.1 GB); no flush"
PREFILL_KERNEL_SOURCES = ["flashattention_forward_fa_gb300/csrc/fa_prefill.cu",
                          "flashattention_forward_fa_gb300/csrc/fa_items.cuh",
                          "flashattention_forward_fa_gb300/csrc/sm103_ptx.cuh"]
DECODE_KERNEL_SOURCES = ["flashattention_forward_fa_gb300/csrc/fa_decode.cu",
                         "flashattention_forward_fa_gb300/csrc/sm103_ptx.cuh"]


# ----------------------------------------------------------------------------- work accounting

def visible_pairs(len_q, len_k, causal: bool, window: int) -> int:
    """Number of (query, key) pairs the mask lets through, summed over sequences (one head)."""
    total = 0
    for lq, lk in zip(len_q, len_k):
        if lq <= 0 or lk <= 0:
            continue
        p = np.arange(lq, dtype=np.int64) + (lk - lq)
        lo = np.zeros(lq, dtype=np.int64)
        hi = np.full(lq, lk, dtype=np.int64)
        if causal:
            hi = np.minimum(hi, p + 1)
            if window > 0:
                lo = np.maximum(lo, p - window + 1)
        elif window > 0:
            lo = np.maximum(lo, p - window + 1)
            hi = np.minimum(hi, p + window)
        total += int(np.maximum(hi - lo, 0).sum())
    return total


def prefill_flops(case, len_q, len_k) -> float:
    return 4.0 * case.d * case.Hq * visible_pairs(len_q, len_k, case.causal, case.window)


def decode_bytes(case, lens) -> float:
    kv = 0
    for n in lens:
        n = max(0, min(n, case.Ncap))
        eff = min(n, case.window) if case.window > 0 else n
        kv += eff * case.Hkv * case.d * 2 * 2          # K and V, bf16, once per KV head
    qo = 2 * case.B * case.Hq * case.d * 2            # q in, o out (bf16)
    return float(kv + qo + case.B * case.Hq * 4)       # + LSE (fp32)


# ----------------------------------------------------------------------------- environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_traffic(summary_name: str, sources) -> float | None:
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", summary_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = re.search(r"^source_sha256:\s*([0-9a-f]{64})", text, re.M)
    val = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    if not sha or not val or sha.group(1) != source_sha(sources):
        return None
    return float(val.group(1))


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.5)  # let the sampler start before the timed region
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU baseline (oracle)

_ORACLE_CACHE: dict = {}


def oracle_sample_rate(target_s: float, seed: int = 0):
    """Time the fp64 oracle on a bounded random sample of llama7b_causal rows.

    Returns (TFLOP/s, seconds, rows, threads).  The sample size is calibrated so the
    timed part takes about ``target_s`` seconds of wall time on the host cores."""
    import oracle
    from fa_workloads import bf16_bits
    case = LLAMA7B_CAUSAL
    if "inputs" not in _ORACLE_CACHE:
        x = make_prefill(case)
        _ORACLE_CACHE["inputs"] = (x, *(bf16_bits(t.reshape(-1, t.shape[-2], t.shape[-1])) for t in (x.q, x.k, x.v)))
    x, qb, kb, vb = _ORACLE_CACHE["inputs"]
    rng = np.random.default_rng(seed)
    threads = oracle.max_threads()

    def run(n):
        rows = np.stack([np.zeros(n, np.int64), rng.integers(0, case.Hq, n), rng.integers(0, case.Nq, n)], 1)
        flops = float(4 * case.d * (rows[:, 2] + 1).sum())          # causal, Nq = Nk: row i sees i + 1 keys
        t0 = time.perf_counter()
        oracle.attention_rows(qb, kb, vb, x.q_off, x.len_q, x.k_off, x.len_k, case.softmax_scale, True, 0,
                              rows.astype(np.int32))
        return flops, time.perf_counter() - t0

    f, s = run(max(threads, 8))
    rate = f / max(s, 1e-6)
    n = int(max(threads, min(case.Hq * case.Nq, target_s * rate / (4 * case.d * case.Nq / 2))))
    f, s = run(n)
    return f / s / 1e12, s, n, threads


# ----------------------------------------------------------------------------- GPU arm

LAST_STATS: dict = {}  # per-fn median / min of the last time_steps call


def time_steps(fns, steps: int, stream):
    """Run ``steps`` steps; each step calls every fn in order.  Events around each fn on the
    launching stream.  Returns (per-fn mean ms, total region ms); per-fn median and min are left
    in LAST_STATS."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)] for _ in range(steps)]
    torch.cuda.synchronize()
    for s in range(steps):
        evs[s][0].record(stream)
        for i, fn in enumerate(fns):
            fn()
            evs[s][i + 1].record(stream)
    torch.cuda.synchronize()
    times = [[evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)] for i in range(len(fns))]
    per = [sum(t) / steps for t in times]
    LAST_STATS["median"] = [statistics.median(t) for t in times]
    LAST_STATS["min"] = [min(t) for t in times]
    total = evs[0][0].elapsed_time(evs[-1][-1])
    return per, total


def pipelined_e2e(run, host_in, dev_in, dev_out, host_out, steps: int, dev) -> float:
    """``steps`` end-to-end steps through the public API with two device buffer sets: step s copies
    its inputs from pinned host memory (one copy stream per input tensor, so the copies can run in
    parallel), runs ``run(s % 2)`` (compute stream) and copies its results back (a result stream),
    so step s+1's input copies and step s-1's result copies overlap step s's kernels.  Returns ms
    per step, timed with CUDA events from the first input copy to the last result copy."""
    s_in = [torch.cuda.Stream(dev) for _ in host_in]
    s_out = torch.cuda.Stream(dev)
    s_cmp = torch.cuda.current_stream(dev)
    ev_in = [[torch.cuda.Event() for _ in host_in] for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    start.record(s_cmp)
    for s in s_in + [s_out]:
        s.wait_stream(s_cmp)                          # nothing starts before the start event
    for st in range(steps):
        b = st % 2
        for j, (d, h) in enumerate(zip(dev_in[b], host_in)):
            with torch.cuda.stream(s_in[j]):
                if st >= 2:
                    s_in[j].wait_event(ev_run[b])     # step st-2 no longer reads these inputs
                d.copy_(h, non_blocking=True)
                ev_in[b][j].record(s_in[j])
        for j in range(len(host_in)):
            s_cmp.wait_event(ev_in[b][j])
        if st >= 2:
            s_cmp.wait_event(ev_out[b])               # step st-2's results have been copied out
        run(b)
        ev_run[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[b])
            for h, d in zip(host_out[b], dev_out[b]):
                h.copy_(d, non_blocking=True)
            ev_out[b].record(s_out)
    s_cmp.wait_stream(s_out)
    for s in s_in:
        s_cmp.wait_stream(s)
    end.record(s_cmp)
    torch.cuda.synchronize(dev)
    return start.elapsed_time(end) / steps


def gpu_arm(args, world, rank, local):
    import flashattention_forward_fa_gb300 as fa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    pc, dc = LLAMA7B_CAUSAL, DECODE_CACHE
    if args.only:
        return single_kernel_run(args, dev, stream)
    px = make_prefill(pc)
    dx = make_decode(dc)
    q, k, v = px.q.to(dev), px.k.to(dev), px.v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((pc.B, pc.Hq, pc.Nq), dtype=torch.float32, device=dev)
    dq, kc, vc = dx.q.to(dev), dx.k_cache.to(dev), dx.v_cache.to(dev)
    lens_host = list(dx.lens)
    lens = torch.tensor(lens_host, dtype=torch.int32, device=dev)
    do = torch.empty_like(dq)
    dl = torch.empty((dc.B, dc.Hq), dtype=torch.float32, device=dev)
    S = fa.fa_decode_max_splits(dc.B, dc.Hq, dc.Hkv, dc.Ncap, dc.window, lens_host, 0)
    ws = torch.empty((fa.decode_workspace_size(dc.B, dc.Hq, dc.d, S) + 3) // 4, dtype=torch.float32, device=dev)

    def prefill():
        fa.fa_fwd(q, k, v, causal=pc.causal, window=pc.window, scale=pc.softmax_scale, out=o, lse=lse)

    def decode():
        fa.fa_decode(dq, kc, vc, lens, window=dc.window, scale=dc.softmax_scale, seqlens_k_host=lens_host,
                     workspace=ws, out=do, lse=dl)

    for _ in range(args.warmup):
        prefill()
        decode()
    torch.cuda.synchronize()
    if fa.fa_device_status() != 0:
        raise RuntimeError("a kernel wait timed out during warm-up")
    barrier(world)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        (pre_ms, dec_ms), total_ms = time_steps([prefill, decode], args.steps, stream)
        (pre_med, dec_med), (pre_min, dec_min) = LAST_STATS["median"], LAST_STATS["min"]
    barrier(world)
    pre_ms_max = max_over_ranks(pre_ms, world)
    dec_ms_max = max_over_ranks(dec_ms, world)
    total_ms_max = max_over_ranks(total_ms, world)
    if fa.fa_device_status() != 0:
        raise RuntimeError("a kernel wait timed out during the timed region")

    flops = prefill_flops(pc, px.len_q, px.len_k)
    dbytes = decode_bytes(dc, lens_host)
    tflops = world * flops / (pre_ms_max * 1e-3) / 1e12
    gbs = world * dbytes / (dec_ms_max * 1e-3) / 1e9

    # end to end through the public API: every step copies its inputs in from pinned host memory,
    # runs, and copies its results back; copies and kernels of neighbouring steps overlap
    e2e_steps = max(4, min(20, args.steps))
    hq, hk, hv = (t.pin_memory() for t in (px.q, px.k, px.v))
    hdq = dx.q.pin_memory()
    hlens = torch.tensor(lens_host, dtype=torch.int32).pin_memory()
    p_in = [(q, k, v), tuple(torch.empty_like(t) for t in (q, k, v))]
    p_out = [(o, lse), (torch.empty_like(o), torch.empty_like(lse))]
    p_host_out = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (o, lse)) for _ in range(2)]
    d_in = [(dq, lens), (torch.empty_like(dq), torch.empty_like(lens))]
    d_out = [(do, dl), (torch.empty_like(do), torch.empty_like(dl))]
    d_host_out = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (do, dl)) for _ in range(2)]
    ws2 = torch.empty_like(ws)  # the second buffer set's decode workspace

    def prefill_into(b):
        (qi, ki, vi), (oi, li) = p_in[b], p_out[b]
        fa.fa_fwd(qi, ki, vi, causal=pc.causal, window=pc.window, scale=pc.softmax_scale, out=oi, lse=li)

    def decode_into(b):
        (qi, li_), (oi, lo) = d_in[b], d_out[b]
        fa.fa_decode(qi, kc, vc, li_, window=dc.window, scale=dc.softmax_scale, seqlens_k_host=lens_host,
                     workspace=ws if b == 0 else ws2, out=oi, lse=lo)

    pe_ms = pipelined_e2e(prefill_into, (hq, hk, hv), p_in, p_out, p_host_out, e2e_steps, dev)
    de_ms = pipelined_e2e(decode_into, (hdq, hlens), d_in, d_out, d_host_out, e2e_steps, dev)
    pe_ms = max_over_ranks(pe_ms, world)
    de_ms = max_over_ranks(de_ms, world)
    ho, hl = p_host_out[(e2e_steps - 1) % 2]
    hdo, hdl = d_host_out[(e2e_steps - 1) % 2]
    assert torch.equal(ho.to(dev), o), "end-to-end output differs from the device-resident run"
    assert torch.equal(hdo.to(dev), do), "end-to-end decode output differs from the device-resident run"
    p_h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    p_d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    d_h2d = hdq.numel() * hdq.element_size() + hlens.numel() * hlens.element_size()
    d_d2h = hdo.numel() * hdo.element_size() + hdl.numel() * hdl.element_size()

    peaks, peak_src = load_peaks()
    tr_pre = profile_traffic("fa_prefill_kernel_llama7b_causal.md", PREFILL_KERNEL_SOURCES)
    tr_dec = profile_traffic("fa_decode_split_kernel_decode_cache.md", DECODE_KERNEL_SOURCES)
    ach_pre = flops / (pre_ms * 1e-3) / 1e12          # this rank's launches
    ach_dec = dbytes / (dec_ms * 1e-3) / 1e9
    out = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms_max / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded randn, bf16)",
        "config": {
            "workload": "llama7b_causal prefill (B=1, Hq=Hkv=32, N=8192, d=128, causal, K x2) + "
                        "decode_cache (B=64, Hq=32, Hkv=8, d=128, cache 8192, len U[512,8192], split-KV)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": L2_NOTE,
            "prefill_flops_per_step": flops,
            "decode_bytes_per_step": dbytes,
            "prefill_ms": round(pre_ms_max, 4),
            "decode_ms": round(dec_ms_max, 4),
            "prefill_ms_median": round(pre_med, 4),
            "prefill_ms_min": round(pre_min, 4),
            "decode_ms_median": round(dec_med, 4),
            "decode_ms_min": round(dec_min, 4),
        },
        "roofline": {"bound": "tensor", "achieved": round(ach_pre, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(ach_pre / peaks["bf16_tflops"], 4),
                     "traffic": tr_pre, "peak_source": f"{peak_src} bf16 dense burst",
                     "kernel": "fa_prefill_kernel<128>"},
        "decode": {
            "value": round(gbs, 1), "unit": "GB/s", "ms": round(dec_ms_max, 4),
            "roofline": {"bound": "hbm", "achieved": round(ach_dec, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(ach_dec / peaks["hbm_gbs"], 4), "traffic": tr_dec,
                         "peak_source": f"{peak_src} HBM copy", "frac_of_8TBs_nominal": round(ach_dec / 8000.0, 4),
                         "kernel": "fa_decode_split_kernel<128> + fa_decode_combine_kernel<128>"},
            "e2e": {"value": round(world * dbytes / (de_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": d_h2d, "d2h_bytes_per_step": d_d2h,
                    "note": "KV cache is resident model state; the step's inputs are q and the lengths; "
                            "copies of neighbouring steps overlap the kernels (two buffer sets, copy streams)"},
        },
        "e2e": {"value": round(world * flops / (pe_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": p_h2d, "d2h_bytes_per_step": p_d2h,
                "note": "every step copies q, k, v in from pinned host memory and O, LSE back; copies of "
                        "neighbouring steps overlap the kernels (two buffer sets, copy streams)"},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_rows:
        out["rows"] = row_measurements(args, dev, stream, peaks,
                                       (pc, px, q, k, v, dc, dx, dq, kc, vc, lens, lens_host))
    return out


def single_kernel_run(args, dev, stream):
    """--only prefill|window|decode: warm-up then ``steps`` launches of one kernel workload
    (llama7b_causal, gqa_window or decode_cache), nothing else (no e2e, no CPU baseline, no clock
    sampling).  Used as the command under ncu."""
    import flashattention_forward_fa_gb300 as fa
    if args.only in ("prefill", "window"):
        pc = LLAMA7B_CAUSAL if args.only == "prefill" else GQA_WINDOW
        px = make_prefill(pc)
        q, k, v = px.q.to(dev), px.k.to(dev), px.v.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((pc.B, pc.Hq, pc.Nq), dtype=torch.float32, device=dev)
        fn = lambda: fa.fa_fwd(q, k, v, causal=pc.causal, window=pc.window, scale=pc.softmax_scale,  # noqa: E731
                               out=o, lse=lse)
        work, unit = prefill_flops(pc, px.len_q, px.len_k) / 1e12, "TFLOP/s"
    else:
        dc = DECODE_CACHE
        dx = make_decode(dc)
        dq, kc, vc = dx.q.to(dev), dx.k_cache.to(dev), dx.v_cache.to(dev)
        lens = torch.tensor(dx.lens, dtype=torch.int32, device=dev)
        do = torch.empty_like(dq)
        dl = torch.empty((dc.B, dc.Hq), dtype=torch.float32, device=dev)
        fn = lambda: fa.fa_decode(dq, kc, vc, lens, scale=dc.softmax_scale, seqlens_k_host=dx.lens,  # noqa: E731
                                  out=do, lse=dl)
        work, unit = decode_bytes(dc, dx.lens) / 1e9, "GB/s"
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    (ms,), _ = time_steps([fn], args.steps, stream)
    ok = fa.fa_device_status() == 0
    return {"partial": True, "only": args.only, "value": round(work / (ms * 1e-3), 2), "unit": unit,
            "ms": round(ms, 4), "steps": args.steps, "warmup": args.warmup, "status_ok": ok}


# ----------------------------------------------------------------------------- the other workloads and options

def time_alone(fn, steps: int, warmup: int, stream) -> float:
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    (ms,), _ = time_steps([fn], steps, stream)
    return ms


def row_measurements(args, dev, stream, peaks, step_inputs):
    """The workloads other than the step's own and the option paths (several new tokens over a
    KV cache, a paged cache, RoPE, ALiBi), each timed alone with CUDA events on the launching
    stream after its own warm-up.  Prefill rows count algorithmic FLOPs (4 d per visible pair),
    decode-like rows algorithmic bytes (each valid cached K/V byte once per KV head, q, o, LSE)."""
    import flashattention_forward_fa_gb300 as fa
    steps, warm = max(3, min(args.steps, 50)), max(3, args.warmup)
    tf_peak, gb_peak = peaks["bf16_tflops"], peaks["hbm_gbs"]
    rows = {}

    def add(name, workload, ms, work, unit, bound, l2):
        val = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
        peak = tf_peak if bound == "tensor" else gb_peak
        rows[name] = {"workload": workload, "ms": round(ms, 4), "value": round(val, 2), "unit": unit,
                      "bound": bound, "frac": round(val / peak, 4), "inputs_vs_l2": l2}

    def prefill_row(name, case, desc, l2, graph=False, **kw):
        x = make_prefill(case)
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        o_pre = torch.empty_like(q)
        if case.layout == "packed":
            cu = torch.tensor([0] + list(np.cumsum(x.len_q)), dtype=torch.int32, device=dev)
            # the batch's metadata, prepared once as a serving loop holds it: the host copy of
            # cu_seqlens as an int32 CPU tensor (passed by address) and the maximum lengths as ints
            host = torch.tensor([0] + [int(c) for c in np.cumsum(x.len_q)], dtype=torch.int32)
            max_q, max_k = int(max(x.len_q)), int(max(x.len_k))
            l_pre = torch.empty((case.Hq, q.shape[0]), dtype=torch.float32, device=dev)

            def fn(out=None, lse=None):
                return fa.fa_fwd_varlen(q, k, v, cu, cu, max_q, max_k, causal=case.causal,
                                        window=case.window, scale=case.softmax_scale, cu_seqlens_q_host=host,
                                        out=out, lse=lse)
        else:
            l_pre = torch.empty((case.B, case.Hq, case.Nq), dtype=torch.float32, device=dev)

            def fn(out=None, lse=None):
                return fa.fa_fwd(q, k, v, causal=case.causal, window=case.window, scale=case.softmax_scale,
                                 out=out, lse=lse, **kw)
        work = prefill_flops(case, x.len_q, x.len_k)
        add(name, desc, time_alone(fn, steps, warm, stream), work, "TFLOP/s", "tensor", l2)
        if graph:
            # launch-bound: the same call with the outputs allocated once (a serving loop's form: no
            # allocation per call), its host time per call, and replays of a captured CUDA graph
            # (no host work per call)
            pre = lambda: fn(out=o_pre, lse=l_pre)  # noqa: E731
            ms_pre = time_alone(pre, steps, warm, stream)
            rows[name]["prealloc_ms_per_call"] = round(ms_pre, 5)
            torch.cuda.synchronize()
            n_host = 200
            t0 = time.perf_counter()
            for _ in range(n_host):
                pre()
            rows[name]["prealloc_host_us_per_call"] = round((time.perf_counter() - t0) / n_host * 1e6, 2)
            torch.cuda.synchronize()
            # back to back: one event pair around n_host calls, as a loop that issues call after
            # call sees them (the per-call events above add their own host time to every call)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for alloc_name, call in (("b2b_ms_per_call", fn), ("prealloc_b2b_ms_per_call", pre)):
                torch.cuda.synchronize()
                ev0.record(stream)
                for _ in range(n_host):
                    call()
                ev1.record(stream)
                torch.cuda.synchronize()
                rows[name][alloc_name] = round(ev0.elapsed_time(ev1) / n_host, 5)
            reps = 20
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(reps):
                    pre()
            g.replay()
            torch.cuda.synchronize()
            (gms,), _ = time_steps([g.replay], max(3, steps // reps), stream)
            rows[name]["graph_ms_per_call"] = round(gms / reps, 5)
            rows[name]["graph_value"] = round(work / (gms / reps * 1e-3) / 1e12, 2)

    prefill_row("tiny_mha", TINY_MHA, "B=1, H=2, N=256, d=64, non-causal (launch-bound)", "inside L2", graph=True)
    prefill_row("bert_varlen", BERT_VARLEN, "B=8, H=12, d=64, len U[128,512] packed, non-causal", "inside L2",
                graph=True)
    prefill_row("gqa_window", GQA_WINDOW, "B=4, Hq=32, Hkv=8, N=4096, d=128, causal, window 1024",
                "larger than L2 (320 MB)")

    pc, px, q, k, v, dc, dx, dq, kc, vc, lens, lens_host = step_inputs
    o = torch.empty_like(q)
    # ALiBi on the step's prefill and decode workloads
    slopes = torch.tensor(fa.alibi_slopes(pc.Hq), dtype=torch.float32, device=dev)
    flops = prefill_flops(pc, px.len_q, px.len_k)
    ms = time_alone(lambda: fa.fa_fwd(q, k, v, causal=True, scale=pc.softmax_scale, out=o, alibi_slopes=slopes),
                    steps, warm, stream)
    add("alibi_prefill", "llama7b_causal + ALiBi (geometric slopes)", ms, flops, "TFLOP/s", "tensor",
        "larger than L2")
    dslopes = torch.tensor(fa.alibi_slopes(dc.Hq), dtype=torch.float32, device=dev)
    do = torch.empty_like(dq)
    dbytes = decode_bytes(dc, lens_host)
    ms = time_alone(lambda: fa.fa_decode(dq, kc, vc, lens, scale=dc.softmax_scale, seqlens_k_host=lens_host,
                                         out=do, alibi_slopes=dslopes), steps, warm, stream)
    add("alibi_decode", "decode_cache + ALiBi", ms, dbytes, "GB/s", "hbm", "larger than L2 (2.1 GB)")

    # RoPE: Q rotated inside the prefill kernel (K rotated once beforehand, as in a cache) ...
    cos_t, sin_t = fa.rope_tables(pc.Nk, pc.d, device=dev)
    kr = k.clone()
    fa.fa_rope(kr, torch.arange(pc.Nk, dtype=torch.int32, device=dev).repeat(pc.B), (cos_t, sin_t))
    ms = time_alone(lambda: fa.fa_fwd(q, kr, v, causal=True, scale=pc.softmax_scale, out=o, rope=(cos_t, sin_t)),
                    steps, warm, stream)
    add("rope_prefill", "llama7b_causal, Q rotated in the kernel (rotary_dim 128)", ms, flops, "TFLOP/s", "tensor",
        "larger than L2")
    # the same work in two passes, for comparison: Q rotated in place by fa_rope (as a model would rotate
    # its fresh Q projection; a copy is rotated again each time, which changes no cost), then the
    # plain kernel
    qr = q.clone()
    qpos = torch.arange(pc.Nq, dtype=torch.int32, device=dev).repeat(pc.B)

    def two_pass():
        fa.fa_rope(qr, qpos, (cos_t, sin_t))
        fa.fa_fwd(qr, kr, v, causal=True, scale=pc.softmax_scale, out=o)

    ms = time_alone(two_pass, steps, warm, stream)
    add("rope_prefill_two_pass", "the same work in two launches: fa_rope on Q in place, then the plain kernel",
        ms, flops, "TFLOP/s", "tensor", "larger than L2")
    del kr, qr
    # ... and the in-place rotation pass itself over a 256 MB K block (4 x 8192 rows)
    xr = torch.randn(4 * pc.Nk, pc.Hkv, pc.d, device=dev).to(torch.bfloat16)
    pos = torch.arange(pc.Nk, dtype=torch.int32, device=dev).repeat(4)
    ms = time_alone(lambda: fa.fa_rope(xr, pos, (cos_t, sin_t)), steps, warm, stream)
    rbytes = 2 * xr.numel() * 2 + pos.numel() * 4
    add("rope_k", "fa_rope in place, [32768, 32, 128] bf16, rotary_dim 128", ms, rbytes, "GB/s", "hbm",
        "larger than L2 (256 MB)")
    del xr

    # several new tokens per sequence over the decode cache (speculative decoding, 4 drafts)
    nt = 4
    g = torch.Generator("cpu").manual_seed(6)
    mq = torch.randn(dc.B, nt, dc.Hq, dc.d, generator=g).to(torch.bfloat16).to(dev)
    mo = torch.empty_like(mq)
    ml = torch.empty((dc.B, dc.Hq, nt), dtype=torch.float32, device=dev)
    S = fa.fa_decode_max_splits(dc.B, dc.Hq, dc.Hkv, dc.Ncap, 0, lens_host, 0)
    mws = torch.empty((fa.decode_workspace_size(dc.B * nt, dc.Hq, dc.d, S) + 3) // 4, dtype=torch.float32,
                      device=dev)
    mbytes = decode_bytes(dc, lens_host) + (nt - 1) * (2 * dc.B * dc.Hq * dc.d * 2 + dc.B * dc.Hq * 4)
    ms = time_alone(lambda: fa.fa_decode(mq, kc, vc, lens, scale=dc.softmax_scale, seqlens_k_host=lens_host,
                                         workspace=mws, out=mo, lse=ml), steps, warm, stream)
    add("multitoken_decode", "decode_cache with 4 new tokens per sequence (bottom-right causal), split-KV decode "
        "kernel", ms, mbytes, "GB/s", "hbm", "larger than L2 (2.1 GB)")
    ms = time_alone(lambda: fa.fa_fwd(mq, kc, vc, causal=True, scale=dc.softmax_scale, seqlens_k=lens, out=mo),
                    steps, warm, stream)
    add("multitoken_decode_prefill_kernel", "the same through fa_fwd with seqlens_k (128-row Q tiles, 4 used)", ms,
        mbytes, "GB/s", "hbm", "larger than L2 (2.1 GB)")
    del mq, mo, mws

    # the decode cache scattered over a page pool (128-token pages in random order)
    page = 128
    nb = dc.Ncap // page
    perm = torch.randperm(dc.B * nb, generator=g).to(dev)
    kp = torch.empty((dc.B * nb, page, dc.Hkv, dc.d), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    kp[perm] = kc.view(dc.B * nb, page, dc.Hkv, dc.d)
    vp[perm] = vc.view(dc.B * nb, page, dc.Hkv, dc.d)
    table = perm.view(dc.B, nb).to(torch.int32).contiguous()
    ms = time_alone(lambda: fa.fa_decode_paged(dq, kp, vp, table, lens, scale=dc.softmax_scale,
                                               seqlens_k_host=lens_host, out=do), steps, warm, stream)
    add("paged_decode", "decode_cache over 128-token pages in random order", ms, dbytes, "GB/s", "hbm",
        "larger than L2 (2.1 GB)")
    del kp, vp
    torch.cuda.synchronize()
    if fa.fa_device_status() != 0:
        raise RuntimeError("a kernel reported an error while the workload rows ran")
    rows["note"] = f"each row {steps} launches after {warm} warm-up; frac against the measured peaks"
    return rows


# ----------------------------------------------------------------------------- reference arm (oracle on CPU)

def reference_arm(args, world, rank):
    """The fp64 oracle as it stands, on the host cores, on bounded samples of the prefill workload."""
    if rank != 0:
        return None
    budget_s = 120.0                                   # the whole --steps/--warmup run
    per_step = max(0.05, min(10.0, budget_s / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample_rate(per_step / 4, seed=1)
    rates, secs, rows = [], [], 0
    for s in range(args.steps):
        r, t, n, threads = oracle_sample_rate(per_step / 2, seed=100 + s)
        rates.append(r)
        secs.append(t)
        rows += n
    value = statistics.median(rates)
    sample = (f"{rows // max(1, args.steps)} random rows per step of llama7b_causal (b=0, random head and "
              f"query row; each row = full causal softmax over its visible keys), fp64")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.mean(secs), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded randn, bf16 inputs widened exactly to fp64)",
        "config": {"workload": "llama7b_causal prefill (B=1, Hq=Hkv=32, N=8192, d=128, causal, K x2), "
                               "sampled rows", "parallelism": "host cores (OpenMP over rows)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", choices=["prefill", "window", "decode"], default=None,
                    help="run one phase alone (for profilers); prints a partial line")
    ap.add_argument("--no-rows", action="store_true",
                    help="skip the per-workload rows (other workloads and option paths) after the step")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=12.0,
                    help="wall time of the oracle CPU baseline sample (rank 0, N=1)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        out = reference_arm(args, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    out = gpu_arm(args, world, rank, local)
    if rank == 0:
        if world == 1 and not args.only:
            r, t, n, threads = oracle_sample_rate(args.cpu_baseline_seconds)
            out["cpu_baseline"] = {
                "value": round(r, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "sample": f"{n} random rows of llama7b_causal (b=0, random head/row, full causal row each), "
                          f"fp64, {t:.1f} s on {threads} host threads"}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
