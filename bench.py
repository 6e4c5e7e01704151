"""Benchmark of the tiled exact attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  * causal prefill forward (fa_fwd) on B=4, Hq=Hkv=16, N=4096, d=128, bf16;
  * split-KV decode (fa_fwd_splitkv: one split kernel whose last CTA per head
    group merges the splits' partials, LSE-weighted) on
    B=8, Hq=32, Hkv=8, KV length 32768, d=128, bf16, query position 32767.
`value` is the prefill's forward TFLOP/s (4 * d * visible (query, key) pairs *
b * hq per launch, over that launch's CUDA-event time); the decode's KV GB/s is
reported beside it.  L2 is flushed (a 256 MiB write) before every step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload.  With N > 1 (torchrun) every rank runs an
independent replica; the line reports the total over ranks and the slowest
rank's time.

Every roofline divides by the measured burst bf16 GEMM peak (each launch lasts
well under a millisecond, between L2 flushes); the sustained peak is reported
beside it.  `--only NAME[,NAME...]` times just the named lines (prefill, decode,
gqa_long, ragged_d64, ragged_d256, backward, e4m3, e4m3_d64, e4m3_d256, paged, decode_e4m3, variants,
decode_b1, decode_d64, e2e, link) and prints them as one JSON object: the form the ncu captures use.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fwd TFLOP/s & % bf16 tensor peak (prefill); decode KV GB/s & % HBM BW"
PREFILL = "causal_prefill"
DECODE = "decode"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _peak_tflops():
    """(burst bf16 TFLOP/s, sustained bf16 TFLOP/s, source)."""
    peaks, src = _peaks()
    burst = float(peaks["bf16_tflops"])
    return burst, float(peaks.get("bf16_tflops_sustained", burst)), src


def _tensor_roofline(tflops, kernel=None, traffic=None, ratio=1.0, dtype_note=""):
    """Roofline object of a tensor-core line against the burst peak (times `ratio` for another dtype)."""
    burst, sustained, src = _peak_tflops()
    pk = burst * ratio
    r = {"bound": "tensor", "achieved": round(tflops, 2), "peak": round(pk, 1), "unit": "TFLOP/s",
         "frac": round(tflops / pk, 4), "traffic": traffic,
         "peak_source": f"{src} bf16 burst GEMM{dtype_note} (launches of well under a millisecond)",
         "frac_of_sustained": round(tflops / (sustained * ratio), 4)}
    if kernel:
        r["kernel"] = kernel
    return r


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# The sources each profiled kernel family is compiled from: a capture stays valid
# while these files are unchanged.
KERNEL_SOURCES = {
    "fa_prefill_kernel": ("fa_prefill.cu", "ptx.cuh", "fa_internal.h", "tc_common.cuh"),
    "fa_decode_kernel": ("fa_decode.cu", "ptx.cuh", "fa_internal.h"),
    "fa_bwd_": ("fa_backward.cu", "ptx.cuh", "fa_internal.h", "tc_common.cuh"),
}


def _kernel_source_hash(kernel: str) -> str | None:
    family = next((k for k in KERNEL_SOURCES if kernel.startswith(k)), None)
    if family is None:
        return None
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, "tiled_exact_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    want = _kernel_source_hash(kernel)
    if want is None:
        return None
    with open(p) as f:
        for line in f:
            parts = line.strip().strip("|").split("|")
            parts = [x.strip() for x in parts]
            if len(parts) >= 3 and parts[0] == kernel and parts[1] == want:
                try:
                    return int(float(parts[2]))
                except ValueError:
                    return None
    return None


def reduce_max_over_ranks(values, dist_mod, device):
    """Element-wise maximum of per-rank timings (the slowest rank sets the job time)."""
    import torch

    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(units_per_rank: float, world_size: int, ms: float) -> float:
    """Whole-job units per second: every rank processes `units_per_rank` in at most `ms`."""
    return units_per_rank * world_size / (ms * 1e-3)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.5)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sms, maxs, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        sms_sorted = sorted(sms)
        med = sms_sorted[len(sms_sorted) // 2] if sms_sorted else None
        return {"sm_mhz": med, "sm_max_mhz": max(maxs) if maxs else None, "reasons": sorted(reasons),
                "samples": len(sms), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------------- our implementation


def _setup(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__

    ws, rank, local = _dist()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    __graft_entry__.build()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    return ws, rank, dev, flush


SECONDARY = ("gqa_long", "ragged_d64", "ragged_d256", "paged", "decode_e4m3", "backward", "e4m3", "e4m3_d64", "e4m3_d256",
             "variants", "decode_b1", "decode_d64", "e2e", "link")


def run_only(args):
    """Time only the named lines (no timed step): what the ncu captures run."""
    import torch

    names = [x for x in args.only.split(",") if x]
    _, _, dev, flush = _setup(args)
    steps = max(1, args.steps)
    out = {}
    for nm in names:
        if nm in ("prefill", "decode"):
            w = WORKLOADS_LAZY()[PREFILL if nm == "prefill" else DECODE]
            out[nm] = bench_config(dev, flush, w, steps=steps, warmup=args.warmup)
        elif nm in ("gqa_long", "ragged_d64", "ragged_d256"):
            out[nm] = bench_config(dev, flush, WORKLOADS_LAZY()[nm], steps=steps, warmup=args.warmup)
        elif nm == "paged":
            out[nm] = bench_paged_decode(dev, flush, steps=steps, warmup=args.warmup)
        elif nm == "backward":
            out[nm] = bench_backward(dev, flush, steps=steps, warmup=args.warmup)
        elif nm == "e4m3":
            out[nm] = bench_e4m3(dev, flush, steps=steps, warmup=args.warmup)
        elif nm == "decode_e4m3":
            out[nm] = bench_decode_e4m3(dev, flush, steps=steps, warmup=args.warmup)
        elif nm in ("e4m3_d64", "e4m3_d256"):
            out[nm] = bench_e4m3(dev, flush, steps=steps, warmup=args.warmup, workload="ragged_" + nm[5:])
        elif nm == "variants":
            out[nm] = bench_variants(dev, flush, steps=steps)
        elif nm in SMALL_DECODES:
            out[nm] = bench_small_decode(dev, flush, nm, steps=steps)
        elif nm in ("e2e", "link"):
            from tiled_exact_attention_gb300 import fa_fwd
            from tiled_exact_attention_gb300.inputs import make_qkv

            wp = WORKLOADS_LAZY()[PREFILL]
            qc, kc, vc = make_qkv(wp)
            stream = torch.cuda.current_stream()
            if nm == "e2e":
                out[nm] = {"ms_per_step": round(bench_e2e(qc, kc, vc, wp, fa_fwd, flush, stream, steps), 4)}
            else:
                out[nm] = bench_link(qc, kc, vc, wp, stream, steps)
        else:
            raise SystemExit(f"unknown line {nm!r}; one of prefill, decode, {', '.join(SECONDARY)}")
    print(json.dumps({"only": out}), flush=True)


def WORKLOADS_LAZY():
    from tiled_exact_attention_gb300.inputs import WORKLOADS

    return WORKLOADS


def run_ours(args):
    import torch
    import torch.distributed as dist

    from tiled_exact_attention_gb300 import fa_fwd, fa_fwd_splitkv, fa_splitkv_default_splits, fa_sync_status
    from tiled_exact_attention_gb300.inputs import WORKLOADS, make_qkv

    ws, rank, dev, flush = _setup(args)

    wp, wd = WORKLOADS[PREFILL], WORKLOADS[DECODE]
    qc, kc, vc = make_qkv(wp)
    q, k, v = qc.to(dev), kc.to(dev), vc.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((wp.b, wp.hq, wp.sq), dtype=torch.float32, device=dev)
    dqc, dkc, dvc = make_qkv(wd)
    dq, dk, dv = dqc.to(dev), dkc.to(dev), dvc.to(dev)
    do = torch.empty_like(dq)
    dlse = torch.empty((wd.b, wd.hq, wd.sq), dtype=torch.float32, device=dev)
    ns = fa_splitkv_default_splits(dq, dk, dv, causal=True, q_pos_offset=wd.offset)
    from tiled_exact_attention_gb300.api import fa_splitkv_workspace_size

    wsb = fa_splitkv_workspace_size(dq, dk, dv, ns, causal=True, q_pos_offset=wd.offset)
    work = torch.empty(wsb, dtype=torch.uint8, device=dev)

    def prefill():
        fa_fwd(q, k, v, causal=True, q_pos_offset=wp.offset, out=o, lse=lse)

    def decode():
        fa_fwd_splitkv(dq, dk, dv, causal=True, q_pos_offset=wd.offset, num_splits=ns, workspace=work, out=do,
                       lse=dlse)

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        prefill()
        decode()
    st = fa_sync_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        evs[i][0].record(stream)
        prefill()
        evs[i][1].record(stream)
        decode()
        evs[i][2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop()
    st = fa_sync_status()
    if st != 0:
        raise RuntimeError(f"device status {st} in the timed region")
    pre_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(K)]
    dec_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(K)]
    pre_avg = sum(pre_ms) / K
    dec_avg = sum(dec_ms) / K
    step_ms = pre_avg + dec_avg
    del q, k, v, o, dq, dk, dv, do, work

    # ---- end-to-end through the public call with host buffers (prefill), and the link alone ----
    e2e_steps = max(3, min(50, K // 20))
    e2e_ms = bench_e2e(qc, kc, vc, wp, fa_fwd, flush, stream, e2e_steps, dist if ws > 1 else None)
    link = bench_link(qc, kc, vc, wp, stream, e2e_steps)

    few = max(10, min(100, K // 50))
    configs = {nm: bench_config(dev, flush, WORKLOADS[nm], steps=few) for nm in ("gqa_long", "ragged_d64",
                                                                                 "ragged_d256")}
    paged = bench_paged_decode(dev, flush, steps=max(20, min(500, K // 10)))
    dec8 = bench_decode_e4m3(dev, flush, steps=max(20, min(500, K // 10)))
    bwd = bench_backward(dev, flush, steps=few)
    e4m3 = bench_e4m3(dev, flush, steps=max(10, min(200, K // 25)))
    e4m3_rag = {f"e4m3_d{w}": bench_e4m3(dev, flush, steps=few, workload=f"ragged_d{w}") for w in (64, 256)}
    variants = bench_variants(dev, flush, steps=few)

    flops = 4.0 * wp.d * wp.visible_pairs_per_head() * wp.b * wp.hq
    kv_bytes = 2 * wd.b * wd.hkv * wd.skv * wd.d * 2
    dec_bytes = kv_bytes + 2 * (wd.b * wd.hq * wd.d * 2) + wd.b * wd.hq * 4

    if ws > 1:
        pre_avg, dec_avg, e2e_ms = reduce_max_over_ranks([pre_avg, dec_avg, e2e_ms], dist, dev)
        step_ms = pre_avg + dec_avg
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = _peaks()
    tflops = job_throughput(flops, ws, pre_avg) / 1e12
    per_gpu_tflops = flops / (pre_avg * 1e-3) / 1e12
    dec_gbs = dec_bytes / (dec_avg * 1e-3) / 1e9
    hbm = float(peaks["hbm_gbs"])
    h2d = sum(t.numel() * t.element_size() for t in (qc, kc, vc))
    d2h = wp.b * wp.sq * wp.hq * wp.d * 2 + wp.b * wp.hq * wp.sq * 4
    pre_traffic = _profiled_traffic("fa_prefill_kernel")
    dec_traffic = _profiled_traffic("fa_decode_kernel")
    e4 = dict(e4m3)
    e4["roofline"] = _tensor_roofline(e4m3["value"], kernel=e4m3["kernel"],
                                      traffic=_profiled_traffic("fa_prefill_kernel_e4m3"), ratio=2.0,
                                      dtype_note=" x 2 (the nominal fp8 : bf16 ratio)")
    for key, val in e4m3_rag.items():
        val["roofline"] = _tensor_roofline(val["value"], kernel=val["kernel"], ratio=2.0,
                                           traffic=_profiled_traffic("fa_prefill_kernel_" + key),
                                           dtype_note=" x 2 (the nominal fp8 : bf16 ratio)")
    bw = dict(bwd)
    bw["roofline"] = _tensor_roofline(bwd["value"], kernel="fa_bwd_dkdv_kernel (the larger of the two product kernels)",
                                      traffic=_profiled_traffic("fa_bwd_dkdv_kernel"))
    line = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: iid N(0,1) bf16 from seeded PCG64, no dataset",
        "config": {
            "workload": "causal prefill B=4 Hq=Hkv=16 N=4096 d=128 bf16 + split-KV decode B=8 Hq=32 Hkv=8 "
                        "KV=32768 d=128 bf16 (query position 32767)",
            "prefill": {"b": wp.b, "sq": wp.sq, "skv": wp.skv, "hq": wp.hq, "hkv": wp.hkv, "d": wp.d,
                        "causal": True, "flops_per_launch": flops, "ms": round(pre_avg, 4)},
            "decode": {"b": wd.b, "skv": wd.skv, "hq": wd.hq, "hkv": wd.hkv, "d": wd.d, "num_splits": ns,
                       "bytes_per_launch": dec_bytes, "ms": round(dec_avg, 4)},
            "l2": "flushed before every step (256 MiB write, outside the kernel events)",
            "parallelism": f"replicas x{ws} (independent problems per GPU)",
            "timing": "CUDA events per phase on the launching stream, mean over the timed steps",
        },
        "decode": {
            "value": round(dec_gbs, 1),
            "unit": "GB/s",
            "ms_per_step": round(dec_avg, 4),
            "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(dec_gbs / hbm, 4), "peak_source": f"{peak_src} copy bandwidth",
                         "traffic": dec_traffic, "spec_peak": 8000.0,
                         "frac_of_spec": round(dec_gbs / 8000.0, 4),
                         "note": "phase time = split kernel with the fused merge (+ a memset of its counters)"},
        },
        "gqa_long": configs["gqa_long"],
        "ragged_d64": configs["ragged_d64"],
        "ragged_d256": configs["ragged_d256"],
        "decode_paged": dict(paged, roofline={"bound": "hbm", "achieved": paged["value"], "peak": hbm,
                                              "unit": "GB/s", "frac": round(paged["value"] / hbm, 4),
                                              "peak_source": f"{peak_src} copy bandwidth", "traffic": None}),
        "decode_e4m3": dec8,
        "e4m3": e4,
        "e4m3_d64": e4m3_rag["e4m3_d64"],
        "e4m3_d256": e4m3_rag["e4m3_d256"],
        "backward": bw,
        "variants": variants,
        "roofline": dict(_tensor_roofline(per_gpu_tflops, kernel="fa_prefill_kernel<128, bf16>", traffic=pre_traffic),
                         spec_peak=2250.0, frac_of_spec=round(per_gpu_tflops / 2250.0, 4)),
        "clocks": clocks,
        "e2e": {"value": round(job_throughput(flops, ws, e2e_ms) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "copy_in_bound_ms": link["h2d_only_ms"],
                "frac_of_copy_bound": round(link["h2d_only_ms"] / e2e_ms, 4),
                "link": link,
                "what": "prefill through fa_fwd with pinned host Q/K/V copied in and O/LSE copied out each step; "
                        "pipelined over two buffer sets (step i + 1 copies in while step i computes and copies out); "
                        "copy_in_bound_ms = the step's inputs copied in alone, no computation: no step can be "
                        "shorter; frac_of_copy_bound = that over ms_per_step"},
        "gpu_launches": K * 2,
        "wall_s_timed_region": round(wall, 3),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def bench_config(dev, flush, w, steps=30, warmup=3):
    """One forward workload of the target set (the long causal GQA prefill, the ragged-tail d = 64 / 256
    forward passes; also the timed step's prefill and decode when asked alone), in TFLOP/s of the visible
    (query, key) pairs (4 d flops per pair and head) or, for the split-KV decode, KV GB/s."""
    import torch

    from tiled_exact_attention_gb300 import fa_fwd, fa_fwd_splitkv, fa_sync_status
    from tiled_exact_attention_gb300.inputs import make_qkv

    q, k, v = (t.to(dev) for t in make_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.b, w.hq, w.sq), dtype=torch.float32, device=dev)
    off = w.offset if w.causal else None
    if w.sq == 1:
        ms = _timed(lambda: fa_fwd_splitkv(q, k, v, causal=True, q_pos_offset=w.offset, out=o, lse=lse), flush,
                    steps, warmup)
        nbytes = 2 * w.b * w.hkv * w.skv * w.d * 2 + 2 * (w.b * w.hq * w.d * 2) + w.b * w.hq * 4
        gbs = nbytes / (ms * 1e-3) / 1e9
        hbm = float(_peaks()[0]["hbm_gbs"])
        return {"value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4), "bytes_per_launch": nbytes,
                "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                             "frac": round(gbs / hbm, 4), "traffic": _profiled_traffic("fa_decode_kernel")}}
    ms = _timed(lambda: fa_fwd(q, k, v, causal=w.causal, q_pos_offset=off, out=o, lse=lse), flush, steps, warmup)
    if fa_sync_status() != 0:
        raise RuntimeError(f"device status set by the {w.name} forward pass")
    flops = 4.0 * w.d * w.visible_pairs_per_head() * w.b * w.hq
    tf = flops / (ms * 1e-3) / 1e12
    dt = "bf16" if w.dtype == "bf16" else "fp16"
    kname = {"gqa_long": "fa_prefill_kernel_gqa", "causal_prefill": "fa_prefill_kernel"}.get(w.name, f"fa_prefill_kernel_d{w.d}")
    return {"value": round(tf, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4), "flops_per_launch": flops,
            "config": {"b": w.b, "sq": w.sq, "skv": w.skv, "hq": w.hq, "hkv": w.hkv, "d": w.d, "dtype": dt,
                       "std": w.std, "causal": w.causal},
            "roofline": _tensor_roofline(tf, kernel=f"fa_prefill_kernel<{w.d}, {dt}>",
                                         traffic=_profiled_traffic(kname),
                                         dtype_note=" (fp16 runs at the bf16 rate)" if dt == "fp16" else ""),
            "steps": steps}


def bench_link(qc, kc, vc, wp, stream, steps):
    """The host link alone: the end-to-end step's copies (pinned Q, K, V in on three streams, O and LSE out on a
    fourth), the same bytes and overlap, with no computation; plus each direction by itself."""
    import torch

    dev = stream.device
    h_in = [t.pin_memory() for t in (qc, kc, vc)]
    d_in = [torch.empty_like(t, device=dev) for t in (qc, kc, vc)]
    o = torch.empty(qc.shape, dtype=qc.dtype, device=dev)
    lse = torch.empty((wp.b, wp.hq, wp.sq), dtype=torch.float32, device=dev)
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    s_in = [torch.cuda.Stream(device=dev) for _ in range(3)]
    s_out = torch.cuda.Stream(device=dev)

    def both(n, do_in=True, do_out=True):
        for si in s_in + [s_out]:
            si.wait_stream(stream)
        for _ in range(n):
            if do_in:
                for j in range(3):
                    with torch.cuda.stream(s_in[j]):
                        d_in[j].copy_(h_in[j], non_blocking=True)
            if do_out:
                with torch.cuda.stream(s_out):
                    ho.copy_(o, non_blocking=True)
                    hl.copy_(lse, non_blocking=True)
        for si in s_in + [s_out]:
            stream.wait_stream(si)

    def timed(**kw):
        both(2, **kw)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        both(steps, **kw)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    h2d = sum(t.numel() * t.element_size() for t in (qc, kc, vc))
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
    ms = timed()
    ms_in = timed(do_out=False)
    ms_out = timed(do_in=False)
    return {"ms_per_step": round(ms, 4), "h2d_only_ms": round(ms_in, 4), "d2h_only_ms": round(ms_out, 4),
            "h2d_gbs": round(h2d / (ms_in * 1e-3) / 1e9, 1), "d2h_gbs": round(d2h / (ms_out * 1e-3) / 1e9, 1),
            "both_gbs": round((h2d + d2h) / (ms * 1e-3) / 1e9, 1),
            "what": "cudaMemcpyAsync from / to pinned host buffers (torch copy_), three copy-in streams and one "
                    "copy-out stream; ms_per_step with both directions at once, h2d_only_ms / d2h_only_ms each alone"}


def bench_backward(dev, flush, steps=30, warmup=3):
    """Backward pass (fa_bwd) on the causal-prefill workload with a seeded upstream gradient; TFLOP/s by the
    usual 2.5x-forward accounting (five products of 2*d flops per visible pair)."""
    import torch

    from tiled_exact_attention_gb300 import fa_bwd, fa_bwd_workspace_size, fa_fwd, fa_sync_status
    from tiled_exact_attention_gb300.inputs import BASE_SEED, WORKLOADS, make_qkv, normal

    w = WORKLOADS["causal_prefill"]
    q, k, v = (t.to(dev) for t in make_qkv(w))
    do = normal(tuple(q.shape), BASE_SEED + w.index, 7, 1.0, q.dtype).to(dev)
    o, lse = fa_fwd(q, k, v, causal=True, q_pos_offset=w.offset)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa_bwd_workspace_size(q, k, v, causal=True, q_pos_offset=w.offset), dtype=torch.uint8,
                     device=dev)

    def step():
        fa_bwd(q, k, v, o, lse, do, causal=True, q_pos_offset=w.offset, dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(warmup):
        flush.zero_()
        step()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    if fa_sync_status() != 0:
        raise RuntimeError("device status set by the backward pass")
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps
    pairs = w.visible_pairs_per_head() * w.b * w.hq
    flops = 2.5 * 4.0 * w.d * pairs
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "config": {"b": w.b, "sq": w.sq, "skv": w.skv, "hq": w.hq, "hkv": w.hkv, "d": w.d, "causal": True},
            "flops_per_launch": flops, "flops_executed_per_launch": 3.5 * 4.0 * w.d * pairs,
            "accounting": "2.5x the forward flops (dV, dP, dQ, dK and the recomputed S); the kernels execute 3.5x "
                          "(S and dP are recomputed by both the dQ and the dK/dV kernel)",
            "kernels": "fa_bwd_dq_kernel (also forms D and L per row) + fa_bwd_dkdv_kernel", "steps": steps}


def bench_e4m3(dev, flush, steps=30, warmup=3, workload="causal_prefill"):
    """The 8-bit forward pass (fa_fwd_e4m3) on a forward workload (the causal prefill, or a ragged-tail
    d = 64 / d = 256 one), its inputs quantised once outside the timed region (fa_quantize_e4m3:
    per-block Q, K scales; V transposed, per-head scale)."""
    import torch

    from tiled_exact_attention_gb300 import fa_fwd_e4m3, fa_sync_status, quantize_qkv_e4m3
    from tiled_exact_attention_gb300.inputs import WORKLOADS, make_qkv

    w = WORKLOADS[workload]
    q, k, v = (t.to(dev) for t in make_qkv(w))
    (q8, qd), (k8, kd), (vt8, vd) = quantize_qkv_e4m3(q, k, v)
    del k, v
    o = torch.empty((w.b, w.sq, w.hq, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.b, w.hq, w.sq), dtype=torch.float32, device=dev)
    off = w.offset if w.causal else None

    def step():
        fa_fwd_e4m3(q8, qd, k8, kd, vt8, vd, causal=w.causal, q_pos_offset=off, out=o, lse=lse)

    for _ in range(warmup):
        flush.zero_()
        step()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    if fa_sync_status() != 0:
        raise RuntimeError("device status set by the e4m3 forward pass")
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps
    flops = 4.0 * w.d * w.visible_pairs_per_head() * w.b * w.hq
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "dtype": "e4m3 inputs, e4m3 P, fp32 accumulation, bf16 O",
            "config": {"b": w.b, "sq": w.sq, "skv": w.skv, "hq": w.hq, "hkv": w.hkv, "d": w.d, "causal": w.causal,
                       "inputs": f"{w.dtype} std {w.std}, quantised outside the timed region"},
            "flops_per_launch": flops, "kernel": f"fa_prefill_kernel<{w.d}, bf16, dense, e4m3>", "steps": steps}


def bench_decode_e4m3(dev, flush, steps=30, warmup=3):
    """Split-KV decode over e4m3 K and V (fa_fwd_splitkv_e4m3) on the decode workload's shape (B=8, Hq=32,
    Hkv=8, KV=32768, d=128, the same seeded values quantised outside the timed region: K with one scale per
    128 keys, V with one per head); KV GB/s of the bytes read (K and V at one byte per element, their scales,
    Q, O and LSE)."""
    import torch

    from tiled_exact_attention_gb300 import fa_fwd_splitkv_e4m3, fa_quantize_e4m3, fa_sync_status
    from tiled_exact_attention_gb300.inputs import WORKLOADS, make_qkv

    w = WORKLOADS[DECODE]
    qc, kc, vc = make_qkv(w)
    q = qc[:, 0].contiguous().to(dev)
    k8, kd = fa_quantize_e4m3(kc.to(dev))
    v8, vd = fa_quantize_e4m3(vc.to(dev), per_head=True)
    o = torch.empty_like(q)
    lse = torch.empty((w.b, w.hq), dtype=torch.float32, device=dev)
    from tiled_exact_attention_gb300 import _lib
    from tiled_exact_attention_gb300.api import make_splitkv_e4m3_args
    import ctypes

    a = make_splitkv_e4m3_args(q, k8, kd, v8, vd, o, lse)
    ws = torch.empty(int(_lib.load().fa_splitkv_e4m3_workspace_size(ctypes.byref(a), 0)), dtype=torch.uint8,
                     device=dev)
    used = fa_fwd_splitkv_e4m3(q, k8, kd, v8, vd, workspace=ws, out=o, lse=lse, return_splits=True)[2]
    ms = _timed(lambda: fa_fwd_splitkv_e4m3(q, k8, kd, v8, vd, workspace=ws, out=o, lse=lse), flush, steps, warmup)
    if fa_sync_status() != 0:
        raise RuntimeError("device status set by the e4m3 decode")
    nbytes = (2 * w.b * w.skv * w.hkv * w.d + (kd.numel() + vd.numel()) * 4 + 2 * w.b * w.hq * w.d * 2
              + w.b * w.hq * 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm = float(_peaks()[0]["hbm_gbs"])
    return {"value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4), "bytes_per_launch": nbytes,
            "config": {"b": w.b, "skv": w.skv, "hq": w.hq, "hkv": w.hkv, "d": w.d, "num_splits": used,
                       "kv": "e4m3 codes, K scale per 128 keys, V scale per head"},
            "keys_per_s": round(w.b * w.hkv * w.skv / (ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "traffic": _profiled_traffic("fa_decode_kernel_e4m3")},
            "steps": steps}


def _timed(step, flush, steps, warmup=3):
    """Mean CUDA-event time (ms) of `step` over `steps` calls, L2 flushed before each."""
    import torch

    for _ in range(warmup):
        flush.zero_()
        step()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps


def bench_variants(dev, flush, steps=20):
    """The mask and layout variants of the forward pass, each on a prefill-sized problem, in TFLOP/s of the
    visible (query, key) pairs (4 d flops per pair and head), against the sustained bf16 peak:
      * window: the causal prefill workload with a sliding window of 1024 keys (local causal);
      * softcap: the causal prefill workload with every score capped to 30 tanh(s / 30);
      * varlen: 16 packed causal sequences, lengths drawn (seeded) from [256, 4096], H = 16, d = 128;
      * decode_g8: split-KV decode with 8 query heads per KV head (B = 8, Hq = 64, Hkv = 8, KV = 32768,
        d = 128), whose heads are the rows of one tensor-core tile; KV GB/s against the measured copy peak;
      * decode_b1 / decode_d64: the split-KV decode at B = 1, and at d = 64.
    The tensor-core lines divide by the burst bf16 peak."""
    import numpy as np
    import torch

    from tiled_exact_attention_gb300 import fa_fwd, fa_fwd_varlen, fa_sync_status
    from tiled_exact_attention_gb300.inputs import BASE_SEED, WORKLOADS, make_qkv, normal

    w = WORKLOADS["causal_prefill"]
    q, k, v = (t.to(dev) for t in make_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.b, w.hq, w.sq), dtype=torch.float32, device=dev)
    out = {}
    wl = 1024
    i = np.arange(w.sq, dtype=np.int64)
    pairs = int((np.minimum(i, wl) + 1).sum())  # row i sees keys max(0, i - wl) .. i
    ms = _timed(lambda: fa_fwd(q, k, v, causal=True, window=(wl, 0), out=o, lse=lse), flush, steps)
    tf = 4.0 * w.d * pairs * w.b * w.hq / (ms * 1e-3) / 1e12
    out["window"] = {"value": round(tf, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
                     "config": {"b": w.b, "sq": w.sq, "hq": w.hq, "d": w.d, "causal": True, "window": [wl, 0]},
                     "roofline": _tensor_roofline(tf)}
    pairs = w.visible_pairs_per_head()
    ms = _timed(lambda: fa_fwd(q, k, v, causal=True, softcap=30.0, out=o, lse=lse), flush, steps)
    tf = 4.0 * w.d * pairs * w.b * w.hq / (ms * 1e-3) / 1e12
    out["softcap"] = {"value": round(tf, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
                      "config": {"b": w.b, "sq": w.sq, "hq": w.hq, "d": w.d, "causal": True, "softcap": 30.0},
                      "roofline": _tensor_roofline(tf)}
    rng = np.random.default_rng(BASE_SEED + 60)
    lens = rng.integers(256, 4097, size=16).astype(np.int64)
    total = int(lens.sum())
    hq, d = 16, 128
    qv = normal((total, hq, d), BASE_SEED + 60, 0).to(dev)
    kv = normal((total, hq, d), BASE_SEED + 60, 1).to(dev)
    vv = normal((total, hq, d), BASE_SEED + 60, 2).to(dev)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(dev)
    ov = torch.empty_like(qv)
    lv = torch.empty((hq, total), dtype=torch.float32, device=dev)
    mx = int(lens.max())
    ms = _timed(lambda: fa_fwd_varlen(qv, kv, vv, cu, cu, max_seqlen_q=mx, causal=True, out=ov, lse=lv), flush,
                steps)
    pairs = int((lens * (lens + 1) // 2).sum())
    tf = 4.0 * d * pairs * hq / (ms * 1e-3) / 1e12
    out["varlen"] = {"value": round(tf, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
                     "config": {"sequences": len(lens), "lengths": [int(x) for x in lens], "hq": hq, "d": d,
                                "causal": True},
                     "roofline": _tensor_roofline(tf)}
    from tiled_exact_attention_gb300 import fa_fwd_splitkv
    from tiled_exact_attention_gb300.api import fa_splitkv_workspace_size
    from tiled_exact_attention_gb300.inputs import make_custom

    del qv, kv, vv, ov, lv
    b, skv, hq, hkv, d = 8, 32768, 64, 8, 128
    qd, kd, vd = (t.to(dev) for t in make_custom(b, 1, skv, hq, hkv, d, "bf16", seed=BASE_SEED + 70))
    od = torch.empty_like(qd)
    ld = torch.empty((b, hq, 1), dtype=torch.float32, device=dev)
    work = torch.empty(fa_splitkv_workspace_size(qd, kd, vd, 0), dtype=torch.uint8, device=dev)
    used = fa_fwd_splitkv(qd, kd, vd, workspace=work, out=od, lse=ld, return_splits=True)[2]
    ms = _timed(lambda: fa_fwd_splitkv(qd, kd, vd, workspace=work, out=od, lse=ld), flush, steps)
    nbytes = 2 * b * skv * hkv * d * 2 + 2 * b * hq * d * 2 + b * hq * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm = float(_peaks()[0]["hbm_gbs"])
    out["decode_g8"] = {"value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
                        "config": {"b": b, "skv": skv, "hq": hq, "hkv": hkv, "d": d, "num_splits": used,
                                   "kernels": "fa_prefill_kernel (heads as rows) + fa_combine_kernel"},
                        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                                     "frac": round(gbs / hbm, 4), "traffic": None}}
    del qd, kd, vd, work
    for key in SMALL_DECODES:
        out[key] = bench_small_decode(dev, flush, key, steps)
    if fa_sync_status() != 0:
        raise RuntimeError("device status set by a forward-pass variant")
    return out


SMALL_DECODES = {"decode_b1": (1, 32, 8, 128), "decode_d64": (8, 32, 8, 64)}  # b, hq, hkv, d


def bench_small_decode(dev, flush, key, steps=30):
    """Split-KV decode at a small batch (decode_b1: B = 1, the decode workload otherwise) or at d = 64
    (decode_d64: B = 8, Hq = 32, Hkv = 8): KV = 32768, the query at the last position; KV GB/s against the
    measured copy peak."""
    import torch

    from tiled_exact_attention_gb300 import fa_fwd_splitkv, fa_sync_status
    from tiled_exact_attention_gb300.api import fa_splitkv_workspace_size
    from tiled_exact_attention_gb300.inputs import BASE_SEED, make_custom

    b, hq, hkv, d = SMALL_DECODES[key]
    skv = 32768
    qd, kd, vd = (t.to(dev) for t in make_custom(b, 1, skv, hq, hkv, d, "bf16", seed=BASE_SEED + 80))
    od = torch.empty_like(qd)
    ld = torch.empty((b, hq, 1), dtype=torch.float32, device=dev)
    work = torch.empty(fa_splitkv_workspace_size(qd, kd, vd, 0, causal=True, q_pos_offset=skv - 1),
                       dtype=torch.uint8, device=dev)
    used = fa_fwd_splitkv(qd, kd, vd, causal=True, q_pos_offset=skv - 1, workspace=work, out=od, lse=ld,
                          return_splits=True)[2]
    ms = _timed(lambda: fa_fwd_splitkv(qd, kd, vd, causal=True, q_pos_offset=skv - 1, workspace=work, out=od,
                                       lse=ld), flush, steps)
    if fa_sync_status() != 0:
        raise RuntimeError(f"device status set by {key}")
    nbytes = 2 * b * skv * hkv * d * 2 + 2 * b * hq * d * 2 + b * hq * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm = float(_peaks()[0]["hbm_gbs"])
    return {"value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "config": {"b": b, "skv": skv, "hq": hq, "hkv": hkv, "d": d, "num_splits": used},
            "bytes_per_launch": nbytes,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "traffic": _profiled_traffic("fa_decode_kernel_" + key[7:])}}


def bench_e2e(qc, kc, vc, wp, fa_fwd, flush, stream, steps, dist=None):
    """Prefill end to end through fa_fwd with host buffers: every step copies its Q, K, V in from pinned host
    memory and its O and LSE out.  Pipelined like a serving loop, two buffer sets in flight: the inputs of step
    i + 1 are copied in (copy stream) while step i computes, and step i's outputs are copied out on a third
    stream; every step's copies stay inside the timed region, from the first copy in to the last copy out."""
    import torch

    dev = stream.device
    h_in = [t.pin_memory() for t in (qc, kc, vc)]
    bufs = []
    for _ in range(2):
        q, k, v = (torch.empty_like(t, device=dev) for t in (qc, kc, vc))
        o = torch.empty_like(q)
        lse = torch.empty((wp.b, wp.hq, wp.sq), dtype=torch.float32, device=dev)
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        bufs.append((q, k, v, o, lse, ho, hl))
    # one copy-in stream per input tensor (the copies run side by side), one copy-out stream
    s_in = [torch.cuda.Stream(device=dev) for _ in range(3)]
    s_out = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done = [[ev(), ev()] for _ in range(3)]
    comp_done, out_done = [ev(), ev()], [ev(), ev()]

    def run(n):
        for i in range(n):
            q, k, v, o, lse, ho, hl = bufs[i % 2]
            for j, (dst, src) in enumerate(zip((q, k, v), h_in)):
                with torch.cuda.stream(s_in[j]):
                    if i >= 2:
                        s_in[j].wait_event(comp_done[i % 2])  # step i - 2 has read this input set
                    dst.copy_(src, non_blocking=True)
                    in_done[j][i % 2].record(s_in[j])
                stream.wait_event(in_done[j][i % 2])
            if i >= 2:
                stream.wait_event(out_done[i % 2])  # step i - 2's outputs have left this output set
            flush.zero_()
            fa_fwd(q, k, v, causal=True, q_pos_offset=wp.offset, out=o, lse=lse)
            comp_done[i % 2].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i % 2])
                ho.copy_(o, non_blocking=True)
                hl.copy_(lse, non_blocking=True)
                out_done[i % 2].record(s_out)
        for si in s_in:
            stream.wait_stream(si)
        stream.wait_stream(s_out)

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    e0.record(stream)
    for si in s_in:  # the first copies start after e0
        si.wait_stream(stream)
    s_out.wait_stream(stream)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def bench_paged_decode(dev, flush, steps=200, warmup=5):
    """Split-KV decode over a paged KV cache: B=8, Hq=32, Hkv=8, d=128, 256-key pages handed out in a
    shuffled order, per-sequence lengths drawn (seeded) from [16384, 49152]; KV GB/s of the valid keys."""
    import numpy as np
    import torch

    from tiled_exact_attention_gb300 import fa_fwd_kvcache, fa_sync_status
    from tiled_exact_attention_gb300.api import make_kvcache_args
    from tiled_exact_attention_gb300.inputs import BASE_SEED, normal

    b, hq, hkv, d, ps = 8, 32, 8, 128, 256
    rng = np.random.default_rng(BASE_SEED + 50)
    lens = rng.integers(16384, 49153, size=b).astype(np.int32)
    pages_per = [int((n + ps - 1) // ps) for n in lens]
    num_pages = sum(pages_per)
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.zeros((b, max(pages_per)), dtype=np.int32)
    nxt = 0
    for i, npg in enumerate(pages_per):
        table[i, :npg] = perm[nxt:nxt + npg]
        nxt += npg
    q = normal((b, hq, d), BASE_SEED + 50, 0).to(dev)
    k = normal((num_pages, ps, hkv, d), BASE_SEED + 50, 1).to(dev)
    v = normal((num_pages, ps, hkv, d), BASE_SEED + 50, 2).to(dev)
    bt = torch.from_numpy(table).to(dev)
    sl = torch.from_numpy(lens).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((b, hq), dtype=torch.float32, device=dev)
    maxlen = int(lens.max())
    from tiled_exact_attention_gb300 import _lib
    import ctypes

    a = make_kvcache_args(q, k, v, o, lse, block_table=bt, seqlens_k=sl, max_seqlen_k=maxlen)
    ws = torch.empty(int(_lib.load().fa_kvcache_workspace_size(ctypes.byref(a), 0)), dtype=torch.uint8, device=dev)

    def step():
        return fa_fwd_kvcache(q, k, v, block_table=bt, seqlens_k=sl, max_seqlen_k=maxlen, workspace=ws, out=o,
                              lse=lse, return_splits=True)

    for _ in range(warmup):
        flush.zero_()
        step()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    ns = 0
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        ns = step()[2]
        e1.record(stream)
    torch.cuda.synchronize()
    if fa_sync_status() != 0:
        raise RuntimeError("device status set by the paged decode")
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps
    nbytes = 2 * int(lens.sum()) * hkv * d * 2 + 2 * b * hq * d * 2 + b * hq * 4
    return {"value": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "config": {"b": b, "hq": hq, "hkv": hkv, "d": d, "page_size": ps, "keys": int(lens.sum()),
                       "seqlens": [int(x) for x in lens], "num_splits": ns, "pages": "shuffled"},
            "bytes_per_launch": nbytes, "steps": steps}


# ------------------------------------------------------------------------- oracle (CPU) arm


def _sample_rows(w, n_rows, seed):
    import numpy as np

    rng = np.random.default_rng(seed)
    idx = rng.choice(w.b * w.hq * w.sq, size=min(n_rows, w.b * w.hq * w.sq), replace=False)
    bi = idx // (w.hq * w.sq)
    hi = (idx // w.sq) % w.hq
    ii = idx % w.sq
    return np.stack([bi, hi, ii], axis=1).astype(np.int64)


def _pairs(w, rows):
    import numpy as np

    if not w.causal:
        return int(rows.shape[0]) * w.skv
    return int(np.clip(rows[:, 2] + w.offset + 1, 0, w.skv).sum())


def cpu_baseline(budget_s=15.0, seed=1):
    """Time the oracle as it stands on the host cores on the prefill workload: the whole
    problem when a calibration run says it takes at most twice the budget, else a random
    sample of its rows sized for the budget; report the algorithmic TFLOP/s."""
    import numpy as np

    import oracle
    from tiled_exact_attention_gb300.inputs import WORKLOADS, make_qkv

    w = WORKLOADS[PREFILL]
    qc, kc, vc = make_qkv(w)
    q, k, v = (t.to(__import__("torch").float64).numpy() for t in (qc, kc, vc))
    total = w.b * w.hq * w.sq
    # calibrate on a small sample, then take the whole problem or a sample sized for the budget
    rows = _sample_rows(w, 256, seed)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, causal=True, q_pos_offset=w.offset, rows=rows)
    t_small = max(time.perf_counter() - t0, 1e-3)
    est_all = t_small * total / 256
    if est_all <= 2 * budget_s:
        rows = oracle.all_rows(w.b, w.hq, w.sq)
        what = "the whole causal prefill workload (every row of every head and batch)"
    else:
        n = int(min(total, max(256, 256 * budget_s / t_small)))
        rows = _sample_rows(w, n, seed + 1)
        what = f"{n} random query rows of the causal prefill workload (all heads/batches)"
    t0 = time.perf_counter()
    oracle.attention(q, k, v, causal=True, q_pos_offset=w.offset, rows=rows)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.d * _pairs(w, rows)
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{what}, {_pairs(w, rows)} visible pairs, {dt:.2f} s, fp64 C oracle with OpenMP",
            "seconds": round(dt, 3)}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from tiled_exact_attention_gb300.inputs import WORKLOADS, make_qkv

    w = WORKLOADS[PREFILL]
    qc, kc, vc = make_qkv(w)
    import torch

    q, k, v = (t.to(torch.float64).numpy() for t in (qc, kc, vc))
    total_budget = 90.0
    rows = _sample_rows(w, 128, 7)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, causal=True, q_pos_offset=w.offset, rows=rows)
    t_small = max(time.perf_counter() - t0, 1e-3)
    per_step = total_budget / max(1, args.steps + args.warmup)
    n = int(min(w.b * w.hq * w.sq, max(16, 128 * per_step / t_small)))
    for i in range(args.warmup):
        oracle.attention(q, k, v, causal=True, q_pos_offset=w.offset, rows=_sample_rows(w, n, 100 + i))
    times, flops = [], 0.0
    for i in range(args.steps):
        rows = _sample_rows(w, n, 1000 + i)
        t0 = time.perf_counter()
        oracle.attention(q, k, v, causal=True, q_pos_offset=w.offset, rows=rows)
        times.append(time.perf_counter() - t0)
        flops += 4.0 * w.d * _pairs(w, rows)
    tt = sum(times)
    val = flops / tt / 1e12
    sample = f"{n} random query rows per step of the causal prefill workload, fp64 C oracle with OpenMP"
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(val, 6),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * tt / max(1, args.steps), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: iid N(0,1) bf16 from seeded PCG64, converted exactly to fp64",
        "config": {"workload": "causal prefill B=4 Hq=Hkv=16 N=4096 d=128 (bounded row sample per step)"},
        "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--only", default="", help="time only these lines (comma-separated); prints them alone")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
