"""Benchmark: CSA forward query-tokens/s and TFLOP/s against the GB300 roofline.

A step is one pass of the whole hot path over one batch of synthetic input:
compress (main KV + indexer K), indexer score + top-k, selected attention with
the local window, indexer KL loss.  The default workload is the sparse warm-up
layer at L = 32768 (r = 4, 64 heads x 128, indexer 8 x 64, top-k 2048, W = 128,
dense teacher over every visible entry), the shape of the DeepSeek-V4 CSA
layers in "DeepSeek-V4 Attention Training Systems" (§2 phase table).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--compressor plain|v4] [--indexer bf16|fp8] [--backward]

Prints one JSON line (rank 0).  Multi-GPU: one process per GPU under
torch.distributed.run; each rank runs its own copy of the workload (the path
has no exchange step on one GPU: replicas only), value = all ranks' tokens /
max-over-ranks time.  ``--impl reference`` times the CPU oracle on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from compressed_sparse_attention_compress_gb300 import inputs as I  # noqa: E402
from compressed_sparse_attention_compress_gb300 import workload as W  # noqa: E402

METRIC = "CSA fwd query-tokens/s at L=32K and TFLOP/s, % of GB300 bf16/HBM roofline"
UNIT = "query-tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 20 ms from before the
    warm-up on; each sample carries nvidia-smi's timestamp, and the summary keeps
    the samples inside the marked timed regions."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.windows = []
        self.lines = []
        self.t_start = time.time()

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t_start = time.time()
        return self

    def settle(self, seconds: float = 0.5):
        """Give nvidia-smi time to start sampling before a timed region."""
        left = seconds - (time.time() - self.t_start)
        if self.proc is not None and left > 0:
            time.sleep(left)

    @staticmethod
    def now():
        return datetime.datetime.now()

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        slack = datetime.timedelta(milliseconds=20)
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                clk, cmax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            if not any(a - slack <= ts <= b + slack for a, b in self.windows):
                continue
            sm.append(clk)
            mx.append(cmax)
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(wl, arrs, seconds_target=15.0, max_rows=None):
    """Time the oracle on a strided sample of query rows of the same workload."""
    import oracle
    cu = arrs["cu_seqlens"]
    threads = oracle.num_threads()
    scale = wl.scale
    t0 = time.perf_counter()
    def comp(s, rope):
        if wl.compressor == "v4":
            return oracle.compress_ex(arrs["x_" + s], arrs["z_" + s], arrs["P_" + s], cu, wl.ratio, wl.overlap,
                                      x_prev=arrs.get(f"x_{s}_prev"), z_prev=arrs.get(f"z_{s}_prev"),
                                      gamma=arrs["g_" + s], eps=wl.norm_eps, rope_dim=rope, theta=wl.rope_theta)
        return oracle.compress(arrs["x_" + s], arrs["z_" + s], arrs["P_" + s], cu, wl.ratio, wl.overlap)

    kv = I.bf16_round(comp("kv", wl.rope_kv).astype(np.float32)) if wl.ratio > 0 else None
    kI = I.bf16_round(comp("I", wl.rope_I).astype(np.float32)) if wl.H_I > 0 else None
    t_comp = time.perf_counter() - t0
    # probe cost on a few rows near the end (the most expensive queries), then size the sample
    n = 8
    while True:
        stride = max(1, wl.T // n)
        rows = np.arange(stride // 2, wl.T, stride, dtype=np.int64)[:n]
        t1 = time.perf_counter()
        if wl.H_I > 0:
            idx_rows = oracle.indexer_topk(arrs["qI"], arrs["w"], kI, cu, wl.ratio, wl.topk, wl.k_pad, rows)
            idx = np.full((wl.T_cap, wl.k_pad), -1, np.int32)
            idx[rows] = idx_rows
            oracle.attention(oracle.KIND_CSA, arrs["q"], kv, None, arrs["x_kv"], None, cu, wl.ratio, wl.window,
                             scale, idx=idx, rows=rows)
            if wl.kl_mode != "none":
                oracle.indexer_kl(arrs["q"], kv, arrs["qI"], arrs["w"], kI, cu, wl.ratio, scale,
                                  idx=idx if wl.kl_mode == "sparse" else None, rows=rows)
        elif wl.ratio > 0:
            oracle.attention(oracle.KIND_HCA, arrs["q"], kv, None, arrs["x_kv"], None, cu, wl.ratio, wl.window,
                             scale, rows=rows)
        else:
            oracle.attention(oracle.KIND_WINDOW, arrs["q"], None, None, arrs["x_kv"], None, cu, 0, wl.window,
                             scale, rows=rows)
        dt = time.perf_counter() - t1
        if dt >= seconds_target or n >= wl.T or (max_rows and n >= max_rows):
            break
        n = min(wl.T, max(n * 2, int(n * seconds_target / max(dt, 1e-3))))
        if max_rows:
            n = min(n, max_rows)
    # rate: sampled rows through the per-query steps + the sample's share of compression
    total = dt + t_comp * len(rows) / wl.T
    return {"value": len(rows) / total, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} query rows strided over the {wl.T}-token workload (one in every {stride}), "
                      f"plus the rows' share of the full-sequence compression; fp64 C oracle, OpenMP"}


def run_reference(args, wl):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    arrs = I.generate(wl, args.seed)
    vals = []
    for _ in range(args.warmup):
        cpu_baseline(wl, arrs, seconds_target=2.0, max_rows=64)
    base = None
    t0 = time.perf_counter()
    per_step = max(1.0, min(args.ref_seconds, 150.0 / max(args.steps, 1)))
    for _ in range(args.steps):
        base = cpu_baseline(wl, arrs, seconds_target=per_step)
        vals.append(base["value"])
    elapsed = time.perf_counter() - t0
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "sample": base["sample"]},
            "cpu_baseline": {**base, "value": v},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, wl):
    import torch
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    from compressed_sparse_attention_compress_gb300.forward import Forward, to_device

    arrs = I.generate(wl, args.seed)
    dev_in = to_device(arrs, wl.io_fp32, local)
    f = Forward(wl, dev_in, device=local)
    stream = torch.cuda.current_stream()
    counts = W.counts(wl)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    # stage boundaries for per-kernel durations (events on the launching stream)
    stages = []
    if wl.ratio > 0:
        stages.append(("compress", f.compress))
        if wl.H_I > 0:
            stages.append(("indexer_topk", f.topk))
    stages.append(("attention", f.attend))
    if wl.kl_mode != "none":
        stages.append(("indexer_kl", f.kl))
    dout = None
    f.keep_stats = bool(args.backward)   # the KL forward hands its normalisers to the indexer backward
    if args.backward:
        # upstream gradient of the attention output: bf16 N(0,1), its own seeded stream
        g = np.random.default_rng(np.random.SeedSequence(args.seed).spawn(len(I.STREAMS) + 1)[-1])
        dout = torch.from_numpy(I.bf16_round(g.standard_normal(tuple(f.out.shape), dtype=np.float32)))
        dout = dout.to(f.out.device, f.out.dtype)
        stages.append(("attention_bwd", lambda: f.backward(dout)))
        if wl.kl_mode != "none":
            stages.append(("indexer_bwd", f.indexer_backward))

    clk = ClockSampler(local).start()   # sampling from before the warm-up; samples kept per timed region
    for _ in range(max(args.warmup, 3)):
        f.run()
    torch.cuda.synchronize()
    assert f.h.device_status() == 0, "device status raised during warm-up"
    clk.settle()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t_dev0 = clk.now()
    for s in range(args.steps):
        ev[s][0].record(stream)
        for i, (_, fn) in enumerate(stages):
            fn()
            ev[s][i + 1].record(stream)
    torch.cuda.synchronize()
    clk.mark(t_dev0, clk.now())
    barrier()
    total_ms = sum(ev[s][0].elapsed_time(ev[s][-1]) for s in range(args.steps))
    stage_ms = {name: sum(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps)) / args.steps
                for i, (name, _) in enumerate(stages)}
    # the median over the steps as well: the first step's first stage also waits
    # for the host to issue it (the device is idle when the timed region opens)
    stage_med = {name: statistics.median([ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps)])
                 for i, (name, _) in enumerate(stages)}
    assert f.h.device_status() == 0, "device status raised during the timed steps"
    ms_step = total_ms / args.steps
    if ws > 1:
        t = torch.tensor([ms_step], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms_step = float(t.item())
    value = ws * wl.T / (ms_step * 1e-3)

    # e2e: the same step through the public API with host buffers (pinned), inputs
    # copied in and the loss (or lse) read back inside the timed region
    host = {k: v.cpu().pin_memory() for k, v in dev_in.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    dout_host = dout.cpu().pin_memory() if dout is not None else None
    if dout_host is not None:
        h2d += dout_host.numel() * dout_host.element_size()
    res = f.kl_sum if wl.kl_mode != "none" else f.lse
    res_host = torch.empty(res.shape, dtype=res.dtype).pin_memory()
    d2h = res_host.numel() * res_host.element_size()

    def e2e_step():
        # inputs copied in stage order on a side stream; each stage waits for its own
        f.run_from_host(host, stream)
        if dout_host is not None:
            # the upstream gradient follows the queries on the copy stream, under the forward
            stream.wait_event(f.copy_from_host(dout, dout_host))
            f.backward(dout, stream)
            if wl.kl_mode != "none":
                f.indexer_backward(stream=stream)
        res_host.copy_(res, non_blocking=True)

    for _ in range(max(3, args.warmup)):   # the first steps after pinning pay a one-time mapping cost
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_e2e0 = clk.now()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk.mark(t_e2e0, clk.now())
    clk.stop()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if ws > 1:
        t = torch.tensor([e2e_ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    peaks, src = _peaks()
    # dominant kernel: the stage with the largest share of the step
    dom = max(stage_ms, key=stage_ms.get)
    per_launch = {"attention": ("tensor", counts["attn_flops"]),
                  "indexer_kl": ("tensor", counts["teacher_flops"]),
                  "indexer_topk": ("tensor", counts["indexer_flops"]),
                  "compress": ("hbm", counts["compress_bytes"]),
                  "attention_bwd": ("tensor", counts["attn_bwd_flops"]),
                  "indexer_bwd": ("tensor", counts["indexer_bwd_flops"])}
    bound, work = per_launch[dom]
    sec = stage_ms[dom] * 1e-3
    # the timed region lasts well under a second: a kernel timed in it is held to
    # the burst tensor rate (the sustained one is reported beside it)
    tpeak = peaks["bf16_tflops"]
    if bound == "tensor":
        achieved = work / sec / 1e12
        peak = tpeak
        unit = "TFLOP/s"
    else:
        achieved = work / sec / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    total_flops = counts["total_flops"]
    if args.backward:
        total_flops += counts["attn_bwd_flops"] + (counts["indexer_bwd_flops"] if wl.kl_mode != "none" else 0)
    tflops = total_flops / (ms_step * 1e-3) / 1e12
    # the HBM-side stages against the copy bandwidth, whichever stage dominates
    def hbm(nbytes, stage, note):
        if stage not in stage_ms or not nbytes:
            return None
        gbs = nbytes / (stage_ms[stage] * 1e-3) / 1e9
        med = nbytes / (stage_med[stage] * 1e-3) / 1e9
        return {"achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                "bytes": int(nbytes), "ms": stage_ms[stage], "ms_median": stage_med[stage],
                "frac_median": med / peaks["hbm_gbs"], "bytes_are": note}
    comp_hbm = hbm(counts["compress_bytes"], "compress", "algorithmic: x, z read once, compressed rows written")
    topk_hbm = hbm(counts["topk_bytes"], "indexer_topk",
                   "algorithmic: qI, w read once, index rows written (scoring is on chip)")
    gather = hbm(counts["gather_bytes"], "attention",
                 "logical: every candidate key row gathered once per query (L2-served; the attention "
                 "stage's whole time, its tensor work included)")
    traffic = _traffic(dom, wl.name)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "global_batch": wl.B * ws, "seq_len": max(wl.lengths),
                   "tokens_per_gpu": wl.T, "ratio": wl.ratio, "heads": wl.H, "head_dim": wl.d, "topk": wl.topk,
                   "window": wl.window, "kl": wl.kl_mode, "compressor": wl.compressor, "indexer": wl.indexer,
                   "backward": bool(args.backward),
                   "parallelism": f"replicas{ws}",
                   "l2": "inputs larger than L2 (q alone is %.0f MB)" % (wl.T_cap * wl.H * wl.d * 2 / 1e6)},
        "tflops": tflops,
        "tflops_frac_of_peak": tflops / tpeak,
        "stage_ms": stage_ms,
        "roofline": {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{src} ({'bf16_tflops, burst' if bound == 'tensor' else 'hbm_gbs'})",
                     **({"frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
                        if bound == "tensor" else {})},
        "compress_hbm": comp_hbm,
        "topk_hbm": topk_hbm,
        "gather": gather,
        "stage_tflops": {k: counts[v] / (stage_ms[k] * 1e-3) / 1e12 for k, v in
                         (("attention", "attn_flops"), ("indexer_kl", "teacher_flops"),
                          ("indexer_topk", "indexer_flops")) if k in stage_ms and counts[v]},
        "attention_bwd": ({"ms": stage_ms["attention_bwd"], "flops": counts["attn_bwd_flops"],
                           "tflops": counts["attn_bwd_flops"] / (stage_ms["attention_bwd"] * 1e-3) / 1e12,
                           "frac": counts["attn_bwd_flops"] / (stage_ms["attention_bwd"] * 1e-3) / 1e12
                           / tpeak} if args.backward else None),
        "indexer_bwd": ({"ms": stage_ms["indexer_bwd"], "flops": counts["indexer_bwd_flops"],
                         "tflops": counts["indexer_bwd_flops"] / (stage_ms["indexer_bwd"] * 1e-3) / 1e12,
                         "frac": counts["indexer_bwd_flops"] / (stage_ms["indexer_bwd"] * 1e-3) / 1e12
                         / tpeak} if args.backward and wl.kl_mode != "none" else None),
        "e2e": {"value": ws * wl.T / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * (f_launches(wl) + (b_launches(wl) if args.backward else 0)),
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and ws >= 1:
        line["cpu_baseline"] = cpu_baseline(wl, arrs, seconds_target=args.ref_seconds)
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def f_launches(wl) -> int:
    """Kernels of ours launched per step (mirrors the dispatch in csrc/)."""
    n = 0
    if wl.ratio > 0:
        if (wl.compressor != "v4" and not wl.separate_v and wl.H_I > 0
                and (wl.d, wl.d_I) in ((128, 64), (64, 32))):
            n += 1                                                              # both compressors + offsets
        else:
            n += 1 + 1 + (1 if wl.separate_v else 0) + (1 if wl.H_I > 0 else 0)   # offsets + compress calls
        if wl.H_I > 0:
            n += 2                                                              # top-k + capacity fill
            if wl.indexer == "fp8":
                n += 2                                                          # quantise qI and kI
    ws_attn = not wl.io_fp32 and wl.H == 64 and wl.d == 128 and not wl.separate_v
    n += 2 if ws_attn else 1                                                    # (capacity rows) + attention
    if wl.kl_mode != "none":
        dense_tc = (wl.kl_mode == "dense" and not wl.io_fp32 and wl.H == 64 and wl.d == 128
                    and wl.H_I == 8 and wl.d_I == 64)
        n += 3 if dense_tc else 2                                               # (zero) + KL + finalize
    return n


def b_launches(wl) -> int:
    """Kernels of ours launched per backward step (mirrors the dispatch in csrc/):
    attention backward = delta + (tcgen05: capacity rows + kernel | warp-level kernel),
    indexer backward = one kernel (its zero fills are memsets)."""
    tc = not wl.io_fp32 and wl.H == 64 and wl.d == 128 and not wl.separate_v
    return (3 if tc else 2) + (1 if wl.kl_mode != "none" else 0)


def _traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel, if current."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    return d.get(workload, {}).get(kernel)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="warmup32k", choices=sorted(I.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--ref-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="add the attention backward (dq, dKV from the saved output and LSE) and, with an "
                         "indexer loss, the indexer backward to every step")
    ap.add_argument("--indexer", default="bf16", choices=["bf16", "fp8"],
                    help="fp8: E4M3 indexer operands (quantised in the step) for the scoring + top-k")
    ap.add_argument("--compressor", default="plain", choices=["plain", "v4"],
                    help="v4: previous-half stream + RMSNorm + RoPE fused into both compressors")
    args = ap.parse_args()
    wl = I.WORKLOADS[args.workload]
    if args.compressor != "plain":
        wl = dataclasses.replace(wl, compressor=args.compressor)
    if args.indexer != "bf16":
        wl = dataclasses.replace(wl, indexer=args.indexer)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
