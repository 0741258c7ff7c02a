#!/usr/bin/env python
"""Benchmark of the Engram per-layer forward step on GB300.

One step = the whole hot path over one batch: the 2,048-token prefill at full
geometry (24 MXFP8 rows of 256 from a 16.0M-row table, wkv 25,600 x 6,144, 4
hyper-connection branches of 5,120).  `value` is device-timed (CUDA events,
inputs resident in HBM) tokens/s per layer of the forward step through the
faster of the two forward entries (engram_forward_staged; the single fused
kernel engram_forward is reported beside it under "fused"); `e2e` is the
same metric through the C ABI with host buffers: append on the host, pinned
H2D of windows and hidden, the forward, D2H of the updated hidden, every step,
with consecutive steps pipelined over an upload, a compute and a download
stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 (torchrun): every rank runs its own replica on its own batches (weak
scaling, no collective on the data path); the time is the max over ranks.
`--impl reference` times the CPU oracle (the plain fp64 definition) on the
host cores on the same workload: each step is a bounded sample of tokens.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "prefill_2048"
# DRAM bytes (read + write) of one launch of the staged forward GEMM
# (k_mma, TMA-fed A on CTA pairs, gate epilogue) at 2,048 tokens, from one ncu
# capture of that kernel (dram__bytes_read.sum 668.1 MB + dram__bytes_write.sum
# 44.8 MB, mean of two launches); the table size does not enter it.  Re-measure
# when the kernel changes.
GEMM_DRAM_BYTES = 713.0e6
# The same for the decode step's stream-K GEMM (256 tokens; dram__bytes_read.sum
# 328.4 MB + dram__bytes_write.sum 9.6 MB, mean of five launches of the
# --decode-small capture).
DECODE_GEMM_DRAM_BYTES = 338.0e6
FLOP_PER_TOKEN = None  # set from the geometry: 2 N K


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip decode / gather / project lines")
    ap.add_argument("--no-host", action="store_true",
                    help="skip the host-table line (pins 17 GB of host memory)")
    ap.add_argument("--cpu-sample", type=int, default=256,
                    help="oracle tokens for cpu_baseline (0: skip)")
    ap.add_argument("--cpu-sample-configs", type=int, default=4096,
                    help="oracle token rows timed for each of the decode, long-prefill and "
                         "host-table lines (0: skip)")
    ap.add_argument("--small", action="store_true",
                    help="profiling case: same kernels and batch, a 4.8M-row table, 2 batches")
    ap.add_argument("--gather-small", action="store_true",
                    help="profiling case of the unfused gather: 50,032 tokens over a 4.8M-row "
                         "table; prints one line with its time and GB/s")
    ap.add_argument("--decode-small", action="store_true",
                    help="profiling case of the decode step: 256 sessions, full wkv, a "
                         "4.8M-row table; prints one line with its ms per step")
    ap.add_argument("--long-small", action="store_true",
                    help="profiling case of the long prefill: 50,032 tokens through two layers "
                         "of 4.8M-row tables; prints one line with its ms per layer")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d["bf16_tflops_sustained"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ---- distributed plumbing (timing only: barrier and max over ranks) -------------------------

class Dist:
    def __init__(self):
        import torch

        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist

            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def shard_sessions(n_sessions: int, rank: int, world: int):
    """Sessions owned by a rank: contiguous, as even as possible (no data exchange)."""
    lo = n_sessions * rank // world
    hi = n_sessions * (rank + 1) // world
    return list(range(lo, hi))


# ---- clocks ------------------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int, interval_ms: int = 50):
        self.gpu = gpu
        self.interval = interval_ms
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval), "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for ln in out.splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows[-3:]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        sm = [r[1] for r in inside]
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "reasons": reasons, "samples": len(inside)}


# ---- the reference arm: the CPU oracle ----------------------------------------------------

def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_inputs(w, T):
    import oracle as O
    import synth

    g = O.Geom(vocab=w.vocab, vc=w.vc, min_n=w.min_n, max_n=w.max_n, heads=w.heads,
               row_dim=w.row_dim, hc=w.hc, d=w.d, pad_cid=w.pad_cid, eps=w.eps)
    p = O.layer_params(g, w.hash_seeds, w.bucket_bases, 0)
    tmap = synth.token_map(w.vocab, w.vc, w.seed)
    win = O.windows(g, tmap, synth.session_tokens(w, 0, T))
    return g, p, win


def run_oracle_timed(w, W, wq, wk, hidden, win, g, p, tokens: np.ndarray, threads: int) -> float:
    import oracle as O

    t0 = time.perf_counter()
    O.forward(g, w.table_seeds[0], p, W, wq, wk, win, hidden, tokens, nthreads=threads,
              want_h64=False)
    return time.perf_counter() - t0


def reference_arm(args, dist: Dist):
    if dist.rank != 0:
        dist.close()
        return
    import oracle as O
    import synth

    O.build()
    w = synth.WORKLOADS[WORKLOAD]
    T = w.tokens_per_session
    W = synth.wkv_bf16(w)
    wq, wk = synth.wq_wk(w)
    hidden = synth.hidden_bf16(w, T)
    g, p, win = oracle_inputs(w, T)
    cores = cpu_cores()
    # size each step's sample so the whole run takes about 20-150 s of wall time
    calib = run_oracle_timed(w, W, wq, wk, hidden, win, g, p, np.arange(cores) % T, cores)
    rate = cores / calib  # tokens/s with all cores
    steps, warm = args.steps, args.warmup
    per_step = max(1, min(T, int(round(20.0 * rate / max(steps, 1)))))
    rng = np.random.default_rng(0)
    sample = rng.integers(0, T, (warm + steps) * per_step)
    run_oracle_timed(w, W, wq, wk, hidden, win, g, p, sample[:warm * per_step], cores)
    elapsed = run_oracle_timed(w, W, wq, wk, hidden, win, g, p, sample[warm * per_step:], cores)
    toks = steps * per_step
    value = toks / elapsed
    line = {
        "metric": "Engram tokens/s per layer (prefill, decode); gather HBM GB/s; wkv TC util %",
        "impl": "reference", "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": 1000.0 * elapsed / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} random tokens of the {T}-token prefill per step, "
                                   f"all steps' tokens run by the oracle over {cores} threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    dist.close()


def workload_config(w) -> dict:
    return {"workload": f"{w.name}: {w.tokens_per_session} tokens, 1 Engram layer, "
                        f"n=2..4 x {w.heads} heads x {w.row_dim}, wkv {w.N}x{w.K} bf16, "
                        f"hc {w.hc} x {w.d}",
            "tokens_per_step": w.sessions * w.tokens_per_session, "layers": 1,
            "table_rows": None, "table_format": "MXFP8 (E4M3 + E8M0 per 32)",
            "l2": "inputs larger than L2: wkv 314.6 MB per step plus a rotating pool of 8 "
                  "hidden/window batches (671 MB)"}


# ---- my arm ------------------------------------------------------------------------------------

def main():
    args = parse_args()
    dist = Dist()
    if args.impl == "reference":
        reference_arm(args, dist)
        return
    if args.decode_small:
        decode_small(args)
        return
    if args.gather_small:
        gather_small(args)
        return
    if args.long_small:
        long_small(args)
        return
    import torch

    import engram_gram_conditional_gb300 as eg
    import oracle as O
    import synth
    from engram_gram_conditional_gb300 import build
    from engram_gram_conditional_gb300.layer import EngramLayerSet

    if dist.rank == 0:
        build.build()
    dist.barrier()
    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    w = synth.WORKLOADS[WORKLOAD]
    POOL = 8
    if args.small:
        import dataclasses

        w = dataclasses.replace(w, bucket_bases=[200_000])
        POOL = 2
    T = w.tokens_per_session
    flop_tok = 2.0 * w.N * w.K
    tmap = synth.token_map(w.vocab, w.vc, w.seed)
    W = synth.wkv_bf16(w)
    wq, wk = synth.wq_wk(w)
    model = EngramLayerSet.from_workload(w, tmap, device=dev)
    model.bind(0, w.table_seeds[0], W, wq, wk)
    rows = model.rows(0)
    ctx = model.ctx

    # a pool of distinct batches per rank (distinct sessions -> distinct rows)
    base_session = dist.rank * POOL
    win_h, hid_h = [], []
    for i in range(POOL):
        s = eg.engram_session_create(ctx)
        win_h.append(eg.engram_session_append(s, synth.session_tokens(w, base_session + i, T)))
        eg.engram_session_destroy(s)
        hid_h.append(synth.normal_bf16((T, w.hc, w.d), 1.0, w.seed, 1000 + base_session + i))
    d_win = [torch.from_numpy(x.view(np.int32)).to(dev) for x in win_h]
    d_hid = [torch.from_numpy(x.view(np.int16)).to(dev) for x in hid_h]
    # one workspace serves both entries: it holds the larger of the two
    d_ws = torch.empty(max(eg.engram_forward_staged_workspace_bytes(ctx, T),
                           eg.engram_workspace_bytes(ctx, T)), dtype=torch.uint8, device=dev)
    sptr = stream.cuda_stream

    def step(i):
        j = i % POOL
        eg.engram_forward_staged(ctx, 0, d_win[j], T, d_hid[j], d_ws, None, sptr)

    def step_fused(i):
        j = i % POOL
        eg.engram_forward(ctx, 0, d_win[j], T, d_hid[j], d_ws, None, sptr)

    for i in range(args.warmup):
        step(i)
    eg.engram_sync(ctx, sptr)
    clocks = ClockSampler(dist.local)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    dist.barrier()
    clk = clocks.stop(t0, t1)
    eg.engram_sync(ctx, sptr)
    ms_local = ev0.elapsed_time(ev1)
    ms = dist.max(ms_local)
    total_tokens = dist.sum(float(T * args.steps))
    value = total_tokens / (ms / 1000.0)
    ms_step = ms / args.steps
    flops_call = flop_tok * T
    achieved = flops_call / (ms_local / args.steps / 1000.0) / 1e12

    # The same step run 2,000 times back to back (0.8 s of GEMMs), long enough
    # for the GPU to reach its power cap: the figure a long prefill stream
    # sees, beside the short timed region above.
    SUSTAINED_STEPS = 2000
    if args.steps >= SUSTAINED_STEPS:
        sustained = {"steps": args.steps, "same_as_timed_region": True}
    else:
        clocks_s = ClockSampler(dist.local)
        clocks_s.start()
        t0s = time.time()
        ms_s = timed(step, SUSTAINED_STEPS, stream)
        clk_s = clocks_s.stop(t0s, time.time())
        ach_s = flops_call / (ms_s / 1000.0) / 1e12
        sustained = {"steps": SUSTAINED_STEPS, "ms_per_step": ms_s,
                     "tokens_per_s": T / (ms_s / 1000.0), "achieved_tflops": ach_s,
                     "frac_of_burst": ach_s / peaks["bf16"],
                     "frac_of_sustained": ach_s / peaks["bf16_sus"],
                     "power_capped": "sw_power_cap" in clk_s.get("reasons", []),
                     "clocks": clk_s}
    eg.engram_sync(ctx, sptr)

    # the single fused kernel (engram_forward) on the same batches
    fused_steps = max(1, min(args.steps, 500))
    for i in range(min(args.warmup, 5)):
        step_fused(i)
    ms_fused = timed(step_fused, fused_steps, stream)
    eg.engram_sync(ctx, sptr)
    fused_tf = flops_call / (ms_fused / 1000.0) / 1e12

    # ---- e2e through the C ABI with host buffers ----
    # Every step appends its tokens on the host, copies its windows and hidden
    # from pinned host memory, runs the forward and copies the updated hidden
    # back.  Three streams and three buffer sets pipeline the steps: step i's
    # upload and step i-1's download (opposite directions of the host link)
    # overlap each other and the compute.  With two sets, step i's upload
    # would wait for step i-2's download, and upload, compute and download
    # would take turns over two steps; with three, the link's two directions
    # bound the step.
    NB = 3
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h_win = [torch.empty((T, 4), dtype=torch.int32, pin_memory=True) for _ in range(NB)]
    h_hid_in = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in hid_h[:2]]
    h_hid_out = [torch.empty((T, w.hc, w.d), dtype=torch.int16, pin_memory=True)
                 for _ in range(NB)]
    e_win = [torch.empty((T, 4), dtype=torch.int32, device=dev) for _ in range(NB)]
    e_hid = [torch.empty((T, w.hc, w.d), dtype=torch.int16, device=dev) for _ in range(NB)]
    ev_in = [torch.cuda.Event() for _ in range(NB)]
    ev_comp = [torch.cuda.Event() for _ in range(NB)]
    ev_out = [torch.cuda.Event() for _ in range(NB)]
    for j in range(NB):  # recorded once so that the first waits return at once
        ev_in[j].record(s_in)
        ev_comp[j].record(stream)
        ev_out[j].record(s_out)
    tok_h = [synth.session_tokens(w, 100 + base_session + i, T) for i in range(2)]
    h_win_np = [x.numpy().view(np.uint32) for x in h_win]

    def e2e_step(i):
        j = i % NB
        ev_in[j].synchronize()  # step i - NB's upload has read h_win[j]
        s = eg.engram_session_create(ctx)
        eg.engram_session_append(s, tok_h[i % 2], None, h_win_np[j])
        eg.engram_session_destroy(s)
        s_in.wait_event(ev_comp[j])  # step i - NB's forward is done with e_win/e_hid[j]
        s_in.wait_event(ev_out[j])   # ... and its download has read e_hid[j]
        with torch.cuda.stream(s_in):
            e_win[j].copy_(h_win[j], non_blocking=True)
            e_hid[j].copy_(h_hid_in[i % 2], non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        eg.engram_forward_staged(ctx, 0, e_win[j], T, e_hid[j], d_ws, None, sptr)
        ev_comp[j].record(stream)
        s_out.wait_event(ev_comp[j])
        with torch.cuda.stream(s_out):
            h_hid_out[j].copy_(e_hid[j], non_blocking=True)
            ev_out[j].record(s_out)

    e2e_steps = max(1, min(args.steps, 500))
    for i in range(min(args.warmup, 5)):
        e2e_step(i)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t_e0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = dist.max(time.perf_counter() - t_e0)
    e2e_value = dist.sum(float(T * e2e_steps)) / e2e_s
    eg.engram_sync(ctx, sptr)

    # the roofline fraction is always read against the measured burst peak, so
    # that runs compare; a run long enough to meet the power cap (seen in the
    # clock samples of the timed region) says so, and its fraction of the
    # sustained peak is given beside it
    capped = "sw_power_cap" in clk.get("reasons", [])
    peak_tc = peaks["bf16"]
    peak_kind = "burst (the timed run met the power cap: see frac_of_sustained)" if capped \
        else "burst"
    line = {
        "metric": "Engram tokens/s per layer (prefill, decode); gather HBM GB/s; wkv TC util %",
        "value": value, "unit": "tokens/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        # the GEMM multiplies FP16 operands that hold the BF16 values exactly
        # (E4M3 x 2^E8M0 rows, wkv scaled by a power of two) into fp32; the
        # gate is fp32; hidden is BF16 in and out
        "scaling": "weak", "vs_baseline": None, "dtype": "f16*f16->f32", "data": "synthetic",
        "config": dict(workload_config(w), table_rows=rows, parallelism=f"replicas x{dist.world}",
                       entry="engram_forward_staged"),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tc,
                     "unit": "TFLOP/s", "frac": achieved / peak_tc,
                     "traffic": GEMM_DRAM_BYTES,
                     "kernel": "engram_forward_staged: k_gather_stage + k_mma (TMA-fed A, gate "
                               "epilogue); time per call covers both launches",
                     "peak_kind": f"bf16 dense {peak_kind}, {peaks['src']}",
                     "frac_of_burst": achieved / peaks["bf16"],
                     "frac_of_sustained": achieved / peaks["bf16_sus"],
                     "flop_per_call": flops_call},
        "sustained": sustained,
        "fused": {"entry": "engram_forward (one kernel: hash, gather and decode into the "
                           "shared-memory operand tiles, GEMM, gate epilogue)",
                  "ms_per_step": ms_fused, "tokens_per_s": T / (ms_fused / 1000.0),
                  "achieved_tflops": fused_tf, "frac": fused_tf / peaks["bf16"],
                  "steps": fused_steps},
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": T * 16 + T * w.hc * w.d * 2,
                "d2h_bytes_per_step": T * w.hc * w.d * 2, "steps": e2e_steps},
        "gpu_launches": 2 * args.steps,  # k_gather_stage + k_mma per step
        "clocks": clk,
    }

    if args.small:
        line["config"]["l2"] = "profiling case: 2 batches, 4.8M-row table"
    if dist.rank == 0 and dist.world == 1 and not args.no_extras and not args.small:
        try:
            line.update(extras(args, w, W, wq, wk, tmap, win_h[0], d_win[0], model, peaks, dev,
                               sptr, stream))
        except Exception as exc:  # extras never hide the main line
            line["extras_error"] = repr(exc)
        try:
            line["long_prefill"] = long_prefill(tmap, peaks, dev, stream)
        except Exception as exc:
            line["long_prefill"] = {"error": repr(exc)}
        if not args.no_host:
            try:
                line["host_table"] = host_pipeline(model, W, wq, wk, tmap, peaks, dev, stream)
            except Exception as exc:
                line["host_table"] = {"error": repr(exc)}
    if dist.rank == 0 and dist.world == 1 and args.cpu_sample > 0:
        line["cpu_baseline"] = cpu_baseline(args, w, W, wq, wk, win_h[0], hid_h[0])
    if dist.rank == 0 and dist.world == 1:
        run_oracle_jobs(args)
    model.close()
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def gather_small(args):
    """engram_gather_dequant (a3 alone) for 50,032 Zipf tokens over a 4.8M-row
    table (1.3 GB, ten times L2), for ncu."""
    import dataclasses

    import torch

    import engram_gram_conditional_gb300 as eg
    import synth
    from engram_gram_conditional_gb300 import build
    from engram_gram_conditional_gb300.layer import EngramLayerSet

    build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    w = dataclasses.replace(synth.WORKLOADS["decode_256"], bucket_bases=[200_000])
    tmap = synth.token_map(w.vocab, w.vc, w.seed)
    wq, wk = synth.wq_wk(w)
    m = EngramLayerSet.from_workload(w, tmap, device=dev)
    m.bind(0, w.table_seeds[0], synth.wkv_bf16(w), wq, wk)
    T = 50_032
    s = eg.engram_session_create(m.ctx)
    win = eg.engram_session_append(s, synth.zipf_tokens(T, w.vocab, seed=5))
    eg.engram_session_destroy(s)
    d_w = torch.from_numpy(win.view(np.int32)).to(dev)
    d_r = torch.empty((T, w.nb), dtype=torch.int32, device=dev)
    d_e = torch.empty((T, w.K), dtype=torch.int16, device=dev)
    sptr = stream.cuda_stream
    eg.engram_hash(m.ctx, 0, d_w, T, d_r, sptr)
    for _ in range(args.warmup):
        eg.engram_gather_dequant(m.ctx, 0, d_r, T, d_e, sptr)
    ms = timed(lambda i: eg.engram_gather_dequant(m.ctx, 0, d_r, T, d_e, sptr), args.steps, stream)
    eg.engram_sync(m.ctx, sptr)
    print(json.dumps({"case": "gather_small", "tokens": T, "table_rows": m.rows(0),
                      "ms": ms, "GB_per_s": T * 18720 / ms / 1e6}), flush=True)
    m.close()


def decode_small(args):
    """The decode step's kernels at full geometry on a small table, for ncu:
    256 sessions (3-token history), one token each per step, staged entry."""
    import dataclasses

    import torch

    import engram_gram_conditional_gb300 as eg
    import synth
    from engram_gram_conditional_gb300 import build
    from engram_gram_conditional_gb300.layer import EngramLayerSet

    build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    wd = dataclasses.replace(synth.WORKLOADS["decode_256"], bucket_bases=[200_000])
    tmap = synth.token_map(wd.vocab, wd.vc, wd.seed)
    wq, wk = synth.wq_wk(wd)
    dm = EngramLayerSet.from_workload(wd, tmap, device=dev)
    dm.bind(0, wd.table_seeds[0], synth.wkv_bf16(wd), wq, wk)
    S = wd.sessions
    sess = [eg.engram_session_create(dm.ctx) for _ in range(S)]
    streams = np.stack([synth.session_tokens(wd, i, wd.history + wd.steps) for i in range(S)])
    for i, s in enumerate(sess):
        eg.engram_session_append(s, streams[i, :wd.history])
    wins = [eg.engram_batch_append(sess, streams[:, wd.history + k]) for k in range(wd.steps)]
    d_wins = torch.from_numpy(np.stack(wins).view(np.int32)).to(dev)
    d_h = torch.from_numpy(synth.normal_bf16((S, wd.hc, wd.d), 1.0, 0, 77).view(np.int16)).to(dev)
    d_ws = torch.empty(eg.engram_forward_staged_workspace_bytes(dm.ctx, S), dtype=torch.uint8,
                       device=dev)
    sptr = stream.cuda_stream

    def fwd(i):
        eg.engram_forward_staged(dm.ctx, 0, d_wins[i % wd.steps], S, d_h, d_ws, None, sptr)

    for i in range(args.warmup):
        fwd(i)
    ms = timed(fwd, args.steps, stream)
    eg.engram_sync(dm.ctx, sptr)
    print(json.dumps({"case": "decode_small", "sessions": S, "table_rows": dm.rows(0),
                      "steps": args.steps, "ms_per_step": ms}), flush=True)
    for s in sess:
        eg.engram_session_destroy(s)
    dm.close()


def prepass_staged(ctx, T, w, d_win, d_h, peaks, sptr, stream, steps):
    """engram_prepass (staged: gather once, tcgen05 projection, kv to HBM) with
    fp32 and with BF16 kv, and the gate on each at the layer entry."""
    import torch

    import engram_gram_conditional_gb300 as eg

    ws = torch.empty(eg.engram_forward_staged_workspace_bytes(ctx, T), dtype=torch.uint8,
                     device=d_win.device)
    res = {"tokens": T}
    for name, fmt, dt, gate in (("f32", eg.KV_F32, torch.float32, eg.engram_gate),
                                ("bf16", eg.KV_BF16, torch.int16, eg.engram_gate_bf16kv)):
        d_kv = torch.empty((T, w.N), dtype=dt, device=d_win.device)
        for _ in range(3):
            eg.engram_prepass(ctx, 0, d_win, T, d_kv, fmt, ws, sptr)
            gate(ctx, 0, d_kv, d_win, T, d_h, None, sptr)
        ms_p = timed(lambda i: eg.engram_prepass(ctx, 0, d_win, T, d_kv, fmt, ws, sptr), steps,
                     stream)
        ms_g = timed(lambda i: gate(ctx, 0, d_kv, d_win, T, d_h, None, sptr), steps, stream)
        eg.engram_sync(ctx, sptr)
        kv_bytes = T * w.N * d_kv.element_size()
        gate_bytes = kv_bytes + T * 2 * w.hc * w.d * 2
        res[name] = {"prepass_ms": ms_p, "layer_entry_gate_ms": ms_g, "kv_bytes": kv_bytes,
                     "gate_GB_per_s": gate_bytes / ms_g / 1e6,
                     "gate_frac": gate_bytes / ms_g / 1e6 / peaks["hbm"]}
        del d_kv
    return res


def timed(fn, steps, stream):
    import torch

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(steps):
        fn(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) / steps


def extras(args, w, W, wq, wk, tmap, win0, d_win0, model, peaks, dev, sptr, stream):
    """Side measurements: the unfused stages at the prefill, and the decode batch."""
    import torch

    import engram_gram_conditional_gb300 as eg
    import synth
    from engram_gram_conditional_gb300.layer import EngramLayerSet

    out = {}
    ctx, T = model.ctx, w.tokens_per_session
    # unfused projection (TMA A operand) and the fused hash+gather+projection
    d_rows = torch.empty((T, w.nb), dtype=torch.int32, device=dev)
    d_emb = torch.empty((T, w.K), dtype=torch.int16, device=dev)
    d_kv = torch.empty((T, w.N), dtype=torch.float32, device=dev)
    eg.engram_hash(ctx, 0, d_win0, T, d_rows, sptr)
    eg.engram_gather_dequant(ctx, 0, d_rows, T, d_emb, sptr)
    for _ in range(3):
        eg.engram_project(ctx, 0, d_emb, T, d_kv, sptr)
    ms_p = timed(lambda i: eg.engram_project(ctx, 0, d_emb, T, d_kv, sptr), 50, stream)
    ms_pw = timed(lambda i: eg.engram_project_windows(ctx, 0, d_win0, T, d_kv, sptr), 50, stream)
    fl = 2.0 * w.N * w.K * T
    out["project"] = {"ms": ms_p, "tflops": fl / ms_p / 1e9,
                      "tc_frac": fl / ms_p / 1e9 / peaks["bf16"]}
    out["project_windows"] = {"ms": ms_pw, "tflops": fl / ms_pw / 1e9,
                              "tc_frac": fl / ms_pw / 1e9 / peaks["bf16"]}
    # hidden-independent pre-pass: hash + gather + projection as soon as the
    # tokens are known (kv fp32 to HBM, off the layer's critical path), then at
    # the layer entry only the gate runs on the stored kv
    d_h = torch.from_numpy(synth.normal_bf16((T, w.hc, w.d), 1.0, w.seed, 4242).view(np.int16)).to(dev)
    for _ in range(3):
        eg.engram_gate(ctx, 0, d_kv, d_win0, T, d_h, None, sptr)
    ms_g = timed(lambda i: eg.engram_gate(ctx, 0, d_kv, d_win0, T, d_h, None, sptr), 50, stream)
    gate_bytes = T * (w.N * 4 + 2 * w.hc * w.d * 2)
    out["prepass"] = {"tokens": T, "prepass_ms": ms_pw, "layer_entry_gate_ms": ms_g,
                      "kv_bytes": T * w.N * 4,
                      "gate_GB_per_s": gate_bytes / ms_g / 1e6,
                      "gate_frac": gate_bytes / ms_g / 1e6 / peaks["hbm"]}
    out["prepass_staged"] = prepass_staged(ctx, T, w, d_win0, d_h, peaks, sptr, stream, 50)
    del d_rows, d_emb, d_kv, d_h

    # decode: 256 sessions x 1 token per step, 384M-row table resident in HBM
    wd = synth.WORKLOADS["decode_256"]
    dm = EngramLayerSet.from_workload(wd, tmap, device=dev)
    dm.bind(0, wd.table_seeds[0], model.tensors[0]["wkv"], wq, wk)
    S = wd.sessions
    sess = [eg.engram_session_create(dm.ctx) for _ in range(S)]
    streams = np.stack([synth.session_tokens(wd, i, wd.history + wd.steps) for i in range(S)])
    for i, s in enumerate(sess):
        eg.engram_session_append(s, streams[i, :wd.history])
    wins = [eg.engram_batch_append(sess, streams[:, wd.history + step])
            for step in range(wd.steps)]
    d_wins = torch.from_numpy(np.stack(wins).view(np.int32)).to(dev)
    d_h = torch.from_numpy(synth.normal_bf16((S, wd.hc, wd.d), 1.0, 0, 77).view(np.int16)).to(dev)
    ws_bytes = max(eg.engram_workspace_bytes(dm.ctx, S),
                   eg.engram_forward_staged_workspace_bytes(dm.ctx, S))
    d_ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    bytes_step = w.N * w.K * 2 + S * (6336 + 81920 + 16)
    entries = {"staged": eg.engram_forward_staged, "fused": eg.engram_forward}
    for name, fwd in entries.items():
        for i in range(5):
            fwd(dm.ctx, 0, d_wins[i], S, d_h, d_ws, None, sptr)
        ms_d = timed(lambda i: fwd(dm.ctx, 0, d_wins[i % wd.steps], S, d_h, d_ws, None, sptr),
                     wd.steps, stream)
        eg.engram_sync(dm.ctx, sptr)
        gbs = bytes_step / ms_d / 1e6
        out["decode" if name == "staged" else "decode_fused"] = {
            "entry": fwd.__name__, "tokens_per_s": S / (ms_d / 1000.0), "ms_per_step": ms_d,
            "sessions": S, "steps": wd.steps, "table_rows": dm.rows(0),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"], "bytes_per_step": bytes_step,
                         "traffic": DECODE_GEMM_DRAM_BYTES if name == "staged" else None}}
    queue_oracle(out["decode"], wd, 0, W, wq, wk, np.stack(wins),
                 f"decode tokens ({wd.steps} steps x {S} sessions, {dm.rows(0):,}-row table)")
    # the decode step as a pre-pass (as soon as the step's tokens are known)
    # plus the gate at the layer entry
    d_kvd = torch.empty((S, w.N), dtype=torch.float32, device=dev)
    for i in range(3):
        eg.engram_project_windows(dm.ctx, 0, d_wins[i], S, d_kvd, sptr)
        eg.engram_gate(dm.ctx, 0, d_kvd, d_wins[i], S, d_h, None, sptr)
    ms_pwd = timed(lambda i: eg.engram_project_windows(dm.ctx, 0, d_wins[i % wd.steps], S, d_kvd,
                                                       sptr), wd.steps, stream)
    ms_gd = timed(lambda i: eg.engram_gate(dm.ctx, 0, d_kvd, d_wins[i % wd.steps], S, d_h, None,
                                           sptr), wd.steps, stream)
    eg.engram_sync(dm.ctx, sptr)
    out["decode_prepass"] = {"sessions": S, "prepass_ms": ms_pwd, "layer_entry_gate_ms": ms_gd}
    out["decode_prepass_staged"] = prepass_staged(dm.ctx, S, wd, d_wins[0], d_h, peaks, sptr,
                                                  stream, wd.steps)
    del d_kvd

    # gather: unfused engram_gather_dequant over the 384M-row table, 50,032 tokens
    Tg = 50_032
    sg = eg.engram_session_create(dm.ctx)
    wg = eg.engram_session_append(sg, synth.zipf_tokens(Tg, wd.vocab, seed=5))
    d_wg = torch.from_numpy(wg.view(np.int32)).to(dev)
    d_rg = torch.empty((Tg, w.nb), dtype=torch.int32, device=dev)
    d_eg = torch.empty((Tg, w.K), dtype=torch.int16, device=dev)
    eg.engram_hash(dm.ctx, 0, d_wg, Tg, d_rg, sptr)
    for _ in range(3):
        eg.engram_gather_dequant(dm.ctx, 0, d_rg, Tg, d_eg, sptr)
    ms_g = timed(lambda i: eg.engram_gather_dequant(dm.ctx, 0, d_rg, Tg, d_eg, sptr), 20, stream)
    eg.engram_sync(dm.ctx, sptr)
    gb_alg = Tg * (w.nb * 4 + w.nb * 264 + w.K * 2)
    out["gather"] = {"tokens": Tg, "table_rows": dm.rows(0), "ms": ms_g,
                     "GB_per_s": gb_alg / ms_g / 1e6, "frac": gb_alg / ms_g / 1e6 / peaks["hbm"],
                     "bytes_per_token": w.nb * 4 + w.nb * 264 + w.K * 2}
    for s in sess + [sg]:
        eg.engram_session_destroy(s)
    dm.close()

    # the BF16-table variant (rows stored dequantised, 512 B, no scales) at the
    # prefill size: the staged forward and the standalone gather
    bm = EngramLayerSet.from_workload(w, tmap, device=dev)
    try:
        bm.bind(0, w.table_seeds[0], model.tensors[0]["wkv"], wq, wk, flags=eg.BIND_TABLE_BF16)
        d_hb = torch.from_numpy(synth.normal_bf16((T, w.hc, w.d), 1.0, w.seed, 5151).view(np.int16)).to(dev)
        d_wsb = torch.empty(eg.engram_forward_staged_workspace_bytes(bm.ctx, T), dtype=torch.uint8,
                            device=dev)
        for _ in range(3):
            eg.engram_forward_staged(bm.ctx, 0, d_win0, T, d_hb, d_wsb, None, sptr)
        ms_b = timed(lambda i: eg.engram_forward_staged(bm.ctx, 0, d_win0, T, d_hb, d_wsb, None,
                                                        sptr), 20, stream)
        d_rb = torch.empty((T, w.nb), dtype=torch.int32, device=dev)
        d_eb = torch.empty((T, w.K), dtype=torch.int16, device=dev)
        eg.engram_hash(bm.ctx, 0, d_win0, T, d_rb, sptr)
        for _ in range(3):
            eg.engram_gather_dequant(bm.ctx, 0, d_rb, T, d_eb, sptr)
        ms_bg = timed(lambda i: eg.engram_gather_dequant(bm.ctx, 0, d_rb, T, d_eb, sptr), 20, stream)
        eg.engram_sync(bm.ctx, sptr)
        gb_b = T * (w.nb * 4 + w.nb * w.row_dim * 2 + w.K * 2)
        out["bf16_table"] = {"tokens": T, "table_rows": bm.rows(0), "row_bytes": w.row_dim * 2,
                             "staged_ms": ms_b, "staged_tflops": fl / ms_b / 1e9,
                             "gather_ms": ms_bg, "gather_GB_per_s": gb_b / ms_bg / 1e6}
    finally:
        bm.close()
    return out


def long_small(args):
    """The long prefill's kernels on 4.8M-row tables, for ncu: same batch,
    chunks and launches, a table the capture can hold."""
    import torch

    from engram_gram_conditional_gb300 import build

    build.build()
    import synth

    dev = torch.device("cuda", 0)
    wl = synth.WORKLOADS["prefill_50k_2layer"]
    tmap = synth.token_map(wl.vocab, wl.vc, wl.seed)
    out = long_prefill(tmap, load_peaks(), dev, torch.cuda.current_stream(), small=True,
                       steps=args.steps)
    print(json.dumps({"case": "long_small", **out}), flush=True)


def long_prefill(tmap, peaks, dev, stream, small=False, steps=6):
    """The long-prefill workload: one history of 50,032 tokens with three image
    spans of 1,024 tokens, appended once and run through layers L1 and L14
    (64M-row tables, primes of L14 after L1's, random-init wkv per layer) with
    the staged forward.  FLOPs count the 46,960 text rows."""
    import dataclasses

    import torch

    import engram_gram_conditional_gb300 as eg
    import synth
    from engram_gram_conditional_gb300.layer import EngramLayerSet

    wl = synth.WORKLOADS["prefill_50k_2layer"]
    if small:
        wl = dataclasses.replace(wl, bucket_bases=[200_000, 200_000])
    lm = EngramLayerSet.from_workload(wl, tmap, device=dev)
    try:
        Ws = []
        for l in range(2):
            q, k = synth.wq_wk(wl, l)
            Ws.append((synth.wkv_bf16(wl, l), q, k))
            lm.bind(l, wl.table_seeds[l], Ws[l][0], q, k)
        T = wl.tokens_per_session
        sess = eg.engram_session_create(lm.ctx)
        win = eg.engram_session_append(sess, synth.session_tokens(wl, 0, T),
                                       synth.image_flags(T, wl.image_spans))
        eg.engram_session_destroy(sess)
        text = int((win[:, 0] != eg.DEAD).sum())
        d_win = torch.from_numpy(win.view(np.int32)).to(dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(wl.seed + 50032)
        d_h = torch.randn((T, wl.hc, wl.d), generator=gen, device=dev).to(torch.bfloat16)
        ws = torch.empty(eg.engram_forward_staged_workspace_bytes(lm.ctx, T), dtype=torch.uint8,
                         device=dev)
        sptr = stream.cuda_stream
        for l in range(2):
            eg.engram_forward_staged(lm.ctx, l, d_win, T, d_h, ws, None, sptr)
        ms = timed(lambda i: eg.engram_forward_staged(lm.ctx, i % 2, d_win, T, d_h, ws, None, sptr),
                   steps, stream)
        eg.engram_sync(lm.ctx, sptr)
        fl = 2.0 * wl.N * wl.K * text
        out = {"tokens": T, "text_tokens": text, "layers": 2,
               "table_rows": [lm.rows(0), lm.rows(1)],
               "ms_per_layer": ms, "tokens_per_s_per_layer": T / (ms / 1000.0),
               "tflops": fl / ms / 1e9, "tc_frac": fl / ms / 1e9 / peaks["bf16"]}
        if not small:
            queue_oracle(out, wl, 0, *Ws[0], win,
                         f"positions of the long prefill, layer L1 ({lm.rows(0):,}-row table)")
        return out
    finally:
        lm.close()


def host_pipeline(model, W, wq, wk, tmap, peaks, dev, stream):
    """The host-table workload: 8 sessions x 1,024 tokens per step, the MXFP8
    table (64M rows, 17 GB) in pinned host memory read through UVA.  Reports the
    host link (a pinned host-to-device copy), the row gather over it, the GEMM
    on the staged rows, and the staged forward run serially or pipelined: the
    rows of step i + 1 staged on a side stream while step i's GEMM runs."""
    import dataclasses

    import torch

    import engram_gram_conditional_gb300 as eg
    import synth
    from engram_gram_conditional_gb300.layer import EngramLayerSet

    with open("/proc/meminfo") as f:
        info = {ln.split(":")[0]: int(ln.split()[1]) * 1024 for ln in f if ":" in ln}
    # The stated table (384,006,168 rows, 101.4 GB) when the host can pin it and
    # keep 48 GB free; else the 64M-row table of the long prefill (16.9 GB).
    avail = info.get("MemAvailable", 0)
    if avail >= 384_006_168 * 264 + 48 * 2**30:
        bases, why = [16_000_000], f"the stated 384M rows ({avail / 2**30:.0f} GB available)"
    elif avail >= 48 * 2**30:
        bases, why = [2_666_666], (f"64M rows: {avail / 2**30:.0f} GB available, below the "
                                   f"101.4 GB table + 48 GB")
    else:
        return {"skipped": "less than 48 GB of host memory available for the pinned table"}
    wh = dataclasses.replace(synth.WORKLOADS["host_table_8x1024"], bucket_bases=bases)
    hm = EngramLayerSet.from_workload(wh, tmap, device=dev)

    def anon_huge() -> int:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("AnonHugePages:"):
                    return int(ln.split()[1]) * 1024
        return 0

    try:
        with open("/sys/kernel/mm/transparent_hugepage/enabled") as f:
            thp_mode = f.read().strip()
    except OSError:
        thp_mode = "unknown"
    try:
        huge0 = anon_huge()
        hm.bind(0, wh.table_seeds[0], model.tensors[0]["wkv"], wq, wk, host_table=True)
        huge_gb = (anon_huge() - huge0) / 2**30
        T = wh.sessions * wh.tokens_per_session
        nbatch = 4
        wins, hids = [], []
        for b in range(nbatch):
            parts = []
            for i in range(wh.sessions):
                s = eg.engram_session_create(hm.ctx)
                parts.append(eg.engram_session_append(
                    s, synth.session_tokens(wh, b * wh.sessions + i, wh.tokens_per_session)))
                eg.engram_session_destroy(s)
            wins.append(torch.from_numpy(np.concatenate(parts).view(np.int32)).to(dev))
            hids.append(torch.from_numpy(
                synth.normal_bf16((T, wh.hc, wh.d), 1.0, wh.seed, 9000 + b).view(np.int16)).to(dev))
        wsb = eg.engram_forward_staged_workspace_bytes(hm.ctx, T)
        ws = [torch.empty(wsb, dtype=torch.uint8, device=dev) for _ in range(2)]
        sptr = stream.cuda_stream
        side = torch.cuda.Stream(device=dev)

        # the host link: a pinned 1 GiB host-to-device copy
        hbuf = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
        dbuf = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(2):
                dbuf.copy_(hbuf, non_blocking=True)
            ms_h2d = timed(lambda i: dbuf.copy_(hbuf, non_blocking=True), 5, stream)
        del hbuf, dbuf
        # the link read through UVA: a kernel (the E8M0 scan of the bind) reading
        # the host table's scale bytes in order, up to 2 GiB
        scales = hm.tensors[0]["scales"]
        n_uva = int(min(scales.nbytes, 2 << 30))
        eg.engram_scale_range(hm.ctx, scales, n_uva)
        t_u0 = time.perf_counter()
        for _ in range(3):
            eg.engram_scale_range(hm.ctx, scales, n_uva)
        uva_gbs = 3 * n_uva / (time.perf_counter() - t_u0) / 1e9

        def stage(i, st):
            eg.engram_stage_rows(hm.ctx, 0, wins[i % nbatch], T, ws[i % 2], st)

        def gemm(i):
            eg.engram_forward_staged_rows(hm.ctx, 0, wins[i % nbatch], T, hids[i % nbatch],
                                          ws[i % 2], None, sptr)

        for i in range(3):
            eg.engram_forward_staged(hm.ctx, 0, wins[i % nbatch], T, hids[i % nbatch], ws[0], None,
                                     sptr)
        ms_stage = timed(lambda i: stage(0, sptr), 10, stream)
        ms_gemm = timed(lambda i: gemm(0), 10, stream)
        steps = 12
        ms_serial = timed(lambda i: eg.engram_forward_staged(
            hm.ctx, 0, wins[i % nbatch], T, hids[i % nbatch], ws[0], None, sptr), steps, stream)

        # pipelined: stage(i + 1) on the side stream overlaps gemm(i) on the main one
        staged = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]

        def pipelined():
            torch.cuda.synchronize()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            side.wait_event(ev0)
            stage(0, side.cuda_stream)
            staged[0].record(side)
            for i in range(steps):
                if i + 1 < steps:
                    if i >= 1:
                        side.wait_event(done[(i + 1) % 2])  # step i - 1 used that workspace
                    stage(i + 1, side.cuda_stream)
                    staged[(i + 1) % 2].record(side)
                stream.wait_event(staged[i % 2])
                gemm(i)
                done[i % 2].record(stream)
            ev1.record(stream)
            torch.cuda.synchronize()
            return ev0.elapsed_time(ev1) / steps

        pipelined()
        ms_pipe = pipelined()
        eg.engram_sync(hm.ctx, sptr)
        link_bytes = T * wh.nb * 264  # codes and scales read over the link per step
        out = {"tokens_per_step": T, "table_rows": hm.rows(0), "table": "pinned host, UVA",
               "table_bytes": hm.rows(0) * 264, "table_choice": why,
               # the table's backing: transparent huge pages gained by the bind
               # (2 MB pages shorten the GPU's translation of random host rows)
               "thp_mode": thp_mode, "huge_pages_GB": huge_gb,
               "h2d_GB_per_s": (1 << 30) / ms_h2d / 1e6,
               "uva_read_GB_per_s": uva_gbs,
               "stage_ms": ms_stage, "stage_link_GB_per_s": link_bytes / ms_stage / 1e6,
               "stage_frac_of_link": (link_bytes / ms_stage / 1e6) / ((1 << 30) / ms_h2d / 1e6),
               "stage_frac_of_uva_read": (link_bytes / ms_stage / 1e6) / uva_gbs,
               "gemm_ms": ms_gemm, "serial_ms_per_step": ms_serial,
               "pipelined_ms_per_step": ms_pipe,
               "pipelined_tokens_per_s": T / (ms_pipe / 1000.0)}
        queue_oracle(out, wh, 0, W, wq, wk, torch.cat(wins).cpu().numpy().view(np.uint32),
                     f"tokens of {nbatch} host-table steps ({hm.rows(0):,}-row table)")
        return out
    finally:
        hm.close()


# Oracle baselines of the side workloads, queued while the GPU lines run and
# timed on the host cores at the end: (line dict, workload, layer, W, wq, wk,
# windows of the workload's tokens, what the tokens are).
_ORACLE_JOBS = []


def queue_oracle(line: dict, wcfg, layer: int, W, wq, wk, win, what: str):
    _ORACLE_JOBS.append((line, wcfg, layer, W, wq, wk, np.asarray(win).reshape(-1, 4), what))


def run_oracle_jobs(args):
    """Each queued workload: the oracle on a stated random subset of its token
    rows (hidden drawn for the sample: the oracle's time does not depend on the
    values), over all host cores, extrapolated linearly to the workload."""
    if args.cpu_sample_configs <= 0:
        for line, *_ in _ORACLE_JOBS:
            line["cpu_baseline"] = {"skipped": "--cpu-sample-configs 0"}
        return
    import oracle as O
    import synth

    O.build()
    cores = cpu_cores()
    for line, wcfg, layer, W, wq, wk, win, what in _ORACLE_JOBS:
        g = O.Geom(vocab=wcfg.vocab, vc=wcfg.vc, min_n=wcfg.min_n, max_n=wcfg.max_n,
                   heads=wcfg.heads, row_dim=wcfg.row_dim, hc=wcfg.hc, d=wcfg.d,
                   pad_cid=wcfg.pad_cid, eps=wcfg.eps)
        p = O.layer_params(g, wcfg.hash_seeds, wcfg.bucket_bases, layer)
        n = min(args.cpu_sample_configs, len(win))
        idx = np.random.default_rng(4096).choice(len(win), n, replace=False)
        win_s = np.ascontiguousarray(win[idx])
        hid_s = synth.normal_bf16((n, wcfg.hc, wcfg.d), 1.0, wcfg.seed, 31337)
        t0 = time.perf_counter()
        O.forward(g, wcfg.table_seeds[layer], p, W, wq, wk, win_s, hid_s, np.arange(n),
                  nthreads=cores, want_h64=False)
        el = time.perf_counter() - t0
        rate = n / el
        line["cpu_baseline"] = {
            "value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} random token rows of the {len(win)} {what} (numpy default_rng(4096)), "
                      f"threads over tokens", "seconds": el,
            "extrapolated": f"linear: the {len(win)} tokens take {len(win) / rate:.0f} s"}


def cpu_baseline(args, w, W, wq, wk, win, hidden):
    import oracle as O

    O.build()
    g = O.Geom(vocab=w.vocab, vc=w.vc, min_n=w.min_n, max_n=w.max_n, heads=w.heads,
               row_dim=w.row_dim, hc=w.hc, d=w.d, pad_cid=w.pad_cid, eps=w.eps)
    p = O.layer_params(g, w.hash_seeds, w.bucket_bases, 0)
    cores = cpu_cores()
    n = max(cores, args.cpu_sample)
    idx = np.random.default_rng(1).integers(0, w.tokens_per_session, n)
    el = run_oracle_timed(w, W, wq, wk, hidden, win, g, p, idx, cores)
    return {"value": n / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} random tokens of the {w.tokens_per_session}-token prefill, "
                      f"threads over tokens", "seconds": el}


if __name__ == "__main__":
    main()
