#!/usr/bin/env python3
"""Benchmark of one QUOKA chunked-prefill step on GB300.

A step is one chunk through the whole hot path: query subselection, cosine
scoring of the history, top-B per KV head, gather, and attention over the kept
history plus the causal chunk.  The workload is the Llama-3-8B-shaped GQA
attention layer: H_q=32, H_kv=8, d=128, one chunk of C=2048 queries over
T=32768 cached keys, N_q=64, B=2048, bf16, synthetic seeded inputs (the
massive-activation recipe of workloads.py).  The metric is chunk tokens per
second (C / step time).

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.  Under torchrun every rank runs
its own replica of the workload (the path has no cross-GPU exchange).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_attention_chunked_gb300 import workloads as wl  # noqa: E402

METRIC = "chunk tokens/sec for QUOKA select+attend at 32K/128K history; % HBM/TC roofline"
WORKLOADS = {"gqa32k": wl.GQA_32K_BF16, "gqa128k": wl.GQA_128K_BF16, "decode32k": wl.DECODE_32K_BF16,
             "tiny": wl.TINY_MHA_FP32}   # tiny: the small parity case, for quick checks of the harness
RAGGED = {"ragged8": wl.RAGGED_8x_BF16}  # one quoka_chunk_attend_varlen call over a ragged batch
FP32_FMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # SMs x FP32 lanes x 2 flop x max SM clock

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one tensor-core attention launch per
# workload, from one ncu capture, and a digest of the kernel sources that capture ran on: once the
# sources change the figure no longer describes the kernel and the bench reports null.
ATTEND_TRAFFIC = {"gqa32k": 33_622_272, "ragged8": 337_428_224}
ATTEND_TRAFFIC_SOURCES = ("attend_tc.cu", "tc_common.cuh")   # the attention kernel and its tcgen05/TMA wrappers
ATTEND_TRAFFIC_SHA256 = "764c4a01c7ebc4af15c9419bfcf06cf8a6f6dd868437799e090c2de03af2a572"


def attend_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ATTEND_TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "sparse_attention_chunked_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def attend_traffic(workload: str):
    if workload not in ATTEND_TRAFFIC or attend_sources_sha256() != ATTEND_TRAFFIC_SHA256:
        return None
    return ATTEND_TRAFFIC[workload]
L2_FLUSH_BYTES = 512 << 20                              # > 3x the 129 MB L2
INPUT_SETS = 3    # timed steps rotate over this many copies of the inputs (> 3x L2 together at 32K history)


# ---------------------------------------------------------------- multi-rank plumbing

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(backend: str):
    rank, world, _ = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)
    return rank, world


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def job_throughput(tokens_per_rank_step: int, world: int, step_ms_max: float) -> float:
    """Whole-job tokens/s: every rank processes its own chunk per step; the slowest rank's step time counts."""
    return tokens_per_rank_step * world / (step_ms_max * 1e-3)


def max_over_ranks(x: float, device="cpu") -> float:
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        t = torch.tensor([x], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return x


# ---------------------------------------------------------------- algorithmic work per stage

def stage_work(cfg: wl.ChunkConfig, gqa: str, query_agg: str = "max") -> dict:
    """Bytes / flops each stage must move or compute (what the method needs, not what the kernels do)."""
    e = 2 if cfg.dtype == "bf16" else 4
    n = min(cfg.N_q, cfg.C)
    B_e = min(cfg.B, cfg.T)
    if query_agg == "mean":       # the mean over tokens is one row per head (max) or per group (mean)
        R = cfg.G if gqa == "max" else 1
    else:
        R = cfg.G * n if gqa == "max" else n
    return {
        "select": {"bytes": cfg.H_q * cfg.C * cfg.d * e},                               # read Q once
        "score": {"bytes": cfg.H_kv * cfg.T * cfg.d * e + cfg.H_kv * cfg.T * 4,         # read K, write scores
                  "flops": 2 * cfg.H_kv * R * cfg.T * cfg.d},
        "topk": {"bytes": cfg.H_kv * cfg.T * 4 + cfg.H_kv * B_e * 4},
        "gather": {"bytes": 2 * 2 * cfg.H_kv * B_e * cfg.d * e},                        # read + write K and V rows
        "attend": {"flops": 4 * cfg.H_q * cfg.d * (cfg.C * B_e + cfg.C * (cfg.C + 1) // 2),
                   "bytes": 2 * cfg.H_q * cfg.C * cfg.d * e + 2 * cfg.H_kv * (B_e + cfg.C) * cfg.d * e},
    }


def dense_flops(cfg: wl.ChunkConfig) -> int:
    return 4 * cfg.H_q * cfg.d * (cfg.C * cfg.T + cfg.C * (cfg.C + 1) // 2)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks during the timed region

class ClockSampler:
    """Samples nvidia-smi every 200 ms in the background (SM clock, max clock, throttle reasons)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.dev = device_index

    def _target(self):
        try:
            props = torch.cuda.get_device_properties(self.dev)
            return "GPU-" + str(props.uuid)
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            return vis.split(",")[self.dev] if vis else str(self.dev)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", self._target()],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        time.sleep(0.05)
        rows = [r for r in self.rows if r[0].replace(".", "").isdigit()]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][1]), "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- the GPU arm

def run_quoka(args, rank, world, local_rank, light=False):
    """One chunk of a WORKLOADS entry.  light: a sub-record of the suite (no end-to-end legs, the CPU
    baseline on one KV group)."""
    from sparse_attention_chunked_gb300 import build as qbuild
    from sparse_attention_chunked_gb300 import quoka as q

    qbuild.build()
    q.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = WORKLOADS[args.workload]
    x = wl.make_chunk(cfg, args.seed)
    Q, Kh, Vh = x.Q.to(dev), x.K_hist.to(dev), x.V_hist.to(dev)
    Kc, Vc = x.K_chunk.to(dev), x.V_chunk.to(dev)
    shape = q.shape_of(Q, Kh)
    params = q.params_of(args.gqa, args.engine, score_fn=args.score_fn, query_agg=args.query_agg)
    ws = q.make_workspace(shape, cfg.N_q, cfg.B, params, device=dev)
    n = min(cfg.N_q, cfg.C)
    H_sel = cfg.H_q if args.gqa == "max" else cfg.H_kv
    B_e = min(cfg.B, cfg.T)
    O = torch.empty_like(Q)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    names = ["select", "score", "topk", "gather", "attend"]

    def new_events(k):
        return [torch.cuda.Event(enable_timing=True) for _ in range(k)]

    # Copies of the step's inputs at other addresses: the timed steps rotate over
    # them, so every step reads inputs last touched INPUT_SETS - 1 steps (several
    # hundred MB of traffic) earlier, i.e. from HBM, without a flush kernel.
    sets = [(Q, Kh, Vh, Kc, Vc)] + [tuple(t.clone() for t in (Q, Kh, Vh, Kc, Vc)) for _ in range(INPUT_SETS - 1)]
    set_bytes = sum(t.numel() * t.element_size() for t in sets[0])
    # each input set's own stage intermediates, for the stage-by-stage breakdown
    inter = [{"q_idx": torch.empty((H_sel, n), dtype=torch.int32, device=dev),
              "scores": torch.empty((cfg.H_kv, cfg.T), dtype=torch.float32, device=dev),
              "sel": torch.empty((cfg.H_kv, B_e), dtype=torch.int32, device=dev),
              "Ks": torch.empty((cfg.H_kv, B_e, cfg.d), dtype=Q.dtype, device=dev),
              "Vs": torch.empty((cfg.H_kv, B_e, cfg.d), dtype=Q.dtype, device=dev)} for _ in sets]

    def stage_call(i, si):
        Qx, Khx, Vhx, Kcx, Vcx = sets[si]
        t = inter[si]
        if i == 0:
            q.quoka_select_queries(shape, Qx, cfg.N_q, params, t["q_idx"], ws, stream)
        elif i == 1:
            q.quoka_score_keys(shape, Qx, t["q_idx"], cfg.N_q, Khx, params, t["scores"], ws, stream)
        elif i == 2:
            q.quoka_topk(shape, t["scores"], cfg.B, t["sel"], ws, stream)
        elif i == 3:
            q.quoka_gather(shape, Khx, Vhx, t["sel"], B_e, t["Ks"], t["Vs"], stream)
        else:
            q.quoka_sparse_attend(shape, Qx, t["Ks"], t["Vs"], B_e, Kcx, Vcx, params, O, None, ws, stream)

    # the key-norm cache of every input set, as quoka_append_kv_norms would have left it when the
    # history was appended (built once, outside the timed region)
    inv_sets = {}
    if args.key_norm_cache:
        for xs in sets:
            inv = torch.empty((cfg.H_kv, cfg.T), dtype=torch.float32, device=dev)
            q.quoka_key_inv_norms(shape, xs[1], 0, cfg.T, inv, stream)
            inv_sets[id(xs[1])] = inv
        torch.cuda.synchronize(dev)

    def step_call(si):
        # the step: one quoka_chunk_attend (every stage of the path)
        Qx, Khx, Vhx, Kcx, Vcx = sets[si]
        if args.key_norm_cache:
            q.quoka_chunk_attend_cached(shape, Qx, Khx, Vhx, Kcx, Vcx, inv_sets[id(Khx)], cfg.N_q, cfg.B, params, O,
                                        None, None, ws, stream)
        else:
            q.quoka_chunk_attend(shape, Qx, Khx, Vhx, Kcx, Vcx, cfg.N_q, cfg.B, params, O, None, None, ws, stream)

    def capture(calls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c()
        return g

    with torch.cuda.stream(stream):   # every call once per set (fills the intermediates, sets up the kernels)
        for si in range(INPUT_SETS):
            for i in range(len(names)):
                stage_call(i, si)
            step_call(si)
    torch.cuda.synchronize(dev)
    # The timed steps: K consecutive steps, rotating over the input sets, captured as ONE graph (the
    # library only enqueues kernels, so a captured call replays the identical launches; consecutive
    # kernels overlap launch and prologue through programmatic dependent launch).  Warm-up: W steps.
    before = q.quoka_launch_count()
    step_graph_k = capture([(lambda si=k % INPUT_SETS: step_call(si)) for k in range(args.steps)])
    launches_per_step = (q.quoka_launch_count() - before) // args.steps
    warm_graph = capture([(lambda si=k % INPUT_SETS: step_call(si)) for k in range(args.warmup)])
    one_step = capture([lambda: step_call(0)])
    # Stage breakdown: each stage call R times back to back on the rotating input sets, one graph each.
    R = max(args.steps, 2 * INPUT_SETS)
    stage_graphs = [capture([(lambda i=i, si=k % INPUT_SETS: stage_call(i, si)) for k in range(R)])
                    for i in range(len(names))]

    sampler = ClockSampler(local_rank)
    sampler.start()
    with torch.cuda.stream(stream):
        t_w = time.perf_counter()
        done = 0
        while done < 1 or time.perf_counter() - t_w < 0.5:   # W warm-up steps; also the clock sampler's lead-in
            warm_graph.replay()
            for g in stage_graphs:
                g.replay()
            done += 1
        warm_graph.replay()
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        e_rot = new_events(2)               # the headline: K steps back to back, rotating input sets
        torch.cuda.nvtx.range_push("timed_steps")   # lets a profiler select exactly these launches
        e_rot[0].record(stream)
        step_graph_k.replay()
        e_rot[1].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        barrier()
        wall = time.perf_counter() - wall0
        stage_ms = {}
        for i, nm in enumerate(names):
            e = new_events(2)
            e[0].record(stream)
            stage_graphs[i].replay()
            e[1].record(stream)
            torch.cuda.synchronize(dev)
            stage_ms[nm] = [e[0].elapsed_time(e[1]) / R]
        step_evs = []
        for _ in range(max(3, args.steps // 4)):
            flush.zero_()                   # L2 written over before this replay (outside the events)
            e = new_events(2)
            e[0].record(stream)
            one_step.replay()
            e[1].record(stream)
            step_evs.append(e)
        torch.cuda.synchronize(dev)
    launches = launches_per_step * args.steps
    assert q.quoka_get_last_device_error(ws, stream) == 0
    step_ms = max_over_ranks(e_rot[0].elapsed_time(e_rot[1]) / args.steps, dev)
    flush_step_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in step_evs), dev)
    staged_ms = sum(v[0] for v in stage_ms.values())

    # dense full-history attention on the same chunk: the speedup reference
    dense_ms = None
    if not args.no_dense:
        Od = torch.empty_like(Q)
        dsteps = max(3, args.steps // 4)
        with torch.cuda.stream(stream):
            for _ in range(2):
                q.quoka_dense_attend(shape, Q, Kh, Vh, Kc, Vc, params, Od, None, ws, stream)
            ts = []
            for _ in range(dsteps):
                flush.zero_()
                e = new_events(2)
                e[0].record(stream)
                q.quoka_dense_attend(shape, Q, Kh, Vh, Kc, Vc, params, Od, None, ws, stream)
                e[1].record(stream)
                ts.append(e)
        torch.cuda.synchronize(dev)
        dense_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ts), dev)

    def measure_e2e():
        # end to end through quoka_chunk_attend: every step's Q, K, V come from pinned host memory and
        # its O goes back to it inside the timed region; the history is a device-resident cache (rotated
        # over the input sets, so it is read from HBM).  Measured two ways: one step at a time on one
        # stream, and as a serving loop where step k's compute overlaps step k+1's upload and step k-1's
        # download (two device buffers, three streams).
        # Q, K_chunk and V_chunk sit back to back in one pinned host buffer and in one device buffer per
        # slot, so a step's inputs go up in one copy; the library takes the three as views of it
        parts = (x.Q, x.K_chunk, x.V_chunk)
        sizes = [t.numel() for t in parts]
        host_in = torch.empty(sum(sizes), dtype=Q.dtype).pin_memory()
        off = 0
        for t, n_el in zip(parts, sizes):
            host_in[off:off + n_el].copy_(t.reshape(-1).to(Q.dtype))
            off += n_el

        def views(buf):
            a, b = sizes[0], sizes[0] + sizes[1]
            return buf[:a].view(Q.shape), buf[a:b].view(Kc.shape), buf[b:].view(Vc.shape)

        Ohs = [torch.empty(O.shape, dtype=O.dtype).pin_memory() for _ in range(2)]
        dev_in = [torch.empty(sum(sizes), dtype=Q.dtype, device=dev) for _ in range(2)]
        bufs = [(*views(dev_in[i]), torch.empty_like(O)) for i in range(2)]
        h2d = host_in.numel() * host_in.element_size()
        d2h = Ohs[0].numel() * Ohs[0].element_size()

        def attend_call(xs, Qd, Kcd, Vcd, Od, st):
            if args.key_norm_cache:
                q.quoka_chunk_attend_cached(shape, Qd, xs[1], xs[2], Kcd, Vcd, inv_sets[id(xs[1])], cfg.N_q, cfg.B, params,
                                            Od, None, None, ws, st)
            else:
                q.quoka_chunk_attend(shape, Qd, xs[1], xs[2], Kcd, Vcd, cfg.N_q, cfg.B, params, Od, None, None, ws, st)

        def e2e_serial_step(k):
            Qd, Kcd, Vcd, Od = bufs[0]
            dev_in[0].copy_(host_in, non_blocking=True)
            attend_call(sets[k % INPUT_SETS], Qd, Kcd, Vcd, Od, stream)
            Ohs[0].copy_(Od, non_blocking=True)

        with torch.cuda.stream(stream):
            for k in range(args.warmup):
                e2e_serial_step(k)
            torch.cuda.synchronize(dev)
            e = new_events(2)
            e[0].record(stream)
            for k in range(args.steps):
                e2e_serial_step(k)
            e[1].record(stream)
        torch.cuda.synchronize(dev)
        e2e_serial_ms = max_over_ranks(e[0].elapsed_time(e[1]) / args.steps, dev)

        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        def e2e_pipelined(n):
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_done = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            for k in range(n):
                b = k % 2
                Qd, Kcd, Vcd, Od = bufs[b]
                with torch.cuda.stream(up):
                    if k >= 2:
                        up.wait_event(ev_done[k - 2])     # buffer b's inputs were consumed by step k-2
                    dev_in[b].copy_(host_in, non_blocking=True)
                    ev_in[k].record(up)
                stream.wait_event(ev_in[k])
                if k >= 2:
                    stream.wait_event(ev_out[k - 2])      # buffer b's output was read back
                attend_call(sets[k % INPUT_SETS], Qd, Kcd, Vcd, Od, stream)
                ev_done[k].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(ev_done[k])
                    Ohs[b].copy_(Od, non_blocking=True)
                    ev_out[k].record(down)
            return ev_out[n - 1]

        e2e_pipelined(args.warmup)
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        e_start.record(up)
        stream.wait_event(e_start)
        last = e2e_pipelined(args.steps)
        down.wait_event(last)
        e_end.record(down)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / args.steps, dev)
        Od2 = bufs[(args.steps - 1) % 2][3]
        assert torch.equal(Od2, O), "chunk_attend and the stage calls disagree"
        return e2e_ms, e2e_serial_ms, h2d, d2h

    e2e_ms = e2e_serial_ms = None
    h2d = d2h = 0
    if not light:
        e2e_ms, e2e_serial_ms, h2d, d2h = measure_e2e()
    clocks = sampler.stop()

    if rank != 0:
        return None
    work = stage_work(cfg, args.gqa, args.query_agg)
    peaks = load_peaks()
    # the roofline line describes the stage that takes longest: attention (tensor cores) for
    # prefill chunks, the scoring pass over the history (HBM) for decode
    dom = max(names, key=lambda nm: statistics.mean(stage_ms[nm]))
    dom_ms = statistics.mean(stage_ms[dom])
    tc_engine = q.uses_tensor_cores("attend", shape, params)
    # a stage whose flops per byte sit below the ridge point is bound by HBM (decode attention: one
    # query row per head), else by the tensor cores (prefill attention)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    att_dense = work["attend"]["flops"] / work["attend"]["bytes"] >= ridge
    if dom == "attend" and tc_engine and att_dense:
        peak, bound, unit = peaks["bf16_tflops"], "tensor", "TFLOP/s"
        achieved = work["attend"]["flops"] / (dom_ms * 1e-3) / 1e12
        peak_source = peaks["source"]
    elif dom == "attend" and att_dense:
        peak, bound, unit = FP32_FMA_PEAK_TFLOPS, "alu", "TFLOP/s"
        achieved = work["attend"]["flops"] / (dom_ms * 1e-3) / 1e12
        peak_source = "derived: 152 SM x 128 FP32 x 2 x 2.07 GHz"
    else:
        peak, bound, unit = peaks["hbm_gbs"], "hbm", "GB/s"
        achieved = work[dom]["bytes"] / (dom_ms * 1e-3) / 1e9
        peak_source = peaks["source"]
    stages = {}
    for nm in names:
        ms = statistics.mean(stage_ms[nm])
        st = {"ms": round(ms, 5)}
        if "bytes" in work[nm]:
            st["GBps"] = round(work[nm]["bytes"] / (ms * 1e-3) / 1e9, 1)
            st["hbm_frac"] = round(st["GBps"] / peaks["hbm_gbs"], 4)
        if "flops" in work[nm]:
            st["TFLOPs"] = round(work[nm]["flops"] / (ms * 1e-3) / 1e12, 2)
        stages[nm] = st
    value = job_throughput(cfg.C, world, step_ms)
    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded massive-activation recipe: biased key channels, shared query direction, "
                "5% outlier queries, planted needles)",
        "config": {"workload": cfg.name, "H_q": cfg.H_q, "H_kv": cfg.H_kv, "d": cfg.d, "C": cfg.C, "T": cfg.T,
                   "N_q": cfg.N_q, "B": cfg.B, "gqa_pool": args.gqa, "engine": args.engine,
                   **variant_keys(args),
                   "l2": f"inputs larger than L2: the timed steps rotate over {INPUT_SETS} copies of the inputs "
                         f"({INPUT_SETS * set_bytes / 2**20:.0f} MB), no flush; l2_write_flush: the same step after "
                         f"a {L2_FLUSH_BYTES >> 20} MB write",
                   "timing": "K consecutive quoka_chunk_attend calls (rotating input sets) captured as one CUDA graph, "
                             "timed with events around its replay; stages: each stage's C-ABI call "
                             f"{max(args.steps, 2 * INPUT_SETS)} times back to back on the rotating sets (the "
                             "separate quoka_topk call does not start from the scorer's histogram as the fused "
                             "step's select does)",
                   "parallelism": f"replicas x{world}"},
        "impl": "quoka",
        "gpu_launches": int(launches),
        "wall_s_timed_region": round(wall, 4),
        "roofline": {"kernel": dom, "bound": bound, "achieved": round(achieved, 2),
                     "peak": round(peak, 1), "unit": unit, "frac": round(achieved / peak, 4),
                     "peak_source": peak_source,
                     "traffic": attend_traffic(args.workload) if (dom == "attend" and tc_engine and att_dense) else None,
                     "traffic_unit": "bytes/launch"},
        "stages": stages,
        "staged_ms_per_step": round(staged_ms, 5),
        "l2_write_flush": {"ms_per_step": round(flush_step_ms, 5),
                           "value": round(job_throughput(cfg.C, world, flush_step_ms), 1)},
        "dense": None if dense_ms is None else {
            "ms_per_step": round(dense_ms, 4), "speedup": round(dense_ms / step_ms, 2),
            "TFLOPs": round(dense_flops(cfg) / (dense_ms * 1e-3) / 1e12, 2)},
        "e2e": None if e2e_ms is None else {
            "value": round(cfg.C * world / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
            "mode": "serving loop: step k's compute overlaps step k+1's upload and step k-1's download "
                    "(two device buffers, three streams; Q, K_chunk and V_chunk packed in one pinned buffer, one "
                    "upload per step); history cache rotated over the input sets",
            "serial_ms_per_step": round(e2e_serial_ms, 4),
            "serial_value": round(cfg.C * world / (e2e_serial_ms * 1e-3), 1)},
        "clocks": clocks,
    }
    if light:
        del res["e2e"]
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(cfg, x, args.gqa, groups=[0] if light else None, score_fn=args.score_fn,
                                           query_agg=args.query_agg)
    return res


def run_quoka_ragged(args, rank, world, local_rank, light=False):
    """The ragged batch: one quoka_chunk_attend_varlen call per step over every sequence's chunk."""
    from sparse_attention_chunked_gb300 import build as qbuild
    from sparse_attention_chunked_gb300 import quoka as q

    qbuild.build()
    q.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = RAGGED[args.workload]
    seqs = wl.make_ragged(cfg, args.seed)
    pk = wl.pack_varlen(seqs)
    cu_T, cu_C = pk["cu_T"], pk["cu_C"]
    names = ("Q", "K_hist", "V_hist", "K_chunk", "V_chunk")
    base = tuple(pk[k].to(dev) for k in names)
    sets = [base] + [tuple(t.clone() for t in base) for _ in range(INPUT_SETS - 1)]
    set_bytes = sum(t.numel() * t.element_size() for t in base)
    vshape = q.varlen_shape_of(len(seqs), cfg.H_q, cfg.H_kv, cfg.d, base[0].dtype)
    params = q.params_of(args.gqa, args.engine, score_fn=args.score_fn, query_agg=args.query_agg)
    T_max = max(b - a for a, b in zip(cu_T, cu_T[1:]))
    n_ws = max(q.quoka_workspace_size_varlen(vshape, cu_T, cu_C, cfg.N_q, cfg.B, params),
               q.quoka_workspace_size_varlen(vshape, cu_T, cu_C, cfg.N_q, T_max, params))
    ws = torch.zeros(n_ws, dtype=torch.uint8, device=dev)
    O = torch.empty_like(base[0])
    B_s = [min(cfg.B, b - a) for a, b in zip(cu_T, cu_T[1:])]
    sel = torch.empty(cfg.H_kv * sum(B_s), dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    new_events = lambda k: [torch.cuda.Event(enable_timing=True) for _ in range(k)]  # noqa: E731

    def call(xs, B, O_out, sel_out=None):
        q.quoka_chunk_attend_varlen(vshape, cu_T, cu_C, *xs, cfg.N_q, B, params, O_out, None, sel_out, ws, stream)

    with torch.cuda.stream(stream):
        call(base, cfg.B, O, sel)       # also leaves every sequence's kept set in sel
        call(base, cfg.B, O)
    torch.cuda.synchronize(dev)
    # K consecutive batches (rotating input sets) as one graph, and W for the warm-up
    def k_graph(k_steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(k_steps):
                call(sets[k % INPUT_SETS], cfg.B, O)
        return g
    before = q.quoka_launch_count()
    step_graph_k = k_graph(args.steps)
    launches_per_step = (q.quoka_launch_count() - before) // args.steps
    warm_graph = k_graph(args.warmup)
    # the attention stage alone over the batch (kept rows gathered once up front), for the roofline: the
    # joint tensor-core launch over every sequence (bf16), else one quoka_sparse_attend per sequence
    G = cfg.H_q // cfg.H_kv
    joint = cfg.dtype == "bf16" and args.engine != "simt" and all(G * (b - a) > 32 for a, b in zip(cu_C, cu_C[1:]))
    cu_B = [0]
    for b in B_s:
        cu_B.append(cu_B[-1] + b)
    Ksel_all = torch.empty((cfg.H_kv * cu_B[-1] * cfg.d,), dtype=base[0].dtype, device=dev)
    Vsel_all = torch.empty_like(Ksel_all)
    O_att = torch.empty_like(base[0])
    att_fns, att_flops, off = [], 0, 0
    for s, x in enumerate(seqs):
        C, T = cu_C[s + 1] - cu_C[s], cu_T[s + 1] - cu_T[s]
        sub = wl.ChunkConfig("seq", cfg.H_q, cfg.H_kv, cfg.d, C, T, cfg.N_q, cfg.B, cfg.dtype, "massive_act")
        sh = q.Shape(0, cfg.H_q, cfg.H_kv, C, T, cfg.d, 0)
        part = lambda t, h, a, b: t[h * cfg.d * a:h * cfg.d * b]  # noqa: E731
        Qs = part(base[0], cfg.H_q, cu_C[s], cu_C[s + 1]).view(cfg.H_q, C, cfg.d)
        Kh = part(base[1], cfg.H_kv, cu_T[s], cu_T[s + 1]).view(cfg.H_kv, T, cfg.d)
        Vh = part(base[2], cfg.H_kv, cu_T[s], cu_T[s + 1]).view(cfg.H_kv, T, cfg.d)
        Kc = part(base[3], cfg.H_kv, cu_C[s], cu_C[s + 1]).view(cfg.H_kv, C, cfg.d)
        Vc = part(base[4], cfg.H_kv, cu_C[s], cu_C[s + 1]).view(cfg.H_kv, C, cfg.d)
        sl = sel[cfg.H_kv * off:cfg.H_kv * (off + B_s[s])].view(cfg.H_kv, B_s[s])
        off += B_s[s]
        Ks = part(Ksel_all, cfg.H_kv, cu_B[s], cu_B[s + 1]).view(cfg.H_kv, B_s[s], cfg.d)
        Vs = part(Vsel_all, cfg.H_kv, cu_B[s], cu_B[s + 1]).view(cfg.H_kv, B_s[s], cfg.d)
        q.quoka_gather(sh, Kh, Vh, sl, B_s[s], Ks, Vs, stream)
        Os = torch.empty_like(Qs)
        att_fns.append((sh, Qs, Ks, Vs, B_s[s], Kc, Vc, Os))
        att_flops += stage_work(sub, args.gqa)["attend"]["flops"]
    torch.cuda.synchronize(dev)
    att_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(att_graph, stream=stream):
        if joint:
            q.quoka_sparse_attend_varlen(vshape, cu_B, cu_C, base[0], Ksel_all, Vsel_all, base[3], base[4], params,
                                         O_att, None, ws, stream)
        else:
            for (sh, Qs, Ks, Vs, b, Kc, Vc, Os) in att_fns:
                q.quoka_sparse_attend(sh, Qs, Ks, Vs, b, Kc, Vc, params, Os, None, ws, stream)

    sampler = ClockSampler(local_rank)
    sampler.start()
    with torch.cuda.stream(stream):
        t_w = time.perf_counter()
        done = 0
        while done < 1 or time.perf_counter() - t_w < 0.5:
            warm_graph.replay()
            att_graph.replay()
            done += 1
        warm_graph.replay()
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        e_rot = new_events(2)
        torch.cuda.nvtx.range_push("timed_steps")
        e_rot[0].record(stream)
        step_graph_k.replay()
        e_rot[1].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(dev)
        barrier()
        att = []                        # the attention stage: back-to-back replays
        n_att = max(3, args.steps // 2)
        e = new_events(2)
        e[0].record(stream)
        for _ in range(n_att):
            att_graph.replay()
        e[1].record(stream)
        att.append(e)
        torch.cuda.synchronize(dev)
        if joint:   # the attention stage alone and the whole call run the same joint launch
            assert torch.equal(O_att, O), "the joint attention stage and the ragged call disagree"
        dense = []
        Od = torch.empty_like(O)
        if not args.no_dense:
            call(base, T_max, Od)      # a budget covering every history: dense chunked attention
            for _ in range(max(3, args.steps // 4)):
                flush.zero_()
                e = new_events(2)
                e[0].record(stream)
                call(base, T_max, Od)
                e[1].record(stream)
                dense.append(e)
        torch.cuda.synchronize(dev)
    assert q.quoka_get_last_device_error(ws, stream) == 0
    step_ms = max_over_ranks(e_rot[0].elapsed_time(e_rot[1]) / args.steps, dev)
    att_ms = statistics.mean(a.elapsed_time(b) for a, b in att) / n_att
    dense_ms = statistics.mean(a.elapsed_time(b) for a, b in dense) if dense else None

    def measure_e2e():
        # end to end: the packed chunk tensors come from pinned host memory, O goes back; a serving loop
        # (step k's compute overlaps step k+1's upload and step k-1's download), as for one chunk
        # the packed Q, K_chunk and V_chunk back to back in one pinned host buffer and one device buffer
        # per slot: one upload per step, the three tensors passed as views of it
        parts = [pk[k] for k in ("Q", "K_chunk", "V_chunk")]
        sizes = [t.numel() for t in parts]
        host_in = torch.cat([t.reshape(-1) for t in parts]).pin_memory()
        dev_in = [torch.empty(sum(sizes), dtype=base[0].dtype, device=dev) for _ in range(2)]

        def views(buf):
            a, b = sizes[0], sizes[0] + sizes[1]
            return [buf[:a].view(base[0].shape), buf[a:b].view(base[3].shape), buf[b:].view(base[4].shape)]

        bufs = [views(dev_in[i]) + [torch.empty_like(O)] for i in range(2)]
        Ohs = [torch.empty(O.shape, dtype=O.dtype).pin_memory() for _ in range(2)]
        h2d = host_in.numel() * host_in.element_size()
        d2h = Ohs[0].numel() * Ohs[0].element_size()
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_pipelined(n):
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_done = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            for k in range(n):
                b = k % 2
                Qd, Kcd, Vcd, Od = bufs[b]
                with torch.cuda.stream(up):
                    if k >= 2:
                        up.wait_event(ev_done[k - 2])
                    dev_in[b].copy_(host_in, non_blocking=True)
                    ev_in[k].record(up)
                stream.wait_event(ev_in[k])
                if k >= 2:
                    stream.wait_event(ev_out[k - 2])
                xs = sets[k % INPUT_SETS]
                call((Qd, xs[1], xs[2], Kcd, Vcd), cfg.B, Od)
                ev_done[k].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(ev_done[k])
                    Ohs[b].copy_(Od, non_blocking=True)
                    ev_out[k].record(down)
            return ev_out[n - 1]

        e2e_pipelined(args.warmup)
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        e_start.record(up)
        stream.wait_event(e_start)
        last = e2e_pipelined(args.steps)
        down.wait_event(last)
        e_end.record(down)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / args.steps, dev)
        O2 = bufs[(args.steps - 1) % 2][3]
        assert torch.equal(O2, O), "the end-to-end call and the timed steps disagree"
        return e2e_ms, h2d, d2h

    e2e_ms, h2d, d2h = (None, 0, 0) if light else measure_e2e()
    clocks = sampler.stop()
    if rank != 0:
        return None
    peaks = load_peaks()
    tokens = cu_C[-1]
    achieved = att_flops / (att_ms * 1e-3) / 1e12
    res = {
        "metric": METRIC,
        "value": round(job_throughput(tokens, world, step_ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded massive-activation recipe per sequence, log-uniform history lengths)",
        "config": {"workload": cfg.name, "nseq": len(seqs), "H_q": cfg.H_q, "H_kv": cfg.H_kv, "d": cfg.d,
                   "C": cfg.C, "T_per_seq": [b - a for a, b in zip(cu_T, cu_T[1:])], "N_q": cfg.N_q, "B": cfg.B,
                   "gqa_pool": args.gqa, "engine": args.engine, **variant_keys(args),
                   "l2": f"inputs larger than L2: the timed steps rotate over {INPUT_SETS} copies of the packed "
                         f"inputs ({INPUT_SETS * set_bytes / 2**20:.0f} MB), no flush",
                   "timing": "K consecutive quoka_chunk_attend_varlen calls (rotating input sets) captured as one "
                             "CUDA graph, timed with events around its replay",
                   "parallelism": f"replicas x{world}"},
        "impl": "quoka",
        "gpu_launches": int(launches_per_step * args.steps),
        "roofline": {"kernel": "attend (all sequences, one joint launch)" if joint else "attend (per sequence)",
                     "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": round(peaks["bf16_tflops"], 1), "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4), "peak_source": peaks["source"],
                     "traffic": attend_traffic(args.workload) if joint else None, "traffic_unit": "bytes/launch"},
        "attend_ms_per_batch": round(att_ms, 5),
        "dense": None if dense_ms is None else {"ms_per_step": round(dense_ms, 4),
                                                "speedup": round(dense_ms / step_ms, 2)},
        "e2e": None if e2e_ms is None else {
            "value": round(tokens * world / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
            "mode": "serving loop: step k's compute overlaps step k+1's upload and step k-1's download "
                    "(two device buffers, three streams; the packed Q, K_chunk and V_chunk in one pinned buffer, "
                    "one upload per step); histories rotated over the input sets"},
        "clocks": clocks,
    }
    if light:
        del res["e2e"]
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_ragged(cfg, seqs, args.gqa)
    return res


def run_sweep(args, rank, world, local_rank):
    """The chunked-prefill sweep: one prompt of 65536 tokens in 32 chunks of 2048, each chunk scored,
    selected and attended against the cache of every earlier chunk, then appended to it (with its key
    norms, which the next chunks' scoring reads).  A step is the whole prompt; per-chunk times are
    reported too.  The cache is preallocated for the whole prompt and filled in place."""
    from sparse_attention_chunked_gb300 import build as qbuild
    from sparse_attention_chunked_gb300 import quoka as q

    qbuild.build()
    q.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = wl.SWEEP_64K_BF16
    sw = wl.make_sweep(cfg, args.seed)
    K_all, V_all = sw.K_all.to(dev), sw.V_all.to(dev)
    Kcache, Vcache = torch.zeros_like(K_all), torch.zeros_like(V_all)
    inv = torch.zeros((cfg.H_kv, cfg.total), dtype=torch.float32, device=dev)   # key-norm cache
    Qs = [t.to(dev) for t in sw.Q]
    Kcs = [K_all[:, i * cfg.C:(i + 1) * cfg.C].contiguous() for i in range(cfg.n_chunks)]
    Vcs = [V_all[:, i * cfg.C:(i + 1) * cfg.C].contiguous() for i in range(cfg.n_chunks)]
    params = q.params_of(args.gqa, args.engine)
    ws = q.make_workspace(q.shape_of(Qs[0], Kcache, T=cfg.total - cfg.C), cfg.N_q, cfg.total, params, device=dev)
    O = torch.empty_like(Qs[0])
    stream = torch.cuda.Stream(dev)

    def chunk_fn(i, B):
        shape = q.shape_of(Qs[i], Kcache, T=i * cfg.C)
        q.quoka_chunk_attend_cached(shape, Qs[i], Kcache, Vcache, Kcs[i], Vcs[i], inv, cfg.N_q, B, params, O, None,
                                    None, ws, stream)
        q.quoka_append_kv_norms(shape, Kcache, Vcache, Kcs[i], Vcs[i], inv, stream)

    def graphs_for(B):
        gs, launches = [], 0
        with torch.cuda.stream(stream):
            for i in range(cfg.n_chunks):
                chunk_fn(i, B)
        torch.cuda.synchronize(dev)
        for i in range(cfg.n_chunks):
            g = torch.cuda.CUDAGraph()
            before = q.quoka_launch_count()
            with torch.cuda.graph(g, stream=stream):
                chunk_fn(i, B)
            launches += q.quoka_launch_count() - before
            gs.append(g)
        return gs, launches

    def time_sweep(gs, reps):
        per = [[] for _ in gs]
        tot = []
        with torch.cuda.stream(stream):
            for _ in range(reps):
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(gs) + 1)]
                evs[0].record(stream)
                for i, g in enumerate(gs):
                    g.replay()
                    evs[i + 1].record(stream)
                torch.cuda.synchronize(dev)
                for i in range(len(gs)):
                    per[i].append(evs[i].elapsed_time(evs[i + 1]))
                tot.append(evs[0].elapsed_time(evs[-1]))
        return [statistics.mean(p) for p in per], statistics.mean(tot)

    gs, launches = graphs_for(cfg.B)
    whole = torch.cuda.CUDAGraph()        # the whole prompt as one graph: the total time
    with torch.cuda.graph(whole, stream=stream):
        for i in range(cfg.n_chunks):
            chunk_fn(i, cfg.B)
    sampler = ClockSampler(local_rank)
    sampler.start()
    with torch.cuda.stream(stream):
        t_w = time.perf_counter()
        while time.perf_counter() - t_w < 0.3:
            for g in gs:
                g.replay()
        torch.cuda.synchronize(dev)
    barrier()
    reps = max(3, args.steps // 4)
    per_ms, _ = time_sweep(gs, reps)
    with torch.cuda.stream(stream):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record(stream)
        for _ in range(reps):
            whole.replay()
        e[1].record(stream)
        torch.cuda.synchronize(dev)
    total_ms = max_over_ranks(e[0].elapsed_time(e[1]) / reps, dev)
    clocks = sampler.stop()
    assert torch.equal(Kcache, K_all) and torch.equal(Vcache, V_all), "the sweep did not rebuild the cache"
    assert q.quoka_get_last_device_error(ws, stream) == 0
    dense_total = None
    if not args.no_dense:   # a budget covering every history: dense chunked prefill of the same prompt
        dgs, _ = graphs_for(cfg.total)
        _, dense_total = time_sweep(dgs, max(2, reps // 2))
    if rank != 0:
        return None
    res = {"workload": cfg.name, "gqa_pool": args.gqa, "n_chunks": cfg.n_chunks, "C": cfg.C, "N_q": cfg.N_q,
           "B": cfg.B, "total_tokens": cfg.total,
           "value": round(cfg.total * world / (total_ms * 1e-3), 1), "unit": "tokens/s",
           "ms_total": round(total_ms, 4),
           "ms_per_chunk": [round(x, 4) for x in per_ms],
           "timing": f"total: the 32 chunks (quoka_chunk_attend_cached + quoka_append_kv_norms each) as one CUDA "
                     f"graph, mean of {reps} replays; per chunk: one graph per chunk, replayed in order with events "
                     f"between them; the cache grows to {2 * K_all.numel() * 2 >> 20} MB, so later chunks read "
                     f"their history from HBM",
           "gpu_launches_per_sweep": int(launches),
           "dense": None if dense_total is None else {"ms_total": round(dense_total, 4),
                                                      "speedup": round(dense_total / total_ms, 2)},
           "clocks": clocks}
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_sweep(cfg, sw, args.gqa)
    return res


# ---------------------------------------------------------------- the CPU oracle

def _blas_threads():
    """Threads of the BLAS numpy uses (OpenBLAS query when it is the loaded library), else the CPU count."""
    try:
        import ctypes
        with open("/proc/self/maps") as f:
            libs = {line.split()[-1] for line in f if "openblas" in line.lower() and line.strip().endswith(".so")
                    or "openblas" in line.lower()}
        for path in libs:
            if os.path.exists(path):
                lib = ctypes.CDLL(path)
                for sym in ("openblas_get_num_threads64_", "openblas_get_num_threads", "scipy_openblas_get_num_threads64_"):
                    if hasattr(lib, sym):
                        return int(getattr(lib, sym)())
    except Exception:
        pass
    return os.cpu_count()


def _oracle_inputs(x, g, G):
    f = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    return (f(x.Q[g * G:(g + 1) * G]), f(x.K_hist[g:g + 1]), f(x.V_hist[g:g + 1]), f(x.K_chunk[g:g + 1]),
            f(x.V_chunk[g:g + 1]))


def variant_keys(args) -> dict:
    """The key-score ablation and the key-norm cache, named in the config only when in force."""
    out = {}
    if getattr(args, "key_norm_cache", False):
        out["key_norm_cache"] = True
    if args.score_fn != "cos":
        out["score_fn"] = args.score_fn
    if args.query_agg != "max":
        out["query_agg"] = args.query_agg
    return out


def cpu_baseline(cfg, x, gqa, groups=None, score_fn="cos", query_agg="max"):
    """The oracle as it stands on this host's cores, on KV groups of the same chunk (each group is an
    independent 1/H_kv share of the chunk's work); reported as the equivalent chunk tokens/s."""
    from oracle import quoka_oracle as qo
    groups = list(range(cfg.H_kv)) if groups is None else groups
    t = 0.0
    for g in groups:
        args = _oracle_inputs(x, g, cfg.G)
        t0 = time.perf_counter()
        qo.chunk_attend(*args, cfg.N_q, cfg.B, gqa, score_fn=score_fn, query_agg=query_agg)
        t += time.perf_counter() - t0
    per_chunk = t * cfg.H_kv / len(groups)
    return {"value": round(cfg.C / per_chunk, 2), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"numpy float64 oracle, {len(groups)} of {cfg.H_kv} KV groups of one chunk "
                      f"({cfg.G} query heads each), {t:.1f} s measured, scaled to a whole chunk"}


def cpu_baseline_ragged(cfg, seqs, gqa):
    """The oracle on one KV group of every sequence, scaled by H_kv to the whole batch."""
    from oracle import quoka_oracle as qo
    t = 0.0
    for x in seqs:
        args = _oracle_inputs(x, 0, cfg.G)
        t0 = time.perf_counter()
        qo.chunk_attend(*args, cfg.N_q, cfg.B, gqa)
        t += time.perf_counter() - t0
    tokens = sum(x.Q.shape[1] for x in seqs)
    return {"value": round(tokens / (t * cfg.H_kv), 2), "unit": "tokens/s", "cores": _blas_threads(),
            "kind": "oracle", "sample": f"numpy float64 oracle, KV group 0 of each of the {len(seqs)} sequences "
                                        f"({cfg.G} query heads each), {t:.1f} s measured, scaled x{cfg.H_kv}"}


def cpu_baseline_sweep(cfg, sw, gqa, sample=(4, 12, 20, 28)):
    """The oracle on KV group 0 of a few chunks of the sweep, spread over the prompt; the mean chunk
    time, scaled by the chunk count and H_kv, stands for the whole sweep."""
    from oracle import quoka_oracle as qo
    G = cfg.H_q // cfg.H_kv
    f = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    t = 0.0
    for i in sample:
        T = i * cfg.C
        args = (f(sw.Q[i][:G]), f(sw.K_all[:1, :T]), f(sw.V_all[:1, :T]), f(sw.K_all[:1, T:T + cfg.C]),
                f(sw.V_all[:1, T:T + cfg.C]))
        t0 = time.perf_counter()
        qo.chunk_attend(*args, cfg.N_q, cfg.B, gqa)
        t += time.perf_counter() - t0
    per_sweep = t / len(sample) * cfg.n_chunks * cfg.H_kv
    return {"value": round(cfg.total / per_sweep, 2), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"numpy float64 oracle, KV group 0 of chunks {list(sample)} ({G} query heads each), "
                      f"{t:.1f} s measured, mean chunk x {cfg.n_chunks} chunks x {cfg.H_kv} groups"}


def run_reference_ragged(args, rank, world):
    """The oracle on the ragged batch: each step is KV group (step mod H_kv) of every sequence, x H_kv."""
    if rank != 0:
        return None
    cfg = RAGGED[args.workload]
    seqs = wl.make_ragged(cfg, args.seed)
    from oracle import quoka_oracle as qo
    times = []
    for k in range(args.warmup + args.steps):
        g = k % cfg.H_kv
        t0 = time.perf_counter()
        for x in seqs:
            qo.chunk_attend(*_oracle_inputs(x, g, cfg.G), cfg.N_q, cfg.B, args.gqa)
        if k >= args.warmup:
            times.append(time.perf_counter() - t0)
    per_batch = statistics.mean(times) * cfg.H_kv
    tokens = sum(x.Q.shape[1] for x in seqs)
    value = round(tokens / per_batch, 2)
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(per_batch * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "nseq": len(seqs), "H_q": cfg.H_q, "H_kv": cfg.H_kv, "d": cfg.d,
                   "C": cfg.C, "N_q": cfg.N_q, "B": cfg.B, "gqa_pool": args.gqa, "parallelism": "host cores"},
        "impl": "reference",
        "gpu_launches": 0,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
                         "sample": f"each step: one of {cfg.H_kv} KV groups of every sequence through the numpy "
                                   f"float64 oracle, scaled x{cfg.H_kv} to the whole batch"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args, rank, world):
    if args.workload in RAGGED:
        return run_reference_ragged(args, rank, world)
    if rank != 0:
        return None
    cfg = WORKLOADS[args.workload]
    x = wl.make_chunk(cfg, args.seed)
    from oracle import quoka_oracle as qo
    inputs = [_oracle_inputs(x, g, cfg.G) for g in range(cfg.H_kv)]
    times = []
    for k in range(args.warmup + args.steps):   # a step: the whole chunk, every KV group
        t0 = time.perf_counter()
        for a in inputs:
            qo.chunk_attend(*a, cfg.N_q, cfg.B, args.gqa, score_fn=args.score_fn, query_agg=args.query_agg)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            times.append(dt)
    per_chunk = statistics.mean(times)
    value = round(cfg.C / per_chunk, 2)
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(per_chunk * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "H_q": cfg.H_q, "H_kv": cfg.H_kv, "d": cfg.d, "C": cfg.C, "T": cfg.T,
                   "N_q": cfg.N_q, "B": cfg.B, "gqa_pool": args.gqa, **variant_keys(args),
                   "parallelism": "host cores"},
        "impl": "reference",
        "gpu_launches": 0,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
                         "sample": f"each step: the whole chunk (all {cfg.H_kv} KV groups) through the numpy "
                                   f"float64 oracle on this host's cores (BLAS threads: {_blas_threads()})"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# The other configurations, measured after the headline in the same run (each a sub-record of the
# headline JSON line with its own step time, stages, roofline, dense reference and CPU sample).
SUITE = (("gqa32k", "mean"), ("gqa128k", "max"), ("gqa128k", "mean"), ("sweep64k", "max"), ("ragged8", "max"),
         ("decode32k", "max"))


def run_suite(args, rank, world, local_rank):
    import copy
    out = {}
    for workload, gqa in SUITE:
        sub = copy.copy(args)
        sub.workload, sub.gqa = workload, gqa
        sub.steps = max(10, args.steps // 2)
        if workload == "decode32k":   # a ~45 us step: more steps for a stable mean at no real cost
            sub.steps = max(100, args.steps)
        if workload == "sweep64k":
            r = run_sweep(sub, rank, world, local_rank)
        elif workload in RAGGED:
            r = run_quoka_ragged(sub, rank, world, local_rank, light=True)
        else:
            r = run_quoka(sub, rank, world, local_rank, light=True)
        torch.cuda.empty_cache()
        if r is not None:
            for k in ("metric", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "data", "impl"):
                r.pop(k, None)
            out[f"{workload}_{gqa}"] = r
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["quoka", "reference"], default="quoka")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(RAGGED) + ["sweep64k"], default="gqa32k")
    ap.add_argument("--gqa", choices=["max", "mean"], default="max")
    ap.add_argument("--engine", choices=["auto", "simt", "tensor"], default="auto")
    ap.add_argument("--score-fn", choices=["cos", "dot"], default="cos",
                    help="key score: cosine (the method) or the dot-product ablation")
    ap.add_argument("--query-agg", choices=["max", "mean"], default="max",
                    help="aggregation over the selected queries: max (the method) or the mean ablation")
    ap.add_argument("--key-norm-cache", action="store_true",
                    help="score with the history's key norms from the cache written at append time")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-suite", action="store_true",
                    help="only the headline line: skip the sub-records of the other configurations")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)     # rank 0 alone; other ranks exit without work
    else:
        dist_init("nccl")
        if args.workload == "sweep64k":
            res = run_sweep(args, rank, world, local_rank)
        else:
            run = run_quoka_ragged if args.workload in RAGGED else run_quoka
            res = run(args, rank, world, local_rank)
            if not args.no_suite and args.workload == "gqa32k" and args.gqa == "max" and not variant_keys(args):
                suite = run_suite(args, rank, world, local_rank)
                if res is not None:
                    res["suite"] = suite
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
