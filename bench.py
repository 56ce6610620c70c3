#!/usr/bin/env python
"""Benchmark of one DSA decode step (indexer scan -> top-2048 -> sparse MLA).

Metric: algorithmic HBM bytes moved per second (GB/s) by dsa_decode_step,
whole job, inputs resident in HBM; also µs per layer-step and the fraction of
the HBM roofline.  Algorithmic bytes = 132 B per context token of every
request (index keys, read once for all its rows) + 576 B per selected latent
row + queries + bf16 output.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl reference]

N > 1 runs under torchrun, one rank per GPU, each rank stepping its own
replica of the workload (independent requests: weak scaling, no data-path
collective).  Rank 0 prints ONE JSON line.  `--impl reference` times the
float64 CPU oracle instead (the only reference this method has), on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dsa_sparse_attention_lightning_gb300 import inputs, traffic  # noqa: E402

METRIC = "DSA decode-step µs/layer and achieved HBM GB/s vs 8 TB/s roofline, 1 GB300"
L2_FLUSH_BYTES = 256 << 20
CLOCK_WINDOW_S = 1.0
# Decode workloads reported beside the headline one: 32K (16 x 4 rows) and 1M
# (one row) beside the 256K headline.
SIDE_CONFIGS = {2: (1, 3), 1: (2, 3), 3: (1, 2)}
# Kernels one step launches: scan 2 (query split + grouping, scan); top-k 1
# (one CTA per row, rows of at most 49,152 scores) or 3 (sample, collect,
# finalize); sparse MLA 3 (query split, attention, combine of cut units).
TOPK_ROW_CAP = 49152


def kernels_per_step(wl) -> int:
    return 2 + (1 if wl.max_pages * inputs.PAGE <= TOPK_ROW_CAP else 3) + 3

# DRAM bytes (read + write) per call of a stage, summed over its kernels, from
# one ncu capture of the current kernels (cold cache, so L2-resident
# intermediates count as DRAM reads).  Stages and workloads not captured on the
# current kernels report null.
NCU_STAGE_TRAFFIC = {
    # the scan kernel on the first 4 of the 16 requests (same per-request shape),
    # its read + write bytes scaled by 4: its traffic grows with the tiles it reads
    ("decode_16x4_ctx262144_h64", "indexer_scan"): 4 * (138.67e6 + 5.33e6),
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# Dense FP8 (E4M3) tensor rate = the bf16 rate x the nominal FP8 / bf16 ratio
# (4.5 / 2.25 PFLOP/s): both contractions of the step run kind::f8f6f4.
FP8_PER_BF16 = 2.0


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"dsa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------- GPU arm
def _step_fn(dsa, inp, wl, ws, out, lse):
    def step():
        dsa.dsa_decode_step(inp["q_idx"], inp["w"], inp["key_cache"], inp["latent_cache"],
                            inp["latent_scale"], inp["block_table"], inp["row_req"],
                            inp["row_len"], inp["q"], softmax_scale=inp["softmax_scale"],
                            k=wl.k, q_scale=inp["q_idx_scale"], out=out, lse=lse, workspace=ws)
    return step


def _graph(fn, stream):
    """Capture fn (a sequence of library launches on `stream`) into a CUDA graph."""
    fn()                                   # warm: one-time kernel attributes are set eagerly
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def _time_launches(fn, n, flush, stream):
    """Mean device time (ms) of fn over n launches, L2 flushed (untimed) before each.

    Each launch is bracketed by its own pair of CUDA events on `stream`; the
    host synchronises once at the end."""
    evs = []
    for _ in range(n):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    evs[-1][1].synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    return statistics.mean(times), times


def rank_workload(config: int, rank: int, requests: int = 0) -> inputs.Workload:
    """Rank r steps its own replica: same shape, its own seed (independent requests).
    requests > 0 keeps only the first `requests` requests (a smaller device
    footprint with the same per-request shape, for profiler captures)."""
    wl = inputs.config(config)
    wl.seed = wl.seed + 1000 * rank
    if 0 < requests < wl.B:
        wl.ctx, wl.rows = wl.ctx[:requests], wl.rows[:requests]
        wl.name = f"{wl.name}_first{requests}requests"
    return wl


def reduce_max_ms(total_ms: float, device) -> float:
    """Max over ranks of the timed region (a control-path reduction, not data)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(total_ms)
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, world: int, steps: int, max_total_ms: float) -> float:
    """Units all ranks processed divided by the slowest rank's time."""
    return bytes_per_step * world * steps / (max_total_ms * 1e-3) / 1e9


def _step_buffers(dsa, wl, dev):
    inp = inputs.make_inputs(wl, device=dev)
    out = torch.empty((wl.R, wl.H, inputs.V_DIM), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.R, wl.H), dtype=torch.float32, device=dev)
    ws = torch.empty(dsa.decode_step_workspace_size(wl.B, wl.R, wl.max_pages, wl.H, wl.k),
                     dtype=torch.uint8, device=dev)
    return inp, out, lse, ws


def _stage_fns(dsa, wl, inp, out, lse, dev):
    """The step's three C-ABI calls, each on its own buffers, with the algorithmic
    bytes of each (None for the selection, which moves no algorithmic bytes)."""
    R, H = wl.R, wl.H
    scores = torch.empty((R, wl.max_pages * inputs.PAGE), dtype=torch.float32, device=dev)
    idx = torch.empty((R, wl.k), dtype=torch.int32, device=dev)
    ws_s = torch.empty(dsa.indexer_score_workspace_size(R), dtype=torch.uint8, device=dev)
    ws_t = torch.empty(dsa.topk_workspace_size(R, scores.shape[1], wl.k), dtype=torch.uint8,
                       device=dev)
    ws_m = torch.empty(dsa.sparse_mla_workspace_size(R, H, wl.k), dtype=torch.uint8, device=dev)
    stages = {
        "indexer_scan": (lambda: dsa.dsa_indexer_score(
            inp["q_idx"], inp["w"], inp["key_cache"], inp["block_table"], inp["row_req"],
            inp["row_len"], q_scale=inp["q_idx_scale"], scores=scores, workspace=ws_s),
            traffic.scan_bytes(wl) + R * inputs.IDX_HEADS * (inputs.IDX_DIM * 2 + 4)),
        "topk": (lambda: dsa.dsa_topk(scores, inp["row_len"], wl.k, idx=idx, workspace=ws_t),
                 None),
        "sparse_mla": (lambda: dsa.dsa_sparse_mla_decode(
            inp["q"], inp["latent_cache"], inp["latent_scale"], inp["block_table"],
            inp["row_req"], inp["row_len"], idx, softmax_scale=inp["softmax_scale"], out=out,
            lse=lse, workspace=ws_m),
            traffic.gather_bytes(wl) + R * H * (inputs.LAT_DIM + inputs.V_DIM) * 2),
    }
    return stages, scores, idx, ws_s


def _time_stages(stages, n, flush, stream):
    """Each stage graph-replayed alone, L2 flushed before every replay."""
    stage_ms = {}
    for name, (fn, _) in stages.items():
        g = _graph(fn, stream)
        for _ in range(3):
            g.replay()
        stage_ms[name] = _time_launches(g.replay, n, flush, stream)[0]
    return stage_ms


def _side_workload(dsa, config, rank, dev, stream, flush, steps, hbm_peak):
    """Step and stage times of another decode workload (reported beside the headline)."""
    wl = rank_workload(config, rank)
    inp, out, lse, ws = _step_buffers(dsa, wl, dev)
    g = _graph(_step_fn(dsa, inp, wl, ws, out, lse), stream)
    for _ in range(3):
        flush()
        g.replay()
    ms = _time_launches(g.replay, steps, flush, stream)[0]
    if dsa.check_device_status(ws) != 0:
        raise RuntimeError(f"device status raised on {wl.name}")
    stages, *_ = _stage_fns(dsa, wl, inp, out, lse, dev)
    stage_ms = _time_stages(stages, steps, flush, stream)
    b = traffic.algorithmic_bytes(wl)
    gbs = b / (ms * 1e-3) / 1e9
    res = {"us_per_step": round(ms * 1e3, 2), "gbs": round(gbs, 1),
           "frac_of_8TBs": round(gbs / 8000.0, 4), "frac_of_measured": round(gbs / hbm_peak, 4),
           "tokens_per_s": round(wl.R / (ms * 1e-3), 1), "algorithmic_bytes": b,
           "stage_us": {k: round(v * 1e3, 2) for k, v in stage_ms.items()}, "steps": steps}
    del inp, out, lse, ws, g, stages
    torch.cuda.empty_cache()
    return wl.name, res


def _packed(tensors, device, pin):
    """One buffer holding every tensor (256-byte aligned slots) and a view of each."""
    offs, o = {}, 0
    for k, t in tensors.items():
        offs[k] = o
        o += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(o, 256), dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = {}
    for k, t in tensors.items():
        n = t.numel() * t.element_size()
        views[k] = buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    return buf, views


def run_gpu(args):
    rank, world, local = _dist()
    import dsa_sparse_attention_lightning_gb300 as dsa
    dsa.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    wl = rank_workload(args.config, rank, args.requests)
    inp, out, lse, ws = _step_buffers(dsa, wl, dev)
    R, H = wl.R, wl.H
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # everything below runs on its own stream: the inputs' generation on the
    # default stream (and the temporaries it freed, whose memory the buffers
    # above may reuse) must be finished before that stream touches them
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    step_eager = _step_fn(dsa, inp, wl, ws, out, lse)
    step_graph = _graph(step_eager, stream)
    step = step_graph.replay

    def flush():
        flush_buf.fill_(1)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if dsa.check_device_status(ws) != 0:
        raise RuntimeError("device status raised during warm-up")

    # ---- timed region: K steps, L2 flushed (untimed) before each; the clock
    # sampler keeps running over at least a second of back-to-back replays of
    # the same step right after it (the timed region alone is shorter than the
    # sampling interval)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        step_ms, _ = _time_launches(step, args.steps, flush, stream)
        torch.cuda.synchronize()
        t_end = time.perf_counter() + CLOCK_WINDOW_S
        window_steps = 0
        while time.perf_counter() < t_end:
            for _ in range(256):
                flush()
                step()
            window_steps += 256
            torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clock_info = clocks.summary()
    clock_info["window"] = (f"timed region plus {window_steps} more replays of the same step "
                            f"(>= {CLOCK_WINDOW_S:g} s)")
    total_ms = reduce_max_ms(step_ms * args.steps, dev)
    bytes_step = traffic.algorithmic_bytes(wl)
    value = whole_job_gbs(bytes_step, world, args.steps, total_ms)
    ms_per_step = total_ms / args.steps

    # ---- per-kernel timing of the step's stages (same inputs, same launches) --
    n_stage = max(20, min(args.steps, 200))
    stages, scores, idx, ws_s = _stage_fns(dsa, wl, inp, out, lse, dev)
    stage_ms = _time_stages(stages, n_stage, flush, stream)
    eager_ms = _time_launches(step_eager, n_stage, flush, stream)[0]

    # ---- the same selection by the decode-context-parallel exchange (8 token
    # shards emulated on this GPU), on the step's scores
    DCP_W = 8
    dcp_idx = torch.empty((R, wl.k), dtype=torch.int32, device=dev)
    dcp_res = torch.empty((R,), dtype=torch.int32, device=dev)
    ws_d = torch.empty(dsa.topk_dcp_workspace_size(R, scores.shape[1], wl.k, DCP_W),
                       dtype=torch.uint8, device=dev)
    dcp_fn = lambda: dsa.dsa_topk_dcp(scores, inp["row_len"], wl.k, DCP_W, idx=dcp_idx,  # noqa: E731
                                      resend=dcp_res, workspace=ws_d)
    g = _graph(dcp_fn, stream)
    for _ in range(3):
        g.replay()
    dcp_ms = _time_launches(g.replay, n_stage, flush, stream)[0]
    torch.cuda.synchronize()
    dcp = {"shards": DCP_W, "us": round(dcp_ms * 1e3, 2), "topk_us": round(stage_ms["topk"] * 1e3, 2),
           "rows_with_resend": int((dcp_res != 0).sum().item()),
           "equals_topk": bool(torch.equal(dcp_idx, idx))}
    del ws_d, dcp_idx, g
    # What one of the W GPUs would run (communication aside): the local top-k
    # and top-c of its own shard (every W-th token of each row), then the top-k
    # of the W x c gathered candidates.  Timed with the library's top-k on a
    # shard of the step's scores and on W x c of a row's scores as stand-ins.
    c_dcp = min(2048, -(-3 * wl.k // (2 * DCP_W)))
    shard = scores[:, 0::DCP_W].contiguous()
    shard_len = ((inp["row_len"] + DCP_W - 1) // DCP_W).to(torch.int32)
    cand = scores[:, :DCP_W * c_dcp].contiguous()
    cand_len = torch.minimum(inp["row_len"], torch.full_like(inp["row_len"], DCP_W * c_dcp))
    torch.cuda.synchronize()
    rank_fns = {
        "local_topk": lambda: dsa.dsa_topk(shard, shard_len, wl.k),
        "local_topc": lambda: dsa.dsa_topk(shard, shard_len, c_dcp),
        "merge_topk": lambda: dsa.dsa_topk(cand, cand_len, wl.k),
    }
    rank_us = {}
    for name, fn in rank_fns.items():
        g = _graph(fn, stream)
        for _ in range(3):
            g.replay()
        rank_us[name] = round(_time_launches(g.replay, n_stage, flush, stream)[0] * 1e3, 2)
        del g
    dcp["per_rank_us"] = {**rank_us, "sum": round(sum(rank_us.values()), 2),
                          "candidates_per_shard": c_dcp}
    del shard, cand
    dominant = max((n for n in stages if stages[n][1] is not None), key=lambda n: stage_ms[n])
    hbm_peak, bf16_peak, peak_kind = _peaks()
    fp8_peak = bf16_peak * FP8_PER_BF16
    # algorithmic FLOPs of the two contractions (indexer scan, attention) per stage time
    tflops = {"indexer_scan": traffic.scan_flops(wl) / (stage_ms["indexer_scan"] * 1e-3) / 1e12,
              "sparse_mla": traffic.mla_flops(wl) / (stage_ms["sparse_mla"] * 1e-3) / 1e12}
    tensor = {"unit": "TFLOP/s", "peak": round(fp8_peak, 1),
              "peak_kind": f"{peak_kind} bf16 x {FP8_PER_BF16:g} (nominal FP8/bf16)",
              "indexer_scan": round(tflops["indexer_scan"], 2),
              "sparse_mla": round(tflops["sparse_mla"], 2),
              "indexer_scan_frac": round(tflops["indexer_scan"] / fp8_peak, 4),
              "sparse_mla_frac": round(tflops["sparse_mla"] / fp8_peak, 4)}
    common = {"traffic": NCU_STAGE_TRAFFIC.get((wl.name, dominant)),
              "stage_us": {k: round(v * 1e3, 2) for k, v in stage_ms.items()},
              "step_frac_of_8TBs": round(bytes_step / (ms_per_step * 1e-3) / 8e12, 4),
              "step_frac_of_measured": round(bytes_step / (ms_per_step * 1e-3) / 1e9 / hbm_peak,
                                             4)}
    if wl.q_idx_fp8:
        # prefill chunk: the indexer is a dense FP8 GEMM, bound by the tensor cores
        dominant = "indexer_scan"
        achieved = tflops[dominant]
        roofline = {"kernel": dominant, "bound": "tensor", "achieved": round(achieved, 2),
                    "peak": round(fp8_peak, 1), "peak_kind": tensor["peak_kind"],
                    "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4), **common}
        roofline["traffic"] = NCU_STAGE_TRAFFIC.get((wl.name, dominant))
    else:
        dom_bytes = stages[dominant][1]
        achieved = dom_bytes / (stage_ms[dominant] * 1e-3) / 1e9
        roofline = {"kernel": dominant, "bound": "hbm", "achieved": round(achieved, 1),
                    "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s",
                    "frac": round(achieved / hbm_peak, 4), **common}

    # ---- end to end through the public API with host buffers: the step's
    # per-step inputs are packed in one pinned host buffer, copied with one
    # host-to-device copy into one device buffer that the call's tensors view;
    # out and lse come back the same way
    per_step = {k: inp[k] for k in ("q_idx", "q_idx_scale", "w", "q", "block_table", "row_req",
                                    "row_len") if inp.get(k) is not None}
    dev_buf, dev_in = _packed(per_step, dev, pin=False)
    host_buf, host_in = _packed(per_step, "cpu", pin=True)
    for k2, t in per_step.items():
        host_in[k2].copy_(t.cpu())
    outs = {"out": out, "lse": lse}
    dev_obuf, dev_out = _packed(outs, dev, pin=False)
    host_obuf, _ = _packed(outs, "cpu", pin=True)
    e2e_inp = dict(inp)
    e2e_inp.update(dev_in)
    e2e_call = _step_fn(dsa, e2e_inp, wl, ws, dev_out["out"], dev_out["lse"])
    h2d = host_buf.numel()
    d2h = host_obuf.numel()

    def e2e_step():
        dev_buf.copy_(host_buf, non_blocking=True)
        e2e_call()
        host_obuf.copy_(dev_obuf, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_serial_ms = _time_launches(e2e_step, n_stage, flush, stream)[0]
    if not torch.equal(host_obuf[:out.numel() * 2].view(torch.bfloat16).view(out.shape).to(dev),
                       out):
        raise RuntimeError("end-to-end output differs from the device-resident step")

    # The same calls as a serving loop runs them: step i + 1's inputs are copied
    # in, and step i's output copied out, on a copy stream while step i
    # computes (two device input and output buffers).  Every step still copies
    # its inputs in and its output out inside the timed region; the caches
    # (larger than L2) are not flushed between steps here.
    bufs = []
    for _ in range(2):
        d_in, v_in = _packed(per_step, dev, pin=False)
        d_out, v_out = _packed(outs, dev, pin=False)
        h_out, _ = _packed(outs, "cpu", pin=True)
        e_inp = dict(inp)
        e_inp.update(v_in)
        bufs.append((d_in, d_out, h_out,
                     _step_fn(dsa, e_inp, wl, ws, v_out["out"], v_out["lse"])))
    copy_stream = torch.cuda.Stream(dev)
    n_pipe = max(20, min(args.steps, 200))

    def e2e_pipelined(n):
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        copy_stream.wait_stream(stream)
        for b in range(2):                          # the first two steps' inputs
            with torch.cuda.stream(copy_stream):
                bufs[b][0].copy_(host_buf, non_blocking=True)
                h2d_done[b].record(copy_stream)
        for i in range(n):
            b = i % 2
            d_in, d_out, h_out, call = bufs[b]
            stream.wait_event(h2d_done[b])
            call()
            comp_done[b].record(stream)
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(comp_done[b])
                h_out.copy_(d_out, non_blocking=True)
                if i + 2 < n:                       # step i + 2's inputs into this buffer
                    d_in.copy_(host_buf, non_blocking=True)
                    h2d_done[b].record(copy_stream)
        stream.wait_stream(copy_stream)
        t1.record(stream)
        t1.synchronize()
        return t0.elapsed_time(t1) / n

    e2e_pipelined(4)
    torch.cuda.synchronize()
    e2e_ms = e2e_pipelined(n_pipe)
    e2e_value = bytes_step * world / (e2e_ms * 1e-3) / 1e9
    for b in range(2):
        got = bufs[b][2][:out.numel() * 2].view(torch.bfloat16).view(out.shape).to(dev)
        if not torch.equal(got, out):
            raise RuntimeError("pipelined end-to-end output differs from the device-resident step")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, inp)

    # ---- the Write step for the step's new tokens (each row's newest position),
    # timed last because it overwrites those tokens in the caches
    gen = torch.Generator(device=dev).manual_seed(wl.seed + 17)
    k_new = torch.randn((R, inputs.IDX_DIM), device=dev, generator=gen).to(torch.bfloat16)
    lat_new = torch.randn((R, inputs.LAT_DIM), device=dev, generator=gen).to(torch.bfloat16)
    ln_w = torch.ones(inputs.IDX_DIM, device=dev)
    ln_b = torch.zeros(inputs.IDX_DIM, device=dev)
    new_pos = (inp["row_len"] - 1).clamp(min=0)
    write_fn = lambda: dsa.dsa_write_kv(k_new, ln_w, ln_b, 1e-6, lat_new,  # noqa: E731
                                        inp["latent_scale"], inp["block_table"], inp["row_req"],
                                        new_pos, inp["key_cache"], inp["latent_cache"])
    g = _graph(write_fn, stream)
    write_ms = _time_launches(g.replay, n_stage, flush, stream)[0]
    write = {"tokens": R, "us": round(write_ms * 1e3, 2),
             "bytes": R * (inputs.IDX_DIM * 2 + inputs.LAT_DIM * 2 + inputs.IDX_DIM + 4 +
                           inputs.LAT_DIM)}

    # ---- the scan over MXFP4 index keys (68 bytes per token) on the same pages
    # and rows: random E2M1 codes with E8M0 scales near 1 (timing only; the
    # parity of this path is in the tests)
    def _mxfp4_leg():
        num_pages = inp["key_cache"].shape[0]
        mx_cache = torch.randint(0, 256, (num_pages, 4352), dtype=torch.uint8, device=dev,
                                 generator=gen)
        mx_cache[:, 4096:] = torch.randint(
            124, 131, (num_pages, 256), dtype=torch.uint8, device=dev, generator=gen)
        mx_qc = torch.randint(0, 256, (R, inputs.IDX_HEADS, 64), dtype=torch.uint8, device=dev,
                              generator=gen)
        mx_qs = torch.randint(124, 131, (R, inputs.IDX_HEADS, 4), dtype=torch.uint8, device=dev,
                              generator=gen)
        mx_fn = lambda: dsa.dsa_indexer_score_mxfp4(mx_qc, mx_qs, inp["w"], mx_cache,  # noqa: E731
                                                    inp["block_table"], inp["row_req"],
                                                    inp["row_len"], scores=scores, workspace=ws_s)
        g = _graph(mx_fn, stream)
        for _ in range(3):
            g.replay()
        mx_ms = _time_launches(g.replay, n_stage, flush, stream)[0]
        mx_bytes = traffic.scan_bytes_mxfp4(wl)
        mx_gbs = mx_bytes / (mx_ms * 1e-3) / 1e9
        mxfp4 = {"us": round(mx_ms * 1e3, 2), "fp8_scan_us": round(stage_ms["indexer_scan"] * 1e3, 2),
                 "speedup_vs_fp8": round(stage_ms["indexer_scan"] / mx_ms, 3),
                 "bytes": mx_bytes, "achieved_gbs": round(mx_gbs, 1),
                 "frac": round(mx_gbs / hbm_peak, 4)}
        del mx_cache
        return mxfp4

    try:
        mxfp4 = _mxfp4_leg()
    except dsa.DSAError as e:                          # reported, never fatal to the step's line
        mxfp4 = {"error": str(e)}

    # ---- sparse MLA over an NVFP4 latent cache (352 bytes per token) for the
    # same rows and selection (timing only; the parity of this path is in the tests)
    def _nvfp4_leg():
        nv_cache, nv_scale = inputs.nvfp4_latent_cache(inp, wl)
        ws_n = torch.empty(dsa.sparse_mla_workspace_size(R, H, wl.k), dtype=torch.uint8,
                           device=dev)
        nv_fn = lambda: dsa.dsa_sparse_mla_decode_nvfp4(  # noqa: E731
            inp["q"], nv_cache, nv_scale, inp["block_table"], inp["row_req"], inp["row_len"],
            idx, softmax_scale=inp["softmax_scale"], out=out, lse=lse, workspace=ws_n)
        g = _graph(nv_fn, stream)
        for _ in range(3):
            g.replay()
        nv_ms = _time_launches(g.replay, n_stage, flush, stream)[0]
        if dsa.check_device_status(ws_n) != 0:
            raise RuntimeError("device status raised by the NVFP4 attention")
        nv_bytes = traffic.gather_bytes_nvfp4(wl) + R * H * (inputs.LAT_DIM + inputs.V_DIM) * 2
        nv_gbs = nv_bytes / (nv_ms * 1e-3) / 1e9
        res = {"us": round(nv_ms * 1e3, 2), "fp8_mla_us": round(stage_ms["sparse_mla"] * 1e3, 2),
               "speedup_vs_fp8": round(stage_ms["sparse_mla"] / nv_ms, 3), "bytes": nv_bytes,
               "achieved_gbs": round(nv_gbs, 1), "frac": round(nv_gbs / hbm_peak, 4)}
        del nv_cache, ws_n, g
        return res

    try:
        nvfp4 = _nvfp4_leg()
    except (dsa.DSAError, RuntimeError) as e:
        nvfp4 = {"error": str(e)}

    # ---- the whole step over MXFP4 index keys and NVFP4 latent rows (the
    # pages' 10,080-byte-per-token caches) on the same pages and rows: random
    # MXFP4 keys and query, random NVFP4 rows (timing only; parity in the tests)
    def _fp4_step_leg():
        num_pages = inp["key_cache"].shape[0]
        kc = torch.randint(0, 256, (num_pages, 4352), dtype=torch.uint8, device=dev,
                           generator=gen)
        kc[:, 4096:] = torch.randint(124, 131, (num_pages, 256), dtype=torch.uint8, device=dev,
                                     generator=gen)
        qc4 = torch.randint(0, 256, (R, inputs.IDX_HEADS, 64), dtype=torch.uint8, device=dev,
                            generator=gen)
        qs4 = torch.randint(124, 131, (R, inputs.IDX_HEADS, 4), dtype=torch.uint8, device=dev,
                            generator=gen)
        nv_cache, nv_scale = inputs.nvfp4_latent_cache(inp, wl)
        ws4 = torch.empty(dsa.decode_step_workspace_size(wl.B, R, wl.max_pages, H, wl.k),
                          dtype=torch.uint8, device=dev)
        fn = lambda: dsa.dsa_decode_step_fp4(  # noqa: E731
            qc4, qs4, inp["w"], kc, nv_cache, nv_scale, inp["block_table"], inp["row_req"],
            inp["row_len"], inp["q"], softmax_scale=inp["softmax_scale"], k=wl.k, out=out,
            lse=lse, workspace=ws4)
        g = _graph(fn, stream)
        for _ in range(3):
            flush()
            g.replay()
        ms = _time_launches(g.replay, n_stage, flush, stream)[0]
        if dsa.check_device_status(ws4) != 0:
            raise RuntimeError("device status raised by the FP4 step")
        b4 = traffic.algorithmic_bytes_fp4(wl)
        gbs = b4 / (ms * 1e-3) / 1e9
        res = {"us_per_step": round(ms * 1e3, 2), "fp8_us_per_step": round(ms_per_step * 1e3, 2),
               "algorithmic_bytes": b4, "gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
               "kv_bytes_per_token": {"index_key": 68, "latent": 352}}
        del kc, nv_cache, ws4, g
        return res

    try:
        fp4_step = _fp4_step_leg()
    except (dsa.DSAError, RuntimeError) as e:
        fp4_step = {"error": str(e)}

    # ---- the other decode workloads, each step graph-replayed with L2 flushed
    del inp, out, lse, ws, stages, scores, idx, ws_s, step_graph, g, dev_buf, dev_obuf, bufs
    torch.cuda.empty_cache()
    side = {}
    if not args.no_side_configs:
        for ci in SIDE_CONFIGS.get(args.config, ()):
            try:
                name, res = _side_workload(dsa, ci, rank, dev, stream, flush, 50, hbm_peak)
                side[name] = res
            except (dsa.DSAError, RuntimeError) as e:
                side[inputs.config(ci).name] = {"error": str(e)}

    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_layer_step": round(ms_per_step * 1e3, 2),
        "tokens_per_s": round(R * world / (ms_per_step * 1e-3), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 (tensor cores), f32 softmax and selection",
        "data": "synthetic",
        "config": {"workload": wl.name, "requests": wl.B, "rows": R, "context": wl.ctx[0],
                   "heads": H, "topk": wl.k, "algorithmic_bytes_per_step": bytes_step,
                   "l2": "flushed before every timed step (256 MiB write, untimed)",
                   "launch": "each step is one CUDA-graph replay of dsa_decode_step",
                   "parallelism": f"replicas{world}"},
        "clocks": clock_info,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                "steps": n_pipe, "serial_ms_per_step": round(e2e_serial_ms, 5),
                "note": "per-step inputs (queries, head weights, block table, rows) packed in "
                        "one pinned host buffer and copied with one host-to-device copy, "
                        "out and lse copied back with one device-to-host copy, every step, "
                        "inside the timed region; step i+1's input copy and step i's output "
                        "copy run on a copy stream beside step i (two device buffers), as a "
                        "serving loop runs them; serial_ms_per_step is copy, step, copy in "
                        "turn with L2 flushed before each; the KV caches are resident layer "
                        "state"},
        "roofline": roofline,
        "tensor": tensor,
        "other_workloads": side,
        "dcp_topk": dcp,
        "write": write,
        "mxfp4_indexer": mxfp4,
        "nvfp4_sparse_mla": nvfp4,
        "fp4_step": fp4_step,
        "eager_ms_per_step": round(eager_ms, 5),
        "cpu_baseline": cpu,
        "gpu_launches": kernels_per_step(wl) * args.steps,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- CPU oracle
def _oracle_sample(wl, inp_host, requests):
    """Host inputs for the rows of the first `requests` requests (caches whole)."""
    rows = [r for r in range(wl.R) if int(inp_host["row_req"][r]) < requests]
    h = dict(inp_host)
    for key in ("q_idx", "q_idx_scale", "w", "row_req", "row_len", "q"):
        if h.get(key) is not None:
            h[key] = np.ascontiguousarray(h[key][rows])
    sample = inputs.Workload(wl.name + "_sample", wl.ctx[:requests], wl.rows[:requests], H=wl.H,
                             k=wl.k, q_idx_fp8=wl.q_idx_fp8)
    return h, sample


def _one_row_sample(wl, inp_host):
    """Host inputs of the first row alone (its request's caches whole)."""
    h = dict(inp_host)
    for key in ("q_idx", "q_idx_scale", "w", "row_req", "row_len", "q"):
        if h.get(key) is not None:
            h[key] = np.ascontiguousarray(h[key][:1])
    n = int(h["row_len"][0])
    sample = inputs.Workload(wl.name + "_row0", [n], [1], H=wl.H, k=wl.k, q_idx_fp8=wl.q_idx_fp8)
    return h, sample


def cpu_baseline(wl, inp, target_s=10.0):
    """Oracle on the first n requests, n grown until the run takes about target_s,
    on every host core; then the first row alone on one core."""
    from oracle import oracle
    host = inputs.to_numpy(inp)
    requests = 1
    while True:
        h, sample = _oracle_sample(wl, host, requests)
        t0 = time.perf_counter()
        oracle.decode_step(h, k=wl.k)
        dt = time.perf_counter() - t0
        if dt >= target_s or requests >= wl.B:
            break
        requests = min(wl.B, max(requests + 1, int(requests * target_s / max(dt, 1e-3))))
    b = traffic.algorithmic_bytes(sample)
    res = {"value": round(b / dt / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
           "kind": "oracle", "seconds": round(dt, 3),
           "sample": f"{requests} of {wl.B} requests ({sample.R} rows) of {wl.name}, full "
                     f"step (scores, top-{wl.k}, attention), float64 C + OpenMP"}
    threads = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        h1, s1 = _one_row_sample(wl, host)
        t0 = time.perf_counter()
        oracle.decode_step(h1, k=wl.k)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(threads)
    res["one_core"] = {"value": round(traffic.algorithmic_bytes(s1) / dt1 / 1e9, 4),
                       "unit": "GB/s", "cores": 1, "seconds": round(dt1, 3),
                       "sample": f"row 0 of {wl.name} ({s1.ctx[0]} tokens), full step"}
    return res


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    from oracle import oracle
    oracle.build()
    wl = inputs.config(args.config)
    inp = inputs.make_inputs(wl, device="cpu")
    host = inputs.to_numpy(inp)
    h, sample = _oracle_sample(wl, host, 1)
    for _ in range(min(args.warmup, 1)):
        oracle.decode_step(h, k=wl.k)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.decode_step(h, k=wl.k)
        times.append(time.perf_counter() - t0)
    b = traffic.algorithmic_bytes(sample)
    value = b * len(times) / sum(times) / 1e9
    cpu = {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
           "kind": "oracle",
           "sample": f"1 of {wl.B} requests ({sample.R} rows) of {wl.name} per step"}
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.mean(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "requests": wl.B, "rows": wl.R, "context": wl.ctx[0],
                   "heads": wl.H, "topk": wl.k, "sample_requests": 1},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2,
                    help="0 tiny, 1 16x4 rows @32K, 2 16x4 @256K (default), 3 1 row @1M, "
                         "4 prefill chunk of 4096 rows @128K")
    ap.add_argument("--impl", default="dsa", choices=["dsa", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side-configs", action="store_true",
                    help="skip the other decode workloads reported beside the headline")
    ap.add_argument("--requests", type=int, default=0,
                    help="keep only the first N requests of the workload (profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "dsa":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
