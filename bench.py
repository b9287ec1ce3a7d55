#!/usr/bin/env python3
"""Benchmark of the compressed-KV hot path on GB300 (one JSON line on stdout).

Workload (Llama-3-8B-shaped KV): 32 layers, 8 KV heads, head_dim 128, 32 query
heads, batch 1, 32768-token context, K turbo4 (3-bit + 1-bit QJL), V turbo4_mse
(3-bit).  K/V are fp16 N(0,1) with 1% outlier channels x20, generated per layer
from a seed.  One step = encode a 4096-token prefill chunk into all 32 layers
(K and V) + one decode-attention step over the full context of all 32 layers.

  value      decode-attention GB/s on the compressed bytes read (all layers),
             inputs resident in HBM, timed with CUDA events on the launch stream;
  e2e        the same metric through the C ABI with pinned host buffers: each
             step copies its K/V chunk and queries host->device and the output
             back, inside the timed region; the copy of step i + 1 overlaps the
             compute of step i on a second stream (two device buffer sets);
  roofline   the decode call against the measured HBM copy bandwidth;
  cpu_baseline  the CPU oracle (NumPy fp64) on a bounded sample of layers.

--impl reference times the CPU oracle as the reference arm on the same metric.
Under torchrun each rank runs the full workload on its own GPU (weak scaling).
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "llama3-8b-32k-turbo4"
METRIC = "turbo-KV decode attention GB/s & % HBM peak; KV encode tokens/s"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="tq", choices=["tq", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target seconds of timed oracle work")
    p.add_argument("--layers", type=int, default=0,
                   help="use only this many layers (small cases for profiler captures; 0 = all)")
    p.add_argument("--workload", default=WORKLOAD, choices=["llama3-8b-32k-turbo4", "llama-70b-128k-turbo4"],
                   help="contiguous batch-1 turbo4 workloads; the default is the benchmark's")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def reduce_max(values, device=None):
    """Elementwise max of per-rank timings over the default process group (identity
    without one).  Timing only: the data path has no collective (weak scaling)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def weak_scaling_value(bytes_per_rank, world, seconds_max):
    """Whole-job throughput: the bytes every rank processed over the slowest rank's time."""
    return world * bytes_per_rank / seconds_max / 1e9


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def source_hash(paths):
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_field(kernel_srcs, record, key):
    """Field `key` of a committed ncu record under profiles/, or None when the record is missing or
    the kernel sources changed since its counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", record)) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256_16") != source_hash(kernel_srcs):
        return None
    return rec.get(key)


def issue_roofline(instr_per_layer, layers, seconds, sm_mhz):
    """Warp instructions issued per second against the issue limit of the GPU: one warp instruction
    per clock on each of the 4 sub-partitions of the 152 SMs, at the median SM clock sampled
    during the timed region."""
    if instr_per_layer is None or not sm_mhz:
        return None
    achieved = instr_per_layer * layers / seconds / 1e9
    peak = 4 * 152 * sm_mhz / 1e3
    return {"achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "G warp instructions/s",
            "frac": round(achieved / peak, 4)}


def profiled_traffic(kernel_srcs, record="decode_traffic.json"):
    """DRAM bytes per call from a committed ncu summary under profiles/ (decode call:
    decode_traffic.json; encode call: encode_traffic.json), or None when the kernel
    sources changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", record)) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256_16") != source_hash(kernel_srcs):
        return None
    return rec.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks sampled every 200 ms around the timed region (see the call site)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.proc or not self.tmp:
            return None
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "window": "1 s of untimed steps of the same workload, then the timed region"}


# ---------------------------------------------------------------------------
# workload construction (device)
# ---------------------------------------------------------------------------

def build_workload(tq, W, torch, dev, layers=0):
    import dataclasses
    wl = W.WORKLOADS[WORKLOAD]
    if layers:
        wl = dataclasses.replace(wl, n_layers=layers)
    if not wl.encode_chunk:  # decode-only recipes: the step still encodes a 4096-token chunk per layer
        wl = dataclasses.replace(wl, encode_chunk=4096)
    L, H, d, T, Hq, chunk = wl.n_layers, wl.n_kv_heads, wl.head_dim, wl.ctx, wl.n_q_heads, wl.encode_chunk
    signs, S = W.wht_signs(wl.wht_seed, d), W.qjl_matrix(wl.qjl_seed, d)
    ctx = tq.tq_context_create(d, wl.wht_seed, wl.qjl_seed, signs, S)
    kview = tq.alloc_view(wl.k_format, d, H, page_size=T, num_pages=1, n_layers=L, device=dev)
    vview = tq.alloc_view(wl.v_format, d, H, page_size=T, num_pages=1, n_layers=L, device=dev)
    k_chunk = torch.empty((L, chunk, H, d), dtype=torch.float16, device=dev)
    v_chunk = torch.empty_like(k_chunk)
    for l in range(L):
        k = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * l, device=dev, outlier_frac=wl.outlier_frac)
        v = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * l + 1, device=dev, outlier_frac=wl.outlier_frac)
        st = tq.tq_encode_kv(ctx, kview, k, vview, v, l, 1, T, T * H * d, H * d)
        assert st == tq.TQ_OK, tq.tq_status_string(st)
        # the chunk re-encodes the last `chunk` tokens, so the cache stays the same across steps
        k_chunk[l].copy_(k[T - chunk:])
        v_chunk[l].copy_(v[T - chunk:])
    q = W.normal_tensor((L, 1, Hq, d), seed=wl.seed * 1000 + 999, device=dev)
    ws_bytes = tq.tq_decode_workspace_bytes(ctx, L, 1, Hq, T)
    return dict(wl=wl, ctx=ctx, kview=kview, vview=vview, k_chunk=k_chunk, v_chunk=v_chunk, q=q,
                seq_lens=torch.tensor([T], dtype=torch.int32, device=dev),
                ws=torch.empty(ws_bytes, dtype=torch.uint8, device=dev), ws_bytes=ws_bytes,
                out=torch.empty((L, 1, Hq, d), dtype=torch.float32, device=dev), signs=signs, S=S)


def encode_step(tq, w, k_chunk, v_chunk, stream):
    wl = w["wl"]
    L, H, d, T, chunk = wl.n_layers, wl.n_kv_heads, wl.head_dim, wl.ctx, wl.encode_chunk
    st = tq.tq_encode_kv(w["ctx"], w["kview"], k_chunk, w["vview"], v_chunk, 0, L, chunk, chunk * H * d, H * d,
                         None, T - chunk, stream)
    assert st == tq.TQ_OK, tq.tq_status_string(st)


def decode_step(tq, w, q, out, stream):
    wl = w["wl"]
    st = tq.tq_decode_attention(w["ctx"], q, 0, wl.n_layers, 1, wl.n_q_heads, w["kview"], w["vview"], 0,
                                w["seq_lens"], wl.ctx, None, 0, 1.0 / math.sqrt(wl.head_dim), 1e-6, w["ws"],
                                w["ws_bytes"], out, stream)
    assert st == tq.TQ_OK, tq.tq_status_string(st)


def decode_bytes(tq, wl):
    per_token_head = tq.tq_vector_bytes(wl.k_format, wl.head_dim) + tq.tq_vector_bytes(wl.v_format, wl.head_dim)
    return wl.n_layers * wl.n_kv_heads * wl.ctx * per_token_head


def encode_bytes(tq, wl):
    """Algorithmic bytes of one encode call: the fp16 K and V chunk read, the codes and headers written."""
    vectors = wl.n_layers * wl.encode_chunk * wl.n_kv_heads
    written = tq.tq_vector_bytes(wl.k_format, wl.head_dim) + tq.tq_vector_bytes(wl.v_format, wl.head_dim)
    return vectors * (2 * 2 * wl.head_dim + written)


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------

def oracle_decode_sample(w, tq, W, torch, dev, target_s, max_layers=8):
    """Times the oracle's decode (dequantisation of the compressed cache + fp64 attention)
    on as many layers as fit in ~target_s seconds; returns (GB/s, layers, seconds, cores)."""
    import numpy as np
    from oracle import tq_oracle as O

    wl = w["wl"]
    L, H, d, T = wl.n_layers, wl.n_kv_heads, wl.head_dim, wl.ctx
    per_layer = decode_bytes(tq, wl) / L
    timed, layers = 0.0, 0
    q = w["q"].cpu().numpy().astype(np.float64)
    for l in range(min(L, max_layers)):
        k = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * l, device=dev, outlier_frac=wl.outlier_frac).cpu().numpy()
        v = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * l + 1, device=dev,
                        outlier_frac=wl.outlier_frac).cpu().numpy()
        ek = O.turbo_encode(k, wl.k_format, w["signs"], w["S"])
        ev = O.turbo_encode(v, wl.v_format, w["signs"], None)
        t0 = time.perf_counter()
        kt = O.turbo_dequant(ek, wl.k_format, w["signs"], w["S"])
        vt = O.turbo_dequant(ev, wl.v_format, w["signs"], None)
        O.decode_attention(q[l, 0], kt, vt, 1.0 / math.sqrt(d), 1e-6)
        timed += time.perf_counter() - t0
        layers += 1
        if timed >= target_s:
            break
    return per_layer * layers / timed / 1e9, layers, timed, os.cpu_count()


def run_reference(args, rank):
    """Reference arm: the CPU oracle on this machine's host cores, on the same metric."""
    if rank != 0:
        return
    import numpy as np
    import torch
    from kv_cache_quantization_turbo_gb300 import workloads as W
    from oracle import tq_oracle as O

    wl = W.WORKLOADS[WORKLOAD]
    H, d, T = wl.n_kv_heads, wl.head_dim, wl.ctx
    signs, S = W.wht_signs(wl.wht_seed, d), W.qjl_matrix(wl.qjl_seed, d)
    k = W.kv_tensor(T, H, d, seed=wl.seed * 1000, outlier_frac=wl.outlier_frac).numpy()
    v = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 1, outlier_frac=wl.outlier_frac).numpy()
    q = W.normal_tensor((wl.n_q_heads, d), seed=wl.seed * 1000 + 999).numpy().astype(np.float64)
    ek = O.turbo_encode(k, wl.k_format, signs, S)
    ev = O.turbo_encode(v, wl.v_format, signs, None)
    bytes_layer = H * T * (d * 4 // 8 + 4 + d * 3 // 8 + 2)

    def step():
        kt = O.turbo_dequant(ek, wl.k_format, signs, S)
        vt = O.turbo_dequant(ev, wl.v_format, signs, None)
        O.decode_attention(q, kt, vt, 1.0 / math.sqrt(d), 1e-6)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = bytes_layer / dt / 1e9
    sample = f"one layer (8 KV heads x {T} tokens, turbo4/turbo4_mse) per step: dequantise + fp64 attention"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers_per_step": 1, "kv_heads": H, "q_heads": wl.n_q_heads,
                   "head_dim": d, "ctx": T, "k_format": wl.k_format, "v_format": wl.v_format},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def main():
    global WORKLOAD
    args = parse()
    WORKLOAD = args.workload
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        run_reference(args, rank)
        return
    import torch

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    import __graft_entry__
    __graft_entry__.build()
    from kv_cache_quantization_turbo_gb300 import tq
    from kv_cache_quantization_turbo_gb300 import workloads as W

    w = build_workload(tq, W, torch, dev, args.layers)
    wl = w["wl"]
    stream = torch.cuda.current_stream(dev)
    dbytes = decode_bytes(tq, wl)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        encode_step(tq, w, w["k_chunk"], w["v_chunk"], stream)
        decode_step(tq, w, w["q"], w["out"], stream)
    barrier()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(local_rank) as clocks:
        # untimed steps for ~1 s, so that the clock record (200 ms samples) spans a steady load
        # that ends where the timed region starts
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 1.0:
            encode_step(tq, w, w["k_chunk"], w["v_chunk"], stream)
            decode_step(tq, w, w["q"], w["out"], stream)
            torch.cuda.synchronize(dev)
        barrier()
        t_wall = time.perf_counter()
        for s in range(args.steps):
            ev[s][0].record(stream)
            encode_step(tq, w, w["k_chunk"], w["v_chunk"], stream)
            ev[s][1].record(stream)
            decode_step(tq, w, w["q"], w["out"], stream)
            ev[s][2].record(stream)
        barrier()
        t_wall = time.perf_counter() - t_wall
    t_enc = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps / 1e3
    t_dec = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps / 1e3
    t_step = sum(e[0].elapsed_time(e[2]) for e in ev) / args.steps / 1e3
    t_enc, t_dec, t_step = reduce_max([t_enc, t_dec, t_step], dev)

    # end to end through the C ABI with pinned host buffers, as a two-stage pipeline: the inputs of
    # step i + 1 are copied on a second stream while step i encodes and decodes (two device buffer
    # sets).  The timed region holds exactly K input copies, K encode + decode steps and K result
    # reads: it starts before the first copy and ends after the last read.
    out_ref = w["out"].cpu()  # the result of the last device-timed step
    k_host = w["k_chunk"].cpu().pin_memory()
    v_host = w["v_chunk"].cpu().pin_memory()
    q_host = w["q"].cpu().pin_memory()
    out_host = torch.empty(w["out"].shape, dtype=torch.float32).pin_memory()
    bufs = [(torch.empty_like(w["k_chunk"]), torch.empty_like(w["v_chunk"]), torch.empty_like(w["q"]))
            for _ in range(2)]
    h2d = k_host.numel() * 2 + v_host.numel() * 2 + q_host.numel() * 4
    d2h = out_host.numel() * 4
    e2e_steps = max(1, args.steps)
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def issue_copy(i):
        b = i & 1
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(consumed[b])  # buffer set b is free once step i - 2 used it
            for dst, src in zip(bufs[b], (k_host, v_host, q_host)):
                dst.copy_(src, non_blocking=True)
            copied[b].record(copy_stream)

    def run_pipeline(n):
        issue_copy(0)
        for i in range(n):
            b = i & 1
            stream.wait_event(copied[b])
            if i + 1 < n:
                issue_copy(i + 1)
            k_dev, v_dev, q_dev = bufs[b]
            encode_step(tq, w, k_dev, v_dev, stream)
            decode_step(tq, w, q_dev, w["out"], stream)
            consumed[b].record(stream)
            out_host.copy_(w["out"], non_blocking=True)

    with torch.cuda.stream(stream):
        run_pipeline(args.warmup)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)
        run_pipeline(e2e_steps)
    e1 = torch.cuda.Event(enable_timing=True)
    e1.record(stream)
    barrier()
    # the pipelined steps reproduce the device-resident result bit for bit (same inputs; every split
    # is owned by one warp and the combine merges in a fixed order)
    assert torch.equal(out_host, out_ref), "end-to-end output differs from the device-timed output"
    t_e2e = e0.elapsed_time(e1) / e2e_steps / 1e3
    t_e2e = reduce_max([t_e2e], dev)[0]
    ok, flags = tq.tq_get_status(w["ctx"])
    assert ok == tq.TQ_OK, f"device status flags {flags}"

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peaks, peak_src = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    value = weak_scaling_value(dbytes, world, t_dec)
    achieved = dbytes / t_dec / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        gbs, nl, secs, cores = oracle_decode_sample(w, tq, W, torch, dev, args.cpu_seconds)
        cpu = {"value": round(gbs, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{nl} of {wl.n_layers} layers (8 KV heads x {wl.ctx} tokens each): oracle dequantisation"
                         f" + fp64 attention, {secs:.1f} s timed"}
    clk = clocks.summary()
    csrc = os.path.join(ROOT, "kv_cache_quantization_turbo_gb300", "csrc")
    dec_srcs = [os.path.join(csrc, f) for f in ("tq_decode_mma.cuh", "tq_decode_mma128.cu", "tq_decode.cu",
                                                 "tq_warp_mma.cuh")]
    enc_srcs = [os.path.join(csrc, f) for f in ("tq_encode.cu", "tq_tc.cuh")]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16-operand/f32-accumulate", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": wl.n_layers, "kv_heads": wl.n_kv_heads,
                   "q_heads": wl.n_q_heads, "head_dim": wl.head_dim, "ctx": wl.ctx, "batch": 1,
                   "k_format": wl.k_format, "v_format": wl.v_format, "encode_chunk": wl.encode_chunk,
                   "skip_threshold": 1e-6, "decode_bytes_per_step": dbytes,
                   "l2": f"inputs larger than L2: each decode step sweeps all {wl.n_layers} layers "
                         f"({dbytes / 1e9:.2f} GB > 129 MB)"},
        "pct_hbm_peak": {"measured": round(100 * achieved / hbm, 2), "nominal": round(100 * achieved /
                                                                                       NOMINAL_HBM_GBS, 2)},
        "decode_tokens_per_s": round(world / t_dec, 2),
        "decode_ms": round(t_dec * 1e3, 4),
        "encode_tokens_per_s": round(world * wl.encode_chunk / t_enc, 1),
        "encode_ms": round(t_enc * 1e3, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": f"{peak_src} hbm_gbs",
                     "kernel": "decode attention call (prologue + split-K attention + combine), one launch set "
                               f"over all {wl.n_layers} layers",
                     "traffic": profiled_traffic(dec_srcs)},
        "roofline_encode": {"bound": "hbm", "achieved": round(encode_bytes(tq, wl) / t_enc / 1e9, 2), "peak": hbm,
                            "unit": "GB/s", "frac": round(encode_bytes(tq, wl) / t_enc / 1e9 / hbm, 4),
                            "peak_source": f"{peak_src} hbm_gbs",
                            "traffic": profiled_traffic(enc_srcs, "encode_traffic.json"),
                            "kernel": f"encode call (K and V kernels) of the {wl.encode_chunk}-token chunk over all "
                                      f"{wl.n_layers} layers: fp16 input read, codes and headers written"},
        "roofline_issue": {
            "bound": "issue",
            "decode": issue_roofline(profiled_field(dec_srcs, "decode_traffic.json", "warp_instructions_per_layer"),
                                     wl.n_layers, t_dec, clk.get("sm_mhz")),
            "encode": issue_roofline(profiled_field(enc_srcs, "encode_traffic.json", "warp_instructions_per_layer"),
                                     wl.n_layers, t_enc, clk.get("sm_mhz")),
            "what": "warp instructions per call (smsp__inst_executed.sum of the attention kernel / of the two "
                    "encode kernels, from the ncu records under profiles/, null once the kernels changed) over "
                    "the call's time; the pipe that binds both calls"},
        "e2e": {"value": round(weak_scaling_value(dbytes, world, t_e2e), 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(t_e2e * 1e3, 3),
                "what": "per step: H2D of the 4096-token K/V chunk (all layers) and q from pinned memory, encode,"
                        " decode, D2H of out; the copy of step i + 1 overlaps step i on a second stream;"
                        " value = decode bytes / time per step"},
        "gpu_launches": 5 * args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
