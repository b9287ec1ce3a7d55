"""Decode-attention (and paged encode) timing on the workload recipes that the benchmark step does not cover.

    python -m kv_cache_quantization_turbo_gb300.decode_timing --workload paged-batch64-turbo3 --head-dim 128
    python -m kv_cache_quantization_turbo_gb300.decode_timing --workload asym-q8k-turbo2v-needles
    python -m kv_cache_quantization_turbo_gb300.decode_timing --workload contiguous --kv-heads 4 --q-heads 64

Builds the recipe's compressed cache on cuda:0 with the library's own encoder (seeded synthetic
inputs from workloads.py), then times whole decode calls (every layer of the recipe, one query
per sequence and query head) with CUDA events on the launching stream after warm-up calls, and
prints one JSON line: algorithmic bytes (the compressed K and V of every attended token, once)
per second.  The paged recipe also times the encode of one layer (every token of every sequence,
K and V, written to its slot in the shuffled pages): fp16 read plus codes written per second.
The caches are several GB, far larger than L2, so no flush is needed between calls.
"""
import argparse
import json
import math

import numpy as np
import torch

from . import tq
from . import workloads as W


def _time(fn, calls, warmup):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(calls):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / calls / 1e3


def _decode_fn(ctx, q, kview, vview, layer_begin, lens, max_ctx, block_table=None, max_blocks=0, tau=1e-6):
    L, B, Hq, d = q.shape
    ws_bytes = tq.tq_decode_workspace_bytes(ctx, L, B, Hq, max_ctx)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((L, B, Hq, d), dtype=torch.float32, device="cuda")
    sl = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    bt = None if block_table is None else torch.as_tensor(block_table.astype(np.int32), device="cuda")

    def run():
        st = tq.tq_decode_attention(ctx, q, 0, L, B, Hq, kview, vview, layer_begin, sl, max_ctx, bt, max_blocks,
                                    1.0 / math.sqrt(d), tau, ws, ws_bytes, out)
        assert st == tq.TQ_OK, tq.tq_status_string(st)
    return run


def _needles(wl):
    """q8_0 K everywhere; V q8_0 on the boundary layers and the recipe's V format elsewhere; one
    sequence of wl.ctx tokens with 16 needles per KV head.  A per-layer format table: one K view of
    every layer, a boundary V view and a middle V view, decoded in one tq_decode_attention_layers call."""
    L, H, d, T, Hq = wl.n_layers, wl.n_kv_heads, wl.head_dim, wl.ctx, wl.n_q_heads
    boundary = sorted(wl.v_format_layers)
    middle = [l for l in range(L) if l not in wl.v_format_layers]
    ctx = tq.tq_context_create(d, wl.wht_seed, wl.qjl_seed, W.wht_signs(wl.wht_seed, d), W.qjl_matrix(wl.qjl_seed, d))
    kview = tq.alloc_view(wl.k_format, d, H, page_size=T, num_pages=1, n_layers=L)
    vb = tq.alloc_view("q8_0", d, H, page_size=T, num_pages=1, n_layers=len(boundary))
    vm = tq.alloc_view(wl.v_format, d, H, page_size=T, num_pages=1, n_layers=len(middle))
    v_views = [vb if l in wl.v_format_layers else vm for l in range(L)]
    v_layers = [boundary.index(l) if l in wl.v_format_layers else middle.index(l) for l in range(L)]
    q = torch.empty((L, 1, Hq, d), dtype=torch.float32, device="cuda")
    for l in range(L):
        k, ql, _ = W.needle_workload(T, H, Hq, d, seed=wl.seed * 1000 + 2 * l, device="cuda")
        v = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * l + 1, device="cuda")
        q[l, 0] = ql
        st = tq.tq_encode_kv_layers(ctx, [kview], [l], [v_views[l]], [v_layers[l]], 1, k, v, T, T * H * d, H * d)
        assert st == tq.TQ_OK, tq.tq_status_string(st)
    ws_bytes = tq.tq_decode_workspace_bytes(ctx, L, 1, Hq, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((L, 1, Hq, d), dtype=torch.float32, device="cuda")
    sl = torch.tensor([T], dtype=torch.int32, device="cuda")
    k_views, k_layers = [kview] * L, list(range(L))

    def run():
        st = tq.tq_decode_attention_layers(ctx, q, 0, L, 1, Hq, k_views, k_layers, v_views, v_layers, sl, T, None, 0,
                                           1.0 / math.sqrt(d), 1e-6, ws, ws_bytes, out)
        assert st == tq.TQ_OK, tq.tq_status_string(st)
    vb_ = lambda f: tq.tq_vector_bytes(f, d)
    nbytes = H * T * (len(boundary) * (vb_(wl.k_format) + vb_("q8_0")) + len(middle) * (vb_(wl.k_format) +
                                                                                        vb_(wl.v_format)))
    cfg = {"layers": L, "kv_heads": H, "q_heads": Hq, "head_dim": d, "ctx": T, "k_format": wl.k_format,
           "v_format": wl.v_format, "boundary_layers_v": "q8_0", "boundary_layers": boundary,
           "calls": "one tq_decode_attention_layers call per decode step"}
    return ctx, run, nbytes, cfg, None


def _paged(wl, d):
    """wl.batch sequences of U[1K, ctx] tokens in shuffled wl.page_size-token pages."""
    L, H, Hq, B, P = wl.n_layers, wl.n_kv_heads, wl.n_q_heads, wl.batch, wl.page_size
    lens = W.seq_lens_uniform(B, 1024, wl.ctx, wl.seed)
    bt, npages = W.shuffled_block_table(lens, P, wl.seed)
    ctx = tq.tq_context_create(d, wl.wht_seed, wl.qjl_seed, W.wht_signs(wl.wht_seed, d), W.qjl_matrix(wl.qjl_seed, d))
    kview = tq.alloc_view(wl.k_format, d, H, page_size=P, num_pages=npages, n_layers=L)
    vview = tq.alloc_view(wl.v_format, d, H, page_size=P, num_pages=npages, n_layers=L)
    slots = np.concatenate([bt[b, np.arange(lens[b]) // P] * P + np.arange(lens[b]) % P for b in range(B)])
    slots_d = torch.as_tensor(slots.astype(np.int64), device="cuda")
    n_tok = int(lens.sum())
    for l in range(L):
        k = W.kv_tensor(n_tok, H, d, seed=wl.seed * 1000 + 2 * l, device="cuda")
        v = W.kv_tensor(n_tok, H, d, seed=wl.seed * 1000 + 2 * l + 1, device="cuda")
        st = tq.tq_encode_kv(ctx, kview, k, vview, v, l, 1, n_tok, n_tok * H * d, H * d, slots_d)
        assert st == tq.TQ_OK, tq.tq_status_string(st)
        if l == 0:
            k0, v0 = k, v  # layer 0's inputs: the encode timing re-encodes them into the same slots
        del k, v

    def encode_layer0():
        st = tq.tq_encode_kv(ctx, kview, k0, vview, v0, 0, 1, n_tok, n_tok * H * d, H * d, slots_d)
        assert st == tq.TQ_OK, tq.tq_status_string(st)
    enc_bytes = n_tok * H * (2 * 2 * d + tq.tq_vector_bytes(wl.k_format, d) + tq.tq_vector_bytes(wl.v_format, d))
    q = W.normal_tensor((L, B, Hq, d), seed=wl.seed * 1000 + 999, device="cuda")
    f = _decode_fn(ctx, q, kview, vview, 0, lens, int(lens.max()), bt, bt.shape[1])
    nbytes = L * H * n_tok * (tq.tq_vector_bytes(wl.k_format, d) + tq.tq_vector_bytes(wl.v_format, d))
    cfg = {"layers": L, "kv_heads": H, "q_heads": Hq, "head_dim": d, "batch": B, "page_size": P,
           "tokens": n_tok, "max_ctx": int(lens.max()), "k_format": wl.k_format, "v_format": wl.v_format}
    return ctx, f, nbytes, cfg, (encode_layer0, n_tok, enc_bytes)


def _contiguous(a):
    """One sequence of a.ctx tokens per layer, contiguous cache, any query-head grouping and format
    pair (e.g. 4 KV heads with 64 query heads: 16 query heads per KV head)."""
    L, H, Hq, d, T = a.layers, a.kv_heads, a.q_heads, a.head_dim, a.ctx
    ctx = tq.tq_context_create(d, 1, 2, W.wht_signs(1, d), W.qjl_matrix(2, d))
    kview = tq.alloc_view(a.k_format, d, H, page_size=T, num_pages=1, n_layers=L)
    vview = tq.alloc_view(a.v_format, d, H, page_size=T, num_pages=1, n_layers=L)
    for l in range(L):
        k = W.kv_tensor(T, H, d, seed=7000 + 2 * l, device="cuda", outlier_frac=0.01)
        v = W.kv_tensor(T, H, d, seed=7001 + 2 * l, device="cuda", outlier_frac=0.01)
        st = tq.tq_encode_kv(ctx, kview, k, vview, v, l, 1, T, T * H * d, H * d)
        assert st == tq.TQ_OK, tq.tq_status_string(st)
        del k, v
    q = W.normal_tensor((L, 1, Hq, d), seed=7999, device="cuda")
    f = _decode_fn(ctx, q, kview, vview, 0, [T], T)
    nbytes = L * H * T * (tq.tq_vector_bytes(a.k_format, d) + tq.tq_vector_bytes(a.v_format, d))
    cfg = {"layers": L, "kv_heads": H, "q_heads": Hq, "head_dim": d, "ctx": T, "k_format": a.k_format,
           "v_format": a.v_format}
    return ctx, f, nbytes, cfg, None


def _prefill(a):
    """Chunked prefill: one sequence of a.ctx cached tokens per layer, the last a.chunk of them the
    chunk's own; every layer's chunk attends causally over the compressed cache (one
    tq_prefill_attention call per layer).  Returns the call plus its attention FLOPs: per chunk
    token i, 2 d (QK) + 2 d (PV) per attended key and query head, and the tensor-core FLOPs the
    kernel issues (score products with high and low query parts of both score parts: 4 QK
    products, plus PV; 64-key tiles up to each 128-row tile's last position)."""
    L, H, Hq, d, T, C = a.layers, a.kv_heads, a.q_heads, a.head_dim, a.ctx, a.chunk
    start = T - C
    ctx = tq.tq_context_create(d, 1, 2, W.wht_signs(1, d), W.qjl_matrix(2, d))
    kview = tq.alloc_view(a.k_format, d, H, page_size=T, num_pages=1, n_layers=L)
    vview = tq.alloc_view(a.v_format, d, H, page_size=T, num_pages=1, n_layers=L)
    for l in range(L):
        k = W.kv_tensor(T, H, d, seed=8000 + 2 * l, device="cuda", outlier_frac=0.01)
        v = W.kv_tensor(T, H, d, seed=8001 + 2 * l, device="cuda", outlier_frac=0.01)
        st = tq.tq_encode_kv(ctx, kview, k, vview, v, l, 1, T, T * H * d, H * d)
        assert st == tq.TQ_OK, tq.tq_status_string(st)
        del k, v
    q = W.normal_tensor((L, C, Hq, d), seed=8999, device="cuda")
    ws_bytes = tq.tq_prefill_workspace_bytes(ctx, C, Hq)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((L, C, Hq, d), dtype=torch.float32, device="cuda")

    def run():
        for l in range(L):
            st = tq.tq_prefill_attention(ctx, q[l], 0, C, Hq, kview, vview, l, 0, None, 0, start, 1.0 / math.sqrt(d),
                                         ws, ws_bytes, out[l])
            assert st == tq.TQ_OK, tq.tq_status_string(st)
    attended = sum(start + i + 1 for i in range(C))
    useful = L * Hq * attended * 4 * d
    G = Hq // H
    rows = C * G
    tiles = 0
    for r0 in range(0, rows, 128):
        last = min(r0 + 128, rows) - 1
        tiles += (start + last // G + 1 + 63) // 64
    issued = L * H * tiles * 128 * 64 * d * 2 * 5  # four QK products and one PV product per tile
    nbytes = L * H * T * (tq.tq_vector_bytes(a.k_format, d) + tq.tq_vector_bytes(a.v_format, d))
    cfg = {"layers": L, "kv_heads": H, "q_heads": Hq, "head_dim": d, "ctx": T, "chunk": C, "start": start,
           "k_format": a.k_format, "v_format": a.v_format, "useful_flops": useful, "tensor_flops": issued}
    return ctx, run, nbytes, cfg, None


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--workload", required=True, choices=["asym-q8k-turbo2v-needles", "paged-batch64-turbo3",
                                                         "contiguous", "prefill"])
    p.add_argument("--chunk", type=int, default=4096, help="prefill only: chunk tokens (the last of --ctx)")
    p.add_argument("--head-dim", type=int, default=128, choices=[64, 128, 256], help="paged and contiguous")
    p.add_argument("--layers", type=int, default=32, help="contiguous only (as the next five)")
    p.add_argument("--kv-heads", type=int, default=4)
    p.add_argument("--q-heads", type=int, default=64)
    p.add_argument("--ctx", type=int, default=32768)
    p.add_argument("--k-format", default="turbo4")
    p.add_argument("--v-format", default="turbo4_mse")
    p.add_argument("--calls", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    args = p.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("decode_timing needs a CUDA device")
    if args.workload == "contiguous":
        ctx, run, nbytes, cfg, enc = _contiguous(args)
    elif args.workload == "prefill":
        ctx, run, nbytes, cfg, enc = _prefill(args)
    else:
        wl = W.WORKLOADS[args.workload]
        ctx, run, nbytes, cfg, enc = _needles(wl) if args.workload == "asym-q8k-turbo2v-needles" else \
            _paged(wl, args.head_dim)
    dt = _time(run, args.calls, args.warmup)
    line = {"metric": "decode_attention_bandwidth", "value": round(nbytes / dt / 1e9, 1), "unit": "GB/s",
            "ms_per_call": round(dt * 1e3, 4), "algorithmic_bytes": int(nbytes), "calls": args.calls,
            "warmup": args.warmup, "workload": args.workload, "config": cfg, "skip_threshold": 1e-6}
    if args.workload == "prefill":
        line["metric"] = "prefill_attention"
        line["tokens_per_s"] = round(cfg["chunk"] * cfg["layers"] / dt, 1)
        line["useful_tflops"] = round(cfg["useful_flops"] / dt / 1e12, 2)
        line["tensor_tflops"] = round(cfg["tensor_flops"] / dt / 1e12, 2)
        line["skip_threshold"] = 0.0
    if enc is not None:
        encode_layer0, n_tok, enc_bytes = enc
        te = _time(encode_layer0, args.calls, args.warmup)
        line["encode_one_layer"] = {"ms": round(te * 1e3, 4), "tokens_per_s": round(n_tok / te, 1),
                                    "gb_per_s": round(enc_bytes / te / 1e9, 1), "algorithmic_bytes": int(enc_bytes)}
    st, flags = tq.tq_get_status(ctx)
    assert st == tq.TQ_OK and flags == 0, (st, flags)
    tq.tq_context_destroy(ctx)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
