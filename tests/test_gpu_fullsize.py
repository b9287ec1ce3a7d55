"""Parity at the benchmark recipes' full sizes, on sampled (layer, KV head) slices.

Each test builds the whole workload on the GPU (all layers, full context) with
the library's encoder and runs decode attention over all layers in one call
(the benchmark's launch configuration), twice:

1. on the cache as the GPU encoded it.  The codes of each sampled slice are
   checked against the oracle (indices bit-exact outside the 1e-6 boundary
   band, QJL signs and rnorm against the oracle's stage 2 on the GPU's own
   indices, headers within 1 ulp), and every query head of the slice must
   match the oracle's fp64 attention over the codes the GPU stored (read back
   and dequantised by the oracle) within 2e-3;
2. after the oracle's own codes are written into the sampled slices: every
   query head of the slice must match the oracle end to end (oracle encode,
   dequantise, attention) within 2e-3.

Inputs are regenerated from their seeds on the same device and copied to the host.
"""
import math

import numpy as np
import pytest
import torch

from kv_cache_quantization_turbo_gb300 import tq
from kv_cache_quantization_turbo_gb300 import workloads as W
from oracle import tq_oracle as O
import gpu_common as C

pytestmark = pytest.mark.gpu


def _gpu_slice(view, layer, kvh, slot_ids):
    """The stored payload and header bytes of KV head kvh at the given slots: [n, 1, bytes]."""
    pay, hdr = C.read_vectors(view, layer)
    pay = C.slot_major(pay, slot_ids, view.page_size)[:, kvh][:, None]
    hdr = C.slot_major(hdr, slot_ids, view.page_size)[:, kvh][:, None]
    return pay, hdr


def _check_codes(view, layer, fmt, x16, kvh, slot_ids, signs, S):
    """Checks the GPU codes of one slice against the oracle.  x16: fp16 [n, d] of KV head kvh at
    the given slots.  Returns (oracle encoding, the GPU's codes in the oracle's form)."""
    enc = C.oracle_encode(fmt, x16[:, None, :], signs, S)
    pay, hdr = _gpu_slice(view, layer, kvh, slot_ids)
    if fmt == "q8_0":
        np.testing.assert_array_equal(pay.view(np.int8), enc[0])
        np.testing.assert_array_equal(hdr.view(np.float16), enc[1])
    else:
        C.check_turbo_codes(fmt, view.head_dim, pay, hdr, enc, S=S)
    return enc, C.gpu_codes(fmt, view.head_dim, pay, hdr)


def _replace(view, layer, fmt, enc, kvh, slot_ids):
    C.write_oracle_codes(view, enc, fmt, slot_ids, layer=layer, head=kvh)


def _attention(q_rows, ek, ev, kfmt, vfmt, signs, S, d, tau=0.0):
    """Oracle attention of one KV head on its codes, q_rows [G, d]; also, per query head,
    the weighted norm of the V terms the oracle's Sparse-V rule drops,
    sum over p_j < tau of p_j ||v~_j||."""
    kt = C.oracle_dequant(kfmt, ek, signs, S)
    vt = C.oracle_dequant(vfmt, ev, signs, S)
    q64 = q_rows.astype(np.float64)
    o_full, _ = O.decode_attention(q64, kt, vt, 1.0 / math.sqrt(d), tau)
    s = (q64 @ kt[:, 0, :].T) / math.sqrt(d)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    bound = np.sum(np.where(p < tau, p, 0.0) * np.linalg.norm(vt[:, 0, :], axis=-1)[None, :], axis=1)
    return o_full, bound


def _within_skip_bound(got, o_full, bound):
    """Sparse V drops a subset of the terms the oracle's rule drops, so the output stays
    within their weighted norm of the full attention (plus the parity tolerance)."""
    dev = np.linalg.norm(np.asarray(got, np.float64) - o_full, axis=-1)
    return bool(np.all(dev <= bound + C.ATTN_RTOL * np.linalg.norm(o_full, axis=-1)))


def _compare(got, want, what):
    err = C.rel_err_per_head(got, want)
    assert err.max() < C.ATTN_RTOL, (what, err.max())


def test_llama3_8b_32k_turbo4_bench_configuration():
    """32 layers x 8 KV heads x 32768 tokens, d 128, 32 query heads, turbo4 / turbo4_mse,
    built, re-encoded and decoded exactly as bench.py does (one decode call over all layers)."""
    C.require_cuda()
    import bench
    dev = torch.device("cuda", 0)
    w = bench.build_workload(tq, W, torch, dev)
    wl = w["wl"]
    d, H, T, L = wl.head_dim, wl.n_kv_heads, wl.ctx, wl.n_layers
    G = wl.n_q_heads // H
    scale = 1.0 / math.sqrt(d)

    def decode_full():
        out = torch.empty_like(w["out"])
        st = tq.tq_decode_attention(w["ctx"], w["q"], 0, L, 1, wl.n_q_heads, w["kview"], w["vview"], 0,
                                    w["seq_lens"], T, None, 0, scale, 0.0, w["ws"], w["ws_bytes"], out)
        assert st == tq.TQ_OK
        torch.cuda.synchronize()
        return out

    try:
        stream = torch.cuda.current_stream()
        bench.encode_step(tq, w, w["k_chunk"], w["v_chunk"], stream)  # the timed encode (last 4096 tokens)
        torch.cuda.synchronize()
        assert tq.tq_get_status(w["ctx"])[0] == tq.TQ_OK
        # 1. the GPU-encoded cache: the timed decode (Sparse V at 1e-6) and the full one
        bench.decode_step(tq, w, w["q"], w["out"], stream)
        torch.cuda.synchronize()
        out_skip = w["out"].clone()
        out_full = decode_full()
        encs = {}
        for layer, kvh in ((0, 3), (31, 6)):
            k = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * layer, device=dev,
                            outlier_frac=wl.outlier_frac)[:, kvh].cpu().numpy()
            v = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * layer + 1, device=dev,
                            outlier_frac=wl.outlier_frac)[:, kvh].cpu().numpy()
            ek, gk = _check_codes(w["kview"], layer, wl.k_format, k, kvh, np.arange(T), w["signs"], w["S"])
            ev, gv = _check_codes(w["vview"], layer, wl.v_format, v, kvh, np.arange(T), w["signs"], w["S"])
            q = w["q"][layer, 0, kvh * G:(kvh + 1) * G].cpu().numpy()
            o_full, bound = _attention(q, gk, gv, wl.k_format, wl.v_format, w["signs"], w["S"], d, 1e-6)
            heads = slice(kvh * G, (kvh + 1) * G)
            _compare(out_full[layer, 0, heads].cpu().numpy(), o_full, ("gpu codes", layer, kvh))
            assert _within_skip_bound(out_skip[layer, 0, heads].cpu().numpy(), o_full, bound)
            encs[layer, kvh] = (ek, ev, q)
        # 2. the oracle's codes in the sampled slices
        for (layer, kvh), (ek, ev, q) in encs.items():
            _replace(w["kview"], layer, wl.k_format, ek, kvh, np.arange(T))
            _replace(w["vview"], layer, wl.v_format, ev, kvh, np.arange(T))
        bench.decode_step(tq, w, w["q"], w["out"], stream)
        torch.cuda.synchronize()
        out_skip = w["out"].clone()
        out_full = decode_full()
        assert tq.tq_get_status(w["ctx"])[0] == tq.TQ_OK
        for (layer, kvh), (ek, ev, q) in encs.items():
            o_full, bound = _attention(q, ek, ev, wl.k_format, wl.v_format, w["signs"], w["S"], d, 1e-6)
            heads = slice(kvh * G, (kvh + 1) * G)
            _compare(out_full[layer, 0, heads].cpu().numpy(), o_full, ("oracle codes", layer, kvh))
            assert _within_skip_bound(out_skip[layer, 0, heads].cpu().numpy(), o_full, bound)
    finally:
        tq.tq_context_destroy(w["ctx"])


def test_llama_70b_128k_turbo4_sampled():
    """80 layers x 8 KV heads x 131072 tokens (9.9 GB compressed), 64 query heads (GQA 8),
    generated layer by layer; one decode call over all 80 layers."""
    C.require_cuda()
    wl = W.WORKLOADS["llama-70b-128k-turbo4"]
    L, H, d, T, Hq = wl.n_layers, wl.n_kv_heads, wl.head_dim, wl.ctx, wl.n_q_heads
    G = Hq // H
    ctx = C.Ctx(d, wl.wht_seed, wl.qjl_seed)
    try:
        kview = tq.alloc_view(wl.k_format, d, H, page_size=T, num_pages=1, n_layers=L)
        vview = tq.alloc_view(wl.v_format, d, H, page_size=T, num_pages=1, n_layers=L)
        for l in range(L):
            k = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * l, device="cuda", outlier_frac=wl.outlier_frac)
            v = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * l + 1, device="cuda", outlier_frac=wl.outlier_frac)
            st = tq.tq_encode_kv(ctx.h, kview, k, vview, v, l, 1, T, T * H * d, H * d)
            assert st == tq.TQ_OK
            del k, v
        q = W.normal_tensor((L, 1, Hq, d), seed=wl.seed * 1000 + 999, device="cuda")
        out = C.decode(ctx, q, kview, vview, [T], T, tau=0.0)  # the GPU-encoded cache
        encs = {}
        for layer, kvh in ((40, 5), (79, 1)):
            k = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * layer, device="cuda",
                            outlier_frac=wl.outlier_frac)[:, kvh].cpu().numpy()
            v = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * layer + 1, device="cuda",
                            outlier_frac=wl.outlier_frac)[:, kvh].cpu().numpy()
            ek, gk = _check_codes(kview, layer, wl.k_format, k, kvh, np.arange(T), ctx.signs, ctx.S)
            ev, gv = _check_codes(vview, layer, wl.v_format, v, kvh, np.arange(T), ctx.signs, ctx.S)
            qr = q[layer, 0, kvh * G:(kvh + 1) * G].cpu().numpy()
            o_full = _attention(qr, gk, gv, wl.k_format, wl.v_format, ctx.signs, ctx.S, d)[0]
            _compare(out[layer, 0, kvh * G:(kvh + 1) * G].cpu().numpy(), o_full, ("gpu codes", layer, kvh))
            encs[layer, kvh] = (ek, ev, qr)
        for (layer, kvh), (ek, ev, qr) in encs.items():
            _replace(kview, layer, wl.k_format, ek, kvh, np.arange(T))
            _replace(vview, layer, wl.v_format, ev, kvh, np.arange(T))
        out = C.decode(ctx, q, kview, vview, [T], T, tau=0.0)
        for (layer, kvh), (ek, ev, qr) in encs.items():
            o_full = _attention(qr, ek, ev, wl.k_format, wl.v_format, ctx.signs, ctx.S, d)[0]
            _compare(out[layer, 0, kvh * G:(kvh + 1) * G].cpu().numpy(), o_full, ("oracle codes", layer, kvh))
        assert tq.tq_get_status(ctx.h)[0] == tq.TQ_OK
    finally:
        ctx.close()


def test_asymmetric_boundary_layers_needles_sampled():
    """64 layers x 4 KV heads x 32768 tokens, 32 query heads (GQA 8): K q8_0; V turbo2_mse
    except the first 2 and last 2 layers (q8_0); queries aligned with 16 needles x8;
    skip threshold 1e-6.  A per-layer format table: one K view of all 64 layers, a 4-layer q8_0 V
    view for the boundary layers and a 60-layer turbo2_mse V view, decoded in one
    tq_decode_attention_layers call."""
    C.require_cuda()
    wl = W.WORKLOADS["asym-q8k-turbo2v-needles"]
    L, H, d, T, Hq = wl.n_layers, wl.n_kv_heads, wl.head_dim, wl.ctx, wl.n_q_heads
    G = Hq // H
    boundary = sorted(wl.v_format_layers)
    middle = [l for l in range(L) if l not in wl.v_format_layers]
    ctx = C.Ctx(d, wl.wht_seed, wl.qjl_seed)
    try:
        kview = tq.alloc_view("q8_0", d, H, page_size=T, num_pages=1, n_layers=L)
        vb = tq.alloc_view("q8_0", d, H, page_size=T, num_pages=1, n_layers=len(boundary))
        vm = tq.alloc_view(wl.v_format, d, H, page_size=T, num_pages=1, n_layers=len(middle))
        v_views = [vb if l in wl.v_format_layers else vm for l in range(L)]
        v_layers = [boundary.index(l) if l in wl.v_format_layers else middle.index(l) for l in range(L)]
        qs = torch.empty((L, 1, Hq, d), dtype=torch.float32, device="cuda")
        for l in range(L):
            k, q, _ = W.needle_workload(T, H, Hq, d, seed=wl.seed * 1000 + 2 * l, device="cuda")
            v = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * l + 1, device="cuda")
            qs[l, 0] = q
            st = tq.tq_encode_kv_layers(ctx.h, [kview], [l], [v_views[l]], [v_layers[l]], 1, k, v, T, T * H * d,
                                        H * d)
            assert st == tq.TQ_OK
        nbytes = tq.tq_decode_workspace_bytes(ctx.h, L, 1, Hq, T)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        lens = torch.tensor([T], dtype=torch.int32, device="cuda")

        def decode_all():
            out = torch.full((L, 1, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
            st = tq.tq_decode_attention_layers(ctx.h, qs, 0, L, 1, Hq, [kview] * L, list(range(L)), v_views, v_layers,
                                               lens, T, None, 0, 1.0 / math.sqrt(d), 1e-6, ws, nbytes, out)
            assert st == tq.TQ_OK
            torch.cuda.synchronize()
            return out

        def pick(out, layer, kvh):
            return out[layer, 0, kvh * G:(kvh + 1) * G].cpu().numpy()

        out = decode_all()  # the GPU-encoded cache
        encs = {}
        for layer, kvh in ((1, 2), (30, 0), (63, 3)):
            k, _, _ = W.needle_workload(T, H, Hq, d, seed=wl.seed * 1000 + 2 * layer, device="cuda")
            v = W.kv_tensor(T, H, d, seed=wl.seed * 1000 + 2 * layer + 1, device="cuda")
            vfmt = wl.v_format_layers.get(layer, wl.v_format)
            vv_, li = v_views[layer], v_layers[layer]
            ek, gk = _check_codes(kview, layer, "q8_0", k[:, kvh].cpu().numpy(), kvh, np.arange(T), ctx.signs, ctx.S)
            ev, gv = _check_codes(vv_, li, vfmt, v[:, kvh].cpu().numpy(), kvh, np.arange(T), ctx.signs, ctx.S)
            qr = qs[layer, 0, kvh * G:(kvh + 1) * G].cpu().numpy()
            o_full, bound = _attention(qr, gk, gv, "q8_0", vfmt, ctx.signs, ctx.S, d, 1e-6)
            got = pick(out, layer, kvh)
            # peaked softmax: what Sparse V drops is far below the parity tolerance
            _compare(got, o_full, ("gpu codes", layer, kvh))
            assert _within_skip_bound(got, o_full, bound)
            encs[layer, kvh] = (vv_, li, vfmt, ek, ev, qr)
        for (layer, kvh), (vv_, li, vfmt, ek, ev, qr) in encs.items():
            _replace(kview, layer, "q8_0", ek, kvh, np.arange(T))
            _replace(vv_, li, vfmt, ev, kvh, np.arange(T))
        out = decode_all()
        for (layer, kvh), (vv_, li, vfmt, ek, ev, qr) in encs.items():
            o_full, bound = _attention(qr, ek, ev, "q8_0", vfmt, ctx.signs, ctx.S, d, 1e-6)
            got = pick(out, layer, kvh)
            _compare(got, o_full, ("oracle codes", layer, kvh))
            assert _within_skip_bound(got, o_full, bound)
        assert tq.tq_get_status(ctx.h)[0] == tq.TQ_OK
    finally:
        ctx.close()


@pytest.mark.parametrize("d", [64, 128, 256])
def test_paged_batch64_turbo3_sampled(d):
    """64 sequences with context ~ U[1K, 16K], 32 layers x 8 KV heads, 32 query heads,
    turbo3 / turbo3_mse in 16-token pages with a shuffled block table."""
    C.require_cuda()
    wl = W.WORKLOADS["paged-batch64-turbo3"]
    L, H, Hq, B, P = wl.n_layers, wl.n_kv_heads, wl.n_q_heads, wl.batch, wl.page_size
    G = Hq // H
    lens = W.seq_lens_uniform(B, 1024, 16384, wl.seed)
    bt, npages = W.shuffled_block_table(lens, P, wl.seed)
    ctx = C.Ctx(d, wl.wht_seed, wl.qjl_seed)
    try:
        kview = tq.alloc_view(wl.k_format, d, H, page_size=P, num_pages=npages, n_layers=L)
        vview = tq.alloc_view(wl.v_format, d, H, page_size=P, num_pages=npages, n_layers=L)
        # slot of every (sequence, token): block_table page * P + in-page offset
        slots = np.concatenate([bt[b, np.arange(lens[b]) // P] * P + np.arange(lens[b]) % P for b in range(B)])
        slots_d = torch.as_tensor(slots.astype(np.int64), device="cuda")
        T_all = int(lens.sum())
        for l in range(L):
            k = W.kv_tensor(T_all, H, d, seed=wl.seed * 1000 + 2 * l, device="cuda")
            v = W.kv_tensor(T_all, H, d, seed=wl.seed * 1000 + 2 * l + 1, device="cuda")
            st = tq.tq_encode_kv(ctx.h, kview, k, vview, v, l, 1, T_all, T_all * H * d, H * d, slots_d)
            assert st == tq.TQ_OK
            del k, v
        q = W.normal_tensor((L, B, Hq, d), seed=wl.seed * 1000 + 999, device="cuda")
        offs = np.concatenate([[0], np.cumsum(lens)])

        def decode():
            return C.decode(ctx, q, kview, vview, lens, int(lens.max()), block_table=bt, max_blocks=bt.shape[1])

        out = decode()  # the GPU-encoded cache
        encs = {}
        for layer, b, kvh in ((3, 0, 1), (17, 37, 7)):
            sl = slots[offs[b]:offs[b + 1]]
            k = W.kv_tensor(T_all, H, d, seed=wl.seed * 1000 + 2 * layer, device="cuda")[offs[b]:offs[b + 1], kvh]
            v = W.kv_tensor(T_all, H, d, seed=wl.seed * 1000 + 2 * layer + 1, device="cuda")[offs[b]:offs[b + 1],
                                                                                                 kvh]
            ek, gk = _check_codes(kview, layer, wl.k_format, k.cpu().numpy(), kvh, sl, ctx.signs, ctx.S)
            ev, gv = _check_codes(vview, layer, wl.v_format, v.cpu().numpy(), kvh, sl, ctx.signs, ctx.S)
            qr = q[layer, b, kvh * G:(kvh + 1) * G].cpu().numpy()
            o_full = _attention(qr, gk, gv, wl.k_format, wl.v_format, ctx.signs, ctx.S, d)[0]
            _compare(out[layer, b, kvh * G:(kvh + 1) * G].cpu().numpy(), o_full, ("gpu codes", layer, b, kvh))
            encs[layer, b, kvh] = (sl, ek, ev, qr)
        for (layer, b, kvh), (sl, ek, ev, qr) in encs.items():
            _replace(kview, layer, wl.k_format, ek, kvh, sl)
            _replace(vview, layer, wl.v_format, ev, kvh, sl)
        out = decode()
        for (layer, b, kvh), (sl, ek, ev, qr) in encs.items():
            o_full = _attention(qr, ek, ev, wl.k_format, wl.v_format, ctx.signs, ctx.S, d)[0]
            _compare(out[layer, b, kvh * G:(kvh + 1) * G].cpu().numpy(), o_full, ("oracle codes", layer, b, kvh))
        st, flags = tq.tq_get_status(ctx.h)
        assert st == tq.TQ_OK, flags
    finally:
        ctx.close()
