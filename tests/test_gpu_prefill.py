"""GPU parity of the chunked-prefill attention (tq_prefill_attention) against the oracle.

The cache is encoded by the library; the oracle dequantises the codes the GPU stored and runs its
fp64 causal prefill attention (prefill_attention), so both sides attend over identical codes.
Every query row of the chunk is compared (relative error 2e-3 per row).  Sizes span several
64-key tiles and 128-row query tiles with ragged ends; chunks start at 0 and deep in the context;
contiguous and paged (shuffled 16-token pages) caches.
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


@pytest.fixture(scope="module")
def ctx128():
    C.require_cuda()
    c = C.Ctx(128)
    yield c
    c.close()


def _run(ctx, kfmt, vfmt, H, G, start, n, page=None, seed=0, q_fp16=False):
    d, T = 128, start + n
    Hq = H * G
    k = W.kv_tensor(T, H, d, seed=seed, device="cuda", outlier_frac=0.01)
    v = W.kv_tensor(T, H, d, seed=seed + 1, device="cuda", outlier_frac=0.01)
    if page is None:
        kv = tq.alloc_view(kfmt, d, H, page_size=T, num_pages=1)
        vv = tq.alloc_view(vfmt, d, H, page_size=T, num_pages=1)
        slots, bt, mb = np.arange(T), None, 0
    else:
        btab, npages = W.shuffled_block_table(np.array([T]), page, seed=seed + 2, extra_pages=3)
        kv = tq.alloc_view(kfmt, d, H, page_size=page, num_pages=npages)
        vv = tq.alloc_view(vfmt, d, H, page_size=page, num_pages=npages)
        slots = btab[0, np.arange(T) // page] * page + np.arange(T) % page
        bt, mb = torch.as_tensor(btab[0], device="cuda"), btab.shape[1]
    st = tq.tq_encode_kv(ctx.h, kv, k, vv, v, 0, 1, T, T * H * d, H * d,
                         None if page is None else torch.as_tensor(slots.astype(np.int64), device="cuda"))
    assert st == tq.TQ_OK
    q = W.normal_tensor((n, Hq, d), seed=seed + 3, device="cuda")
    if q_fp16:
        q = q.half()
    ws_bytes = tq.tq_prefill_workspace_bytes(ctx.h, n, Hq)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((n, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
    st = tq.tq_prefill_attention(ctx.h, q, int(q_fp16), n, Hq, kv, vv, 0, 0, bt, mb, start, 1 / math.sqrt(d), ws,
                                 ws_bytes, out)
    assert st == tq.TQ_OK, tq.tq_status_string(st)
    torch.cuda.synchronize()
    assert tq.tq_get_status(ctx.h)[0] == tq.TQ_OK
    kp, kh = C.read_vectors(kv)
    vp, vh = C.read_vectors(vv)
    kp, kh, vp, vh = (C.slot_major(x, slots, kv.page_size) for x in (kp, kh, vp, vh))  # [T, H, bytes]
    kt = C.oracle_dequant(kfmt, C.gpu_codes(kfmt, d, kp, kh), ctx.signs, ctx.S)
    vt = C.oracle_dequant(vfmt, C.gpu_codes(vfmt, d, vp, vh), ctx.signs, ctx.S)
    want = O.prefill_attention(q.float().cpu().numpy().astype(np.float64), kt, vt, start, 1 / math.sqrt(d))
    got = out.cpu().numpy()
    err = C.rel_err_per_head(got.reshape(-1, d), want.reshape(-1, d))
    assert err.max() < C.ATTN_RTOL, err.max()


@pytest.mark.parametrize("kfmt,vfmt", [("turbo4", "turbo4_mse"), ("turbo3", "turbo3_mse"), ("turbo2", "turbo2_mse"),
                                       ("turbo4", "turbo2_mse")])
def test_prefill_format_pairs(ctx128, kfmt, vfmt):
    """Chunk of 150 tokens after 200 cached ones, GQA 4: three 128-row query tiles per KV head
    (the last ragged), keys in six 64-key tiles (the last ragged)."""
    _run(ctx128, kfmt, vfmt, H=2, G=4, start=200, n=150, seed=1)


@pytest.mark.parametrize("G,start,n", [(1, 0, 1), (1, 0, 129), (4, 0, 64), (8, 1000, 300), (16, 37, 40)])
def test_prefill_shapes(ctx128, G, start, n):
    """Head groupings 1..16, chunks from the start of the context and deep in it, a one-token chunk."""
    _run(ctx128, "turbo4", "turbo4_mse", H=2, G=G, start=start, n=n, seed=10 + G)


def test_prefill_paged_and_fp16_queries(ctx128):
    """Shuffled 16-token pages through a block table; fp16 queries."""
    _run(ctx128, "turbo3", "turbo3_mse", H=2, G=4, start=333, n=200, page=16, seed=30, q_fp16=True)


def test_prefill_rejects_bad_arguments(ctx128):
    d = 128
    kv = tq.alloc_view("turbo4", d, 2, page_size=64, num_pages=1)
    vv = tq.alloc_view("turbo4_mse", d, 2, page_size=64, num_pages=1)
    q = torch.zeros((10, 8, d), device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    args = dict(softmax_scale=0.1, workspace=ws, workspace_bytes=ws.numel(), out=out)

    def call(kview, vview, n, start, wsb=None):
        return tq.tq_prefill_attention(ctx128.h, q, 0, n, 8, kview, vview, 0, 0, None, 0, start, 0.1, ws,
                                       ws.numel() if wsb is None else wsb, out)
    assert call(kv, vv, 10, 54) == tq.TQ_OK
    assert call(kv, vv, 10, 55) == tq.TQ_ERR_INVALID_ARG  # past the page's capacity
    assert call(vv, vv, 10, 0) == tq.TQ_ERR_UNSUPPORTED  # a turbo-MSE K
    assert call(kv, tq.alloc_view("q8_0", d, 2, page_size=64, num_pages=1), 10, 0) == tq.TQ_ERR_UNSUPPORTED
    assert call(kv, vv, 10, 0, wsb=16) == tq.TQ_ERR_WORKSPACE
    torch.cuda.synchronize()


def test_prefill_full_size_sampled_rows(ctx128):
    """The timed configuration: a 4096-token chunk at the end of a 32768-token context, 8 KV heads,
    GQA 4 (32 query heads), turbo4 / turbo4_mse, one call as the timing runs it.  Sampled rows
    (chunk token, query head): the first and last tokens, 128-row tile boundaries (32 tokens of a
    KV head's 4 query heads), 64-key tile boundaries of the causal edge, on three KV heads, against
    the oracle over the codes the GPU stored for those heads."""
    d, H, G, n, start = 128, 8, 4, 4096, 28672
    T, Hq = start + n, H * G
    k = W.kv_tensor(T, H, d, seed=41, device="cuda", outlier_frac=0.01)
    v = W.kv_tensor(T, H, d, seed=42, device="cuda", outlier_frac=0.01)
    kv = tq.alloc_view("turbo4", d, H, page_size=T, num_pages=1)
    vv = tq.alloc_view("turbo4_mse", d, H, page_size=T, num_pages=1)
    assert tq.tq_encode_kv(ctx128.h, kv, k, vv, v, 0, 1, T, T * H * d, H * d, None) == tq.TQ_OK
    del k, v
    q = W.normal_tensor((n, Hq, d), seed=43, device="cuda")
    ws_bytes = tq.tq_prefill_workspace_bytes(ctx128.h, n, Hq)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((n, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
    st = tq.tq_prefill_attention(ctx128.h, q, 0, n, Hq, kv, vv, 0, 0, None, 0, start, 1 / math.sqrt(d), ws,
                                 ws_bytes, out)
    assert st == tq.TQ_OK, tq.tq_status_string(st)
    torch.cuda.synchronize()
    assert tq.tq_get_status(ctx128.h)[0] == tq.TQ_OK
    got_all = out.cpu().numpy()
    assert np.isfinite(got_all).all()
    kp, kh = C.read_vectors(kv)
    vp, vh = C.read_vectors(vv)
    qn = q.cpu().numpy().astype(np.float64)
    tokens = [0, 1, 31, 32, 63, 64, 95, 96, 127, 128, 2047, 2048, 4063, 4064, 4094, 4095]
    errs = []
    for kvh in (0, 3, 7):
        kt = C.oracle_dequant("turbo4", C.gpu_codes("turbo4", d, kp[0, kvh], kh[0, kvh]), ctx128.signs, ctx128.S)
        vt = C.oracle_dequant("turbo4_mse", C.gpu_codes("turbo4_mse", d, vp[0, kvh], vh[0, kvh]), ctx128.signs,
                              ctx128.S)
        for j, i in enumerate(tokens):
            h = kvh * G + (j + kvh) % G
            want = O.prefill_attention(qn[i:i + 1, h:h + 1], kt[:, None], vt[:, None], start + i, 1 / math.sqrt(d))
            errs.append(C.rel_err_per_head(got_all[i, h][None], want[0, 0][None])[0])
    assert max(errs) < C.ATTN_RTOL, max(errs)
