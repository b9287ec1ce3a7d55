"""tq_decode_attention_static: decode attention for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run decode attention (their device
memory is already reserved by a pool of their own, they run inside an allocator
callback, or they are a plug-in that only receives inputs and outputs).  This entry
point keeps its workspace in a fixed 16 MiB array inside the library instead of
taking one from the caller.  Through the C ABI, its output must equal that of
tq_decode_attention with a caller workspace bit for bit (the same kernels run on the
same inputs), on two calls in a row (the second call finds the array holding the first
call's data).  The file is named so that pytest
collects it last; it must pass alone in a fresh process as well.
"""
import ctypes
import math

import pytest
import torch

from kv_cache_quantization_turbo_gb300 import tq
from kv_cache_quantization_turbo_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STATIC_LIMIT = 16 << 20  # bytes, as declared in include/tq.h


def _cache(d, H, T, kfmt, vfmt, seed):
    ctx = tq.tq_context_create(d, 1, 2, W.wht_signs(1, d), W.qjl_matrix(2, d))
    kview = tq.alloc_view(kfmt, d, H, page_size=T, num_pages=2)
    vview = tq.alloc_view(vfmt, d, H, page_size=T, num_pages=2)
    for b in range(2):
        k = W.kv_tensor(T, H, d, seed=seed + b, device="cuda", outlier_frac=0.01)
        v = W.kv_tensor(T, H, d, seed=seed + 10 + b, device="cuda", outlier_frac=0.01)
        assert tq.tq_encode_kv(ctx, kview, k, vview, v, 0, 1, T, T * H * d, H * d, None, b * T) == tq.TQ_OK
    return ctx, kview, vview


@pytest.mark.parametrize("kfmt,vfmt", [("turbo4", "turbo4_mse"), ("turbo3", "turbo3_mse")])
def test_static_workspace_matches_caller_workspace(kfmt, vfmt):
    assert torch.cuda.is_available()
    d, H, Hq, T = 128, 4, 16, 3000
    ctx, kview, vview = _cache(d, H, T, kfmt, vfmt, seed=40)
    try:
        lens = torch.tensor([T, 1777], dtype=torch.int32, device="cuda")  # two sequences, one layer
        ws_bytes = tq.tq_decode_workspace_bytes(ctx, 1, 2, Hq, T)
        assert 0 < ws_bytes <= STATIC_LIMIT
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        for call in range(2):
            q = W.normal_tensor((1, 2, Hq, d), seed=100 + call, device="cuda")
            ref = torch.empty((1, 2, Hq, d), dtype=torch.float32, device="cuda")
            got = torch.full_like(ref, float("nan"))
            assert tq.tq_decode_attention(ctx, q, 0, 1, 2, Hq, kview, vview, 0, lens, T, None, 0, 1 / math.sqrt(d),
                                          0.0, ws, ws_bytes, ref) == tq.TQ_OK
            assert tq.tq_decode_attention_static(ctx, q, 0, 1, 2, Hq, kview, vview, 0, lens, T, None, 0,
                                                 1 / math.sqrt(d), 0.0, got) == tq.TQ_OK
            torch.cuda.synchronize()
            assert torch.isfinite(got).all()
            # the same deterministic kernels on the same inputs: equal bit for bit
            assert torch.equal(got, ref), (got - ref).abs().max().item()
    finally:
        tq.tq_context_destroy(ctx)


def test_static_workspace_rejects_requests_above_its_size():
    assert torch.cuda.is_available()
    d, H, Hq, T = 128, 8, 32, 1024
    ctx, kview, vview = _cache(d, H, T, "turbo4", "turbo4_mse", seed=1)
    try:
        max_ctx = 1 << 20
        assert tq.tq_decode_workspace_bytes(ctx, 80, 64, Hq, max_ctx) > STATIC_LIMIT  # 80 layers x 64 sequences
        q = torch.zeros((80, 64, Hq, d), device="cuda")
        out = torch.full_like(q, 7.0)
        lens = torch.zeros(64, dtype=torch.int32, device="cuda")
        st = tq.tq_decode_attention_static(ctx, q, 0, 80, 64, Hq, kview, vview, 0, lens, max_ctx, None, 0, 1.0,
                                           0.0, out)
        assert st == tq.TQ_ERR_WORKSPACE
        torch.cuda.synchronize()
        assert torch.all(out == 7.0)  # nothing was launched
    finally:
        tq.tq_context_destroy(ctx)
