"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on seeded inputs.

Sizes span several tiles/batches and ragged tails; every comparison follows
the rules in gpu_common (bit-exact codes outside the 1e-6 band, fp16 headers
within 1 ulp, attention within 2e-3 relative per query head).
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

TURBO_K = ["turbo2", "turbo3", "turbo4"]
TURBO_V = ["turbo2_mse", "turbo3_mse", "turbo4_mse"]


@pytest.fixture(scope="module", params=[64, 128, 256])
def ctx(request):
    C.require_cuda()
    c = C.Ctx(request.param)
    yield c
    c.close()


@pytest.fixture(scope="module")
def ctx128():
    C.require_cuda()
    c = C.Ctx(128)
    yield c
    c.close()


def test_context_tables_are_the_inputs(ctx):
    s, S, cb, bd = tq.tq_context_get_tables(ctx.h, ctx.d)
    np.testing.assert_array_equal(s, ctx.signs)
    np.testing.assert_array_equal(S, ctx.S)
    for b in (1, 2, 3):
        c, bb = O.codebook(b, ctx.d)
        np.testing.assert_array_equal(cb[b - 1, : 1 << b].astype(np.float64), c)
        np.testing.assert_array_equal(bd[b - 1, : (1 << b) - 1].astype(np.float64), bb)


# ---------------------------------------------------------------------------
# encode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", TURBO_K + TURBO_V)
def test_encode_turbo_bit_exact(ctx, fmt):
    d, H, T = ctx.d, 4, 301  # ragged: not a multiple of any batch size
    x = W.kv_tensor(T, H, d, seed=10 + d, device="cuda", outliers_per_head=4)
    view = tq.alloc_view(fmt, d, H, page_size=T, num_pages=1)
    C.encode(ctx, view, x, is_k=fmt in TURBO_K)
    pay, hdr = C.read_vectors(view)
    enc = O.turbo_encode(x.cpu().numpy(), fmt, ctx.signs, ctx.S)
    # view order is [page, head, slot]; oracle order is [token, head]
    C.check_turbo_codes(fmt, d, pay[0].transpose(1, 0, 2), hdr[0].transpose(1, 0, 2), enc, S=ctx.S)


@pytest.mark.parametrize("fmt", ["turbo4", "turbo3_mse"])
def test_encode_scattered_slots_multi_layer(ctx128, fmt):
    """Paged view, shuffled slots, two layers written at layer_begin = 1."""
    d, H, T, P, pages = 128, 8, 200, 16, 20
    x = torch.stack([W.kv_tensor(T, H, d, seed=s, device="cuda", outlier_frac=0.01) for s in (3, 4)])
    view = tq.alloc_view(fmt, d, H, page_size=P, num_pages=pages, n_layers=3)
    rng = np.random.default_rng(0)
    slots = rng.permutation(P * pages)[:T].astype(np.int64)
    C.encode(ctx128, view, x, is_k=fmt in TURBO_K, layer_begin=1, slots=torch.as_tensor(slots, device="cuda"))
    for l in (0, 1):
        pay, hdr = C.read_vectors(view, layer=1 + l)
        enc = O.turbo_encode(x[l].cpu().numpy(), fmt, ctx128.signs, ctx128.S)
        C.check_turbo_codes(fmt, d, C.slot_major(pay, slots, P), C.slot_major(hdr, slots, P), enc, S=ctx128.S)
    pay0, hdr0 = C.read_vectors(view, layer=0)
    assert not pay0.any() and not hdr0.any()  # untouched layer


@pytest.mark.parametrize("H", [3, 6, 12])
def test_encode_tensor_core_partial_batches_and_strides(ctx128, H):
    """d = 128 (the tensor-core encoder): head counts that do not divide 128, so a batch holds
    H * floor(128 / H) < 128 rows, a ragged token count, two layers, and K and V read in place from
    one interleaved [layer][token][K | V][head][d] buffer (token stride 2 H d, layer stride 2 T H d)."""
    d, T, L = 128, 173, 2
    kv = torch.stack([torch.stack([W.kv_tensor(T, H, d, seed=40 + 10 * l + j, device="cuda", outliers_per_head=2)
                                   for j in (0, 1)], dim=1) for l in range(L)])  # [L, T, 2, H, d]
    assert kv.is_contiguous()
    for fmt, j in (("turbo4", 0), ("turbo3_mse", 1)):
        is_k = j == 0
        view = tq.alloc_view(fmt, d, H, page_size=T, num_pages=1, n_layers=L)
        x = kv[:, :, j]  # a strided view of the interleaved buffer
        args = (view, x, None, None) if is_k else (None, None, view, x)
        st = tq.tq_encode_kv(ctx128.h, *args, 0, L, T, T * 2 * H * d, 2 * H * d, None, 0, None)
        assert st == tq.TQ_OK, tq.tq_status_string(st)
        for l in range(L):
            pay, hdr = C.read_vectors(view, layer=l)
            enc = O.turbo_encode(x[l].cpu().numpy(), fmt, ctx128.signs, ctx128.S)
            C.check_turbo_codes(fmt, d, pay[0].transpose(1, 0, 2), hdr[0].transpose(1, 0, 2), enc, S=ctx128.S)


def test_encode_zero_and_single_vectors(ctx128):
    """Zero vectors (every rotated coordinate exactly 0: the tie rule decides, identically on
    both sides), a basis vector, and the all-ones vector, whose rotated coordinates are
    multiples of 1/d and so often sit exactly on the middle boundary (band rule)."""
    d, H = 128, 2
    x = torch.zeros((3, H, d), dtype=torch.float16, device="cuda")
    x[1, 0, 5] = 1.0
    x[2, 1] = 1.0
    zero = np.array([[True, True], [False, True], [True, False]])
    for fmt in ("turbo3", "turbo2_mse"):
        view = tq.alloc_view(fmt, d, H, page_size=3, num_pages=1)
        C.encode(ctx128, view, x, is_k=fmt in TURBO_K)
        pay, hdr = C.read_vectors(view)
        enc = O.turbo_encode(x.cpu().numpy(), fmt, ctx128.signs, ctx128.S)
        pay, hdr = pay[0].transpose(1, 0, 2), hdr[0].transpose(1, 0, 2)
        C.check_turbo_codes(fmt, d, pay[zero], hdr[zero], {k: v[zero] for k, v in enc.items()}, exact=True,
                            S=ctx128.S)
        C.check_turbo_codes(fmt, d, pay[~zero], hdr[~zero], {k: v[~zero] for k, v in enc.items()},
                            band_limit=False, S=ctx128.S)


def test_encode_q8_0_bit_exact(ctx):
    d, H, T = ctx.d, 3, 77
    x = W.kv_tensor(T, H, d, seed=21, device="cuda", outliers_per_head=2)
    x[5, 1, :32] = 0  # an all-zero block
    view = tq.alloc_view("q8_0", d, H, page_size=T, num_pages=1)
    C.encode(ctx, view, x, is_k=True)
    pay, hdr = C.read_vectors(view)
    q, dl = O.q8_0_encode(x.cpu().numpy())
    np.testing.assert_array_equal(pay[0].transpose(1, 0, 2).view(np.int8), q)
    np.testing.assert_array_equal(hdr[0].transpose(1, 0, 2).view(np.float16), dl)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_encode_minmax_bit_exact(ctx, bits):
    d, H, T = ctx.d, 2, 65
    x = W.kv_tensor(T, H, d, seed=31, device="cuda", outliers_per_head=3)
    x[3, 0, :64] = 0.25  # a flat group
    view = tq.alloc_view("minmax", d, H, page_size=T, num_pages=1, bits=bits)
    C.encode(ctx, view, x, is_k=False)
    pay, hdr = C.read_vectors(view)
    q, sc, zr = O.minmax_encode(x.cpu().numpy().astype(np.float32), bits=bits)
    from _layout import unpack_codes
    np.testing.assert_array_equal(unpack_codes(pay[0].transpose(1, 0, 2), d, bits), q)
    h = hdr[0].transpose(1, 0, 2).view(np.float16).reshape(T, H, d // 64, 2)
    np.testing.assert_array_equal(h[..., 0], sc)
    np.testing.assert_array_equal(h[..., 1], zr)


def test_encode_flags_out_of_range_slot(ctx128):
    d, H = 128, 1
    x = W.kv_tensor(2, H, d, seed=1, device="cuda")
    view = tq.alloc_view("turbo4_mse", d, H, page_size=4, num_pages=1)
    tq.tq_get_status(ctx128.h)  # clear
    C.encode(ctx128, view, x, is_k=False, slots=torch.tensor([1, 99], device="cuda"))
    st, flags = tq.tq_get_status(ctx128.h)
    assert st == tq.TQ_ERR_INVALID_ARG and flags & 4
    pay, _ = C.read_vectors(view)
    assert pay[0, 0, 1].any() and not pay[0, 0, 0].any()


# ---------------------------------------------------------------------------
# dequantize (on oracle-written codes, so both sides see identical codes)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", TURBO_K + TURBO_V + ["q8_0"])
def test_dequantize_matches_oracle(ctx, fmt):
    d, H, T = ctx.d, 3, 50
    x16 = W.kv_tensor(T, H, d, seed=41, outliers_per_head=2).numpy()
    enc = C.oracle_encode(fmt, x16, ctx.signs, ctx.S)
    view = tq.alloc_view(fmt, d, H, page_size=64, num_pages=1)
    C.write_oracle_codes(view, enc, fmt, np.arange(T))
    out = torch.empty((T, H, d), dtype=torch.float32, device="cuda")
    for inc in (0, 1):
        assert tq.tq_dequantize(ctx.h, view, 0, None, 0, T, inc, out) == tq.TQ_OK
        torch.cuda.synchronize()
        if fmt == "q8_0":
            want = O.q8_0_dequant(*enc)
        else:
            want = O.turbo_dequant(enc, fmt, ctx.signs, ctx.S, include_qjl=bool(inc))
        err = np.abs(out.cpu().numpy() - want).max() / np.abs(want).max()
        assert err < 2e-6, err


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_minmax_round_trip_matches_oracle(ctx128, bits):
    d, H, T = 128, 8, 40
    x = W.kv_tensor(T, H, d, seed=51, device="cuda", outliers_per_head=4)
    view = tq.alloc_view("minmax", d, H, page_size=T, num_pages=1, bits=bits)
    C.encode(ctx128, view, x, is_k=False)
    out = torch.empty((T, H, d), dtype=torch.float32, device="cuda")
    assert tq.tq_dequantize(ctx128.h, view, 0, None, 0, T, 0, out) == tq.TQ_OK
    torch.cuda.synchronize()
    want = O.minmax_dequant(*O.minmax_encode(x.cpu().numpy().astype(np.float32), bits=bits))
    np.testing.assert_allclose(out.cpu().numpy(), want, rtol=1e-6, atol=1e-6)


# ---------------------------------------------------------------------------
# decode attention
# ---------------------------------------------------------------------------

def _oracle_attention(q, kt, vt, tau=0.0, d=128):
    o_full, o_skip = O.decode_attention(q, kt, vt, 1.0 / math.sqrt(d), tau)
    return o_full, o_skip


def test_decode_tiny_workload_end_to_end(ctx128):
    """Single layer, 8 KV heads x 1024 tokens, d 128, 4 outlier channels per head x20,
    K turbo3, V turbo3_mse, 32 query heads (GQA 4): GPU encode + GPU decode.

    Every query head is compared twice, none excluded: (1) the GPU decode of the GPU-encoded
    cache against oracle attention over the codes the GPU stored (read back and dequantised by
    the oracle), which holds whatever the two sides decided inside the 1e-6 band; (2) the GPU
    decode of the oracle's own codes written into the cache against the oracle end to end
    (oracle encode, dequantise, attention)."""
    wl = W.WORKLOADS["tiny-d128-h8-t1024-turbo3"]
    d, H, T, Hq = wl.head_dim, wl.n_kv_heads, wl.ctx, wl.n_q_heads
    G = Hq // H
    k = W.kv_tensor(T, H, d, seed=wl.seed, device="cuda", outliers_per_head=4)
    v = W.kv_tensor(T, H, d, seed=wl.seed + 100, device="cuda", outliers_per_head=4)
    q = W.normal_tensor((1, 1, Hq, d), seed=wl.seed + 200, device="cuda")
    kv = tq.alloc_view("turbo3", d, H, page_size=T, num_pages=1)
    vv = tq.alloc_view("turbo3_mse", d, H, page_size=T, num_pages=1)
    C.encode(ctx128, kv, k, True)
    C.encode(ctx128, vv, v, False)
    out = C.decode(ctx128, q, kv, vv, [T], T)[0, 0].cpu().numpy()
    ek = O.turbo_encode(k.cpu().numpy(), "turbo3", ctx128.signs, ctx128.S)
    ev = O.turbo_encode(v.cpu().numpy(), "turbo3_mse", ctx128.signs, None)
    # codes: indices bit-exact outside the band; signs and rnorm from the GPU's own indices
    kp, kh = C.read_vectors(kv)
    vp, vh = C.read_vectors(vv)
    kp, kh, vp, vh = (a[0].transpose(1, 0, 2) for a in (kp, kh, vp, vh))  # [T, H, bytes]
    C.check_turbo_codes("turbo3", d, kp, kh, ek, S=ctx128.S)
    C.check_turbo_codes("turbo3_mse", d, vp, vh, ev)
    q64 = q[0, 0].cpu().numpy().astype(np.float64)
    for h in range(H):
        sl = slice(h, h + 1)
        want, _ = C.oracle_attention_on_gpu_codes("turbo3", "turbo3_mse", d, kp[:, sl], kh[:, sl], vp[:, sl],
                                                  vh[:, sl], q64[h * G:(h + 1) * G], ctx128.signs, ctx128.S)
        err = C.rel_err_per_head(out[h * G:(h + 1) * G], want)
        assert err.max() < C.ATTN_RTOL, (h, err.max())
    # the oracle's own codes in the same cache: the GPU decode against the oracle end to end
    C.write_oracle_codes(kv, ek, "turbo3", np.arange(T))
    C.write_oracle_codes(vv, ev, "turbo3_mse", np.arange(T))
    out2 = C.decode(ctx128, q, kv, vv, [T], T)[0, 0].cpu().numpy()
    kt = O.turbo_dequant(ek, "turbo3", ctx128.signs, ctx128.S)
    vt = O.turbo_dequant(ev, "turbo3_mse", ctx128.signs, None)
    o_full, _ = _oracle_attention(q64, kt, vt)
    err = C.rel_err_per_head(out2, o_full)
    assert err.max() < C.ATTN_RTOL, err.max()


def _oracle_cache(ctx, kfmt, vfmt, T, H, seed, outliers=0, frac=0.0):
    d = ctx.d
    k16 = W.kv_tensor(T, H, d, seed=seed, outliers_per_head=outliers, outlier_frac=frac).numpy()
    v16 = W.kv_tensor(T, H, d, seed=seed + 1, outliers_per_head=outliers, outlier_frac=frac).numpy()
    ek = C.oracle_encode(kfmt, k16, ctx.signs, ctx.S)
    ev = C.oracle_encode(vfmt, v16, ctx.signs, ctx.S)
    return ek, ev, C.oracle_dequant(kfmt, ek, ctx.signs, ctx.S), C.oracle_dequant(vfmt, ev, ctx.signs, ctx.S)


def _slice_enc(enc, sl):
    if isinstance(enc, tuple):
        return tuple(e[sl] for e in enc)
    return {k: v[sl] for k, v in enc.items()}


@pytest.mark.parametrize("kfmt,vfmt", [("turbo4", "turbo4_mse"), ("turbo2", "turbo2_mse"), ("turbo3", "q8_0"),
                                       ("q8_0", "turbo2_mse"), ("q8_0", "q8_0"), ("turbo3_mse", "turbo3_mse")])
def test_decode_on_oracle_codes(ctx, kfmt, vfmt):
    """Identical codes on both sides: ragged batch (0, 1, 700 tokens and a full page),
    several splits, GQA 4, fp32 and fp16 queries."""
    d, H, G, page = ctx.d, 2, 4, 1024
    lens = [0, 1, 700, page]
    B = len(lens)
    kview = tq.alloc_view(kfmt, d, H, page_size=page, num_pages=B)
    vview = tq.alloc_view(vfmt, d, H, page_size=page, num_pages=B)
    caches = []
    for b, L in enumerate(lens):
        ek, ev, kt, vt = _oracle_cache(ctx, kfmt, vfmt, max(L, 1), H, seed=100 + b, outliers=2)
        C.write_oracle_codes(kview, ek, kfmt, b * page + np.arange(max(L, 1)))
        C.write_oracle_codes(vview, ev, vfmt, b * page + np.arange(max(L, 1)))
        caches.append((kt[:L], vt[:L]))
    for qdt in (torch.float32, torch.float16):
        q = W.normal_tensor((1, B, H * G, d), seed=7, device="cuda").to(qdt)
        out = C.decode(ctx, q, kview, vview, lens, page)
        for b, L in enumerate(lens):
            if L == 0:
                assert torch.all(out[0, b] == 0)
                continue
            o_full, _ = O.decode_attention(q[0, b].float().cpu().numpy().astype(np.float64), caches[b][0],
                                           caches[b][1], 1.0 / math.sqrt(d))
            err = C.rel_err_per_head(out[0, b].cpu().numpy(), o_full)
            assert err.max() < C.ATTN_RTOL, (b, err.max())


MMA_K = ["turbo2", "turbo3", "turbo4", "q8_0"]
MMA_V = ["turbo2_mse", "turbo3_mse", "turbo4_mse", "q8_0"]
_MMA_LENS = [0, 1, 17, 300, 613]
_mma_codes = {}


def _mma_oracle(ctx, fmt, is_k):
    """Oracle codes and dequantised vectors of one role (K or V) for every sequence of
    _MMA_LENS, concatenated; shared by the format pairs of one head_dim."""
    key = (ctx.d, fmt, is_k)
    if key not in _mma_codes:
        T = sum(_MMA_LENS)
        x16 = W.kv_tensor(T, 2, ctx.d, seed=31 if is_k else 37, outlier_frac=0.01).numpy()
        enc = C.oracle_encode(fmt, x16, ctx.signs, ctx.S)
        _mma_codes[key] = (enc, C.oracle_dequant(fmt, enc, ctx.signs, ctx.S))
    return _mma_codes[key]


@pytest.mark.parametrize("G", [4, 8, 16])
@pytest.mark.parametrize("vfmt", MMA_V)
@pytest.mark.parametrize("kfmt", MMA_K)
def test_decode_tensor_core_format_pairs_paged(ctx, kfmt, vfmt, G):
    """Every K x V format pair of the tensor-core decode kernels at head_dim 64/128/256, with
    4 query heads per KV head (high/low fp16 query columns), 8 (two heads per column pair) and 16
    (four query products, two V products; at d 256 two head halves per work item):
    16-token pages in shuffled order, lengths 0, 1, 17, 300, 613 (ragged tiles, several
    256-token splits), Sparse V at 1e-6; identical codes on both sides."""
    d, H, P = ctx.d, 2, 16
    lens = np.array(_MMA_LENS)
    bt, npages = W.shuffled_block_table(lens, P, seed=11, extra_pages=3)
    ek, kt = _mma_oracle(ctx, kfmt, True)
    ev, vt = _mma_oracle(ctx, vfmt, False)
    kview = tq.alloc_view(kfmt, d, H, page_size=P, num_pages=npages)
    vview = tq.alloc_view(vfmt, d, H, page_size=P, num_pages=npages)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    slots = np.concatenate([bt[b, np.arange(L) // P] * P + np.arange(L) % P for b, L in enumerate(lens)])
    C.write_oracle_codes(kview, ek, kfmt, slots)
    C.write_oracle_codes(vview, ev, vfmt, slots)
    q = W.normal_tensor((1, len(lens), H * G, d), seed=13, device="cuda")
    out = C.decode(ctx, q, kview, vview, lens, int(lens.max()), block_table=bt, max_blocks=bt.shape[1], tau=1e-6)
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.all(out[0, b] == 0)
            continue
        sl = slice(starts[b], starts[b] + L)
        o_full, _ = O.decode_attention(q[0, b].cpu().numpy().astype(np.float64), kt[sl], vt[sl], 1.0 / math.sqrt(d))
        err = C.rel_err_per_head(out[0, b].cpu().numpy(), o_full)
        assert err.max() < C.ATTN_RTOL, (b, err.max())


def test_decode_pages_not_a_multiple_of_16_tokens(ctx128):
    """24-token pages in shuffled order (the CUDA-core attention kernel's block-table path), lengths
    0, 5, 24, 100, 333, GQA 4, Sparse V at 1e-6; identical codes on both sides."""
    d, H, G, P = 128, 2, 4, 24
    lens = np.array([0, 5, 24, 100, 333])
    bt, npages = W.shuffled_block_table(lens, P, seed=21, extra_pages=2)
    T = int(lens.sum())
    ek, ev, kt, vt = _oracle_cache(ctx128, "turbo4", "turbo4_mse", T, H, seed=23, frac=0.01)
    kview = tq.alloc_view("turbo4", d, H, page_size=P, num_pages=npages)
    vview = tq.alloc_view("turbo4_mse", d, H, page_size=P, num_pages=npages)
    slots = np.concatenate([bt[b, np.arange(L) // P] * P + np.arange(L) % P for b, L in enumerate(lens)])
    C.write_oracle_codes(kview, ek, "turbo4", slots)
    C.write_oracle_codes(vview, ev, "turbo4_mse", slots)
    q = W.normal_tensor((1, len(lens), H * G, d), seed=25, device="cuda")
    out = C.decode(ctx128, q, kview, vview, lens, int(lens.max()), block_table=bt, max_blocks=bt.shape[1], tau=1e-6)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.all(out[0, b] == 0)
            continue
        sl = slice(starts[b], starts[b] + L)
        o_full, _ = O.decode_attention(q[0, b].cpu().numpy().astype(np.float64), kt[sl], vt[sl], 1.0 / math.sqrt(d))
        assert C.rel_err_per_head(out[0, b].cpu().numpy(), o_full).max() < C.ATTN_RTOL


@pytest.mark.parametrize("G", [1, 3, 6, 8, 9, 12, 16])
def test_decode_gqa_groups(ctx128, G):
    """turbo4 / turbo4_mse, 333 tokens: G 1 and 3 leave column pairs of the high / low query
    layout empty, G 6 leaves two of the second product's pairs empty, G 8 fills both products,
    and G 9, 12, 16 run two launches over the halves of each KV head's query heads (5 + 4, 6 + 6,
    8 + 8)."""
    d, H, T = 128, 2, 333
    ek, ev, kt, vt = _oracle_cache(ctx128, "turbo4", "turbo4_mse", T, H, seed=9, frac=0.01)
    kview = tq.alloc_view("turbo4", d, H, page_size=T, num_pages=1)
    vview = tq.alloc_view("turbo4_mse", d, H, page_size=T, num_pages=1)
    C.write_oracle_codes(kview, ek, "turbo4", np.arange(T))
    C.write_oracle_codes(vview, ev, "turbo4_mse", np.arange(T))
    q = W.normal_tensor((1, 1, H * G, d), seed=8, device="cuda")
    out = C.decode(ctx128, q, kview, vview, [T], T)
    o_full, _ = O.decode_attention(q[0, 0].cpu().numpy().astype(np.float64), kt, vt, 1.0 / math.sqrt(d))
    assert C.rel_err_per_head(out[0, 0].cpu().numpy(), o_full).max() < C.ATTN_RTOL


def test_decode_paged_equals_contiguous_and_layers(ctx128):
    """Shuffled 16-token pages give the same result as a contiguous cache; three layers with
    layer_begin = 1 read the right layers."""
    d, H, Hq, P, B = 128, 4, 16, 16, 3
    lens = np.array([100, 37, 256])
    nl = 2
    max_ctx = int(lens.max())
    bt, npages = W.shuffled_block_table(lens, P, seed=3, extra_pages=5)
    kc = tq.alloc_view("turbo4", d, H, page_size=max_ctx, num_pages=B, n_layers=3)
    vc = tq.alloc_view("turbo4_mse", d, H, page_size=max_ctx, num_pages=B, n_layers=3)
    kp = tq.alloc_view("turbo4", d, H, page_size=P, num_pages=npages, n_layers=3)
    vp = tq.alloc_view("turbo4_mse", d, H, page_size=P, num_pages=npages, n_layers=3)
    inputs = {}
    for l in range(nl):
        for b in range(B):
            L = int(lens[b])
            k = W.kv_tensor(L, H, d, seed=50 + 10 * l + b, device="cuda", outlier_frac=0.01)
            v = W.kv_tensor(L, H, d, seed=70 + 10 * l + b, device="cuda", outlier_frac=0.01)
            inputs[l, b] = (k.cpu().numpy(), v.cpu().numpy())
            t = np.arange(L)
            phys = torch.as_tensor(bt[b, t // P] * P + t % P, dtype=torch.int64, device="cuda")
            for view_k, view_v, slots, sb in ((kc, vc, None, b * max_ctx), (kp, vp, phys, 0)):
                C.encode(ctx128, view_k, k.unsqueeze(0), True, layer_begin=1 + l, slots=slots, slot_begin=sb)
                C.encode(ctx128, view_v, v.unsqueeze(0), False, layer_begin=1 + l, slots=slots, slot_begin=sb)
    q = W.normal_tensor((nl, B, Hq, d), seed=5, device="cuda")
    o_c = C.decode(ctx128, q, kc, vc, lens, max_ctx, layer_begin=1)
    o_p = C.decode(ctx128, q, kp, vp, lens, max_ctx, block_table=bt, max_blocks=bt.shape[1], layer_begin=1)
    torch.testing.assert_close(o_p, o_c, rtol=0, atol=0)
    # and each layer / sequence agrees with the oracle on the GPU's own encoded cache
    for l in range(nl):
        for b in range(B):
            k, v = inputs[l, b]
            kt = O.turbo_dequant(O.turbo_encode(k, "turbo4", ctx128.signs, ctx128.S), "turbo4", ctx128.signs,
                                 ctx128.S)
            vt = O.turbo_dequant(O.turbo_encode(v, "turbo4_mse", ctx128.signs, None), "turbo4_mse",
                                 ctx128.signs, None)
            o, _ = O.decode_attention(q[l, b].cpu().numpy().astype(np.float64), kt, vt, 1 / math.sqrt(d))
            assert C.rel_err_per_head(o_c[l, b].cpu().numpy(), o).max() < C.ATTN_RTOL


def test_decode_sparse_v_needles(ctx128):
    """Peaked softmax (query aligned with 16 needle keys x8): skipping V terms below 1e-6
    stays within the skip bound of the full result and within 2e-3 of the oracle."""
    d, H, Hq, T = 128, 2, 16, 4096
    k, q, pos = W.needle_workload(T, H, Hq, d, seed=4)
    v = W.kv_tensor(T, H, d, seed=5)
    ek = O.q8_0_encode(k.numpy())
    ev = O.turbo_encode(v.numpy(), "turbo2_mse", ctx128.signs, None)
    kview = tq.alloc_view("q8_0", d, H, page_size=T, num_pages=1)
    vview = tq.alloc_view("turbo2_mse", d, H, page_size=T, num_pages=1)
    C.write_oracle_codes(kview, ek, "q8_0", np.arange(T))
    C.write_oracle_codes(vview, ev, "turbo2_mse", np.arange(T))
    kt, vt = O.q8_0_dequant(*ek), O.turbo_dequant(ev, "turbo2_mse", ctx128.signs, None)
    qd = q.reshape(1, 1, Hq, d).cuda()
    o_full, o_skip = O.decode_attention(q.numpy().astype(np.float64), kt, vt, 1 / math.sqrt(d), 1e-6)
    bound = 1e-6 * np.sum(np.linalg.norm(vt, axis=-1), axis=0)  # per KV head
    assert np.all(np.linalg.norm(o_full - o_skip, axis=-1) <= np.repeat(bound, Hq // H))
    for tau in (0.0, 1e-6):
        out = C.decode(ctx128, qd, kview, vview, [T], T, tau=tau)[0, 0].cpu().numpy()
        assert C.rel_err_per_head(out, o_full).max() < C.ATTN_RTOL
        if tau:
            assert np.all(np.linalg.norm(out - o_full, axis=-1) <= np.repeat(bound, Hq // H) + 2e-3 *
                          np.linalg.norm(o_full, axis=-1))


def test_decode_flags_bad_block_table_and_long_sequence(ctx128):
    d, H, P = 128, 1, 16
    kview = tq.alloc_view("turbo4", d, H, page_size=P, num_pages=2)
    vview = tq.alloc_view("turbo4_mse", d, H, page_size=P, num_pages=2)
    q = W.normal_tensor((1, 1, 1, d), seed=1, device="cuda")
    tq.tq_get_status(ctx128.h)
    C.decode(ctx128, q, kview, vview, [32], 32, block_table=[[0, 7]], max_blocks=2)
    st, flags = tq.tq_get_status(ctx128.h)
    assert st == tq.TQ_ERR_INVALID_ARG and flags & 2
    C.decode(ctx128, q, kview, vview, [40], 32, block_table=[[0, 1]], max_blocks=2)
    st, flags = tq.tq_get_status(ctx128.h)
    assert flags & 1


def test_encode_rejects_misaligned_inputs(ctx128):
    d, H, T = 128, 2, 16
    view = tq.alloc_view("turbo4_mse", d, H, page_size=T, num_pages=1)
    x = torch.zeros((T + 1, H, d), dtype=torch.float16, device="cuda")
    ok = tq.tq_encode_kv(ctx128.h, None, None, view, x, 0, 1, T, T * H * d, H * d)
    assert ok == tq.TQ_OK
    # input pointer not 16-byte aligned
    assert tq.tq_encode_kv(ctx128.h, None, None, view, x.data_ptr() + 2, 0, 1, T, T * H * d, H * d) == \
        tq.TQ_ERR_INVALID_ARG
    # token stride not a multiple of 8 elements
    assert tq.tq_encode_kv(ctx128.h, None, None, view, x, 0, 1, T - 1, (T - 1) * (H * d + 1), H * d + 1) == \
        tq.TQ_ERR_INVALID_ARG
    torch.cuda.synchronize()


def test_decode_rejects_bad_arguments(ctx128):
    d = 128
    kview = tq.alloc_view("turbo4", d, 2, page_size=64, num_pages=1)
    vview = tq.alloc_view("turbo4_mse", d, 2, page_size=64, num_pages=1)
    kmse = tq.alloc_view("turbo4", d, 2, page_size=64, num_pages=1)
    q = torch.zeros((1, 1, 3, d), device="cuda")
    out = torch.empty_like(q)
    sl = torch.tensor([10], dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    # 3 query heads over 2 KV heads
    assert tq.tq_decode_attention(ctx128.h, q, 0, 1, 1, 3, kview, vview, 0, sl, 64, None, 0, 1.0, 0.0, ws,
                                  ws.numel(), out) == tq.TQ_ERR_UNSUPPORTED
    q = torch.zeros((1, 1, 4, d), device="cuda")
    out = torch.empty_like(q)
    # V with a QJL format
    assert tq.tq_decode_attention(ctx128.h, q, 0, 1, 1, 4, kview, kmse, 0, sl, 64, None, 0, 1.0, 0.0, ws,
                                  ws.numel(), out) == tq.TQ_ERR_UNSUPPORTED
    # workspace too small
    assert tq.tq_decode_attention(ctx128.h, q, 0, 1, 1, 4, kview, vview, 0, sl, 64, None, 0, 1.0, 0.0, ws, 16,
                                  out) == tq.TQ_ERR_WORKSPACE
    # context capacity exceeded without a block table
    assert tq.tq_decode_attention(ctx128.h, q, 0, 1, 1, 4, kview, vview, 0, sl, 65, None, 0, 1.0, 0.0, ws,
                                  ws.numel(), out) == tq.TQ_ERR_INVALID_ARG


def test_per_layer_views_boundary_v_in_one_call(ctx128):
    """A per-layer format table: 6 layers, K turbo4 in one view; V q8_0 on the first and the last
    layer (a 2-layer view) and turbo2_mse between (a 4-layer view).  One tq_encode_kv_layers call
    and one tq_decode_attention_layers call; the result equals the per-group calls bit for bit (the
    same 256-token splits) and every query head matches oracle attention over the stored codes."""
    d, H, Hq, T, L = 128, 2, 8, 700, 6
    G = Hq // H
    kview = tq.alloc_view("turbo4", d, H, page_size=T, num_pages=1, n_layers=L)
    vb = tq.alloc_view("q8_0", d, H, page_size=T, num_pages=1, n_layers=2)
    vm = tq.alloc_view("turbo2_mse", d, H, page_size=T, num_pages=1, n_layers=4)
    v_views = [vb, vm, vm, vm, vm, vb]
    v_layers = [0, 0, 1, 2, 3, 1]
    k = torch.stack([W.kv_tensor(T, H, d, seed=90 + l, device="cuda", outlier_frac=0.01) for l in range(L)])
    v = torch.stack([W.kv_tensor(T, H, d, seed=190 + l, device="cuda", outlier_frac=0.01) for l in range(L)])
    st = tq.tq_encode_kv_layers(ctx128.h, [kview] * L, list(range(L)), v_views, v_layers, L, k, v, T, T * H * d, H * d)
    assert st == tq.TQ_OK, tq.tq_status_string(st)
    q = W.normal_tensor((L, 1, Hq, d), seed=91, device="cuda")
    lens = torch.tensor([T], dtype=torch.int32, device="cuda")
    nbytes = tq.tq_decode_workspace_bytes(ctx128.h, L, 1, Hq, T)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((L, 1, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
    st = tq.tq_decode_attention_layers(ctx128.h, q, 0, L, 1, Hq, [kview] * L, list(range(L)), v_views, v_layers,
                                       lens, T, None, 0, 1 / math.sqrt(d), 1e-6, ws, nbytes, out)
    assert st == tq.TQ_OK, tq.tq_status_string(st)
    # the same layers decoded group by group with the plain entry point
    ref = torch.empty_like(out)
    for (l0, n, vv, vl0) in ((0, 1, vb, 0), (1, 4, vm, 0), (5, 1, vb, 1)):
        o = torch.empty((n, 1, Hq, d), dtype=torch.float32, device="cuda")
        # layer l0 of the K view and layer vl0 of the V view: views advanced by whole layers
        kvec = H * T
        ksub = tq.CacheView("turbo4", d, H, T, 1, n,
                            kview.payload[l0 * kvec * 64:], kview.header[l0 * kvec * 4:])
        pb, hb = tq.tq_payload_bytes(vv.fmt, d), tq.tq_header_bytes(vv.fmt, d)
        vsub = tq.CacheView(vv.fmt, d, H, T, 1, n, vv.payload[vl0 * kvec * pb:], vv.header[vl0 * kvec * hb:])
        ws2 = torch.empty(tq.tq_decode_workspace_bytes(ctx128.h, n, 1, Hq, T), dtype=torch.uint8, device="cuda")
        assert tq.tq_decode_attention(ctx128.h, q[l0:l0 + n].contiguous(), 0, n, 1, Hq, ksub, vsub, 0, lens, T, None,
                                      0, 1 / math.sqrt(d), 1e-6, ws2, ws2.numel(), o) == tq.TQ_OK
        ref[l0:l0 + n] = o
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # every head against the oracle over the codes stored in each layer's views
    for l in range(L):
        vv, vl = v_views[l], v_layers[l]
        kp, kh = C.read_vectors(kview, l)
        vp, vh = C.read_vectors(vv, vl)
        for h in range(H):
            sl = (0, h)  # page 0, KV head h: [T, bytes]
            want, _ = C.oracle_attention_on_gpu_codes("turbo4", vv.fmt, d, kp[sl][:, None], kh[sl][:, None],
                                                      vp[sl][:, None], vh[sl][:, None],
                                                      q[l, 0, h * G:(h + 1) * G].cpu().numpy(), ctx128.signs,
                                                      ctx128.S)
            assert C.rel_err_per_head(out[l, 0, h * G:(h + 1) * G].cpu().numpy(), want).max() < C.ATTN_RTOL, (l, h)
