"""Shared helpers of the GPU parity tests: contexts, encoding through the C ABI,
reading caches back, and the parity rules.

Parity rules (stated by the method's acceptance criteria):
  * indices and QJL signs match the oracle bit-exactly except coordinates whose
    fp64 value lies within 1e-6 of a decision boundary (or of 0 for the sign);
    those are counted and must be <= 1e-4 of the elements;
  * fp16 headers within 1 ulp;
  * attention outputs within a relative error of 2e-3 per query head.
"""
import math

import numpy as np
import torch

from kv_cache_quantization_turbo_gb300 import tq
from kv_cache_quantization_turbo_gb300 import workloads as W
from oracle import tq_oracle as O
from _layout import code_bits, header_halves, split_turbo, unpack_codes, pack_codes, join_turbo

BAND = 1e-6
BAND_FRACTION = 1e-4
ATTN_RTOL = 2e-3


def require_cuda():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"


class Ctx:
    """A library context whose tables come from the shared seeded generators."""

    def __init__(self, d, wht_seed=1, qjl_seed=2):
        self.d = d
        self.signs = W.wht_signs(wht_seed, d)
        self.S = W.qjl_matrix(qjl_seed, d)
        self.h = tq.tq_context_create(d, wht_seed, qjl_seed, self.signs, self.S)

    def close(self):
        tq.tq_context_destroy(self.h)


def encode(ctx, view, x, is_k, layer_begin=0, slots=None, slot_begin=0, stream=None):
    """x: fp16 cuda [L, T, H, d] or [T, H, d]."""
    if x.dim() == 3:
        x = x.unsqueeze(0)
    L, T, H, d = x.shape
    x = x.contiguous()
    args = (view, x, None, None) if is_k else (None, None, view, x)
    st = tq.tq_encode_kv(ctx.h, *args, layer_begin, L, T, T * H * d, H * d, slots, slot_begin, stream)
    assert st == tq.TQ_OK, tq.tq_status_string(st)


def read_vectors(view, layer=0):
    """Payload and header bytes of a view's layer as numpy [num_pages, H, page_size, bytes]."""
    torch.cuda.synchronize()
    pb = tq.tq_payload_bytes(view.fmt, view.head_dim, view.bits)
    hb = tq.tq_header_bytes(view.fmt, view.head_dim, view.bits)
    n = view.num_pages * view.n_kv_heads * view.page_size
    pay = view.payload.view(view.n_layers, n, pb)[layer].cpu().numpy()
    hdr = view.header.view(view.n_layers, n, hb)[layer].cpu().numpy()
    shp = (view.num_pages, view.n_kv_heads, view.page_size)
    return pay.reshape(shp + (pb,)), hdr.reshape(shp + (hb,))


def slot_major(arr, slots, page_size):
    """[pages, H, page_size, ...] -> [len(slots), H, ...] for the given slot ids."""
    slots = np.asarray(slots)
    return arr[slots // page_size, :, slots % page_size]


def near_boundary(y, boundaries):
    return np.min(np.abs(y[..., None] - boundaries), axis=-1) < BAND


def check_turbo_codes(fmt, d, gpu_pay, gpu_hdr, enc, exact=False, band_limit=True, S=None):
    """Bit-exact comparison with the band exclusion; returns counts for reporting.

    Indices are compared with the oracle's.  QJL signs and rnorm (K formats, S required) are
    compared with the oracle's stage 2 run on the indices the GPU stored (O.qjl_stage): where the
    two sides decided an index differently inside the band, the residual differs, and every sign
    and the rnorm of that vector are still checked against what the GPU's own index implies.
    exact=True: no mismatch at all (inputs whose coordinates are exactly zero on both sides, so
    the tie rule decides identically).  band_limit=False: the band-population limit, a property
    of random data, is not applied (inputs constructed to put many coordinates on a boundary)."""
    bits, has_qjl = O.TURBO_FORMATS[fmt]
    codes = unpack_codes(gpu_pay, d, code_bits(fmt))
    idx, sigma = split_turbo(codes, fmt)
    _, bnd = O.codebook(bits, d)
    band = near_boundary(enc["y"], bnd)
    mism = idx != enc["idx"]
    n_el = idx.size
    if exact:
        assert not mism.any(), f"{int(mism.sum())} index mismatches"
    else:
        assert np.all(band[mism]), f"{int((mism & ~band).sum())} index mismatches outside the 1e-6 band"
        if band_limit:
            assert band.sum() <= max(BAND_FRACTION * n_el, 3), f"band too populated: {band.sum()} of {n_el}"
    hdr = header_halves(gpu_hdr, 2 if has_qjl else 1)
    from _layout import f16_ulp_diff
    assert f16_ulp_diff(hdr[..., 0], enc["n16"]).max() <= 1
    out = {"idx_mismatch": int(mism.sum()), "band": int(band.sum()), "elements": n_el,
           "vectors_with_band_index": int(mism.any(axis=-1).sum())}
    if has_qjl:
        assert S is not None, "the QJL check needs the projection matrix"
        st = O.qjl_stage(enc["y"], enc["n"], idx, bits, S)
        sband = np.abs(st["proj"]) < BAND
        smism = sigma != st["sigma"]
        if exact:
            assert not smism.any(), f"{int(smism.sum())} sign mismatches"
        else:
            assert np.all(sband[smism]), f"{int((smism & ~sband).sum())} sign mismatches outside the band"
            if band_limit:
                assert sband.sum() <= max(BAND_FRACTION * n_el, 3), f"sign band too populated: {sband.sum()}"
        assert f16_ulp_diff(hdr[..., 1], st["rnorm16"]).max() <= 1
        out["sigma_mismatch"] = int(smism.sum())
    return out


def gpu_codes(fmt, d, gpu_pay, gpu_hdr):
    """The stored fields of GPU-written vectors in the oracle's form, so that the oracle can
    dequantise the GPU's own codes: turbo {"idx", "n16"[, "sigma", "rnorm16"]}; q8_0 (q, delta16)."""
    if fmt == "q8_0":
        return gpu_pay.view(np.int8), gpu_hdr.view(np.float16)
    bits, has_qjl = O.TURBO_FORMATS[fmt]
    idx, sigma = split_turbo(unpack_codes(gpu_pay, d, code_bits(fmt)), fmt)
    hdr = header_halves(gpu_hdr, 2 if has_qjl else 1)
    enc = {"idx": idx, "n16": hdr[..., 0].copy()}
    if has_qjl:
        enc.update({"sigma": sigma, "rnorm16": hdr[..., 1].copy()})
    return enc


def write_oracle_codes(view, enc, fmt, slots, layer=0, head=None):
    """Packs oracle-encoded vectors [n_slots, H, ...] into a view at the given slots;
    with head=h, enc holds one head ([n_slots, 1, ...]) written to KV head h only."""
    torch.cuda.synchronize()
    d, H, P = view.head_dim, view.n_kv_heads, view.page_size
    pb = tq.tq_payload_bytes(fmt, d)
    hb = tq.tq_header_bytes(fmt, d)
    n = view.num_pages * H * P
    pay = view.payload.view(view.n_layers, n, pb)[layer].cpu().numpy().reshape(view.num_pages, H, P, pb)
    hdr = view.header.view(view.n_layers, n, hb)[layer].cpu().numpy().reshape(view.num_pages, H, P, hb)
    slots = np.asarray(slots)
    hs = slice(None) if head is None else slice(head, head + 1)
    if fmt == "q8_0":
        q, dl = enc
        pay[slots // P, hs, slots % P] = q.view(np.uint8)
        hdr[slots // P, hs, slots % P] = dl.astype(np.float16).view(np.uint8).reshape(dl.shape[:-1] + (-1,))
    else:
        bits, has_qjl = O.TURBO_FORMATS[fmt]
        codes = join_turbo(enc["idx"], enc.get("sigma"), fmt)
        pay[slots // P, hs, slots % P] = pack_codes(codes, code_bits(fmt))
        if has_qjl:
            h = np.stack([enc["n16"], enc["rnorm16"]], axis=-1).astype(np.float16)
        else:
            h = enc["n16"][..., None].astype(np.float16)
        hdr[slots // P, hs, slots % P] = h.view(np.uint8)
    view.payload.view(view.n_layers, n * pb)[layer].copy_(torch.from_numpy(pay.reshape(-1)))
    view.header.view(view.n_layers, n * hb)[layer].copy_(torch.from_numpy(hdr.reshape(-1)))


def oracle_dequant(fmt, enc, signs, S):
    if fmt == "q8_0":
        return O.q8_0_dequant(*enc)
    return O.turbo_dequant(enc, fmt, signs, S)


def oracle_encode(fmt, x16, signs, S):
    if fmt == "q8_0":
        return O.q8_0_encode(x16)
    return O.turbo_encode(x16, fmt, signs, S)


def decode(ctx, q, k_view, v_view, seq_lens, max_ctx, block_table=None, max_blocks=0, layer_begin=0,
           scale=None, tau=0.0, n_layers=1):
    """q: cuda [L, B, Hq, d] fp32/fp16 -> out [L, B, Hq, d] fp32."""
    L, B, Hq, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    nbytes = tq.tq_decode_workspace_bytes(ctx.h, L, B, Hq, max_ctx)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((L, B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
    sl = torch.as_tensor(np.asarray(seq_lens, dtype=np.int32), device="cuda")
    bt = None if block_table is None else torch.as_tensor(np.asarray(block_table, np.int32), device="cuda")
    st = tq.tq_decode_attention(ctx.h, q.contiguous(), int(q.dtype == torch.float16), L, B, Hq, k_view, v_view,
                                layer_begin, sl, max_ctx, bt, max_blocks, scale, tau, ws, nbytes, out)
    assert st == tq.TQ_OK, tq.tq_status_string(st)
    torch.cuda.synchronize()
    return out


def rel_err_per_head(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    num = np.linalg.norm(got - want, axis=-1)
    den = np.maximum(np.linalg.norm(want, axis=-1), 1e-30)
    return num / den


def oracle_attention_on_gpu_codes(kfmt, vfmt, d, kpay, khdr, vpay, vhdr, q_rows, signs, S, tau=0.0):
    """Oracle attention (fp64) over the codes a GPU stored for one KV head's tokens:
    kpay/khdr/vpay/vhdr [T, 1, bytes] read back from the caches, dequantised by the oracle;
    q_rows [G, d].  Returns (o_full, o_skip) [G, d]."""
    kt = oracle_dequant(kfmt, gpu_codes(kfmt, d, kpay, khdr), signs, S)
    vt = oracle_dequant(vfmt, gpu_codes(vfmt, d, vpay, vhdr), signs, S)
    return O.decode_attention(np.asarray(q_rows, np.float64), kt, vt, 1.0 / math.sqrt(d), tau)
