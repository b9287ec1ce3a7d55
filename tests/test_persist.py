"""Persistence of a compressed cache (tq_cache_save / tq_cache_file_info / tq_cache_load).

CPU tests use host arrays (host_memory = 1): the file round-trips every byte, its header is the
documented magic line plus one JSON object, and every mismatch (geometry, tables, size, a flipped
data byte, trailing bytes) is rejected.  The GPU test encodes a cache with the library, saves it,
loads it into a fresh view and checks that decode attention over the loaded cache equals decode
attention over the original bit for bit.
"""
import json
import math
import os

import numpy as np
import pytest

tq = pytest.importorskip("kv_cache_quantization_turbo_gb300.tq", reason="libtq.so not built")
from kv_cache_quantization_turbo_gb300 import workloads as W  # noqa: E402


def _host_view(fmt, d, H, P, pages, L, bits=0, seed=0):
    pb, hb = tq.tq_payload_bytes(fmt, d, bits), tq.tq_header_bytes(fmt, d, bits)
    n = L * pages * H * P
    rng = np.random.default_rng(seed)
    pay = rng.integers(0, 256, n * pb, dtype=np.uint8)
    hdr = rng.integers(0, 256, n * hb, dtype=np.uint8)
    return tq.CacheView(fmt, d, H, P, pages, L, pay, hdr, bits)


def _empty_like(v):
    return tq.CacheView(v.fmt, v.head_dim, v.n_kv_heads, v.page_size, v.num_pages, v.n_layers,
                        np.zeros_like(v.payload), np.zeros_like(v.header), v.bits)


@pytest.mark.parametrize("fmt,bits", [("turbo4", 0), ("turbo3_mse", 0), ("q8_0", 0), ("minmax", 3)])
def test_host_round_trip_and_header(tmp_path, fmt, bits):
    v = _host_view(fmt, 128, 3, 16, 5, 2, bits, seed=1)
    path = str(tmp_path / "cache.tq")
    assert tq.tq_cache_save(None, v, path) == tq.TQ_OK
    assert not os.path.exists(path + ".partial")
    raw = open(path, "rb").read()
    assert raw[:9] == b"TQCACHE1\n"
    line = raw[9:raw.index(b"\n", 9)]
    meta = json.loads(line)  # the metadata record is plain JSON
    assert meta["format"] == fmt and meta["head_dim"] == 128 and meta["n_kv_heads"] == 3
    assert meta["page_size"] == 16 and meta["num_pages"] == 5 and meta["n_layers"] == 2
    assert meta["bits"] == bits and meta["payload_bytes"] == v.payload.size and meta["header_bytes"] == v.header.size
    off = (9 + len(line) + 1 + 4095) // 4096 * 4096
    assert not any(raw[9 + len(line) + 1:off])  # zero padding
    np.testing.assert_array_equal(np.frombuffer(raw[off:off + v.payload.size], np.uint8), v.payload)
    np.testing.assert_array_equal(np.frombuffer(raw[off + v.payload.size:], np.uint8), v.header)
    st, geo, th = tq.tq_cache_file_info(path)
    assert st == tq.TQ_OK and th == 0
    assert geo == {"format": tq.FORMATS[fmt], "head_dim": 128, "n_kv_heads": 3, "page_size": 16, "num_pages": 5,
                   "n_layers": 2, "bits": bits}
    w = _empty_like(v)
    assert tq.tq_cache_load(None, w, path) == tq.TQ_OK
    np.testing.assert_array_equal(w.payload, v.payload)
    np.testing.assert_array_equal(w.header, v.header)


def test_host_load_rejects_mismatches(tmp_path):
    v = _host_view("turbo4", 64, 2, 32, 3, 1, seed=2)
    path = str(tmp_path / "c.tq")
    assert tq.tq_cache_save(None, v, path) == tq.TQ_OK
    for change in ({"num_pages": 4}, {"page_size": 16}, {"n_kv_heads": 1}, {"n_layers": 2}):
        kw = dict(fmt="turbo4", d=64, H=2, P=32, pages=3, L=1)
        kw.update({"pages" if k == "num_pages" else "P" if k == "page_size" else "H" if k == "n_kv_heads" else "L": x
                   for k, x in change.items()})
        w = _host_view(**kw)
        assert tq.tq_cache_load(None, w, path) == tq.TQ_ERR_INVALID_ARG, change
    w = _host_view("turbo4_mse", 64, 2, 32, 3, 1)  # another format
    assert tq.tq_cache_load(None, w, path) == tq.TQ_ERR_INVALID_ARG
    raw = bytearray(open(path, "rb").read())
    bad = str(tmp_path / "flipped.tq")
    raw[-5] ^= 0x10  # one flipped bit in the header array
    open(bad, "wb").write(raw)
    assert tq.tq_cache_load(None, _empty_like(v), bad) == tq.TQ_ERR_INVALID_ARG
    open(bad, "wb").write(bytes(raw[:-1]))  # truncated
    assert tq.tq_cache_load(None, _empty_like(v), bad) == tq.TQ_ERR_INVALID_ARG
    open(bad, "wb").write(bytes(open(path, "rb").read()) + b"\0")  # trailing byte
    assert tq.tq_cache_load(None, _empty_like(v), bad) == tq.TQ_ERR_INVALID_ARG
    open(bad, "wb").write(b"not a cache\n")
    assert tq.tq_cache_file_info(bad)[0] == tq.TQ_ERR_INVALID_ARG
    assert tq.tq_cache_file_info(str(tmp_path / "missing.tq"))[0] == tq.TQ_ERR_INVALID_ARG


@pytest.mark.gpu
def test_decode_of_a_loaded_cache_equals_the_original(tmp_path):
    import torch

    assert torch.cuda.is_available()
    d, H, Hq, T, L = 128, 4, 16, 1000, 2
    ctx = tq.tq_context_create(d, 1, 2, W.wht_signs(1, d), W.qjl_matrix(2, d))
    other = tq.tq_context_create(d, 1, 3)  # another QJL matrix
    try:
        kv = tq.alloc_view("turbo4", d, H, page_size=T, num_pages=1, n_layers=L)
        vv = tq.alloc_view("turbo3_mse", d, H, page_size=T, num_pages=1, n_layers=L)
        for l in range(L):
            k = W.kv_tensor(T, H, d, seed=60 + l, device="cuda", outlier_frac=0.01)
            v = W.kv_tensor(T, H, d, seed=70 + l, device="cuda", outlier_frac=0.01)
            assert tq.tq_encode_kv(ctx, kv, k, vv, v, l, 1, T, T * H * d, H * d) == tq.TQ_OK
        pk, pv = str(tmp_path / "k.tq"), str(tmp_path / "v.tq")
        assert tq.tq_cache_save(ctx, kv, pk) == tq.TQ_OK and tq.tq_cache_save(ctx, vv, pv) == tq.TQ_OK
        st, geo, th = tq.tq_cache_file_info(pk)
        assert st == tq.TQ_OK and th == tq.tq_context_tables_hash(ctx) != tq.tq_context_tables_hash(other)
        kl = tq.alloc_view("turbo4", d, H, page_size=T, num_pages=1, n_layers=L)
        vl = tq.alloc_view("turbo3_mse", d, H, page_size=T, num_pages=1, n_layers=L)
        assert tq.tq_cache_load(other, kl, pk) == tq.TQ_ERR_INVALID_ARG  # codes made with other tables
        assert tq.tq_cache_load(ctx, kl, pk) == tq.TQ_OK and tq.tq_cache_load(ctx, vl, pv) == tq.TQ_OK
        assert torch.equal(kl.payload, kv.payload) and torch.equal(vl.header, vv.header)
        q = W.normal_tensor((L, 1, Hq, d), seed=80, device="cuda")
        lens = torch.tensor([T], dtype=torch.int32, device="cuda")
        nbytes = tq.tq_decode_workspace_bytes(ctx, L, 1, Hq, T)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        outs = []
        for kview, vview in ((kv, vv), (kl, vl)):
            out = torch.empty((L, 1, Hq, d), dtype=torch.float32, device="cuda")
            assert tq.tq_decode_attention(ctx, q, 0, L, 1, Hq, kview, vview, 0, lens, T, None, 0, 1 / math.sqrt(d),
                                          1e-6, ws, nbytes, out) == tq.TQ_OK
            outs.append(out)
        torch.cuda.synchronize()
        assert torch.equal(outs[0], outs[1])
    finally:
        tq.tq_context_destroy(ctx)
        tq.tq_context_destroy(other)
