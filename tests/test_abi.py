"""The C ABI without a GPU: the library loads, exports every declared symbol, and its
host-only functions (sizes, codebook, default random tables, argument checks) behave."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle import tq_oracle as O

tq = pytest.importorskip("kv_cache_quantization_turbo_gb300.tq", reason="libtq.so not built")
from kv_cache_quantization_turbo_gb300 import workloads as W  # noqa: E402
from _layout import code_bits  # noqa: E402


def _declared():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    lib = ctypes.CDLL(tq.LIB_PATH)
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n
    # and the binding wraps each of them under the same name
    assert set(names) <= set(tq.EXPORTED)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_sizes_follow_the_documented_layout(d):
    for fmt in ("turbo2", "turbo3", "turbo4", "turbo2_mse", "turbo3_mse", "turbo4_mse"):
        w = code_bits(fmt)
        assert tq.tq_payload_bytes(fmt, d) == d * w // 8
        assert tq.tq_header_bytes(fmt, d) == (4 if not fmt.endswith("_mse") else 2)
        # payload bits per element match the pages' format table
        assert tq.tq_payload_bytes(fmt, d) * 8 // d == O.payload_bits_per_element(fmt)
    assert tq.tq_payload_bytes("q8_0", d) == d and tq.tq_header_bytes("q8_0", d) == d // 16
    for b in (2, 3, 4):
        assert tq.tq_payload_bytes("minmax", d, b) == d * b // 8
        assert tq.tq_header_bytes("minmax", d, b) == d // 16
    assert tq.tq_payload_bytes("minmax", d, 5) == 0
    assert tq.tq_payload_bytes("turbo4", 96) == 0 and tq.tq_payload_bytes("turbo4", 512) == 0
    # d=128 compressed bytes per vector: 68 (turbo4 K) + 50 (turbo4 V) = 118
    if d == 128:
        assert tq.tq_vector_bytes("turbo4", d) + tq.tq_vector_bytes("turbo4_mse", d) == 118


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_library_codebook_equals_oracle(bits, d):
    c, b = tq.tq_codebook_build(bits, d)
    oc, ob = O.codebook(bits, d)
    # independent fp64 Lloyd iterations: same fixed point, equal after fp32 rounding
    np.testing.assert_array_equal(c.astype(np.float64), oc)
    np.testing.assert_array_equal(b.astype(np.float64), ob)


def test_codebook_rejects_bad_args():
    f = np.zeros(16, np.float32)
    assert tq._lib.tq_codebook_build(0, 128, f.ctypes.data, f.ctypes.data) == tq.TQ_ERR_INVALID_ARG
    assert tq._lib.tq_codebook_build(5, 128, f.ctypes.data, f.ctypes.data) == tq.TQ_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [64, 128, 256])
def test_default_tables_equal_the_input_generator(d):
    np.testing.assert_array_equal(tq.tq_signs_generate(1, d), W.wht_signs(1, d))
    S_lib = tq.tq_qjl_matrix_generate(2, d)
    S_gen = W.qjl_matrix(2, d)
    ulp = np.abs(S_lib.view(np.int32).astype(np.int64) - S_gen.view(np.int32).astype(np.int64))
    assert ulp.max() <= 1 and np.count_nonzero(ulp) <= 4  # libm vs numpy transcendental rounding


def test_status_strings_and_null_handles():
    assert tq.tq_status_string(0) == "ok"
    assert tq.tq_format_name("turbo4_mse") == "turbo4_mse"
    assert tq._lib.tq_encode_kv(None, None, None, None, None, 0, 1, 1, 0, 0, None, 0, None) == tq.TQ_ERR_INVALID_ARG
    assert tq._lib.tq_dequantize(None, None, 0, None, 0, 1, 0, None, None) == tq.TQ_ERR_INVALID_ARG
    assert tq._lib.tq_decode_workspace_bytes(None, 1, 1, 1, 1) == 0
    assert tq._lib.tq_context_destroy(None) == tq.TQ_ERR_INVALID_ARG


def test_context_rejects_unsupported_dim_before_touching_a_device():
    out = ctypes.c_void_p()
    assert tq._lib.tq_context_create(96, 1, 2, None, None, ctypes.byref(out)) == tq.TQ_ERR_UNSUPPORTED
    bad = np.array([1, 0] * 32, np.int8)
    st = tq._lib.tq_context_create(64, 1, 2, bad.ctypes.data, None, ctypes.byref(out))
    assert st == tq.TQ_ERR_INVALID_ARG


def test_layout_pack_unpack_round_trip():
    from _layout import pack_codes, unpack_codes
    rng = np.random.default_rng(0)
    for w in (1, 2, 3, 4):
        for d in (64, 128, 256):
            c = rng.integers(0, 1 << w, size=(7, d))
            p = pack_codes(c, w)
            assert p.shape == (7, d * w // 8)
            np.testing.assert_array_equal(unpack_codes(p, d, w), c)
    # coordinate i at bit offset w*i, little endian: codes 1,2,3,... at w=4 -> bytes 0x21, 0x43
    assert list(pack_codes(np.array([[1, 2, 3, 4] + [0] * 60]), 4)[0, :2]) == [0x21, 0x43]
