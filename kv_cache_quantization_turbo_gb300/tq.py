"""ctypes binding of libtq.so (include/tq.h): argument marshalling only.

Every function keeps the C name.  Device buffers are passed as torch tensors
(their data_ptr()) or raw integer addresses; streams as torch.cuda.Stream or
raw handles.  The compute runs in the library's CUDA kernels; importing this
module without the built library raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtq.so")

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_WORKSPACE, TQ_ERR_CUDA, TQ_ERR_OOM = range(6)

FORMATS = {
    "turbo2": 0, "turbo3": 1, "turbo4": 2,
    "turbo2_mse": 3, "turbo3_mse": 4, "turbo4_mse": 5,
    "q8_0": 6, "minmax": 7,
}

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with kv_cache_quantization_turbo_gb300.build.build()")
_lib = ctypes.CDLL(LIB_PATH)


class tq_cache_view(ctypes.Structure):
    _fields_ = [
        ("format", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int64), ("n_layers", ctypes.c_int32),
        ("bits", ctypes.c_int32), ("payload", ctypes.c_void_p), ("header", ctypes.c_void_p),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int
_U32 = ctypes.c_uint32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_VP = ctypes.POINTER(tq_cache_view)

_SIGS = {
    "tq_status_string": (ctypes.c_char_p, [_I]),
    "tq_format_name": (ctypes.c_char_p, [_I]),
    "tq_payload_bytes": (_SZ, [_I, _I, _I]),
    "tq_header_bytes": (_SZ, [_I, _I, _I]),
    "tq_vector_bytes": (_SZ, [_I, _I, _I]),
    "tq_codebook_build": (_I, [_I, _I, _P, _P]),
    "tq_signs_generate": (_I, [_U32, _I, _P]),
    "tq_qjl_matrix_generate": (_I, [_U32, _I, _P]),
    "tq_context_create": (_I, [_I, _U32, _U32, _P, _P, ctypes.POINTER(_P)]),
    "tq_context_destroy": (_I, [_P]),
    "tq_context_get_tables": (_I, [_P, _P, _P, _P, _P]),
    "tq_get_status": (_I, [_P, ctypes.POINTER(_U32)]),
    "tq_encode_kv": (_I, [_P, _VP, _P, _VP, _P, _I, _I, _I, _I64, _I64, _P, _I64, _P]),
    "tq_decode_workspace_bytes": (_SZ, [_P, _I, _I, _I, _I]),
    "tq_decode_attention": (_I, [_P, _P, _I, _I, _I, _I, _VP, _VP, _I, _P, _I, _P, _I, _F, _F, _P, _SZ,
                                 _P, _P]),
    "tq_dequantize": (_I, [_P, _VP, _I, _P, _I64, _I, _I, _P, _P]),
    "tq_decode_attention_static": (_I, [_P, _P, _I, _I, _I, _I, _VP, _VP, _I, _P, _I, _P, _I, _F, _F, _P, _P]),
    "tq_encode_kv_layers": (_I, [_P, _VP, _P, _VP, _P, _I, _P, _P, _I, _I64, _I64, _P, _I64, _P]),
    "tq_decode_attention_layers": (_I, [_P, _P, _I, _I, _I, _I, _VP, _P, _VP, _P, _P, _I, _P, _I, _F, _F, _P, _SZ,
                                        _P, _P]),
    "tq_prefill_workspace_bytes": (_SZ, [_P, _I, _I]),
    "tq_prefill_attention": (_I, [_P, _P, _I, _I, _I, _VP, _VP, _I, _I, _P, _I, _I, _F, _P, _SZ, _P, _P]),
    "tq_context_tables_hash": (_I, [_P, ctypes.POINTER(ctypes.c_uint64)]),
    "tq_cache_save": (_I, [_P, _VP, _I, ctypes.c_char_p]),
    "tq_cache_file_info": (_I, [ctypes.c_char_p, _VP, ctypes.POINTER(ctypes.c_uint64)]),
    "tq_cache_load": (_I, [_P, _VP, _I, ctypes.c_char_p]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


class TQError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {tq_status_string(status)} ({status})")
        self.status = status


def _check(status: int, what: str) -> int:
    if status != TQ_OK:
        raise TQError(status, what)
    return status


def _ptr(x) -> int | None:
    """Device/host address of a tensor, an ndarray, an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(type(x))


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _fmt(f) -> int:
    return FORMATS[f] if isinstance(f, str) else int(f)


# ---- pure host functions ----

def tq_status_string(status: int) -> str:
    return _lib.tq_status_string(status).decode()


def tq_format_name(fmt) -> str:
    return _lib.tq_format_name(_fmt(fmt)).decode()


def tq_payload_bytes(fmt, head_dim: int, bits: int = 0) -> int:
    return _lib.tq_payload_bytes(_fmt(fmt), head_dim, bits)


def tq_header_bytes(fmt, head_dim: int, bits: int = 0) -> int:
    return _lib.tq_header_bytes(_fmt(fmt), head_dim, bits)


def tq_vector_bytes(fmt, head_dim: int, bits: int = 0) -> int:
    return _lib.tq_vector_bytes(_fmt(fmt), head_dim, bits)


def tq_codebook_build(bits: int, head_dim: int):
    """Returns (centroids, boundaries) as numpy float32 arrays."""
    import numpy as np

    c = np.zeros(1 << bits, np.float32)
    b = np.zeros(max((1 << bits) - 1, 1), np.float32)
    _check(_lib.tq_codebook_build(bits, head_dim, c.ctypes.data, b.ctypes.data), "tq_codebook_build")
    return c, b[: (1 << bits) - 1]


def tq_signs_generate(seed: int, head_dim: int):
    import numpy as np

    s = np.zeros(head_dim, np.int8)
    _check(_lib.tq_signs_generate(seed, head_dim, s.ctypes.data), "tq_signs_generate")
    return s


def tq_qjl_matrix_generate(seed: int, head_dim: int):
    import numpy as np

    S = np.zeros((head_dim, head_dim), np.float32)
    _check(_lib.tq_qjl_matrix_generate(seed, head_dim, S.ctypes.data), "tq_qjl_matrix_generate")
    return S


# ---- context ----

def tq_context_create(head_dim: int, wht_seed: int = 1, qjl_seed: int = 2, signs=None, qjl=None) -> int:
    """Returns the context handle (an integer).  signs/qjl: host numpy arrays or None."""
    import numpy as np

    out = _P()
    s = None if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
    S = None if qjl is None else np.ascontiguousarray(qjl, dtype=np.float32)
    _check(_lib.tq_context_create(head_dim, wht_seed, qjl_seed, _ptr(s), _ptr(S), ctypes.byref(out)),
           "tq_context_create")
    return out.value


def tq_context_destroy(ctx: int) -> None:
    _check(_lib.tq_context_destroy(ctx), "tq_context_destroy")


def tq_context_get_tables(ctx: int, head_dim: int):
    """Returns (signs int8 [d], S float32 [d, d], centroids [3, 8], boundaries [3, 7])."""
    import numpy as np

    s = np.zeros(head_dim, np.int8)
    S = np.zeros((head_dim, head_dim), np.float32)
    c = np.zeros((3, 8), np.float32)
    b = np.zeros((3, 7), np.float32)
    _check(_lib.tq_context_get_tables(ctx, s.ctypes.data, S.ctypes.data, c.ctypes.data, b.ctypes.data),
           "tq_context_get_tables")
    return s, S, c, b


def tq_get_status(ctx: int) -> tuple[int, int]:
    """Returns (status, flags); synchronises the device."""
    f = _U32(0)
    st = _lib.tq_get_status(ctx, ctypes.byref(f))
    return st, f.value


# ---- views ----

@dataclass
class CacheView:
    """A cache view plus the torch tensors that own its memory."""
    fmt: str
    head_dim: int
    n_kv_heads: int
    page_size: int
    num_pages: int
    n_layers: int
    payload: object
    header: object
    bits: int = 0

    def c_view(self) -> tq_cache_view:
        return tq_cache_view(_fmt(self.fmt), self.head_dim, self.n_kv_heads, self.page_size, self.num_pages,
                             self.n_layers, self.bits, _ptr(self.payload), _ptr(self.header))

    @property
    def compressed_bytes_per_vector(self) -> int:
        return tq_vector_bytes(self.fmt, self.head_dim, self.bits)


def alloc_view(fmt, head_dim: int, n_kv_heads: int, page_size: int, num_pages: int, n_layers: int = 1,
               bits: int = 0, device="cuda") -> CacheView:
    """Allocates a zeroed view's payload and header with torch (the caller owns them)."""
    import torch

    n = n_layers * num_pages * n_kv_heads * page_size
    pb, hb = tq_payload_bytes(fmt, head_dim, bits), tq_header_bytes(fmt, head_dim, bits)
    if pb == 0:
        raise ValueError(f"unsupported view: {fmt} d={head_dim} bits={bits}")
    payload = torch.zeros(n * pb, dtype=torch.uint8, device=device)
    header = torch.zeros(n * hb, dtype=torch.uint8, device=device)
    return CacheView(fmt if isinstance(fmt, str) else tq_format_name(fmt), head_dim, n_kv_heads, page_size,
                     num_pages, n_layers, payload, header, bits)


def _view_arg(v):
    if v is None:
        return None
    cv = v.c_view() if isinstance(v, CacheView) else v
    return ctypes.byref(cv), cv


# ---- device entry points ----

def tq_encode_kv(ctx: int, k_view, k, v_view, v, layer_begin: int, n_layers: int, n_tokens: int,
                 in_layer_stride: int, in_token_stride: int, slots=None, slot_begin: int = 0,
                 stream=None) -> int:
    ka, va = _view_arg(k_view), _view_arg(v_view)
    return _lib.tq_encode_kv(ctx, ka[0] if ka else None, _ptr(k), va[0] if va else None, _ptr(v), layer_begin,
                             n_layers, n_tokens, in_layer_stride, in_token_stride, _ptr(slots), slot_begin,
                             _stream(stream))


def tq_decode_workspace_bytes(ctx: int, n_layers: int, batch: int, n_q_heads: int, max_ctx: int) -> int:
    return _lib.tq_decode_workspace_bytes(ctx, n_layers, batch, n_q_heads, max_ctx)


def tq_decode_attention(ctx: int, q, q_is_fp16: int, n_layers: int, batch: int, n_q_heads: int, k_view, v_view,
                        layer_begin: int, seq_lens, max_ctx: int, block_table, max_blocks_per_seq: int,
                        softmax_scale: float, skip_threshold: float, workspace, workspace_bytes: int, out,
                        stream=None) -> int:
    ka, va = _view_arg(k_view), _view_arg(v_view)
    return _lib.tq_decode_attention(ctx, _ptr(q), q_is_fp16, n_layers, batch, n_q_heads, ka[0], va[0], layer_begin,
                                    _ptr(seq_lens), max_ctx, _ptr(block_table), max_blocks_per_seq,
                                    softmax_scale, skip_threshold, _ptr(workspace), workspace_bytes, _ptr(out),
                                    _stream(stream))


def tq_decode_attention_static(ctx: int, q, q_is_fp16: int, n_layers: int, batch: int, n_q_heads: int, k_view,
                               v_view, layer_begin: int, seq_lens, max_ctx: int, block_table,
                               max_blocks_per_seq: int, softmax_scale: float, skip_threshold: float, out,
                               stream=None) -> int:
    ka, va = _view_arg(k_view), _view_arg(v_view)
    return _lib.tq_decode_attention_static(ctx, _ptr(q), q_is_fp16, n_layers, batch, n_q_heads, ka[0], va[0],
                                           layer_begin, _ptr(seq_lens), max_ctx, _ptr(block_table),
                                           max_blocks_per_seq, softmax_scale, skip_threshold, _ptr(out),
                                           _stream(stream))


def tq_dequantize(ctx: int, view, layer: int, slots, slot_begin: int, n: int, include_qjl: int, out,
                  stream=None) -> int:
    va = _view_arg(view)
    return _lib.tq_dequantize(ctx, va[0], layer, _ptr(slots), slot_begin, n, include_qjl, _ptr(out),
                              _stream(stream))


# ---- persistence ----

def _host_view(v) -> tuple:
    """(c view, host_memory flag) for a CacheView over torch tensors or numpy arrays."""
    cv = v.c_view() if isinstance(v, CacheView) else v
    host = 1
    if isinstance(v, CacheView) and hasattr(v.payload, "is_cuda") and v.payload.is_cuda:
        host = 0
    return cv, host


def tq_context_tables_hash(ctx: int) -> int:
    h = ctypes.c_uint64(0)
    _check(_lib.tq_context_tables_hash(ctx, ctypes.byref(h)), "tq_context_tables_hash")
    return h.value


def tq_cache_save(ctx, view, path: str) -> int:
    """Saves a view (device tensors or host arrays); ctx may be None.  Returns the status."""
    cv, host = _host_view(view)
    return _lib.tq_cache_save(ctx, ctypes.byref(cv), host, os.fsencode(path))


def tq_cache_file_info(path: str):
    """Returns (status, geometry dict, tables_hash)."""
    cv = tq_cache_view()
    h = ctypes.c_uint64(0)
    st = _lib.tq_cache_file_info(os.fsencode(path), ctypes.byref(cv), ctypes.byref(h))
    geo = {k: getattr(cv, k) for k in ("format", "head_dim", "n_kv_heads", "page_size", "num_pages", "n_layers",
                                       "bits")}
    return st, geo, h.value


def tq_cache_load(ctx, view, path: str) -> int:
    """Loads a file into a view of the same geometry (device tensors or host arrays); ctx may be None."""
    cv, host = _host_view(view)
    return _lib.tq_cache_load(ctx, ctypes.byref(cv), host, os.fsencode(path))


# ---- per-layer views ----

def _view_array(views):
    """(ctypes array of tq_cache_view, keep-alive) for a list of CacheView, or (None, None)."""
    if views is None:
        return None, None
    arr = (tq_cache_view * len(views))(*[v.c_view() if isinstance(v, CacheView) else v for v in views])
    return arr, arr


def _layer_array(layers):
    if layers is None:
        return None
    return (ctypes.c_int32 * len(layers))(*[int(x) for x in layers])


def tq_encode_kv_layers(ctx: int, k_views, k_view_layers, v_views, v_view_layers, n_layers: int, k, v,
                        n_tokens: int, in_layer_stride: int, in_token_stride: int, slots=None, slot_begin: int = 0,
                        stream=None) -> int:
    """k_views / v_views: lists of n_layers CacheView (or None); *_view_layers: lists of ints."""
    ka, kkeep = _view_array(k_views)
    va, vkeep = _view_array(v_views)
    kl, vl = _layer_array(k_view_layers), _layer_array(v_view_layers)
    return _lib.tq_encode_kv_layers(ctx, ka, kl, va, vl, n_layers, _ptr(k), _ptr(v), n_tokens, in_layer_stride,
                                    in_token_stride, _ptr(slots), slot_begin, _stream(stream))


def tq_decode_attention_layers(ctx: int, q, q_is_fp16: int, n_layers: int, batch: int, n_q_heads: int, k_views,
                               k_view_layers, v_views, v_view_layers, seq_lens, max_ctx: int, block_table,
                               max_blocks_per_seq: int, softmax_scale: float, skip_threshold: float, workspace,
                               workspace_bytes: int, out, stream=None) -> int:
    ka, kkeep = _view_array(k_views)
    va, vkeep = _view_array(v_views)
    return _lib.tq_decode_attention_layers(ctx, _ptr(q), q_is_fp16, n_layers, batch, n_q_heads, ka,
                                           _layer_array(k_view_layers), va, _layer_array(v_view_layers),
                                           _ptr(seq_lens), max_ctx, _ptr(block_table), max_blocks_per_seq,
                                           softmax_scale, skip_threshold, _ptr(workspace), workspace_bytes, _ptr(out),
                                           _stream(stream))


# ---- chunked-prefill attention ----

def tq_prefill_workspace_bytes(ctx: int, n_tokens: int, n_q_heads: int) -> int:
    return _lib.tq_prefill_workspace_bytes(ctx, n_tokens, n_q_heads)


def tq_prefill_attention(ctx: int, q, q_is_fp16: int, n_tokens: int, n_q_heads: int, k_view, v_view, layer: int,
                         seq: int, block_table, max_blocks: int, start: int, softmax_scale: float, workspace,
                         workspace_bytes: int, out, stream=None) -> int:
    ka, va = _view_arg(k_view), _view_arg(v_view)
    return _lib.tq_prefill_attention(ctx, _ptr(q), q_is_fp16, n_tokens, n_q_heads, ka[0], va[0], layer, seq,
                                     _ptr(block_table), max_blocks, start, softmax_scale, _ptr(workspace),
                                     workspace_bytes, _ptr(out), _stream(stream))
