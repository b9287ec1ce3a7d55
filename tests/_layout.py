"""Test-side packing/unpacking of the stored byte layout documented in include/tq.h.

Used to read codes out of the CUDA path's caches (bit-exact comparisons with
the oracle) and to write oracle-produced codes into caches (decode parity on
identical codes).  Written from the header's description, not from the kernels.
"""
import numpy as np

TURBO = {"turbo2": (1, 1), "turbo3": (2, 1), "turbo4": (3, 1),
         "turbo2_mse": (1, 0), "turbo3_mse": (2, 0), "turbo4_mse": (3, 0)}


def code_bits(fmt, bits=0):
    if fmt in TURBO:
        b, q = TURBO[fmt]
        return b + q
    if fmt == "minmax":
        return bits
    raise ValueError(fmt)


def unpack_codes(payload: np.ndarray, d: int, w: int) -> np.ndarray:
    """payload uint8 [..., d*w/8] -> codes [..., d]: coordinate i at bit offset w*i, little endian."""
    bits = np.unpackbits(payload, axis=-1, bitorder="little").reshape(payload.shape[:-1] + (d, w))
    return (bits.astype(np.int64) << np.arange(w)).sum(axis=-1)


def pack_codes(codes: np.ndarray, w: int) -> np.ndarray:
    """codes [..., d] -> payload uint8 [..., d*w/8]."""
    codes = np.asarray(codes, dtype=np.int64)
    bits = ((codes[..., None] >> np.arange(w)) & 1).astype(np.uint8)
    flat = bits.reshape(codes.shape[:-1] + (codes.shape[-1] * w,))
    return np.packbits(flat, axis=-1, bitorder="little")


def split_turbo(codes: np.ndarray, fmt: str):
    """(idx, sigma or None) from turbo codes: bits [0, b) index, bit b QJL sign (K only)."""
    b, q = TURBO[fmt]
    idx = codes & ((1 << b) - 1)
    return idx, ((codes >> b) & 1).astype(bool) if q else None


def join_turbo(idx: np.ndarray, sigma, fmt: str) -> np.ndarray:
    b, q = TURBO[fmt]
    c = np.asarray(idx, dtype=np.int64)
    if q:
        c = c | (np.asarray(sigma, dtype=np.int64) << b)
    return c


def header_halves(header: np.ndarray, n_halves: int) -> np.ndarray:
    """header uint8 [..., 2*n] -> float16 [..., n]."""
    return header.view(np.float16).reshape(header.shape[:-1] + (n_halves,))


def f16_ulp_diff(a, b) -> np.ndarray:
    """Distance in units in the last place between fp16 arrays (same sign assumed)."""
    ia = np.asarray(a, dtype=np.float16).view(np.int16).astype(np.int64)
    ib = np.asarray(b, dtype=np.float16).view(np.int16).astype(np.int64)
    return np.abs(ia - ib)
