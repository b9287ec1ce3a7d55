"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds no arithmetic of the compression method itself: it only draws
random numbers (the method's random tables and the synthetic K/V/q tensors)
from fixed seeds, so that both sides of a parity check see identical inputs.

Random tables of the method
---------------------------
* ``wht_signs(seed, d)``: the diagonal of the random sign flip that precedes
  the Walsh-Hadamard rotation ("TurboQuant+ KV cache compression",
  Stage 1 step list: random Walsh-Hadamard rotation).
* ``qjl_matrix(seed, d)``: the d x d iid N(0, 1) projection of the 1-bit QJL
  residual sketch ("TurboQuant+ KV cache compression", Stage 2: multiply by a
  random projection matrix and keep the sign).

Both are counter-based: element ``k`` depends only on ``(seed, k)``.  The
counter generator is SplitMix64 as published by Steele, Lea and Flood (2014)
and in Vigna's reference ``splitmix64.c``: ``z = c + 0x9E3779B97F4A7C15``;
``z = (z ^ z>>30) * 0xBF58476D1CE4E5B9``; ``z = (z ^ z>>27) * 0x94D049BB133111EB``;
``out = z ^ z>>31``.  The native library carries its own implementation of the
same definition for callers that do not pass tables in.

Synthetic K/V/q
---------------
fp16 N(0, 1) tensors with outlier channels scaled x20, as the benchmark
recipes describe (4 fixed channels per KV head, or 1% of the H x d channel
space).  Bulk tensors are drawn with ``torch.Generator`` on the requested
device; everything a test compares is copied from the same tensor.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(counters) -> np.ndarray:
    """SplitMix64 output for each 64-bit counter value (one ``next()`` from state c)."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = c + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def _counters(seed: int, n: int, start: int = 0) -> np.ndarray:
    if not (0 <= seed < 2**32):
        raise ValueError("seed must fit in 32 bits")
    return (np.uint64(seed) << np.uint64(32)) + np.arange(start, start + n, dtype=np.uint64)


def wht_signs(seed: int, d: int) -> np.ndarray:
    """int8 [d] of +-1: s_i = -1 iff the top bit of SplitMix64((seed << 32) + i) is set."""
    z = splitmix64(_counters(seed, d))
    return np.where((z >> np.uint64(63)) == 1, -1, 1).astype(np.int8)


def uniform53(seed: int, n: int, start: int = 0) -> np.ndarray:
    """fp64 uniforms in (0, 1]: ((SplitMix64(c) >> 11) + 1) * 2^-53."""
    z = splitmix64(_counters(seed, n, start))
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def qjl_matrix(seed: int, d: int) -> np.ndarray:
    """fp32 [d, d] (row j = projection j) of iid N(0, 1).

    Element e = j*d + i uses the cosine branch of Box-Muller on the uniforms at
    counters 2e and 2e+1, evaluated in fp64 and rounded to fp32.
    """
    u = uniform53(seed, 2 * d * d)
    u1, u2 = u[0::2], u[1::2]
    g = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return g.astype(np.float32).reshape(d, d)


# ---------------------------------------------------------------------------
# synthetic tensors
# ---------------------------------------------------------------------------

def _torch():
    import torch  # local import: the oracle-only tests do not need torch

    return torch


def outlier_channels_per_head(seed: int, n_heads: int, d: int, per_head: int) -> np.ndarray:
    """[n_heads, per_head] channel ids: randperm(d)[:per_head] per head from a seeded PCG64."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.stack([rng.permutation(d)[:per_head] for _ in range(n_heads)])


def outlier_channels_fraction(seed: int, n_heads: int, d: int, frac: float) -> np.ndarray:
    """Flat ids into the H*d channel space: round(frac*H*d) distinct channels."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k = max(1, int(round(frac * n_heads * d)))
    return np.sort(rng.permutation(n_heads * d)[:k])


def kv_tensor(n_tokens: int, n_heads: int, d: int, seed: int, *, device="cpu",
              outliers_per_head: int = 0, outlier_frac: float = 0.0,
              outlier_scale: float = 20.0, outlier_seed: int | None = None):
    """fp16 [n_tokens, n_heads, d]: N(0,1) from torch.Generator(seed), outlier channels x scale."""
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn((n_tokens, n_heads, d), generator=g, device=device, dtype=torch.float32)
    oseed = seed + 1_000_003 if outlier_seed is None else outlier_seed
    if outliers_per_head:
        ch = outlier_channels_per_head(oseed, n_heads, d, outliers_per_head)
        for h in range(n_heads):
            x[:, h, torch.as_tensor(ch[h], device=device)] *= outlier_scale
    elif outlier_frac > 0:
        flat = torch.as_tensor(outlier_channels_fraction(oseed, n_heads, d, outlier_frac), device=device)
        x.view(n_tokens, n_heads * d)[:, flat] *= outlier_scale
    return x.to(torch.float16)


def normal_tensor(shape, seed: int, *, device="cpu", dtype=None, scale: float = 1.0):
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32) * scale
    return x if dtype is None else x.to(dtype)


def needle_workload(n_tokens: int, n_kv_heads: int, n_q_heads: int, d: int, seed: int, *,
                    n_needles: int = 16, q_scale: float = 8.0, noise_std: float = 0.1, device="cpu"):
    """Peaked-softmax recipe: per KV head, ``n_needles`` seeded positions whose K equals one
    shared N(0, I) vector u; every query head of the group is q_scale*u plus N(0, noise_std^2).

    Returns (k fp16 [T, H, d], q fp32 [Hq, d], needle positions int64 [H, n_needles]).
    """
    torch = _torch()
    k = kv_tensor(n_tokens, n_kv_heads, d, seed, device=device)
    u = normal_tensor((n_kv_heads, d), seed + 11, device=device)
    rng = np.random.Generator(np.random.PCG64(seed + 13))
    pos = np.stack([np.sort(rng.choice(n_tokens, size=n_needles, replace=False)) for _ in range(n_kv_heads)])
    for h in range(n_kv_heads):
        k[torch.as_tensor(pos[h], device=device), h, :] = u[h].to(torch.float16)
    G = n_q_heads // n_kv_heads
    noise = normal_tensor((n_q_heads, d), seed + 17, device=device, scale=noise_std)
    q = u.to(torch.float16).float().repeat_interleave(G, dim=0) * q_scale + noise
    return k, q, torch.as_tensor(pos)


def seq_lens_uniform(n_seqs: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """int32 [n_seqs] context lengths uniform in [lo, hi] from a seeded PCG64."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(lo, hi + 1, size=n_seqs).astype(np.int32)


def shuffled_block_table(seq_lens: np.ndarray, page_size: int, seed: int, extra_pages: int = 0):
    """Assign a random physical page to each logical page of each sequence.

    Returns (block_table int32 [B, max_blocks] padded with -1, num_pages).
    """
    blocks = [(int(L) + page_size - 1) // page_size for L in seq_lens]
    total = sum(blocks) + extra_pages
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(total).astype(np.int32)
    mb = max(blocks) if blocks else 0
    bt = np.full((len(blocks), max(mb, 1)), -1, dtype=np.int32)
    o = 0
    for b, nb in enumerate(blocks):
        bt[b, :nb] = perm[o:o + nb]
        o += nb
    return bt, total


@dataclass
class Workload:
    """One benchmark recipe: shapes, formats and seeds (no arithmetic)."""
    name: str
    n_layers: int
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    ctx: int
    k_format: str
    v_format: str
    batch: int = 1
    seed: int = 0
    wht_seed: int = 1
    qjl_seed: int = 2
    outliers_per_head: int = 0
    outlier_frac: float = 0.0
    encode_chunk: int = 0
    page_size: int = 0
    v_format_layers: dict = field(default_factory=dict)
    note: str = ""


WORKLOADS = {
    "tiny-d128-h8-t1024-turbo3": Workload(
        "tiny-d128-h8-t1024-turbo3", n_layers=1, n_kv_heads=8, n_q_heads=32, head_dim=128,
        ctx=1024, k_format="turbo3", v_format="turbo3_mse", seed=0, wht_seed=1, qjl_seed=2,
        outliers_per_head=4,
        note="single layer, 4 outlier channels per head x20, one decode step, GQA 4"),
    "llama3-8b-32k-turbo4": Workload(
        "llama3-8b-32k-turbo4", n_layers=32, n_kv_heads=8, n_q_heads=32, head_dim=128,
        ctx=32768, k_format="turbo4", v_format="turbo4_mse", seed=2, wht_seed=1, qjl_seed=2,
        outlier_frac=0.01, encode_chunk=4096,
        note="32 layers, 1% outlier channels x20, encode a 4096-token chunk + decode all layers"),
    "llama-70b-128k-turbo4": Workload(
        "llama-70b-128k-turbo4", n_layers=80, n_kv_heads=8, n_q_heads=64, head_dim=128,
        ctx=131072, k_format="turbo4", v_format="turbo4_mse", seed=3, wht_seed=1, qjl_seed=2,
        outlier_frac=0.01, note="80 layers, GQA 8, cache generated layer by layer"),
    "asym-q8k-turbo2v-needles": Workload(
        "asym-q8k-turbo2v-needles", n_layers=64, n_kv_heads=4, n_q_heads=32, head_dim=128,
        ctx=32768, k_format="q8_0", v_format="turbo2_mse", seed=4, wht_seed=1, qjl_seed=2,
        v_format_layers={0: "q8_0", 1: "q8_0", 62: "q8_0", 63: "q8_0"},
        note="q8_0 K, turbo2 V except 2+2 boundary layers at q8_0, 16 needles per KV head"),
    "paged-batch64-turbo3": Workload(
        "paged-batch64-turbo3", n_layers=32, n_kv_heads=8, n_q_heads=32, head_dim=128,
        ctx=16384, k_format="turbo3", v_format="turbo3_mse", batch=64, seed=5, wht_seed=1,
        qjl_seed=2, page_size=16,
        note="64 sequences, ctx ~ U[1K,16K], 16-token pages, shuffled block table; d in {64,128,256}"),
}
