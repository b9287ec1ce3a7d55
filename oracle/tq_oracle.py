"""CPU oracle for TurboQuant-style KV-cache compression and compressed-cache decode attention.

TEST INFRASTRUCTURE.  This module is the independent, slow, obviously correct
restatement of what the CUDA path computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it.  It shares no code, table or constant generator
with the CUDA library; the random tables of the method (sign diagonal, QJL
projection) are inputs, drawn by the seeded generator module that both sides
use.

Arithmetic is fp64 NumPy except where the method turns floating point into an
integer through a single formula that the pages spell out (q8_0, min-max): there
both sides take the decision in IEEE fp32, the precision of the kernel.

Sources (page title, then section):
  [TQ+]   "TurboQuant+ KV cache compression" (quidproquo.cc, 2026-04-01):
          Stage 1 "PolarQuant: rotation + scalar quantisation" step list;
          Stage 2 "QJL: 1-bit residual compression" step list;
          the format table (turbo2/3/4 bits per element);
          "K/V asymmetric strategy" (K: both stages, V: stage 1 only).
  [DEEP]  "TurboQuant+ deep dive: 2-bit KV cache ..." (chenxutan.com):
          section 2.3 QJL (sign rule ``projection > 0``);
          section 3.3 sparse V dequantisation (mask V after softmax);
          section 2.1 traditional quantisation (absmax / (2^(n-1)-1), round).
  [INTRO] "TurboQuant+: 3.8x compression ..." (yeyulingfeng.com):
          core content item 4, Sparse V (skip V where the weight < 1e-6);
          item 3, Boundary V (first 2 + last 2 layers at q8_0).
  [MAC]   "mac-code TurboQuant analysis" (GitHub issue walter-grace/mac-code #1):
          section 2.1 per-group asymmetric min-max quantisation and its worked
          example [0.1, 0.5, 0.9] at 4 bits.

Readings where the pages are silent are named "reading" in the docstrings.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# formats: name -> (index bits of stage 1, has the QJL stage)
# [TQ+] format table: turbo2 = 1-bit + 1-bit, turbo3 = 2-bit + 1-bit,
# turbo4 = 3-bit + 1-bit.  [TQ+] K/V asymmetry: V keeps stage 1 only.
# ---------------------------------------------------------------------------
TURBO_FORMATS = {
    "turbo2": (1, True), "turbo3": (2, True), "turbo4": (3, True),
    "turbo2_mse": (1, False), "turbo3_mse": (2, False), "turbo4_mse": (3, False),
}


# ---------------------------------------------------------------------------
# Walsh-Hadamard rotation
# ---------------------------------------------------------------------------

def hadamard(d: int) -> np.ndarray:
    """Orthonormal Sylvester Hadamard matrix H_d / sqrt(d), built by the Kronecker recursion.

    [TQ+] Stage 1 step 2: Walsh-Hadamard random rotation, orthogonal and
    distance preserving.  Reading: natural (Sylvester) order, 1/sqrt(d) scale,
    d = head_dim must be a power of two.
    """
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h / math.sqrt(d)


def rotate(x_unit: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """y = H_d diag(s) x  ([TQ+] Stage 1 step 2; reading: sign flip first, then H)."""
    d = x_unit.shape[-1]
    return (x_unit * signs.astype(np.float64)) @ hadamard(d).T


def unrotate(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """x = diag(s) H_d y, the inverse of ``rotate`` (H is symmetric and orthonormal)."""
    d = y.shape[-1]
    return (y @ hadamard(d)) * signs.astype(np.float64)


# ---------------------------------------------------------------------------
# Lloyd-Max codebook
# ---------------------------------------------------------------------------

def _phi(t):
    return np.exp(-0.5 * t * t) / math.sqrt(2.0 * math.pi)


def _Phi(t):
    return 0.5 * (1.0 + np.vectorize(math.erf)(t / math.sqrt(2.0)))


def lloyd_max_gaussian(bits: int, d: int, tol: float = 1e-13, max_iter: int = 200000):
    """Lloyd-Max quantiser for N(0, 1/d) with 2^bits levels, in fp64.

    [TQ+] Stage 1 step 3: the optimal codebook for the Gaussian is precomputed
    with Lloyd's algorithm.  Reading: the coordinate law after the rotation is
    taken as N(0, 1/d).  Iteration: boundaries are midpoints of neighbouring
    centroids; each centroid is the conditional mean of its cell,
    sigma * (phi(a/sigma) - phi(b/sigma)) / (Phi(b/sigma) - Phi(a/sigma));
    start from the N(0, 1) quantile midpoints; stop when no centroid moves by
    more than tol * sigma; finally make the codebook exactly odd-symmetric.

    Returns (centroids [2^bits], boundaries [2^bits - 1]) ascending, fp64.
    """
    L = 1 << bits
    sigma = 1.0 / math.sqrt(d)
    from scipy.special import ndtri  # inverse normal CDF, only for the starting point

    c = ndtri((np.arange(L) + 0.5) / L)  # in units of sigma
    for _ in range(max_iter):
        b = 0.5 * (c[:-1] + c[1:])
        lo = np.concatenate(([-np.inf], b))
        hi = np.concatenate((b, [np.inf]))
        num = _phi(lo) - _phi(hi)
        den = _Phi(hi) - _Phi(lo)
        c_new = num / den
        moved = np.max(np.abs(c_new - c))
        c = c_new
        if moved < tol:
            break
    # N(0, 1/d) is symmetric, so the optimal quantiser is odd: c[L-1-k] = -c[k]
    # (reading).  Mirroring removes rounding asymmetry so the middle boundary
    # is exactly 0 and a zero coordinate takes the upper index on any machine.
    c = 0.5 * (c - c[::-1])
    c = c * sigma
    return c, 0.5 * (c[:-1] + c[1:])


def codebook(bits: int, d: int):
    """The stored codebook: fp32 centroids and fp32 boundaries (midpoints taken in fp64).

    Returned as fp64 arrays holding fp32-representable values.  Reading: both
    tables are kept in fp32, the boundaries being the fp64 midpoints rounded.
    """
    c, b = lloyd_max_gaussian(bits, d)
    return c.astype(np.float32).astype(np.float64), b.astype(np.float32).astype(np.float64)


def gaussian_mse(bits: int, d: int = 1) -> float:
    """Expected squared error of the Lloyd-Max quantiser on N(0, 1/d) (closed form over cells)."""
    c, b = lloyd_max_gaussian(bits, d)
    s = 1.0 / math.sqrt(d)
    lo = np.concatenate(([-np.inf], b)) / s
    hi = np.concatenate((b, [np.inf])) / s
    cc = c / s
    # E[(X - c)^2; a < X < b] for X ~ N(0,1):
    # = [Phi]_a^b (1 + c^2) - 2c [phi(a) - phi(b)] + [a phi(a) - b phi(b)]
    def tphi(t):
        return np.where(np.isinf(t), 0.0, t * _phi(np.where(np.isinf(t), 0.0, t)))
    P = _Phi(hi) - _Phi(lo)
    m1 = _phi(lo) - _phi(hi)
    m2 = P + tphi(lo) - tphi(hi)
    return float(np.sum(m2 - 2 * cc * m1 + cc * cc * P)) * s * s


def quantize(y: np.ndarray, boundaries: np.ndarray) -> np.ndarray:
    """idx_i = #{j : y_i >= beta_j}  ([TQ+] Stage 1 step 3; reading: a tie goes up)."""
    return np.sum(y[..., None] >= boundaries, axis=-1).astype(np.int64)


# ---------------------------------------------------------------------------
# TurboQuant encode / decode
# ---------------------------------------------------------------------------

def turbo_encode(x16: np.ndarray, fmt: str, signs: np.ndarray, S: np.ndarray | None):
    """Encode vectors x [..., d] (fp16 values) with a turbo format.

    Stage 1 ([TQ+] Stage 1 step list):
      1. n = ||x||, x_hat = x / n (x_hat = 0 when n = 0);
      2. y = H diag(s) x_hat;
      3. idx = Lloyd-Max index of each coordinate of y;
      4. store idx and n.
    Stage 2, K formats only ([TQ+] Stage 2 step list, [DEEP] 2.3 sign rule):
      5. r = y - c[idx] (residual in the unit rotated space: the rotation
         preserves norms and inner products, reading);
      6. store the residual norm rnorm = n * ||r||;
      7. sigma_j = [(S r)_j > 0], one bit per dimension (S is d x d).
    Norms are stored as fp16 (round to nearest even).

    Returns a dict with the stored fields (n16, idx, and for K rnorm16, sigma)
    plus the fp64 intermediates y and proj = S r used to locate decision
    boundaries in parity tests.
    """
    bits, has_qjl = TURBO_FORMATS[fmt]
    x = np.asarray(x16, dtype=np.float16).astype(np.float64)
    d = x.shape[-1]
    n = np.sqrt(np.sum(x * x, axis=-1))
    safe = np.where(n > 0, n, 1.0)
    x_hat = np.where((n > 0)[..., None], x / safe[..., None], 0.0)
    y = rotate(x_hat, signs)
    c, b = codebook(bits, d)
    idx = quantize(y, b)
    out = {"n16": n.astype(np.float16), "idx": idx, "y": y, "n": n}
    if has_qjl:
        out.update(qjl_stage(y, n, idx, bits, S))
    return out


def qjl_stage(y: np.ndarray, n: np.ndarray, idx: np.ndarray, bits: int, S) -> dict:
    """Stage 2 of a K format for given stage-1 indices ([TQ+] Stage 2 step list, [DEEP] 2.3).

    y [..., d]: the rotated unit vectors; n [...]: their norms; idx [..., d]: the
    stage-1 indices, whoever chose them (``turbo_encode`` passes its own; a
    parity check passes the indices a GPU stored, so that the rest of a vector
    whose index was decided differently inside the 1e-6 band is still checked).
      1. r = y - c[idx] (residual of the stage-1 reconstruction, unit rotated space);
      2. rnorm = n * ||r||, stored as fp16;
      3. sigma_j = [(S r)_j > 0].
    Returns {"rnorm16", "sigma", "proj" (= S r, fp64), "r"}.
    """
    d = y.shape[-1]
    c, _ = codebook(bits, d)
    r = y - c[np.asarray(idx)]
    rn = np.sqrt(np.sum(r * r, axis=-1))
    proj = r @ np.asarray(S, dtype=np.float64).T
    return {"rnorm16": (np.asarray(n) * rn).astype(np.float16), "sigma": proj > 0, "proj": proj, "r": r}


QJL_CONST = math.sqrt(math.pi / 2.0)


def turbo_dequant(enc: dict, fmt: str, signs: np.ndarray, S: np.ndarray | None,
                  include_qjl: bool = True) -> np.ndarray:
    """Reconstruct x~ [..., d] from stored fields.

    MSE part: n * diag(s) H c[idx].  QJL part (K, vector form): the residual
    estimate rnorm * sqrt(pi/2) / d * S^T (2 sigma - 1) in the rotated space,
    mapped back with diag(s) H.  The constant follows from
    E[sign(g.r) g] = sqrt(2/pi) r / ||r|| for g ~ N(0, I) (reading: the pages'
    garbled decoder is replaced by this unbiased form, m = d projections).
    """
    bits, has_qjl = TURBO_FORMATS[fmt]
    idx = enc["idx"]
    d = idx.shape[-1]
    c, _ = codebook(bits, d)
    n = enc["n16"].astype(np.float64)
    y_hat = n[..., None] * c[idx]
    if has_qjl and include_qjl:
        pm = np.where(enc["sigma"], 1.0, -1.0)
        rn = enc["rnorm16"].astype(np.float64)
        y_hat = y_hat + (rn * QJL_CONST / d)[..., None] * (pm @ np.asarray(S, dtype=np.float64))
    return unrotate(y_hat, signs)


def qjl_inner_product_estimate(q: np.ndarray, r: np.ndarray, S: np.ndarray) -> np.ndarray:
    """<q, r> ~= ||r|| sqrt(pi/2) / m <S q, sign(S r)>, m = rows of S (sign 0 -> -1)."""
    S = np.asarray(S, dtype=np.float64)
    m = S.shape[0]
    pm = np.where(r @ S.T > 0, 1.0, -1.0)
    return np.linalg.norm(r, axis=-1) * QJL_CONST / m * np.sum((q @ S.T) * pm, axis=-1)


# ---------------------------------------------------------------------------
# q8_0 and min-max baselines
# ---------------------------------------------------------------------------

def q8_0_encode(x16: np.ndarray):
    """q8_0: per block of 32 along d, delta = max|x| / 127, q = round half away (x / delta).

    [DEEP] 2.1 absmax rule scale = max|x| / (2^(n-1) - 1), q = round(x / scale),
    with n = 8 over blocks of 32 (the q8_0 cache type of the pages).  Reading:
    delta and x / delta are IEEE fp32 divisions (the kernel's precision, since
    they decide an integer); delta is stored as fp16; delta = 0 gives q = 0.
    Returns (q int8 [..., d], delta16 [..., d/32]).
    """
    x = np.asarray(x16, dtype=np.float16).astype(np.float32)
    d = x.shape[-1]
    blk = x.reshape(x.shape[:-1] + (d // 32, 32))
    amax = np.max(np.abs(blk), axis=-1)
    delta = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(delta > 0, delta, np.float32(1.0)).astype(np.float32)
    t = (blk / safe[..., None]).astype(np.float32)
    q = np.sign(t) * np.floor(np.abs(t).astype(np.float64) + 0.5)
    q = np.where((delta > 0)[..., None], q, 0.0)
    return q.reshape(x.shape).astype(np.int8), delta.astype(np.float16)


def q8_0_dequant(q: np.ndarray, delta16: np.ndarray) -> np.ndarray:
    d = q.shape[-1]
    blk = q.astype(np.float64).reshape(q.shape[:-1] + (d // 32, 32))
    return (blk * delta16.astype(np.float64)[..., None]).reshape(q.shape)


def minmax_encode(x, bits: int = 3, group: int = 64):
    """Per-group asymmetric min-max ([MAC] 2.1 and its worked example).

    Groups of ``group`` consecutive elements along the last axis (reading).
    scale = (max - min) / (2^bits - 1), zero = min, q = round((x - zero) / scale),
    in IEEE fp32 step by step; the example's 7.5 -> 8 fixes round half up,
    taken as floor(v + 0.5) (reading); q is clipped to [0, 2^bits - 1]; a flat
    group gets scale 0 and q = 0.  scale and zero are stored as fp16.
    Returns (q uint8 [..., d], scale16 [..., d/group], zero16 [..., d/group]).
    """
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    g = x.reshape(x.shape[:-1] + (d // group, group))
    mn = np.min(g, axis=-1).astype(np.float32)
    mx = np.max(g, axis=-1).astype(np.float32)
    scale = ((mx - mn) / np.float32((1 << bits) - 1)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    t = ((g - mn[..., None]).astype(np.float32) / safe[..., None]).astype(np.float32)
    t = (t + np.float32(0.5)).astype(np.float32)
    q = np.clip(np.floor(t), 0, (1 << bits) - 1)
    q = np.where((scale > 0)[..., None], q, 0.0)
    return q.reshape(x.shape).astype(np.uint8), scale.astype(np.float16), mn.astype(np.float16)


def minmax_dequant(q, scale16, zero16, group: int = 64) -> np.ndarray:
    """x~ = q * scale + zero ([MAC] 2.1, dequantisation)."""
    d = q.shape[-1]
    g = q.astype(np.float64).reshape(q.shape[:-1] + (d // group, group))
    out = g * scale16.astype(np.float64)[..., None] + zero16.astype(np.float64)[..., None]
    return out.reshape(q.shape)


# ---------------------------------------------------------------------------
# decode attention
# ---------------------------------------------------------------------------

def decode_attention(q: np.ndarray, k_tilde: np.ndarray, v_tilde: np.ndarray,
                     scale: float, tau: float = 0.0):
    """Single-token decode attention over a dequantised cache, fp64.

    q [Hq, d]; k_tilde, v_tilde [T, Hkv, d].  Query head h reads KV head
    floor(h / G), G = Hq / Hkv (reading).  s_j = scale <q, k~_j> over every
    cached token (reading: no mask; scale = 1/sqrt(d) by default); p =
    softmax(s); o_full = sum_j p_j v~_j.  o_skip drops the V terms whose final
    weight p_j is below tau while keeping the softmax denominator ([INTRO]
    item 4: skip V where the attention weight is below 1e-6; [DEEP] 3.3 masks V
    after the softmax).  Returns (o_full, o_skip) [Hq, d].
    """
    Hq, d = q.shape
    T, Hkv, _ = k_tilde.shape
    G = Hq // Hkv
    o_full = np.zeros((Hq, d))
    o_skip = np.zeros((Hq, d))
    if T == 0:
        return o_full, o_skip
    for h in range(Hq):
        kv = h // G
        s = scale * (k_tilde[:, kv, :] @ q[h].astype(np.float64))
        m = np.max(s)
        e = np.exp(s - m)
        p = e / np.sum(e)
        o_full[h] = p @ v_tilde[:, kv, :]
        o_skip[h] = np.where(p >= tau, p, 0.0) @ v_tilde[:, kv, :]
    return o_full, o_skip


def prefill_attention(q: np.ndarray, k_tilde: np.ndarray, v_tilde: np.ndarray, start: int,
                      scale: float) -> np.ndarray:
    """Chunked-prefill attention over a dequantised cache, fp64.

    A chunk of C new tokens at positions start .. start + C - 1 attends to the cache, which already
    holds them ("TurboQuant+: 3.8x compression ...", core content item 1: prefill reads the
    quantised cache; reading: causal, each token attends to every cached token up to and including
    its own position).  q [C, Hq, d]; k_tilde, v_tilde [T, Hkv, d] with T >= start + C.  Query
    head h reads KV head floor(h / G) (reading, as for decode).  For chunk token i:
    s_j = scale <q_i, k~_j> for j <= start + i; p = softmax(s); o_i = sum_j p_j v~_j.
    Returns o [C, Hq, d].
    """
    C, Hq, d = q.shape
    T, Hkv, _ = k_tilde.shape
    G = Hq // Hkv
    out = np.zeros((C, Hq, d))
    for i in range(C):
        n = start + i + 1
        for h in range(Hq):
            kv = h // G
            s = scale * (k_tilde[:n, kv, :] @ np.asarray(q[i, h], dtype=np.float64))
            e = np.exp(s - np.max(s))
            out[i, h] = (e / np.sum(e)) @ v_tilde[:n, kv, :]
    return out


def compressed_scores(q: np.ndarray, k_enc: dict, fmt: str, signs, S, scale: float):
    """Scores computed in the compressed domain, without reconstructing K.

    With q_rot = H diag(s) q and Sq = S q_rot, for K token j:
      s_j = scale * ( n_j <q_rot, c[idx_j]> + rnorm_j sqrt(pi/2)/d <Sq, 2 sigma_j - 1> ).
    By linearity this equals scale <q, k~_j> for the vector-form dequantisation;
    q is rotated once per query ("rotate q once", the decode recipe).
    q [Hq, d] for one KV head's tokens: k_enc fields [T, d] / [T].  Returns [Hq, T].
    """
    bits, has_qjl = TURBO_FORMATS[fmt]
    d = q.shape[-1]
    c, _ = codebook(bits, d)
    q_rot = rotate(np.asarray(q, dtype=np.float64), signs)
    n = k_enc["n16"].astype(np.float64)
    s = n[None, :] * (q_rot @ c[k_enc["idx"]].T)
    if has_qjl:
        Sq = q_rot @ np.asarray(S, dtype=np.float64).T
        pm = np.where(k_enc["sigma"], 1.0, -1.0)
        s = s + k_enc["rnorm16"].astype(np.float64)[None, :] * QJL_CONST / d * (Sq @ pm.T)
    return scale * s


def kv_cache_bytes_fp16(n_layers: int, n_kv_heads: int, head_dim: int, ctx: int, batch: int = 1) -> int:
    """2 (K and V) x layers x heads x head_dim x context x 2 bytes ([TQ+] cache-size formula)."""
    return 2 * batch * n_layers * n_kv_heads * head_dim * ctx * 2


def payload_bits_per_element(fmt: str) -> int:
    """Stored code bits per element, without per-vector norms ([TQ+] format table)."""
    if fmt in TURBO_FORMATS:
        bits, has_qjl = TURBO_FORMATS[fmt]
        return bits + (1 if has_qjl else 0)
    if fmt == "q8_0":
        return 8
    raise ValueError(fmt)
