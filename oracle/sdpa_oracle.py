"""Float64 CPU oracle for scaled dot-product attention (forward, backward, decode).

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
definition that the CUDA library is checked against.  Only the test suite,
the smoke check and the benchmark's CPU legs (its CPU baseline and its
reference arm) may import it; the library itself never does, and it shares
no code with the CUDA path.

Everything is NumPy float64, one (batch, query head) problem at a time, in the
order and notation of the course chapter "Scaled dot-product attention
(forward and backward)": scores S = alpha*Q*K^T, masked softmax P, output
O = P*V, and the hand-derived backward of its section 2.3.

Sources for each step (page title, section):
  * definition O = softmax(alpha*Q*K^T + mask)*V and the default scale
    1/sqrt(d): "Scaled dot-product attention (forward and backward)",
    Key Takeaways and section 2.1;
  * additive mask, -inf where blocked, applied before the softmax, and an
    all-blocked row giving zeros: same page, section 2.2, and
    "ScaledDotProductAttentionBackward" (Notes: additive mask, engine-side
    causal j <= i);
  * causal = lower triangle tril(diagonal=0), top-left aligned:
    "Understanding PyTorch Scaled Dot-Product Attention", section 3;
  * grouped-query heads by repeat_interleave (query head h reads KV head
    floor(h / (Hq/Hkv))): same page, section 4;
  * backward dV = P^T dO, dP = dO V^T, dS = P o (dP - D), D_i = sum_j P_ij dP_ij
    = dO_i . O_i, dQ = alpha dS K, dK = alpha dS^T Q: "Scaled dot-product
    attention (forward and backward)", section 2.3;
  * log-sum-exp statistics max + ln(sum exp(s - max)), natural log, fp32
    shape (B, Hq, L): "Attention" (cuDNN), Scaled Dot Product Attention,
    Returns ("stats");
  * padding by per-batch lengths seq_len_q / seq_len_kv, diagonal alignment
    (TOP_LEFT: the diagonal starts at the top-left; BOTTOM_RIGHT: at the
    bottom-right, aligned with the actual lengths) and the diagonal band
    (right bound: columns beyond row + right_bound masked; left bound: columns
    at or before row - left_bound masked): "Attention" (cuDNN), Configurable
    Options (Padding mask, Diagonal masking options) and Scaled Dot Product
    Attention, Args (seq_len_q, seq_len_kv, diagonal_alignment,
    diagonal_band_left_bound, diagonal_band_right_bound);
  * attention dropout: one uniform u per weight, keep where u >= p, kept
    weights scaled by 1/(1-p): O = (P o m) V with m = keep / (1 - p); the
    backward replays m: dV = (P o m)^T dO, dP = (dO V^T) o m, the softmax
    VJP unchanged ("Scaled dot-product attention (forward and backward)",
    section 2.5); the uniforms come from a Philox counter-based generator
    with a seed and an offset ("Attention" (cuDNN), Configurable Options:
    Dropout, Philox RNG dropout);
  * paged K/V caches: K_cache[b, h, s, d] = K_container[page_table_k[b, s / bs_k],
    h, s mod bs_k, d], likewise V, with containers (num_blocks, H, bs, D) and
    page tables (B, ceil(S / bs)): "Attention" (cuDNN), Configurable Options
    (Paged attention, Offset calculation) and Tensors (Page Table K / V).

Readings where the pages are silent:
  * a fully blocked row has LSE = -inf, O = 0, dQ = 0 and contributes nothing
    to dK/dV; padded query rows (i >= seq_len_q[b]) are such rows;
  * dropout uniforms (the pages fix the rule u >= p and name a Philox
    generator with a seed and an offset, not its width or layout):
    Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers:
    as easy as 1, 2, 3", SC 2011) with key (seed mod 2^32, seed // 2^32) and
    counter (j // 8, i, b * Hq + h, offset), offset < 2^32; its four 32-bit
    words give 8 uniforms of 16 bits, word t // 2, bits 16 * (t % 2).. for key
    j = 8 * (j // 8) + t; keep iff u16 >= ceil(p * 65536) (so the drop
    probability is p rounded up to a multiple of 2^-16), scale 1 / (1 - p);
  * "row" and "column" of the band bounds are measured from the aligned
    diagonal (row i's diagonal column is i, or i + seq_len_kv - seq_len_q
    when bottom-right aligned), and the band, the padding, the additive mask
    and is_causal (top-left j <= i) all apply together;
  * the scale multiplies Q*K^T only, never the mask;
  * only -inf blocks; a finite large negative number is just a number.

Every function here is pinned by tests against the page's hand-worked
example, central differences, invariants and a library cross-check.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "default_scale", "ref_forward", "ref_backward", "ref_forward_rows", "ref_backward_rows",
    "ref_group", "causal_bias", "band_bias", "Band", "gather_paged", "ref_forward_paged",
    "philox4x32_10", "dropout_keep", "Dropout",
]

NEG_INF = -np.inf


def default_scale(E: int) -> float:
    """Default alpha = 1/sqrt(d) (course chapter, section 2.1 "Why scale?")."""
    return 1.0 / math.sqrt(E)


def _scores(q: np.ndarray, k: np.ndarray, alpha: float) -> np.ndarray:
    """S = alpha * Q K^T, [L, S] (course chapter, symbol table of section 2)."""
    return alpha * (q @ k.T)


def causal_bias(L: int, S: int) -> np.ndarray:
    """Engine-side causal mask: 0 where j <= i, -inf where j > i (top-left tril)."""
    i = np.arange(L)[:, None]
    j = np.arange(S)[None, :]
    return np.where(j <= i, 0.0, NEG_INF)


class Band:
    """Padding and diagonal-band options of one call (cuDNN "Attention" page).

    seq_len_q, seq_len_kv: per-batch actual lengths (sequences of B ints) or
    None for "the full length"; alignment: "top_left" or "bottom_right";
    right_bound: None or an int >= 0 (0 = causal about the aligned
    diagonal); left_bound: None or an int >= 1 (a window of left_bound keys
    ending at the diagonal).
    """

    def __init__(self, seq_len_q=None, seq_len_kv=None, alignment="top_left", right_bound=None,
                 left_bound=None):
        if alignment not in ("top_left", "bottom_right"):
            raise ValueError("alignment is top_left or bottom_right")
        if right_bound is not None and right_bound < 0:
            raise ValueError("right_bound must be >= 0")
        if left_bound is not None and left_bound < 1:
            raise ValueError("left_bound must be >= 1")
        self.seq_len_q = None if seq_len_q is None else [int(x) for x in seq_len_q]
        self.seq_len_kv = None if seq_len_kv is None else [int(x) for x in seq_len_kv]
        self.alignment, self.right_bound, self.left_bound = alignment, right_bound, left_bound

    def lengths(self, b, L, S):
        Lb = L if self.seq_len_q is None else min(max(self.seq_len_q[b], 0), L)
        Sb = S if self.seq_len_kv is None else min(max(self.seq_len_kv[b], 0), S)
        return Lb, Sb


def band_bias(L: int, S: int, band: "Band", b: int) -> np.ndarray:
    """0 where key j is visible to query i of batch b, -inf where it is masked.

    Padding: rows i >= seq_len_q[b] and columns j >= seq_len_kv[b] are
    masked.  The aligned diagonal of row i is column i (top-left) or
    i + seq_len_kv[b] - seq_len_q[b] (bottom-right).  Right bound r: columns
    beyond diagonal + r are masked; left bound w: columns at or before
    diagonal - w are masked.
    """
    Lb, Sb = band.lengths(b, L, S)
    i = np.arange(L)[:, None]
    j = np.arange(S)[None, :]
    diag = i + (Sb - Lb if band.alignment == "bottom_right" else 0)
    visible = (i < Lb) & (j < Sb)
    if band.right_bound is not None:
        visible &= j <= diag + band.right_bound
    if band.left_bound is not None:
        visible &= j > diag - band.left_bound
    return np.where(visible, 0.0, NEG_INF)


# ------------------------------------------------------------------ dropout
_PHILOX_M = (0xD2511F53, 0xCD9E8D57)   # round multipliers
_PHILOX_W = (0x9E3779B9, 0xBB67AE85)   # key increments (Weyl sequence)
_M32 = (1 << 32) - 1
_M64 = (1 << 64) - 1


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds on one 128-bit counter (Python integers, exact).

    A round multiplies counter words 0 and 2 by the two multipliers (64-bit
    products split into high and low halves), mixes the high halves with
    words 1, 3 and the key, and bumps the key by the Weyl constants.
    """
    c = [int(x) & _M32 for x in counter]
    k = [int(x) & _M32 for x in key]
    for _ in range(10):
        p0 = _PHILOX_M[0] * c[0]
        p1 = _PHILOX_M[1] * c[2]
        c = [(p1 >> 32) ^ c[1] ^ k[0], p1 & _M32, (p0 >> 32) ^ c[3] ^ k[1], p0 & _M32]
        k = [(k[0] + _PHILOX_W[0]) & _M32, (k[1] + _PHILOX_W[1]) & _M32]
    return c


def _philox_arrays(c0, c1, c2, c3, k0, k1):
    """philox4x32_10 applied elementwise to counter arrays (same arithmetic, vectorised:
    a 32 x 32-bit product is exact in uint64)."""
    m32 = np.uint64(_M32)
    c = [np.asarray(x, dtype=np.uint64) & m32 for x in (c0, c1, c2, c3)]
    k = [np.uint64(k0 & _M32), np.uint64(k1 & _M32)]
    for _ in range(10):
        p0 = c[0] * np.uint64(_PHILOX_M[0])
        p1 = c[2] * np.uint64(_PHILOX_M[1])
        c = [(p1 >> np.uint64(32)) ^ c[1] ^ k[0], p1 & m32, (p0 >> np.uint64(32)) ^ c[3] ^ k[1], p0 & m32]
        k = [(k[0] + np.uint64(_PHILOX_W[0])) & m32, (k[1] + np.uint64(_PHILOX_W[1])) & m32]
    return c


class Dropout:
    """Attention dropout of one call: probability p in [0, 1), 64-bit seed, 32-bit offset."""

    def __init__(self, p: float, seed: int, offset: int = 0):
        if not (0.0 <= p < 1.0):
            raise ValueError("dropout probability must be in [0, 1)")
        if not (0 <= int(offset) <= _M32):
            raise ValueError("dropout offset must be in [0, 2^32)")
        self.p, self.seed, self.offset = float(p), int(seed) & _M64, int(offset)

    def threshold16(self) -> int:
        """Uniforms below this 16-bit value drop their weight: ceil(p * 2^16)."""
        return int(math.ceil(self.p * 65536.0))


def dropout_keep(dropout: "Dropout", bh: int, rows, S: int) -> np.ndarray:
    """keep[r, j] for query rows `rows` of head bh (= b * Hq + h) and keys 0..S-1."""
    rows = np.asarray(rows, dtype=np.int64)
    ngroups = (S + 7) // 8
    g = np.arange(ngroups, dtype=np.uint64)[None, :]
    i = rows.astype(np.uint64)[:, None]
    shape = (len(rows), ngroups)
    w = _philox_arrays(np.broadcast_to(g, shape), np.broadcast_to(i, shape), np.full(shape, bh, np.uint64),
                       np.full(shape, dropout.offset, np.uint64), dropout.seed & _M32, dropout.seed >> 32)
    u16 = np.empty((len(rows), ngroups * 8), dtype=np.uint64)
    for t in range(8):
        u16[:, t::8] = (w[t // 2] >> np.uint64(16 * (t % 2))) & np.uint64(0xFFFF)
    return u16[:, :S] >= np.uint64(dropout.threshold16())


def _masked_softmax(s: np.ndarray, bias: np.ndarray):
    """Row softmax of s + bias over the keys, stable, all -inf rows -> zeros.

    Returns (P, lse) with lse_i = m_i + ln(sum_j exp(t_ij - m_i)) and -inf
    for a row with every key blocked (course chapter, section 2.2; cuDNN
    "Attention" page, stats).
    """
    t = s + bias
    m = t.max(axis=1)
    open_row = np.isfinite(m)
    m_safe = np.where(open_row, m, 0.0)
    e = np.exp(t - m_safe[:, None])            # exp(-inf) = 0 exactly
    z = e.sum(axis=1)
    P = np.zeros_like(t)
    P[open_row] = e[open_row] / z[open_row, None]
    lse = np.full(t.shape[0], NEG_INF)
    lse[open_row] = m[open_row] + np.log(z[open_row])
    return P, lse


def _row_D(P: np.ndarray, dP: np.ndarray) -> np.ndarray:
    """D_i = sum_j P_ij dP_ij (course chapter, section 2.3)."""
    return (P * dP).sum(axis=1)


def _softmax_vjp(P: np.ndarray, dP: np.ndarray, D: np.ndarray) -> np.ndarray:
    """dS = P o (dP - D) (course chapter, section 2.3)."""
    return P * (dP - D[:, None])


def _dq(dS: np.ndarray, k: np.ndarray, alpha: float) -> np.ndarray:
    """dQ = alpha dS K (course chapter, section 2.3)."""
    return alpha * (dS @ k)


def _dk(dS: np.ndarray, q: np.ndarray, alpha: float) -> np.ndarray:
    """dK = alpha dS^T Q (course chapter, section 2.3; note the transpose)."""
    return alpha * (dS.T @ q)


def _as64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):                   # a torch tensor (bf16 is upcast exactly)
        x = x.detach().to("cpu")
        import torch  # local: only to read the tensor's values
        x = x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _check_shapes(q, k, v, mask, enable_gqa):
    B, Hq, L, E = q.shape
    Bk, Hkv, S, Ek = k.shape
    if k.ndim != 4 or q.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, T, D]")
    if Bk != B or v.shape[0] != B:
        raise ValueError("batch sizes differ")
    if Ek != E:
        raise ValueError("q and k widths differ")
    if v.shape[1] != Hkv or v.shape[2] != S:
        raise ValueError("k and v disagree on heads or length")
    if Hq != Hkv and not enable_gqa:
        raise ValueError("Hq != Hkv needs enable_gqa")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if mask is not None:
        if mask.ndim != 4 or mask.shape[2:] != (L, S) or mask.shape[0] not in (1, B) \
                or mask.shape[1] not in (1, Hq):
            raise ValueError("mask must be [B|1, Hq|1, L, S]")
    return B, Hq, Hkv, L, S, E, v.shape[3]


def _head_bias(mask, b, h, L, S, is_causal, band=None):
    bias = np.zeros((L, S))
    if mask is not None:
        bias = bias + mask[min(b, mask.shape[0] - 1), min(h, mask.shape[1] - 1)]
    if is_causal:
        bias = bias + causal_bias(L, S)
    if band is not None:
        bias = bias + band_bias(L, S, band, b)
    return bias


def _alpha(scale, E):
    if scale is None:
        return default_scale(E)
    if not (scale >= 0.0) or math.isinf(scale):
        raise ValueError("scale must be finite and >= 0")
    return float(scale)


def _head_forward(q, k, v, bias, alpha, m=None):
    """O = (P o m) V (m = None: no dropout), LSE and P (before dropout)."""
    P, lse = _masked_softmax(_scores(q, k, alpha), bias)
    return (P if m is None else P * m) @ v, lse, P


def _dropout_m(dropout, b, h, Hq, L, S):
    """m = keep / (1 - p) of head (b, h), or None without dropout (course chapter, section 2.5)."""
    if dropout is None or dropout.p == 0.0:
        return None
    return dropout_keep(dropout, b * Hq + h, np.arange(L), S) / (1.0 - dropout.p)


def ref_forward(q, k, v, mask=None, scale=None, is_causal=False, enable_gqa=False,
                return_P=False, band=None, dropout=None):
    """O [B,Hq,L,Ev] and LSE [B,Hq,L] of softmax(alpha*Q*K^T + mask + causal + band)*V.

    Query head h reads KV head h // (Hq // Hkv) (repeat_interleave).  band:
    None or a Band (padding lengths, diagonal alignment and bounds).  dropout:
    None or a Dropout; P (returned on request) and LSE are before dropout.
    """
    q, k, v, mask = _as64(q), _as64(k), _as64(v), _as64(mask)
    B, Hq, Hkv, L, S, E, Ev = _check_shapes(q, k, v, mask, enable_gqa)
    G = Hq // Hkv
    alpha = _alpha(scale, E)
    O = np.zeros((B, Hq, L, Ev))
    LSE = np.zeros((B, Hq, L))
    Ps = np.zeros((B, Hq, L, S)) if return_P else None
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            o, lse, P = _head_forward(q[b, h], k[b, kv], v[b, kv],
                                      _head_bias(mask, b, h, L, S, is_causal, band), alpha,
                                      _dropout_m(dropout, b, h, Hq, L, S))
            O[b, h], LSE[b, h] = o, lse
            if return_P:
                Ps[b, h] = P
    return (O, LSE, Ps) if return_P else (O, LSE)


def _head_backward(q, k, v, P, o, dO, alpha, m=None):
    """dQ, dK, dV, D of one head; with dropout m: dV = (P o m)^T dO, dP = (dO V^T) o m."""
    dV = (P if m is None else P * m).T @ dO
    dP = dO @ v.T
    if m is not None:
        dP = dP * m
    D = _row_D(P, dP)
    # the identity D_i = dO_i . O_i of section 2.3 must hold for the oracle's own P
    np.testing.assert_allclose(D, (dO * o).sum(axis=1), rtol=1e-9, atol=1e-9)
    dS = _softmax_vjp(P, dP, D)
    return _dq(dS, k, alpha), _dk(dS, q, alpha), dV, D


def ref_backward(q, k, v, dO, mask=None, scale=None, is_causal=False, enable_gqa=False,
                 return_D=False, band=None, dropout=None):
    """dQ [B,Hq,L,E], dK [B,Hkv,S,E], dV [B,Hkv,S,Ev] of L = sum(O * dO).

    dK and dV of a KV head are summed over the Hq/Hkv query heads that read it
    (chain rule through repeat_interleave).  P is recomputed from the
    definition, never taken from another implementation.
    """
    q, k, v, dO, mask = _as64(q), _as64(k), _as64(v), _as64(dO), _as64(mask)
    B, Hq, Hkv, L, S, E, Ev = _check_shapes(q, k, v, mask, enable_gqa)
    G = Hq // Hkv
    alpha = _alpha(scale, E)
    dQ = np.zeros((B, Hq, L, E))
    dK = np.zeros((B, Hkv, S, E))
    dV = np.zeros((B, Hkv, S, Ev))
    Dall = np.zeros((B, Hq, L))
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            bias = _head_bias(mask, b, h, L, S, is_causal, band)
            m = _dropout_m(dropout, b, h, Hq, L, S)
            o, _, P = _head_forward(q[b, h], k[b, kv], v[b, kv], bias, alpha, m)
            dq, dk, dv, D = _head_backward(q[b, h], k[b, kv], v[b, kv], P, o, dO[b, h], alpha, m)
            dQ[b, h] = dq
            dK[b, kv] += dk
            dV[b, kv] += dv
            Dall[b, h] = D
    return (dQ, dK, dV, Dall) if return_D else (dQ, dK, dV)


def ref_forward_rows(q, k, v, b, h, rows, mask=None, scale=None, is_causal=False,
                     enable_gqa=False, band=None, dropout=None):
    """O and LSE of selected query rows of one (b, h): for sampled checks of large runs.

    Each row is an independent problem (course chapter, section 2.1: every
    query is computed independently), so a row needs only its own q_i and all
    keys.
    """
    G = q.shape[1] // k.shape[1]
    kv = h // G
    rows = np.asarray(rows)
    L, S, E = q.shape[2], k.shape[2], q.shape[3]
    alpha = _alpha(scale, E)
    qh = _as64(q[b, h][rows])
    kh = _as64(k[b, kv])
    vh = _as64(v[b, kv])
    bias = np.zeros((len(rows), S))
    if mask is not None:
        m = mask[min(b, mask.shape[0] - 1), min(h, mask.shape[1] - 1)]
        bias = bias + _as64(m[rows])
    if is_causal:
        bias = bias + causal_bias(L, S)[rows]
    if band is not None:
        bias = bias + band_bias(L, S, band, b)[rows]
    P, lse = _masked_softmax(_scores(qh, kh, alpha), bias)
    if dropout is not None and dropout.p > 0.0:
        P = P * (dropout_keep(dropout, b * q.shape[1] + h, rows, S) / (1.0 - dropout.p))
    return P @ vh, lse


def ref_backward_rows(q, k, v, dO, b, h, rows, mask=None, scale=None, is_causal=False,
                      enable_gqa=False, band=None):
    """dQ of selected query rows of one (b, h): for sampled checks of large runs.

    Row i of dQ needs only row i of P, dP = dO V^T and D (course chapter,
    section 2.3: dS_i = P_i o (dP_i - D_i), D_i = sum_j P_ij dP_ij, dQ_i =
    alpha dS_i K), so, like the forward's rows, it is a closed sub-problem.
    """
    G = q.shape[1] // k.shape[1]
    kv = h // G
    rows = np.asarray(rows)
    L, S, E = q.shape[2], k.shape[2], q.shape[3]
    alpha = _alpha(scale, E)
    qh = _as64(q[b, h][rows])
    kh = _as64(k[b, kv])
    vh = _as64(v[b, kv])
    dOh = _as64(dO[b, h][rows])
    bias = np.zeros((len(rows), S))
    if mask is not None:
        m = mask[min(b, mask.shape[0] - 1), min(h, mask.shape[1] - 1)]
        bias = bias + _as64(m[rows])
    if is_causal:
        bias = bias + causal_bias(L, S)[rows]
    if band is not None:
        bias = bias + band_bias(L, S, band, b)[rows]
    P, _ = _masked_softmax(_scores(qh, kh, alpha), bias)
    dP = dOh @ vh.T
    dS = _softmax_vjp(P, dP, _row_D(P, dP))
    return _dq(dS, kh, alpha)


def ref_group(q, k, v, dO, b, kv, mask=None, scale=None, is_causal=False, band=None, dropout=None):
    """Forward and backward of the G query heads sharing KV head (b, kv).

    Returns (O [G,L,Ev], LSE [G,L], dQ [G,L,E], dK [S,E], dV [S,Ev]) for
    sampled checks of large runs: one KV group is a closed sub-problem (the
    heads are independent, course chapter section 2.1, and dK, dV of a KV head
    sum only its own group's terms, section 2.3).  Each head keeps its index
    (b, h) in the whole problem, so its padding lengths and its dropout mask
    (section 2.5) are the ones the full call draws.
    """
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    L, S, E = q.shape[2], k.shape[2], q.shape[3]
    alpha = _alpha(scale, E)
    kh, vh = _as64(k[b, kv]), _as64(v[b, kv])
    mg = None if mask is None else _as64(mask[min(b, mask.shape[0] - 1)])      # [mask_h, L, S]
    O, LSE, dQ = [], [], []
    dK, dV = np.zeros((S, E)), np.zeros((S, vh.shape[1]))
    for h in range(kv * G, (kv + 1) * G):
        bias = np.zeros((L, S))
        if mg is not None:
            bias = bias + mg[min(h, mg.shape[0] - 1)]
        if is_causal:
            bias = bias + causal_bias(L, S)
        if band is not None:
            bias = bias + band_bias(L, S, band, b)
        m = _dropout_m(dropout, b, h, Hq, L, S)
        qh = _as64(q[b, h])
        o, lse, P = _head_forward(qh, kh, vh, bias, alpha, m)
        O.append(o)
        LSE.append(lse)
        if dO is not None:
            dq, dk, dv, _ = _head_backward(qh, kh, vh, P, o, _as64(dO[b, h]), alpha, m)
            dQ.append(dq)
            dK += dk
            dV += dv
    out = [np.stack(O), np.stack(LSE)]
    if dO is not None:
        out += [np.stack(dQ), dK, dV]
    return tuple(out)


def gather_paged(container, page_table, block_size: int, S: int) -> np.ndarray:
    """Dense cache [B, H, S, D] of a paged container [num_blocks, H, block_size, D].

    cache[b, h, s, d] = container[page_table[b, s // block_size], h, s % block_size, d]
    (cuDNN "Attention", Paged attention, Offset calculation).  A table entry
    outside [0, num_blocks), or a block index past the table's width, gives
    zeros: such positions lie past the sequence's length and are masked.
    """
    c = _as64(container)
    table = np.asarray(page_table.cpu() if hasattr(page_table, "cpu") else page_table, dtype=np.int64)
    nb, H, bs, D = c.shape
    if bs != block_size:
        raise ValueError("container block size differs from block_size")
    B = table.shape[0]
    out = np.zeros((B, H, S, D))
    for b in range(B):
        for s in range(S):
            blk = s // block_size
            if blk >= table.shape[1]:
                continue
            page = int(table[b, blk])
            if 0 <= page < nb:
                out[b, :, s, :] = c[page, :, s % block_size, :]
    return out


def ref_forward_paged(q, k_container, v_container, page_table_k, page_table_v, block_size_k: int,
                      block_size_v: int, S: int, mask=None, scale=None, enable_gqa=False, band=None):
    """Forward (O, LSE) with paged K/V: the plain forward on the gathered caches."""
    k = gather_paged(k_container, page_table_k, block_size_k, S)
    v = gather_paged(v_container, page_table_v, block_size_v, S)
    return ref_forward(q, k, v, mask, scale, False, enable_gqa, band=band)
