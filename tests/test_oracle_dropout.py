"""Pins of the oracle's attention dropout (course chapter "Scaled dot-product
attention (forward and backward)", section 2.5; cuDNN "Attention", Philox RNG
dropout).

The generator (Philox4x32-10) is pinned against Triton's own Philox run by its
CPU interpreter (an independent library implementation of the same function),
the vectorised path against the scalar one, the mask layout against the
documented counter rule; the dropout math by
p = 0 reducing to the plain oracle, the kept fraction, unbiasedness over
seeds, and central differences with the mask replayed.  The chapter's three
dropout pitfalls (s07: dV ignores the mask, s08: dP ignores it, s09: keeping
u < p) are planted and each is caught.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from oracle import sdpa_oracle as so
from workloads import random_inputs

M32 = (1 << 32) - 1

# Triton's Philox (triton.language.philox: 32-bit counter words, key = the 64-bit seed's
# low and high halves, 10 rounds) evaluated by Triton's CPU interpreter in a child process.
_TRITON_PHILOX = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl

@triton.jit
def _philox_kernel(out, c0p, c1p, c2p, c3p, seed, N: tl.constexpr):
    n = tl.arange(0, N)
    r0, r1, r2, r3 = tl.philox(seed, tl.load(c0p + n), tl.load(c1p + n), tl.load(c2p + n), tl.load(c3p + n), 10)
    tl.store(out + 4 * n, r0)
    tl.store(out + 4 * n + 1, r1)
    tl.store(out + 4 * n + 2, r2)
    tl.store(out + 4 * n + 3, r3)

res = []
for ctrs, seed in json.loads(sys.stdin.read()):
    cols = [torch.tensor([c[w] for c in ctrs], dtype=torch.int64).to(torch.uint32) for w in range(4)]
    out = torch.zeros(4 * len(ctrs), dtype=torch.uint32)
    _philox_kernel[(1,)](out, *cols, seed, N=len(ctrs))
    res.append([int(x) & 0xFFFFFFFF for x in out.to(torch.int64)])
print(json.dumps(res))
"""


def _np(x):
    return None if x is None else x.to(torch.float64).numpy()


def pin_philox_matches_triton():
    pytest.importorskip("triton")
    rng = np.random.default_rng(5)
    ctrs = [[0, 0, 0, 0], [1, 0, 0, 0], [0, 1, 2, 3], [M32, M32, M32, M32], [7, 3, 99, 2 ** 31 + 5]]
    ctrs += [[int(x) for x in rng.integers(0, 2 ** 32, 4)] for _ in range(3)]
    seeds = [0, 123456789, 2 ** 40 + 7, 2 ** 63 + 12345]
    env = dict(os.environ, TRITON_INTERPRET="1")
    got = subprocess.run([sys.executable, "-c", _TRITON_PHILOX], input=json.dumps([[ctrs, sd] for sd in seeds]),
                         capture_output=True, text=True, env=env, timeout=300, check=True)
    words = json.loads(got.stdout.strip().splitlines()[-1])
    for sd, w in zip(seeds, words):
        for n, ctr in enumerate(ctrs):
            assert w[4 * n:4 * n + 4] == oracle.philox4x32_10(ctr, [sd & M32, sd >> 32]), (ctr, sd)


def pin_vectorised_philox_matches_scalar():
    rng = np.random.default_rng(6)
    c = rng.integers(0, 2 ** 32, (4, 64), dtype=np.int64).astype(np.uint64)
    c[0, :3] = [0, M32, 2 ** 31]
    k0, k1 = 0xFEDCBA98, 42
    w = so._philox_arrays(c[0], c[1], c[2], c[3], k0, k1)
    for n in range(c.shape[1]):
        assert [int(w[t][n]) for t in range(4)] == oracle.philox4x32_10([int(x) for x in c[:, n]], [k0, k1])


def pin_mask_layout():
    """keep(i, j) of head bh: 16-bit chunk j % 8 of Philox((j // 8, i, bh, offset), seed) >= ceil(p 2^16)."""
    seed = 2 ** 40 + 7
    d = oracle.Dropout(0.37, seed=seed, offset=12345)
    keep = oracle.dropout_keep(d, 5, [0, 3, 17], 40)
    thr = int(np.ceil(0.37 * 65536))
    for r, i in enumerate([0, 3, 17]):
        for j in range(40):
            words = oracle.philox4x32_10([j // 8, i, 5, 12345], [seed & M32, seed >> 32])
            u = (words[(j % 8) // 2] >> (16 * (j % 2))) & 0xFFFF
            assert keep[r, j] == (u >= thr)


def pin_p_zero_is_plain():
    q, k, v, dO, mask = random_inputs(2, 4, 2, 9, 11, 5, 3, torch.float64, seed=60, mask_kind="bias", p_block=0.2)
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    d = oracle.Dropout(0.0, seed=1)
    a = oracle.ref_forward(q, k, v, mask, 0.4, True, True, dropout=d)
    b = oracle.ref_forward(q, k, v, mask, 0.4, True, True)
    np.testing.assert_array_equal(a[0], b[0])
    ga = oracle.ref_backward(q, k, v, dO, mask, 0.4, True, True, dropout=d)
    gb = oracle.ref_backward(q, k, v, dO, mask, 0.4, True, True)
    for x, y in zip(ga, gb):
        np.testing.assert_array_equal(x, y)


def pin_keep_fraction():
    for p in (0.1, 0.3, 0.7):
        keep = oracle.dropout_keep(oracle.Dropout(p, seed=11, offset=3), 2, np.arange(64), 4096)
        n = keep.size
        want = 1.0 - np.ceil(p * 65536) / 65536
        assert abs(keep.mean() - want) < 5 * np.sqrt(want * (1 - want) / n)


def pin_unbiased_over_seeds():
    """E_m[(P o m) V] = P V: the mean over 200 seeds approaches the plain output."""
    q, k, v, _, _ = random_inputs(1, 1, 1, 6, 40, 4, 3, torch.float64, seed=61)
    q, k, v = _np(q), _np(k), _np(v)
    O, _ = oracle.ref_forward(q, k, v, None, 0.5)
    acc = np.zeros_like(O)
    for s in range(200):
        acc += oracle.ref_forward(q, k, v, None, 0.5, dropout=oracle.Dropout(0.25, seed=s))[0]
    assert np.abs(acc / 200 - O).max() < 0.06


def pin_dropout_gradcheck():
    """Central differences of sum(O * g) with the mask replayed (fixed seed and offset)."""
    q, k, v, dO, mask = random_inputs(1, 2, 1, 5, 7, 3, 2, torch.float64, seed=62, mask_kind="bias", p_block=0.2)
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    d = oracle.Dropout(0.4, seed=9, offset=2)
    dQ, dK, dV = oracle.ref_backward(q, k, v, dO, mask, 0.6, True, True, dropout=d)

    def f(qq, kk, vv):
        return float((oracle.ref_forward(qq, kk, vv, mask, 0.6, True, True, dropout=d)[0] * dO).sum())
    h = 1e-6
    for x, g in ((q, dQ), (k, dK), (v, dV)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            fp = f(q, k, v)
            x[idx] = old - h
            fm = f(q, k, v)
            x[idx] = old
            fd[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(g, fd, atol=2e-7, rtol=1e-6)


def pin_identity_values_show_the_mask():
    """With V = I, O = P o m: zero exactly where dropped, P / (1 - p) where kept."""
    S = 24
    q, k, _, _, _ = random_inputs(1, 1, 1, 5, S, 4, 4, torch.float64, seed=63)
    q, k = _np(q), _np(k)
    v = np.eye(S)[None, None]
    d = oracle.Dropout(0.3, seed=4)
    O, _, P = oracle.ref_forward(q, k, v, None, 0.5, return_P=True, dropout=d)
    keep = oracle.dropout_keep(d, 0, np.arange(5), S)
    np.testing.assert_allclose(O[0, 0], np.where(keep, P[0, 0] / 0.7, 0.0), atol=1e-15)


DROPOUT_PINS = [pin_philox_matches_triton, pin_vectorised_philox_matches_scalar, pin_mask_layout, pin_p_zero_is_plain,
                pin_keep_fraction, pin_unbiased_over_seeds, pin_dropout_gradcheck, pin_identity_values_show_the_mask]


@pytest.mark.parametrize("pin", DROPOUT_PINS, ids=[p.__name__ for p in DROPOUT_PINS])
def test_dropout_pin(pin):
    pin()


def _m_dv_ignores_mask(q, k, v, P, o, dO, alpha, m=None):
    dq, dk, _, D = _orig_backward(q, k, v, P, o, dO, alpha, m)
    return dq, dk, P.T @ dO, D


def _m_dp_ignores_mask(q, k, v, P, o, dO, alpha, m=None):
    dV = (P if m is None else P * m).T @ dO
    dP = dO @ v.T
    D = (dO * o).sum(axis=1)
    dS = P * (dP - D[:, None])
    return alpha * (dS @ k), alpha * (dS.T @ q), dV, D


def _m_keep_below_p(dropout, bh, rows, S):
    return ~_orig_keep(dropout, bh, rows, S)


_orig_backward = so._head_backward
_orig_keep = so.dropout_keep
DROPOUT_MUTANTS = {"s07_dv_ignores_mask": ("_head_backward", _m_dv_ignores_mask),
                   "s08_dp_ignores_mask": ("_head_backward", _m_dp_ignores_mask),
                   "s09_keep_u_below_p": ("dropout_keep", _m_keep_below_p)}


@pytest.mark.parametrize("name", sorted(DROPOUT_MUTANTS))
def test_dropout_mutants_are_caught(name, monkeypatch):
    attr, fn = DROPOUT_MUTANTS[name]
    monkeypatch.setattr(so, attr, fn)
    if attr == "dropout_keep":
        monkeypatch.setattr(oracle, "dropout_keep", fn)
    failed = []
    for pin in DROPOUT_PINS:
        try:
            pin()
        except Exception:   # noqa: BLE001 - any failure counts as caught
            failed.append(pin.__name__)
    assert failed, f"dropout mutant {name} survived every pin"


def test_dropout_rejects_bad_probability_and_offset():
    for p in (-0.1, 1.0, 1.5):
        with pytest.raises(ValueError):
            oracle.Dropout(p, seed=0)
    for off in (-1, 2 ** 32):
        with pytest.raises(ValueError):
            oracle.Dropout(0.1, seed=0, offset=off)
