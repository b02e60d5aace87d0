"""Pins of the oracle's padding and diagonal-band options.

The options come from the cuDNN "Attention" page (Configurable Options:
Padding mask, Diagonal masking options; Scaled Dot Product Attention, Args
seq_len_q, seq_len_kv, diagonal_alignment, diagonal_band_left_bound,
diagonal_band_right_bound).  None of the checks below retypes the band rule:
each one reduces a banded or padded problem to the plain (or plain causal)
oracle on a sliced or shifted problem, uses a closed form, an invariant, or
central differences.  ``test_band_mutants_are_caught`` plants plausible
mistakes in ``band_bias`` and checks that a pin fails for each.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import sdpa_oracle as so
from workloads import random_inputs

Band = oracle.Band


def _np(x):
    return None if x is None else x.to(torch.float64).numpy()


def _inputs(B, Hq, Hkv, L, S, E, Ev, seed):
    q, k, v, dO, _ = random_inputs(B, Hq, Hkv, L, S, E, Ev, torch.float64, seed=seed)
    return _np(q), _np(k), _np(v), _np(dO)


def pin_padding_is_truncation():
    """Padded batches equal the unpadded problems cut to their lengths (the page's
    example batch "aa" / "bbb" with max length 8 is the first case)."""
    cases = [
        # B, Hq, Hkv, L, S, E, Ev, seq_len_q, seq_len_kv, causal
        (2, 1, 1, 8, 8, 4, 3, [2, 3], [2, 3], False),
        (3, 4, 2, 7, 9, 5, 3, [2, 7, 5], [3, 9, 4], True),
        (2, 2, 2, 6, 5, 3, 2, [0, 4], [5, 0], False),
    ]
    for n, (B, Hq, Hkv, L, S, E, Ev, lq, lk, causal) in enumerate(cases):
        q, k, v, dO = _inputs(B, Hq, Hkv, L, S, E, Ev, 40 + n)
        band = Band(lq, lk)
        gqa = Hq != Hkv
        O, LSE = oracle.ref_forward(q, k, v, None, 0.4, causal, gqa, band=band)
        dQ, dK, dV = oracle.ref_backward(q, k, v, dO, None, 0.4, causal, gqa, band=band)
        for b in range(B):
            Lb, Sb = lq[b], lk[b]
            # padded query rows, and every row of a batch without keys: zeros, LSE -inf
            dead = slice(Lb, L) if Sb > 0 else slice(0, L)
            assert np.all(O[b, :, dead] == 0.0) and np.all(np.isneginf(LSE[b, :, dead]))
            assert np.all(dQ[b, :, dead] == 0.0)
            assert np.all(dK[b, :, Sb:] == 0.0) and np.all(dV[b, :, Sb:] == 0.0)
            if Lb == 0 or Sb == 0:
                assert np.all(dK[b] == 0.0) and np.all(dV[b] == 0.0)
                continue
            sl = (slice(b, b + 1), slice(None))
            qt, kt, vt, dOt = q[sl][:, :, :Lb], k[sl][:, :, :Sb], v[sl][:, :, :Sb], dO[sl][:, :, :Lb]
            Ot, LSEt = oracle.ref_forward(qt, kt, vt, None, 0.4, causal, gqa)
            dQt, dKt, dVt = oracle.ref_backward(qt, kt, vt, dOt, None, 0.4, causal, gqa)
            np.testing.assert_allclose(O[b, :, :Lb], Ot[0], atol=1e-13)
            np.testing.assert_allclose(LSE[b, :, :Lb], LSEt[0], atol=1e-13)
            np.testing.assert_allclose(dQ[b, :, :Lb], dQt[0], atol=1e-13)
            np.testing.assert_allclose(dK[b, :, :Sb], dKt[0], atol=1e-13)
            np.testing.assert_allclose(dV[b, :, :Sb], dVt[0], atol=1e-13)


def pin_bottom_right_is_suffix_of_top_left():
    """Bottom-right causal (prefix-LM / decode diagonal): the L query rows are the
    last L rows of a top-left causal problem with as many queries as keys; with
    padding, the last seq_len_q rows of one with seq_len_kv queries."""
    B, Hq, Hkv, L, S, E, Ev = 2, 2, 1, 5, 9, 4, 3
    q, k, v, _ = _inputs(B, Hq, Hkv, L, S, E, Ev, 50)
    rng = np.random.default_rng(51)
    pre = rng.standard_normal((B, Hq, S - L, E))            # arbitrary earlier queries
    qfull = np.concatenate([pre, q], axis=2)
    O, LSE = oracle.ref_forward(q, k, v, None, 0.5, False, True, band=Band(alignment="bottom_right", right_bound=0))
    Of, LSEf = oracle.ref_forward(qfull, k, v, None, 0.5, True, True)
    np.testing.assert_allclose(O, Of[:, :, S - L:], atol=1e-13)
    np.testing.assert_allclose(LSE, LSEf[:, :, S - L:], atol=1e-13)
    # L == S: bottom-right and top-left coincide
    q2, k2, v2, _ = _inputs(1, 1, 1, 6, 6, 3, 2, 52)
    a = oracle.ref_forward(q2, k2, v2, None, 0.5, False, band=Band(alignment="bottom_right", right_bound=0))
    c = oracle.ref_forward(q2, k2, v2, None, 0.5, True)
    np.testing.assert_allclose(a[0], c[0], atol=1e-14)
    # with padding: aligned to the actual lengths.  Row i sees keys j <= i + Sb - Lb:
    # Sb >= Lb is the suffix of a top-left problem with Sb - Lb earlier queries;
    # Sb < Lb leaves the first Lb - Sb rows without keys and the rest top-left causal.
    lq, lk = [3, 5], [7, 4]
    O, LSE = oracle.ref_forward(q, k, v, None, 0.5, False, True,
                                band=Band(lq, lk, alignment="bottom_right", right_bound=0))
    for b in range(B):
        Lb, Sb = lq[b], lk[b]
        kb, vb = k[b:b + 1, :, :Sb], v[b:b + 1, :, :Sb]
        if Sb >= Lb:
            qq = np.concatenate([pre[b:b + 1, :, :Sb - Lb], q[b:b + 1, :, :Lb]], axis=2)
            Oc, Lc = oracle.ref_forward(qq, kb, vb, None, 0.5, True, True)
            np.testing.assert_allclose(O[b, :, :Lb], Oc[0, :, Sb - Lb:], atol=1e-13)
            np.testing.assert_allclose(LSE[b, :, :Lb], Lc[0, :, Sb - Lb:], atol=1e-13)
        else:
            assert np.all(O[b, :, :Lb - Sb] == 0.0) and np.all(np.isneginf(LSE[b, :, :Lb - Sb]))
            Oc, Lc = oracle.ref_forward(q[b:b + 1, :, Lb - Sb:Lb], kb, vb, None, 0.5, True, True)
            np.testing.assert_allclose(O[b, :, Lb - Sb:Lb], Oc[0], atol=1e-13)
            np.testing.assert_allclose(LSE[b, :, Lb - Sb:Lb], Lc[0], atol=1e-13)
        assert np.all(O[b, :, Lb:] == 0.0)


def pin_right_bound_is_shifted_causal():
    """Right bound r: row i sees the keys causal row i + r would see; r = 0 is
    is_causal; r >= S removes the bound."""
    B, Hq, L, S, E, Ev, r = 1, 2, 5, 8, 3, 2, 2
    q, k, v, _ = _inputs(B, Hq, Hq, L, S, E, Ev, 60)
    pre = np.random.default_rng(61).standard_normal((B, Hq, r, E))
    O, _ = oracle.ref_forward(q, k, v, None, 0.7, band=Band(right_bound=r))
    Oc, _ = oracle.ref_forward(np.concatenate([pre, q], axis=2), k, v, None, 0.7, True)
    np.testing.assert_allclose(O, Oc[:, :, r:], atol=1e-13)
    a = oracle.ref_forward(q, k, v, None, 0.7, band=Band(right_bound=0))
    c = oracle.ref_forward(q, k, v, None, 0.7, True)
    np.testing.assert_allclose(a[0], c[0], atol=1e-14)
    a = oracle.ref_forward(q, k, v, None, 0.7, band=Band(right_bound=S))
    c = oracle.ref_forward(q, k, v, None, 0.7)
    np.testing.assert_allclose(a[0], c[0], atol=1e-14)


def pin_left_bound_window():
    """Causal window of w keys: row i equals plain attention over keys
    max(0, i-w+1)..i; w = 1 gives O_i = v_i and LSE_i = alpha q_i.k_i; a window
    wider than the sequence changes nothing."""
    B, Hq, L, S, E, Ev, w, alpha = 1, 2, 7, 7, 4, 3, 3, 0.6
    q, k, v, _ = _inputs(B, Hq, Hq, L, S, E, Ev, 70)
    O, LSE = oracle.ref_forward(q, k, v, None, alpha, True, band=Band(left_bound=w))
    for i in range(L):
        lo = max(0, i - w + 1)
        Oi, Li = oracle.ref_forward(q[:, :, i:i + 1], k[:, :, lo:i + 1], v[:, :, lo:i + 1], None, alpha)
        np.testing.assert_allclose(O[:, :, i], Oi[:, :, 0], atol=1e-13)
        np.testing.assert_allclose(LSE[:, :, i], Li[:, :, 0], atol=1e-13)
    O1, L1 = oracle.ref_forward(q, k, v, None, alpha, True, band=Band(left_bound=1))
    np.testing.assert_allclose(O1, v, atol=1e-13)
    np.testing.assert_allclose(L1, alpha * (q * k).sum(-1), atol=1e-13)
    a = oracle.ref_forward(q, k, v, None, alpha, True, band=Band(left_bound=L + S))
    c = oracle.ref_forward(q, k, v, None, alpha, True)
    np.testing.assert_allclose(a[0], c[0], atol=1e-14)


def pin_window_locality():
    """With a bottom-right band, changing keys/values outside a row's band leaves
    that row's output unchanged; changing one inside changes it."""
    L, S, E = 4, 10, 3
    q, k, v, _ = _inputs(1, 1, 1, L, S, E, E, 80)
    band = Band(alignment="bottom_right", right_bound=1, left_bound=3)
    O, _ = oracle.ref_forward(q, k, v, None, 0.5, band=band)
    for i in range(L):
        d = i + S - L
        inside = [j for j in range(S) if d - 3 < j <= d + 1]
        outside = [j for j in range(S) if j not in inside]
        k2, v2 = k.copy(), v.copy()
        k2[0, 0, outside] += 3.0
        v2[0, 0, outside] -= 2.0
        O2, _ = oracle.ref_forward(q, k2, v2, None, 0.5, band=band)
        np.testing.assert_allclose(O2[0, 0, i], O[0, 0, i], atol=1e-14)
        v3 = v.copy()
        v3[0, 0, inside[0]] += 1.0
        O3, _ = oracle.ref_forward(q, k, v3, None, 0.5, band=band)
        assert np.abs(O3[0, 0, i] - O[0, 0, i]).max() > 1e-6


def pin_band_gradcheck():
    """Central differences of sum(O * g) under padding, bottom-right alignment and both bounds."""
    B, Hq, Hkv, L, S, E, Ev = 2, 2, 1, 4, 6, 3, 2
    q, k, v, dO = _inputs(B, Hq, Hkv, L, S, E, Ev, 90)
    band = Band([3, 4], [5, 6], alignment="bottom_right", right_bound=1, left_bound=3)
    dQ, dK, dV = oracle.ref_backward(q, k, v, dO, None, 0.45, False, True, band=band)

    def f(qq, kk, vv):
        O, _ = oracle.ref_forward(qq, kk, vv, None, 0.45, False, True, band=band)
        return float((O * dO).sum())
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


BAND_PINS = [pin_padding_is_truncation, pin_bottom_right_is_suffix_of_top_left, pin_right_bound_is_shifted_causal,
             pin_left_bound_window, pin_window_locality, pin_band_gradcheck]


@pytest.mark.parametrize("pin", BAND_PINS, ids=[p.__name__ for p in BAND_PINS])
def test_band_pin(pin):
    pin()


# --------------------------------------------------------------------------- mutants
def _mutant(kind):
    def band_bias(L, S, band, b):
        Lb, Sb = band.lengths(b, L, S)
        i = np.arange(L)[:, None]
        j = np.arange(S)[None, :]
        off = Sb - Lb if band.alignment == "bottom_right" else 0
        if kind == "br_offset_sign":
            off = -off
        diag = i + off
        visible = (j < Sb) if kind == "pad_rows_open" else (i < Lb) & (j < Sb)
        if kind == "pad_keys_open":
            visible = i < Lb
        if band.right_bound is not None:
            visible &= (j < diag + band.right_bound) if kind == "right_strict" else (j <= diag + band.right_bound)
        if band.left_bound is not None:
            visible &= (j >= diag - band.left_bound) if kind == "left_inclusive" else (j > diag - band.left_bound)
        if kind == "br_uses_max_lengths" and band.alignment == "bottom_right":
            visible = (i < Lb) & (j < Sb)
            diag = i + (S - L)
            if band.right_bound is not None:
                visible &= j <= diag + band.right_bound
            if band.left_bound is not None:
                visible &= j > diag - band.left_bound
        return np.where(visible, 0.0, -np.inf)
    return band_bias


BAND_MUTANTS = ["br_offset_sign", "pad_rows_open", "pad_keys_open", "right_strict", "left_inclusive",
                "br_uses_max_lengths"]


@pytest.mark.parametrize("kind", BAND_MUTANTS)
def test_band_mutants_are_caught(kind, monkeypatch):
    monkeypatch.setattr(so, "band_bias", _mutant(kind))
    failed = []
    for pin in BAND_PINS:
        try:
            pin()
        except Exception:   # noqa: BLE001 - any failure counts as caught
            failed.append(pin.__name__)
    assert failed, f"band mutant {kind} survived every pin"


def test_band_rejects_bad_options():
    with pytest.raises(ValueError):
        Band(alignment="middle")
    with pytest.raises(ValueError):
        Band(right_bound=-1)
    with pytest.raises(ValueError):
        Band(left_bound=0)
