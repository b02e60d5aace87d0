"""Pins of the float64 oracle against what the pages and mathematics fix.

Nothing here retypes the oracle's formulas: every check is either a value
printed on a page (the hand-worked example), central differences, a closed
form, an invariant, a reduction to a simpler case, or an independent library
routine (torch's CPU float64 attention).  ``test_mutants_are_caught`` plants
each applicable pitfall of the course chapter "Scaled dot-product attention
(forward and backward)", section 5, into the oracle and checks that at least
one pin fails, so the pins have teeth.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import sdpa_oracle as so
from workloads import random_inputs

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "hand_example.json")


def _np(x):
    return None if x is None else x.to(torch.float64).numpy()


def _hand():
    with open(GOLDEN) as f:
        g = json.load(f)
    q = np.array(g["q"], float)[None, None]
    k = np.array(g["k"], float)[None, None]
    v = np.array(g["v"], float)[None, None]
    dO = np.array(g["dO"], float)[None, None]
    return g, q, k, v, dO


# --------------------------------------------------------------------------- pins
# Each pin is a plain function raising on failure, so the mutant test can run
# all of them under a planted mistake.

def pin_hand_forward():
    """Course chapter section 3: P and O of the worked example (default scale 1/sqrt(4))."""
    g, q, k, v, _ = _hand()
    O, LSE, P = oracle.ref_forward(q, k, v, scale=None, return_P=True)
    tol = 0.5 * 10.0 ** -g["printed_decimals"] + 1e-12
    np.testing.assert_allclose(P[0, 0], np.array(g["P"]), atol=tol, rtol=0)
    np.testing.assert_allclose(O[0, 0], np.array(g["O"]), atol=tol, rtol=0)
    # printed normaliser 11.107 (3 decimals): lse = ln(normaliser) within its rounding
    assert abs(LSE[0, 0, 0] - math.log(g["normaliser"])) < 0.0005 / g["normaliser"] + 1e-12


def pin_hand_backward():
    """Course chapter section 3: dV, D, dQ, dK of the worked example with dO = (1, 0)."""
    g, q, k, v, dO = _hand()
    dQ, dK, dV, D = oracle.ref_backward(q, k, v, dO, scale=None, return_D=True)
    tol = 0.5 * 10.0 ** -g["printed_decimals"] + 1e-12
    np.testing.assert_allclose(dV[0, 0], np.array(g["dV"]), atol=tol, rtol=0)
    np.testing.assert_allclose(D[0, 0], np.array(g["D"]), atol=tol, rtol=0)
    np.testing.assert_allclose(dQ[0, 0], np.array(g["dQ"]), atol=tol, rtol=0)
    np.testing.assert_allclose(dK[0, 0], np.array(g["dK"]), atol=tol, rtol=0)


GRAD_CASES = [
    # B, Hq, Hkv, L, S, E, Ev, causal, mask_kind, mask_shape, scale
    (1, 1, 1, 3, 5, 4, 3, False, "none", None, 0.7),
    (2, 2, 1, 4, 3, 3, 2, True, "none", None, None),
    (1, 4, 2, 5, 5, 4, 3, True, "bias", (1, 4), 0.5),
    (2, 2, 2, 3, 6, 2, 2, False, "bias", (2, 1), 1.3),
]


def _fd_grads(q, k, v, g, mask, scale, causal, gqa, h=1e-6):
    """Central differences of f = sum(O * g) with respect to q, k and v."""
    def f(qq, kk, vv):
        O, _ = oracle.ref_forward(qq, kk, vv, mask, scale, causal, gqa)
        return float((O * g).sum())
    out = []
    for which, x in enumerate((q, k, v)):
        grad = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = [q, k, v]; args_p[which] = xp
            args_m = [q, k, v]; args_m[which] = xm
            grad[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
        out.append(grad)
    return out


def pin_gradcheck():
    """Course chapter section 4 (test_gradcheck_float64): every gradient element vs central differences."""
    for i, (B, Hq, Hkv, L, S, E, Ev, causal, mk, ms, scale) in enumerate(GRAD_CASES):
        q, k, v, dO, mask = random_inputs(B, Hq, Hkv, L, S, E, Ev, torch.float64, seed=10 + i,
                                          mask_shape=ms, mask_kind=mk, p_block=0.2)
        q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
        gqa = Hq != Hkv
        dQ, dK, dV = oracle.ref_backward(q, k, v, dO, mask, scale, causal, gqa)
        fq, fk, fv = _fd_grads(q, k, v, dO, mask, scale, causal, gqa)
        np.testing.assert_allclose(dQ, fq, atol=2e-7, rtol=1e-6)
        np.testing.assert_allclose(dK, fk, atol=2e-7, rtol=1e-6)
        np.testing.assert_allclose(dV, fv, atol=2e-7, rtol=1e-6)


def pin_lse_is_log_normaliser():
    """d(LSE_i)/dq_i = alpha * sum_j P_ij k_j (the gradient of log-sum-exp is the softmax)."""
    q, k, v, _, mask = random_inputs(1, 1, 1, 3, 4, 3, 2, torch.float64, seed=3,
                                     mask_kind="bias", mask_shape=(1, 1), p_block=0.2)
    q, k, v, mask = _np(q), _np(k), _np(v), _np(mask)
    alpha = 0.8
    _, LSE, P = oracle.ref_forward(q, k, v, mask, alpha, return_P=True)
    h = 1e-6
    for i in range(3):
        for e in range(3):
            qp = q.copy(); qp[0, 0, i, e] += h
            qm = q.copy(); qm[0, 0, i, e] -= h
            fd = (oracle.ref_forward(qp, k, v, mask, alpha)[1][0, 0, i]
                  - oracle.ref_forward(qm, k, v, mask, alpha)[1][0, 0, i]) / (2 * h)
            an = alpha * (P[0, 0, i] @ k[0, 0][:, e])
            assert abs(fd - an) < 1e-7


def pin_rows_sum_to_one_and_blocked_zero():
    """Section 2.2: blocked weights exactly 0, open rows sum to 1 (test_masked_keys_get_no_weight_or_gradient)."""
    q, k, v, dO, mask = random_inputs(2, 2, 2, 6, 7, 4, 3, torch.float64, seed=5,
                                      mask_kind="block", mask_shape=(2, 2), p_block=0.3)
    mask[..., 2] = float("-inf")          # key 2 blocked for every query: no gradient at all
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    O, LSE, P = oracle.ref_forward(q, k, v, mask, None, return_P=True)
    blocked = np.isneginf(mask)
    assert np.all(P[np.broadcast_to(blocked, P.shape)] == 0.0)
    rows_open = ~np.all(blocked, axis=-1)
    np.testing.assert_allclose(P.sum(-1)[np.broadcast_to(rows_open, P.shape[:-1])], 1.0, atol=1e-12)
    dQ, dK, dV = oracle.ref_backward(q, k, v, dO, mask, None)
    assert np.all(dK[:, :, 2] == 0.0) and np.all(dV[:, :, 2] == 0.0)


def pin_fully_masked_row():
    """Section 2.2 / test_fully_masked_row_gives_zeros: zeros, never NaN; LSE = -inf (the reading taken)."""
    q, k, v, dO, mask = random_inputs(1, 2, 2, 5, 4, 3, 3, torch.float64, seed=6,
                                      mask_kind="bias", mask_shape=(1, 1), p_block=0.1)
    mask[0, 0, 3, :] = float("-inf")
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    O, LSE = oracle.ref_forward(q, k, v, mask)
    dQ, dK, dV = oracle.ref_backward(q, k, v, dO, mask)
    for x in (O, dQ, dK, dV):
        assert not np.isnan(x).any() and np.isfinite(x).all()
    assert np.all(O[:, :, 3] == 0.0) and np.all(dQ[:, :, 3] == 0.0)
    assert np.all(np.isneginf(LSE[:, :, 3]))
    assert np.isfinite(np.delete(LSE, 3, axis=2)).all()
    # the masked row adds nothing: dK/dV equal those of the same problem with that query's dO zeroed
    dO2 = dO.copy(); dO2[:, :, 3] = 0.0
    _, dK2, dV2 = oracle.ref_backward(q, k, v, dO2, mask)
    np.testing.assert_array_equal(dK, dK2)
    np.testing.assert_array_equal(dV, dV2)


def pin_large_scores_one_hot():
    """test_large_scores_do_not_overflow: scores of order 1e4 give a clean one-hot."""
    q = np.zeros((1, 1, 1, 2)); q[0, 0, 0] = [100.0, 0.0]
    k = np.array([[[[100.0, 0.0], [80.0, 0.0], [-100.0, 0.0]]]])
    v = np.array([[[[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]]]])
    O, LSE, P = oracle.ref_forward(q, k, v, scale=1.0, return_P=True)
    assert np.array_equal(P[0, 0, 0], [1.0, 0.0, 0.0])
    assert np.array_equal(O[0, 0, 0], [1.0, 2.0])
    assert LSE[0, 0, 0] == 1e4


def pin_dk_sums_to_zero():
    """Softmax rows sum to 1, so sum_j dS_ij = 0 and therefore sum_j dK_j = 0 (pitfall 4's symptom)."""
    q, k, v, dO, mask = random_inputs(2, 4, 2, 5, 6, 3, 4, torch.float64, seed=7,
                                      mask_kind="bias", mask_shape=(2, 4), p_block=0.2)
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    _, dK, _ = oracle.ref_backward(q, k, v, dO, mask, 0.6, True, True)
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-12)


def pin_D_identity():
    """Section 2.3: D_i = sum_j P_ij dP_ij equals dO_i . O_i."""
    q, k, v, dO, mask = random_inputs(1, 2, 1, 4, 5, 3, 3, torch.float64, seed=8,
                                      mask_kind="bias", mask_shape=(1, 2), p_block=0.2)
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    O, _ = oracle.ref_forward(q, k, v, mask, None, False, True)
    _, _, _, D = oracle.ref_backward(q, k, v, dO, mask, None, False, True, return_D=True)
    np.testing.assert_allclose(D, (dO * O).sum(-1), atol=1e-12)


def pin_key_permutation_equivariance():
    """test_key_permutation_equivariance: permuting keys with their values changes nothing but the order."""
    q, k, v, dO, mask = random_inputs(1, 2, 2, 4, 6, 3, 2, torch.float64, seed=9,
                                      mask_kind="bias", mask_shape=(1, 2), p_block=0.2)
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    perm = np.array([3, 0, 5, 1, 4, 2])
    O, L = oracle.ref_forward(q, k, v, mask)
    Op, Lp = oracle.ref_forward(q, k[:, :, perm], v[:, :, perm], mask[..., perm])
    np.testing.assert_allclose(O, Op, atol=1e-12)
    np.testing.assert_allclose(L, Lp, atol=1e-12)
    dQ, dK, dV = oracle.ref_backward(q, k, v, dO, mask)
    dQp, dKp, dVp = oracle.ref_backward(q, k[:, :, perm], v[:, :, perm], dO, mask[..., perm])
    np.testing.assert_allclose(dQ, dQp, atol=1e-12)
    np.testing.assert_allclose(dK[:, :, perm], dKp, atol=1e-12)
    np.testing.assert_allclose(dV[:, :, perm], dVp, atol=1e-12)


def pin_queries_independent():
    """test_queries_are_independent: permuted or single queries give the same rows."""
    q, k, v, dO, mask = random_inputs(1, 1, 1, 5, 4, 3, 2, torch.float64, seed=11,
                                      mask_kind="bias", mask_shape=(1, 1), p_block=0.2)
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    perm = np.array([4, 2, 0, 3, 1])
    O, L = oracle.ref_forward(q, k, v, mask)
    Op, Lp = oracle.ref_forward(q[:, :, perm], k, v, mask[:, :, perm])
    np.testing.assert_allclose(O[:, :, perm], Op, atol=1e-12)
    np.testing.assert_allclose(L[:, :, perm], Lp, atol=1e-12)
    for i in range(5):
        Oi, Li = oracle.ref_forward(q[:, :, i:i + 1], k, v, mask[:, :, i:i + 1])
        np.testing.assert_allclose(Oi[:, :, 0], O[:, :, i], atol=1e-12)
    dQ, dK, dV = oracle.ref_backward(q, k, v, dO, mask)
    dQp, dKp, dVp = oracle.ref_backward(q[:, :, perm], k, v, dO[:, :, perm], mask[:, :, perm])
    np.testing.assert_allclose(dQ[:, :, perm], dQp, atol=1e-12)
    np.testing.assert_allclose(dK, dKp, atol=1e-12)


def pin_batched_equals_per_item():
    """Each batch item is its own problem (course chapter, section 2.1: the batch index only
    selects inputs): a batch of three with a per-item mask gives, item by item, exactly what
    each item gives alone."""
    q, k, v, dO, mask = random_inputs(3, 4, 2, 5, 7, 3, 2, torch.float64, seed=13,
                                      mask_kind="bias", mask_shape=(3, 4), p_block=0.2)
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    O, L = oracle.ref_forward(q, k, v, mask, 0.7, True, True)
    grads = oracle.ref_backward(q, k, v, dO, mask, 0.7, True, True)
    for b in range(3):
        sl = slice(b, b + 1)
        Ob, Lb = oracle.ref_forward(q[sl], k[sl], v[sl], mask[sl], 0.7, True, True)
        np.testing.assert_allclose(O[sl], Ob, atol=1e-13)
        np.testing.assert_allclose(L[sl], Lb, atol=1e-13)
        for g, gb in zip(grads, oracle.ref_backward(q[sl], k[sl], v[sl], dO[sl], mask[sl], 0.7, True, True)):
            np.testing.assert_allclose(g[sl], gb, atol=1e-13)


def pin_gqa_is_repeat_interleave():
    """"Understanding PyTorch SDPA" section 4: GQA equals repeat_interleave of K/V; gradients sum over the group."""
    G, Hkv = 3, 2
    q, k, v, dO, mask = random_inputs(2, G * Hkv, Hkv, 4, 5, 3, 2, torch.float64, seed=12,
                                      mask_kind="bias", mask_shape=(2, G * Hkv), p_block=0.2)
    q, k, v, dO, mask = _np(q), _np(k), _np(v), _np(dO), _np(mask)
    kx = np.repeat(k, G, axis=1)          # kv0,kv0,kv0,kv1,kv1,kv1 (repeat_interleave order)
    vx = np.repeat(v, G, axis=1)
    O, L = oracle.ref_forward(q, k, v, mask, 0.4, True, True)
    Ox, Lx = oracle.ref_forward(q, kx, vx, mask, 0.4, True, False)
    np.testing.assert_allclose(O, Ox, atol=1e-12)
    np.testing.assert_allclose(L, Lx, atol=1e-12)
    dQ, dK, dV = oracle.ref_backward(q, k, v, dO, mask, 0.4, True, True)
    dQx, dKx, dVx = oracle.ref_backward(q, kx, vx, dO, mask, 0.4, True, False)
    np.testing.assert_allclose(dQ, dQx, atol=1e-12)
    np.testing.assert_allclose(dK, dKx.reshape(2, Hkv, G, 5, 3).sum(2), atol=1e-12)
    np.testing.assert_allclose(dV, dVx.reshape(2, Hkv, G, 5, 2).sum(2), atol=1e-12)


def pin_zero_scale_is_mean():
    """alpha = 0: every open key has weight 1/#open, O = mean of open values, LSE = ln(#open)."""
    q, k, v, _, mask = random_inputs(1, 1, 1, 4, 6, 3, 2, torch.float64, seed=13,
                                     mask_kind="block", mask_shape=(1, 1), p_block=0.4)
    mask[0, 0, :, 0] = 0.0                # at least one open key per row
    q, k, v, mask = _np(q), _np(k), _np(v), _np(mask)
    O, L = oracle.ref_forward(q, k, v, mask, 0.0)
    for i in range(4):
        open_ = np.isfinite(mask[0, 0, i])
        np.testing.assert_allclose(O[0, 0, i], v[0, 0][open_].mean(0), atol=1e-13)
        np.testing.assert_allclose(L[0, 0, i], math.log(open_.sum()), atol=1e-13)


def pin_single_key():
    """S = 1: P = 1, O = v_0 for every query and all gradients but dV vanish."""
    q, k, v, dO, _ = random_inputs(1, 2, 1, 3, 1, 4, 3, torch.float64, seed=14)
    q, k, v, dO = _np(q), _np(k), _np(v), _np(dO)
    O, L = oracle.ref_forward(q, k, v, None, None, False, True)
    np.testing.assert_allclose(O, np.broadcast_to(v[:, :1, :1], O.shape), atol=1e-14)
    dQ, dK, dV = oracle.ref_backward(q, k, v, dO, None, None, False, True)
    assert np.all(dQ == 0) and np.all(dK == 0)
    np.testing.assert_allclose(dV[0, 0, 0], dO[0].sum(axis=(0, 1)), atol=1e-13)


def pin_causal_first_row():
    """Causal with L = S: query 0 sees key 0 only, so O_0 = v_0 and its LSE is its own score."""
    q, k, v, _, _ = random_inputs(1, 1, 1, 5, 5, 3, 2, torch.float64, seed=15)
    q, k, v = _np(q), _np(k), _np(v)
    O, L = oracle.ref_forward(q, k, v, None, 0.9, True)
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, 0], atol=1e-15)
    np.testing.assert_allclose(L[0, 0, 0], 0.9 * q[0, 0, 0] @ k[0, 0, 0], atol=1e-14)


def pin_default_scale_variance():
    """Section 2.1 (test_score_variance_is_one): with the default scale, score differences have variance 2.

    With no mask, log(P_i0 / P_i1) = s_i0 - s_i1, so the weights reveal the
    scaled score differences; for N(0,1) entries each scaled score has
    variance 1 and the difference of two independent ones variance 2.
    """
    rng = np.random.default_rng(16)
    n = 6000
    for d in (4, 64):
        q = rng.standard_normal((n, 1, 1, d))
        k = rng.standard_normal((n, 1, 2, d))
        v = np.zeros((n, 1, 2, 1))
        _, _, P = oracle.ref_forward(q, k, v, return_P=True)
        diff = np.log(P[:, 0, 0, 0]) - np.log(P[:, 0, 0, 1])
        assert abs(diff.var() - 2.0) < 0.2, (d, diff.var())


def pin_torch_cross_check():
    """Independent library routine: torch's CPU float64 attention and autograd on small cases."""
    F = torch.nn.functional
    cases = [(2, 4, 2, 7, 9, 8, 5, True, (2, 4)), (1, 2, 2, 6, 6, 4, 4, False, (1, 1)),
             (2, 3, 1, 5, 8, 6, 3, False, None)]
    for i, (B, Hq, Hkv, L, S, E, Ev, causal, ms) in enumerate(cases):
        q, k, v, dO, mask = random_inputs(B, Hq, Hkv, L, S, E, Ev, torch.float64, seed=20 + i,
                                          mask_shape=ms, mask_kind="bias" if ms else "none",
                                          p_block=0.1)
        if mask is not None:
            mask[..., 0] = 0.0            # no fully masked rows: torch returns NaN there
        bias = torch.zeros(1, 1, L, S, dtype=torch.float64) if mask is None else mask.clone()
        if causal:
            bias = bias + torch.triu(torch.full((L, S), float("-inf"), dtype=torch.float64), 1)
        tq, tk, tv = (x.clone().requires_grad_(True) for x in (q, k, v))
        out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=bias, scale=0.3,
                                             enable_gqa=Hq != Hkv)
        out.backward(dO)
        O, LSE = oracle.ref_forward(q, k, v, mask, 0.3, causal, Hq != Hkv)
        dQ, dK, dV = oracle.ref_backward(q, k, v, dO, mask, 0.3, causal, Hq != Hkv)
        np.testing.assert_allclose(O, out.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(dQ, tq.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dK, tk.grad.numpy(), atol=1e-11)
        np.testing.assert_allclose(dV, tv.grad.numpy(), atol=1e-11)
        G = Hq // Hkv
        s = 0.3 * (q @ k.repeat_interleave(G, 1).transpose(-1, -2)) + bias
        np.testing.assert_allclose(LSE, torch.logsumexp(s, -1).numpy(), atol=1e-12)


PINS = [pin_hand_forward, pin_hand_backward, pin_gradcheck, pin_lse_is_log_normaliser,
        pin_rows_sum_to_one_and_blocked_zero, pin_fully_masked_row, pin_large_scores_one_hot,
        pin_dk_sums_to_zero, pin_D_identity, pin_key_permutation_equivariance,
        pin_queries_independent, pin_batched_equals_per_item, pin_gqa_is_repeat_interleave, pin_zero_scale_is_mean,
        pin_single_key, pin_causal_first_row, pin_default_scale_variance, pin_torch_cross_check]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# --------------------------------------------------------------------------- mutants
# The pitfalls of section 5 without dropout; the dropout ones (s07-s09) are
# planted in tests/test_oracle_dropout.py.

def _m_scale_1_over_d(E):
    return 1.0 / E


def _m_softmax_query_axis(s, bias):
    orig = so.__dict__["_orig_masked_softmax"]
    t = s + bias
    Pt, _ = orig(t.T, np.zeros_like(t.T))
    return Pt.T, orig(s, bias)[1]


def _m_mask_after_softmax(s, bias):
    orig = so.__dict__["_orig_masked_softmax"]
    P, lse = orig(s, np.zeros_like(s))
    return P * np.isfinite(bias), lse


def _m_vjp_without_D(P, dP, D):
    return P * dP


def _m_dk_no_transpose(dS, q, alpha):
    return alpha * (dS @ q)


def _m_dq_no_scale(dS, k, alpha):
    return dS @ k


def _m_minus_1e9(s, bias):
    return so.__dict__["_orig_masked_softmax"](s, np.where(np.isneginf(bias), -1e9, bias))


def _m_mask_of_batch_zero(mask, b, h, L, S, is_causal, band=None):
    return so.__dict__["_orig_head_bias"](mask, 0, h, L, S, is_causal, band)


MUTANTS = {
    "s01_scale_1_over_d": ("default_scale", _m_scale_1_over_d),
    "s02_softmax_over_queries": ("_masked_softmax", _m_softmax_query_axis),
    "s03_mask_after_softmax": ("_masked_softmax", _m_mask_after_softmax),
    "s04_vjp_without_D": ("_softmax_vjp", _m_vjp_without_D),
    "s05_dk_without_transpose": ("_dk", _m_dk_no_transpose),
    "s06_dq_without_scale": ("_dq", _m_dq_no_scale),
    "s10_mask_with_minus_1e9": ("_masked_softmax", _m_minus_1e9),
    "x01_mask_of_batch_zero": ("_head_bias", _m_mask_of_batch_zero),   # a broadcast-index slip
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setitem(so.__dict__, "_orig_masked_softmax", so._masked_softmax)
    monkeypatch.setitem(so.__dict__, "_orig_head_bias", so._head_bias)
    monkeypatch.setattr(so, attr, fn)
    failed = []
    for pin in PINS:
        if pin is pin_default_scale_variance and attr != "default_scale":
            continue                        # slow; only relevant to the scale mutant
        try:
            pin()
        except Exception:                   # noqa: BLE001 - any failure counts as caught
            failed.append(pin.__name__)
    assert failed, f"mutant {name} survived every pin"


def test_default_scale_is_inverse_sqrt_d():
    """test_default_scale_is_inverse_sqrt_d: scale=None equals 1/sqrt(E) explicitly."""
    q, k, v, _, _ = random_inputs(1, 1, 1, 3, 4, 9, 2, torch.float64, seed=30)
    a = oracle.ref_forward(q, k, v, None, None)
    b = oracle.ref_forward(q, k, v, None, 1.0 / 3.0)
    np.testing.assert_array_equal(a[0], b[0])


def test_rejects_bad_arguments():
    """test_rejects_bad_arguments: mismatched shapes and bad scales fail loudly."""
    q, k, v, _, _ = random_inputs(1, 2, 1, 3, 4, 4, 2, torch.float64, seed=31)
    with pytest.raises(ValueError):
        oracle.ref_forward(q, k, v)                       # GQA without enable_gqa
    with pytest.raises(ValueError):
        oracle.ref_forward(q, k[..., :3], v, enable_gqa=True)
    with pytest.raises(ValueError):
        oracle.ref_forward(q, k, v, scale=-1.0, enable_gqa=True)
    with pytest.raises(ValueError):
        oracle.ref_forward(q, k, v, scale=float("inf"), enable_gqa=True)
    with pytest.raises(ValueError):
        oracle.ref_forward(q, k, v, mask=torch.zeros(1, 1, 3, 5), enable_gqa=True)


def test_group_and_rows_helpers_match_full():
    """The sampled-check helpers agree with the full oracle (they restrict it, nothing more)."""
    q, k, v, dO, mask = random_inputs(2, 4, 2, 6, 7, 3, 3, torch.float64, seed=32,
                                      mask_kind="bias", mask_shape=(2, 1), p_block=0.2)
    O, L = oracle.ref_forward(q, k, v, mask, 0.5, True, True)
    dQ, dK, dV = oracle.ref_backward(q, k, v, dO, mask, 0.5, True, True)
    Og, Lg, dQg, dKg, dVg = oracle.ref_group(q, k, v, dO, 1, 1, mask, 0.5, True)
    np.testing.assert_allclose(Og, O[1, 2:4], atol=1e-13)
    np.testing.assert_allclose(Lg, L[1, 2:4], atol=1e-13)
    np.testing.assert_allclose(dQg, dQ[1, 2:4], atol=1e-13)
    np.testing.assert_allclose(dKg, dK[1, 1], atol=1e-13)
    np.testing.assert_allclose(dVg, dV[1, 1], atol=1e-13)
    Or, Lr = oracle.ref_forward_rows(q, k, v, 1, 3, [0, 4, 5], mask, 0.5, True, True)
    np.testing.assert_allclose(Or, O[1, 3, [0, 4, 5]], atol=1e-13)
    np.testing.assert_allclose(Lr, L[1, 3, [0, 4, 5]], atol=1e-13)
    dQr = oracle.ref_backward_rows(q, k, v, dO, 1, 3, [0, 4, 5], mask, 0.5, True, True)
    np.testing.assert_allclose(dQr, dQ[1, 3, [0, 4, 5]], atol=1e-13)
    band = oracle.Band([6, 4], [7, 5], "bottom_right", 0, 3)
    dQb = oracle.ref_backward(q, k, v, dO, mask, 0.5, False, True, band=band)[0]
    dQrb = oracle.ref_backward_rows(q, k, v, dO, 0, 1, [1, 2, 5], mask, 0.5, False, True, band=band)
    np.testing.assert_allclose(dQrb, dQb[0, 1, [1, 2, 5]], atol=1e-13)
    # the group restriction keeps each head's padding lengths and dropout mask
    drop = oracle.Dropout(0.3, seed=12345, offset=7)
    Od, Ld = oracle.ref_forward(q, k, v, mask, 0.5, False, True, band=band, dropout=drop)
    dQd, dKd, dVd = oracle.ref_backward(q, k, v, dO, mask, 0.5, False, True, band=band, dropout=drop)
    for b, kv in ((0, 0), (1, 1)):
        Og, Lg, dQg, dKg, dVg = oracle.ref_group(q, k, v, dO, b, kv, mask, 0.5, False, band=band, dropout=drop)
        hs = slice(2 * kv, 2 * kv + 2)
        np.testing.assert_allclose(Og, Od[b, hs], atol=1e-13)
        np.testing.assert_allclose(Lg, Ld[b, hs], atol=1e-13)
        np.testing.assert_allclose(dQg, dQd[b, hs], atol=1e-13)
        np.testing.assert_allclose(dKg, dKd[b, kv], atol=1e-13)
        np.testing.assert_allclose(dVg, dVd[b, kv], atol=1e-13)
    # and the dropout is live there: without it the group's O differs
    assert np.abs(oracle.ref_group(q, k, v, None, 1, 1, mask, 0.5, False, band=band)[0] - Od[1, 2:4]).max() > 1e-3
    # the row restriction's band and dropout branches: each row keeps its batch's lengths
    # and its own (b, h, row) dropout counters
    Ob, Lb = oracle.ref_forward(q, k, v, mask, 0.5, False, True, band=band)
    for b, h, rows in ((0, 1, [1, 2, 5]), (1, 3, [0, 3, 4])):
        Orb, Lrb = oracle.ref_forward_rows(q, k, v, b, h, rows, mask, 0.5, False, True, band=band)
        np.testing.assert_allclose(Orb, Ob[b, h, rows], atol=1e-13)
        np.testing.assert_array_equal(np.isneginf(Lrb), np.isneginf(Lb[b, h, rows]))
        fin = np.isfinite(Lrb)
        np.testing.assert_allclose(Lrb[fin], Lb[b, h, rows][fin], atol=1e-13)
        Ord, Lrd = oracle.ref_forward_rows(q, k, v, b, h, rows, mask, 0.5, False, True, band=band, dropout=drop)
        np.testing.assert_allclose(Ord, Od[b, h, rows], atol=1e-13)
        np.testing.assert_allclose(Lrd[fin], Ld[b, h, rows][fin], atol=1e-13)
    # both branches are live on these rows: dropping either changes the result
    Orx, _ = oracle.ref_forward_rows(q, k, v, 1, 3, [0, 3, 4], mask, 0.5, False, True, band=band)
    assert np.abs(Orx - Od[1, 3, [0, 3, 4]]).max() > 1e-3
    Orx, _ = oracle.ref_forward_rows(q, k, v, 1, 3, [0, 3, 4], mask, 0.5, False, True)
    assert np.abs(Orx - Ob[1, 3, [0, 3, 4]]).max() > 1e-3


def test_repeated_keys_equal_log_multiplicity_bias():
    """Attention over keys that repeat (key r present n_r times, in any order) equals
    attention over the distinct keys with the additive bias ln n_r: each distinct key's
    weight is n_r e^(s_r) / sum_r n_r e^(s_r) either way.  Large-size GPU tests rely on it."""
    rng = np.random.default_rng(81)
    P, E, Ev = 5, 4, 3
    counts = np.array([1, 3, 2, 4, 1])
    kb, vb = rng.standard_normal((P, E)), rng.standard_normal((P, Ev))
    q = rng.standard_normal((1, 2, 3, E))
    order = rng.permutation(np.repeat(np.arange(P), counts))
    k_full, v_full = kb[order][None, None], vb[order][None, None]
    O1, L1 = oracle.ref_forward(q, k_full, v_full, None, 0.7, False, True)
    bias = np.broadcast_to(np.log(counts).astype(np.float64), (1, 1, 3, P)).copy()   # [1, 1, L, P]
    O2, L2 = oracle.ref_forward(q, kb[None, None], vb[None, None], bias, 0.7, False, True)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)
