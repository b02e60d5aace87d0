"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle.

Same seeded inputs on both sides (workloads module).  Tolerances:
  fp32 inputs: max |err| <= 1e-4 on O, <= 1e-3 on dQ/dK/dV, <= 1e-5 on finite LSE;
  bf16 inputs with fp32 accumulation: relative L2 ||x - ref|| / ||ref|| <= 5e-3 on O and
  <= 1e-2 on each gradient (whole tensor), |err| <= 1e-3 on finite LSE;
  and, for both, exact zeros where masking forces them (O and dQ rows of fully
  masked queries, dK/dV rows of keys blocked for every query of their group),
  LSE = -inf exactly on fully masked rows and no NaN/Inf anywhere else.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_sm_gb300 as sdpa
from workloads import random_inputs

pytestmark = pytest.mark.gpu

F32_O, F32_G, F32_LSE = 1e-4, 1e-3, 1e-5
BF_O, BF_G, BF_LSE = 5e-3, 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdpa.build()
    sdpa.load_library()
    assert sdpa.last_device_status() == 0


def rel_l2(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / (den if den > 0 else 1.0)


def to64(t):
    return t.detach().float().cpu().double().numpy()


def blocked_keys(mask, causal, B, Hq, Hkv, L, S):
    """[B, Hkv, S] True where the key is blocked for every query of every head of its group."""
    G = Hq // Hkv
    out = np.zeros((B, Hkv, S), bool)
    cb = oracle.causal_bias(L, S) if causal else np.zeros((L, S))
    for b in range(B):
        for kv in range(Hkv):
            allb = np.ones(S, bool)
            for h in range(kv * G, (kv + 1) * G):
                m = np.zeros((L, S)) if mask is None else mask[min(b, mask.shape[0] - 1), min(h, mask.shape[1] - 1)]
                allb &= np.all(np.isneginf(m + cb), axis=0)
            out[b, kv] = allb
    return out


def check_forward(o, lse, ref_o, ref_lse, bf16):
    o64, l64 = to64(o), lse.detach().cpu().double().numpy()
    dead = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l64), dead), "LSE = -inf exactly on the fully masked rows only"
    assert np.isfinite(o64).all()
    assert np.all(o64[dead] == 0.0), "fully masked rows give O = 0 exactly"
    live = ~dead
    if live.any():
        lerr = np.abs(l64[live] - ref_lse[live]).max()
        assert lerr <= (BF_LSE if bf16 else F32_LSE), f"LSE err {lerr}"
    if bf16:
        e = rel_l2(o64, ref_o)
        assert e <= BF_O, f"O rel-L2 {e}"
    else:
        e = np.abs(o64 - ref_o).max()
        assert e <= F32_O, f"O max err {e}"


def check_backward(grads, refs, dead_rows, blocked, bf16):
    dq, dk, dv = (to64(g) for g in grads)
    for name, x, r in (("dQ", dq, refs[0]), ("dK", dk, refs[1]), ("dV", dv, refs[2])):
        assert np.isfinite(x).all(), name
        if bf16:
            e = rel_l2(x, r)
            assert e <= BF_G, f"{name} rel-L2 {e}"
        else:
            e = np.abs(x - r).max()
            assert e <= F32_G, f"{name} max err {e}"
    assert np.all(dq[dead_rows] == 0.0), "dQ rows of fully masked queries are exactly 0"
    assert np.all(dk[blocked] == 0.0) and np.all(dv[blocked] == 0.0), "keys blocked for every query get 0"


def run_case(B, Hq, Hkv, L, S, E, Ev, dtype, causal, mask_kind="none", mask_shape=None, full_rows=0,
             scale=None, seed=0, backward=True, p_block=0.25, k_growth=0.0):
    q, k, v, dO, mask = random_inputs(B, Hq, Hkv, L, S, E, Ev, dtype, seed=seed, mask_shape=mask_shape,
                                      mask_kind=mask_kind, full_rows=full_rows, p_block=p_block)
    if k_growth:   # key j scaled by 1 + k_growth * j / S: the scores grow along the keys
        g = 1.0 + k_growth * torch.arange(S, dtype=torch.float32) / S
        k = (k.float() * g[None, None, :, None]).to(dtype)
    gqa = Hq != Hkv
    bf16 = dtype == torch.bfloat16
    ref_o, ref_lse = oracle.ref_forward(q, k, v, mask, scale, causal, gqa)
    dev = [x.cuda() if x is not None else None for x in (q, k, v, dO, mask)]
    qd, kd, vd, dOd, md = dev
    o, lse = sdpa.sdpa_forward(qd, kd, vd, md, scale, causal, gqa)
    torch.cuda.synchronize()
    check_forward(o, lse, ref_o, ref_lse, bf16)
    if backward:
        dq, dk, dv = sdpa.sdpa_backward(qd, kd, vd, o, dOd, lse, md, scale, causal, gqa)
        torch.cuda.synchronize()
        refs = oracle.ref_backward(q, k, v, dO, mask, scale, causal, gqa)
        m64 = None if mask is None else mask.double().numpy()
        check_backward((dq, dk, dv), refs, np.isneginf(ref_lse), blocked_keys(m64, causal, B, Hq, Hkv, L, S),
                       bf16)
    assert sdpa.last_device_status() == 0


@pytest.mark.parametrize("causal", [False, True])
def test_row_max_growing_across_key_tiles(causal):
    """Scores that grow along the keys (key j scaled by 1 + 7 j / S, so a 128-key tile's row max
    rises by about 2 natural-log units per tile): the running row max moves past the kernels'
    rescale threshold (2^8 in the exponentials) several times per row, so O is rescaled and the
    exponentials of those tiles are taken again with the new max."""
    run_case(1, 4, 2, 700, 1000, 128, 128, torch.bfloat16, causal, seed=41, k_growth=7.0)


# ----------------------------------------------------------------------------- fp32
@pytest.mark.parametrize("causal", [False, True])
def test_tiny_fp32_workload(causal):
    """B=2, Hq=Hkv=2, L=S=64, E=Ev=16, N(0,1), seed 0, scale 1/4; no mask, then causal."""
    run_case(2, 2, 2, 64, 64, 16, 16, torch.float32, causal, scale=0.25, seed=0)


def test_hand_example_on_gpu():
    """Course chapter section 3 worked example (E=4, Ev=2, L=1, S=3) on the fp32 kernels."""
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")))
    q = torch.tensor(g["q"], dtype=torch.float32)[None, None].cuda()
    k = torch.tensor(g["k"], dtype=torch.float32)[None, None].cuda()
    v = torch.tensor(g["v"], dtype=torch.float32)[None, None].cuda()
    dO = torch.tensor(g["dO"], dtype=torch.float32)[None, None].cuda()
    o, lse = sdpa.sdpa_forward(q, k, v)
    dq, dk, dv = sdpa.sdpa_backward(q, k, v, o, dO, lse)
    tol = 0.5e-6 + 1e-6
    np.testing.assert_allclose(o.cpu().numpy()[0, 0], g["O"], atol=tol)
    np.testing.assert_allclose(dq.cpu().numpy()[0, 0], g["dQ"], atol=tol)
    np.testing.assert_allclose(dk.cpu().numpy()[0, 0], g["dK"], atol=tol)
    np.testing.assert_allclose(dv.cpu().numpy()[0, 0], g["dV"], atol=tol)
    assert abs(lse.item() - math.log(g["normaliser"])) < 1e-4


@pytest.mark.parametrize("case", [
    (1, 4, 2, 37, 91, 24, 8, True, "bias", (1, 4), 2),
    (2, 2, 2, 130, 70, 128, 128, False, "bias", (2, 1), 3),
    (1, 3, 1, 65, 200, 33, 17, True, "none", None, 0),
])
def test_fp32_ragged_masked(case):
    B, Hq, Hkv, L, S, E, Ev, causal, mk, ms, fr = case
    run_case(B, Hq, Hkv, L, S, E, Ev, torch.float32, causal, mk, ms, fr, scale=0.3, seed=5)


# ----------------------------------------------------------------------------- bf16 prefill
BF16_CASES = [
    # B, Hq, Hkv, L, S, E, Ev, causal, mask_kind, mask_shape, full_rows
    (1, 2, 2, 300, 260, 64, 64, True, "none", None, 0),
    (2, 8, 2, 257, 385, 128, 128, False, "bias", (2, 1), 3),
    (1, 4, 1, 130, 700, 128, 128, True, "none", None, 0),
    (1, 2, 2, 700, 130, 64, 64, True, "none", None, 0),
    (1, 4, 4, 200, 300, 128, 128, False, "bias", (1, 4), 2),
    (1, 2, 1, 256, 256, 128, 64, True, "block", (1, 1), 1),
    (1, 2, 2, 129, 129, 64, 128, False, "none", None, 0),
    (1, 2, 2, 96, 80, 32, 40, True, "bias", (1, 1), 1),     # widths outside {64,128}: CUDA-core path
    (1, 8, 2, 100, 300, 128, 128, True, "none", None, 0),   # key tiles past every query: dK = dV = 0
    (2, 4, 1, 333, 333, 128, 128, True, "bias", (2, 4), 2), # GQA causal + per-head mask, ragged
    (1, 2, 2, 64, 1000, 128, 128, False, "block", (1, 2), 0),
    # rows of a multiple of 4 keys: the backward stages the mask through shared memory
    (2, 4, 2, 190, 512, 64, 64, False, "bias", (2, 4), 2),
    (2, 4, 4, 257, 388, 128, 128, True, "bias", (2, 4), 1),
    (3, 2, 1, 100, 132, 128, 128, False, "block", (3, 1), 1),
    # more work units than SMs: the persistent forward walks several units per CTA
    (2, 96, 32, 300, 333, 128, 128, True, "bias", (2, 1), 2),
    (1, 200, 200, 130, 140, 64, 64, False, "none", None, 0),
    # large query groups: sixteen query heads on one KV head (MQA), eight per KV head with a
    # per-head mask (S not a multiple of 4: the mask is read from global memory)
    (1, 16, 1, 200, 300, 128, 128, True, "none", None, 0),
    (2, 8, 1, 150, 150, 64, 64, False, "bias", (2, 8), 1),
    # one query row under the causal mask: key 0 alone is open, dK = dV = 0 past it
    (2, 4, 2, 1, 100, 128, 128, True, "none", None, 0),
]


@pytest.mark.parametrize("case", BF16_CASES, ids=[str(i) for i in range(len(BF16_CASES))])
def test_bf16_prefill(case):
    B, Hq, Hkv, L, S, E, Ev, causal, mk, ms, fr = case
    run_case(B, Hq, Hkv, L, S, E, Ev, torch.bfloat16, causal, mk, ms, fr, seed=7)


# One, two and three iterations per backward CTA (64-row query tiles times the heads of
# its group): the two S^T buffers, the two dS^T buffers and, with a staged mask, the
# dS^T hand-over deferred to the next iteration, each at its first uses and at the end.
ITER_CASES = [
    # B, Hq, Hkv, L, S, E, causal, mask kind, mask shape
    (1, 1, 1, 64, 64, 128, False, "none", None),       # 1 iteration
    (1, 1, 1, 128, 128, 128, False, "none", None),     # 2
    (1, 1, 1, 192, 192, 64, False, "none", None),      # 3
    (2, 3, 1, 64, 64, 128, False, "none", None),       # 3: one query tile, three heads
    (1, 2, 1, 320, 320, 128, True, "none", None),      # 10 down to 2 per key tile
    (1, 1, 1, 64, 64, 128, False, "bias", (1, 1)),     # staged mask, 1 iteration
    (1, 1, 1, 128, 128, 128, False, "bias", (1, 1)),   # 2
    (2, 2, 2, 192, 192, 64, False, "block", (2, 2)),   # 3
]


@pytest.mark.parametrize("case", ITER_CASES, ids=[str(i) for i in range(len(ITER_CASES))])
def test_backward_iteration_counts(case):
    B, Hq, Hkv, L, S, E, causal, mk, ms = case
    run_case(B, Hq, Hkv, L, S, E, E, torch.bfloat16, causal, mk, ms, 0, seed=21)


def test_bf16_large_scores_no_overflow():
    """Scores of order 1e3-1e4 stay finite and match (the max is subtracted first)."""
    q, k, v, dO, _ = random_inputs(1, 2, 2, 200, 300, 64, 64, torch.bfloat16, seed=9)
    q = (q.float() * 40).bfloat16()
    ref_o, ref_lse = oracle.ref_forward(q, k, v, None, 1.0)
    o, lse = sdpa.sdpa_forward(q.cuda(), k.cuda(), v.cuda(), None, 1.0)
    check_forward(o, lse, ref_o, ref_lse, True)


# ----------------------------------------------------------------------------- decode
@pytest.mark.parametrize("splits,S", [(1, 1000), (2, 1000), (7, 1000), (0, 1000), (64, 4095)])
def test_decode_split_invariance(splits, S):
    """Split-KV decode equals the oracle for any split count (merge exact up to fp32 rounding).

    With 64-key stages, S = 4095 and 64 requested splits give 64 splits of 64 keys,
    the last one 63."""
    B, Hq, Hkv, E = 2, 8, 2, 128
    q, k, v, _, _ = random_inputs(B, Hq, Hkv, 1, S, E, E, torch.bfloat16, seed=11)
    ref_o, ref_lse = oracle.ref_forward(q, k, v, None, None, False, True)
    o, lse = sdpa.sdpa_decode(q.cuda(), k.cuda(), v.cuda(), None, None, True, splits)
    check_forward(o, lse, ref_o, ref_lse, True)
    o1, lse1 = sdpa.sdpa_decode(q.cuda(), k.cuda(), v.cuda(), None, None, True, 1)
    np.testing.assert_allclose(lse.cpu().numpy(), lse1.cpu().numpy(), atol=2e-5)


def test_decode_with_mask_and_rows():
    """Decode with an additive mask (one fully masked query) and G*L > 8 rows per group."""
    B, Hq, Hkv, L, S, E = 1, 6, 1, 3, 777, 64
    q, k, v, _, mask = random_inputs(B, Hq, Hkv, L, S, E, E, torch.bfloat16, seed=12, mask_kind="bias",
                                     mask_shape=(1, Hq), full_rows=1)
    ref_o, ref_lse = oracle.ref_forward(q, k, v, mask, None, False, True)
    o, lse = sdpa.sdpa_decode(q.cuda(), k.cuda(), v.cuda(), mask.cuda(), None, True, 3)
    check_forward(o, lse, ref_o, ref_lse, True)


def test_decode_mqa_groups():
    """Decode with 32 query heads on one KV head (four row groups of 8 per split) and a ragged
    S, for the automatic split count and for an explicit one."""
    B, Hq, Hkv, S, E = 2, 32, 1, 2049, 128
    q, k, v, _, _ = random_inputs(B, Hq, Hkv, 1, S, E, E, torch.bfloat16, seed=14)
    ref_o, ref_lse = oracle.ref_forward(q, k, v, None, None, False, True)
    for splits in (0, 5):
        o, lse = sdpa.sdpa_decode(q.cuda(), k.cuda(), v.cuda(), None, None, True, splits)
        check_forward(o, lse, ref_o, ref_lse, True)


def test_forward_routes_l1_to_decode():
    B, Hq, Hkv, S, E = 3, 4, 4, 513, 64
    q, k, v, _, _ = random_inputs(B, Hq, Hkv, 1, S, E, E, torch.bfloat16, seed=13)
    ref_o, ref_lse = oracle.ref_forward(q, k, v)
    o, lse = sdpa.sdpa_forward(q.cuda(), k.cuda(), v.cuda())
    check_forward(o, lse, ref_o, ref_lse, True)


@pytest.mark.parametrize("causal,mask_kind", [(True, "none"), (False, "bias")])
def test_bf16_zero_scale(causal, mask_kind):
    """alpha = 0: every open key gets the same weight (the mean of the open values)."""
    run_case(1, 4, 2, 200, 260, 128, 128, torch.bfloat16, causal, mask_kind, (1, 1) if mask_kind != "none" else None,
             1 if mask_kind != "none" else 0, scale=0.0, seed=31)



def test_masked_runs_are_bit_identical():
    """The staged additive mask is recycled between TMA fills and the softmax / elementwise
    warps' reads; a missing order between the two shows as run-to-run differences.  O, LSE,
    dK and dV of repeated calls must match bit for bit (dQ is summed in a varying order)."""
    B, Hq, Hkv, L, S, E = 4, 8, 8, 1024, 1024, 128
    q, k, v, dO, mask = random_inputs(B, Hq, Hkv, L, S, E, E, torch.bfloat16, seed=51, mask_kind="bias",
                                      mask_shape=(B, 1), full_rows=2)
    qd, kd, vd, dOd, md = q.cuda(), k.cuda(), v.cuda(), dO.cuda(), mask.cuda()
    o0, l0 = sdpa.sdpa_forward(qd, kd, vd, md)
    g0 = sdpa.sdpa_backward(qd, kd, vd, o0, dOd, l0, md)
    for _ in range(3):
        o1, l1 = sdpa.sdpa_forward(qd, kd, vd, md)
        g1 = sdpa.sdpa_backward(qd, kd, vd, o0, dOd, l0, md)
        torch.cuda.synchronize()
        assert torch.equal(o0, o1) and torch.equal(l0, l1)
        assert torch.equal(g0[1], g1[1]) and torch.equal(g0[2], g1[2])
    assert sdpa.last_device_status() == 0
