"""GPU parity of padding (seq_len_q / seq_len_kv), diagonal alignment and band
bounds: the *_opts entry points against the float64 oracle with the same Band.

Cases cover every kernel path (bf16 tensor-core prefill and backward at E = 128
and 64, the CUDA-core fp32 and bf16 kernels, the split-KV decode), batches of
length 0 and 1, keys shorter than queries under bottom-right alignment (leading
rows without keys), windows narrower and wider than a tile, a right bound past
the diagonal, and bands combined with an additive mask.  Tolerances are the
ones of test_gpu_parity.py, with exact zeros where padding or the band forces
them.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_sm_gb300 as sdpa
from test_gpu_parity import check_backward, check_forward
from workloads import random_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdpa.build()
    sdpa.load_library()
    assert sdpa.last_device_status() == 0


def _bands(B, lq, lk, align, right, left):
    ob = oracle.Band(lq, lk, align, right, left)
    gb = sdpa.Band(None if lq is None else torch.tensor(lq, dtype=torch.int32, device="cuda"),
                   None if lk is None else torch.tensor(lk, dtype=torch.int32, device="cuda"),
                   align, right, left)
    return ob, gb


def _blocked_keys(mask, band, B, Hq, Hkv, L, S):
    """[B, Hkv, S]: keys blocked for every query of every head of their group."""
    G = Hq // Hkv
    out = np.zeros((B, Hkv, S), bool)
    for b in range(B):
        bb = oracle.band_bias(L, S, band, b)
        for kv in range(Hkv):
            allb = np.ones(S, bool)
            for h in range(kv * G, (kv + 1) * G):
                m = np.zeros((L, S)) if mask is None else mask[min(b, mask.shape[0] - 1), min(h, mask.shape[1] - 1)]
                allb &= np.all(np.isneginf(m + bb), axis=0)
            out[b, kv] = allb
    return out


def _run(B, Hq, Hkv, L, S, E, Ev, dtype, lq, lk, align, right, left, mask_kind="none", seed=0, backward=True):
    q, k, v, dO, mask = random_inputs(B, Hq, Hkv, L, S, E, Ev, dtype, seed=seed, mask_kind=mask_kind,
                                      mask_shape=(B, 1) if mask_kind != "none" else None, p_block=0.2)
    ob, gb = _bands(B, lq, lk, align, right, left)
    gqa = Hq != Hkv
    bf16 = dtype == torch.bfloat16
    ref_o, ref_lse = oracle.ref_forward(q, k, v, mask, None, False, gqa, band=ob)
    qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    md = None if mask is None else mask.cuda()
    o, lse = sdpa.sdpa_forward(qd, kd, vd, md, None, False, gqa, band=gb)
    torch.cuda.synchronize()
    check_forward(o, lse, ref_o, ref_lse, bf16)
    if backward:
        dq, dk, dv = sdpa.sdpa_backward(qd, kd, vd, o, dOd, lse, md, None, False, gqa, band=gb)
        torch.cuda.synchronize()
        refs = oracle.ref_backward(q, k, v, dO, mask, None, False, gqa, band=ob)
        m64 = None if mask is None else mask.double().numpy()
        check_backward((dq, dk, dv), refs, np.isneginf(ref_lse), _blocked_keys(m64, ob, B, Hq, Hkv, L, S), bf16)
    assert sdpa.last_device_status() == 0


PREFILL = [
    # B, Hq, Hkv, L, S, E, Ev, dtype, seq_len_q, seq_len_kv, alignment, right, left, mask
    (3, 4, 2, 300, 333, 128, 128, "bf16", [300, 129, 0], [333, 1, 200], "top_left", None, None, "none"),
    (3, 4, 2, 300, 333, 128, 128, "bf16", [300, 129, 0], [333, 1, 200], "top_left", 0, None, "none"),
    (2, 2, 2, 200, 700, 128, 128, "bf16", None, None, "bottom_right", 0, None, "none"),
    (2, 4, 1, 257, 640, 128, 128, "bf16", [150, 40], [600, 30], "bottom_right", 0, None, "none"),
    (1, 2, 2, 500, 500, 128, 128, "bf16", None, None, "top_left", 0, 100, "none"),
    (2, 2, 1, 400, 450, 128, 128, "bf16", [400, 333], None, "top_left", 0, 300, "bias"),
    (1, 2, 2, 400, 400, 128, 128, "bf16", None, None, "top_left", 50, 64, "none"),
    (2, 2, 2, 300, 900, 64, 64, "bf16", [300, 200], [900, 450], "bottom_right", 0, 256, "none"),
    (1, 3, 3, 260, 260, 64, 128, "bf16", None, [200], "top_left", 0, 70, "none"),
    # rows of a multiple of 4 keys: the additive mask is staged by TMA, the padded units come from the counter
    (2, 4, 2, 300, 512, 128, 128, "bf16", [300, 200], [512, 256], "bottom_right", 0, 100, "bias"),
    (3, 2, 2, 260, 388, 64, 64, "bf16", [260, 0, 129], [388, 100, 200], "top_left", 0, None, "bias"),
    (1, 2, 1, 150, 170, 32, 40, "bf16", [150], [120], "bottom_right", 0, 50, "bias"),   # CUDA-core bf16
    (2, 2, 2, 70, 90, 24, 16, "f32", [70, 33], [90, 10], "bottom_right", 0, 20, "bias"),
    (2, 2, 1, 64, 64, 16, 16, "f32", [64, 0], [64, 64], "top_left", 3, 8, "none"),
]


@pytest.mark.parametrize("case", PREFILL, ids=[str(i) for i in range(len(PREFILL))])
def test_band_prefill(case):
    B, Hq, Hkv, L, S, E, Ev, dt, lq, lk, align, right, left, mk = case
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    _run(B, Hq, Hkv, L, S, E, Ev, dtype, lq, lk, align, right, left, mk, seed=100 + PREFILL.index(case))


@pytest.mark.parametrize("splits", [0, 1, 7])
def test_band_decode_cache_lengths_and_window(splits):
    """Decode against per-sequence cache lengths (one empty, one of length 1) and a
    bottom-right window, with 1 and 3 query rows; any split count."""
    for L, lq in ((1, None), (3, [3, 3, 2, 3])):
        B, Hq, Hkv, S, E = 4, 8, 2, 3000, 128
        q, k, v, _, _ = random_inputs(B, Hq, Hkv, L, S, E, E, torch.bfloat16, seed=200 + L)
        for right, left in ((None, None), (0, 700)):
            ob, gb = _bands(B, lq, [3000, 1, 1500, 0], "bottom_right", right, left)
            ref_o, ref_lse = oracle.ref_forward(q, k, v, None, None, False, True, band=ob)
            o, lse = sdpa.sdpa_decode(q.cuda(), k.cuda(), v.cuda(), None, None, True, splits, band=gb)
            torch.cuda.synchronize()
            check_forward(o, lse, ref_o, ref_lse, True)
    assert sdpa.last_device_status() == 0


def test_band_forward_routes_l1_to_decode():
    B, Hq, Hkv, S, E = 2, 4, 4, 777, 64
    q, k, v, _, _ = random_inputs(B, Hq, Hkv, 1, S, E, E, torch.bfloat16, seed=210)
    ob, gb = _bands(B, None, [777, 300], "bottom_right", 0, 128)
    ref_o, ref_lse = oracle.ref_forward(q, k, v, None, None, False, False, band=ob)
    o, lse = sdpa.sdpa_forward(q.cuda(), k.cuda(), v.cuda(), band=gb)
    torch.cuda.synchronize()
    check_forward(o, lse, ref_o, ref_lse, True)


def test_plain_causal_equals_top_left_right_bound_zero():
    """is_causal and the band {top_left, right_bound 0} give bit-identical O, LSE, dK and
    dV (dQ is summed by bulk reductions whose order between key tiles is not fixed, so two
    runs may differ in the last bits of dQ)."""
    q, k, v, dO, _ = random_inputs(1, 4, 2, 300, 300, 128, 128, torch.bfloat16, seed=220)
    qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o1, l1 = sdpa.sdpa_forward(qd, kd, vd, None, None, True, True)
    o2, l2 = sdpa.sdpa_forward(qd, kd, vd, None, None, False, True, band=sdpa.Band(right_bound=0))
    g1 = sdpa.sdpa_backward(qd, kd, vd, o1, dOd, l1, None, None, True, True)
    g2 = sdpa.sdpa_backward(qd, kd, vd, o2, dOd, l2, None, None, False, True, band=sdpa.Band(right_bound=0))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    d = (g1[0].float() - g2[0].float()).norm() / g1[0].float().norm()
    assert d <= 1e-3, d


def test_padded_counter_schedule_equals_fixed_order():
    """With padding lengths the tensor-core forward takes work units from a counter in its
    workspace; without a workspace it walks a fixed list.  Units are independent, so both
    give bit-identical outputs, and both match the oracle."""
    B, Hq, Hkv, L, S, E = 6, 8, 2, 1100, 1100, 128
    lq, lk = [1100, 37, 900, 0, 640, 1], [1100, 500, 900, 10, 1100, 1]
    q, k, v, _, _ = random_inputs(B, Hq, Hkv, L, S, E, E, torch.bfloat16, seed=230)
    ob, gb = _bands(B, lq, lk, "bottom_right", 0, None)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = sdpa.sdpa_forward(qd, kd, vd, None, None, False, True, band=gb)   # counter (workspace given)
    none = torch.empty(0, dtype=torch.uint8, device="cuda")
    o2, l2 = sdpa.sdpa_forward(qd, kd, vd, None, None, False, True, band=gb, workspace=none)
    torch.cuda.synchronize()
    assert sdpa.last_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref_o, ref_lse = oracle.ref_forward(q, k, v, None, None, False, True, band=ob)
    check_forward(o1, lse=l1, ref_o=ref_o, ref_lse=ref_lse, bf16=True)
