"""GPU parity of attention dropout (course chapter section 2.5; cuDNN Philox RNG
dropout) against the float64 oracle with the same Philox4x32-10 mask.

The mask itself is compared bit for bit (an integer decision): with V = I the
output row is P o keep / (1 - p), so its zero pattern is the dropped set.  The
forward and backward are compared with the oracle's on every kernel path
(bf16 tensor cores at E = 128 and 64, CUDA-core bf16 and fp32), with causal,
GQA, masks and bands; p = 0 reproduces the plain call; a call is determined by
its seed and offset.
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


@pytest.mark.parametrize("dtype,E", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 16)])
def test_dropout_mask_bit_exact(dtype, E):
    B, Hq, L, S = 2, 3, 200, 128 if E != 16 else 64
    q, k, _, _, _ = random_inputs(B, Hq, Hq, L, S, E, E, dtype, seed=400 + E)
    v = torch.eye(S, dtype=dtype)[None, None].expand(B, Hq, S, S).contiguous()
    if S < 128 and dtype == torch.bfloat16:
        v = torch.nn.functional.pad(v, (0, 128 - S))
    d = oracle.Dropout(0.35, seed=77, offset=5)
    o, _ = sdpa.sdpa_forward(q.cuda(), k.cuda(), v.cuda(), None, 0.1, dropout=sdpa.Dropout(0.35, 77, 5))
    torch.cuda.synchronize()
    got_kept = (o[..., :S].float().cpu() != 0).numpy()
    for b in range(B):
        for h in range(Hq):
            keep = oracle.dropout_keep(d, b * Hq + h, np.arange(L), S)
            assert np.array_equal(got_kept[b, h], keep), (b, h)


CASES = [
    # B, Hq, Hkv, L, S, E, Ev, dtype, causal, mask, band
    (2, 4, 2, 300, 333, 128, 128, "bf16", True, "none", None),
    (1, 4, 4, 257, 400, 128, 128, "bf16", False, "bias", None),
    (2, 2, 2, 260, 260, 64, 64, "bf16", True, "none", None),
    (1, 4, 1, 300, 300, 128, 128, "bf16", False, "none", ([300], [250], "top_left", 0, 100)),
    (1, 2, 1, 120, 90, 32, 40, "bf16", True, "bias", None),       # CUDA-core bf16
    (2, 2, 2, 64, 64, 16, 16, "f32", True, "none", None),
    (1, 2, 1, 70, 90, 24, 16, "f32", False, "bias", ([70], [80], "bottom_right", 0, 30)),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_dropout_forward_backward(case):
    B, Hq, Hkv, L, S, E, Ev, dt, causal, mk, bd = case
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    n = CASES.index(case)
    q, k, v, dO, mask = random_inputs(B, Hq, Hkv, L, S, E, Ev, dtype, seed=410 + n, mask_kind=mk,
                                      mask_shape=(B, 1) if mk != "none" else None, p_block=0.2)
    od = oracle.Dropout(0.2, seed=1234 + n, offset=99)
    gd = sdpa.Dropout(0.2, 1234 + n, 99)
    ob = gb = None
    if bd is not None:
        lq, lk, align, right, left = bd
        ob = oracle.Band(lq, lk, align, right, left)
        gb = sdpa.Band(torch.tensor(lq, dtype=torch.int32, device="cuda"),
                       torch.tensor(lk, dtype=torch.int32, device="cuda"), align, right, left)
        causal = False
    gqa = Hq != Hkv
    bf16 = dtype == torch.bfloat16
    ref_o, ref_lse = oracle.ref_forward(q, k, v, mask, None, causal, gqa, band=ob, dropout=od)
    qd, kd, vd, dOd = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    md = None if mask is None else mask.cuda()
    o, lse = sdpa.sdpa_forward(qd, kd, vd, md, None, causal, gqa, band=gb, dropout=gd)
    torch.cuda.synchronize()
    check_forward(o, lse, ref_o, ref_lse, bf16)
    grads = sdpa.sdpa_backward(qd, kd, vd, o, dOd, lse, md, None, causal, gqa, band=gb, dropout=gd)
    torch.cuda.synchronize()
    refs = oracle.ref_backward(q, k, v, dO, mask, None, causal, gqa, band=ob, dropout=od)
    dead = np.isneginf(ref_lse)
    check_backward(grads, refs, dead, np.zeros((B, Hkv, S), bool), bf16)
    assert sdpa.last_device_status() == 0


def test_dropout_zero_is_plain_and_seed_determines_the_call():
    q, k, v, dO, _ = random_inputs(1, 4, 2, 300, 300, 128, 128, torch.bfloat16, seed=430)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o0, l0 = sdpa.sdpa_forward(qd, kd, vd, None, None, True, True)
    o1, l1 = sdpa.sdpa_forward(qd, kd, vd, None, None, True, True, dropout=sdpa.Dropout(0.0, 5))
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    a, _ = sdpa.sdpa_forward(qd, kd, vd, None, None, True, True, dropout=sdpa.Dropout(0.3, 5, 1))
    b, _ = sdpa.sdpa_forward(qd, kd, vd, None, None, True, True, dropout=sdpa.Dropout(0.3, 5, 1))
    c, _ = sdpa.sdpa_forward(qd, kd, vd, None, None, True, True, dropout=sdpa.Dropout(0.3, 5, 2))
    torch.cuda.synchronize()
    assert torch.equal(a, b) and not torch.equal(a, c)
