"""GPU parity at sizes past 2^31 elements in one tensor, where 32-bit offsets would wrap.

The outputs are checked on closed sub-problems the float64 oracle computes exactly:

* prefill: Q, O, dO and dQ hold 2^31 + 131,072 elements each (B = 1, Hq = 128,
  Hkv = 8, L = 131,077, S = 333, E = 128).  Sampled query rows are independent
  problems (course chapter "Scaled dot-product attention (forward and backward)",
  section 2.1), so their O and LSE come from the oracle's row restriction.  The
  backward runs with dO zero except on the sampled rows of one KV group: then dQ is
  zero on every other row, dK and dV are zero outside that group, and the group's
  dK and dV are those of the sampled rows alone (every term of section 2.3 carries
  a factor dO_i), which the oracle computes on the compressed problem.
* decode: K and V hold 2^24 + 77 keys x 128 = 2^31 + 9,856 elements each.  The keys
  repeat with period 4,099, and attention over keys repeated n_r times equals
  attention over the 4,099 distinct keys with the additive bias ln n_r (softmax
  weights e^(s_r) n_r / sum; pinned on the CPU in test_oracle.py), which the
  oracle computes.

Inputs are drawn on the GPU from seeded generators; only the sampled rows and the
small tensors are copied to the host.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_sm_gb300 as sdpa
from test_gpu_parity import check_forward

pytestmark = pytest.mark.gpu

BF_O, BF_G = 5e-3, 1e-2


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
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30))


def f64(t):
    return t.detach().float().cpu().double().numpy()


def test_prefill_past_2g_elements():
    B, Hq, Hkv, L, S, E = 1, 128, 8, 131077, 333, 128
    assert Hq * L * E > 2 ** 31
    G = Hq // Hkv
    g = torch.Generator(device="cuda").manual_seed(71)
    q = torch.randn(B, Hq, L, E, device="cuda", dtype=torch.bfloat16, generator=g)
    k = torch.randn(B, Hkv, S, E, device="cuda", dtype=torch.bfloat16, generator=g)
    v = torch.randn(B, Hkv, S, E, device="cuda", dtype=torch.bfloat16, generator=g)
    o, lse = sdpa.sdpa_forward(q, k, v, None, None, False, True)
    torch.cuda.synchronize()
    assert sdpa.last_device_status() == 0
    kc, vc = f64(k), f64(v)
    rows = np.array([0, 1, 127, 128, 65535, 65536, L - 2, L - 1])
    for h in (0, 55, 127):
        qr = f64(q[0, h, torch.from_numpy(rows).cuda()])[None, None]
        ref_o, ref_lse = oracle.ref_forward_rows(qr, kc[:, h // G:h // G + 1], vc[:, h // G:h // G + 1], 0, 0,
                                                 np.arange(len(rows)))
        got_o = f64(o[0, h, torch.from_numpy(rows).cuda()])
        got_lse = f64(lse[0, h, torch.from_numpy(rows).cuda()])
        assert rel_l2(got_o, ref_o) <= BF_O, (h, rel_l2(got_o, ref_o))
        assert np.abs(got_lse - ref_lse).max() <= 1e-3
    # backward with dO zero except on sampled rows of KV group 3
    kv = 3
    heads = [kv * G, kv * G + 7, kv * G + G - 1]
    dO = torch.zeros_like(q)
    gd = torch.Generator(device="cuda").manual_seed(72)
    idx = torch.from_numpy(rows).cuda()
    for h in heads:
        dO[0, h, idx] = torch.randn(len(rows), E, device="cuda", dtype=torch.bfloat16, generator=gd)
    dq, dk, dv = sdpa.sdpa_backward(q, k, v, o, dO, lse, None, None, False, True)
    torch.cuda.synchronize()
    assert sdpa.last_device_status() == 0
    # the compressed problem: the sampled rows of the group's heads against KV head kv
    qs = np.stack([f64(q[0, h, idx]) for h in heads])[None]        # [1, 3, R, E]
    dOs = np.stack([f64(dO[0, h, idx]) for h in heads])[None]
    ks, vs = kc[:, kv:kv + 1], vc[:, kv:kv + 1]
    ref_dq, ref_dk, ref_dv = oracle.ref_backward(qs, ks, vs, dOs, None, None, False, True)
    got_dq = np.stack([f64(dq[0, h, idx]) for h in heads])
    assert rel_l2(got_dq, ref_dq[0]) <= BF_G, rel_l2(got_dq, ref_dq[0])
    assert rel_l2(f64(dk[0, kv]), ref_dk[0, 0]) <= BF_G, rel_l2(f64(dk[0, kv]), ref_dk[0, 0])
    assert rel_l2(f64(dv[0, kv]), ref_dv[0, 0]) <= BF_G, rel_l2(f64(dv[0, kv]), ref_dv[0, 0])
    # zero everywhere else
    for h in heads:
        dq[0, h, idx] = 0
    assert int(torch.count_nonzero(dq)) == 0
    others = [i for i in range(Hkv) if i != kv]
    assert int(torch.count_nonzero(dk[0, others])) == 0 and int(torch.count_nonzero(dv[0, others])) == 0


@pytest.mark.parametrize("splits", [0, 5])
def test_decode_past_2g_elements(splits):
    B, Hq, Hkv, S, E, P = 1, 8, 1, 2 ** 24 + 77, 128, 4099
    assert S * E > 2 ** 31
    g = torch.Generator(device="cuda").manual_seed(73)
    q = torch.randn(B, Hq, 1, E, device="cuda", dtype=torch.bfloat16, generator=g)
    kb = torch.randn(B, Hkv, P, E, device="cuda", dtype=torch.bfloat16, generator=g)
    vb = torch.randn(B, Hkv, P, E, device="cuda", dtype=torch.bfloat16, generator=g)
    reps = -(-S // P)
    k = kb.repeat(1, 1, reps, 1)[:, :, :S].contiguous()
    v = vb.repeat(1, 1, reps, 1)[:, :, :S].contiguous()
    o, lse = sdpa.sdpa_decode(q, k, v, None, None, True, splits)
    torch.cuda.synchronize()
    assert sdpa.last_device_status() == 0
    del k, v
    n = np.array([(S - 1 - r) // P + 1 for r in range(P)], dtype=np.float64)   # copies of key r
    bias = np.log(n)[None, None, None, :]                                          # [1, 1, 1, P]
    ref_o, ref_lse = oracle.ref_forward(f64(q), f64(kb), f64(vb), bias, None, False, True)
    check_forward(o, lse, ref_o, ref_lse, True)
