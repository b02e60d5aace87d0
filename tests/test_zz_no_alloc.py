"""sdpa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers only own their input and output buffers: an operator plugin
inside another runtime that gets no scratch space, or a serving loop whose
device memory is fixed at start-up and may not call cudaMalloc afterwards.
sdpa_decode_noalloc gives them the split-KV decode with its split partials in
the library's own fixed device array instead of a caller workspace.  These
checks call it through the C ABI, call after call, and compare each result
with the float64 oracle (the tolerances of every bf16 parity test) and with
sdpa_decode (which takes a workspace) at the same split count: both run the
same kernels on the same partial layout, so the two must agree bit for bit.
The shared array keeps the previous call's partials, so a second call with
other inputs must not see stale data.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_sm_gb300 as sdpa
from workloads import random_inputs

pytestmark = pytest.mark.gpu

O_REL_L2 = 5e-3     # bf16 output tolerance used by every bf16 parity test
LSE_ABS = 1e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdpa.build()
    return sdpa.load_library()


def _noalloc(lib, q, k, v, mask, scale, gqa, splits):
    B, Hq, L, _ = q.shape
    o = torch.full((B, Hq, L, v.shape[3]), float("nan"), dtype=q.dtype, device=q.device)
    lse = torch.full((B, Hq, L), float("nan"), dtype=torch.float32, device=q.device)
    shp = sdpa._shape(q, k, v, mask)
    P = ctypes.c_void_p
    st = lib.sdpa_decode_noalloc(ctypes.byref(shp), P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()),
                                 None if mask is None else P(mask.data_ptr()),
                                 float("nan") if scale is None else float(scale), int(gqa), int(splits),
                                 P(o.data_ptr()), P(lse.data_ptr()),
                                 P(torch.cuda.current_stream().cuda_stream))
    return st, o, lse


def _against_oracle(o, lse, q, k, v, mask):
    """o, lse of a decode call against the float64 oracle on the same (CPU) inputs."""
    ref_o, ref_lse = oracle.ref_forward(q.cpu(), k.cpu(), v.cpu(), None if mask is None else mask.cpu(), None,
                                        False, True)
    a = o.float().cpu().double().numpy()
    assert np.isfinite(a).all()
    rel = np.linalg.norm(a - ref_o) / max(np.linalg.norm(ref_o), 1e-30)
    assert rel <= O_REL_L2, rel
    la = lse.cpu().double().numpy()
    dead = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(la), dead)
    assert np.all(a[dead] == 0.0)
    assert (~dead).any()
    assert np.abs(la[~dead] - ref_lse[~dead]).max() <= LSE_ABS


def _bit_identical(o, lse, o_ref, lse_ref):
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))


CALLS = [
    # B, Hq, Hkv, L, S, E, mask, splits, seed
    (4, 16, 4, 1, 3000, 128, False, 0, 21),
    (2, 8, 2, 2, 1500, 64, True, 5, 22),     # one of the two query rows fully masked
]


def test_noalloc_matches_oracle_and_workspace_decode_on_consecutive_calls(lib):
    for B, Hq, Hkv, L, S, E, with_mask, splits, seed in CALLS:
        q, k, v, _, mask = random_inputs(B, Hq, Hkv, L, S, E, E, torch.bfloat16, seed=seed,
                                         mask_kind="bias" if with_mask else "none", mask_shape=(1, Hq),
                                         full_rows=1 if with_mask else 0)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        md = None if mask is None else mask.cuda()
        st, o, lse = _noalloc(lib, qd, kd, vd, md, None, True, splits)
        o_ref, lse_ref = sdpa.sdpa_decode(qd, kd, vd, md, None, True, splits)
        torch.cuda.synchronize()
        assert st == 0, lib.sdpa_status_string(st)
        _against_oracle(o, lse, q, k, v, mask)
        _bit_identical(o, lse, o_ref, lse_ref)
    assert sdpa.last_device_status() == 0


def test_noalloc_rejects_scratch_beyond_the_maximum(lib):
    # 2*64 rows x 128 splits x (128 + 1) floats = 8.45 MB > SDPA_DECODE_STATIC_SCRATCH_BYTES (8 MiB)
    q, k, v, _, _ = random_inputs(2, 64, 8, 1, 8192, 128, 128, torch.bfloat16, seed=23)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    st, _, _ = _noalloc(lib, q, k, v, None, None, True, 128)
    assert st == 2   # SDPA_ERR_UNSUPPORTED, nothing enqueued
    st, o, lse = _noalloc(lib, q, k, v, None, None, True, 16)   # 1.06 MB: fits
    o_ref, lse_ref = sdpa.sdpa_decode(q, k, v, None, None, True, 16)
    torch.cuda.synchronize()
    assert st == 0
    _against_oracle(o, lse, q, k, v, None)
    _bit_identical(o, lse, o_ref, lse_ref)
