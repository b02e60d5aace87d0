"""sdpa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers only own their input and output buffers: an operator plugin
inside another runtime that gets no scratch space, or a serving loop whose
device memory is fixed at start-up and may not call cudaMalloc afterwards.
sdpa_decode_noalloc gives them the split-KV decode with its split partials in
the library's own fixed device array instead of a caller workspace.  These
checks call it through the C ABI and compare it with sdpa_decode (which takes
a workspace), call after call: the shared array keeps the previous call's
partials, so a second call with other inputs must not see stale data.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def _compare(o, lse, o_ref, lse_ref):
    a = o.float().cpu().double().numpy()
    r = o_ref.float().cpu().double().numpy()
    assert np.isfinite(a).all()
    rel = np.linalg.norm(a - r) / max(np.linalg.norm(r), 1e-30)
    assert rel <= O_REL_L2, rel
    la, lr = lse.cpu().double().numpy(), lse_ref.cpu().double().numpy()
    assert np.array_equal(np.isneginf(la), np.isneginf(lr))
    fin = np.isfinite(lr)
    assert fin.any()
    assert np.abs(la[fin] - lr[fin]).max() <= LSE_ABS


CALLS = [
    # B, Hq, Hkv, L, S, E, mask, splits, seed
    (4, 16, 4, 1, 3000, 128, False, 0, 21),
    (2, 8, 2, 2, 1500, 64, True, 5, 22),     # one of the two query rows fully masked
]


def test_noalloc_matches_workspace_decode_on_consecutive_calls(lib):
    for B, Hq, Hkv, L, S, E, with_mask, splits, seed in CALLS:
        q, k, v, _, mask = random_inputs(B, Hq, Hkv, L, S, E, E, torch.bfloat16, seed=seed,
                                         mask_kind="bias" if with_mask else "none", mask_shape=(1, Hq),
                                         full_rows=1 if with_mask else 0)
        q, k, v = q.cuda(), k.cuda(), v.cuda()
        mask = None if mask is None else mask.cuda()
        o_ref, lse_ref = sdpa.sdpa_decode(q, k, v, mask, None, True, splits)
        st, o, lse = _noalloc(lib, q, k, v, mask, None, True, splits)
        torch.cuda.synchronize()
        assert st == 0, lib.sdpa_status_string(st)
        _compare(o, lse, o_ref, lse_ref)
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
    _compare(o, lse, o_ref, lse_ref)
