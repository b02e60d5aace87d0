"""Forward, backward and decode calls captured in a CUDA graph.

For problems small enough that the host's per-call work (argument checks,
tensor-map encoding, launches) is comparable to the device time, a caller
captures its steps once and replays them.  The library's calls only enqueue
work on the given stream (kernel launches, programmatic dependent launches
included, and the padded forward's counter reset), so a captured step must
give the same bits as the direct calls: O, LSE, dK and dV exactly, and dQ up
to the order of its fp32 reductions (the key-tile CTAs add into the dQ
accumulator in whatever order they finish, run to run, captured or not).
The first call on the device runs before the capture, as the library's
per-context set-up requires.
"""
import pytest
import torch

import scaled_dot_product_sm_gb300 as sdpa
from workloads import random_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdpa.build()
    sdpa.load_library()


def _same(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


@pytest.mark.parametrize("padded", [False, True])
def test_captured_training_step_matches_direct_calls(padded):
    B, Hq, Hkv, L, E = 2, 8, 2, 700, 128
    q, k, v, dO, _ = random_inputs(B, Hq, Hkv, L, L, E, E, torch.bfloat16, seed=61)
    q, k, v, dO = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    band = None
    if padded:
        lens = torch.tensor([700, 413], dtype=torch.int32, device="cuda")
        band = sdpa.Band(lens, lens, "top_left", 0, None)
    o, lse = torch.empty_like(q), torch.empty(B, Hq, L, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fws = torch.empty(max(16, sdpa.forward_workspace_bytes(q, k, v)), dtype=torch.uint8, device="cuda")
    bws = torch.empty(sdpa.backward_workspace_bytes(q, k, v), dtype=torch.uint8, device="cuda")

    def step():
        sdpa.sdpa_forward(q, k, v, None, None, band is None, True, out=o, lse=lse, workspace=fws, band=band)
        sdpa.sdpa_backward(q, k, v, o, dO, lse, None, None, band is None, True, dq=dq, dk=dk, dv=dv, workspace=bws,
                           band=band)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (o, lse, dq, dk, dv):
        t.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert sdpa.last_device_status() == 0
    for got, want in zip((o, lse, dk, dv), (ref[0], ref[1], ref[3], ref[4])):
        assert _same(got, want)
    err = float((dq.float() - ref[2].float()).norm() / ref[2].float().norm())
    assert err <= 1e-4, err


def test_captured_decode_matches_direct_call():
    q, k, v, _, _ = random_inputs(4, 16, 4, 1, 5000, 128, 128, torch.bfloat16, seed=62)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o, lse = torch.empty(4, 16, 1, 128, dtype=torch.bfloat16, device="cuda"), torch.empty(4, 16, 1, device="cuda")
    ws = torch.empty(sdpa.decode_workspace_bytes(q, k, v, 0), dtype=torch.uint8, device="cuda")

    def call():
        sdpa.sdpa_decode(q, k, v, None, None, True, 0, out=o, lse=lse, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = (o.clone(), lse.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    o.fill_(float("nan"))
    lse.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert _same(o, ref[0]) and _same(lse, ref[1])
