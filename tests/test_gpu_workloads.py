"""Full-size workloads, in the launch configuration the benchmark times.

The benchmark's workloads include the padding-length, sliding-window and dropout
variants, which run here with the same lengths, window and (seed 0, offset 0)
dropout as in the benchmark.

Each workload runs whole on the GPU; the float64 oracle then recomputes every
closed sub-problem of it (each KV group: the Hq/Hkv query heads sharing a KV
head, with all their keys and queries), so every output element of the call is
compared with the oracle, with the same tolerances as the small cases, group by
group.  (Every leading index is an independent problem: course chapter
"Scaled dot-product attention (forward and backward)", section 2.4.)  The
persistent forward hands units to CTAs in a fixed snake order and the backward
walks its key tiles in waves, so checking every group covers every CTA and
every wave.  Properties that hold at any size are checked on the whole tensors
as well: no NaN/Inf, LSE = -inf exactly on fully masked rows (and only there),
zero O/dQ rows there, and zero dK/dV rows for keys that no query may see.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_sm_gb300 as sdpa
import workloads

pytestmark = pytest.mark.gpu

BF_O, BF_G, BF_LSE = 5e-3, 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdpa.build()
    sdpa.load_library()


def rel_l2(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30))


def run_workload(name, groups=None):
    """Runs workload `name` whole on the GPU and compares the KV groups `groups`
    ((b, kv) pairs; None = every group) with the oracle."""
    w = workloads.get(name)
    q, k, v, dO, mask = workloads.make_inputs(w, seed=0, with_grad="bwd" in w.phases)
    dev = [None if x is None else x.cuda() for x in (q, k, v, dO, mask)]
    qd, kd, vd, dOd, md = dev
    spec = workloads.make_band(w, seed=0)
    band = ob = None
    if spec is not None:
        lens = [None if spec[n] is None else torch.tensor(spec[n], dtype=torch.int32, device="cuda")
                for n in ("seq_len_q", "seq_len_kv")]
        band = sdpa.Band(*lens, spec["alignment"], spec["right_bound"], spec["left_bound"])
        ob = oracle.Band(spec["seq_len_q"], spec["seq_len_kv"], spec["alignment"], spec["right_bound"],
                         spec["left_bound"])
    drop = sdpa.Dropout(w.dropout, 0, 0) if w.dropout > 0 else None
    odrop = oracle.Dropout(w.dropout, 0, 0) if w.dropout > 0 else None
    o, lse = sdpa.sdpa_forward(qd, kd, vd, md, w.scale, w.is_causal, w.enable_gqa, band=band, dropout=drop)
    grads = None
    if "bwd" in w.phases:
        grads = sdpa.sdpa_backward(qd, kd, vd, o, dOd, lse, md, w.scale, w.is_causal, w.enable_gqa, band=band,
                                   dropout=drop)
    torch.cuda.synchronize()
    assert sdpa.last_device_status() == 0
    assert torch.isfinite(o).all()
    if grads is not None:
        for g in grads:
            assert torch.isfinite(g).all()
    G = w.Hq // w.Hkv
    if groups is None:
        groups = [(b, kv) for b in range(w.B) for kv in range(w.Hkv)]
    o_h, lse_h = o.float().cpu(), lse.cpu()
    g_h = None if grads is None else [g.float().cpu() for g in grads]
    worst = {"O": 0.0, "dQ": 0.0, "dK": 0.0, "dV": 0.0, "LSE": 0.0}
    for b, kv in groups:
        sl = slice(kv * G, (kv + 1) * G)
        out = oracle.ref_group(q, k, v, dO, b, kv, mask, w.scale, w.is_causal, band=ob, dropout=odrop)
        ref_o, ref_lse = out[0], out[1]
        lg = lse_h[b, sl].double().numpy()
        dead = np.isneginf(ref_lse)
        assert np.array_equal(np.isneginf(lg), dead), (name, b, kv)
        if (~dead).any():
            e_l = float(np.abs(lg[~dead] - ref_lse[~dead]).max())
            assert e_l <= BF_LSE, (name, b, kv, e_l)
            worst["LSE"] = max(worst["LSE"], e_l)
        og = o_h[b, sl].double().numpy()
        assert np.all(og[dead] == 0.0)
        e_o = rel_l2(og, ref_o)
        assert e_o <= BF_O, (name, b, kv, e_o)
        worst["O"] = max(worst["O"], e_o)
        if g_h is not None:
            dq, dk, dv = g_h
            dqg = dq[b, sl].double().numpy()
            e_q = rel_l2(dqg, out[2])
            e_k = rel_l2(dk[b, kv].double().numpy(), out[3])
            e_v = rel_l2(dv[b, kv].double().numpy(), out[4])
            assert max(e_q, e_k, e_v) <= BF_G, (name, b, kv, e_q, e_k, e_v)
            assert np.all(dqg[dead] == 0.0)
            worst.update(dQ=max(worst["dQ"], e_q), dK=max(worst["dK"], e_k), dV=max(worst["dV"], e_v))
    print(f"{name}: {len(groups)} KV groups vs the oracle; worst rel-L2 / LSE abs error {worst}")
    return w, q, k, v, mask, o, lse, grads


def test_mha_causal_e64():
    run_workload("mha_causal_e64")


def test_gqa_causal_e128():
    run_workload("gqa_causal_e128")


def test_padded_mask_e128():
    w, q, k, v, mask, o, lse, grads = run_workload("padded_mask_e128")
    m = mask[:, 0]                                         # [B, L, S]
    dead_rows = torch.isneginf(m).all(dim=-1)              # [B, L]
    lse_dead = torch.isneginf(lse).cpu()                   # [B, H, L]
    assert torch.equal(lse_dead, dead_rows[:, None, :].expand_as(lse_dead))
    assert (o.cpu()[dead_rows[:, None, :].expand(-1, w.Hq, -1)] == 0).all()
    dq, dk, dv = grads
    assert (dq.cpu()[dead_rows[:, None, :].expand(-1, w.Hq, -1)] == 0).all()
    dead_keys = torch.isneginf(m).all(dim=1)               # [B, S]: blocked for every query
    sel = dead_keys[:, None, :].expand(-1, w.Hkv, -1)
    assert (dk.cpu()[sel] == 0).all() and (dv.cpu()[sel] == 0).all()


def test_gqa_decode_s32k():
    run_workload("gqa_decode_s32k")


def test_padded_seqlen_e128():
    """Padding lengths instead of a mask: keys at or past a sequence's length get exact zero dK, dV."""
    w, q, k, v, mask, o, lse, grads = run_workload("padded_seqlen_e128")
    lens = workloads.make_band(w, seed=0)["seq_len_kv"]
    dq, dk, dv = grads
    for b, n in enumerate(lens):
        assert int(torch.count_nonzero(dk[b, :, n:])) == 0 and int(torch.count_nonzero(dv[b, :, n:])) == 0


def test_gqa_swa_e128():
    run_workload("gqa_swa_e128")


def test_gqa_causal_dropout_e128():
    run_workload("gqa_causal_dropout_e128")
