"""GPU parity of the paged-KV decode (sdpa_decode_paged) against the oracle.

K/V caches are cut into blocks, shuffled into containers with spare blocks, and
addressed through page tables whose entries past each sequence's length are
garbage (other blocks, -1, past the container).  Results must match the
float64 oracle on the gathered caches (bf16 tolerances) and be bit-identical
to the dense decode of the same caches with the same split count.
"""
import numpy as np
import pytest
import torch

import oracle
import scaled_dot_product_sm_gb300 as sdpa
from test_gpu_parity import check_forward
from workloads import random_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdpa.build()
    sdpa.load_library()


def _paginate(dense, bs, lens, rng, spare=3):
    """Container [nblk, H, bs, D] and table [B, ceil(S/bs)] holding `dense` [B, H, S, D]."""
    B, H, S, D = dense.shape
    nb_seq = (S + bs - 1) // bs
    pad = nb_seq * bs - S
    d = torch.nn.functional.pad(dense, (0, 0, 0, pad)) if pad else dense
    blocks = d.reshape(B, H, nb_seq, bs, D).permute(0, 2, 1, 3, 4).reshape(B * nb_seq, H, bs, D)
    nblk = B * nb_seq + spare
    perm = torch.from_numpy(rng.permutation(nblk)[:B * nb_seq])
    noise = torch.Generator().manual_seed(int(rng.integers(0, 2**31)))
    container = torch.randn(nblk, H, bs, D, generator=noise).to(dense.dtype)   # spare blocks hold noise
    container[perm] = blocks
    table = perm.reshape(B, nb_seq).to(torch.int32).clone()
    for b in range(B):                                     # entries past the length: garbage
        first_unused = (lens[b] + bs - 1) // bs
        for i in range(first_unused, nb_seq):
            table[b, i] = int(rng.choice([-1, nblk + 5, int(rng.integers(0, nblk))]))
    return container, table


CASES = [
    # B, Hq, Hkv, L, S, E, bs_k, bs_v, lens, splits
    (4, 8, 2, 1, 2000, 128, 64, 64, [2000, 1, 1337, 0], 0),
    (3, 8, 2, 1, 1500, 128, 16, 16, [1500, 700, 65], 5),
    (2, 4, 1, 2, 1000, 64, 8, 128, [1000, 333], 0),
    (2, 16, 2, 1, 4096, 128, 256, 32, [4096, 2500], 3),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_paged_decode(case):
    B, Hq, Hkv, L, S, E, bs_k, bs_v, lens, splits = case
    rng = np.random.default_rng(300 + CASES.index(case))
    q, k, v, _, _ = random_inputs(B, Hq, Hkv, L, S, E, E, torch.bfloat16, seed=300 + CASES.index(case))
    kc, tk = _paginate(k, bs_k, lens, rng)
    vc, tv = _paginate(v, bs_v, lens, rng)
    width = max(tk.shape[1], tv.shape[1])
    tk = torch.nn.functional.pad(tk, (0, width - tk.shape[1]), value=-1)
    tv = torch.nn.functional.pad(tv, (0, width - tv.shape[1]), value=-1)
    ob = oracle.Band(None, lens, "bottom_right", 0, None)
    ref_o, ref_lse = oracle.ref_forward_paged(q, kc, vc, tk.numpy(), tv.numpy(), bs_k, bs_v, S, None, None, True,
                                              ob)
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    gb = sdpa.Band(None, lens_d, "bottom_right", 0, None)
    o, lse = sdpa.sdpa_decode_paged(q.cuda(), kc.cuda(), vc.cuda(), tk.cuda(), tv.cuda(), S, None, None, True,
                                    splits, band=gb)
    torch.cuda.synchronize()
    check_forward(o, lse, ref_o, ref_lse, True)
    # the dense decode of the same caches, same splits: bit-identical
    od, lsed = sdpa.sdpa_decode(q.cuda(), k.cuda(), v.cuda(), None, None, True, splits, band=gb)
    torch.cuda.synchronize()
    assert torch.equal(o, od) and torch.equal(lse, lsed)
    assert sdpa.last_device_status() == 0


def test_paged_decode_full_size():
    """The 32k-key GQA decode workload (B = 16, Hq = 32, Hkv = 8, S = 32768) with its caches cut into
    64-key blocks shuffled across one container: bit-identical to the dense decode, and sampled KV
    groups match the oracle."""
    import workloads
    w = workloads.get("gqa_decode_s32k")
    q, k, v, _, _ = workloads.make_inputs(w, seed=0, with_grad=False)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    bs = 64
    nb = w.S // bs
    perm = torch.randperm(w.B * nb, device="cuda", generator=torch.Generator(device="cuda").manual_seed(5))

    def container(x):   # block i of sequence b lands at perm[b * nb + i]
        B, H, S, D = x.shape
        blocks = x.reshape(B, H, nb, bs, D).permute(0, 2, 1, 3, 4).reshape(B * nb, H, bs, D)
        c = torch.empty_like(blocks)
        c[perm] = blocks
        return c
    table = perm.reshape(w.B, nb).to(torch.int32).contiguous()
    o, lse = sdpa.sdpa_decode_paged(qd, container(kd), container(vd), table, table, w.S, None, w.scale, True, 0)
    od, lsed = sdpa.sdpa_decode(qd, kd, vd, None, w.scale, True, 0)
    torch.cuda.synchronize()
    assert sdpa.last_device_status() == 0
    assert torch.equal(o, od) and torch.equal(lse, lsed)
    G = w.Hq // w.Hkv
    for b, kv in ((0, 0), (9, 3), (15, 7)):
        ref_o, ref_lse = oracle.ref_group(q, k, v, None, b, kv, None, w.scale, False)
        sl = slice(kv * G, (kv + 1) * G)
        got = o[b, sl].float().cpu().double().numpy()
        assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= 5e-3
        assert np.abs(lse[b, sl].cpu().double().numpy() - ref_lse).max() <= 1e-3
