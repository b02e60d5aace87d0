"""Pins of the oracle's paged K/V gather (cuDNN "Attention" page, Paged attention:
K_cache[b,h,s,d] = K_container[page_table_k[b, s / bs_k], h, s mod bs_k, d]).

The gather is checked against a dense cache laid out block by block (identity
table), the same cache with its blocks shuffled, a tiny hand-worked table, and
the independence of a padded sequence's result from table entries past its
length.  A planted off-by-one in the offset is caught.
"""
import numpy as np
import pytest

import oracle
from oracle import sdpa_oracle as so


def _dense(B, H, S, D, seed):
    return np.random.default_rng(seed).standard_normal((B, H, S, D))


def _to_container(dense, bs, perm=None):
    """Blocks of bs keys of every sequence, one after another; perm reorders them."""
    B, H, S, D = dense.shape
    nblk = S // bs
    blocks = dense.reshape(B, H, nblk, bs, D).transpose(0, 2, 1, 3, 4).reshape(B * nblk, H, bs, D)
    table = np.arange(B * nblk).reshape(B, nblk)
    if perm is not None:                 # block i of the layout moves to position perm[i]
        moved = np.empty_like(blocks)
        moved[perm] = blocks
        blocks, table = moved, perm[table]
    return blocks, table


def pin_identity_layout():
    dense = _dense(2, 3, 16, 4, 1)
    c, t = _to_container(dense, 4)
    np.testing.assert_array_equal(oracle.gather_paged(c, t, 4, 16), dense)


def pin_shuffled_blocks():
    dense = _dense(3, 2, 24, 5, 2)
    perm = np.random.default_rng(3).permutation(3 * 24 // 8)
    c, t = _to_container(dense, 8, perm)
    np.testing.assert_array_equal(oracle.gather_paged(c, t, 8, 24), dense)


def pin_hand_table():
    # container of 3 blocks of 2 keys, one head, width 1: block p holds values 10p, 10p+1
    c = np.array([[[[0.0], [1.0]]], [[[10.0], [11.0]]], [[[20.0], [21.0]]]])
    got = oracle.gather_paged(c, [[2, 0], [1, 1]], 2, 4)
    np.testing.assert_array_equal(got[0, 0, :, 0], [20.0, 21.0, 0.0, 1.0])
    np.testing.assert_array_equal(got[1, 0, :, 0], [10.0, 11.0, 10.0, 11.0])


def pin_entries_past_length_do_not_matter():
    B, Hq, Hkv, S, E, bs = 2, 4, 2, 32, 8, 8
    rng = np.random.default_rng(4)
    q = rng.standard_normal((B, Hq, 1, E))
    kc = rng.standard_normal((10, Hkv, bs, E))
    vc = rng.standard_normal((10, Hkv, bs, E))
    table = rng.integers(0, 10, (B, S // bs))
    lens = [13, 24]
    band = oracle.Band(None, lens, "bottom_right", 0, None)
    O, L = oracle.ref_forward_paged(q, kc, vc, table, table, bs, bs, S, None, 0.3, True, band)
    t2 = table.copy()
    t2[0, 2:] = [7, 99]          # blocks past sequence 0's 13 keys (and an out-of-range entry)
    t2[1, 3:] = 5
    O2, L2 = oracle.ref_forward_paged(q, kc, vc, t2, t2, bs, bs, S, None, 0.3, True, band)
    np.testing.assert_array_equal(O, O2)
    np.testing.assert_array_equal(L, L2)


PAGED_PINS = [pin_identity_layout, pin_shuffled_blocks, pin_hand_table, pin_entries_past_length_do_not_matter]


@pytest.mark.parametrize("pin", PAGED_PINS, ids=[p.__name__ for p in PAGED_PINS])
def test_paged_pin(pin):
    pin()


def test_paged_offset_mutant_is_caught(monkeypatch):
    real = so.gather_paged

    def off_by_one(container, page_table, block_size, S):
        out = real(container, page_table, block_size, S)
        return np.roll(out, 1, axis=2)   # keys shifted by one position
    monkeypatch.setattr(so, "gather_paged", off_by_one)
    monkeypatch.setattr(oracle, "gather_paged", off_by_one)
    failed = 0
    for pin in PAGED_PINS[:3]:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0


def test_paged_rejects_block_size_mismatch():
    with pytest.raises(ValueError):
        oracle.gather_paged(np.zeros((2, 1, 4, 1)), [[0]], 8, 8)
