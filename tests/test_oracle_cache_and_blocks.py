"""Pins for the oracle's cache ops and host block manager (CPU only)."""

import json
import os

import numpy as np
import pytest

import oracle
from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- block manager

def test_lifecycle_of_fig_19_6():
    g = json.load(open(os.path.join(GOLDEN, "kvs_fig19_6_lifecycle.json")))
    bs = g["block_size"]
    assert len(g["prompt"].split()) == g["prompt_tokens"]
    pool = oracle.BlockPool(16)
    t = oracle.BlockTable(pool, bs)
    for _ in range(g["prompt_tokens"]):
        t.append_slot()
    assert len(t.mapping) == g["prompt_blocks"]
    for allocates in g["allocates_on_decode_token"]:
        before = len(t.mapping)
        t.append_slot()
        assert (len(t.mapping) > before) == allocates
    t.release_all()
    assert sorted(pool.free_list) == list(range(16))


def test_allocation_takes_the_end_of_the_free_list_and_exhausts():
    pool = oracle.BlockPool(3)
    assert [pool.allocate() for _ in range(3)] == [2, 1, 0]
    with pytest.raises(oracle.BlockExhausted):
        pool.allocate()
    pool.release(1)
    assert pool.allocate() == 1


def test_slots_address_block_and_offset():
    pool = oracle.BlockPool(8)
    t = oracle.BlockTable(pool, 4)
    slots = [t.append_slot() for _ in range(10)]
    for n, s in enumerate(slots):
        assert s // 4 == t.mapping[n // 4] and s % 4 == n % 4


def test_copy_on_write_with_eight_samples():
    bs, S = 4, 8
    pool = oracle.BlockPool(64)
    parent = oracle.BlockTable(pool, bs)
    for _ in range(6):                      # block 1 is partial (2 of 4)
        parent.append_slot()
    kids = [parent] + [parent.fork() for _ in range(S - 1)]
    shared_tail = parent.mapping[1]
    assert pool.ref_counts[shared_tail] == S and pool.ref_counts[parent.mapping[0]] == S
    for kid in kids:                        # each sample writes its own next token
        kid.append_slot()
    copies = [c for kid in kids for c in kid.copies]
    assert len(copies) == S - 1              # the last writer finds refcount 1
    assert all(src == shared_tail for src, _ in copies)
    assert len({dst for _, dst in copies}) == S - 1
    assert pool.ref_counts[shared_tail] == 1
    assert pool.ref_counts[parent.mapping[0]] == S   # full prompt block still shared
    for kid in kids:
        kid.release_all()
    assert len(pool.free_list) == 64


@pytest.mark.parametrize("bs", [4, 16, 32])
def test_tail_waste_is_below_one_block(bs):
    rng = np.random.default_rng(bs)
    pool = oracle.BlockPool(4096)
    for L in rng.integers(1, 500, size=40):
        t = oracle.BlockTable(pool, bs)
        for _ in range(int(L)):
            t.append_slot()
        assert 0 <= len(t.mapping) * bs - L <= bs - 1
        t.release_all()


def test_13b_sequence_kv_size_claim():
    g = json.load(open(os.path.join(GOLDEN, "sch_13b_kv_size.json")))
    per_token = 2 * g["layers"] * g["heads"] * g["head_dim"] * g["bytes_per_element"]
    assert per_token == 819_200
    assert 2048 * per_token < g["claim_bytes"] < 2100 * per_token


# ---------------------------------------------------------------- cache ops

def test_reshape_and_cache_writes_only_addressed_slots():
    rng = np.random.default_rng(0)
    NB, bs, H, D = 6, 4, 2, 3
    k = rng.standard_normal((NB, bs, H, D))
    v = rng.standard_normal((NB, bs, H, D))
    key = rng.standard_normal((4, H, D))
    val = rng.standard_normal((4, H, D))
    slots = np.array([5, -1, 23, 8])
    k2, v2 = oracle.reshape_and_cache(key, val, slots, k, v)
    touched = {(1, 1), (5, 3), (2, 0)}
    for blk in range(NB):
        for off in range(bs):
            if (blk, off) in touched:
                continue
            assert np.array_equal(k2[blk, off], k[blk, off])
            assert np.array_equal(v2[blk, off], v[blk, off])
    assert np.array_equal(k2[1, 1], key[0]) and np.array_equal(v2[5, 3], val[2])
    assert np.array_equal(k2[2, 0], key[3])
    assert np.array_equal(k, oracle.reshape_and_cache(key, val, np.full(4, -1), k, v)[0])


def test_append_then_gather_round_trip_bf16_bits():
    rng = np.random.default_rng(1)
    bs, H, D, T = 4, 2, 8, 11
    pool = oracle.BlockPool(9)
    t = oracle.BlockTable(pool, bs)
    bits = rng.integers(0, 1 << 16, size=(T, H, D), dtype=np.uint16)
    k = np.zeros((9, bs, H, D), np.uint16)
    slots = np.array([t.append_slot() for _ in range(T)])
    k2, _ = oracle.reshape_and_cache(bits, bits, slots, k, k)
    K, _ = A.gather_context(k2, k2, t.mapping, T)
    assert np.array_equal(K.astype(np.uint16), bits)


def test_copy_blocks_is_bit_identical_and_local():
    rng = np.random.default_rng(2)
    k = rng.integers(0, 1 << 16, size=(10, 4, 2, 8), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(10, 4, 2, 8), dtype=np.uint16)
    pairs = np.array([[1, 7], [1, 8], [4, 9]])
    k2, v2 = oracle.copy_blocks(k, v, pairs)
    for src, dst in pairs:
        assert np.array_equal(k2[dst], k[src]) and np.array_equal(v2[dst], v[src])
    for blk in range(10):
        if blk not in (7, 8, 9):
            assert np.array_equal(k2[blk], k[blk]) and np.array_equal(v2[blk], v[blk])


def test_swap_out_and_back_is_identity():
    rng = np.random.default_rng(3)
    dev_k = rng.integers(0, 1 << 16, size=(12, 4, 2, 8), dtype=np.uint16)
    dev_v = rng.integers(0, 1 << 16, size=(12, 4, 2, 8), dtype=np.uint16)
    host_k = np.zeros((5, 4, 2, 8), np.uint16)
    host_v = np.zeros((5, 4, 2, 8), np.uint16)
    out_pairs = np.array([[3, 0], [7, 4], [11, 2]])
    hk, hv = oracle.swap_blocks(host_k, host_v, dev_k, dev_v, out_pairs)
    for s, d in out_pairs:
        assert np.array_equal(hk[d], dev_k[s]) and np.array_equal(hv[d], dev_v[s])
    assert not hk[1].any() and not hk[3].any()           # untouched host blocks
    # back into fresh device blocks, then a table remap sees the same data
    back = np.array([[0, 9], [4, 10], [2, 1]])
    k2, v2 = oracle.swap_blocks(np.zeros_like(dev_k), np.zeros_like(dev_v), hk, hv, back)
    assert np.array_equal(k2[9], dev_k[3]) and np.array_equal(v2[10], dev_v[7]) and np.array_equal(k2[1], dev_k[11])
