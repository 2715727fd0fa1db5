"""The seeded workloads have the structure their docstrings promise (CPU)."""

import numpy as np
import torch
import pytest

from paged_kv_cache_307_gb300 import workloads as W
import oracle


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c4b32", "c5"])
def test_small_cases_are_well_formed(name):
    c = W.decode_case(name, small=True)
    s = c.spec
    B = c.q.shape[0]
    assert c.q.dtype == W.DTYPES[s.dtype] and c.k_cache.shape[1:] == (s.bs, s.Hkv, s.D)
    lens = c.context_lens.numpy()
    tables = c.block_tables.numpy()
    NB = c.num_blocks
    used = []
    for b in range(B):
        n = -(-int(lens[b]) // s.bs)
        assert (tables[b, :n] >= 0).all() and (tables[b, :n] < NB).all()
        assert (tables[b, n:] == NB).all()
        used.extend(tables[b, :n].tolist())
        # slot of the newest token, as the oracle's block table addresses it
        L = int(lens[b])
        slot = int(c.slot_mapping[b])
        if slot >= 0:
            assert slot == int(tables[b, (L - 1) // s.bs]) * s.bs + (L - 1) % s.bs
            assert torch.isnan(c.k_cache[slot // s.bs, slot % s.bs].float()).all()
    if name != "c5":
        assert len(set(used)) == len(used)   # private blocks only
    c2 = W.decode_case(name, small=True)
    assert torch.equal(c.q, c2.q) and torch.equal(c.block_tables, c2.block_tables)


def test_c1_is_the_worked_example_shape():
    c = W.decode_case("c1")
    assert c.num_blocks == 16 and int(c.context_lens[0]) == 10
    assert (c.block_tables[0, :3] < 16).all() and c.block_tables.shape[1] == 3


def test_c2_lengths_and_pool():
    c = W.decode_case("c2", nan_fill=False)
    lens = c.context_lens.numpy()
    assert lens.min() >= 128 and lens.max() <= 2048 and len(lens) == 64
    assert c.block_tables.shape[1] == 128


def test_c5_shares_prompt_blocks_eight_ways():
    c = W.decode_case("c5", small=True)
    P, S = c.extra["prompts"], c.extra["samples"]
    tables = c.block_tables.numpy()
    pre = c.extra["prefix"] // c.spec.bs
    for p in range(P):
        rows = tables[p * S:(p + 1) * S, :pre]
        assert (rows == rows[0]).all()
    assert (c.context_lens.numpy() >= c.extra["prefix"]).all()


def test_c5_group_descriptor_is_the_sharing_the_tables_hold():
    for small in (True, False):
        c = W.decode_case("c5", small=small, nan_fill=False)
        gs, sb = oracle.shared_prefix_groups(c.block_tables.numpy(), c.context_lens.numpy(), c.spec.bs)
        assert np.array_equal(gs, c.extra["group_start"].numpy())
        assert np.array_equal(sb, c.extra["shared_blocks"].numpy())


def test_cow_pairs_follow_the_block_manager():
    cc = W.cow_case(small=True)
    P, S = len(cc["prompt_len"]), cc["samples"]
    pairs = cc["pairs"].numpy()
    assert pairs.shape == (P * (S - 1), 2)
    assert len(set(pairs[:, 1].tolist())) == len(pairs)
    assert not set(pairs[:, 1].tolist()) & set(pairs[:, 0].tolist())
    # the oracle's block manager asks for the same number of copies per prompt
    for p in range(P):
        pool = oracle.BlockPool(256)
        parent = oracle.BlockTable(pool, cc["block_size"])
        for _ in range(int(cc["prompt_len"][p])):
            parent.append_slot()
        kids = [parent] + [parent.fork() for _ in range(S - 1)]
        for kid in kids:
            kid.append_slot()
        assert sum(len(k.copies) for k in kids) == (pairs[:, 0] == cc["prompt_blocks"][p, -1]).sum()


def test_full_size_c4_lengths_only():
    rng = np.random.default_rng(W.SPECS["c4"].seed)
    lens = W._lengths(W.SPECS["c4"], 256, rng)
    assert lens.min() >= 1024 and lens.max() <= 32768
