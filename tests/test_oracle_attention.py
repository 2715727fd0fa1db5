"""Pins for the float64 attention oracle (CPU only).

Each check ties the oracle to something other than itself: exactly rounded
brute force, closed forms, the worked example the pages print, and
invariants.  ``test_planted_mistakes_are_caught`` plants plausible mistakes
in copies of the oracle and shows that a pin here fails for each.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_pool(rng, NB, bs, Hkv, D):
    return rng.standard_normal((NB, bs, Hkv, D)), rng.standard_normal((NB, bs, Hkv, D))


def scattered_case(rng, B, Hq, Hkv, D, bs, lens, nan_tail=True):
    nblk = [-(-L // bs) for L in lens]
    NB = sum(nblk) + 5
    k, v = rand_pool(rng, NB, bs, Hkv, D)
    perm = rng.permutation(NB)
    maxb = max(nblk) if nblk else 1
    tables = np.full((B, max(maxb, 1)), NB, dtype=np.int64)
    off = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[off:off + n]
        off += n
        if nan_tail and n:
            valid = lens[b] - (n - 1) * bs
            k[tables[b, n - 1], valid:] = np.nan
            v[tables[b, n - 1], valid:] = np.nan
    k[perm[off:]] = np.nan
    v[perm[off:]] = np.nan
    q = rng.standard_normal((B, Hq, D))
    return q, k, v, tables, np.array(lens)


# ---------------------------------------------------------------- definition pins

@pytest.mark.parametrize("T,Hq,Hkv,D", [(1, 1, 1, 1), (3, 2, 1, 4), (9, 4, 2, 3), (7, 3, 3, 2)])
def test_dense_matches_exact_brute_force(T, Hq, Hkv, D):
    rng = np.random.default_rng(T * 100 + Hq)
    q = rng.standard_normal((Hq, D)) * 2
    K = rng.standard_normal((T, Hkv, D))
    V = rng.standard_normal((T, Hkv, D))
    s = 0.7
    np.testing.assert_allclose(A.dense_attention(q, K, V, s),
                               A.brute_force_attention(q, K, V, s), rtol=0, atol=1e-13)


def test_closed_form_two_tokens_with_scale():
    # q=2, keys 1 and 0, scale 1/2: scores 1 and 0, weights e/(1+e), 1/(1+e)
    q = np.array([[2.0]])
    K = np.array([[[1.0]], [[0.0]]])
    V = np.array([[[1.0]], [[0.0]]])
    out = A.dense_attention(q, K, V, 0.5)
    assert abs(out[0, 0] - math.e / (1 + math.e)) < 1e-15


def test_closed_form_single_token_is_its_value():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((4, 8))
    K = rng.standard_normal((1, 2, 8))
    V = rng.standard_normal((1, 2, 8))
    out = A.dense_attention(q, K, V, 0.3)
    np.testing.assert_array_equal(out[:2], np.broadcast_to(V[0, 0], (2, 8)))
    np.testing.assert_array_equal(out[2:], np.broadcast_to(V[0, 1], (2, 8)))


def test_closed_form_identical_keys_give_mean_value():
    rng = np.random.default_rng(1)
    T = 6
    K = np.broadcast_to(rng.standard_normal((1, 1, 5)), (T, 1, 5)).copy()
    V = rng.standard_normal((T, 1, 5))
    out = A.dense_attention(rng.standard_normal((1, 5)), K, V, 1.0)
    np.testing.assert_allclose(out[0], V[:, 0].mean(axis=0), atol=1e-15)


def test_closed_form_dominant_score_selects_its_value():
    T, D = 5, 4
    K = np.zeros((T, 1, D))
    K[3, 0, 0] = 1.0
    V = np.arange(T * D, dtype=np.float64).reshape(T, 1, D)
    q = np.zeros((1, D))
    q[0, 0] = 1e4
    out = A.dense_attention(q, K, V, 1.0)
    np.testing.assert_array_equal(out[0], V[3, 0])


def test_gqa_head_grouping():
    # 4 query heads over 2 KV heads: heads 0,1 read KV head 0, heads 2,3 head 1
    T, D = 3, 2
    K = np.random.default_rng(2).standard_normal((T, 2, D))
    V = np.zeros((T, 2, D))
    V[:, 0] = 1.0
    V[:, 1] = 2.0
    out = A.dense_attention(np.random.default_rng(3).standard_normal((4, D)), K, V, 1.0)
    np.testing.assert_allclose(out[:, 0], [1, 1, 2, 2], atol=1e-15)


def test_empty_context_is_zero():
    q = np.ones((2, 3))
    K = np.zeros((0, 1, 3))
    assert not A.dense_attention(q, K, K, 1.0).any()
    k = np.full((2, 4, 1, 3), np.nan)
    assert not A.paged_attention_walk(q, k, k, [0], 0, 1.0).any()


# ---------------------------------------------------------------- paged walk

@pytest.mark.parametrize("bs,Hq,Hkv,D,lens", [
    (4, 8, 8, 32, [10]),
    (16, 4, 2, 16, [1, 16, 17, 100]),
    (8, 6, 3, 8, [33, 5, 64]),
    (32, 2, 1, 4, [31, 96, 97]),
])
def test_walk_equals_dense(bs, Hq, Hkv, D, lens):
    rng = np.random.default_rng(sum(lens) + bs)
    q, k, v, tables, L = scattered_case(rng, len(lens), Hq, Hkv, D, bs, lens)
    walk = A.paged_decode(q, k, v, tables, L, 0.25, method="walk")
    dense = A.paged_decode(q, k, v, tables, L, 0.25, method="dense")
    assert np.isfinite(walk).all()          # NaN slots past `valid` never read
    np.testing.assert_allclose(walk, dense, rtol=0, atol=1e-12)


def test_worked_example_of_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "kvs_19_2_3_worked_example.json")))
    NB, bs, H, D, T = g["num_blocks"], g["block_size"], g["num_heads"], g["head_dim"], g["seq_len"]
    rng = np.random.default_rng(11)
    pool = oracle.BlockPool(NB)
    table = oracle.BlockTable(pool, bs)
    k = np.zeros((NB, bs, H, D))
    v = np.zeros((NB, bs, H, D))
    keys = rng.standard_normal((T, H, D))
    vals = rng.standard_normal((T, H, D))
    slots = [table.append_slot() for _ in range(T)]
    k, v = oracle.reshape_and_cache(keys, vals, np.array(slots), k, v)
    assert len(table.mapping) == g["blocks_used"]
    valid = [min(bs, T - j * bs) for j in range(len(table.mapping))]
    assert valid == g["valid_per_block"]
    q = rng.standard_normal((H, D))
    scale = 1.0 / math.sqrt(D)
    paged = A.paged_attention_walk(q, k, v, table.mapping, table.num_filled, scale)
    standard = A.dense_attention(q, keys, vals, scale)
    assert np.abs(paged - standard).max() < g["max_error_bound"]
    # the same walk carried out in fp32 lands near the printed 2^-22 scale
    q32, k32, v32 = q.astype(np.float32), k.astype(np.float32), v.astype(np.float32)
    ref = A.dense_attention(q32, keys.astype(np.float32), vals.astype(np.float32), scale)
    err32 = np.abs(_walk_fp32(q32, k32, v32, table.mapping, T, np.float32(scale)) - ref).max()
    assert err32 < g["max_error_bound"]
    table.release_all()
    assert len(pool.free_list) == g["free_after_release"]


def _walk_fp32(q, k, v, mapping, L, scale):
    """The block walk with every operation in float32 (used only to show the
    pages' fp32 error scale)."""
    H, D = q.shape
    bs = k.shape[1]
    out = np.zeros((H, D), np.float32)
    for h in range(H):
        m, l, o, left = np.float32(-np.inf), np.float32(0), np.zeros(D, np.float32), L
        for phys in mapping:
            valid = min(bs, left)
            left -= valid
            s = (k[phys, :valid, h] @ q[h]) * scale
            mn = np.float32(max(m, s.max()))
            c = np.exp(np.float32(m - mn)) if np.isfinite(m) else np.float32(0)
            p = np.exp(s - mn).astype(np.float32)
            l, o, m = l * c + p.sum(dtype=np.float32), o * c + p @ v[phys, :valid, h], mn
        out[h] = o / l
    return out


def test_fixed_block_table_of_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "os_block_table_example.json")))
    table = g["logical_to_physical"]
    bs, D = 2, 3
    NB = max(table) + 1
    k = np.full((NB, bs, 1, D), np.nan)
    v = np.full((NB, bs, 1, D), np.nan)
    for blk in table:                       # each block's rows carry its id
        k[blk] = 0.0
        v[blk, :, 0, :] = blk
    L = len(table) * bs
    K, V = A.gather_context(k, v, table, L)
    assert [int(V[t, 0, 0]) for t in range(L)] == [p for p in table for _ in range(bs)]
    out = A.paged_attention_walk(np.zeros((1, D)), k, v, table, L, 1.0)
    # all keys equal -> uniform weights -> mean of the ids
    assert abs(out[0, 0] - np.mean(table)) < 1e-13


def test_permutation_of_physical_ids_is_invisible():
    rng = np.random.default_rng(5)
    q, k, v, tables, L = scattered_case(rng, 3, 4, 2, 8, 4, [13, 1, 30])
    NB = k.shape[0]
    perm = rng.permutation(NB)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    t2 = np.where(tables < NB, perm[np.minimum(tables, NB - 1)], NB)
    a = A.paged_decode(q, k, v, tables, L, 0.5)
    b = A.paged_decode(q, k2, v2, t2, L, 0.5)
    np.testing.assert_array_equal(a, b)


def test_shared_blocks_equal_private_copies():
    rng = np.random.default_rng(6)
    bs, H, D = 4, 2, 8
    k, v = rand_pool(rng, 12, bs, H, D)
    shared = [3, 7]
    tables_shared = np.array([[3, 7, 1], [3, 7, 2]])
    k2, v2 = oracle.copy_blocks(k, v, [(3, 9), (7, 10)])
    tables_private = np.array([[3, 7, 1], [9, 10, 2]])
    q = rng.standard_normal((2, H, D))
    L = np.array([10, 11])
    a = A.paged_decode(q, k, v, tables_shared, L, 0.3)
    b = A.paged_decode(q, k2, v2, tables_private, L, 0.3)
    np.testing.assert_array_equal(a, b)
    assert shared == [3, 7]


# ---------------------------------------------------------------- split-K

@pytest.mark.parametrize("part", [4, 16, 100, 512, 4096])
def test_split_merge_equals_single_pass(part):
    rng = np.random.default_rng(part)
    q, k, v, tables, L = scattered_case(rng, 4, 4, 1, 16, 16, [1, 511, 512, 1500])
    np.testing.assert_allclose(A.paged_decode_split(q, k, v, tables, L, 0.2, part),
                               A.paged_decode(q, k, v, tables, L, 0.2), rtol=0, atol=1e-12)


def test_single_partition_state_normalises_to_dense():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((2, 4))
    K = rng.standard_normal((5, 1, 4))
    V = rng.standard_normal((5, 1, 4))
    m, l, o = A.decode_partials(q, K, V, 1.0, 64)
    assert m.shape == (1, 2)
    np.testing.assert_allclose(o[0] / l[0][:, None], A.dense_attention(q, K, V, 1.0), atol=1e-14)


# ---------------------------------------------------------------- chunked prefill

def test_prefill_rows_are_decode_at_their_position():
    rng = np.random.default_rng(12)
    bs, Hq, Hkv, D, Tq = 4, 4, 2, 8, 6
    lens = [9, 14]
    q1, k, v, tables, L = scattered_case(rng, 2, Hq, Hkv, D, bs, lens)
    q = rng.standard_normal((2, Tq, Hq, D))
    out = A.paged_prefill(q, k, v, tables, L, 0.4)
    for b in range(2):
        for i in range(Tq):
            pos = L[b] - Tq + i
            ref = A.paged_attention_walk(q[b, i], k, v, tables[b], pos + 1, 0.4)
            np.testing.assert_allclose(out[b, i], ref, atol=1e-12)


def test_prefill_brute_force_and_padding_rows():
    rng = np.random.default_rng(13)
    bs, H, D, Tq = 2, 2, 3, 4
    q1, k, v, tables, L = scattered_case(rng, 1, H, H, D, bs, [3])
    q = rng.standard_normal((1, Tq, H, D))
    out = A.paged_prefill(q, k, v, tables, L, 1.0)
    assert not out[0, 0].any()              # position -1: padding row
    K, V = A.gather_context(k, v, tables[0], 3)
    for i in range(1, Tq):
        pos = 3 - Tq + i
        np.testing.assert_allclose(
            out[0, i], A.brute_force_attention(q[0, i], K[:pos + 1], V[:pos + 1], 1.0), atol=1e-13)


# ---------------------------------------------------------------- sensitivity

def _pins_pass(walk=None, dense=None, merge=None):
    """Run a subset of the pins above against (possibly mutated) functions."""
    walk = walk or A.paged_attention_walk
    dense = dense or A.dense_attention
    merge = merge or A.merge_partials
    ok = True
    # brute force
    rng = np.random.default_rng(21)
    q = rng.standard_normal((4, 3))
    K = rng.standard_normal((9, 2, 3))
    V = rng.standard_normal((9, 2, 3))
    ok &= np.allclose(dense(q, K, V, 0.7), A.brute_force_attention(q, K, V, 0.7), atol=1e-12)
    # walk vs brute force through the pool (NaN tails)
    rng = np.random.default_rng(22)
    qb, k, v, tables, L = scattered_case(rng, 2, 4, 2, 8, 4, [10, 7])
    for b in range(2):
        Kc, Vc = A.gather_context(k, v, tables[b], L[b])
        w = walk(qb[b], k, v, tables[b], L[b], 0.5)
        ok &= bool(np.isfinite(w).all()) and np.allclose(
            w, A.brute_force_attention(qb[b], Kc, Vc, 0.5), atol=1e-12)
    # split/merge vs brute force
    Kc, Vc = A.gather_context(k, v, tables[0], L[0])
    m, l, o = A.decode_partials(qb[0], Kc, Vc, 0.5, 4)
    ok &= np.allclose(merge(m, l, o), A.brute_force_attention(qb[0], Kc, Vc, 0.5), atol=1e-12)
    return bool(ok)


def test_planted_mistakes_are_caught():
    assert _pins_pass()

    def dense_no_scale(q, K, V, scale):
        return A.dense_attention(q, K, V, 1.0)

    def dense_wrong_group(q, K, V, scale):          # h % Hkv instead of h // G
        Hq, Hkv = q.shape[0], K.shape[1]
        out = np.zeros_like(q, dtype=np.float64)
        for h in range(Hq):
            out[h] = A.dense_attention(q[h:h + 1], K[:, h % Hkv:h % Hkv + 1], V[:, h % Hkv:h % Hkv + 1], scale)[0]
        return out

    def dense_transposed(q, K, V, scale):           # weights applied to K
        return A.dense_attention(q, K, K, scale)

    def walk_no_rescale(q, k, v, row, L, scale):    # forgets exp(m - m')
        Hq, D = q.shape
        bs, Hkv = k.shape[1], k.shape[2]
        G = Hq // Hkv
        out = np.zeros((Hq, D))
        for h in range(Hq):
            m, l, o, left = -np.inf, 0.0, np.zeros(D), L
            for j in range(-(-L // bs)):
                valid = min(bs, left)
                left -= valid
                s = (k[row[j], :valid, h // G] @ q[h]) * scale
                mn = max(m, s.max())
                p = np.exp(s - mn)
                l, o, m = l + p.sum(), o + p @ v[row[j], :valid, h // G], mn
            out[h] = o / l
        return out

    def walk_reads_whole_block(q, k, v, row, L, scale):  # ignores `valid`
        bs = k.shape[1]
        return A.paged_attention_walk(q, k, v, row, -(-L // bs) * bs, scale)

    def merge_unweighted(m, l, o):
        return o.sum(axis=0) / l.sum(axis=0)[:, None]

    assert not _pins_pass(dense=dense_no_scale)
    assert not _pins_pass(dense=dense_wrong_group)
    assert not _pins_pass(dense=dense_transposed)
    assert not _pins_pass(walk=walk_no_rescale)
    assert not _pins_pass(walk=walk_reads_whole_block)
    assert not _pins_pass(merge=merge_unweighted)


def test_varlen_round_reduces_to_decode_and_fixed_chunks():
    """A mixed round: decode rows equal single-query decode; a uniform round
    equals the fixed-count tile; empty sequences contribute no rows."""
    rng = np.random.default_rng(17)
    NB, bs, Hkv, G, D = 24, 4, 2, 2, 8
    k = rng.standard_normal((NB, bs, Hkv, D))
    v = rng.standard_normal((NB, bs, Hkv, D))
    tables = rng.permutation(NB)[:18].reshape(3, 6)
    lens = np.array([13, 7, 20])
    n = np.array([1, 0, 5])                        # decode, empty, a 5-token chunk
    qs = np.concatenate([[0], np.cumsum(n)])
    q = rng.standard_normal((int(qs[-1]), Hkv * G, D))
    out = oracle.paged_prefill_varlen(q, qs, k, v, tables, lens, 0.3)
    dec = oracle.paged_decode(q[0:1], k, v, tables[0:1], lens[0:1], 0.3)
    assert np.abs(out[0] - dec[0]).max() <= 1e-12
    chunk = oracle.paged_prefill(q[1:6][None], k, v, tables[2:3], lens[2:3], 0.3)[0]
    assert np.abs(out[1:6] - chunk).max() <= 1e-12
    # a row's output depends only on its own query and its causal prefix
    q2 = q.copy()
    q2[3] += 1.0
    out2 = oracle.paged_prefill_varlen(q2, qs, k, v, tables, lens, 0.3)
    assert np.array_equal(np.delete(out2, 3, axis=0), np.delete(out, 3, axis=0))



# ---------------------------------------------------------------- shared prefixes

def shared_case(rng, P, S, pre_blocks, tails, bs=4, Hq=4, Hkv=2, D=8):
    """P prompts x S samples: every sample's table starts with its prompt's
    pre_blocks physical blocks, followed by private blocks for its tail;
    unused slots and blocks are NaN."""
    B = P * S
    lens = [pre_blocks * bs + int(t) for t in tails]
    nblk = [-(-L // bs) for L in lens]
    NB = P * pre_blocks + sum(n - pre_blocks for n in nblk) + 3
    k, v = rand_pool(rng, NB, bs, Hkv, D)
    perm = rng.permutation(NB)
    tables = np.full((B, max(nblk)), NB, dtype=np.int64)
    off = 0
    for p in range(P):
        pb = perm[off:off + pre_blocks]
        off += pre_blocks
        for s in range(S):
            b = p * S + s
            tables[b, :pre_blocks] = pb
            n = nblk[b] - pre_blocks
            tables[b, pre_blocks:pre_blocks + n] = perm[off:off + n]
            off += n
            if n:
                valid = lens[b] - (nblk[b] - 1) * bs
                k[tables[b, nblk[b] - 1], valid:] = np.nan
                v[tables[b, nblk[b] - 1], valid:] = np.nan
    k[perm[off:]] = np.nan
    v[perm[off:]] = np.nan
    q = rng.standard_normal((B, Hq, D))
    gs = np.arange(0, B + 1, S)
    return q, k, v, tables, np.array(lens), gs, np.full(P, pre_blocks)


def _shared_pins_pass(decode_shared=None):
    """The shared-prefix pins, run against a given implementation."""
    f = decode_shared or A.paged_decode_shared_prefix
    rng = np.random.default_rng(41)
    ok = True
    # real sharing: equals the plain decode (and brute force for one member)
    q, k, v, t, L, gs, sb = shared_case(rng, 3, 4, 3, [0, 5, 1, 9, 4, 4, 0, 2, 7, 3, 6, 11])
    got = f(q, k, v, t, L, 0.4, gs, sb)
    ok &= bool(np.isfinite(got).all()) and np.abs(got - A.paged_decode(q, k, v, t, L, 0.4)).max() <= 1e-12
    Kc, Vc = A.gather_context(k, v, t[5], L[5])
    ok &= np.abs(got[5] - A.brute_force_attention(q[5], Kc, Vc, 0.4)).max() <= 1e-12
    # a claimed prefix longer than a member's full blocks is clamped
    L2 = L.copy()
    L2[1] = 2 * 4 + 3                   # member 1 holds only 2 full blocks of the 3 shared
    got = f(q, k, v, t, L2, 0.4, gs, np.array([3, 3, 3]))
    ok &= np.abs(got - A.paged_decode(q, k, v, t, L2, 0.4)).max() <= 1e-12
    # the shared blocks are read through the first member's row
    t3 = t.copy()
    t3[6, 0] = t[0, 0]                  # member 2 of prompt 1 now points elsewhere
    want = A.paged_decode(q, k, v, t, L, 0.4)
    got = f(q, k, v, t3, L, 0.4, gs, sb)
    ok &= np.abs(got - want).max() <= 1e-12
    return bool(ok)


def test_shared_prefix_decode_pins():
    assert _shared_pins_pass()


def test_shared_prefix_decode_equals_plain_decode_on_many_shapes():
    rng = np.random.default_rng(42)
    for P, S, pre, bs, Hq, Hkv in ((1, 8, 5, 4, 8, 2), (4, 2, 1, 8, 4, 4), (2, 3, 6, 4, 6, 3)):
        tails = rng.integers(0, 3 * bs, size=P * S)
        q, k, v, t, L, gs, sb = shared_case(rng, P, S, pre, tails, bs=bs, Hq=Hq, Hkv=Hkv)
        got = A.paged_decode_shared_prefix(q, k, v, t, L, 0.3, gs, sb)
        assert np.abs(got - A.paged_decode(q, k, v, t, L, 0.3)).max() <= 1e-12


def test_shared_prefix_groups_of_one_and_empty_contexts():
    rng = np.random.default_rng(43)
    q, k, v, t, L = scattered_case(rng, 4, 4, 2, 8, 4, [0, 9, 1, 16])
    # every sequence its own group with nothing shared, including L = 0
    gs, sb = np.arange(5), np.zeros(4, dtype=np.int64)
    got = A.paged_decode_shared_prefix(q, k, v, t, L, 0.5, gs, sb)
    np.testing.assert_allclose(got, A.paged_decode(q, k, v, t, L, 0.5), rtol=0, atol=1e-12)
    assert np.array_equal(got[0], np.zeros_like(got[0]))


def test_invalid_group_descriptor_is_ignored():
    rng = np.random.default_rng(44)
    q, k, v, t, L, gs, sb = shared_case(rng, 2, 2, 2, [1, 2, 3, 4])
    want = A.paged_decode(q, k, v, t, L, 0.5)
    for bad in ([0, 2, 3], [1, 2, 4], [0, 3, 2, 4]):
        got = A.paged_decode_shared_prefix(q, k, v, t, L, 0.5, np.array(bad), np.full(len(bad) - 1, 2))
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_shared_prefix_groups_are_found_from_the_tables():
    rng = np.random.default_rng(45)
    q, k, v, t, L, gs, sb = shared_case(rng, 3, 4, 3, [2, 0, 5, 1, 4, 4, 3, 2, 7, 3, 6, 1])
    g2, s2 = A.shared_prefix_groups(t, L, 4)
    assert np.array_equal(g2, gs) and np.array_equal(s2, sb)
    # brute force: the longest run of leading entries common to every pair of members
    for g in range(len(g2) - 1):
        rows = range(g2[g], g2[g + 1])
        n = min(min(int(L[b]) // 4 for b in rows),
                min(next((j for j in range(t.shape[1]) if t[a, j] != t[b, j]), t.shape[1])
                    for a in rows for b in rows))
        assert s2[g] == n
    # a sample that has copied its first block on write leaves the group
    t2 = t.copy()
    t2[4, 0] = k.shape[0] - 1
    g3, s3 = A.shared_prefix_groups(t2, L, 4)
    assert list(g3) == [0, 4, 5, 8, 12] and list(s3) == [3, 0, 3, 3]
    # a divergent second block shortens the group's shared run
    t2 = t.copy()
    t2[9, 1] = k.shape[0] - 2
    g4, s4 = A.shared_prefix_groups(t2, L, 4)
    assert list(g4) == list(gs) and list(s4) == [3, 3, 1]


def test_planted_shared_prefix_mistakes_are_caught():
    def unweighted_merge(q, k, v, t, L, scale, gs, sb):
        out = np.zeros(q.shape)
        bs = k.shape[1]
        for g in range(len(gs) - 1):
            s0, s1 = int(gs[g]), int(gs[g + 1])
            S = min([int(sb[g])] + [int(L[b]) // bs for b in range(s0, s1)])
            Ks, Vs = A.gather_context(k, v, t[s0], S * bs)
            for b in range(s0, s1):
                Kf, Vf = A.gather_context(k, v, t[b], int(L[b]))
                m1, l1, o1 = A.decode_partials(q[b], Ks, Vs, scale, S * bs)
                if int(L[b]) > S * bs:
                    m2, l2, o2 = A.decode_partials(q[b], Kf[S * bs:], Vf[S * bs:], scale, int(L[b]) - S * bs)
                    out[b] = (o1[0] + o2[0]) / (l1[0] + l2[0])[:, None]
                else:
                    out[b] = o1[0] / l1[0][:, None]
        return out

    def tail_one_block_late(q, k, v, t, L, scale, gs, sb):
        L = np.asarray(L)
        out = A.paged_decode_shared_prefix(q, k, v, t, L, scale, gs, sb)
        bs = k.shape[1]
        for g in range(len(gs) - 1):
            s0, s1 = int(gs[g]), int(gs[g + 1])
            S = min([int(sb[g])] + [int(L[b]) // bs for b in range(s0, s1)])
            Ks, Vs = A.gather_context(k, v, t[s0], S * bs)
            for b in range(s0, s1):
                Kf, Vf = A.gather_context(k, v, t[b], int(L[b]))
                keep = np.concatenate([Ks, Kf[(S + 1) * bs:]]), np.concatenate([Vs, Vf[(S + 1) * bs:]])
                out[b] = A.dense_attention(q[b], keep[0], keep[1], scale)
        return out

    def leaders_query(q, k, v, t, L, scale, gs, sb):
        q2 = q.copy()
        for g in range(len(gs) - 1):
            q2[int(gs[g]):int(gs[g + 1])] = q[int(gs[g])]
        return A.paged_decode_shared_prefix(q2, k, v, t, L, scale, gs, sb)

    def members_own_rows(q, k, v, t, L, scale, gs, sb):   # never reads through the first member's row
        return A.paged_decode(q, k, v, t, L, scale)

    assert _shared_pins_pass()
    for bad in (unweighted_merge, tail_one_block_late, leaders_query, members_own_rows):
        assert not _shared_pins_pass(bad), bad.__name__
