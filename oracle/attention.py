"""Attention over a paged KV cache, float64, written for a reader to check by eye.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Layout, as the page [KVS] "19.2 KV Cache 系统化管理" fixes it in §19.2.3 (the
block pool stores keys and values as ``[num_blocks, block_size, num_heads,
head_dim]``):

    k_cache, v_cache : [NB, bs, Hkv, D]
    q                : [Hq, D] for one sequence, [B, Hq, D] for a batch
    block table row  : physical block id of logical block j, j = 0, 1, ...
    context length L : tokens held by the sequence; the token at logical
                       position t sits in physical block table[t // bs] at
                       slot t % bs ([OS] §三: the attention kernel looks the
                       logical block up in the block table, then forms the
                       physical block address and the offset inside it).

Readings where the pages are silent (each listed again in the design notes):

* scale is an argument; the pages use 1/sqrt(head_dim) ([KVS] §19.2.3).
* GQA (not on the pages): query head h reads KV head h // (Hq / Hkv).
* an empty context (L == 0) gives a zero output (the pages would give 0/0).
* split-K partitions are ``part`` tokens long, aligned at token 0; their merge
  follows from the associativity of the online-softmax update of §19.2.3.
* chunked prefill ([OS] §8.1): the Tq query tokens are the LAST Tq tokens of
  the context, query i sits at position L - Tq + i and attends causally to
  positions 0..L - Tq + i; a query whose position is negative is padding and
  gives zeros.
"""

import math

import numpy as np


def _as_f64(a):
    a = np.asarray(a)
    if a.dtype != np.float64:
        a = a.astype(np.float64)
    return a


def dense_attention(q, K, V, scale):
    """Softmax attention of each query head over a contiguous context.

    Definition (the "standard attention" that [KVS] §19.2.3 checks the paged
    version against): for query head h with KV head g = h // G,

        s_t   = scale * <q[h], K[t, g]>
        w_t   = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u)
        out_h = sum_t w_t V[t, g]

    q: [Hq, D]; K, V: [T, Hkv, D].  Two passes (max, then normalised weights).
    Returns [Hq, D] float64; zeros when T == 0.
    """
    q = _as_f64(q)
    K = _as_f64(K)
    V = _as_f64(V)
    Hq, D = q.shape
    T, Hkv, Dk = K.shape
    assert Dk == D and V.shape == K.shape and Hq % Hkv == 0
    G = Hq // Hkv
    out = np.zeros((Hq, D), dtype=np.float64)
    if T == 0:
        return out
    for h in range(Hq):
        g = h // G
        s = (K[:, g, :] @ q[h]) * scale            # [T]
        w = np.exp(s - s.max())
        w = w / w.sum()
        out[h] = w @ V[:, g, :]
    return out


def brute_force_attention(q, K, V, scale):
    """The same definition as ``dense_attention`` with scalar Python loops and
    ``math.fsum`` (exactly rounded sums).  For tiny inputs only; it is the pin
    that ``dense_attention`` is checked against."""
    q = _as_f64(q)
    K = _as_f64(K)
    V = _as_f64(V)
    Hq, D = q.shape
    T, Hkv, _ = K.shape
    G = Hq // Hkv
    out = np.zeros((Hq, D), dtype=np.float64)
    if T == 0:
        return out
    for h in range(Hq):
        g = h // G
        scores = [scale * math.fsum(float(q[h, d]) * float(K[t, g, d]) for d in range(D))
                  for t in range(T)]
        mx = max(scores)
        e = [math.exp(s - mx) for s in scores]
        z = math.fsum(e)
        for d in range(D):
            out[h, d] = math.fsum(e[t] * float(V[t, g, d]) for t in range(T)) / z
    return out


def gather_context(k_cache, v_cache, table_row, L):
    """Copy a sequence's L tokens out of the pool into contiguous [L, Hkv, D]
    arrays, token t from block table_row[t // bs], slot t % bs ([OS] §三)."""
    bs = k_cache.shape[1]
    idx_blk = np.array([int(table_row[t // bs]) for t in range(L)], dtype=np.int64)
    idx_off = np.arange(L, dtype=np.int64) % bs
    return _as_f64(k_cache[idx_blk, idx_off]), _as_f64(v_cache[idx_blk, idx_off])


def paged_attention_walk(q, k_cache, v_cache, table_row, L, scale):
    """Block-by-block paged attention with an online softmax, the algorithm of
    [KVS] §19.2.3 (Fig 19-5: the operator walks the block table and
    accumulates block by block), generalised to GQA.

    State per query head: running maximum m, running sum of exponentials l,
    unnormalised output o; start m = -inf, l = 0, o = 0.  For each mapped block
    only ``valid = min(bs, tokens left)`` slots are read.  With the block's
    scores s and m' = max(m, max s):

        l <- l * exp(m - m') + sum exp(s - m')
        o <- o * exp(m - m') + sum exp(s - m') v
        m <- m'

    and the result is o / l once every block has been seen.
    """
    q = _as_f64(q)
    Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    G = Hq // Hkv
    out = np.zeros((Hq, D), dtype=np.float64)
    if L == 0:
        return out
    nblk = -(-L // bs)
    for h in range(Hq):
        g = h // G
        m = -np.inf
        l = 0.0
        o = np.zeros(D, dtype=np.float64)
        left = L
        for j in range(nblk):
            phys = int(table_row[j])
            valid = min(bs, left)
            left -= valid
            keys = _as_f64(k_cache[phys, :valid, g, :])   # [valid, D]
            vals = _as_f64(v_cache[phys, :valid, g, :])
            s = (keys @ q[h]) * scale
            m_new = max(m, float(s.max()))
            carry = math.exp(m - m_new) if m != -np.inf else 0.0
            p = np.exp(s - m_new)
            l = l * carry + p.sum()
            o = o * carry + p @ vals
            m = m_new
        out[h] = o / l
    return out


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, method="dense"):
    """Decode attention for a batch: out[b] = attention of q[b] over sequence
    b's paged context.  ``method='dense'`` gathers then applies the definition;
    ``method='walk'`` runs the block-by-block online softmax.  [B, Hq, D] f64."""
    q = _as_f64(q)
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(context_lens[b])
        if method == "walk":
            out[b] = paged_attention_walk(q[b], k_cache, v_cache, block_tables[b], L, scale)
        else:
            K, V = gather_context(k_cache, v_cache, block_tables[b], L)
            out[b] = dense_attention(q[b], K, V, scale)
    return out


def decode_partials(q, K, V, scale, part):
    """Split one sequence's context into partitions of ``part`` tokens starting
    at token 0 and return, per partition i and query head h, the online-softmax
    state over that partition alone:

        m_i = max_t s_t,  l_i = sum_t exp(s_t - m_i),  o_i = sum_t exp(s_t - m_i) v_t

    (unnormalised).  Returns arrays m [P, Hq], l [P, Hq], o [P, Hq, D]."""
    q = _as_f64(q)
    K = _as_f64(K)
    V = _as_f64(V)
    Hq, D = q.shape
    T, Hkv, _ = K.shape
    G = Hq // Hkv
    P = -(-T // part)
    m = np.full((P, Hq), -np.inf)
    l = np.zeros((P, Hq))
    o = np.zeros((P, Hq, D))
    for i in range(P):
        lo, hi = i * part, min(T, (i + 1) * part)
        for h in range(Hq):
            g = h // G
            s = (K[lo:hi, g, :] @ q[h]) * scale
            m[i, h] = s.max()
            e = np.exp(s - m[i, h])
            l[i, h] = e.sum()
            o[i, h] = e @ V[lo:hi, g, :]
    return m, l, o


def merge_partials(m, l, o):
    """Log-sum-exp merge of partition states: with M = max_i m_i,

        out = sum_i exp(m_i - M) o_i / sum_i exp(m_i - M) l_i

    which is the online-softmax update of [KVS] §19.2.3 applied to whole
    partitions instead of single blocks.  m, l: [P, Hq]; o: [P, Hq, D]."""
    M = m.max(axis=0)                      # [Hq]
    w = np.exp(m - M[None, :])             # [P, Hq]
    num = (w[:, :, None] * o).sum(axis=0)  # [Hq, D]
    den = (w * l).sum(axis=0)              # [Hq]
    return num / den[:, None]


def paged_decode_split(q, k_cache, v_cache, block_tables, context_lens, scale, part):
    """Split-K decode: per sequence, partition states then their merge."""
    q = _as_f64(q)
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(context_lens[b])
        if L == 0:
            continue
        K, V = gather_context(k_cache, v_cache, block_tables[b], L)
        m, l, o = decode_partials(q[b], K, V, scale, part)
        out[b] = merge_partials(m, l, o)
    return out


def paged_prefill(q, k_cache, v_cache, block_tables, context_lens, scale):
    """Causal chunked-prefill tile over the paged cache ([OS] §8.1).

    q: [B, Tq, Hq, D].  The tile is the last Tq tokens of each sequence's
    context (their K/V already appended), so query i of sequence b sits at
    position pos = L_b - Tq + i and attends to positions 0..pos.  Returns
    [B, Tq, Hq, D] f64; rows with pos < 0 are zero."""
    q = _as_f64(q)
    B, Tq, Hq, D = q.shape
    out = np.zeros((B, Tq, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(context_lens[b])
        K, V = gather_context(k_cache, v_cache, block_tables[b], L)
        for i in range(Tq):
            pos = L - Tq + i
            if pos < 0:
                continue
            out[b, i] = dense_attention(q[b, i], K[:pos + 1], V[:pos + 1], scale)
    return out


def paged_prefill_varlen(q, query_start, k_cache, v_cache, block_tables, context_lens, scale):
    """Attention for a mixed round: sequence b contributes the query rows
    q[query_start[b]:query_start[b+1]] ([rows, Hq, D]), its last
    n_b = query_start[b+1] - query_start[b] tokens, their K/V already in the
    pool.  [OS] §8.1–8.2: one round holds decode tokens (n_b = 1) and prefill
    chunk tokens under one token budget; a chunk continues from the tokens
    already computed.  Each row attends causally to its paged context, as in
    ``paged_prefill``.  Returns [rows, Hq, D] f64; rows at negative
    positions are zero."""
    q = _as_f64(q)
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(len(context_lens)):
        s0, s1 = int(query_start[b]), int(query_start[b + 1])
        if s1 <= s0:
            continue
        out[s0:s1] = paged_prefill(q[s0:s1][None], k_cache, v_cache, block_tables[b:b + 1],
                                   context_lens[b:b + 1], scale)[0]
    return out



# ---------------------------------------------------------------- shared prefixes

def shared_prefix_groups(block_tables, context_lens, block_size):
    """Find the sequences that share a prompt's physical blocks.

    [KVS] §19.2.2 (copy-on-write and prefix sharing) and §19.2.5: samples
    drawn from one prompt point their block tables at the same physical
    blocks for the prompt (reference count = number of samples); [OS] §四
    names beam search and parallel sampling as the cases.  A group is a
    maximal run of adjacent sequences whose first block is one and the same
    full physical block; its shared length is the number of leading table
    entries that all members hold in common, counting only blocks that every
    member fills completely (at most floor(L_b / bs) for each member b).  A
    sequence alone is a group of one with no shared blocks.

    Returns (group_start [n+1], shared_blocks [n]) as int64 arrays."""
    lens = [int(x) for x in context_lens]
    B = len(lens)
    starts = [0]
    for b in range(1, B):
        same = (lens[b] >= block_size and lens[b - 1] >= block_size
                and int(block_tables[b][0]) == int(block_tables[b - 1][0]))
        if not same:
            starts.append(b)
    starts.append(B)
    shared = []
    for g in range(len(starts) - 1):
        members = range(starts[g], starts[g + 1])
        if len(members) < 2:
            shared.append(0)
            continue
        cap = min(lens[b] // block_size for b in members)
        lead = starts[g]
        n = 0
        while n < cap and all(int(block_tables[b][n]) == int(block_tables[lead][n]) for b in members):
            n += 1
        shared.append(n)
    return np.array(starts, dtype=np.int64), np.array(shared, dtype=np.int64)


def _valid_groups(group_start, B):
    gs = [int(x) for x in group_start]
    return len(gs) >= 1 and gs[0] == 0 and gs[-1] == B and all(a <= b for a, b in zip(gs, gs[1:]))


def paged_decode_shared_prefix(q, k_cache, v_cache, block_tables, context_lens, scale,
                               group_start, shared_blocks):
    """Decode of a batch whose sequences share prompt blocks, with each shared
    block's keys and values read once for all the sequences of its group.

    Sequences group_start[g] .. group_start[g+1]-1 form group g; they declare
    that the first shared_blocks[g] entries of their block-table rows name the
    same physical blocks ([KVS] §19.2.5, Fig 19-8: every sample's table points
    at the prompt's blocks).  The shared part actually used is

        S_g = min(shared_blocks[g], min over members b of floor(L_b / bs))

    whole blocks (each member holds every one of them completely), taken from
    the FIRST member's table row.  For each member b and query head h:

      * the state (m, l, o) of the online softmax of [KVS] §19.2.3 over the
        S_g * bs shared tokens (one partition, as in ``decode_partials``);
      * the state over b's own tokens S_g * bs .. L_b - 1, read through b's
        own table row;
      * the two merged by ``merge_partials`` (the log-sum-exp combination);
        a part with no tokens is left out, and a sequence with none at all
        gives zeros.

    When the members' rows really share those blocks this is exactly
    ``paged_decode`` (the merge is the associativity of the online softmax).
    A descriptor that does not cover the batch as non-decreasing runs from 0
    to B is ignored (plain decode)."""
    q = _as_f64(q)
    B, Hq, D = q.shape
    bs = k_cache.shape[1]
    if not _valid_groups(group_start, B):
        return paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for g in range(len(group_start) - 1):
        s0, s1 = int(group_start[g]), int(group_start[g + 1])
        if s1 <= s0:
            continue
        S = min([int(shared_blocks[g])] + [int(context_lens[b]) // bs for b in range(s0, s1)])
        S = max(S, 0)
        Ts = S * bs
        Ks, Vs = gather_context(k_cache, v_cache, block_tables[s0], Ts)
        for b in range(s0, s1):
            L = int(context_lens[b])
            parts = []
            if Ts > 0:
                parts.append(decode_partials(q[b], Ks, Vs, scale, Ts))
            if L > Ts:
                Kf, Vf = gather_context(k_cache, v_cache, block_tables[b], L)
                Kt, Vt = Kf[Ts:], Vf[Ts:]
                parts.append(decode_partials(q[b], Kt, Vt, scale, L - Ts))
            if not parts:
                continue
            m = np.concatenate([p[0] for p in parts], axis=0)
            l = np.concatenate([p[1] for p in parts], axis=0)
            o = np.concatenate([p[2] for p in parts], axis=0)
            out[b] = merge_partials(m, l, o)
    return out
