"""One decode step (append + paged decode) captured once as a CUDA graph and
replayed with new inputs written into the captured buffers: every replay
must give the bits the eager calls give, and match the oracle.

The graph holds device pointers and the tensor maps of the pools by value,
so new tokens, new queries, grown lengths and edited block tables take
effect by overwriting the captured tensors in place.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_307_gb300 import workloads as W
from _helpers import f64, oracle_decode, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_307_gb300 import build
    build.build()
    from paged_kv_cache_307_gb300 import _lib
    assert torch.cuda.is_available()
    _lib.last_error()
    return _lib


def _cuda_case(name, **kw):
    c = W.decode_case(name, **kw)
    for f in ("q", "k_cache", "v_cache", "block_tables", "context_lens", "key", "value", "slot_mapping"):
        setattr(c, f, getattr(c, f).cuda())
    return c


def _fresh_inputs(c, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return {"q": torch.randn(c.q.shape, generator=g, device="cuda").to(c.q.dtype),
            "key": torch.randn(c.key.shape, generator=g, device="cuda").to(c.key.dtype),
            "value": torch.randn(c.value.shape, generator=g, device="cuda").to(c.value.dtype)}


@pytest.mark.parametrize("name,partition", [("c2", 0), ("c2", 64), ("c4", 0), ("c5", 0), ("c1", 0)])
def test_graph_replay_matches_eager(pa, name, partition):
    c = _cuda_case(name, small=True)
    if c.spec.bs > 0 and partition % c.spec.bs:
        partition = 4 * c.spec.bs
    k0, v0 = c.k_cache.clone(), c.v_cache.clone()
    ws = pa.alloc_workspace(c.q, c.k_cache, c.block_tables, partition)
    inputs = [_fresh_inputs(c, s) for s in (1, 2, 3)]

    def step(kc, vc, q, key, value, out):
        pa.reshape_and_cache(key, value, c.slot_mapping, kc, vc)
        pa.decode(out, q, kc, vc, c.block_tables, c.context_lens, c.scale, partition_size=partition,
                  workspace=ws)

    # eager, one step per input set, on one pool
    eager = []
    kc, vc = k0.clone(), v0.clone()
    for x in inputs:
        o = torch.empty_like(c.q)
        step(kc, vc, x["q"], x["key"], x["value"], o)
        eager.append(o)
    torch.cuda.synchronize()
    assert pa.last_error() == 0

    # graph: static buffers, captured once (after an eager warm-up on the side stream)
    kg, vg = k0.clone(), v0.clone()
    sq, skey, sval = c.q.clone(), c.key.clone(), c.value.clone()
    sout = torch.empty_like(c.q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(kg, vg, sq, skey, sval, sout)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(kg, vg, sq, skey, sval, sout)
    kg.copy_(k0)
    vg.copy_(v0)
    for x, e in zip(inputs, eager):
        sq.copy_(x["q"])
        skey.copy_(x["key"])
        sval.copy_(x["value"])
        graph.replay()
        torch.cuda.synchronize()
        assert pa.last_error() == 0
        assert torch.equal(sout.view(torch.int16 if sout.element_size() == 2 else torch.int32),
                           e.view(torch.int16 if e.element_size() == 2 else torch.int32))
    assert torch.equal(kg.view(torch.uint8), kc.view(torch.uint8))


def test_graph_replay_follows_growing_contexts(pa):
    """Three decode steps of the same requests: each step the lengths grow by
    one and the new token's slot moves; the captured graph reads the updated
    lengths, slots and tables and matches the oracle each step."""
    c = _cuda_case("c2", small=True)
    bs = c.spec.bs
    B = c.q.shape[0]
    free = sorted(set(range(c.num_blocks)) - set(c.block_tables.cpu().numpy().ravel().tolist()))
    ws = pa.alloc_workspace(c.q, c.k_cache, c.block_tables, 0)
    sq, skey, sval = c.q.clone(), c.key.clone(), c.value.clone()
    out = torch.empty_like(c.q)

    def step():
        pa.reshape_and_cache(skey, sval, c.slot_mapping, c.k_cache, c.v_cache)
        pa.decode(out, sq, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, workspace=ws)

    # the first step runs eagerly as the warm-up; it appends the case's own token
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for it in range(3):
        lens = c.context_lens.cpu().numpy() + 1
        tables = c.block_tables.cpu().numpy()
        slots = np.empty(B, np.int64)
        for b in range(B):
            L = int(lens[b])
            j = (L - 1) // bs
            if j >= tables.shape[1]:
                pytest.skip("case has no room to grow")
            if (L - 1) % bs == 0:                 # the new token opens a block
                tables[b, j] = free.pop()
            slots[b] = int(tables[b, j]) * bs + (L - 1) % bs
        x = _fresh_inputs(c, 10 + it)
        sq.copy_(x["q"])
        skey.copy_(x["key"])
        sval.copy_(x["value"])
        c.context_lens.copy_(torch.from_numpy(lens.astype(np.int32)))
        c.block_tables.copy_(torch.from_numpy(tables))
        c.slot_mapping.copy_(torch.from_numpy(slots))
        pool_k, pool_v = c.k_cache.clone(), c.v_cache.clone()     # before this step's append
        graph.replay()
        torch.cuda.synchronize()
        assert pa.last_error() == 0
        ref_case = W.decode_case("c2", small=True)
        ref_case.q, ref_case.key, ref_case.value = sq.cpu(), skey.cpu(), sval.cpu()
        ref_case.k_cache, ref_case.v_cache = pool_k.cpu(), pool_v.cpu()
        ref_case.block_tables, ref_case.context_lens = c.block_tables.cpu(), c.context_lens.cpu()
        ref_case.slot_mapping = c.slot_mapping.cpu()
        assert_close(f64(out), oracle_decode(ref_case), "bf16")
