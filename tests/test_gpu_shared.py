"""pa_decode_shared (shared prompt blocks read once per group) through the C
ABI against the float64 oracle, on the GPU.

The result must be that of plain decode ("19.2 KV Cache 系统化管理" §19.2.5:
samples of one prompt share its physical blocks), within the bf16 tolerance
(max 2e-2, mean 2e-3 against float64); where the caller's descriptor does not
match the tables, the result must follow the descriptor's documented reading
(``oracle.paged_decode_shared_prefix``) and the device flags it.
"""

import numpy as np
import pytest
import torch

import oracle
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


def _case(small=True, device="cuda", **kw):
    c = W.decode_case("c5", small=small, device=device, **kw)
    return c


def _run(pa, c, partition=0, gs=None, sb=None, append=True):
    if append:
        pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
    gs = c.extra["group_start"] if gs is None else gs
    sb = c.extra["shared_blocks"] if sb is None else sb
    out = torch.full_like(c.q, float("nan"))
    pa.decode_shared(out, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, gs, sb, c.scale,
                     partition_size=partition)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("partition", [0, 64, 512, -1])
def test_shared_matches_oracle_c5_small(pa, partition):
    c = _case()
    ref = oracle_decode(c)                        # before the pool is touched
    out = _run(pa, c, partition)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


# (Hq, Hkv, head_dim, block_size, samples, prefix tokens, max tail):
# 8 rows per KV head (MHA, 8 samples), 16 (G = 2), 32, row chunks (64
# rows), head_dim 64 with block_size 8, KV heads not a multiple of 4, odd
# sample counts, prompts that end inside a block, block sizes 8 and 32
SHAPES = [
    (32, 8, 128, 16, 8, 128, 40),
    (8, 8, 128, 16, 8, 96, 30),
    (16, 8, 128, 16, 8, 64, 20),
    (64, 8, 128, 16, 8, 64, 20),
    (32, 8, 64, 8, 4, 64, 20),
    (24, 6, 128, 32, 3, 96, 70),
    (12, 6, 128, 16, 5, 48, 33),
    (4, 4, 128, 16, 2, 32, 17),
    (32, 8, 128, 8, 8, 200, 60),
    (32, 8, 128, 32, 8, 160, 100),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_shared_shape_variants(pa, shape):
    Hq, Hkv, D, bs, S, prefix, tmax = shape
    c = _case(B=3 * S, Hq=Hq, Hkv=Hkv, D=D, bs=bs, len_dist=("shared", 3, S, prefix, tmax))
    ref = oracle_decode(c)
    out = _run(pa, c)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


def test_shared_full_size_c5_sampled(pa):
    c = _case(small=False)
    lens = c.context_lens.cpu().numpy()
    rng = np.random.default_rng(7)
    S = c.extra["samples"]
    seqs = sorted(set(list(range(S)) + list(range(len(lens) - S, len(lens))) +
                      [int(np.argmax(lens)), int(np.argmin(lens))] +
                      rng.choice(len(lens), 6, replace=False).tolist()))
    ref = oracle_decode(c, seqs)
    out = _run(pa, c)
    assert pa.last_error() == 0
    got = f64(out)
    assert np.isfinite(got).all()
    vmax = float(torch.nan_to_num(c.v_cache.float(), nan=0.0).abs().max())
    assert np.abs(got).max() <= vmax + 1e-6            # convex combinations of V rows
    assert_close(got[seqs], ref, "bf16")
    # against the plain decode of the same pool (any size)
    plain = torch.empty_like(c.q)
    pa.decode(plain, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    torch.cuda.synchronize()
    d = np.abs(got - f64(plain))
    assert d.max() <= 2e-2 and d.mean() <= 1e-3


# The automatic shared partition depends on the batch (1024-token partitions
# for 64 prompts, 512 for 32, 256 for 16 and 8): each choice against the
# oracle on sampled sequences and against plain decode on all of them.
@pytest.mark.parametrize("batch", [64, 128, 256])
def test_shared_automatic_partition_by_batch(pa, batch):
    c = _case(small=False, B=batch)
    lens = c.context_lens.cpu().numpy()
    S = c.extra["samples"]
    rng = np.random.default_rng(batch)
    seqs = sorted(set(list(range(S)) + [int(np.argmax(lens)), int(np.argmin(lens))] +
                      rng.choice(len(lens), 4, replace=False).tolist()))
    ref = oracle_decode(c, seqs)
    out = _run(pa, c)
    assert pa.last_error() == 0
    got = f64(out)
    assert_close(got[seqs], ref, "bf16")
    plain = torch.empty_like(c.q)
    pa.decode(plain, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
    torch.cuda.synchronize()
    d = np.abs(got - f64(plain))
    assert d.max() <= 2e-2 and d.mean() <= 1e-3


def test_invalid_descriptor_is_flagged_and_ignored(pa):
    c = _case()
    ref = oracle_decode(c)
    B = c.q.shape[0]
    for bad in ([0, 8, 7, B], [1, 8, B], [0, 8, B + 1]):
        gs = torch.tensor(bad, dtype=torch.int32, device="cuda")
        sb = torch.full((len(bad) - 1,), 64, dtype=torch.int32, device="cuda")
        cc = _case()
        out = _run(pa, cc, gs=gs, sb=sb)
        assert pa.last_error() == pa.DEV_BAD_GROUP
        assert_close(f64(out), ref, "bf16")


def test_member_outside_the_shared_blocks_is_flagged(pa):
    c = _case(nan_fill=False)
    pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
    tables = c.block_tables.clone()
    tables[3, 5] = tables[9, 5]                   # member 3 of prompt 0 names another prompt's block
    c.block_tables = tables
    k, v = f64(c.k_cache), f64(c.v_cache)
    want = oracle.paged_decode_shared_prefix(f64(c.q), k, v, tables.cpu().numpy(), c.context_lens.cpu().numpy(),
                                             c.scale, c.extra["group_start"].cpu().numpy(),
                                             c.extra["shared_blocks"].cpu().numpy())
    out = _run(pa, c, append=False)
    assert pa.last_error() == pa.DEV_BAD_GROUP
    assert_close(f64(out), want, "bf16")
    # and that reading is not the plain decode of the altered tables
    plain = oracle.paged_decode(f64(c.q), k, v, tables.cpu().numpy(), c.context_lens.cpu().numpy(), c.scale)
    assert np.abs(plain[3] - want[3]).max() > 1e-3


def test_claimed_prefix_is_clamped_to_full_blocks(pa):
    c = _case()
    pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
    lens = c.context_lens.clone()
    lens[1] = 1024 - 21                          # member 1 ends inside the shared blocks
    lens[10] = 1024 - 16                         # member 2 of prompt 1 holds one block fewer
    c.context_lens = lens
    sm = c.slot_mapping.clone()
    sm[1] = sm[10] = -1                          # their appended tokens now lie past their contexts
    c.slot_mapping = sm
    ref = oracle_decode(c)
    sb = torch.full_like(c.extra["shared_blocks"], 70)     # claims more than any member holds
    out = _run(pa, c, sb=sb, append=False)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


def test_singletons_and_empty_contexts(pa):
    c = _case(B=16)
    lens = c.context_lens.clone()
    lens[0] = 0
    lens[5] = 1
    c.context_lens = lens
    sm = c.slot_mapping.clone()
    sm[0] = sm[5] = -1                           # no append past the shortened contexts
    c.slot_mapping = sm
    ref = oracle_decode(c)
    B = c.q.shape[0]
    gs = torch.arange(B + 1, dtype=torch.int32, device="cuda")
    sb = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = _run(pa, c, gs=gs, sb=sb)
    assert pa.last_error() == 0
    assert torch.equal(out[0].float(), torch.zeros_like(out[0].float()))
    assert_close(f64(out), ref, "bf16")
    # empty groups between real ones
    c2 = _case(B=16)
    ref2 = oracle_decode(c2)
    gs = torch.tensor([0, 0, 8, 8, 16, 16], dtype=torch.int32, device="cuda")
    sb = torch.tensor([5, 64, 0, 64, 3], dtype=torch.int32, device="cuda")
    out = _run(pa, c2, gs=gs, sb=sb)
    assert pa.last_error() == 0
    assert_close(f64(out), ref2, "bf16")


def test_shared_permuted_pool_is_bit_identical(pa):
    c = _case()
    pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
    out1 = _run(pa, c, append=False)
    NB = c.num_blocks
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(3)).cuda()
    k2, v2 = torch.empty_like(c.k_cache), torch.empty_like(c.v_cache)
    k2[perm], v2[perm] = c.k_cache, c.v_cache
    t = c.block_tables.long()
    t2 = torch.where(t < NB, perm[t.clamp(max=NB - 1)], t).int().contiguous()
    c.k_cache, c.v_cache, c.block_tables = k2, v2, t2
    out2 = _run(pa, c, append=False)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_shared_graph_replay_is_bit_identical(pa):
    c = _case()
    pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
    ws = pa.alloc_shared_workspace(c.q, c.k_cache, c.block_tables, c.extra["shared_blocks"].shape[0])
    out = torch.empty_like(c.q)

    def step():
        pa.decode_shared(out, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.extra["group_start"],
                         c.extra["shared_blocks"], c.scale, workspace=ws)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pa.last_error() == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_shared_back_to_back_on_a_side_stream(pa):
    """Three calls in a row on a user stream sharing one workspace (the work
    counter is cleared before each, the merge waits for its decode kernel on
    the device): the first and third give the current stream's bits, the
    middle one (another query batch) its own."""
    c = _case()
    ref = _run(pa, c, partition=64)
    q2 = c.q.flip(0).contiguous()
    gs, sb = c.extra["group_start"], c.extra["shared_blocks"]
    ws = pa.alloc_shared_workspace(c.q, c.k_cache, c.block_tables, sb.shape[0], partition_size=64)
    outs = [torch.full_like(c.q, float("nan")) for _ in range(3)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for o, q in zip(outs, (c.q, q2, c.q)):
            pa.decode_shared(o, q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, gs, sb, c.scale,
                             partition_size=64, workspace=ws, stream=side)
    side.synchronize()
    assert pa.last_error() == 0
    assert torch.equal(outs[0].view(torch.int16), ref.view(torch.int16))
    assert torch.equal(outs[2].view(torch.int16), ref.view(torch.int16))
    mid = torch.full_like(c.q, float("nan"))
    pa.decode_shared(mid, q2, c.k_cache, c.v_cache, c.block_tables, c.context_lens, gs, sb, c.scale,
                     partition_size=64)
    torch.cuda.synchronize()
    assert torch.equal(outs[1].view(torch.int16), mid.view(torch.int16))


def test_unsupported_shapes_run_plain_decode(pa):
    # fp32 pools and groups of more than 8 query heads take pa_decode's path
    # unchanged
    for name, over in (("c1", {}), ("c4", {"Hq": 64, "Hkv": 4, "D": 64}), ("c4", {"Hq": 128, "Hkv": 2})):
        c = W.decode_case(name, small=True, device="cuda", **over)
        pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
        B = c.q.shape[0]
        gs = torch.tensor([0, B], dtype=torch.int32, device="cuda")
        sb = torch.zeros(1, dtype=torch.int32, device="cuda")
        a, b = torch.empty_like(c.q), torch.empty_like(c.q)
        pa.decode(a, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale)
        pa.decode_shared(b, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, gs, sb, c.scale)
        torch.cuda.synchronize()
        assert pa.last_error() == 0
        assert torch.equal(a.view(torch.int16) if a.element_size() == 2 else a.view(torch.int32),
                           b.view(torch.int16) if b.element_size() == 2 else b.view(torch.int32))
