"""CUDA path (through the C ABI) against the float64 oracle, on the GPU.

Small cases run the whole batch through the oracle; full-size cases run in
the launch configuration the benchmark times and compare sampled sequences
one by one, plus properties that hold at any size.  The append and the block
copy must be bit-exact; attention must meet max|err| <= 1e-5 (fp32) or
max <= 2e-2 and mean <= 2e-3 (bf16, fp32 accumulation).
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_307_gb300 import workloads as W
from _helpers import f64, bits, oracle_decode, gpu_decode, assert_close

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


# ------------------------------------------------------------------ append / copy

@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c4b32", "c5"])
def test_reshape_and_cache_bit_exact(pa, name):
    c = _cuda_case(name, small=True)
    exp_k, exp_v = oracle.reshape_and_cache(bits(c.key), bits(c.value), c.slot_mapping.cpu().numpy(),
                                            bits(c.k_cache), bits(c.v_cache))
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    pa.reshape_and_cache(c.key, c.value, c.slot_mapping, kc, vc)
    assert pa.last_error() == 0
    assert np.array_equal(bits(kc), exp_k) and np.array_equal(bits(vc), exp_v)


def test_reshape_and_cache_padding_and_bad_slot(pa):
    c = _cuda_case("c2", small=True)
    slots = c.slot_mapping.clone()
    slots[0] = -1
    slots[1] = c.num_blocks * c.spec.bs + 3            # outside the pool
    exp_k, exp_v = oracle.reshape_and_cache(bits(c.key)[2:], bits(c.value)[2:], slots.cpu().numpy()[2:],
                                            bits(c.k_cache), bits(c.v_cache))
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    pa.reshape_and_cache(c.key, c.value, slots, kc, vc)
    assert pa.last_error() == pa.DEV_BAD_SLOT
    assert np.array_equal(bits(kc), exp_k) and np.array_equal(bits(vc), exp_v)


@pytest.mark.parametrize("small", [True, False])
def test_copy_blocks_bit_exact(pa, small):
    cc = W.cow_case(small=small, device="cuda")
    k, v, pairs = cc["k_cache"], cc["v_cache"], cc["pairs"]
    exp_k, exp_v = oracle.copy_blocks(bits(k), bits(v), pairs.cpu().numpy())
    pa.copy_blocks(k, v, pairs)
    assert pa.last_error() == 0
    assert np.array_equal(bits(k), exp_k) and np.array_equal(bits(v), exp_v)


def test_copy_blocks_fp32_and_bad_pair(pa):
    g = torch.Generator(device="cuda").manual_seed(7)
    k = torch.randn(12, 8, 2, 64, device="cuda", generator=g)
    v = torch.randn(12, 8, 2, 64, device="cuda", generator=g)
    pairs = torch.tensor([[1, 5], [2, 6], [3, 40]], dtype=torch.int64, device="cuda")
    exp_k, exp_v = oracle.copy_blocks(bits(k), bits(v), pairs.cpu().numpy()[:2])
    pa.copy_blocks(k, v, pairs)
    assert pa.last_error() == pa.DEV_BAD_BLOCK
    assert np.array_equal(bits(k), exp_k) and np.array_equal(bits(v), exp_v)


def test_copy_blocks_onto_itself_changes_nothing(pa):
    g = torch.Generator(device="cuda").manual_seed(8)
    k = torch.randn(6, 16, 2, 64, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(6, 16, 2, 64, device="cuda", generator=g).to(torch.bfloat16)
    before_k, before_v = bits(k), bits(v)
    pa.copy_blocks(k, v, torch.tensor([[4, 4], [2, 2]], dtype=torch.int64, device="cuda"))
    assert pa.last_error() == 0
    assert np.array_equal(bits(k), before_k) and np.array_equal(bits(v), before_v)


@pytest.mark.parametrize("dtype,bs,H,D", [("bf16", 16, 8, 128), ("f32", 16, 2, 64), ("bf16", 32, 8, 128),
                                         ("bf16", 4, 1, 32)])
def test_swap_out_to_pinned_host_and_back(pa, dtype, bs, H, D):
    """Preempt: blocks of a device pool go to a page-locked host pool and come
    back into different device blocks; byte-exact both ways, and decode over
    the remapped table gives bit-identical output."""
    dt = W.DTYPES[dtype]
    g = torch.Generator(device="cuda").manual_seed(bs * D)
    NB, NH = 40, 12
    dev_k = torch.randn(NB, bs, H, D, device="cuda", generator=g).to(dt)
    dev_v = torch.randn(NB, bs, H, D, device="cuda", generator=g).to(dt)
    host_k = torch.zeros(NH, bs, H, D, dtype=dt).pin_memory()
    host_v = torch.zeros(NH, bs, H, D, dtype=dt).pin_memory()
    out_pairs = torch.tensor([[3, 0], [17, 5], [39, 11], [8, 2]], dtype=torch.int64)
    exp_hk, exp_hv = oracle.swap_blocks(bits(host_k), bits(host_v), bits(dev_k), bits(dev_v), out_pairs.numpy())
    pa.swap_blocks(host_k, host_v, dev_k, dev_v, out_pairs.cuda())
    torch.cuda.synchronize()
    assert pa.last_error() == 0
    assert np.array_equal(bits(host_k), exp_hk) and np.array_equal(bits(host_v), exp_hv)
    # swap in to other device blocks of a second pool
    back = torch.tensor([[0, 21], [5, 22], [11, 23], [2, 24]], dtype=torch.int64)
    new_k, new_v = torch.zeros_like(dev_k), torch.zeros_like(dev_v)
    exp_k, exp_v = oracle.swap_blocks(bits(new_k), bits(new_v), exp_hk, exp_hv, back.numpy())
    pa.swap_blocks(new_k, new_v, host_k, host_v, back.cuda())
    assert pa.last_error() == 0
    assert np.array_equal(bits(new_k), exp_k) and np.array_equal(bits(new_v), exp_v)
    for (s, _), (_, d) in zip(out_pairs.tolist(), back.tolist()):
        assert np.array_equal(bits(new_k)[d], bits(dev_k)[s]) and np.array_equal(bits(new_v)[d], bits(dev_v)[s])


def test_swap_restores_decode_bit_identically(pa):
    c = _cuda_case("c4", small=True)
    pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
    out1 = gpu_decode(c, append=False)
    # swap sequence 0 out, wipe its device blocks, swap it back in elsewhere
    L = int(c.context_lens[0])
    n = -(-L // c.spec.bs)
    blocks = c.block_tables[0, :n].long()
    hk = torch.empty((n,) + c.k_cache.shape[1:], dtype=c.k_cache.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    ar = torch.arange(n, device="cuda")
    pa.swap_blocks(hk, hv, c.k_cache, c.v_cache, torch.stack([blocks, ar], 1).contiguous())
    c.k_cache[blocks] = float("nan")
    c.v_cache[blocks] = float("nan")
    k = torch.cat([c.k_cache, torch.empty((n,) + c.k_cache.shape[1:], dtype=c.k_cache.dtype, device="cuda")])
    v = torch.cat([c.v_cache, torch.empty_like(k[c.num_blocks:])])
    new = ar + c.num_blocks
    pa.swap_blocks(k, v, hk, hv, torch.stack([ar, new], 1).contiguous())
    t = c.block_tables.clone()
    t[t == c.num_blocks] = k.shape[0]
    t[0, :n] = new.int()
    c.k_cache, c.v_cache, c.block_tables = k, v, t.contiguous()
    out2 = gpu_decode(c, append=False)
    assert pa.last_error() == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_swap_bad_pair_is_flagged_and_skipped(pa):
    k = torch.randn(6, 16, 2, 64, device="cuda")
    v = torch.randn(6, 16, 2, 64, device="cuda")
    hk = torch.zeros(3, 16, 2, 64).pin_memory()
    hv = torch.zeros(3, 16, 2, 64).pin_memory()
    pa.swap_blocks(hk, hv, k, v, torch.tensor([[1, 0], [2, 3], [9, 1]], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert pa.last_error() == pa.DEV_BAD_BLOCK
    exp_k, exp_v = oracle.swap_blocks(np.zeros((3, 16, 2, 64), np.float32), np.zeros((3, 16, 2, 64), np.float32),
                                      bits(k).view(np.float32), bits(v).view(np.float32), np.array([[1, 0]]))
    assert np.array_equal(hk.numpy(), exp_k) and np.array_equal(hv.numpy(), exp_v)


# ------------------------------------------------------------------ decode, small

@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c4b32", "c5"])
@pytest.mark.parametrize("partition", [0, -1, 64])
def test_decode_matches_oracle(pa, name, partition):
    c = _cuda_case(name, small=True)
    ref = oracle_decode(c)
    if partition > 0 and partition % c.spec.bs:
        partition = 4 * c.spec.bs
    out = gpu_decode(c, partition_size=partition)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, c.spec.dtype)


def test_worked_example_error_scale(pa):
    """c1: the pages' 10-token / block_size-4 fp32 example; their CPU check
    printed a 2.38e-07 max error and asserted < 1e-5."""
    c = _cuda_case("c1")
    ref = oracle_decode(c)
    err = np.abs(f64(gpu_decode(c)) - ref).max()
    assert err < 1e-5
    assert err < 1e-6          # same order as the printed fp32 figure


@pytest.mark.parametrize("lens", [[1, 15, 16, 17], [511, 512, 513, 1024], [2047, 2048, 3, 1000]])
@pytest.mark.parametrize("partition", [0, 16, 512, -1])
def test_decode_ragged_boundaries(pa, lens, partition):
    c = _cuda_case("c2", lens=lens)
    ref = oracle_decode(c)
    out = gpu_decode(c, partition_size=partition)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


@pytest.mark.parametrize("G", [1, 2, 3, 4, 8, 16, 32])
def test_decode_gqa_group_sizes(pa, G):
    c = _cuda_case("c4", small=True)
    # reuse the c4 pool (8 KV heads) with G query heads per KV head
    g = torch.Generator(device="cuda").manual_seed(G)
    c.q = torch.randn(c.q.shape[0], 8 * G, c.spec.D, generator=g, device="cuda").to(c.q.dtype)
    c.spec = W.Spec(**{**c.spec.__dict__, "Hq": 8 * G})
    ref = oracle_decode(c)
    out = gpu_decode(c)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


@pytest.mark.parametrize("Hq,Hkv,D,bs", [(16, 4, 64, 8), (32, 8, 64, 32), (8, 2, 128, 8), (16, 8, 128, 32),
                                         (12, 4, 128, 16), (8, 4, 32, 16), (8, 2, 128, 4)])
@pytest.mark.parametrize("partition", [0, -1])
def test_decode_shape_variants(pa, Hq, Hkv, D, bs, partition):
    """Tensor-core GQA path (bf16, head_dim 64/128, G a power of two, block
    size >= 8) and the CUDA-core path for the rest, against the oracle."""
    c = _cuda_case("c4", B=3, Hq=Hq, Hkv=Hkv, D=D, bs=bs, len_dist=("uniform", 1, 1500))
    ref = oracle_decode(c)
    out = gpu_decode(c, partition_size=partition)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


def test_empty_context_gives_zeros(pa):
    c = _cuda_case("c4", small=True)
    c.context_lens[1] = 0
    c.slot_mapping[1] = -1
    out = gpu_decode(c)
    assert pa.last_error() == 0
    assert (out[1] == 0).all()
    ref = oracle_decode(c)
    assert_close(f64(out), ref, "bf16")


def test_bad_block_id_and_length_are_flagged(pa):
    c = _cuda_case("c2", small=True)
    ref = oracle_decode(c)
    c.block_tables[0, 0] = c.num_blocks + 5
    out = gpu_decode(c)
    assert pa.last_error() & pa.DEV_BAD_BLOCK
    assert_close(f64(out)[1:], ref[1:], "bf16")       # other sequences unaffected
    c = _cuda_case("c2", small=True)
    c.context_lens[2] = c.max_blocks * c.spec.bs + 1
    c.slot_mapping[2] = -1
    gpu_decode(c)
    assert pa.last_error() & pa.DEV_BAD_LEN


def test_bounded_wait_gives_up_and_the_context_stays_usable(pa):
    # a pipeline wait that nothing will satisfy ends after its limit with
    # PA_DEV_TIMEOUT, which the host reads; the next calls run normally
    assert pa.last_error() == 0
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    pa.selftest_bounded_wait(20_000_000)           # 20 ms
    t1.record()
    torch.cuda.synchronize()
    assert t0.elapsed_time(t1) >= 19.0              # it waited out its limit
    assert pa.last_error() == pa.DEV_TIMEOUT
    assert pa.last_error() == 0                     # the bit is cleared once read
    c = _cuda_case("c2", small=True)
    out = gpu_decode(c)
    assert pa.last_error() == 0
    assert_close(f64(out), oracle_decode(c), "bf16")


def test_permuted_pool_gives_bit_identical_output(pa):
    c = _cuda_case("c4", small=True)
    out1 = gpu_decode(c)
    perm = torch.randperm(c.num_blocks, generator=torch.Generator().manual_seed(1)).cuda()
    k2 = torch.empty_like(c.k_cache)
    v2 = torch.empty_like(c.v_cache)
    k2[perm] = c.k_cache
    v2[perm] = c.v_cache
    t = c.block_tables.long()
    valid = t < c.num_blocks
    t2 = torch.where(valid, perm[t.clamp(max=c.num_blocks - 1)], t).int()
    s = c.slot_mapping
    s2 = perm[s // c.spec.bs] * c.spec.bs + s % c.spec.bs
    c.k_cache, c.v_cache, c.block_tables, c.slot_mapping = k2, v2, t2.contiguous(), s2.contiguous()
    out2 = gpu_decode(c)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("name,partition", [("c2", 64), ("c4", 64), ("c3", 0)])
def test_decode_on_a_side_stream_is_bit_identical(pa, name, partition):
    """Split-K decode enqueued on a user stream (the merge is then a
    programmatic dependent of the decode kernel) gives the same bits as on
    the current stream, and back to back calls on that stream do not see
    each other's partials."""
    c = _cuda_case(name, small=True)
    pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
    torch.cuda.synchronize()
    ref = torch.full_like(c.q, float("nan"))
    pa.decode(ref, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, partition_size=partition)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    ws = pa.alloc_workspace(c.q, c.k_cache, c.block_tables, partition_size=partition)
    outs = [torch.full_like(c.q, float("nan")) for _ in range(3)]
    q2 = c.q.flip(0).contiguous()          # a second, different case between two identical ones
    with torch.cuda.stream(side):
        pa.decode(outs[0], c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale,
                  partition_size=partition, workspace=ws, stream=side)
        pa.decode(outs[1], q2, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale,
                  partition_size=partition, workspace=ws, stream=side)
        pa.decode(outs[2], c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale,
                  partition_size=partition, workspace=ws, stream=side)
    side.synchronize()
    assert pa.last_error() == 0
    assert torch.equal(outs[0].view(torch.int16), ref.view(torch.int16))
    assert torch.equal(outs[2].view(torch.int16), ref.view(torch.int16))
    assert_close(f64(ref), oracle_decode(c), "bf16")


def test_shared_prefix_equals_private_copies(pa):
    c = _cuda_case("c5", small=True)
    pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
    out_shared = gpu_decode(c, append=False)
    assert torch.isfinite(out_shared.float()).all()
    # give every sequence private copies of its prompt blocks via pa_copy_blocks
    tables = c.block_tables.cpu().numpy().copy()
    pre = c.extra["prefix"] // c.spec.bs
    free = list(c.extra["free_blocks"])
    need = (c.q.shape[0] - c.extra["prompts"]) * pre
    k = torch.cat([c.k_cache, torch.empty((need,) + c.k_cache.shape[1:], dtype=c.k_cache.dtype,
                                          device="cuda")])
    v = torch.cat([c.v_cache, torch.empty_like(k[c.num_blocks:])])
    tables[tables == c.num_blocks] = k.shape[0]        # unused entries stay out of range
    nxt = c.num_blocks
    pairs = []
    for b in range(c.q.shape[0]):
        if b % c.extra["samples"] == 0:
            continue                      # the first sample keeps the originals
        for j in range(pre):
            pairs.append((int(tables[b, j]), nxt))
            tables[b, j] = nxt
            nxt += 1
    pa.copy_blocks(k, v, torch.tensor(pairs, dtype=torch.int64, device="cuda"))
    c.k_cache, c.v_cache = k, v
    c.block_tables = torch.from_numpy(tables).cuda()
    out_private = gpu_decode(c, append=False)
    assert pa.last_error() == 0 and free is not None
    assert torch.equal(out_shared.view(torch.int16), out_private.view(torch.int16))


# ------------------------------------------------------------------ full size

def _full_check(pa, name, n_sample=6, partition=0):
    c = W.decode_case(name, device="cuda")
    lens = c.context_lens.cpu().numpy()
    rng = np.random.default_rng(99)
    seqs = sorted(set([int(np.argmax(lens)), int(np.argmin(lens))] +
                      rng.choice(len(lens), n_sample, replace=False).tolist()))
    ref = oracle_decode(c, seqs)                     # before the pool is touched
    out = gpu_decode(c, partition_size=partition, clone=False)
    assert pa.last_error() == 0
    got = f64(out)
    assert np.isfinite(got).all()
    # every output is a convex combination of V rows
    vmax = float(torch.nan_to_num(c.v_cache.float(), nan=0.0).abs().max())
    assert np.abs(got).max() <= vmax + 1e-6
    return assert_close(got[seqs], ref, c.spec.dtype), c, out


@pytest.mark.parametrize("name", ["c2", "c3", "c5"])
def test_full_size_sampled(pa, name):
    _full_check(pa, name)


@pytest.mark.parametrize("partition", [0, 512])
@pytest.mark.parametrize("name", ["c4", "c4b32"])
def test_full_size_gqa_split_sampled(pa, name, partition):
    # automatic (2048-token) partitions and the configuration's 512-token ones
    (_, c, out) = _full_check(pa, name, n_sample=3, partition=partition)
    del c, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("lens", [[511, 512, 513, 1024, 1537], [2047, 2048, 2049, 1, 4095]])
@pytest.mark.parametrize("partition", [512, 2048])
def test_gqa_ragged_partition_boundaries(pa, lens, partition):
    # grouped-query path (tokens in M) across 512- and 2048-token partition edges
    c = _cuda_case("c4", lens=lens)
    ref = oracle_decode(c)
    out = gpu_decode(c, partition_size=partition)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


def test_full_c2_split_equals_unsplit(pa):
    c = W.decode_case("c2", device="cuda")
    a = gpu_decode(c, partition_size=0)
    b = gpu_decode(c, partition_size=-1)
    assert_close(f64(a), f64(b), "bf16")
