"""e4m3 KV cache with per-token scales, through the C ABI, against the oracle.

The append quantises on both sides in float32 and must match byte for byte
(codes and scales).  Decode over the e4m3 pool must match the float64 decode
of the dequantised pool within the bf16 tolerance (fp32 accumulation, bf16
output).  Inputs come from the seeded generators only.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_307_gb300 import workloads as W
from _helpers import f64, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_307_gb300 import build
    build.build()
    from paged_kv_cache_307_gb300 import _lib
    assert torch.cuda.is_available()
    _lib.last_error()
    return _lib


def _case(name, small=True, device="cuda", **kw):
    c = W.fp8_case(W.decode_case(name, small=small, **kw))
    if device == "cuda":
        for f in ("q", "k_cache", "v_cache", "block_tables", "context_lens", "key", "value", "slot_mapping"):
            setattr(c, f, getattr(c, f).cuda())
        c.extra["k_scale"] = c.extra["k_scale"].cuda()
        c.extra["v_scale"] = c.extra["v_scale"].cuda()
    return c


def _np(t):
    return t.detach().cpu().numpy()


def oracle_fp8(c, seqs=None):
    """Oracle: quantise-append each sequence's newest token, then decode over
    the dequantised pool (only the blocks the chosen sequences use)."""
    s = c.spec
    lens = _np(c.context_lens)
    tables = _np(c.block_tables)
    seqs = list(range(len(lens))) if seqs is None else list(seqs)
    used = sorted({int(tables[b, j]) for b in seqs for j in range(-(-int(lens[b]) // s.bs))})
    index = {blk: i for i, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=c.k_cache.device)
    kc, vc = _np(c.k_cache.index_select(0, idx)), _np(c.v_cache.index_select(0, idx))
    ks, vs = _np(c.extra["k_scale"].index_select(0, idx)), _np(c.extra["v_scale"].index_select(0, idx))
    nt = np.zeros((len(seqs), tables.shape[1]), dtype=np.int64)
    for r, b in enumerate(seqs):
        for j in range(-(-int(lens[b]) // s.bs)):
            nt[r, j] = index[int(tables[b, j])]
    slots = _np(c.slot_mapping)
    new = [-1 if slots[b] < 0 else index[int(slots[b]) // s.bs] * s.bs + int(slots[b]) % s.bs for b in seqs]
    key, val = f64(c.key)[seqs], f64(c.value)[seqs]
    kc, vc, ks, vs = oracle.reshape_and_cache_fp8(key, val, np.array(new), kc, vc, ks, vs)
    return oracle.paged_decode_fp8(f64(c.q)[seqs], kc, vc, ks, vs, nt, lens[seqs], c.scale)


def gpu_fp8(pa, c, partition_size=0, clone=True):
    kc = c.k_cache.clone() if clone else c.k_cache
    vc = c.v_cache.clone() if clone else c.v_cache
    ks = c.extra["k_scale"].clone() if clone else c.extra["k_scale"]
    vs = c.extra["v_scale"].clone() if clone else c.extra["v_scale"]
    pa.reshape_and_cache_fp8(c.key, c.value, c.slot_mapping, kc, vc, ks, vs)
    out = torch.full_like(c.q, float("nan"))
    pa.decode_fp8(out, c.q, kc, vc, ks, vs, c.block_tables, c.context_lens, c.scale, partition_size=partition_size)
    torch.cuda.synchronize()
    return out, (kc, vc, ks, vs)


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("name", ["c2", "c4", "c5"])
def test_append_fp8_bit_exact(pa, name):
    c = _case(name)
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    ks, vs = c.extra["k_scale"].clone(), c.extra["v_scale"].clone()
    pa.reshape_and_cache_fp8(c.key, c.value, c.slot_mapping, kc, vc, ks, vs)
    assert pa.last_error() == 0
    e = oracle.reshape_and_cache_fp8(f64(c.key), f64(c.value), _np(c.slot_mapping), _np(c.k_cache),
                                     _np(c.v_cache), _np(c.extra["k_scale"]), _np(c.extra["v_scale"]))
    assert np.array_equal(_np(kc), e[0]) and np.array_equal(_np(vc), e[1])
    assert np.array_equal(_np(ks).view(np.uint32), e[2].view(np.uint32))
    assert np.array_equal(_np(vs).view(np.uint32), e[3].view(np.uint32))


def test_append_fp8_from_fp32_with_zero_and_extreme_tokens(pa):
    g = torch.Generator(device="cuda").manual_seed(11)
    NB, bs, H, D, T = 8, 16, 4, 64, 6
    key = torch.randn(T, H, D, device="cuda", generator=g)
    val = torch.randn(T, H, D, device="cuda", generator=g) * 1e-3
    key[1] = 0.0                                # zero vector: scale 0, codes 0
    key[2] *= 1e4                               # large magnitudes
    key[3, 0, 0] = -key[3].abs().max() * 2      # a negative maximum
    val[4] = -0.0
    slots = torch.tensor([0, 17, 33, 50, 101, -1], dtype=torch.int64, device="cuda")
    kc = torch.zeros(NB, bs, H, D, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.full((NB, bs), 7.0, device="cuda")
    vs = torch.full((NB, bs), 7.0, device="cuda")
    e = oracle.reshape_and_cache_fp8(f64(key).astype(np.float32), f64(val).astype(np.float32), _np(slots),
                                     _np(kc), _np(vc), _np(ks), _np(vs))
    pa.reshape_and_cache_fp8(key, val, slots, kc, vc, ks, vs)
    assert pa.last_error() == 0
    assert np.array_equal(_np(kc), e[0]) and np.array_equal(_np(vc), e[1])
    assert np.array_equal(_np(ks).view(np.uint32), e[2].view(np.uint32))
    assert np.array_equal(_np(vs).view(np.uint32), e[3].view(np.uint32))
    assert float(ks[1, 1]) == 0.0 and not kc[1, 1].any()


def test_append_fp8_bad_slot(pa):
    c = _case("c2")
    slots = c.slot_mapping.clone()
    slots[0] = c.num_blocks * c.spec.bs + 1
    kc, vc = c.k_cache.clone(), c.v_cache.clone()
    ks, vs = c.extra["k_scale"].clone(), c.extra["v_scale"].clone()
    pa.reshape_and_cache_fp8(c.key, c.value, slots, kc, vc, ks, vs)
    assert pa.last_error() == pa.DEV_BAD_SLOT


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("name", ["c2", "c3", "c4", "c4b32", "c5"])
@pytest.mark.parametrize("partition", [0, -1, 64])
def test_decode_fp8_matches_oracle(pa, name, partition):
    c = _case(name)
    ref = oracle_fp8(c)
    out, _ = gpu_fp8(pa, c, partition_size=partition)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


@pytest.mark.parametrize("Hq,Hkv,D,bs", [(8, 8, 128, 16), (16, 4, 64, 8), (32, 8, 64, 32), (8, 2, 128, 8),
                                         (16, 8, 128, 32), (12, 4, 128, 16), (8, 4, 32, 16), (8, 2, 128, 4),
                                         (64, 8, 128, 16), (6, 2, 64, 16), (32, 2, 128, 16), (64, 2, 128, 16),
                                         (8, 1, 128, 16)])
def test_decode_fp8_shape_variants(pa, Hq, Hkv, D, bs):
    c = _case("c4", B=3, Hq=Hq, Hkv=Hkv, D=D, bs=bs, len_dist=("uniform", 1, 1500))
    ref = oracle_fp8(c)
    out, _ = gpu_fp8(pa, c)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


@pytest.mark.parametrize("lens", [[1, 15, 16, 17], [511, 512, 513, 1024]])
def test_decode_fp8_ragged(pa, lens):
    c = _case("c2", lens=lens)
    ref = oracle_fp8(c)
    for partition in (0, 16, -1):
        out, _ = gpu_fp8(pa, c, partition_size=partition)
        assert pa.last_error() == 0
        assert_close(f64(out), ref, "bf16")


def test_decode_fp8_zero_scale_tokens_and_empty_context(pa):
    c = _case("c4")
    c.extra["k_scale"][c.block_tables[0, 0].long(), :5] = 0.0     # keys quantised from zero vectors
    c.extra["v_scale"][c.block_tables[1, 0].long(), 2:9] = 0.0
    c.context_lens[2] = 0
    c.slot_mapping[2] = -1
    ref = oracle_fp8(c)
    out, _ = gpu_fp8(pa, c)
    assert pa.last_error() == 0
    assert (out[2] == 0).all()
    assert_close(f64(out), ref, "bf16")


@pytest.mark.parametrize("name", ["c2", "c5"])
def test_decode_fp8_full_size_sampled(pa, name):
    c = W.fp8_case(W.decode_case(name, device="cuda"))
    lens = _np(c.context_lens)
    rng = np.random.default_rng(7)
    seqs = sorted(set([int(np.argmax(lens)), int(np.argmin(lens))] +
                      rng.choice(len(lens), 5, replace=False).tolist()))
    ref = oracle_fp8(c, seqs)
    out, (_, vc, _, vs) = gpu_fp8(pa, c, clone=False)
    assert pa.last_error() == 0
    got = f64(out)
    assert np.isfinite(got).all()
    assert_close(got[seqs], ref, "bf16")


def test_fp8_is_close_to_full_precision(pa):
    """Quantisation error, not parity: quantise every token of a bf16 pool
    with the fp8 append, decode, and stay near the float64 decode of the
    unquantised pool (e4m3 keeps 3 mantissa bits)."""
    from _helpers import oracle_decode
    c = W.decode_case("c2", small=True, device="cuda", nan_fill=False)
    s = c.spec
    lens = _np(c.context_lens)
    tables = _np(c.block_tables)
    slots = np.array([int(tables[b, t // s.bs]) * s.bs + t % s.bs
                      for b in range(len(lens)) for t in range(int(lens[b]) - 1)], dtype=np.int64)
    st = torch.from_numpy(slots).cuda()
    key = c.k_cache.view(-1, s.Hkv, s.D)[st].contiguous()
    val = c.v_cache.view(-1, s.Hkv, s.D)[st].contiguous()
    kc = torch.zeros(c.k_cache.shape, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros(c.k_cache.shape[:2], device="cuda")
    vs = torch.zeros_like(ks)
    pa.reshape_and_cache_fp8(key, val, st, kc, vc, ks, vs)
    pa.reshape_and_cache_fp8(c.key, c.value, c.slot_mapping, kc, vc, ks, vs)
    out = torch.empty_like(c.q)
    pa.decode_fp8(out, c.q, kc, vc, ks, vs, c.block_tables, c.context_lens, c.scale)
    torch.cuda.synchronize()
    assert pa.last_error() == 0
    ref = oracle_decode(c)
    err = np.abs(f64(out) - ref)
    assert err.max() < 0.05 and err.mean() < 0.01


def test_copy_blocks_fp8_with_scales(pa):
    cc = W.cow_case(small=True, device="cuda")
    k, v, pairs = cc["k_cache"], cc["v_cache"], cc["pairs"]
    fc = W.fp8_case(W.DecodeCase(W.SPECS["c5"], 1.0, k[:1, 0], k, v, None, None, None, None, None))
    kc, vc = fc.k_cache, fc.v_cache
    ks, vs = fc.extra["k_scale"], fc.extra["v_scale"]
    ek, ev = oracle.copy_blocks(_np(kc), _np(vc), _np(pairs))
    eks, evs = oracle.copy_blocks(_np(ks), _np(vs), _np(pairs))
    pa.copy_blocks_fp8(kc, vc, ks, vs, pairs)
    torch.cuda.synchronize()
    assert pa.last_error() == 0
    assert np.array_equal(_np(kc), ek) and np.array_equal(_np(vc), ev)
    assert np.array_equal(_np(ks).view(np.uint32), eks.view(np.uint32))
    assert np.array_equal(_np(vs).view(np.uint32), evs.view(np.uint32))
