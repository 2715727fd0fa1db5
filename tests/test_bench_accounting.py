"""The benchmark's work accounting against closed forms, and the structure of
the e4m3 and mixed-round inputs (CPU).

The roofline figures divide these counts by measured time, so each is pinned
to an expression derived by hand from the workload definition rather than to
the helper's own loop.
"""

import numpy as np
import pytest
import torch

from paged_kv_cache_307_gb300 import workloads as W


def test_causal_tile_flops_closed_form():
    # queries at positions L-Tq .. L-1, query i sees L-Tq+i+1 keys:
    # sum = Tq*(L-Tq) + Tq*(Tq+1)/2 pairs, 4*Hq*D flops per pair (QK^T and PV)
    L, Tq, Hq, D, P = 1024, 512, 32, 128, 64
    pairs = Tq * (L - Tq) + Tq * (Tq + 1) // 2
    assert W.prefill_flops([L] * P, Tq, Hq, D) == P * pairs * 4 * Hq * D
    # the chunked-prefill tile of 64 prompts is about 412 GFLOP
    assert W.prefill_flops([L] * P, Tq, Hq, D) == pytest.approx(412.6e9, rel=1e-3)
    # a prompt shorter than the tile only counts its real positions
    assert W.prefill_flops([3], 5, 1, 1) == 4 * (1 + 2 + 3)


def test_mixed_round_flops_reduce_to_decode_and_prefill():
    Hq, D = 32, 128
    # a decode request (one query at position L-1) sees all L keys
    assert W.varlen_flops([100], [1], Hq, D) == 4 * Hq * D * 100
    # a prefill chunk counts exactly what the causal tile counts
    assert W.varlen_flops([1024], [512], Hq, D) == W.prefill_flops([1024], 512, Hq, D)
    assert W.varlen_flops([1024, 77], [512, 1], Hq, D) == \
        W.prefill_flops([1024], 512, Hq, D) + 4 * Hq * D * 77


def test_c2_algorithmic_bytes_per_token():
    c = W.decode_case("c2", nan_fill=False)
    lens = c.context_lens.numpy().astype(np.int64)
    B, Hq, D = c.q.shape
    # K and V rows of 32 KV heads x 128 dims in bf16: 16 384 bytes per token
    per_token = 2 * 32 * 128 * 2
    assert W._kv_token_bytes(c) == per_token == 16384
    tables = sum(-(-int(L) // 16) for L in lens) * 4 + 4 * B
    assert W.algorithmic_decode_bytes(c) == int(lens.sum()) * per_token + 2 * B * Hq * D * 2 + tables
    # private blocks only: counting each physical block once changes nothing
    assert W.unique_decode_bytes(c) == W.algorithmic_decode_bytes(c)


def test_shared_prompts_are_counted_once_in_unique_bytes():
    c = W.decode_case("c5", small=True, nan_fill=False)
    assert W.unique_decode_bytes(c) < W.algorithmic_decode_bytes(c)
    # the difference is exactly the prompt blocks read by the 7 other siblings
    P, S, bs = c.extra["prompts"], c.extra["samples"], c.spec.bs
    shared_tokens = (c.extra["prefix"] // bs) * bs
    saved = P * (S - 1) * shared_tokens * W._kv_token_bytes(c)
    assert W.algorithmic_decode_bytes(c) - W.unique_decode_bytes(c) == saved


def test_fp8_inputs_follow_their_recipe():
    c = W.decode_case("c1", nan_fill=True)
    f = W.fp8_case(c)
    NB, bs = c.k_cache.shape[:2]
    ks, vs = f.extra["k_scale"], f.extra["v_scale"]
    assert f.k_cache.dtype == torch.uint8 and ks.shape == (NB, bs) and ks.dtype == torch.float32
    nan = torch.isnan(c.k_cache.float()).flatten(2).any(-1)
    assert nan.any() and (~nan).any()
    # scales of live slots drawn from [0.5, 1.5] / 112; NaN slots carry NaN scales and NaN codes
    live = ks[~nan]
    assert (live >= 0.5 / 112 - 1e-9).all() and (live <= 1.5 / 112 + 1e-9).all()
    assert torch.isnan(ks[nan]).all() and torch.isnan(vs[nan]).all()
    assert ((f.k_cache[nan] & 0x7F) == 0x7F).all()
    # live codes are torch's e4m3 cast of the clipped pool x 112
    x = (c.k_cache.float() * 112.0).clamp(-448.0, 448.0)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(f.k_cache[~nan], ref[~nan])
    # the byte count per token adds the two fp32 scales to the code bytes
    assert W._kv_token_bytes(f) == 2 * c.spec.Hkv * c.spec.D + 8
    # the same seed gives the same scales
    assert torch.equal(W.fp8_case(c).extra["v_scale"][~nan], vs[~nan])


def test_mixed_round_packing():
    m = W.mixed_case(small=True)
    qs = m["query_start"].numpy()
    lens = m["context_lens"].numpy()
    npf, nd = m["n_prefill"], m["n_decode"]
    assert len(qs) == npf + nd + 1 and qs[0] == 0 and qs[-1] == m["q"].shape[0]
    nq = np.diff(qs)
    assert (nq[:npf] == 512).all() and (nq[npf:] == 1).all()
    assert (lens[:npf] == 1024).all() and (lens[npf:] >= 128).all() and (lens[npf:] <= 2048).all()
    # every query's context fits its table row
    bs = m["block_size"]
    assert (-(-lens // bs) <= m["block_tables"].shape[1]).all()


def _sampler_with(lines, t0, t1):
    import bench
    s = bench.ClockSampler(0)
    s.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout=None: 0,
                            "kill": lambda self: None})()
    s.t = type("T", (), {"join": lambda self, timeout=None: None})()
    s.lines = list(lines)
    s.t0, s.t1 = t0, t1
    return s.stop()


def _smi(ts, mhz, reasons=("Not Active",) * 4):
    import datetime
    stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(mhz), "2070", "900.0", "0x0"] + list(reasons))


def test_clock_record_keeps_the_timed_region():
    # 20 ms samples from 1000.00 s: an idle lead-in at 1000 MHz, the timed
    # region at 2070 MHz from 1000.30 to 1000.50 s, a tail at 1500 MHz
    t = [1000.0 + 0.02 * i for i in range(40)]
    mhz = [1000 if x < 1000.3 else 2070 if x <= 1000.5 else 1500 for x in t]
    r = _sampler_with([_smi(x, m) for x, m in zip(t, mhz)], 1000.3, 1000.5)
    assert r["sm_mhz"] == 2070 and r["which"] == "inside the timed region"
    assert r["samples"] == 11 and r["reasons"] == [] and r["region_ms"] == pytest.approx(200.0)
    # a throttle reason inside the region is reported, one outside it is not
    lines = [_smi(x, m, ("Active",) + ("Not Active",) * 3 if x < 1000.1 else ("Not Active",) * 3 + ("Active",)
                  if 1000.35 < x < 1000.45 else ("Not Active",) * 4) for x, m in zip(t, mhz)]
    assert _sampler_with(lines, 1000.3, 1000.5)["reasons"] == ["sw_power_cap"]


def test_clock_record_of_a_region_shorter_than_the_sampling_interval():
    t = [1000.0 + 0.02 * i for i in range(10)]
    mhz = [1800, 1800, 1800, 2070, 2070, 1900, 1900, 1900, 1900, 1900]
    # a 4 ms region between the samples at 1000.06 and 1000.08
    r = _sampler_with([_smi(x, m) for x, m in zip(t, mhz)], 1000.0705, 1000.0745)
    assert r["which"].startswith("nearest") and r["samples"] == 2 and r["sm_mhz"] == 2070
