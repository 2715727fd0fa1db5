"""Chunked-prefill tile on the tensor cores (through the C ABI) against the
float64 oracle.  bf16 inputs, fp32 accumulation, P rounded to bf16: the
bf16 tolerance applies (max 2e-2, mean 2e-3)."""

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


def _oracle(case, seqs=None):
    lens = case["context_lens"].cpu().numpy()
    tables = case["block_tables"].cpu().numpy()
    bs = case["block_size"]
    seqs = list(range(len(lens))) if seqs is None else list(seqs)
    used = sorted({int(tables[b, j]) for b in seqs for j in range(-(-int(lens[b]) // bs))})
    index = {blk: i for i, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=case["k_cache"].device)
    k = f64(case["k_cache"].index_select(0, idx))
    v = f64(case["v_cache"].index_select(0, idx))
    nt = np.zeros((len(seqs), tables.shape[1]), dtype=np.int64)
    for r, b in enumerate(seqs):
        for j in range(-(-int(lens[b]) // bs)):
            nt[r, j] = index[int(tables[b, j])]
    q = f64(case["q"])[seqs]
    return oracle.paged_prefill(q, k, v, nt, lens[seqs], case["scale"])


def _run(pa, case):
    out = torch.full_like(case["q"], float("nan"))
    pa.prefill(out, case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
               case["context_lens"], case["scale"])
    torch.cuda.synchronize()
    return out


def test_prefill_c5_small(pa):
    case = W.prefill_case(small=True, device="cuda")
    ref = _oracle(case)
    out = _run(pa, case)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (32, 4), (32, 2)])
def test_prefill_group_sizes(pa, Hq, Hkv):
    case = W.prefill_case(device="cuda", Hq=Hq, Hkv=Hkv, Tq=160, lens=[300, 161])
    ref = _oracle(case)
    out = _run(pa, case)
    assert pa.last_error() == 0
    assert_close(f64(out), ref, "bf16")


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_prefill_block_sizes_and_ragged_tails(pa, bs):
    # lengths that end mid-block and mid-tile, one shorter than the tile
    case = W.prefill_case(device="cuda", bs=bs, Tq=200, lens=[131, 517, 77])
    ref = _oracle(case)
    out = _run(pa, case)
    assert pa.last_error() == 0
    got = f64(out)
    assert not got[2, :200 - 77].any()          # rows before position 0 are zero
    assert_close(got, ref, "bf16")


def test_prefill_single_query_equals_decode(pa):
    """Tq = 1 is a decode step: the tile row equals pa_decode's output."""
    case = W.prefill_case(device="cuda", Tq=1, lens=[700, 33, 1024])
    out = _run(pa, case)
    dec = torch.empty_like(case["q"][:, 0])
    pa.decode(dec, case["q"][:, 0].contiguous(), case["k_cache"], case["v_cache"], case["block_tables"],
              case["context_lens"], case["scale"])
    torch.cuda.synchronize()
    assert_close(f64(out[:, 0]), f64(dec), "bf16")
    assert_close(f64(out), _oracle(case), "bf16")


def test_prefill_full_size_sampled(pa):
    case = W.prefill_case(device="cuda")
    seqs = [0, 37]
    ref = _oracle(case, seqs)
    out = _run(pa, case)
    assert pa.last_error() == 0
    got = f64(out)
    assert np.isfinite(got).all()
    assert_close(got[seqs], ref, "bf16")


# ------------------------------------------------------------------ mixed rounds (ragged query counts)

def _oracle_varlen(case, seqs=None):
    lens = case["context_lens"].cpu().numpy()
    tables = case["block_tables"].cpu().numpy()
    qs = case["query_start"].cpu().numpy()
    bs = case["block_size"]
    seqs = list(range(len(lens))) if seqs is None else list(seqs)
    used = sorted({int(tables[b, j]) for b in seqs for j in range(-(-int(lens[b]) // bs))})
    index = {blk: i for i, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=case["k_cache"].device)
    k = f64(case["k_cache"].index_select(0, idx))
    v = f64(case["v_cache"].index_select(0, idx))
    nt = np.zeros((len(seqs), tables.shape[1]), dtype=np.int64)
    for r, b in enumerate(seqs):
        for j in range(-(-int(lens[b]) // bs)):
            nt[r, j] = index[int(tables[b, j])]
    rows = [np.arange(qs[b], qs[b + 1]) for b in seqs]
    sub_qs = np.concatenate([[0], np.cumsum([len(r) for r in rows])])
    q = f64(case["q"])[np.concatenate(rows)] if sub_qs[-1] else f64(case["q"])[:0]
    return oracle.paged_prefill_varlen(q, sub_qs, k, v, nt, lens[seqs], case["scale"]), np.concatenate(rows)


def _run_varlen(pa, case):
    out = torch.full_like(case["q"], float("nan"))
    pa.prefill_varlen(out, case["q"], case["query_start"], case["k_cache"], case["v_cache"],
                      case["block_tables"], case["context_lens"], case["scale"])
    torch.cuda.synchronize()
    return out


def test_mixed_round_small(pa):
    case = W.mixed_case(small=True, device="cuda")
    ref, rows = _oracle_varlen(case)
    out = _run_varlen(pa, case)
    assert pa.last_error() == 0
    assert_close(f64(out)[rows], ref, "bf16")


@pytest.mark.parametrize("chunk", [1, 2, 3, 31, 32, 33, 100])
def test_mixed_round_ragged_chunks_and_empty_sequences(pa, chunk):
    case = W.mixed_case(small=True, device="cuda", chunk=chunk, prefix=300, n_decode=5, n_prefill=3)
    # give sequence 1 no work this round: drop its rows from the packing
    qs = case["query_start"].cpu().numpy().astype(np.int64)
    n = np.diff(qs)
    keep = np.concatenate([np.arange(qs[b], qs[b + 1]) for b in range(len(n)) if b != 1])
    n[1] = 0
    case["q"] = case["q"][torch.from_numpy(keep).cuda()].contiguous()
    case["query_start"] = torch.from_numpy(np.concatenate([[0], np.cumsum(n)]).astype(np.int32)).cuda()
    ref, rows = _oracle_varlen(case)
    out = _run_varlen(pa, case)
    assert pa.last_error() == 0
    assert_close(f64(out)[rows], ref, "bf16")


@pytest.mark.parametrize("heads,dq", [((16, 8), 1), ((16, 8), 3), ((16, 8), 4), ((16, 8), 5), ((8, 8), 8), ((32, 4), 1),
                                      ((32, 8), 2)])
def test_short_requests_in_a_round(pa, heads, dq):
    """Requests with a few query positions each (a decode step, or a short
    causal run such as a speculative step) beside prefill chunks, for several
    group sizes: every row sees its own causal limit."""
    case = W.mixed_case(small=True, device="cuda", heads=heads, decode_queries=dq, n_prefill=2, chunk=40,
                        prefix=200, n_decode=7, decode_lens=("uniform", 1, 300))
    ref, rows = _oracle_varlen(case)
    out = _run_varlen(pa, case)
    assert pa.last_error() == 0
    assert_close(f64(out)[rows], ref, "bf16")


@pytest.mark.parametrize("kind", ["decreasing", "past_the_rows"])
def test_bad_query_start_is_flagged_and_skipped(pa, kind):
    """A decreasing pair of starts, or a start past the query rows, is
    flagged PA_DEV_BAD_LEN and those sequences write nothing; the others
    are unaffected."""
    case = W.mixed_case(small=True, device="cuda", n_prefill=3, chunk=40, prefix=200, n_decode=6)
    qs = case["query_start"].cpu().numpy().astype(np.int64)
    B = len(qs) - 1
    ok_seqs = [0] + list(range(4, B - 1))
    if kind == "decreasing":
        qs[2] = qs[3] + 1                     # sequence 2 decreasing; 1 and 3 overlap it
    else:
        qs[B] = qs[B - 1] + case["q"].shape[0]   # the last sequence ends past the rows
        ok_seqs = [0, 1, 2, 3] + ok_seqs[1:]
    case["query_start"] = torch.from_numpy(qs.astype(np.int32)).cuda()
    out = _run_varlen(pa, case)
    assert pa.last_error() & pa.DEV_BAD_LEN
    ref, rows = _oracle_varlen(case, ok_seqs)
    assert_close(f64(out)[rows], ref, "bf16")
    assert pa.last_error() == 0


def test_uniform_round_equals_fixed_count_tile(pa):
    case = W.prefill_case(small=True, device="cuda", Tq=96)
    fixed = _run(pa, case)
    P, Tq, Hq, D = case["q"].shape
    vl = dict(case, q=case["q"].reshape(P * Tq, Hq, D),
              query_start=torch.arange(0, (P + 1) * Tq, Tq, dtype=torch.int32, device="cuda"))
    out = _run_varlen(pa, vl)
    assert pa.last_error() == 0
    assert torch.equal(out.view(torch.int16), fixed.reshape(P * Tq, Hq, D).view(torch.int16))


def test_decode_only_round_matches_decode_oracle(pa):
    case = W.mixed_case(small=True, device="cuda", n_prefill=0, n_decode=12)
    ref, rows = _oracle_varlen(case)
    out = _run_varlen(pa, case)
    assert pa.last_error() == 0
    assert_close(f64(out)[rows], ref, "bf16")


def test_mixed_round_full_size_sampled(pa):
    case = W.mixed_case(device="cuda")
    lens = case["context_lens"].cpu().numpy()
    rng = np.random.default_rng(3)
    seqs = sorted(set([0, int(case["n_prefill"]) - 1] +
                      (case["n_prefill"] + rng.choice(case["n_decode"], 6, replace=False)).tolist()))
    ref, rows = _oracle_varlen(case, seqs)
    out = _run_varlen(pa, case)
    assert pa.last_error() == 0
    got = f64(out)
    assert np.isfinite(got).all()
    assert_close(got[rows], ref, "bf16")
    assert len(lens) == case["n_prefill"] + case["n_decode"]
