"""Marshalling shared by the GPU tests: run the oracle and the CUDA path on the
same seeded case and compare.  Oracle inputs come from the workload tensors
(widened exactly to float64), never from a CUDA-path result."""

import numpy as np
import torch

import oracle

TOL = {"f32": dict(max=1e-5, mean=1e-5), "bf16": dict(max=2e-2, mean=2e-3)}


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def bits(t):
    """Bit pattern view (exact comparisons, NaN-safe)."""
    t = t.detach().to("cpu").contiguous()
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).numpy()


def compact(case, seqs=None):
    """The pool blocks the chosen sequences use, as float64 arrays, with the
    block tables renumbered to index them."""
    s = case.spec
    lens = case.context_lens.cpu().numpy()
    tables = case.block_tables.cpu().numpy()
    seqs = range(len(lens)) if seqs is None else seqs
    used = sorted({int(tables[b, j]) for b in seqs for j in range(-(-int(lens[b]) // s.bs))})
    index = {blk: i for i, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=case.k_cache.device)
    k = f64(case.k_cache.index_select(0, idx)) if used else np.zeros((0, s.bs, s.Hkv, s.D))
    v = f64(case.v_cache.index_select(0, idx)) if used else np.zeros((0, s.bs, s.Hkv, s.D))
    nt = np.zeros((len(list(seqs)), tables.shape[1]), dtype=np.int64)
    for r, b in enumerate(seqs):
        for j in range(-(-int(lens[b]) // s.bs)):
            nt[r, j] = index[int(tables[b, j])]
    return k, v, nt, index


def oracle_decode(case, seqs=None):
    """Oracle: append each sequence's newest token, then dense attention."""
    lens = case.context_lens.cpu().numpy()
    seqs = list(range(len(lens))) if seqs is None else list(seqs)
    k, v, nt, index = compact(case, seqs)
    s = case.spec
    slots = case.slot_mapping.cpu().numpy()
    key, val = f64(case.key), f64(case.value)
    new_slots = []
    for b in seqs:
        sl = int(slots[b])
        new_slots.append(-1 if sl < 0 else index[sl // s.bs] * s.bs + sl % s.bs)
    k, v = oracle.reshape_and_cache(key[seqs], val[seqs], np.array(new_slots), k, v)
    q = f64(case.q)[seqs]
    return oracle.paged_decode(q, k, v, nt, lens[seqs], case.scale)


def gpu_decode(case, partition_size=0, append=True, clone=True):
    """Append (on copies of the pools unless clone=False), then decode."""
    from paged_kv_cache_307_gb300 import _lib as pa
    kc = case.k_cache.clone() if clone else case.k_cache
    vc = case.v_cache.clone() if clone else case.v_cache
    if append:
        pa.reshape_and_cache(case.key, case.value, case.slot_mapping, kc, vc)
    out = torch.full_like(case.q, float("nan"))
    pa.decode(out, case.q, kc, vc, case.block_tables, case.context_lens,
              case.scale, partition_size=partition_size)
    torch.cuda.synchronize()
    return out


def assert_close(got, ref, dtype):
    tol = TOL[dtype]
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), "non-finite output"
    assert err.max() <= tol["max"], "max abs err %.3g > %.3g" % (err.max(), tol["max"])
    assert err.mean() <= tol["mean"], "mean abs err %.3g > %.3g" % (err.mean(), tol["mean"])
    return float(err.max()), float(err.mean())
