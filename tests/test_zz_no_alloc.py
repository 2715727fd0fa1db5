"""pa_decode_noalloc: decode for callers that cannot allocate device memory
when they call in (a plug-in whose host engine owns all device allocations,
or a latency-critical path that cannot risk an allocation call that may
synchronise the device).  It uses a scratch array built into the library
instead of a workspace.  These tests call it through the C ABI and check it
bit for bit against pa_decode with a caller-provided workspace, on two
different calls in a row (the array keeps the previous call's contents,
which must not leak into the next result).  This file sorts last so that a
run stopping at the first failure has already run every other test."""

import ctypes

import pytest
import torch

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


def _noalloc(pa, out, c, partition):
    s = torch.cuda.current_stream()
    NB, bs, Hkv, D = c.k_cache.shape
    B, Hq, _ = c.q.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return pa.lib.pa_decode_noalloc(p(out), p(c.q), p(c.k_cache), p(c.v_cache), p(c.block_tables),
                                    c.block_tables.shape[1], p(c.context_lens), B, Hq, Hkv, D, bs, NB,
                                    ctypes.c_float(c.scale), partition, pa.PA_BF16, ctypes.c_void_p(s.cuda_stream))


def _reference(pa, c, partition):
    ref = torch.empty_like(c.q)
    pa.decode(ref, c.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, c.scale, partition_size=partition)
    torch.cuda.synchronize()
    return ref


# Two calls in a row on different cases: the second has fewer partitions per
# sequence than the first left in the array, so stale partials from the first
# call would change its result if they leaked into the merge.
@pytest.mark.parametrize("first,second", [(("c4", 0), ("c3", 64)), (("c2", 16), ("c2", 0)), (("c3", 64), ("c4", 512))])
def test_noalloc_matches_workspace_decode_on_two_calls(pa, first, second):
    for name, partition in (first, second):
        c = W.decode_case(name, small=True, device="cuda")
        pa.reshape_and_cache(c.key, c.value, c.slot_mapping, c.k_cache, c.v_cache)
        ref = _reference(pa, c, partition)
        out = torch.full_like(c.q, float("nan"))
        assert _noalloc(pa, out, c, partition) == 0
        torch.cuda.synchronize()
        assert pa.last_error() == 0
        # the same kernels over the same partitions: bit-identical
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (name, partition)
        assert_close(f64(out), f64(ref), "bf16")


def test_noalloc_rejects_sizes_beyond_its_scratch(pa):
    # full-size GQA workload: its split-K scratch is far above the built-in limit
    B, Hq, Hkv, D, maxb, bs = 256, 32, 8, 128, 2048, 16
    need = pa.workspace_bytes(B, Hq, Hkv, D, maxb, bs, 0)
    assert need > 32 * 1024 * 1024
    fake = torch.empty(16, device="cuda")
    p = ctypes.c_void_p(fake.data_ptr())
    rc = pa.lib.pa_decode_noalloc(p, p, p, p, p, maxb, p, B, Hq, Hkv, D, bs, 10, ctypes.c_float(1.0), 0,
                                  pa.PA_BF16, ctypes.c_void_p(0))
    assert rc == -5
    assert b"scratch" in pa.lib.pa_last_host_error()
