"""The C-ABI library loads on a machine without a GPU and exports every
function include/pa.h declares; host-side argument checks need no GPU."""

import ctypes

import pytest

from paged_kv_cache_307_gb300 import build as B


@pytest.fixture(scope="module")
def pa():
    B.build()
    from paged_kv_cache_307_gb300 import _lib
    return _lib


def test_every_declared_symbol_is_exported(pa):
    names = pa.declared_functions()
    assert {"pa_decode", "pa_reshape_and_cache", "pa_copy_blocks", "pa_last_error"} <= set(names)
    for n in names:
        assert hasattr(pa.lib, n), n


def test_version_and_error_text(pa):
    assert pa.lib.pa_version() >= 100
    assert b"aligned" in pa.lib.pa_strerror(-4)
    assert b"block" in pa.lib.pa_strerror(1)


def test_workspace_and_partition_arithmetic(pa):
    # 64 seqs x 32 heads, 128 blocks of 16 -> 2048 tokens -> 8 partitions of 256
    assert pa.partition_size(64, 32, 32, 128, 128, 16, 0) == 256
    rows = 64 * 32 * 8
    ml = (rows * 8 + 255) // 256 * 256
    # (m, l) pairs, partial outputs, then 256 bytes for the work-item counter
    assert pa.workspace_bytes(64, 32, 32, 128, 128, 16, 0) == ml + rows * 128 * 4 + 256
    assert pa.workspace_bytes(64, 32, 32, 128, 128, 16, -1) == 0          # never split
    assert pa.partition_size(1, 8, 8, 32, 3, 4, 0) == 12                   # fits one partition
    assert pa.partition_size(1, 8, 8, 32, 3, 4, 6) == -2                   # not a block multiple
    # e4m3 pools: 512-token partitions for MHA, the grouped-query rule of pa_decode
    assert pa.partition_size(64, 32, 32, 128, 128, 16, 0, fp8=True) == 512
    # grouped queries: 2048 while the batch gives >= 912 unsplit items
    # (num_seqs * ceil(Hkv / 4)), else finer: 2048 * 128 items / 2432 = 107 -> 256
    assert pa.partition_size(64, 32, 8, 128, 128, 16, 0, fp8=True) == 256
    assert pa.partition_size(64, 32, 8, 128, 128, 16, 0) == 256
    assert pa.partition_size(456, 32, 8, 128, 128, 16, 0) == 2048               # 912 items
    assert pa.partition_size(455, 32, 8, 128, 128, 16, 0) == 512                # 2048 * 910 / 2432 = 766
    assert pa.partition_size(256, 32, 8, 128, 2048, 16, 0) == 2048             # 32768 * 512 / 2432 = 6898
    assert pa.partition_size(256, 32, 8, 128, 80, 16, 0) == 256                # 1280 * 512 / 2432 = 269
    assert pa.partition_size(512, 32, 8, 128, 81, 16, 0) == 1296               # 1024 items: no split
    assert pa.partition_size(64, 32, 32, 128, 128, 16, 64, fp8=True) == 64
    assert pa.partition_size(1, 8, 8, 32, 3, 4, 0, fp8=True) == 12
    # shared-prefix decode: per (sequence, head) slots for ceil(max_ctx / 1024) + 1
    # partitions (1024-token shared partitions), a partition count per sequence,
    # never less than pa_decode's
    rows = 512 * 32 * (-(-1280 // 1024) + 1)
    # partition counts (B ints) and the item counter, rounded to 256 bytes: (512 + 1) * 4 -> 2304
    assert pa.shared_workspace_bytes(512, 32, 8, 128, 80, 16, 0, 64) == 2304 + rows * 8 + rows * 128 * 4
    assert pa.shared_workspace_bytes(64, 32, 32, 128, 128, 16, 0, 8) >= pa.workspace_bytes(64, 32, 32, 128, 128, 16)
    # shapes the shared path does not take fall back to pa_decode's workspace
    assert pa.shared_workspace_bytes(4, 256, 4, 128, 80, 16, 0, 1) == pa.workspace_bytes(4, 256, 4, 128, 80, 16, 0)
    assert pa.shared_workspace_bytes(4, 64, 4, 64, 80, 16, 0, 1) == pa.workspace_bytes(4, 64, 4, 64, 80, 16, 0)


def test_host_side_rejections_launch_nothing(pa):
    L = pa.lib
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: every call below is rejected first
    # head_dim 48 unsupported
    assert L.pa_decode(fake, fake, fake, fake, fake, 4, fake, 2, 8, 8, 48, 16, 10, 1.0, 0, null, 0, 1, null) == -2
    # heads not a multiple of kv heads
    assert L.pa_decode(fake, fake, fake, fake, fake, 4, fake, 2, 6, 4, 64, 16, 10, 1.0, 0, null, 0, 1, null) == -2
    # block size 12 unsupported
    assert L.pa_copy_blocks(fake, fake, fake, 3, 10, 12, 2, 64, 1, null) == -2
    # unknown dtype
    assert L.pa_reshape_and_cache(fake, fake, fake, 3, fake, fake, 10, 16, 2, 64, 7, null) == -3
    # null pool
    assert L.pa_copy_blocks(null, fake, fake, 3, 10, 16, 2, 64, 1, null) == -1
    # misaligned pointer
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert L.pa_reshape_and_cache(fake, odd, fake, 3, fake, fake, 10, 16, 2, 64, 1, null) == -4
    # split needed but no workspace (4 partitions)
    assert L.pa_decode(fake, fake, fake, fake, fake, 128, fake, 2, 8, 8, 128, 16, 10, 1.0, 512, null, 0, 1,
                       null) == -5
    # prefill: head_dim 64 and non-positive scale are rejected
    assert L.pa_prefill_paged(fake, fake, 16, fake, fake, fake, 8, fake, 2, 8, 8, 64, 16, 10, 1.0, 1, null) == -2
    assert L.pa_prefill_paged(fake, fake, 16, fake, fake, fake, 8, fake, 2, 8, 8, 128, 16, 10, -1.0, 1, null) == -2
    # bounded-wait health check: a limit of 0 or above 2 s is rejected
    assert L.pa_selftest_bounded_wait(0, null) == -2
    assert L.pa_selftest_bounded_wait(3_000_000_000, null) == -2
    # swap: null source pool, misaligned destination, unsupported block size
    assert L.pa_swap_blocks(fake, fake, 4, null, fake, 10, fake, 2, 16, 2, 64, 1, null) == -1
    assert L.pa_swap_blocks(odd, fake, 4, fake, fake, 10, fake, 2, 16, 2, 64, 1, null) == -4
    assert L.pa_swap_blocks(fake, fake, 4, fake, fake, 10, fake, 2, 12, 2, 64, 1, null) == -2
    # e4m3 pools: fp32 queries are not supported, scales are required and aligned
    assert L.pa_decode_fp8(fake, fake, fake, fake, fake, fake, fake, 4, fake, 2, 8, 8, 128, 16, 10, 1.0, 0,
                           null, 0, 0, null) == -3
    assert L.pa_decode_fp8(fake, fake, fake, fake, null, fake, fake, 4, fake, 2, 8, 8, 128, 16, 10, 1.0, 0,
                           null, 0, 1, null) == -1
    assert L.pa_decode_fp8(fake, fake, fake, fake, odd, fake, fake, 4, fake, 2, 8, 8, 128, 16, 10, 1.0, 0,
                           null, 0, 1, null) == -4
    assert L.pa_reshape_and_cache_fp8(fake, fake, fake, 3, fake, fake, null, fake, 10, 16, 2, 64, 1, null) == -1
    assert L.pa_reshape_and_cache_fp8(fake, fake, fake, 3, fake, fake, fake, fake, 10, 16, 2, 64, 2, null) == -3
    # copies accept e4m3 pools and the [NB, bs, 1, 1] fp32 scale rows, not blocks of a partial chunk
    assert L.pa_copy_blocks(fake, fake, fake, 0, 10, 16, 1, 1, 0, null) == 0
    assert L.pa_copy_blocks(fake, fake, fake, 0, 10, 4, 1, 1, 2, null) == -2      # 4 bytes per block
    # shared-prefix decode: a descriptor is required when groups are named; the
    # workspace is checked before anything is launched; partitions are whole blocks
    assert L.pa_decode_shared(fake, fake, fake, fake, fake, 80, fake, 16, null, fake, 2, 32, 8, 128, 16, 10, 1.0,
                              0, null, 0, 1, null) == -1
    assert L.pa_decode_shared(fake, fake, fake, fake, fake, 80, fake, 16, fake, fake, 2, 32, 8, 128, 16, 10, 1.0,
                              0, null, 0, 1, null) == -5
    assert L.pa_decode_shared(fake, fake, fake, fake, fake, 80, fake, 16, fake, fake, 2, 32, 8, 128, 16, 10, 1.0,
                              24, null, 0, 1, null) == -2
    assert L.pa_decode_shared(fake, fake, fake, fake, fake, 80, fake, 16, fake, fake, -1, 32, 8, 128, 16, 10, 1.0,
                              0, null, 0, 1, null) == -2
    # empty inputs are a no-op success
    assert L.pa_copy_blocks(null, null, null, 0, 10, 16, 2, 64, 1, null) == 0
    assert L.pa_swap_blocks(null, null, 4, null, null, 10, null, 0, 16, 2, 64, 1, null) == 0
