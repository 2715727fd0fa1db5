"""ctypes binding to libpa.so: argument marshalling only.

Every step of the path runs in libpa's CUDA kernels; this module turns torch
tensors into raw device pointers and sizes, passes torch's current CUDA
stream, and raises on a non-zero return.  There is no fallback: if libpa.so
is missing the import of this module fails.
"""

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "pa.h")

if not os.path.exists(LIB_PATH):
    raise ImportError("libpa.so is not built (run paged_kv_cache_307_gb300.build.build()): " + LIB_PATH)

lib = ctypes.CDLL(LIB_PATH)

PA_F32, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
DEV_BAD_BLOCK, DEV_BAD_SLOT, DEV_BAD_LEN, DEV_TIMEOUT, DEV_BAD_GROUP = 1, 2, 4, 8, 16

_p, _i, _f, _sz, _i64p, _i32p = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                                 ctypes.c_void_p, ctypes.c_void_p)

lib.pa_reshape_and_cache.argtypes = [_p, _p, _i64p, _i, _p, _p, _i, _i, _i, _i, _i, _p]
lib.pa_reshape_and_cache.restype = _i
lib.pa_decode.argtypes = [_p, _p, _p, _p, _i32p, _i, _i32p, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _i, _p]
lib.pa_decode.restype = _i
lib.pa_decode_noalloc.argtypes = [_p, _p, _p, _p, _i32p, _i, _i32p, _i, _i, _i, _i, _i, _i, _f, _i, _i, _p]
lib.pa_decode_noalloc.restype = _i
lib.pa_decode_shared.argtypes = [_p, _p, _p, _p, _i32p, _i, _i32p, _i, _i32p, _i32p, _i, _i, _i, _i, _i, _i, _f, _i,
                                 _p, _sz, _i, _p]
lib.pa_decode_shared.restype = _i
lib.pa_decode_shared_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i]
lib.pa_decode_shared_workspace_bytes.restype = _sz
lib.pa_decode_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
lib.pa_decode_workspace_bytes.restype = _sz
lib.pa_decode_partition_size.argtypes = [_i, _i, _i, _i, _i, _i, _i]
lib.pa_decode_partition_size.restype = _i
lib.pa_decode_fp8_partition_size.argtypes = [_i, _i, _i, _i, _i, _i, _i]
lib.pa_decode_fp8_partition_size.restype = _i
lib.pa_copy_blocks.argtypes = [_p, _p, _i64p, _i, _i, _i, _i, _i, _i, _p]
lib.pa_copy_blocks.restype = _i
lib.pa_prefill_paged.argtypes = [_p, _p, _i, _p, _p, _i32p, _i, _i32p, _i, _i, _i, _i, _i, _i, _f, _i, _p]
lib.pa_prefill_paged.restype = _i
lib.pa_reshape_and_cache_fp8.argtypes = [_p, _p, _i64p, _i, _p, _p, _p, _p, _i, _i, _i, _i, _i, _p]
lib.pa_reshape_and_cache_fp8.restype = _i
lib.pa_decode_fp8.argtypes = [_p, _p, _p, _p, _p, _p, _i32p, _i, _i32p, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz,
                              _i, _p]
lib.pa_decode_fp8.restype = _i
lib.pa_prefill_varlen.argtypes = [_p, _p, _i32p, _i, _p, _p, _i32p, _i, _i32p, _i, _i, _i, _i, _i, _i, _f, _i, _p]
lib.pa_prefill_varlen.restype = _i
lib.pa_swap_blocks.argtypes = [_p, _p, _i, _p, _p, _i, _i64p, _i, _i, _i, _i, _i, _p]
lib.pa_swap_blocks.restype = _i
lib.pa_last_error.argtypes = []
lib.pa_last_error.restype = _i
lib.pa_strerror.argtypes = [_i]
lib.pa_strerror.restype = ctypes.c_char_p
lib.pa_last_host_error.argtypes = []
lib.pa_last_host_error.restype = ctypes.c_char_p
lib.pa_version.argtypes = []
lib.pa_version.restype = _i
lib.pa_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, _p]
lib.pa_selftest_bounded_wait.restype = _i


class PAError(RuntimeError):
    def __init__(self, code, what):
        extra = lib.pa_last_host_error().decode() if code == -6 else ""
        super().__init__("%s failed: %s (%d)%s" % (what, lib.pa_strerror(code).decode(), code,
                                                   (": " + extra) if extra else ""))
        self.code = code


def declared_functions():
    """Names of the functions include/pa.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", text)))


def _dtype(t):
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.uint8:
        return PA_FP8_E4M3          # e4m3 codes
    raise TypeError("unsupported dtype %s" % t.dtype)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(code, what):
    if code != 0:
        raise PAError(code, what)


def _contig(*ts):
    for t in ts:
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def reshape_and_cache(key, value, slot_mapping, k_cache, v_cache, stream=None):
    """Append key/value [T, Hkv, D] into the pool slots named by slot_mapping."""
    _contig(key, value, slot_mapping, k_cache, v_cache)
    NB, bs, H, D = k_cache.shape
    assert slot_mapping.dtype == torch.int64
    _check(lib.pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(slot_mapping), key.shape[0],
                                    _ptr(k_cache), _ptr(v_cache), NB, bs, H, D, _dtype(k_cache),
                                    _stream(stream)), "pa_reshape_and_cache")


def reshape_and_cache_fp8(key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None):
    """Quantise key/value [T, Hkv, D] (bf16 or fp32) per token into an e4m3
    pool (uint8 codes [NB, bs, Hkv, D]) and its scales (fp32 [NB, bs])."""
    _contig(key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale)
    assert k_cache.dtype == torch.uint8 and k_scale.dtype == torch.float32
    assert slot_mapping.dtype == torch.int64
    NB, bs, H, D = k_cache.shape
    assert k_scale.shape == (NB, bs) and v_scale.shape == (NB, bs)
    _check(lib.pa_reshape_and_cache_fp8(_ptr(key), _ptr(value), _ptr(slot_mapping), key.shape[0],
                                        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), NB, bs, H, D,
                                        _dtype(key), _stream(stream)), "pa_reshape_and_cache_fp8")


def workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks, block_size, partition_size=0):
    return lib.pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks,
                                         block_size, partition_size)


def partition_size(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks, block_size, partition_size=0,
                   fp8=False):
    f = lib.pa_decode_fp8_partition_size if fp8 else lib.pa_decode_partition_size
    return f(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks, block_size, partition_size)


def alloc_workspace(q, k_cache, block_tables, partition_size=0):
    B, Hq, D = q.shape
    n = workspace_bytes(B, Hq, k_cache.shape[2], D, block_tables.shape[1], k_cache.shape[1], partition_size)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)


def decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, partition_size=0,
           workspace=None, stream=None):
    """out[B,Hq,D] = paged decode attention of q[B,Hq,D] over the pool."""
    _contig(out, q, k_cache, v_cache, block_tables, context_lens)
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    if workspace is None:
        workspace = alloc_workspace(q, k_cache, block_tables, partition_size)
    _check(lib.pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                         block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, bs, NB,
                         ctypes.c_float(scale), partition_size, _ptr(workspace), workspace.numel(),
                         _dtype(q), _stream(stream)), "pa_decode")
    return out


def shared_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks, block_size,
                           partition_size=0, num_groups=1):
    return lib.pa_decode_shared_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks,
                                                block_size, partition_size, num_groups)


def alloc_shared_workspace(q, k_cache, block_tables, num_groups, partition_size=0):
    B, Hq, D = q.shape
    n = shared_workspace_bytes(B, Hq, k_cache.shape[2], D, block_tables.shape[1], k_cache.shape[1],
                               partition_size, num_groups)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)


def decode_shared(out, q, k_cache, v_cache, block_tables, context_lens, group_start, shared_blocks, scale,
                  partition_size=0, workspace=None, stream=None):
    """out[B,Hq,D] = paged decode attention of q over the pool, reading the
    shared prompt blocks of each group (sequences group_start[g] ..
    group_start[g+1]-1 share their first shared_blocks[g] table entries)
    once for the whole group."""
    _contig(out, q, k_cache, v_cache, block_tables, context_lens, group_start, shared_blocks)
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert group_start.dtype == torch.int32 and shared_blocks.dtype == torch.int32
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    ng = shared_blocks.shape[0]
    assert group_start.shape[0] == ng + 1
    if workspace is None:
        workspace = alloc_shared_workspace(q, k_cache, block_tables, ng, partition_size)
    _check(lib.pa_decode_shared(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                block_tables.shape[1], _ptr(context_lens), B, _ptr(group_start),
                                _ptr(shared_blocks), ng, Hq, Hkv, D, bs, NB, ctypes.c_float(scale), partition_size,
                                _ptr(workspace), workspace.numel(), _dtype(q), _stream(stream)), "pa_decode_shared")
    return out


def decode_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
               partition_size=0, workspace=None, stream=None):
    """out[B,Hq,D] (bf16) = paged decode attention of q over an e4m3 pool."""
    _contig(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens)
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert k_cache.dtype == torch.uint8 and k_scale.dtype == torch.float32
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    if workspace is None:
        workspace = alloc_workspace(q, k_cache, block_tables, partition_size)
    _check(lib.pa_decode_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                             _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, bs, NB,
                             ctypes.c_float(scale), partition_size, _ptr(workspace), workspace.numel(), _dtype(q),
                             _stream(stream)), "pa_decode_fp8")
    return out


def copy_blocks_fp8(k_cache, v_cache, k_scale, v_scale, pairs, stream=None):
    """Copy-on-write for an e4m3 pool: the codes, then the scale rows."""
    copy_blocks(k_cache, v_cache, pairs, stream)
    NB, bs = k_scale.shape
    copy_blocks(k_scale.view(NB, bs, 1, 1), v_scale.view(NB, bs, 1, 1), pairs, stream)


def copy_blocks(k_cache, v_cache, pairs, stream=None):
    """Copy-on-write: block pairs[i,1] becomes a copy of block pairs[i,0]."""
    _contig(k_cache, v_cache, pairs)
    assert pairs.dtype == torch.int64
    NB, bs, H, D = k_cache.shape
    _check(lib.pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0], NB, bs, H, D,
                              _dtype(k_cache), _stream(stream)), "pa_copy_blocks")


def prefill(out, q, k_cache, v_cache, block_tables, context_lens, scale, stream=None):
    """Causal chunked-prefill tile: q/out [B, Tq, Hq, D], the last Tq tokens
    of each context."""
    _contig(out, q, k_cache, v_cache, block_tables, context_lens)
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    B, Tq, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    _check(lib.pa_prefill_paged(_ptr(out), _ptr(q), Tq, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, bs, NB,
                                ctypes.c_float(scale), _dtype(q), _stream(stream)), "pa_prefill_paged")
    return out


def prefill_varlen(out, q, query_start, k_cache, v_cache, block_tables, context_lens, scale, stream=None):
    """Mixed round: q/out [rows, Hq, D], sequence b's rows are
    query_start[b]..query_start[b+1]-1, the last tokens of its context."""
    _contig(out, q, query_start, k_cache, v_cache, block_tables, context_lens)
    assert query_start.dtype == torch.int32 and block_tables.dtype == torch.int32
    rows, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    B = context_lens.shape[0]
    _check(lib.pa_prefill_varlen(_ptr(out), _ptr(q), _ptr(query_start), rows, _ptr(k_cache), _ptr(v_cache),
                                 _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, bs,
                                 NB, ctypes.c_float(scale), _dtype(q), _stream(stream)), "pa_prefill_varlen")
    return out


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs, stream=None):
    """Block pairs[i,1] of (dst_k, dst_v) becomes a copy of block pairs[i,0]
    of (src_k, src_v).  Either pool may be pinned host memory."""
    _contig(dst_k, dst_v, src_k, src_v, pairs)
    assert pairs.dtype == torch.int64 and pairs.is_cuda
    assert dst_k.shape[1:] == src_k.shape[1:] and dst_k.dtype == src_k.dtype
    _, bs, H, D = dst_k.shape
    _check(lib.pa_swap_blocks(_ptr(dst_k), _ptr(dst_v), dst_k.shape[0], _ptr(src_k), _ptr(src_v), src_k.shape[0],
                              _ptr(pairs), pairs.shape[0], bs, H, D, _dtype(dst_k), _stream(stream)),
           "pa_swap_blocks")


def selftest_bounded_wait(limit_ns, stream=None):
    """Launch the bounded-wait health check (one warp waits on an mbarrier
    nothing arrives at, giving up after ``limit_ns``)."""
    _check(lib.pa_selftest_bounded_wait(int(limit_ns), _stream(stream)), "pa_selftest_bounded_wait")


def last_error():
    """Sticky device-detected condition bits (and clear them); synchronises."""
    code = lib.pa_last_error()
    if code < 0:
        raise PAError(code, "pa_last_error")
    return code
