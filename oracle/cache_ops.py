"""KV append and copy-on-write block copy on the pool arrays.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Both functions move values without arithmetic, so they work on any dtype and
the GPU path must match them byte for byte (bf16 pools are handled as their
uint16 bit patterns).  They return new arrays and leave their inputs alone.
"""

import numpy as np


def reshape_and_cache(key, value, slot_mapping, k_cache, v_cache):
    """Write token t's key/value rows ([T, Hkv, D]) into the pool slot that
    ``slot_mapping[t]`` names: block slot // bs, offset slot % bs.

    This is the write of one token's K/V into a given slot of a given
    physical block, and the block/offset split of a running token count by
    the block size, from [KVS] "19.2 KV Cache 系统化管理" §19.2.3 (block
    pool write and block-table append); Fig 19-6 has decode append into the
    partly filled last block.  A negative slot is padding and is skipped (a
    reading: the pages have no padding).  Slots must be unique within a call.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    bs = kc.shape[1]
    for t in range(len(slot_mapping)):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        blk, off = s // bs, s % bs
        kc[blk, off] = key[t]
        vc[blk, off] = value[t]
    return kc, vc


def copy_blocks(k_cache, v_cache, pairs):
    """Copy-on-write block copy: for each (src, dst) pair the whole physical
    block dst (every slot, every head) becomes a copy of block src, in K and V.

    [KVS] §19.2.2 Fig 19-8 (allocate a new block and copy the original
    contents before the table is remapped) and [OS] §四 (copy what is
    needed).  Copying the whole block is the reading taken: it contains what
    is needed and is exact.  Pairs apply in order; callers keep dsts distinct
    and never use a dst as another pair's src, so the order does not matter.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    for src, dst in np.asarray(pairs).reshape(-1, 2):
        kc[int(dst)] = kc[int(src)]
        vc[int(dst)] = vc[int(src)]
    return kc, vc


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs):
    """Preemption by swapping: block pairs[i, 1] of the destination pool
    becomes a copy of block pairs[i, 0] of the source pool (whole blocks, K and
    V).  [KVS] "19.2 KV Cache 系统化管理" §19.2.6 (swap a preempted request's KV
    cache out to CPU memory and back when memory frees up) and [OS] §九.  The
    two pools may differ in block count; every pair must name valid blocks and
    the destination blocks must be distinct."""
    kc = np.array(dst_k, copy=True)
    vc = np.array(dst_v, copy=True)
    for src, dst in np.asarray(pairs).reshape(-1, 2):
        kc[int(dst)] = src_k[int(src)]
        vc[int(dst)] = src_v[int(src)]
    return kc, vc
