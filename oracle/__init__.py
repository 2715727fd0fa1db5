"""Float64 CPU oracle for paged KV-cache attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import, call or execute anything under ``oracle/``.  It shares
no code with the CUDA library (no kernels, headers, helpers or tables) and does
not import the ``paged_kv_cache_307_gb300`` package.

Pages this oracle restates (cited by title and section everywhere below):

* [KVS]  "19.2 KV Cache 系统化管理" (paper.xwysyy.cn, llm-fullstack-book 19_2):
  §19.2.2 block tables, Fig 19-6 lifecycle, Fig 19-8 copy-on-write;
  §19.2.3 the simplified implementation (block pool, block table, paged
  attention with an online softmax, and its check against dense attention);
  §19.2.5 prefix sharing (``paged_decode_shared_prefix``).
* [OS]   "LLM 推理引擎的内存管理与调度：PagedAttention、Prefix Cache 与
  Continuous Batching" (zhouzhq2021.github.io): §三 block-table diagram,
  §四 reference counts and copy-on-write, §8.1 chunked prefill.
  §19.2.4 KV cache quantisation (per-token scaled FP8, ``quant.py``).
* [SCH]  "KV Cache、PagedAttention 与调度器" (gongshangzheng.github.io):
  the 13B-per-sequence KV size claim.

Every function works in float64 on exactly widened inputs (bf16 -> f64 and
f32 -> f64 are exact), so the oracle's own rounding is ~1e-16 relative and
negligible against every tolerance the GPU path is held to.

Pinning (see ``tests/test_oracle_*.py``): dense attention is pinned by brute
force with ``math.fsum`` and closed forms; the paged walk, split/merge and
prefill are pinned against dense attention and against each other; the
cache ops against byte-level invariants; the block manager against the worked
examples the pages print.  No function here is "parity unpinned".
"""

from .attention import (  # noqa: F401
    dense_attention,
    brute_force_attention,
    gather_context,
    paged_attention_walk,
    paged_decode,
    decode_partials,
    merge_partials,
    paged_decode_split,
    paged_prefill,
    paged_prefill_varlen,
    shared_prefix_groups,
    paged_decode_shared_prefix,
)
from .cache_ops import reshape_and_cache, copy_blocks, swap_blocks  # noqa: F401
from .quant import (  # noqa: F401
    e4m3_decode,
    e4m3_encode,
    quantize_token,
    dequantize,
    reshape_and_cache_fp8,
    paged_decode_fp8,
)
from .block_manager import BlockPool, BlockTable, BlockExhausted  # noqa: F401
