"""Paged KV-cache decode for GB300 (sm_103a): the hot path of PagedAttention.

Device calls (hand-written CUDA behind the C ABI of ``libpagedkv.so``):

* :func:`paged_attn_decode` — single-query decode attention walking each
  sequence's block table, with split-context partitions and GQA grouping
  (grouped heads and small single-head calls on the tcgen05 tensor cores,
  single-head groups with many (sequence, head) pairs on the CUDA cores);
* :func:`kv_append` — scatter of each step's new K/V into its slot;
* :func:`paged_attn_decode_append` — both in one launch (the new token is
  written to its slot and used directly);
* :func:`block_copy` — block-granular copy-on-write;
* :func:`paged_attn_prefill` — causal multi-query (chunked prompt) attention
  over the paged cache on the tcgen05 tensor cores.

Host: :class:`BlockAllocator`, the refcounted block allocator that decides
slots and copy-on-write pairs.  The library is loaded on first use and there
is no fallback: a missing library raises.
"""

from ._lib import PagedKVError, load as load_library  # noqa: F401
from .ops import (  # noqa: F401
    paged_attn_decode,
    paged_attn_decode_append,
    paged_attn_prefill,
    contiguous_attn_decode,
    kv_append,
    block_copy,
    check_copy_pairs,
    device_status,
    debug_wait_timeout,
    decode_workspace_size,
    decode_partition_size,
    decode_uses_tensor_cores,
    set_decode_path,
)
from .allocator import BlockAllocator, OutOfBlocks  # noqa: F401
