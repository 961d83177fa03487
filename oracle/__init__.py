"""CPU oracle for the paged KV-cache decode path — TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct restatement of what the paged
decode path computes, in float64 numpy (plus pure-Python loops for the block
allocator).  It exists so that the CUDA kernels can be checked against
something written straight from the source pages.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  The product package (``paged_kv_cache_247_gb300``) never imports it and
shares no code, constants or helpers with it.

Sources (cited by page title and section throughout):

* "800 kilobytes per token" (shashforge.dev) — byte arithmetic, blocks of
  sixteen, copy-on-write.
* "Only 20.4% of your KV cache held actual tokens: how PagedAttention put a
  page table inside the attention kernel" (blog.teqners.com) — block table,
  on-demand allocation, refcounts, the kernel that follows the table.
* "The KV cache is a systems problem" (rsw.lol) — bytes-per-token formula,
  the 33-token example, ownership rules for shared prefixes.

Modules:

* :mod:`oracle.facts` — closed-form byte and block counts.
* :mod:`oracle.attention` — paged single-query decode attention and paged
  multi-query (chunked prompt) attention in fp64.
* :mod:`oracle.cache_ops` — the slot scatter (append) and block copy.
* :mod:`oracle.allocator` — a pure-Python refcounted block allocator model.

Every function here is pinned by ``tests/test_oracle_pins.py`` and
``tests/test_oracle_allocator.py`` to facts and invariants that do not come
from the oracle itself; no function is "parity unpinned".
"""

from .facts import (  # noqa: F401
    kv_bytes_per_token,
    blocks_for_tokens,
    unused_tail_slots,
)
from .attention import (  # noqa: F401
    paged_decode_attention, paged_prefill_attention, gather_sequence_kv)
from .cache_ops import kv_append, block_copy  # noqa: F401
from .allocator import OracleAllocator, OracleOutOfBlocks  # noqa: F401
