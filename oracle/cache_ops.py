"""Cache-maintenance operations as plain loops (oracle, test infrastructure).

* ``kv_append`` — each decode step adds one token of K and V per sequence;
  the cache grows token by token ("Only 20.4% of your KV cache held actual
  tokens", section "Why the KV cache is the thing that limits your batch") and
  logical blocks fill left to right (section "The page table, relocated into
  attention").  A token's destination is given as a flat slot
  ``phys_block * B + offset``; a negative slot marks a padding token that is
  skipped.
* ``block_copy`` — copy-on-write at block granularity: allocate a fresh
  block, copy one block's worth of data, decrement the refcount ("Only 20.4%
  ...", section "The part everyone forgets: pages enable sharing, not just
  packing"; "800 kilobytes per token", section "The old answer, imported
  honestly").  The oracle copies whole K and V blocks, pair by pair.

Both operate on copies and return them; they are byte copies, so the result
is exact for any dtype.
"""

import numpy as np


def kv_append(k, v, k_cache, v_cache, slot_mapping):
    """Write token t's K/V (all KV heads) into slot ``slot_mapping[t]``.

    Args:
      k, v: ``[num_tokens, num_kv_heads, head_dim]``.
      k_cache, v_cache: ``[num_blocks, num_kv_heads, block_size, head_dim]``.
      slot_mapping: ``[num_tokens]`` integers; negative entries are skipped.

    Returns new ``(k_cache, v_cache)`` arrays.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    block_size = k_cache.shape[2]
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        block, offset = divmod(int(slot), block_size)
        if block >= k_cache.shape[0]:
            raise IndexError("slot beyond the physical pool")
        k_out[block, :, offset, :] = k[t]
        v_out[block, :, offset, :] = v[t]
    return k_out, v_out


def block_copy(k_cache, v_cache, src_dst_pairs):
    """Copy whole physical blocks ``src -> dst`` in both caches, in pair order."""
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    for src, dst in np.asarray(src_dst_pairs).reshape(-1, 2).tolist():
        k_out[dst] = k_out[src]
        v_out[dst] = v_out[src]
    return k_out, v_out
