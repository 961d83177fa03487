"""Closed-form KV-cache byte and block arithmetic (oracle, test infrastructure).

* Bytes per token: "The KV cache is a systems problem", section "Calculate
  bytes per token before choosing a batch" gives the formula
  2 (keys and values) x layers x KV heads x head dimension x element bytes.
  "Only 20.4% of your KV cache held actual tokens", section "Why the KV cache
  is the thing that limits your batch" applies the same product to OPT-13B
  with the hidden size (40 heads x 128) in place of KV heads x head dim.
* Blocks: a sequence occupies ceil(n / B) fixed-size blocks, the last one
  partially filled ("Only 20.4% ...", section "The page table, relocated into
  attention": logical blocks are filled left to right and a new block is taken
  only when all earlier ones are full).
"""


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, element_bytes: int) -> int:
    """K and V bytes one token adds to the cache, over all layers."""
    return 2 * layers * kv_heads * head_dim * element_bytes


def blocks_for_tokens(num_tokens: int, block_size: int) -> int:
    """Physical blocks a sequence of ``num_tokens`` positions holds.

    Blocks fill left to right and a fresh block is taken only once every
    earlier block is full, so the count is the ceiling of n / B.
    """
    if num_tokens < 0 or block_size <= 0:
        raise ValueError("num_tokens must be >= 0 and block_size > 0")
    return -(-num_tokens // block_size)


def unused_tail_slots(num_tokens: int, block_size: int) -> int:
    """Unfilled token positions in the sequence's last block."""
    return blocks_for_tokens(num_tokens, block_size) * block_size - num_tokens
