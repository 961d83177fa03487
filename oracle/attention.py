"""Paged single-query decode attention, fp64 (oracle, test infrastructure).

What it computes ("Only 20.4% of your KV cache held actual tokens", section
"The page table, relocated into attention"): the attention kernel follows
each sequence's block table and gathers keys and values from non-contiguous
physical blocks instead of one flat tensor.  Paging changes where K and V
live, not the result, so the oracle first rebuilds each sequence's contiguous
K and V by walking its table and then applies the plain definition of one
decode step of scaled dot-product attention:

    out[s, h] = softmax(scale * K_s[:, kvh] @ q[s, h]) @ V_s[:, kvh]

Readings taken where the pages are silent (each is listed with its reason in
the design notes):

* cache layout ``[num_blocks, num_kv_heads, block_size, head_dim]``, K and V
  in separate arrays; token position t of a sequence sits in logical block
  t // B at offset t % B (logical blocks fill left to right);
* query head h reads KV head h // G with G = Hq / Hkv (contiguous groups:
  "The KV cache is a systems problem", section "Calculate bytes per token
  before choosing a batch", notes that groups of query heads share K and V);
* the step's new token is already in the cache, so every one of the
  ``context_lens[s]`` positions is attended to (no causal mask);
* positions at or beyond ``context_lens[s]`` are never read;
* a sequence with ``context_lens[s] == 0`` has an all-zero output.

Inputs may be any numpy float arrays (fp16, fp32, fp64); they are widened to
fp64 exactly before any arithmetic.  bf16 data is widened by the caller
(numpy has no bf16 type).
"""

import numpy as np


def gather_sequence_kv(k_cache, v_cache, block_table_row, context_len):
    """Follow one sequence's block table; return contiguous K, V in fp64.

    Returns two arrays of shape ``[context_len, num_kv_heads, head_dim]``.
    Only the first ceil(context_len / B) table entries are read, and only the
    first ``context_len`` positions are kept.
    """
    block_size = k_cache.shape[2]
    n_blocks = -(-int(context_len) // block_size)
    ids = np.asarray(block_table_row[:n_blocks], dtype=np.int64)
    if n_blocks and (ids.min() < 0 or ids.max() >= k_cache.shape[0]):
        raise IndexError("block table entry outside the physical pool")
    # [n_blocks, Hkv, B, d] -> [n_blocks, B, Hkv, d] -> [n_blocks*B, Hkv, d]
    k = np.asarray(k_cache[ids], dtype=np.float64).transpose(0, 2, 1, 3)
    v = np.asarray(v_cache[ids], dtype=np.float64).transpose(0, 2, 1, 3)
    k = k.reshape(n_blocks * block_size, k_cache.shape[1], k_cache.shape[3])
    v = v.reshape(n_blocks * block_size, v_cache.shape[1], v_cache.shape[3])
    return k[:context_len], v[:context_len]


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale,
                           pairs=None):
    """Reference decode attention over a paged cache, in fp64.

    Args:
      q: ``[num_seqs, num_q_heads, head_dim]``.
      k_cache, v_cache: ``[num_blocks, num_kv_heads, block_size, head_dim]``.
      block_tables: ``[num_seqs, max_blocks_per_seq]`` integer physical ids.
      context_lens: ``[num_seqs]`` integer token counts.
      scale: softmax temperature applied to q.k.
      pairs: optional iterable of ``(s, h)``; when given, only those outputs
        are computed (the rest of the returned array stays NaN) so that large
        workloads can be checked on a sample.

    Returns:
      ``[num_seqs, num_q_heads, head_dim]`` float64.
    """
    q = np.asarray(q)
    num_seqs, num_q_heads, head_dim = q.shape
    num_kv_heads = k_cache.shape[1]
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = num_q_heads // num_kv_heads
    out = np.full((num_seqs, num_q_heads, head_dim), np.nan)
    if pairs is None:
        wanted = {s: list(range(num_q_heads)) for s in range(num_seqs)}
    else:
        wanted = {}
        for s, h in pairs:
            wanted.setdefault(int(s), []).append(int(h))
    for s, heads in wanted.items():
        n = int(context_lens[s])
        if n == 0:
            out[s, heads] = 0.0
            continue
        k_seq, v_seq = gather_sequence_kv(k_cache, v_cache, block_tables[s], n)
        for h in heads:
            kvh = h // group
            logits = scale * (k_seq[:, kvh, :] @ q[s, h].astype(np.float64))
            weights = np.exp(logits - logits.max())
            weights /= weights.sum()
            out[s, h] = weights @ v_seq[:, kvh, :]
    return out


def paged_prefill_attention(q, k_cache, v_cache, block_tables, context_lens, query_start, scale):
    """Multi-query (chunked prompt) attention over a paged cache, in fp64.

    Sequence s contributes ``L_s = query_start[s+1] - query_start[s]`` query
    rows ``q[query_start[s] : query_start[s+1]]``: the last L_s positions of
    its context, whose K/V are already in the cache.  Query j sits at position
    ``p = context_lens[s] - L_s + j`` and attends to positions ``0 .. p``
    (causal), through the block table as in decode.  This is prompt processing
    in chunks ("The KV cache is a systems problem", section "Memory savings
    change the scheduling question": prompt chunks share the step budget with
    decoding); with L_s = 1 it is one decode step.

    Args:
      q: ``[total_queries, num_q_heads, head_dim]``.
      query_start: ``[num_seqs + 1]`` non-decreasing offsets, ``query_start[0] = 0``.
      context_lens: ``[num_seqs]`` with ``context_lens[s] >= L_s``.
    Returns ``[total_queries, num_q_heads, head_dim]`` float64.
    """
    q = np.asarray(q)
    total, num_q_heads, head_dim = q.shape
    group = num_q_heads // k_cache.shape[1]
    out = np.zeros((total, num_q_heads, head_dim))
    for s in range(len(context_lens)):
        q0, q1 = int(query_start[s]), int(query_start[s + 1])
        n_q, ctx = q1 - q0, int(context_lens[s])
        if n_q == 0:
            continue
        if n_q > ctx:
            raise ValueError("a chunk cannot be longer than its context")
        k_seq, v_seq = gather_sequence_kv(k_cache, v_cache, block_tables[s], ctx)
        for j in range(n_q):
            pos = ctx - n_q + j
            for h in range(num_q_heads):
                kvh = h // group
                logits = scale * (k_seq[:pos + 1, kvh, :] @ q[q0 + j, h].astype(np.float64))
                weights = np.exp(logits - logits.max())
                weights /= weights.sum()
                out[q0 + j, h] = weights @ v_seq[:pos + 1, kvh, :]
    return out
