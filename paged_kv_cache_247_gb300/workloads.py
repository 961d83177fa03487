"""Seeded synthetic inputs for the paged decode path.

This module only draws inputs: context lengths, a random assignment of
physical block ids to each sequence's logical blocks, and N(0, 1) query, key
and value data.  It holds none of the attention arithmetic and imports neither
the kernels nor the CPU oracle, so both sides can be fed from it.

Shapes follow the workloads the pages discuss: an OPT-13B layer (40 heads of
128, fp16, "800 kilobytes per token"), the grouped-query shape of "The KV cache
is a systems problem" (32 query heads over 8 KV heads of 128), blocks of 16
tokens by default, and variable request lengths.

Structure (lengths, permutations) is drawn with ``numpy.random.default_rng``
on the host; tensor values with a seeded ``torch.Generator`` on the target
device, which keeps multi-GiB caches cheap to build.  Positions a sequence
does not hold and pool blocks no sequence maps can be filled with NaN
(``poison=True``) so that any read of them shows up in the output.
"""

from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


def context_lens_uniform(seed, num_seqs, lo, hi):
    """Integer lengths uniform in [lo, hi]."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=num_seqs).astype(np.int64)


def context_lens_lognormal(seed, num_seqs, median, sigma, lo, hi):
    """round(exp(N(ln median, sigma))) clipped to [lo, hi]."""
    rng = np.random.default_rng(seed)
    x = np.exp(np.log(median) + sigma * rng.standard_normal(num_seqs))
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def _randn(shape, gen, device, dtype):
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    step = 1 << 28  # draw in chunks to bound the fp32 staging buffer
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32).to(dtype)
    return out


@dataclass
class DecodeCase:
    """One batch of decode inputs over a paged cache (all torch tensors)."""
    q: torch.Tensor             # [S, Hq, d]
    k_cache: torch.Tensor       # [NB, Hkv, B, d]
    v_cache: torch.Tensor       # [NB, Hkv, B, d]
    block_tables: torch.Tensor  # int32 [S, max_blocks_per_seq], -1 padded
    context_lens: torch.Tensor  # int32 [S]
    scale: float
    block_size: int
    max_context_len: int
    meta: dict = field(default_factory=dict)

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]


def make_decode_case(seed, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     dtype, context_lens, pool_factor=1.0, pool_blocks=None,
                     max_blocks_per_seq=None, poison=False, device="cpu"):
    """Build a decode batch whose logical blocks sit at random physical ids.

    ``pool_blocks`` (or ``pool_factor`` x the blocks needed) sets the pool
    size; ids are a seeded permutation of the pool handed out in order.
    """
    tdtype = DTYPES[dtype] if isinstance(dtype, str) else dtype
    lens = np.asarray(context_lens, dtype=np.int64)
    per_seq = [int(-(-int(n) // block_size)) for n in lens]
    needed = sum(per_seq)
    if pool_blocks is None:
        pool_blocks = max(1, int(np.ceil(needed * pool_factor)))
    if pool_blocks < needed:
        raise ValueError("pool smaller than the blocks the batch needs")
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max([1] + per_seq)
    rng = np.random.default_rng(seed)
    perm = rng.permutation(pool_blocks)
    tables = np.full((len(lens), max_blocks_per_seq), -1, dtype=np.int32)
    cursor = 0
    for s, nb in enumerate(per_seq):
        tables[s, :nb] = perm[cursor:cursor + nb]
        cursor += nb

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 1000003 + 17)
    q = _randn((len(lens), num_q_heads, head_dim), gen, device, tdtype)
    cache_shape = (pool_blocks, num_kv_heads, block_size, head_dim)
    k_cache = _randn(cache_shape, gen, device, tdtype)
    v_cache = _randn(cache_shape, gen, device, tdtype)

    if poison:
        nan = float("nan")
        used = np.zeros(pool_blocks, dtype=bool)
        used[perm[:cursor]] = True
        unused = torch.from_numpy(np.nonzero(~used)[0]).to(device)
        if unused.numel():
            k_cache[unused] = nan
            v_cache[unused] = nan
        for s, n in enumerate(lens.tolist()):
            nb = per_seq[s]
            held = n - (nb - 1) * block_size if nb else 0
            if nb and held < block_size:
                last = int(tables[s, nb - 1])
                k_cache[last, :, held:, :] = nan
                v_cache[last, :, held:, :] = nan

    return DecodeCase(
        q=q, k_cache=k_cache, v_cache=v_cache,
        block_tables=torch.from_numpy(tables).to(device),
        context_lens=torch.from_numpy(lens.astype(np.int32)).to(device),
        scale=1.0 / float(np.sqrt(head_dim)), block_size=block_size,
        max_context_len=int(lens.max()) if len(lens) else 0,
        meta={"seed": seed, "dtype": dtype if isinstance(dtype, str) else str(dtype),
              "pool_blocks": pool_blocks, "blocks_needed": needed},
    )


def new_tokens(seed, num_tokens, num_kv_heads, head_dim, dtype, device="cpu"):
    """N(0, 1) K and V rows ``[T, Hkv, d]`` for one append."""
    tdtype = DTYPES[dtype] if isinstance(dtype, str) else dtype
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 7919 + 5)
    k = _randn((num_tokens, num_kv_heads, head_dim), gen, device, tdtype)
    v = _randn((num_tokens, num_kv_heads, head_dim), gen, device, tdtype)
    return k, v


def last_position_slots(case):
    """Flat slot (phys * B + offset) of each sequence's last held position.

    A decode step appends its new token there before attending over the
    whole context, so a repeated step rewrites the same slot.
    """
    tables = case.block_tables.cpu().numpy()
    lens = case.context_lens.cpu().numpy()
    B = case.block_size
    slots = np.full(len(lens), -1, dtype=np.int64)
    for s, n in enumerate(lens.tolist()):
        if n > 0:
            slots[s] = int(tables[s, (n - 1) // B]) * B + (n - 1) % B
    return torch.from_numpy(slots)


# ---- the named workloads -------------------------------------------------

TINY = dict(num_seqs=4, num_q_heads=8, num_kv_heads=8, head_dim=64, block_size=16,
            dtype="fp16", ctx_lo=1, ctx_hi=200, pool_blocks=64, seed=0)
OPT13B_LAYER = dict(num_seqs=64, num_q_heads=40, num_kv_heads=40, head_dim=128,
                    block_size=16, dtype="fp16", median=500, sigma=1.0, ctx_lo=16,
                    ctx_hi=2048, pool_factor=1.3, seed=1)
GQA_4K = dict(num_seqs=256, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
              dtype="bf16", ctx=4096, pool_blocks=65536, seed=2)
SHARED_PREFIX = dict(num_prompts=16, samples=8, prompt_lo=100, prompt_hi=700,
                     num_q_heads=40, num_kv_heads=40, head_dim=128, dtype="fp16",
                     block_size=16, steps=200, seed=3)
SWEEP = dict(block_sizes=(8, 16, 32, 64, 128), num_q_heads=32, num_kv_heads=8,
             head_dim=128, dtype="bf16", batches=(8, 64), ctxs=(1024, 8192, 32768), seed=4)


def tiny_decode(device="cpu", poison=True):
    w = TINY
    lens = context_lens_uniform(w["seed"], w["num_seqs"], w["ctx_lo"], w["ctx_hi"])
    return make_decode_case(w["seed"], w["num_seqs"], w["num_q_heads"], w["num_kv_heads"],
                            w["head_dim"], w["block_size"], w["dtype"], lens,
                            pool_blocks=w["pool_blocks"], poison=poison, device=device)


def opt13b_layer_decode(device="cpu", poison=False, num_seqs=None):
    w = OPT13B_LAYER
    n = w["num_seqs"] if num_seqs is None else num_seqs
    lens = context_lens_lognormal(w["seed"], n, w["median"], w["sigma"],
                                  w["ctx_lo"], w["ctx_hi"])
    return make_decode_case(w["seed"], n, w["num_q_heads"], w["num_kv_heads"],
                            w["head_dim"], w["block_size"], w["dtype"], lens,
                            pool_factor=w["pool_factor"], poison=poison, device=device)


def gqa_4k_decode(device="cpu", poison=False, num_seqs=None):
    w = GQA_4K
    n = w["num_seqs"] if num_seqs is None else num_seqs
    lens = np.full(n, w["ctx"], dtype=np.int64)
    # the workload's pool, in proportion when fewer sequences are asked for
    pool = max(w["pool_blocks"] * n // w["num_seqs"], n * w["ctx"] // w["block_size"])
    return make_decode_case(w["seed"], n, w["num_q_heads"], w["num_kv_heads"],
                            w["head_dim"], w["block_size"], w["dtype"], lens,
                            pool_blocks=pool, poison=poison, device=device)


def sweep_decode(block_size, num_seqs, ctx, device="cpu", poison=False):
    w = SWEEP
    lens = np.full(num_seqs, ctx, dtype=np.int64)
    seed = w["seed"] * 100000 + block_size * 1000 + num_seqs * 10 + ctx % 7
    return make_decode_case(seed, num_seqs, w["num_q_heads"], w["num_kv_heads"],
                            w["head_dim"], block_size, w["dtype"], lens,
                            pool_factor=1.0, poison=poison, device=device)


def shared_prefix_prompts():
    """Prompt lengths of the parallel-sampling workload."""
    w = SHARED_PREFIX
    return context_lens_uniform(w["seed"], w["num_prompts"], w["prompt_lo"], w["prompt_hi"])


PREFILL_CHUNKS = dict(num_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                      dtype="bf16", ctx=4096, chunk=2048, seed=5)


def prefill_chunks(device="cpu", num_seqs=None):
    """Chunked prompt processing: each sequence's context is `ctx` tokens, the
    last `chunk` of which are the queries (their K/V already cached)."""
    w = PREFILL_CHUNKS
    n = w["num_seqs"] if num_seqs is None else num_seqs
    lens = np.full(n, w["ctx"], dtype=np.int64)
    case = make_decode_case(w["seed"], n, w["num_q_heads"], w["num_kv_heads"], w["head_dim"],
                            w["block_size"], w["dtype"], lens, pool_factor=1.0, device=device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w["seed"]) * 31 + 7)
    q = _randn((n * w["chunk"], w["num_q_heads"], w["head_dim"]), gen, device, DTYPES[w["dtype"]])
    query_start = torch.arange(0, n + 1, dtype=torch.int32, device=device) * w["chunk"]
    return case, q, query_start
