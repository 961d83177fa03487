"""GPU parity of the tensor-core chunked-prompt (multi-query) attention.

Each sequence's last L_s positions attend causally over its paged context;
the kernel runs on tcgen05 with the softmax weights rounded to the operand
type before P.V, so results are compared with the fp64 oracle under the
same tolerances as decode.  Cases cover whole prompts, partial chunks, one
query (which must agree with decode), several 128-row query tiles and
128-key tiles, ragged and NaN-poisoned block tails, every block size and
grouped heads."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import _lib
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import TOL, assert_within_tol, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status(lib, cuda_device):
    pkv.device_status(clear=True)
    yield
    assert pkv.device_status(clear=True) == 0


def _run(case, chunks, seed):
    dev = case.q.device
    S, Hq, D = case.q.shape
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    gen = torch.Generator(device=dev).manual_seed(seed)
    q = torch.randn((int(qs[-1]), Hq, D), generator=gen, device=dev).to(case.q.dtype)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attn_prefill(out, q, torch.from_numpy(qs).to(dev), case.k_cache, case.v_cache,
                           case.block_tables, case.context_lens, case.scale,
                           case.max_context_len, int(max(chunks)))
    torch.cuda.synchronize()
    ref = oracle.paged_prefill_attention(to_f64(q), to_f64(case.k_cache), to_f64(case.v_cache),
                                         case.block_tables.cpu().numpy(),
                                         case.context_lens.cpu().numpy(), qs, case.scale)
    return q, out, ref, qs


@pytest.mark.parametrize("dtype,hq,hkv,D,B", [
    ("bf16", 8, 8, 128, 16), ("fp16", 8, 8, 128, 16), ("bf16", 32, 8, 128, 16),
    ("fp16", 16, 2, 64, 8), ("bf16", 12, 4, 128, 128), ("bf16", 6, 2, 64, 32),
    ("fp16", 4, 4, 64, 64), ("bf16", 32, 1, 128, 16), ("fp16", 24, 4, 64, 32),
    # groups of 5 (padded to 8 rows a query), 64 and 128 (one query per row tile):
    # each row tile's Q is one copy of G' heads x 128 / G' queries
    ("bf16", 10, 2, 128, 32), ("bf16", 64, 1, 64, 16), ("fp16", 128, 1, 128, 16)])
def test_prefill_matches_oracle(cuda_device, dtype, hq, hkv, D, B):
    lens = [1, 17, 130, 300, 64, 257]
    chunks = [1, 17, 130, 45, 1, 200]   # whole prompt, partial chunks, single queries
    case = W.make_decode_case(hq * 3 + B, len(lens), hq, hkv, D, B, dtype, lens, pool_factor=1.3,
                              poison=True, device=cuda_device)
    q, out, ref, qs = _run(case, chunks, seed=B + hq)
    assert_within_tol(out, ref, W.DTYPES[dtype], f"prefill {dtype} {hq}/{hkv} D={D} B={B}")


def test_single_query_agrees_with_decode(cuda_device):
    lens = [5, 700, 1500, 33]
    case = W.make_decode_case(77, len(lens), 32, 8, 128, 16, "bf16", lens, pool_factor=1.2,
                              device=cuda_device)
    q, out, ref, qs = _run(case, [1] * len(lens), seed=3)
    dec = torch.empty_like(q)
    pkv.paged_attn_decode(dec, q, case.k_cache, case.v_cache, case.block_tables,
                          case.context_lens, case.scale, case.max_context_len)
    torch.cuda.synchronize()
    assert_within_tol(out, ref, torch.bfloat16, "prefill L=1")
    assert_within_tol(dec, ref, torch.bfloat16, "decode")


def test_long_prompt_chunks(cuda_device):
    """A 2,000-token prompt processed as chunks of 512 against a growing context."""
    case = W.make_decode_case(5, 1, 32, 8, 128, 16, "bf16", [2000], pool_factor=1.0,
                              device=cuda_device)
    for done in (512, 1024, 1536, 2000):
        chunk = min(512, done) if done < 2000 else 2000 - 1536
        case.context_lens.fill_(done)
        q, out, ref, qs = _run(case, [chunk], seed=done)
        assert_within_tol(out, ref, torch.bfloat16, f"chunk ending at {done}")


def test_prefill_full_size_sampled(cuda_device):
    """The bench's workload (8 sequences x 2,048-query chunks over 4,096 tokens,
    32 q / 8 kv heads, D = 128, B = 16, bf16) in the bench's launch, checked on
    sampled outputs: causal attention of the query at position p is decode
    attention over positions 0..p, which the oracle computes for one query
    from that sequence's own blocks."""
    case, q, qs = W.prefill_chunks(device=cuda_device)
    w = W.PREFILL_CHUNKS
    out = torch.full_like(q, float("nan"))
    pkv.paged_attn_prefill(out, q, qs, case.k_cache, case.v_cache, case.block_tables,
                           case.context_lens, case.scale, case.max_context_len, w["chunk"])
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    S, L, B = w["num_seqs"], w["chunk"], w["block_size"]
    rng = np.random.default_rng(11)
    # the first and last query of a sequence, both row tiles of a CTA, and random ones
    picks = [(0, 0), (S - 1, L - 1), (1, 63), (2, 64), (3, 1000)]
    picks += [(int(rng.integers(S)), int(rng.integers(L))) for _ in range(7)]
    tables = case.block_tables.cpu().numpy()
    for s, j in picks:
        p = int(case.context_lens[s]) - L + j
        nb = -(-(p + 1) // B)
        blocks = torch.from_numpy(tables[s, :nb].astype(np.int64)).to(cuda_device)
        k_sub, v_sub = to_f64(case.k_cache[blocks]), to_f64(case.v_cache[blocks])
        row = int(qs[s]) + j
        ref = oracle.paged_decode_attention(to_f64(q[row:row + 1]), k_sub, v_sub,
                                            np.arange(nb)[None, :], np.array([p + 1]), case.scale)
        assert_within_tol(out[row:row + 1], ref, torch.bfloat16, f"prefill seq {s} query {j}")


def test_prefill_long_context_sampled(cuda_device):
    """Chunks at the end of 32k-token contexts: 256 key tiles per row tile, so
    the K and V rings wrap around many times, with a chunk that ends in a
    partial row tile; checked on sampled queries against decode attention
    over each query's visible prefix."""
    lens = [32768, 30001]
    chunks = [192, 77]
    case = W.make_decode_case(31, len(lens), 32, 8, 128, 16, "bf16", lens, pool_factor=1.0,
                              device=cuda_device)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    gen = torch.Generator(device=cuda_device).manual_seed(12)
    q = torch.randn((int(qs[-1]), 32, 128), generator=gen, device=cuda_device).to(torch.bfloat16)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attn_prefill(out, q, torch.from_numpy(qs).to(cuda_device), case.k_cache,
                           case.v_cache, case.block_tables, case.context_lens, case.scale,
                           case.max_context_len, max(chunks))
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    tables = case.block_tables.cpu().numpy()
    B = 16
    for s, j in [(0, 0), (0, 31), (0, 32), (0, 191), (1, 0), (1, 64), (1, 76)]:
        p = lens[s] - chunks[s] + j
        nb = -(-(p + 1) // B)
        blocks = torch.from_numpy(tables[s, :nb].astype(np.int64)).to(cuda_device)
        k_sub, v_sub = to_f64(case.k_cache[blocks]), to_f64(case.v_cache[blocks])
        row = int(qs[s]) + j
        ref = oracle.paged_decode_attention(to_f64(q[row:row + 1]), k_sub, v_sub,
                                            np.arange(nb)[None, :], np.array([p + 1]), case.scale)
        assert_within_tol(out[row:row + 1], ref, torch.bfloat16, f"long context seq {s} query {j}")


@pytest.mark.parametrize("dtype,hq,D,lens,chunks", [
    ("bf16", 32, 128, [1500, 1300], [1500, 1200]),  # 8 queries a CTA: 188 query tiles
    ("fp16", 128, 64, [400, 150], [400, 150]),      # 2 queries a CTA: 200 query tiles
])
def test_prefill_more_query_tiles_than_sms(cuda_device, dtype, hq, D, lens, chunks):
    """Large groups (one KV head): more query tiles per (sequence, KV head) than
    the device has SMs, so each launch-order group holds one pair and the Q
    rows fetched ahead for the next wave belong to the same sequence; every
    output against the oracle."""
    case = W.make_decode_case(hq + D, len(lens), hq, 1, D, 16, dtype, lens, pool_factor=1.2,
                              poison=True, device=cuda_device)
    q, out, ref, qs = _run(case, chunks, seed=hq)
    assert_within_tol(out, ref, W.DTYPES[dtype], f"prefill {hq}/1 D={D} chunks {chunks}")


def test_prefill_whole_prompts_sampled(cuda_device):
    """The prefill shape sweep's whole-prompt case (16 prompts of 100-700
    tokens, each queried whole, 40 MHA heads, fp16): 760 of its 1,920 CTAs
    find no queries; sampled queries of every prompt against decode attention
    over their visible prefix, on every head."""
    rng = np.random.default_rng(11)
    prompts = [int(x) for x in rng.integers(100, 701, size=16)]
    case = W.make_decode_case(704, len(prompts), 40, 40, 128, 16, "fp16", prompts,
                              pool_factor=1.0, device=cuda_device)
    qs = np.concatenate([[0], np.cumsum(prompts)]).astype(np.int32)
    gen = torch.Generator(device=cuda_device).manual_seed(4)
    q = torch.randn((int(qs[-1]), 40, 128), generator=gen, device=cuda_device).half()
    out = torch.full_like(q, float("nan"))
    pkv.paged_attn_prefill(out, q, torch.from_numpy(qs).to(cuda_device), case.k_cache,
                           case.v_cache, case.block_tables, case.context_lens, case.scale,
                           case.max_context_len, max(prompts))
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    tables = case.block_tables.cpu().numpy()
    pick = np.random.default_rng(5)
    for s, n in enumerate(prompts):
        for j in (0, n - 1, int(pick.integers(n))):
            nb = -(-(j + 1) // 16)
            blocks = torch.from_numpy(tables[s, :nb].astype(np.int64)).to(cuda_device)
            k_sub, v_sub = to_f64(case.k_cache[blocks]), to_f64(case.v_cache[blocks])
            row = int(qs[s]) + j
            ref = oracle.paged_decode_attention(to_f64(q[row:row + 1]), k_sub, v_sub,
                                                np.arange(nb)[None, :], np.array([j + 1]),
                                                case.scale)
            assert_within_tol(out[row:row + 1], ref, torch.float16, f"prompt {s} query {j}")


def test_prefill_empty_chunks_and_bad_context(cuda_device):
    """Sequences without queries leave nothing to do; a context shorter than
    its chunk is flagged (PKV_DEV_BAD_CONTEXT_LEN = 2) and skipped, while the
    other sequences are still computed exactly."""
    lens = [40, 300, 0, 129]
    case = W.make_decode_case(21, len(lens), 8, 2, 128, 16, "bf16", lens, pool_factor=1.2,
                              poison=True, device=cuda_device)
    chunks = [0, 33, 0, 129]
    q, out, ref, qs = _run(case, chunks, seed=4)
    assert_within_tol(out, ref, torch.bfloat16, "prefill with empty chunks")
    assert pkv.device_status(clear=True) == 0
    # sequence 0 now claims 41 queries against a 40-token context
    chunks = [41, 33, 0, 129]
    qs2 = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    gen = torch.Generator(device=cuda_device).manual_seed(9)
    q2 = torch.randn((int(qs2[-1]), 8, 128), generator=gen, device=cuda_device).to(torch.bfloat16)
    out2 = torch.full_like(q2, float("nan"))
    pkv.paged_attn_prefill(out2, q2, torch.from_numpy(qs2).to(cuda_device), case.k_cache,
                           case.v_cache, case.block_tables, case.context_lens, case.scale,
                           case.max_context_len, 129)
    assert pkv.device_status(clear=True) == 2
    assert torch.isnan(out2[:41]).all()  # the bad sequence is not written
    ok_lens = case.context_lens.cpu().numpy().copy()
    ok_lens[0] = 41
    ref2 = oracle.paged_prefill_attention(to_f64(q2[41:]), to_f64(case.k_cache),
                                          to_f64(case.v_cache),
                                          case.block_tables.cpu().numpy()[1:], ok_lens[1:],
                                          qs2[1:] - 41, case.scale)
    assert_within_tol(out2[41:], ref2, torch.bfloat16, "prefill next to a bad sequence")


def test_rows_past_total_queries_untouched(lib, cuda_device):
    """q and out hold total_queries rows; with total_queries below
    query_start[S] the rows from total_queries on are neither read (the Q
    copies read zeros there) nor written, and the rows before it are exact.
    Only the kernel's own bounds keep the last sequence's tail rows out of
    memory that q and out do not own."""
    lens = [300, 200]
    chunks = [150, 100]
    case = W.make_decode_case(31, len(lens), 32, 8, 128, 16, "bf16", lens, pool_factor=1.2,
                              device=cuda_device)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    gen = torch.Generator(device=cuda_device).manual_seed(8)
    q = torch.randn((int(qs[-1]), 32, 128), generator=gen, device=cuda_device).to(torch.bfloat16)
    out = torch.full_like(q, float("nan"))
    total = 190  # 40 rows of sequence 1 are inside, 60 past the end
    qs_dev = torch.from_numpy(qs).to(cuda_device)
    st = lib.pkv_paged_attn_prefill(
        out.data_ptr(), q.data_ptr(), total, qs_dev.data_ptr(), max(chunks),
        case.k_cache.data_ptr(), case.v_cache.data_ptr(), case.block_tables.data_ptr(),
        case.block_tables.shape[1], case.context_lens.data_ptr(), case.max_context_len, 2, 32,
        8, 128, 16, case.k_cache.shape[0], case.scale, _lib.PKV_BF16,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.isnan(out[total:]).all()
    ref = oracle.paged_prefill_attention(to_f64(q), to_f64(case.k_cache), to_f64(case.v_cache),
                                         case.block_tables.cpu().numpy(),
                                         case.context_lens.cpu().numpy(), qs, case.scale)
    assert_within_tol(out[:total], ref[:total], torch.bfloat16, "rows below total_queries")
