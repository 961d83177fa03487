"""GPU parity of paged decode attention against the fp64 oracle.

Every case runs the CUDA kernels through the C ABI and compares with the
oracle on the same seeded inputs: element by element on small cases (several
32-token stages, ragged tails, NaN-poisoned unused slots and blocks) and on
sampled (sequence, head) outputs at the full workload sizes.  Each case runs
with the library's default kernel choice and with the CUDA-core kernel
forced, so both decode kernels are checked on every shape."""

import numpy as np
import pytest
import torch

import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import TOL, assert_within_tol, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[0, 1], ids=["default-path", "cuda-cores"])
def _clean_status(request, lib, cuda_device):
    """Every case runs twice: with the library's choice of kernel (grouped
    heads of 128 on the tensor cores) and with the CUDA-core kernel forced."""
    assert lib.pkv_set_decode_path(request.param) == 0
    pkv.device_status(clear=True)
    yield
    lib.pkv_set_decode_path(0)
    assert pkv.device_status(clear=True) == 0, "kernel raised a device status flag"


def run(case, partition_size=0):
    out = torch.empty_like(case.q)
    pkv.paged_attn_decode(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                          case.context_lens, case.scale, case.max_context_len,
                          partition_size=partition_size)
    torch.cuda.synchronize()
    return out


def test_tiny_workload_every_output(cuda_device):
    case = W.tiny_decode(device=cuda_device, poison=True)
    ref = oracle_decode(case)
    out = run(case)
    assert_within_tol(out, ref, torch.float16, "tiny")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (12, 4), (8, 2), (16, 2), (6, 2), (32, 1)])
def test_shapes_and_groups(cuda_device, dtype, head_dim, hq, hkv):
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 100, 127, 129, 250, 511, 700]
    case = W.make_decode_case(hq * 31 + hkv + head_dim, len(lens), hq, hkv, head_dim, 16, dtype,
                              lens, pool_factor=1.5, poison=True, device=cuda_device)
    ref = oracle_decode(case)
    for part in (0, 64, 512):
        assert_within_tol(run(case, part), ref, W.DTYPES[dtype], f"partition {part}")


@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128])
def test_block_sizes_ragged(cuda_device, block_size):
    lens = [1, block_size - 1, block_size, block_size + 1, 3 * block_size + 7, 600, 1025]
    case = W.make_decode_case(block_size, len(lens), 8, 2, 128, block_size, "bf16", lens,
                              pool_factor=1.2, poison=True, device=cuda_device)
    ref = oracle_decode(case)
    for part in (0, 32, 96, 1024):
        assert_within_tol(run(case, part), ref, torch.bfloat16, f"B={block_size} part={part}")


def test_empty_and_single_token_contexts(cuda_device):
    lens = [0, 1, 0, 5, 1]
    case = W.make_decode_case(77, len(lens), 8, 8, 128, 16, "fp16", lens, pool_blocks=20,
                              max_blocks_per_seq=4, poison=True, device=cuda_device)
    case.max_context_len = 40  # a loose host bound is allowed
    for part in (0, 32):
        out = run(case, part)
        assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
        assert_within_tol(out, oracle_decode(case), torch.float16, f"part {part}")
    # a one-token context returns that token's value row exactly (p = 1)
    out = run(case)
    tbl = case.block_tables.cpu()
    v_row = case.v_cache[int(tbl[1, 0]), :, 0, :]
    assert torch.equal(out[1], v_row)


def test_split_matches_unsplit(cuda_device):
    lens = [3000, 17, 4096, 2049]
    case = W.make_decode_case(5, len(lens), 32, 8, 128, 16, "bf16", lens, pool_factor=1.1,
                              device=cuda_device)
    ref = oracle_decode(case)
    outs = {}
    for part in (0, 128, 512, 1024, 4096):
        outs[part] = run(case, part)
        assert_within_tol(outs[part], ref, torch.bfloat16, f"partition {part}")
    # one partition covering everything is the unsplit path; results agree
    # with the split ones to a few bf16 ulps
    diff = (outs[4096].float() - outs[512].float()).abs().max().item()
    assert diff < 2e-2


def test_opt13b_layer_full_size(cuda_device):
    """40 MHA heads of 128, fp16, 64 sequences with lognormal lengths."""
    case = W.opt13b_layer_decode(device=cuda_device)
    lens = case.context_lens.cpu().numpy()
    out = run(case)
    # sample: the longest, the shortest and six random sequences, all heads
    rng = np.random.default_rng(0)
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens))} |
                  set(rng.choice(len(lens), 6, replace=False).tolist()))
    ref = oracle_decode(case, seqs)
    assert_within_tol(out[seqs], ref, torch.float16, "opt13b")


def test_gqa_4k_full_size(cuda_device):
    """32 query heads over 8 KV heads, bf16, 256 sequences of 4096 tokens."""
    case = W.gqa_4k_decode(device=cuda_device)
    out = run(case)
    seqs = [0, 97, 255]
    ref = oracle_decode(case, seqs)
    assert_within_tol(out[seqs], ref, torch.bfloat16, "gqa 4k")
    del case
    torch.cuda.empty_cache()


@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("num_seqs,ctx", [(8, 1024), (8, 8192), (8, 32768), (64, 1024),
                                          (64, 8192), (64, 32768)])
def test_block_size_and_long_context_sweep(cuda_device, block_size, num_seqs, ctx):
    case = W.sweep_decode(block_size, num_seqs, ctx, device=cuda_device)
    out = run(case)
    seqs = [0, num_seqs - 1]
    heads = [0, 5, 31]
    ref = oracle_decode(case, seqs, heads)
    for i, s in enumerate(seqs):
        for h in heads:
            assert_within_tol(out[s, h], ref[i, h], torch.bfloat16, f"s={s} h={h}")
    del case, out
    torch.cuda.empty_cache()


def test_permuted_pool_gives_same_output(cuda_device):
    """Moving every block to another physical id (and the table with it)
    leaves the output bit-identical."""
    lens = [100, 333, 17, 1000]
    case = W.make_decode_case(9, len(lens), 8, 2, 64, 16, "fp16", lens, pool_factor=1.3,
                              device=cuda_device)
    out1 = run(case)
    NB = case.k_cache.shape[0]
    pi = torch.randperm(NB, generator=torch.Generator().manual_seed(3)).to(cuda_device)
    k2 = torch.empty_like(case.k_cache)
    v2 = torch.empty_like(case.v_cache)
    k2[pi] = case.k_cache
    v2[pi] = case.v_cache
    t = case.block_tables.long()
    t2 = torch.where(t >= 0, pi[t.clamp(min=0)], t).to(torch.int32)
    case.k_cache, case.v_cache, case.block_tables = k2, v2, t2.contiguous()
    assert torch.equal(run(case), out1)
