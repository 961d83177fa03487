"""GPU parity of the tensor-core grouped-head decode kernel against the fp64
oracle.

The kernel puts 128 keys of a tile on the MMA's M dimension and the group's
query heads on N (padded to 16 or 32); for head size 64 the P.V product puts
the heads on M instead.  Both head sizes run every case, covering groups that fill
N exactly and groups that leave padding (3, 6, 12, 20), contexts that end
inside, at and just past a 128-key tile and a block, every block size,
NaN-poisoned tails and unused blocks, split and unsplit partitions, the
fused append, and the lazily moved running maximum (a later tile exceeding
the first one's maximum by far, so the accumulated output is rescaled in
tensor memory).  The path is forced with pkv_set_decode_path(2) and put
back to the default afterwards."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import assert_within_tol, oracle_decode, raw_bytes, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tc_path(lib, cuda_device):
    pkv.device_status(clear=True)
    assert lib.pkv_set_decode_path(2) == 0
    yield
    lib.pkv_set_decode_path(0)
    assert pkv.device_status(clear=True) == 0, "kernel raised a device status flag"


def run(case, partition_size=0):
    out = torch.full_like(case.q, float("nan"))
    pkv.paged_attn_decode(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                          case.context_lens, case.scale, case.max_context_len,
                          partition_size=partition_size)
    torch.cuda.synchronize()
    return out


LENS = [1, 2, 15, 16, 17, 127, 128, 129, 255, 256, 257, 700, 1500]


@pytest.mark.parametrize("head_dim", [128, 64])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (12, 4), (16, 4), (24, 4), (16, 2), (48, 4),
                                    (32, 2), (40, 2), (64, 2), (32, 1)])
def test_groups_ragged(cuda_device, dtype, hq, hkv, head_dim):
    case = W.make_decode_case(hq * 13 + hkv + head_dim, len(LENS), hq, hkv, head_dim, 16, dtype,
                              LENS, pool_factor=1.4, poison=True, device=cuda_device)
    assert pkv.decode_uses_tensor_cores(len(LENS), hq, hkv, head_dim, case.max_context_len)
    ref = oracle_decode(case)
    for part in (0, 128, 256, 1024):
        assert_within_tol(run(case, part), ref, W.DTYPES[dtype],
                          f"G={hq // hkv} D={head_dim} part={part}")


@pytest.mark.parametrize("head_dim", [128, 64])
@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128])
def test_block_sizes(cuda_device, block_size, head_dim):
    lens = [1, block_size - 1, block_size, block_size + 1, 3 * block_size + 7, 600, 1025]
    case = W.make_decode_case(block_size + 3, len(lens), 64, 8, head_dim, block_size, "bf16",
                              lens, pool_factor=1.2, poison=True, device=cuda_device)
    ref = oracle_decode(case)
    for part in (0, 128, 384):
        assert_within_tol(run(case, part), ref, torch.bfloat16,
                          f"B={block_size} D={head_dim} part={part}")


@pytest.mark.parametrize("head_dim", [128, 64])
def test_empty_and_single_token_contexts(cuda_device, head_dim):
    lens = [0, 1, 0, 5, 1]
    case = W.make_decode_case(78, len(lens), 64, 8, head_dim, 16, "fp16", lens, pool_blocks=20,
                              max_blocks_per_seq=4, poison=True, device=cuda_device)
    case.max_context_len = 40  # a loose host bound is allowed
    out = run(case)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert_within_tol(out, oracle_decode(case), torch.float16, "empty/single")
    # one key: its weight is exp2(0) = 1 exactly, so the output is V_0
    tbl = case.block_tables.cpu()
    for s in (1, 4):
        v_row = case.v_cache[int(tbl[s, 0]), :, 0, :]  # [Hkv, D]
        assert torch.equal(out[s], v_row.repeat_interleave(8, dim=0))


@pytest.mark.parametrize("head_dim", [128, 64])
def test_running_max_moves_late(cuda_device, head_dim):
    """A key late in the context dominates (its logit is far above the first
    tile's maximum), and logits with a large scale keep moving the maximum:
    the accumulated output must be rescaled, not overflow or go stale."""
    lens = [300, 1000, 2000, 129]
    case = W.make_decode_case(91, len(lens), 32, 4, head_dim, 16, "bf16", lens, pool_factor=1.1,
                              device=cuda_device)
    tbl = case.block_tables.cpu()
    for s, pos in ((0, 290), (1, 700), (2, 1999), (3, 128)):
        blk, off = int(tbl[s, pos // 16]), pos % 16
        # key of KV head 0 at `pos` along query head 0's direction: a logit
        # of about 3 * |q|^2 * scale, tens of units above the rest
        case.k_cache[blk, 0, off] = (3.0 * case.q[s, 0].float()).to(torch.bfloat16)
    ref = oracle_decode(case)
    for part in (0, 128, 512):
        assert_within_tol(run(case, part), ref, torch.bfloat16, f"dominant key part={part}")
    case.scale = 1.0  # logits ~ N(0, 128): maxima keep growing across tiles
    ref = oracle_decode(case)
    for part in (0, 256):
        assert_within_tol(run(case, part), ref, torch.bfloat16, f"scale 1 part={part}")


@pytest.mark.parametrize("dtype,hq,hkv,B,D", [("bf16", 32, 8, 16, 128), ("fp16", 64, 8, 8, 128),
                                               ("bf16", 24, 4, 128, 128), ("fp16", 32, 8, 16, 64),
                                               ("bf16", 64, 4, 32, 64)])
def test_fused_append_equals_separate_and_oracle(cuda_device, dtype, hq, hkv, B, D):
    lens = [1, 0, B - 1, B, B + 1, 127, 128, 129, 600, 1500]
    case = W.make_decode_case(hq * 5 + B + D, len(lens), hq, hkv, D, B, dtype, lens,
                              pool_factor=1.3, poison=True, device=cuda_device)
    k_new, v_new = W.new_tokens(B + hq + 1, len(lens), hkv, D, dtype, device=cuda_device)
    k0, v0 = to_f64(case.k_cache), to_f64(case.v_cache)
    slots = W.last_position_slots(case)
    k1, v1 = oracle.kv_append(to_f64(k_new), to_f64(v_new), k0, v0, slots.numpy())
    ref = oracle.paged_decode_attention(to_f64(case.q), k1, v1, case.block_tables.cpu().numpy(),
                                        case.context_lens.cpu().numpy(), case.scale)
    for part in (0, 128, 512):
        ka, va = case.k_cache.clone(), case.v_cache.clone()
        kb, vb = case.k_cache.clone(), case.v_cache.clone()
        out_a, out_b = torch.empty_like(case.q), torch.empty_like(case.q)
        pkv.kv_append(k_new, v_new, ka, va, slots.to(cuda_device))
        pkv.paged_attn_decode(out_a, case.q, ka, va, case.block_tables, case.context_lens,
                              case.scale, case.max_context_len, partition_size=part)
        pkv.paged_attn_decode_append(out_b, case.q, k_new, v_new, kb, vb, case.block_tables,
                                     case.context_lens, case.scale, case.max_context_len,
                                     partition_size=part)
        torch.cuda.synchronize()
        assert np.array_equal(raw_bytes(kb), raw_bytes(ka))
        assert np.array_equal(raw_bytes(vb), raw_bytes(va))
        assert torch.equal(out_b, out_a), f"fused != separate (partition {part})"
        assert_within_tol(out_b, ref, W.DTYPES[dtype], f"fused partition {part}")


@pytest.mark.parametrize("group,head_dim", [(4, 128), (8, 128), (32, 128), (8, 64), (32, 64)])
def test_long_contexts_sampled(cuda_device, group, head_dim):
    """32 sequences x 4096 tokens over 8 KV heads (the query-head group sweep
    of the bench) plus 8 x 32k, sampled sequences, every head."""
    case = W.make_decode_case(6, 32, 8 * group, 8, head_dim, 16, "bf16", [4096] * 32,
                              device=cuda_device)
    out = run(case)
    assert_within_tol(out[[0, 31]], oracle_decode(case, [0, 31]), torch.bfloat16,
                      f"G={group} D={head_dim} 32x4k")
    del case, out
    case = W.sweep_decode(16, 8, 32768, device=cuda_device)
    out = run(case)
    heads = [0, 13, 31]
    ref = oracle_decode(case, [0, 7], heads)
    for i, s in enumerate((0, 7)):
        for h in heads:
            assert_within_tol(out[s, h], ref[i, h], torch.bfloat16, f"8x32k s={s} h={h}")
    del case, out
    torch.cuda.empty_cache()


def test_default_path_takes_grouped_heads(lib, cuda_device):
    """By default grouped heads go to the tensor-core kernel (its partitions
    are whole 128-key tiles), and so do single-head groups with few (sequence,
    KV head) pairs (8 x 8 here); both agree with the oracle."""
    lib.pkv_set_decode_path(0)
    assert lib.pkv_get_decode_path() == 0
    for hq, hkv in ((64, 8), (32, 8), (8, 8)):
        part = pkv.decode_partition_size(8, hq, hkv, 128, 8192)
        assert pkv.decode_uses_tensor_cores(8, hq, hkv, 128, 8192)
        assert part > 0 and part % 128 == 0
        lens = [8192, 100, 5000, 7777, 1, 4096, 3000, 8000]
        case = W.make_decode_case(hq + 1, 8, hq, hkv, 128, 16, "bf16", lens, pool_factor=1.1,
                                  device=cuda_device)
        out = run(case)
        assert_within_tol(out[[0, 3, 4]], oracle_decode(case, [0, 3, 4]), torch.bfloat16,
                          f"default path {hq}/{hkv}")
        del case, out
    torch.cuda.empty_cache()
