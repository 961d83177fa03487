"""max_context_len is a host-side upper bound on the contexts, not their
maximum: callers often pass the model's limit (or the block table's capacity)
while every context is much shorter.  The grid and the split partitions are
then sized for contexts that no sequence has, so most work items find no keys
and the reduction merges fewer partitions than it was launched with.  The
outputs must not change, and no table entry past a context (-1 here, which a
read would flag as a bad block id) may be read."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import assert_within_tol, oracle_decode, raw_bytes, to_f64

pytestmark = pytest.mark.gpu

LENS = [1, 100, 700, 33, 0, 2048, 129, 5]
BOUND = 16384


@pytest.fixture(autouse=True)
def _clean(lib, cuda_device):
    pkv.device_status(clear=True)
    yield
    lib.pkv_set_decode_path(0)
    assert pkv.device_status(clear=True) == 0


def _case(seed, hq, hkv, D, B, dtype, device, lens=LENS):
    return W.make_decode_case(seed, len(lens), hq, hkv, D, B, dtype, lens, pool_factor=1.3,
                              max_blocks_per_seq=BOUND // B, poison=True, device=device)


@pytest.mark.parametrize("hq,hkv,D,B,dtype", [(8, 8, 128, 16, "fp16"), (32, 8, 128, 16, "bf16"),
                                              (64, 2, 64, 32, "bf16")])
@pytest.mark.parametrize("part", [0, 512])
def test_decode_with_loose_bound(lib, cuda_device, hq, hkv, D, B, dtype, part):
    case = _case(hq + B, hq, hkv, D, B, dtype, cuda_device)
    ref = oracle_decode(case)
    for path in (0, 1, 2):
        assert lib.pkv_set_decode_path(path) == 0
        outs = []
        for bound in (case.max_context_len, BOUND):
            out = torch.full_like(case.q, float("nan"))
            pkv.paged_attn_decode(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                                  case.context_lens, case.scale, bound, partition_size=part)
            torch.cuda.synchronize()
            assert_within_tol(out, ref, W.DTYPES[dtype], f"path {path} bound {bound}")
            outs.append(out)
        if part:
            # the same partition, so the same kernels over the same keys
            assert torch.equal(outs[0], outs[1]), f"path {path}: the bound changed the result"


def test_fused_step_with_loose_bound(cuda_device):
    lens = [max(1, n) for n in LENS]
    case = _case(7, 40, 40, 128, 16, "fp16", cuda_device, lens)
    k_new, v_new = W.new_tokens(7, len(lens), 40, 128, "fp16", device=cuda_device)
    tables = case.block_tables.cpu().numpy()
    slots = torch.tensor([int(tables[s, (n - 1) // 16]) * 16 + (n - 1) % 16
                          for s, n in enumerate(lens)], dtype=torch.int64, device=cuda_device)
    kc_ref, vc_ref = case.k_cache.clone(), case.v_cache.clone()
    pkv.kv_append(k_new, v_new, kc_ref, vc_ref, slots)
    out = torch.full_like(case.q, float("nan"))
    pkv.paged_attn_decode_append(out, case.q, k_new, v_new, case.k_cache, case.v_cache,
                                 case.block_tables, case.context_lens, case.scale, BOUND)
    torch.cuda.synchronize()
    assert np.array_equal(raw_bytes(case.k_cache), raw_bytes(kc_ref))
    assert np.array_equal(raw_bytes(case.v_cache), raw_bytes(vc_ref))
    assert_within_tol(out, oracle_decode(case), torch.float16, "fused step, loose bound")


def test_prefill_with_loose_bound(cuda_device):
    lens = [max(1, n) for n in LENS]
    chunks = [min(n, c) for n, c in zip(lens, [1, 100, 300, 33, 1, 200, 129, 5])]
    case = _case(9, 32, 8, 128, 16, "bf16", cuda_device, lens)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    gen = torch.Generator(device=cuda_device).manual_seed(9)
    q = torch.randn((int(qs[-1]), 32, 128), generator=gen, device=cuda_device).bfloat16()
    ref = oracle.paged_prefill_attention(to_f64(q), to_f64(case.k_cache), to_f64(case.v_cache),
                                         case.block_tables.cpu().numpy(),
                                         case.context_lens.cpu().numpy(), qs, case.scale)
    outs = []
    for bound in (case.max_context_len, BOUND):
        out = torch.full_like(q, float("nan"))
        pkv.paged_attn_prefill(out, q, torch.from_numpy(qs).to(cuda_device), case.k_cache,
                               case.v_cache, case.block_tables, case.context_lens, case.scale,
                               bound, max(chunks))
        torch.cuda.synchronize()
        assert_within_tol(out, ref, torch.bfloat16, f"prefill bound {bound}")
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
