"""The contiguous-cache baseline (no block table) on the GPU.

"The KV cache is a systems problem", section "When the extra machinery is not
worth it", asks for a simple contiguous baseline compared under identical
token distributions.  Here the same tokens are laid out both ways: each
sequence reserved at full capacity ([S, Hkv, capacity, D], positions past the
context NaN-poisoned), and paged through a shuffled pool.  Both must match the
oracle, and the two layouts must give bit-identical outputs for the same
partitioning, since only the addresses differ."""

import numpy as np
import pytest
import torch

import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import assert_within_tol, oracle_decode

pytestmark = pytest.mark.gpu


def contiguous_from_paged(case, capacity):
    """Lay each sequence's tokens out contiguously (torch indexing only)."""
    S, Hq, D = case.q.shape
    Hkv, B = case.k_cache.shape[1], case.block_size
    shape = (S, Hkv, capacity, D)
    kc = torch.full(shape, float("nan"), dtype=case.q.dtype, device=case.q.device)
    vc = torch.full(shape, float("nan"), dtype=case.q.dtype, device=case.q.device)
    tables = case.block_tables.long()
    for s, n in enumerate(case.context_lens.tolist()):
        nb = -(-n // B)
        if nb == 0:
            continue
        ids = tables[s, :nb]
        kc[s, :, :n] = case.k_cache[ids].permute(1, 0, 2, 3).reshape(Hkv, nb * B, D)[:, :n]
        vc[s, :, :n] = case.v_cache[ids].permute(1, 0, 2, 3).reshape(Hkv, nb * B, D)[:, :n]
    return kc, vc


@pytest.fixture(autouse=True)
def _clean_status(lib, cuda_device):
    """The contiguous call runs the CUDA-core kernel; the paged calls it is
    compared with bit for bit run the same kernel (setting 1)."""
    pkv.device_status(clear=True)
    assert lib.pkv_set_decode_path(1) == 0
    yield
    lib.pkv_set_decode_path(0)
    assert pkv.device_status(clear=True) == 0


@pytest.mark.parametrize("dtype,hq,hkv,D", [("fp16", 8, 8, 128), ("bf16", 32, 8, 128),
                                            ("fp16", 8, 2, 64)])
def test_contiguous_matches_oracle_and_paged(cuda_device, dtype, hq, hkv, D):
    lens = [1, 31, 32, 33, 200, 1000, 0, 2047]
    case = W.make_decode_case(41 + hq, len(lens), hq, hkv, D, 16, dtype, lens, pool_factor=1.2,
                              poison=True, device=cuda_device)
    capacity = 2048
    kc, vc = contiguous_from_paged(case, capacity)
    ref = oracle_decode(case)
    for part in (0, 256, 2048):
        out_c = torch.empty_like(case.q)
        pkv.contiguous_attn_decode(out_c, case.q, kc, vc, case.context_lens, case.scale,
                                   partition_size=part)
        assert_within_tol(out_c, ref, W.DTYPES[dtype], f"contiguous part={part}")
        if part:
            out_p = torch.empty_like(case.q)
            pkv.paged_attn_decode(out_p, case.q, case.k_cache, case.v_cache, case.block_tables,
                                  case.context_lens, case.scale, capacity, partition_size=part)
            torch.cuda.synchronize()
            assert torch.equal(out_c, out_p)
