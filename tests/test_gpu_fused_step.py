"""The fused decode step (append the new token, then attend, in one launch)
against the two separate calls and the oracle.

The fused call must leave the caches bit-identical to kv_append and produce
the same output bits as kv_append followed by paged decode (the new row
reaches the same shared-memory row either way), and match the fp64 oracle
applied to the appended cache it computes itself from the inputs."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import assert_within_tol, raw_bytes, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[0, 1], ids=["default-path", "cuda-cores"])
def _clean_status(request, lib, cuda_device):
    """Both decode kernels: the library's choice and the CUDA-core one."""
    assert lib.pkv_set_decode_path(request.param) == 0
    pkv.device_status(clear=True)
    yield
    lib.pkv_set_decode_path(0)
    assert pkv.device_status(clear=True) == 0


def _both_paths(case, k_new, v_new, part):
    slots = W.last_position_slots(case).to(case.q.device)
    ka, va = case.k_cache.clone(), case.v_cache.clone()
    kb, vb = case.k_cache.clone(), case.v_cache.clone()
    out_a = torch.empty_like(case.q)
    out_b = torch.empty_like(case.q)
    pkv.kv_append(k_new, v_new, ka, va, slots)
    pkv.paged_attn_decode(out_a, case.q, ka, va, case.block_tables, case.context_lens,
                          case.scale, case.max_context_len, partition_size=part)
    pkv.paged_attn_decode_append(out_b, case.q, k_new, v_new, kb, vb, case.block_tables,
                                 case.context_lens, case.scale, case.max_context_len,
                                 partition_size=part)
    torch.cuda.synchronize()
    return (out_a, ka, va), (out_b, kb, vb), slots


@pytest.mark.parametrize("dtype,hq,hkv,D,B", [("fp16", 8, 8, 128, 16), ("bf16", 32, 8, 128, 16),
                                              ("bf16", 16, 2, 128, 8), ("fp16", 8, 2, 64, 128),
                                              ("bf16", 12, 4, 64, 32)])
def test_fused_equals_separate_and_oracle(cuda_device, dtype, hq, hkv, D, B):
    lens = [1, 0, B - 1, B, B + 1, 31, 32, 33, 600, 1500]
    case = W.make_decode_case(hq * 7 + B, len(lens), hq, hkv, D, B, dtype, lens, pool_factor=1.3,
                              poison=True, device=cuda_device)
    k_new, v_new = W.new_tokens(B + hq, len(lens), hkv, D, dtype, device=cuda_device)
    # oracle inputs: the pristine cache and the new rows, before any kernel runs
    k0, v0 = to_f64(case.k_cache), to_f64(case.v_cache)
    slots_host = W.last_position_slots(case).numpy()
    k1, v1 = oracle.kv_append(to_f64(k_new), to_f64(v_new), k0, v0, slots_host)
    ref = oracle.paged_decode_attention(to_f64(case.q), k1, v1, case.block_tables.cpu().numpy(),
                                        case.context_lens.cpu().numpy(), case.scale)
    for part in (0, 32, 512):
        (out_a, ka, va), (out_b, kb, vb), _ = _both_paths(case, k_new, v_new, part)
        assert np.array_equal(raw_bytes(kb), raw_bytes(ka))
        assert np.array_equal(raw_bytes(vb), raw_bytes(va))
        assert torch.equal(out_b, out_a), f"fused != separate (partition {part})"
        assert_within_tol(out_b, ref, W.DTYPES[dtype], f"fused partition {part}")


def test_fused_opt13b_layer_full_size(cuda_device):
    case = W.opt13b_layer_decode(device=cuda_device)
    S, Hq, D = case.q.shape
    k_new, v_new = W.new_tokens(11, S, case.k_cache.shape[1], D, "fp16", device=cuda_device)
    (out_a, ka, va), (out_b, kb, vb), _ = _both_paths(case, k_new, v_new, 0)
    assert torch.equal(kb, ka) and torch.equal(vb, va)
    assert torch.equal(out_b, out_a)
