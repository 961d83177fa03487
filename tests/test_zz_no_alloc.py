"""The allocation-free decode entry point (pkv_paged_attn_decode_noalloc).

It exists for callers that cannot allocate device memory while they run (a
serving engine that owns all device memory through its own pool, or a
latency-critical loop where cudaMalloc could synchronise the device).  It
keeps the split-context partials in a fixed array inside the library instead
of a caller workspace.  This file is collected last so that a run stopping at
the first failure has already run every other test."""

import ctypes

import pytest
import torch

import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import _lib
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import assert_within_tol, oracle_decode

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20  # PKV_NOALLOC_SCRATCH_BYTES in include/pagedkv.h


def _call_noalloc(lib, out, case, partition_size=0):
    S, Hq, D = case.q.shape
    NB, Hkv, B, _ = case.k_cache.shape
    dtype = _lib.PKV_F16 if case.q.dtype == torch.float16 else _lib.PKV_BF16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pkv_paged_attn_decode_noalloc(
        out.data_ptr(), case.q.data_ptr(), case.k_cache.data_ptr(), case.v_cache.data_ptr(),
        case.block_tables.data_ptr(), case.block_tables.shape[1], case.context_lens.data_ptr(),
        case.max_context_len, S, Hq, Hkv, D, B, NB, case.scale, dtype, partition_size, stream)


def _with_workspace(case, partition_size=0):
    out = torch.empty_like(case.q)
    pkv.paged_attn_decode(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                          case.context_lens, case.scale, case.max_context_len,
                          partition_size=partition_size)
    return out


def test_noalloc_matches_workspace_entry_point(lib, cuda_device):
    pkv.device_status(clear=True)
    # Two different batches in a row: both split their contexts, so the
    # second call reuses the array the first one left filled, with fewer
    # partitions per sequence in places (a stale partial would show).
    first = W.make_decode_case(21, 8, 32, 8, 128, 16, "bf16",
                               [8192, 100, 5000, 7777, 1, 4096, 3000, 8000], pool_factor=1.1,
                               device=cuda_device)
    second = W.opt13b_layer_decode(device=cuda_device)
    for case, part, sample in ((first, 0, range(8)), (second, 512, (0, 7, 21, 40, 63))):
        S, Hq, D = case.q.shape
        Hkv = case.k_cache.shape[1]
        need = pkv.decode_workspace_size(S, Hq, Hkv, D, case.max_context_len, part)
        assert 0 < need <= SCRATCH_BYTES
        ref = _with_workspace(case, part)
        out = torch.full_like(case.q, float("nan"))
        assert _call_noalloc(lib, out, case, part) == 0
        torch.cuda.synchronize()
        # the same kernels at the same partition size: the same bits
        assert torch.equal(out, ref), "noalloc differs from the workspace entry point"
        # and the oracle on sampled sequences, all heads
        sample = list(sample)
        assert_within_tol(out[sample], oracle_decode(case, sample), case.q.dtype,
                          "noalloc vs oracle")
    assert pkv.device_status(clear=True) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(lib, cuda_device):
    case = W.make_decode_case(3, 2, 8, 8, 64, 16, "fp16", [40, 7], device=cuda_device)
    case.max_context_len = 1 << 20  # needs far more than the fixed scratch
    case.block_tables = torch.zeros((2, (1 << 20) // 16), dtype=torch.int32, device=cuda_device)
    out = torch.zeros_like(case.q)
    assert _call_noalloc(lib, out, case, partition_size=32) == 3  # PKV_ERR_WORKSPACE_TOO_SMALL
    assert torch.count_nonzero(out) == 0  # nothing was enqueued
