"""The kernels' bounded waits on a GPU: a wait that nothing completes gives
up after its limit, the device status reports it, and the context is still
usable afterwards (a decode right after matches the oracle).  No GPU fault,
trap or hang is involved: the wait simply runs out."""

import time

import pytest
import torch

import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import TOL, assert_within_tol, oracle_decode

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = 8  # PKV_DEV_WAIT_TIMEOUT


def test_wait_runs_out_and_context_stays_usable(lib, cuda_device):
    pkv.device_status(clear=True)
    t0 = time.perf_counter()
    pkv.debug_wait_timeout()
    flags = pkv.device_status(clear=True)  # synchronises: the kernel has ended
    elapsed = time.perf_counter() - t0
    assert flags & WAIT_TIMEOUT
    assert 1.0 < elapsed < 30.0  # the 2 s limit, not an endless wait
    assert pkv.device_status(clear=True) == 0
    # the same context runs a decode correctly
    case = W.tiny_decode(device=cuda_device, poison=True)
    out = torch.empty_like(case.q)
    pkv.paged_attn_decode(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                          case.context_lens, case.scale, case.max_context_len)
    assert pkv.device_status(clear=True) == 0
    assert_within_tol(out, oracle_decode(case), torch.float16, "decode after a timed-out wait")
