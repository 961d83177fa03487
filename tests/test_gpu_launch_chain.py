"""Back-to-back launches of the library's kernels with nothing else between
them on the stream (no copies, no other kernels), as a serving loop issues
them.

Each kernel of the library is launched so that it may be placed on the GPU
while the kernel before it still runs, and waits for that kernel before it
touches memory.  These chains check both directions of that contract:

* every kernel sees what the kernels before it wrote (the new rows of
  kv_append, the blocks block_copy filled, the split partials the reduction
  merges);
* no kernel overwrites what an earlier one is still reading: each step's
  block_copy overwrites a block that the previous step's decode attended
  over, so a copy that ran early would change that decode's output.

All inputs are staged on the device first; the outputs are checked against
the fp64 oracle replaying the same operations in the same order."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import assert_within_tol, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[0, 1], ids=["default-path", "cuda-cores"])
def _clean_status(request, lib, cuda_device):
    """Both decode kernels: the library's choice (grouped heads of 128 on the
    tensor cores) and the CUDA-core one."""
    assert lib.pkv_set_decode_path(request.param) == 0
    pkv.device_status(clear=True)
    yield
    lib.pkv_set_decode_path(0)
    assert pkv.device_status(clear=True) == 0


@pytest.mark.parametrize("dtype,hq,hkv,D,B", [("bf16", 16, 4, 128, 16), ("fp16", 8, 8, 64, 32)])
def test_adjacent_launch_chain(cuda_device, dtype, hq, hkv, D, B):
    T = 10
    base = np.array([40, 300, 17, 900, 1, 128], dtype=np.int64)
    S = len(base)
    final = base + T
    case = W.make_decode_case(hq * 5 + B, S, hq, hkv, D, B, dtype, final, pool_factor=1.6,
                              poison=False, device=cuda_device)
    tdt = case.q.dtype
    tables = case.block_tables.cpu().numpy()
    used = set(int(b) for b in tables[tables >= 0])
    spare = [b for b in range(case.k_cache.shape[0]) if b not in used]
    assert len(spare) >= T
    # Step t > 0 overwrites logical block t of the longest sequence (inside
    # every step's context) with a spare block of different contents.
    victim_seq = int(np.argmax(base))
    assert base[victim_seq] // B > T
    pairs_np = [np.array([[spare[t], int(tables[victim_seq, t])]], dtype=np.int64)
                for t in range(T)]
    slots_np = np.empty((T, S), dtype=np.int64)
    for t in range(T):
        pos = base + t
        slots_np[t] = tables[np.arange(S), pos // B].astype(np.int64) * B + pos % B
    ctx_np = np.stack([(base + t + 1).astype(np.int32) for t in range(T)])

    k_new, v_new = W.new_tokens(77 + hq, T * S, hkv, D, dtype, device=cuda_device)
    k_new, v_new = k_new.view(T, S, hkv, D), v_new.view(T, S, hkv, D)
    gen = torch.Generator(device=cuda_device).manual_seed(5 + D)
    q_all = torch.randn((T, S, hq, D), generator=gen, device=cuda_device).to(tdt)
    pairs_all = torch.from_numpy(np.stack(pairs_np)).to(cuda_device)
    slots_all = torch.from_numpy(slots_np).to(cuda_device)
    ctx_all = torch.from_numpy(ctx_np).to(cuda_device)
    out_all = torch.empty((T, S, hq, D), dtype=tdt, device=cuda_device)
    kc, vc = case.k_cache, case.v_cache
    k_h, v_h = to_f64(kc), to_f64(vc)
    max_ctx = int(final.max())
    torch.cuda.synchronize()

    for t in range(T):
        if t > 0:
            pkv.block_copy(kc, vc, pairs_all[t])
        part = (64, 0, 32)[t % 3]  # split into many partitions, automatic, finest
        if t % 2 == 0:
            pkv.kv_append(k_new[t], v_new[t], kc, vc, slots_all[t])
            pkv.paged_attn_decode(out_all[t], q_all[t], kc, vc, case.block_tables, ctx_all[t],
                                  case.scale, max_ctx, partition_size=part)
        else:
            pkv.paged_attn_decode_append(out_all[t], q_all[t], k_new[t], v_new[t], kc, vc,
                                         case.block_tables, ctx_all[t], case.scale, max_ctx,
                                         partition_size=part)
    torch.cuda.synchronize()

    kn, vn, q64 = to_f64(k_new), to_f64(v_new), to_f64(q_all)
    for t in range(T):
        if t > 0:
            k_h, v_h = oracle.block_copy(k_h, v_h, pairs_np[t])
        k_h, v_h = oracle.kv_append(kn[t], vn[t], k_h, v_h, slots_np[t])
        ref = oracle.paged_decode_attention(q64[t], k_h, v_h, tables, ctx_np[t], case.scale)
        assert_within_tol(out_all[t], ref, tdt, f"step {t}")
    assert np.array_equal(to_f64(kc), k_h)
    assert np.array_equal(to_f64(vc), v_h)
