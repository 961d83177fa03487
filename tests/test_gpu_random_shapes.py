"""Seeded random shapes against the fp64 oracle: decode on both kernels (the
library's choice and each kernel forced), the fused append + decode step and
chunked prefill.

The fixed-shape tests pick their cases by hand; these draw them: batch size,
query and KV heads (any group from 1 to 32, powers of two or not), head size,
block size, dtype, context lengths from 0 up to several thousand tokens with
duplicates, partitions from the library's choice down to one tile, and the
number of work items relative to the SMs.  Every output is compared with the
oracle; caches after the fused step bit for bit with kv_append's."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import assert_within_tol, oracle_decode, raw_bytes, to_f64

pytestmark = pytest.mark.gpu

N_CASES = 48


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([1, 1, 2, 3, 4, 5, 8, 12, 16, 32]))
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([8, 16, 32, 64, 128]))
    dtype = str(rng.choice(["fp16", "bf16"]))
    S = int(rng.integers(1, 40))
    kind = rng.integers(3)
    if kind == 0:      # short, ragged, with empty contexts
        lens = rng.integers(0, 300, size=S)
    elif kind == 1:    # lognormal around a few hundred, clipped
        lens = np.clip(rng.lognormal(6.0, 1.0, size=S), 1, 3000).astype(np.int64)
    else:              # a few long ones among short ones, duplicates
        lens = rng.choice([1, 17, 128, 129, 1000, 4097], size=S)
    part = int(rng.choice([0, 0, 128, 256, 512, 1024]))
    lens = [int(x) for x in lens]
    # keep the oracle's share small: at most 60k (token, KV head) pairs
    while len(lens) > 1 and sum(lens) * hkv > 60000:
        lens.pop()
    lens[0] = min(lens[0], 60000 // hkv)
    return dict(S=len(lens), hq=hkv * group, hkv=hkv, D=D, B=B, dtype=dtype, lens=lens, part=part)


@pytest.fixture(autouse=True)
def _clean(lib, cuda_device):
    pkv.device_status(clear=True)
    yield
    lib.pkv_set_decode_path(0)
    assert pkv.device_status(clear=True) == 0


@pytest.mark.parametrize("seed", range(N_CASES))
def test_decode_random(lib, cuda_device, seed):
    c = draw(seed)
    case = W.make_decode_case(2000 + seed, c["S"], c["hq"], c["hkv"], c["D"], c["B"], c["dtype"],
                              c["lens"], pool_factor=1.3, poison=True, device=cuda_device)
    ref = oracle_decode(case)
    tdt = W.DTYPES[c["dtype"]]
    for path in (0, 1, 2):
        if path == 2 and c["hq"] // c["hkv"] > 128:
            continue
        assert lib.pkv_set_decode_path(path) == 0
        out = torch.full_like(case.q, float("nan"))
        pkv.paged_attn_decode(out, case.q, case.k_cache, case.v_cache, case.block_tables,
                              case.context_lens, case.scale, case.max_context_len,
                              partition_size=c["part"])
        torch.cuda.synchronize()
        assert_within_tol(out, ref, tdt, f"seed {seed} path {path} {c}")
    lib.pkv_set_decode_path(0)


@pytest.mark.parametrize("seed", range(0, N_CASES, 3))
def test_fused_step_random(lib, cuda_device, seed):
    """The fused step writes the new token at position ctx - 1 and attends over
    it: caches equal kv_append's, output the oracle's on the appended cache."""
    c = draw(seed)
    lens = [max(1, x) for x in c["lens"]]
    case = W.make_decode_case(3000 + seed, c["S"], c["hq"], c["hkv"], c["D"], c["B"], c["dtype"],
                              lens, pool_factor=1.3, device=cuda_device)
    k_new, v_new = W.new_tokens(seed, c["S"], c["hkv"], c["D"], c["dtype"], device=cuda_device)
    tables = case.block_tables.cpu().numpy()
    slots = torch.tensor([int(tables[s, (n - 1) // c["B"]]) * c["B"] + (n - 1) % c["B"]
                          for s, n in enumerate(lens)], dtype=torch.int64, device=cuda_device)
    kc_ref, vc_ref = case.k_cache.clone(), case.v_cache.clone()
    pkv.kv_append(k_new, v_new, kc_ref, vc_ref, slots)
    out = torch.full_like(case.q, float("nan"))
    pkv.paged_attn_decode_append(out, case.q, k_new, v_new, case.k_cache, case.v_cache,
                                 case.block_tables, case.context_lens, case.scale,
                                 case.max_context_len, partition_size=c["part"])
    torch.cuda.synchronize()
    assert np.array_equal(raw_bytes(case.k_cache), raw_bytes(kc_ref))
    assert np.array_equal(raw_bytes(case.v_cache), raw_bytes(vc_ref))
    assert_within_tol(out, oracle_decode(case), W.DTYPES[c["dtype"]], f"fused seed {seed} {c}")


@pytest.mark.parametrize("seed", range(1, N_CASES, 3))
def test_prefill_random(cuda_device, seed):
    """Chunks of random length at the end of random contexts (every chunk no
    longer than its context), over the whole batch against the oracle."""
    c = draw(seed)
    rng = np.random.default_rng(4000 + seed)
    lens = [max(1, min(x, 1500)) for x in c["lens"]]
    chunks = [int(rng.integers(0, min(n, 160) + 1)) for n in lens]
    # the oracle's share: at most 3e7 (query, key, head) triples
    while len(lens) > 1 and sum(q * n for q, n in zip(chunks, lens)) * c["hq"] > 3e7:
        lens.pop()
        chunks.pop()
    case = W.make_decode_case(5000 + seed, len(lens), c["hq"], c["hkv"], c["D"], c["B"],
                              c["dtype"], lens, pool_factor=1.3, poison=True, device=cuda_device)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    total = max(1, int(qs[-1]))
    gen = torch.Generator(device=cuda_device).manual_seed(seed)
    q = torch.randn((total, c["hq"], c["D"]), generator=gen, device=cuda_device).to(case.q.dtype)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attn_prefill(out, q, torch.from_numpy(qs).to(cuda_device), case.k_cache,
                           case.v_cache, case.block_tables, case.context_lens, case.scale,
                           case.max_context_len, max(1, max(chunks)))
    torch.cuda.synchronize()
    if qs[-1] == 0:
        assert torch.isnan(out).all()   # nothing to compute: nothing written
        return
    ref = oracle.paged_prefill_attention(to_f64(q[:qs[-1]]), to_f64(case.k_cache),
                                         to_f64(case.v_cache), case.block_tables.cpu().numpy(),
                                         case.context_lens.cpu().numpy(), qs, case.scale)
    assert_within_tol(out[:qs[-1]], ref, W.DTYPES[c["dtype"]], f"prefill seed {seed} {c}")
