"""GPU parity of kv_append and block_copy: bit-exact against the oracle's
scatter and copy on the same seeded inputs, including the large instances
(a whole prompt fill, a batch of copy-on-write pairs)."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import raw_bytes

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status(lib, cuda_device):
    pkv.device_status(clear=True)
    yield
    flags = pkv.device_status(clear=True)
    assert flags == 0, f"device status {flags}"


def _cache(seed, nb, hkv, B, D, dtype, device):
    g = torch.Generator(device=device).manual_seed(seed)
    k = torch.randn((nb, hkv, B, D), generator=g, device=device).to(W.DTYPES[dtype])
    v = torch.randn((nb, hkv, B, D), generator=g, device=device).to(W.DTYPES[dtype])
    return k, v


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("B,D,hkv,T", [(16, 128, 40, 64), (8, 64, 8, 33), (128, 128, 8, 300),
                                       (32, 64, 1, 7)])
def test_kv_append_bit_exact(cuda_device, dtype, B, D, hkv, T):
    nb = max(8, 2 * T // B + 4)
    kc, vc = _cache(T, nb, hkv, B, D, dtype, cuda_device)
    k, v = W.new_tokens(T + 1, T, hkv, D, dtype, device=cuda_device)
    rng = np.random.default_rng(T)
    slots = rng.choice(nb * B, size=T, replace=False).astype(np.int64)
    slots[::5] = -1  # padding tokens are skipped
    want_k, want_v = oracle.kv_append(raw_bytes(k), raw_bytes(v), raw_bytes(kc), raw_bytes(vc),
                                      slots)
    pkv.kv_append(k, v, kc, vc, torch.from_numpy(slots).to(cuda_device))
    torch.cuda.synchronize()
    assert np.array_equal(raw_bytes(kc), want_k)
    assert np.array_equal(raw_bytes(vc), want_v)


def test_kv_append_prompt_fill_large(cuda_device):
    """A whole prompt fill: ~6.4k tokens x 40 heads x 128 (about 130 MB)."""
    hkv, D, B = 40, 128, 16
    T = 6400
    nb = T // B + 16
    kc, vc = _cache(1, nb, hkv, B, D, "fp16", cuda_device)
    k, v = W.new_tokens(2, T, hkv, D, "fp16", device=cuda_device)
    perm = np.random.default_rng(5).permutation(nb)[: T // B]
    slots = (perm[:, None] * B + np.arange(B)[None, :]).reshape(-1).astype(np.int64)
    want_k, want_v = oracle.kv_append(raw_bytes(k), raw_bytes(v), raw_bytes(kc), raw_bytes(vc),
                                      slots)
    pkv.kv_append(k, v, kc, vc, torch.from_numpy(slots).to(cuda_device))
    torch.cuda.synchronize()
    assert np.array_equal(raw_bytes(kc), want_k)
    assert np.array_equal(raw_bytes(vc), want_v)


@pytest.mark.parametrize("B,D,hkv,P", [(16, 128, 40, 112), (8, 64, 2, 3), (128, 128, 8, 17)])
def test_block_copy_bit_exact(cuda_device, B, D, hkv, P):
    nb = 2 * P + 5
    kc, vc = _cache(P, nb, hkv, B, D, "fp16", cuda_device)
    ids = np.random.default_rng(P).permutation(nb)
    pairs = np.stack([ids[:P], ids[P:2 * P]], axis=1).astype(np.int64)  # distinct, disjoint
    want_k, want_v = oracle.block_copy(raw_bytes(kc), raw_bytes(vc), pairs)
    pkv.block_copy(kc, vc, torch.from_numpy(pairs).to(cuda_device))
    torch.cuda.synchronize()
    assert np.array_equal(raw_bytes(kc), want_k)
    assert np.array_equal(raw_bytes(vc), want_v)


def test_bad_ids_are_flagged_not_faulted(cuda_device):
    """Out-of-pool ids are caught by the kernels' own bounds checks: the access
    is skipped (or redirected inside the pool) and a status flag is raised."""
    kc, vc = _cache(0, 8, 2, 16, 64, "fp16", cuda_device)
    before_k = raw_bytes(kc)
    k, v = W.new_tokens(0, 2, 2, 64, "fp16", device=cuda_device)
    pkv.kv_append(k, v, kc, vc, torch.tensor([8 * 16, 8 * 16 + 5], device=cuda_device))
    assert pkv.device_status(clear=True) == pkv._lib.DEV_BAD_SLOT
    assert np.array_equal(raw_bytes(kc), before_k)
    pkv.block_copy(kc, vc, torch.tensor([[0, 8]], device=cuda_device))
    assert pkv.device_status(clear=True) == pkv._lib.DEV_BAD_BLOCK_ID
    assert np.array_equal(raw_bytes(kc), before_k)
    q = torch.randn((1, 2, 64), device=cuda_device).half()
    out = torch.empty_like(q)
    tables = torch.tensor([[3, 99]], dtype=torch.int32, device=cuda_device)
    lens = torch.tensor([20], dtype=torch.int32, device=cuda_device)
    pkv.paged_attn_decode(out, q, kc, vc, tables, lens, 0.1, 32)
    assert pkv.device_status(clear=True) == pkv._lib.DEV_BAD_BLOCK_ID
    lens = torch.tensor([40], dtype=torch.int32, device=cuda_device)  # beyond max_context_len
    tables = torch.tensor([[3, 4]], dtype=torch.int32, device=cuda_device)
    pkv.paged_attn_decode(out, q, kc, vc, tables, lens, 0.1, 32)
    assert pkv.device_status(clear=True) == pkv._lib.DEV_BAD_CONTEXT_LEN
