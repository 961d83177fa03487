"""The C ABI on a machine without a GPU: the library loads, exports every
symbol include/pagedkv.h declares, and rejects bad arguments on the host
before anything is enqueued (none of these calls reaches CUDA)."""

import ctypes
import os
import re

import numpy as np
import pytest

from paged_kv_cache_247_gb300 import _lib as L

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "pagedkv.h")


def declared_functions():
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pkv_paged_attn_decode", "pkv_kv_append", "pkv_block_copy",
                     "pkv_decode_workspace_size", "pkv_alloc_create", "pkv_alloc_append_slot"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing
    # and the binding attaches a signature to each of them
    assert set(declared_functions()) == set(L.SIGNATURES)


def test_status_strings(lib):
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(3) == b"workspace too small"
    assert lib.pkv_version() == 1


def _decode(lib, **over):
    a = dict(out=16, q=16, k=16, v=16, tables=16, mbps=4, lens=16, maxctx=64, S=2, Hq=8,
             Hkv=2, D=128, B=16, NB=10, scale=0.1, dtype=0, part=0, ws=None, wsb=0)
    a.update(over)
    return lib.pkv_paged_attn_decode(a["out"], a["q"], a["k"], a["v"], a["tables"], a["mbps"],
                                     a["lens"], a["maxctx"], a["S"], a["Hq"], a["Hkv"], a["D"],
                                     a["B"], a["NB"], a["scale"], a["dtype"], a["part"], a["ws"],
                                     a["wsb"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(Hq=6, Hkv=4), 1),             # Hq not a multiple of Hkv
    (dict(D=96), 2),                    # head_dim not built
    (dict(B=24), 2),                    # block size not built
    (dict(dtype=7), 1),
    (dict(part=48), 1),                 # partition not a multiple of 32
    (dict(q=None), 1),
    (dict(q=8), 1),                     # misaligned
    (dict(tables=2), 1),                # misaligned int32
    (dict(mbps=3), 1),                  # 3 * 16 < 64 = max context
    (dict(maxctx=-1), 1),
    (dict(scale=float("inf")), 1),
    (dict(S=70000), 2),                 # grid limit
    (dict(maxctx=4096, part=512), 3),   # split needs workspace
    (dict(S=0, q=None), 0),             # empty batch is a no-op
])
def test_decode_host_validation(lib, over, expect):
    if over.get("maxctx") == 4096:
        over["mbps"] = 256
    assert _decode(lib, **over) == expect


def test_workspace_size_arithmetic(lib):
    # explicit partitions: 8 sequences, 32 heads, 32k context, 512 tokens -> 64 parts
    assert lib.pkv_decode_workspace_size(8, 32, 8, 128, 32768, 512) == 8 * 32 * 64 * (128 + 2) * 4
    assert lib.pkv_decode_workspace_size(8, 32, 8, 128, 4096, 4096) == 0
    assert lib.pkv_decode_workspace_size(8, 32, 8, 128, 4097, 4096) == 8 * 32 * 2 * 130 * 4
    assert lib.pkv_decode_workspace_size(8, 32, 8, 96, 100, 0) == ctypes.c_size_t(-1).value
    assert lib.pkv_decode_workspace_size(8, 32, 8, 128, 100, 48) == ctypes.c_size_t(-1).value


def test_auto_partition_policy(lib):
    """The CUDA-core kernel's choice (assumes a GB300 without a device: 152
    SMs, 3 CTAs each)."""
    part = lib.pkv_decode_partition_size
    assert part(64, 40, 40, 128, 2048) == 2048      # 2560 units: enough CTAs unsplit
    assert lib.pkv_set_decode_path(1) == 0
    try:
        assert part(8, 32, 8, 128, 100) == 128          # short context: one partition
        assert part(256, 32, 8, 128, 4096) == 2048      # long contexts: 2048-token partitions
        # 64 or 128 units: the fewest whole waves of CTAs (within 5 % below k x 456)
        assert part(8, 32, 8, 128, 8192) == 1184        # 7 parts: 448 CTAs, one wave
        assert part(16, 32, 8, 128, 8192) == 1184       # 7 parts: 896 CTAs, two waves
        assert part(8, 32, 8, 128, 32768) == 1568       # 21 parts: 1344 CTAs, three waves
        assert part(16, 32, 8, 128, 16384) == 1184      # 14 parts: 1792 CTAs, four waves
        assert part(32, 32, 8, 128, 4096) == 1024       # no whole-wave split: ~four waves
        assert part(128, 32, 8, 128, 2048) == 1024      # 1024 units: two partitions
        assert part(8, 32, 8, 128, 1024) == 256         # 64 units: split finer to fill the GPU
        assert part(64, 32, 8, 128, 1024) == 1024       # 512 units: not worth splitting 1k
    finally:
        lib.pkv_set_decode_path(0)
    for args in [(1, 1, 1, 64, 5), (3, 12, 4, 64, 100000), (200, 64, 8, 128, 777)]:
        p = part(*args)
        assert p > 0 and p % 32 == 0
        ws = lib.pkv_decode_workspace_size(*args, 0)
        parts = -(-args[4] // p)
        assert ws == (0 if parts <= 1 else args[0] * args[1] * parts * (args[3] + 2) * 4)


def test_tensor_core_partition_policy(lib):
    """The tensor-core kernel's choice (grouped heads): whole 128-key tiles,
    minimising a model of the persistent kernel's time (152 SMs assumed) in
    tiles at an SM's share of HBM: rounds of items on ceil(items / rounds)
    CTAs, each round's tiles times the fraction of the SMs it occupies but
    at least half, half a tile per item and two tiles for a split.  The
    shapes below are the ones measured on GB300, where the model picks the
    fastest partition."""
    import math
    part = lib.pkv_decode_partition_size

    def model(S, hkv, ctx, parts, sms=152):
        tiles = -(-ctx // 128)
        items = S * hkv * parts
        avg = tiles / parts
        rounds = math.ceil(items / sms)
        ctas = math.ceil(items / rounds)
        return rounds * avg * max(ctas / sms, 0.5) + rounds * 0.5 + (2.0 if parts > 1 else 0.0)

    for S, ctx, want in [(8, 100, 128), (8, 1024, 1024), (64, 1024, 1024), (8, 8192, 4096),
                         (64, 8192, 8192), (8, 32768, 16384), (64, 32768, 32768),
                         (32, 4096, 4096), (256, 4096, 4096)]:
        p = part(S, 32, 8, 128, ctx)
        assert p == want, (S, ctx, p)
        tiles = -(-ctx // 128)
        parts = -(-tiles // (p // 128))
        assert model(S, 8, ctx, parts) <= min(model(S, 8, ctx, n) for n in range(1, 17)) + 1e-9
    # groups of 2 to 32 share the policy, and so do single-head groups with
    # fewer than 8 (sequence, KV head) pairs per SM; with more they take the
    # CUDA-core kernel and its partitions (any multiple of 32)
    assert part(8, 16, 8, 128, 8192) == part(8, 256, 8, 128, 8192) == 4096
    assert part(8, 8, 8, 128, 8192) == 4096
    assert lib.pkv_decode_uses_tensor_cores(8, 8, 8, 128, 8192, 0) == 1
    assert lib.pkv_decode_uses_tensor_cores(8, 16, 8, 64, 8192, 0) == 1
    sms = 152  # no device here: the library assumes a GB300
    assert lib.pkv_decode_uses_tensor_cores(8 * sms // 40 + 1, 40, 40, 128, 2048, 0) == 0
    assert lib.pkv_decode_uses_tensor_cores(8 * sms // 40, 40, 40, 128, 2048, 0) == 1
    assert lib.pkv_decode_uses_tensor_cores(64, 40, 40, 128, 2048, 0) == 0  # the OPT-13B layer
    assert part(256, 8, 8, 128, 2000) % 128 != 0  # CUDA-core kernel: one partition, not whole tiles


def test_auto_partition_properties(lib):
    """Whatever branch picks it, the automatic partition is a positive multiple
    of 32 (of 128 on the tensor-core kernel), on the CUDA-core kernel at most
    2048 tokens unless one partition covers the whole context, and its
    workspace size matches the partition count it implies."""
    part = lib.pkv_decode_partition_size
    ws = lib.pkv_decode_workspace_size
    for S in (1, 3, 8, 16, 37, 64, 128, 256, 1000):
        for hq, hkv in ((8, 8), (32, 8), (40, 40), (12, 4), (64, 8)):
            for ctx in (1, 31, 32, 33, 700, 1024, 2049, 5000, 8192, 32768, 100000):
                p = part(S, hq, hkv, 128, ctx)
                assert p > 0 and p % 32 == 0, (S, hq, hkv, ctx, p)
                parts = -(-ctx // p)
                if lib.pkv_decode_uses_tensor_cores(S, hq, hkv, 128, ctx, 0):
                    assert p % 128 == 0, (S, hq, hkv, ctx, p)
                else:
                    assert p <= 2048 or parts == 1, (S, hq, hkv, ctx, p)
                assert ws(S, hq, hkv, 128, ctx, 0) == (
                    0 if parts <= 1 else S * hq * parts * (128 + 2) * 4), (S, hq, hkv, ctx, p)


def test_append_and_copy_host_validation(lib):
    assert lib.pkv_kv_append(None, None, None, None, None, 0, 8, 128, 16, 4, 0, None) == 0
    assert lib.pkv_kv_append(16, 16, 16, 16, 16, 3, 8, 80, 16, 4, 0, None) == 2
    assert lib.pkv_kv_append(16, 16, 16, 16, 12, 3, 8, 128, 16, 4, 0, None) == 1
    assert lib.pkv_kv_append(16, 16, 16, 16, 16, -1, 8, 128, 16, 4, 0, None) == 1
    # more than 2^31 16-byte chunks of K in one call (2^24 + 1 tokens x 8 heads x
    # 128): refused on the host before anything touches the device
    assert lib.pkv_kv_append(16, 16, 16, 16, 16, (1 << 24) + 1, 8, 128, 16, 4, 0, None) == 2
    assert lib.pkv_block_copy(None, None, None, 0, 4, 4096, None) == 0
    assert lib.pkv_block_copy(16, 16, 16, 2, 4, 4090, None) == 1
    assert lib.pkv_block_copy(16, 16, None, 2, 4, 4096, None) == 1


def _prefill(lib, **over):
    a = dict(out=16, q=16, T=16, qs=16, mql=8, k=16, v=16, tables=16, mbps=4, lens=16, maxctx=64,
             S=2, Hq=8, Hkv=2, D=128, B=16, NB=10, scale=0.1, dtype=1)
    a.update(over)
    return lib.pkv_paged_attn_prefill(a["out"], a["q"], a["T"], a["qs"], a["mql"], a["k"], a["v"],
                                      a["tables"], a["mbps"], a["lens"], a["maxctx"], a["S"],
                                      a["Hq"], a["Hkv"], a["D"], a["B"], a["NB"], a["scale"],
                                      a["dtype"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(Hq=6, Hkv=4), 1),             # Hq not a multiple of Hkv
    (dict(D=96), 2),                    # head_dim not built
    (dict(B=24), 2),                    # block size not built
    (dict(B=4), 2),                     # runs shorter than an 8-row TMA group
    (dict(dtype=7), 1),
    (dict(Hq=256, Hkv=1), 2),           # group larger than a 128-row tile
    (dict(mql=-1), 1),
    (dict(scale=float("nan")), 1),
    (dict(qs=None), 1),
    (dict(k=8), 1),                     # misaligned cache
    (dict(qs=2), 1),                    # misaligned int32 offsets
    (dict(mbps=3), 1),                  # 3 * 16 < 64 = max context
    (dict(NB=0), 1),
    (dict(S=70000), 2),                 # grid limit
    (dict(S=0, q=None), 0),             # empty batch is a no-op
    (dict(mql=0, q=None), 0),           # no queries: a no-op
    (dict(T=-1), 1),                    # negative row count of q and out
    (dict(T=0, q=None), 0),             # no rows: a no-op
])
def test_prefill_host_validation(lib, over, expect):
    assert _prefill(lib, **over) == expect


def test_copy_pair_validation():
    from paged_kv_cache_247_gb300.ops import check_copy_pairs
    check_copy_pairs([[0, 5], [1, 6], [2, 7]], 8)
    check_copy_pairs(np.zeros((0, 2), dtype=np.int64), 8)
    for bad in ([[0, 5], [1, 5]],        # destination twice
                [[0, 5], [5, 6]],        # 5 is a destination and a source
                [[0, 8]], [[-1, 3]]):    # ids outside the pool
        with pytest.raises(ValueError):
            check_copy_pairs(bad, 8)


def test_decode_path_switch(lib):
    """The process-wide decode-path control: values 0-2 only, and the
    partition it implies (tensor-core partitions are whole 128-key tiles;
    without a device the library assumes a GB300's 152 SMs)."""
    assert lib.pkv_get_decode_path() == 0
    try:
        for bad in (-1, 3):
            assert lib.pkv_set_decode_path(bad) == 1
            assert lib.pkv_get_decode_path() == 0
        # groups of 8 and more go to the tensor cores by default
        assert lib.pkv_decode_partition_size(8, 64, 8, 128, 8192) % 128 == 0
        assert lib.pkv_decode_partition_size(8, 256, 8, 128, 32768) % 128 == 0
        assert lib.pkv_set_decode_path(2) == 0
        assert lib.pkv_decode_partition_size(8, 32, 8, 128, 8192) % 128 == 0
        # forced, single-head groups run on the tensor cores whatever their number
        # of (sequence, head) pairs; head size 64 has both
        assert lib.pkv_decode_uses_tensor_cores(8, 8, 8, 128, 8192, 0) == 1
        assert lib.pkv_decode_uses_tensor_cores(256, 40, 40, 128, 2048, 0) == 1
        assert lib.pkv_decode_uses_tensor_cores(8, 64, 8, 64, 8192, 0) == 1
        assert lib.pkv_decode_uses_tensor_cores(8, 64, 8, 64, 8192, 96) == 0  # not whole tiles
        for args in ((8, 8, 8, 128, 8192), (8, 64, 8, 64, 8192)):
            assert lib.pkv_decode_partition_size(*args) % 32 == 0
        assert lib.pkv_set_decode_path(1) == 0
        assert lib.pkv_get_decode_path() == 1
    finally:
        lib.pkv_set_decode_path(0)
