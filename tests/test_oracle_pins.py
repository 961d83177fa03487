"""Pins for the CPU oracle: facts the pages print, closed forms, invariants,
library routines and brute force — nothing here re-derives a value from the
oracle itself.  Runs on CPU (not marked gpu)."""

import inspect
import json
import math
import os
import types

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import attention as oracle_attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


@pytest.fixture(scope="module")
def facts():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------- facts ----

def test_opt13b_800_kib_per_token(facts):
    f = facts["opt13b_bytes_per_token"]
    direct = 2 * f["hidden"] * f["layers"] * f["element_bytes"]
    assert direct == f["printed_kb"] * 1024 == 819200
    # hidden 5120 = 40 heads x 128 head dim
    assert oracle.kv_bytes_per_token(f["layers"], 40, 128, f["element_bytes"]) == direct


def test_opt13b_request_sizes(facts):
    per_token = oracle.kv_bytes_per_token(40, 40, 128, 2)
    a = facts["opt13b_2000_token_request"]
    assert round(per_token * a["tokens"] / 1e9, 1) == a["printed_gb"]
    b = facts["opt13b_2048_token_request"]
    assert per_token * b["tokens"] == 1_677_721_600
    assert round(per_token * b["tokens"] / 2**30, 1) == b["printed_gb"]


def test_illustrative_gqa_snippet(facts):
    f = facts["illustrative_gqa_bytes_per_token"]
    bpt = oracle.kv_bytes_per_token(f["layers"], f["kv_heads"], f["head_dim"], f["element_bytes"])
    assert bpt == f["printed_bytes"]
    assert bpt // 1024 == f["printed_kib"]
    assert bpt * f["sequence_tokens"] // 1024**2 == f["printed_mib_per_sequence"]


def test_thirty_three_tokens(facts):
    f = facts["thirty_three_token_sequence"]
    assert oracle.blocks_for_tokens(f["tokens"], f["block_size"]) == f["printed_blocks"]
    unused = oracle.unused_tail_slots(f["tokens"], f["block_size"])
    assert unused == f["printed_unused_positions"]
    assert unused * f["bytes_per_token"] / 2**20 == f["printed_tail_mib"]


def test_fragmentation_bound(facts):
    f = facts["internal_fragmentation_bound"]
    worst = max(oracle.unused_tail_slots(n, f["block_size"]) for n in range(1, 5000))
    assert worst == f["printed_max_unused"]
    assert all(oracle.unused_tail_slots(n, 16) < 16 for n in range(0, 2049))
    assert facts["default_block_size"]["printed_tokens"] == 16


def test_seven_token_prompt_reading(facts):
    f = facts["seven_token_prompt"]
    assert oracle.blocks_for_tokens(f["tokens"], f["printed_block_slots"]) == 1
    assert oracle.blocks_for_tokens(f["tokens"], 4) == f["printed_blocks"]


# ------------------------------------------------------------ attention ----

def _pool_from_contiguous(rng, ks, vs, block_size, extra_blocks=3, poison=True):
    """Scatter per-sequence contiguous K/V ([n, Hkv, d]) into a shuffled pool.

    Written from the pages' rule: logical blocks fill left to right, so
    position t is in logical block t // B at offset t % B.
    """
    hkv, d = ks[0].shape[1], ks[0].shape[2]
    counts = [-(-len(k) // block_size) for k in ks]
    nb = sum(counts) + extra_blocks
    perm = rng.permutation(nb)
    k_cache = np.full((nb, hkv, block_size, d), np.nan if poison else 0.0)
    v_cache = np.full_like(k_cache, np.nan if poison else 0.0)
    tables = np.full((len(ks), max(counts + [1])), -1, dtype=np.int64)
    cur = 0
    for s, (k, v) in enumerate(zip(ks, vs)):
        for j in range(counts[s]):
            tables[s, j] = perm[cur]
            cur += 1
        for t in range(len(k)):
            phys = tables[s, t // block_size]
            k_cache[phys, :, t % block_size, :] = k[t]
            v_cache[phys, :, t % block_size, :] = v[t]
    return k_cache, v_cache, tables


def _random_batch(seed, lens, hq, hkv, d, block_size):
    rng = np.random.default_rng(seed)
    ks = [rng.standard_normal((n, hkv, d)) for n in lens]
    vs = [rng.standard_normal((n, hkv, d)) for n in lens]
    q = rng.standard_normal((len(lens), hq, d))
    k_cache, v_cache, tables = _pool_from_contiguous(rng, ks, vs, block_size)
    return q, ks, vs, k_cache, v_cache, tables


def _brute_force(q, k_cache, v_cache, tables, lens, scale):
    """Pure-Python loops straight from softmax(q.K * scale) V."""
    S, Hq, d = q.shape
    Hkv, B = k_cache.shape[1], k_cache.shape[2]
    G = Hq // Hkv
    out = np.zeros((S, Hq, d))
    for s in range(S):
        for h in range(Hq):
            kvh = h // G
            logits = []
            for t in range(lens[s]):
                blk = tables[s][t // B]
                off = t % B
                logits.append(scale * sum(float(q[s, h, j]) * float(k_cache[blk, kvh, off, j])
                                          for j in range(d)))
            if not logits:
                continue
            mx = max(logits)
            w = [math.exp(x - mx) for x in logits]
            tot = sum(w)
            for j in range(d):
                acc = 0.0
                for t in range(lens[s]):
                    blk = tables[s][t // B]
                    acc += w[t] * float(v_cache[blk, kvh, t % B, j])
                out[s, h, j] = acc / tot
    return out


def _sdpa(q, ks, vs, scale):
    """torch's fp64 CPU scaled_dot_product_attention on contiguous K/V (GQA-aware)."""
    outs = []
    for s in range(q.shape[0]):
        qs = torch.from_numpy(q[s]).unsqueeze(0).unsqueeze(2)            # [1, Hq, 1, d]
        k = torch.from_numpy(ks[s]).permute(1, 0, 2).unsqueeze(0)         # [1, Hkv, n, d]
        v = torch.from_numpy(vs[s]).permute(1, 0, 2).unsqueeze(0)
        o = F.scaled_dot_product_attention(qs, k, v, scale=scale, enable_gqa=True)
        outs.append(o[0, :, 0, :].numpy())
    return np.stack(outs)


def test_brute_force_tiny():
    lens = [1, 5, 16, 17, 33]
    q, ks, vs, kc, vc, tables = _random_batch(11, lens, hq=4, hkv=2, d=8, block_size=4)
    scale = 0.37
    got = oracle.paged_decode_attention(q, kc, vc, tables, lens, scale)
    ref = _brute_force(q, kc, vc, tables, lens, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("hq,hkv,d,B", [(8, 8, 64, 16), (32, 8, 128, 16), (6, 2, 16, 8),
                                        (4, 1, 32, 128), (8, 2, 64, 32)])
def test_equals_unpaged_sdpa(hq, hkv, d, B):
    lens = [1, B - 1, B, B + 1, 3 * B + 5, 200]
    q, ks, vs, kc, vc, tables = _random_batch(hq * 1000 + B, lens, hq, hkv, d, B)
    scale = 1.0 / math.sqrt(d)
    got = oracle.paged_decode_attention(q, kc, vc, tables, lens, scale)
    np.testing.assert_allclose(got, _sdpa(q, ks, vs, scale), rtol=1e-10, atol=1e-12)


def test_permutation_invariance():
    lens = [7, 40, 64, 129]
    q, ks, vs, kc, vc, tables = _random_batch(3, lens, hq=8, hkv=4, d=16, block_size=16)
    base = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.25)
    rng = np.random.default_rng(99)
    pi = rng.permutation(kc.shape[0])
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    tables2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1)
    again = oracle.paged_decode_attention(q, kc2, vc2, tables2, lens, 0.25)
    assert np.array_equal(base, again)


def test_single_token_returns_its_value():
    q, ks, vs, kc, vc, tables = _random_batch(5, [1, 1], hq=4, hkv=2, d=8, block_size=16)
    out = oracle.paged_decode_attention(q, kc, vc, tables, [1, 1], 3.0)
    for s in range(2):
        for h in range(4):
            assert np.array_equal(out[s, h], vs[s][0, h // 2])


def test_zero_query_is_mean_of_values():
    lens = [3, 50]
    q, ks, vs, kc, vc, tables = _random_batch(6, lens, hq=2, hkv=2, d=8, block_size=16)
    out = oracle.paged_decode_attention(np.zeros_like(q), kc, vc, tables, lens, 1.0)
    for s in range(2):
        for h in range(2):
            np.testing.assert_allclose(out[s, h], vs[s][:, h].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_equal_keys_is_mean_of_values():
    rng = np.random.default_rng(7)
    n, d = 37, 8
    krow = rng.standard_normal((1, 1, d))
    ks = [np.repeat(krow, n, axis=0)]
    vs = [rng.standard_normal((n, 1, d))]
    kc, vc, tables = _pool_from_contiguous(rng, ks, vs, 8)
    q = rng.standard_normal((1, 1, d))
    out = oracle.paged_decode_attention(q, kc, vc, tables, [n], 0.9)
    np.testing.assert_allclose(out[0, 0], vs[0][:, 0].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_sharp_softmax_picks_argmax():
    lens = [40]
    q, ks, vs, kc, vc, tables = _random_batch(8, lens, hq=1, hkv=1, d=16, block_size=16)
    logits = ks[0][:, 0] @ q[0, 0]
    best = int(np.argmax(logits))
    out = oracle.paged_decode_attention(q, kc, vc, tables, lens, 1e4)
    np.testing.assert_allclose(out[0, 0], vs[0][best, 0], atol=1e-9)


def test_empty_context_is_zero():
    q, ks, vs, kc, vc, tables = _random_batch(9, [4, 1], hq=2, hkv=1, d=8, block_size=4)
    out = oracle.paged_decode_attention(q, kc, vc, tables, [0, 1], 1.0)
    assert np.all(out[0] == 0.0)


def test_shared_prefix_matches_unshared_copies():
    rng = np.random.default_rng(12)
    B, hkv, d = 4, 2, 8
    prefix_k = rng.standard_normal((10, hkv, d))
    prefix_v = rng.standard_normal((10, hkv, d))
    tails = [(rng.standard_normal((3, hkv, d)), rng.standard_normal((3, hkv, d))) for _ in range(2)]
    # unshared: each sample owns a full copy of the prefix
    ks = [np.concatenate([prefix_k, tk]) for tk, _ in tails]
    vs = [np.concatenate([prefix_v, tv]) for _, tv in tails]
    kc, vc, tables = _pool_from_contiguous(rng, ks, vs, B)
    q = rng.standard_normal((2, 4, d))
    ref = oracle.paged_decode_attention(q, kc, vc, tables, [13, 13], 0.5)
    # shared: both samples map the two full prefix blocks to the same physical
    # blocks; the partial third block was copied on write and then diverged.
    kc2, vc2 = kc.copy(), vc.copy()
    tables2 = tables.copy()
    tables2[1, :2] = tables[0, :2]
    kc2[tables[1, :2]] = np.nan
    vc2[tables[1, :2]] = np.nan
    got = oracle.paged_decode_attention(q, kc2, vc2, tables2, [13, 13], 0.5)
    assert np.array_equal(ref, got)


def test_positions_past_context_are_never_read():
    lens = [5, 18]
    q, ks, vs, kc, vc, tables = _random_batch(10, lens, hq=2, hkv=2, d=8, block_size=16)
    assert np.isnan(kc).any()  # unused tails and spare blocks are NaN-poisoned
    out = oracle.paged_decode_attention(q, kc, vc, tables, lens, 1.0)
    assert np.isfinite(out).all()


def test_sampled_pairs_match_full():
    lens = [9, 30, 2]
    q, ks, vs, kc, vc, tables = _random_batch(13, lens, hq=4, hkv=2, d=8, block_size=4)
    full = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.5)
    pairs = [(0, 3), (2, 0), (1, 1)]
    part = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.5, pairs=pairs)
    for s, h in pairs:
        assert np.array_equal(part[s, h], full[s, h])
    assert np.isnan(part[0, 0]).all()


# --------------------------------------- planted mistakes must be caught ----

def _mutated_attention(old, new):
    src = inspect.getsource(oracle_attention)
    assert old in src, old
    mod = types.ModuleType("mutated_attention")
    exec(compile(src.replace(old, new), "mutated_attention", "exec"), mod.__dict__)
    return mod


def _pins_pass(mod):
    """Run the brute-force, SDPA and sharp-softmax pins against ``mod``."""
    try:
        lens = [1, 5, 16, 17, 33]
        q, ks, vs, kc, vc, tables = _random_batch(11, lens, hq=4, hkv=2, d=8, block_size=4)
        got = mod.paged_decode_attention(q, kc, vc, tables, lens, 0.37)
        if not np.allclose(got, _brute_force(q, kc, vc, tables, lens, 0.37), rtol=1e-10, atol=1e-12):
            return False
        lens = [1, 15, 16, 17, 53, 200]
        q, ks, vs, kc, vc, tables = _random_batch(5, lens, 8, 2, 16, 16)
        if not np.allclose(mod.paged_decode_attention(q, kc, vc, tables, lens, 0.25),
                           _sdpa(q, ks, vs, 0.25), rtol=1e-10, atol=1e-12):
            return False
        q, ks, vs, kc, vc, tables = _random_batch(8, [40], 1, 1, 16, 16)
        best = int(np.argmax(ks[0][:, 0] @ q[0, 0]))
        out = mod.paged_decode_attention(q, kc, vc, tables, [40], 1e4)
        return bool(np.allclose(out[0, 0], vs[0][best, 0], atol=1e-9))
    except Exception:
        return False


def test_unmutated_oracle_passes_pins():
    assert _pins_pass(oracle_attention)


@pytest.mark.parametrize("old,new", [
    ("kvh = h // group", "kvh = h % num_kv_heads"),             # wrong GQA head map
    (".transpose(0, 2, 1, 3)", ".transpose(0, 1, 2, 3)"),        # tokens/heads mixed up
    ("logits = scale * (", "logits = ("),                        # dropped scale
    ("weights /= weights.sum()", "weights /= weights.max()"),    # wrong normaliser
    ("np.exp(logits - logits.max())", "np.exp(logits.max() - logits)"),  # sign flip
    ("return k[:context_len], v[:context_len]", "return k, v"),  # reads past the context
    ("ids = np.asarray(block_table_row[:n_blocks]", "ids = np.asarray(block_table_row[1:n_blocks + 1]"),
])
def test_planted_mistake_is_caught(old, new):
    assert not _pins_pass(_mutated_attention(old, new))


# ------------------------------------------------------------ cache ops ----

def test_kv_append_then_gather_reads_back():
    rng = np.random.default_rng(21)
    NB, hkv, B, d = 6, 2, 4, 8
    kc = rng.standard_normal((NB, hkv, B, d)).astype(np.float16)
    vc = rng.standard_normal((NB, hkv, B, d)).astype(np.float16)
    table = np.array([4, 1, 3])
    positions = [0, 5, 11, 6]
    slots = [table[p // B] * B + p % B for p in positions] + [-1]
    k = rng.standard_normal((5, hkv, d)).astype(np.float16)
    v = rng.standard_normal((5, hkv, d)).astype(np.float16)
    k2, v2 = oracle.kv_append(k, v, kc, vc, slots)
    kseq, vseq = oracle.gather_sequence_kv(k2, v2, table, 12)
    for i, p in enumerate(positions):
        assert np.array_equal(kseq[p], k[i].astype(np.float64))
        assert np.array_equal(vseq[p], v[i].astype(np.float64))
    changed = (k2.view(np.uint16) != kc.view(np.uint16)).reshape(NB, hkv, B, d).any(axis=(1, 3))
    assert changed.sum() <= len(positions)  # padding token (slot -1) wrote nothing
    untouched = np.ones((NB, B), bool)
    for s in slots[:-1]:
        untouched[s // B, s % B] = False
    assert np.array_equal(k2.view(np.uint16)[untouched.nonzero()[0], :, untouched.nonzero()[1]],
                          kc.view(np.uint16)[untouched.nonzero()[0], :, untouched.nonzero()[1]])


def test_block_copy_copies_exact_bytes():
    rng = np.random.default_rng(22)
    kc = rng.standard_normal((8, 2, 4, 8)).astype(np.float16)
    vc = rng.standard_normal((8, 2, 4, 8)).astype(np.float16)
    pairs = [(1, 5), (3, 0)]
    k2, v2 = oracle.block_copy(kc, vc, pairs)
    for src, dst in pairs:
        assert np.array_equal(k2[dst].view(np.uint16), kc[src].view(np.uint16))
        assert np.array_equal(v2[dst].view(np.uint16), vc[src].view(np.uint16))
    for b in (1, 2, 3, 4, 6, 7):
        assert np.array_equal(k2[b].view(np.uint16), kc[b].view(np.uint16))


# ------------------------------------------------------ chunked prompt ----

def _prefill_batch(seed, lens, chunks, hq, hkv, d, block_size):
    rng = np.random.default_rng(seed)
    ks = [rng.standard_normal((n, hkv, d)) for n in lens]
    vs = [rng.standard_normal((n, hkv, d)) for n in lens]
    kc, vc, tables = _pool_from_contiguous(rng, ks, vs, block_size)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int64)
    q = rng.standard_normal((int(qs[-1]), hq, d))
    return q, ks, vs, kc, vc, tables, qs


def _sdpa_prefill(q, ks, vs, lens, qs, scale):
    """torch SDPA with an explicit causal-with-offset mask, per sequence."""
    out = np.zeros_like(q)
    for s in range(len(lens)):
        q0, q1 = qs[s], qs[s + 1]
        n_q, n = q1 - q0, lens[s]
        if n_q == 0:
            continue
        qt = torch.from_numpy(q[q0:q1]).permute(1, 0, 2).unsqueeze(0)      # [1, Hq, L, d]
        k = torch.from_numpy(ks[s]).permute(1, 0, 2).unsqueeze(0)           # [1, Hkv, n, d]
        v = torch.from_numpy(vs[s]).permute(1, 0, 2).unsqueeze(0)
        pos = torch.arange(n - n_q, n).unsqueeze(1)
        mask = torch.arange(n).unsqueeze(0) <= pos                           # [L, n]
        o = F.scaled_dot_product_attention(qt, k, v, attn_mask=mask, scale=scale, enable_gqa=True)
        out[q0:q1] = o[0].permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("hq,hkv,d,B", [(4, 4, 16, 4), (8, 2, 32, 16), (6, 3, 8, 8)])
def test_prefill_equals_masked_sdpa(hq, hkv, d, B):
    lens = [1, 9, 33, 64, 100]
    chunks = [1, 9, 5, 64, 17]  # whole prompt, partial chunks, one token
    q, ks, vs, kc, vc, tables, qs = _prefill_batch(hq * 10 + B, lens, chunks, hq, hkv, d, B)
    got = oracle.paged_prefill_attention(q, kc, vc, tables, lens, qs, 0.3)
    np.testing.assert_allclose(got, _sdpa_prefill(q, ks, vs, lens, qs, 0.3), rtol=1e-10, atol=1e-12)


def test_prefill_whole_prompt_is_causal_attention():
    lens = [40]
    q, ks, vs, kc, vc, tables, qs = _prefill_batch(3, lens, [40], 4, 2, 16, 16)
    got = oracle.paged_prefill_attention(q, kc, vc, tables, lens, qs, 0.25)
    qt = torch.from_numpy(q).permute(1, 0, 2).unsqueeze(0)
    k = torch.from_numpy(ks[0]).permute(1, 0, 2).unsqueeze(0)
    v = torch.from_numpy(vs[0]).permute(1, 0, 2).unsqueeze(0)
    ref = F.scaled_dot_product_attention(qt, k, v, is_causal=True, scale=0.25, enable_gqa=True)
    np.testing.assert_allclose(got, ref[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_prefill_brute_force_tiny():
    lens = [7, 12]
    q, ks, vs, kc, vc, tables, qs = _prefill_batch(4, lens, [3, 5], 2, 1, 4, 4)
    got = oracle.paged_prefill_attention(q, kc, vc, tables, lens, qs, 0.7)
    for s in range(2):
        for j in range(qs[s + 1] - qs[s]):
            pos = lens[s] - (qs[s + 1] - qs[s]) + j
            for h in range(2):
                lg = [0.7 * sum(q[qs[s] + j, h, i] * ks[s][t, 0, i] for i in range(4)) for t in range(pos + 1)]
                mx = max(lg)
                w = [math.exp(x - mx) for x in lg]
                for i in range(4):
                    ref = sum(w[t] * vs[s][t, 0, i] for t in range(pos + 1)) / sum(w)
                    assert abs(got[qs[s] + j, h, i] - ref) < 1e-12


@pytest.mark.parametrize("old,new", [
    ("logits = scale * (k_seq[:pos + 1, kvh, :]", "logits = scale * (k_seq[:pos, kvh, :]"),
    ("out[q0 + j, h] = weights @ v_seq[:pos + 1, kvh, :]", "out[q0 + j, h] = weights @ v_seq[1:pos + 2, kvh, :]"),
    ("pos = ctx - n_q + j", "pos = j"),
])
def test_prefill_planted_mistake_is_caught(old, new):
    mod = _mutated_attention(old, new)
    lens = [9, 33, 64]
    q, ks, vs, kc, vc, tables, qs = _prefill_batch(12, lens, [9, 5, 17], 8, 2, 16, 16)
    try:
        got = mod.paged_prefill_attention(q, kc, vc, tables, lens, qs, 0.3)
    except Exception:
        return
    assert not np.allclose(got, _sdpa_prefill(q, ks, vs, lens, qs, 0.3), rtol=1e-8, atol=1e-10)
