"""Helpers shared by the GPU parity tests: moving seeded inputs to the oracle
and comparing within the stated tolerances."""

import numpy as np
import torch

import oracle

# |err| <= atol + rtol * |ref|, per output element, against the fp64 oracle.
TOL = {torch.float16: (4e-3, 1e-2), torch.bfloat16: (2e-2, 2e-2)}


def to_f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def oracle_decode(case, seqs=None, heads=None):
    """Oracle output for the listed sequences (all heads unless given),
    reading only the blocks those sequences map (relabelled to a small pool;
    the oracle is pinned to be invariant under such relabelling)."""
    S, Hq, D = case.q.shape
    B = case.block_size
    seqs = list(range(S)) if seqs is None else list(seqs)
    tables = case.block_tables.cpu().numpy()
    lens = case.context_lens.cpu().numpy()
    used = sorted({int(b) for s in seqs for b in tables[s, :-(-int(lens[s]) // B)]})
    remap = {b: i for i, b in enumerate(used)}
    idx = torch.tensor(used if used else [0], dtype=torch.long, device=case.k_cache.device)
    k_small = to_f64(case.k_cache.index_select(0, idx))
    v_small = to_f64(case.v_cache.index_select(0, idx))
    sub_tables = np.full((len(seqs), tables.shape[1]), -1, dtype=np.int64)
    for i, s in enumerate(seqs):
        nb = -(-int(lens[s]) // B)
        sub_tables[i, :nb] = [remap[int(b)] for b in tables[s, :nb]]
    q = to_f64(case.q[seqs])
    pairs = None
    if heads is not None:
        pairs = [(i, h) for i in range(len(seqs)) for h in heads]
    out = oracle.paged_decode_attention(q, k_small, v_small, sub_tables, lens[seqs], case.scale,
                                        pairs=pairs)
    return out


def assert_within_tol(got, ref, dtype, what=""):
    atol, rtol = TOL[dtype]
    g = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst at {i}: "
                             f"got {g[i]}, ref {ref[i]}")
    return float(err.max())


def raw_bytes(t):
    """CPU int16 view of a half/bf16 tensor, for bit-exact comparison."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy()
