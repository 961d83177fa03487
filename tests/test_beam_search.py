"""Beam search on the paged cache: beams share every block up to their
divergence point, the sharing pattern changes every step as beams are kept
or dropped, dead beams only release their references, and a surviving beam
copies at most one block ("Only 20.4% of your KV cache held actual tokens",
section "The part everyone forgets: pages enable sharing, not just packing").

The CPU part drives the native allocator and the oracle model through the
same beam schedule; the GPU part runs decode over the beams and checks it
against the oracle, with each beam's inputs rebuilt from its token history."""

import numpy as np
import pytest
import torch

import oracle


def beam_schedule(seed, width, steps, prompt_len):
    """Synthetic beam search: each step every live beam proposes two
    continuations with random scores and the best `width` survive."""
    rng = np.random.default_rng(seed)
    plan = []
    for _ in range(steps):
        scores = rng.random((width, 2))
        order = np.argsort(-scores.ravel())[:width]
        plan.append([int(o // 2) for o in order])  # parent beam index of each survivor
    return plan


def run_beams(alloc, plan, width, prompt_len, on_step=None):
    """Apply the schedule to an allocator with the native/oracle interface.

    Returns per-step lists of (copy pairs, live beam ids)."""
    alloc.add_seq(0, prompt_len)
    beams = [0]
    for j in range(1, width):  # initial beams share the whole prompt
        alloc.fork(0, j)
        beams.append(j)
    next_id = width
    history = []
    for parents in plan:
        new_beams = []
        for p in parents:
            alloc.fork(beams[p], next_id)
            new_beams.append(next_id)
            next_id += 1
        for b in beams:  # dropped and superseded beams release their blocks
            alloc.free_seq(b)
        beams = new_beams
        slots, pairs = alloc.append_slots(beams)
        history.append((np.asarray(pairs).reshape(-1, 2), list(beams), list(slots)))
        if on_step is not None:
            on_step(beams, slots, pairs)
    return beams, history


@pytest.mark.parametrize("prompt_len", [37, 48])
def test_beam_sharing_and_copy_bound(lib, prompt_len):
    from paged_kv_cache_247_gb300 import BlockAllocator
    width, steps, B, NB = 4, 60, 16, 64
    plan = beam_schedule(prompt_len, width, steps, prompt_len)
    nat, model = BlockAllocator(NB, B), oracle.OracleAllocator(NB, B)
    beams_n, hist_n = run_beams(nat, plan, width, prompt_len)
    beams_m, hist_m = run_beams(model, plan, width, prompt_len)
    for (pn, bn, sn), (pm, bm, sm) in zip(hist_n, hist_m):
        assert pn.tolist() == pm.tolist() and sn == list(sm)
        # at most one block copied per surviving beam and step
        assert len(pn) <= width
        assert len(set(pn[:, 1].tolist())) == len(pn)
    st = nat.stats()
    assert st == model.stats()
    # sharing: the beams hold far fewer blocks than unshared copies would
    unshared = width * -(-(prompt_len + steps) // B)
    assert st["used_blocks"] < unshared
    for b in beams_n:
        nat.free_seq(b)
        model.free_seq(b)
    assert nat.stats()["free_blocks"] == NB and model.stats()["free_blocks"] == NB


@pytest.mark.gpu
def test_beam_decode_on_gpu(lib, cuda_device):
    import paged_kv_cache_247_gb300 as pkv
    from paged_kv_cache_247_gb300 import workloads as W
    from _gpu_util import assert_within_tol
    width, steps, B, NB, H, D = 4, 40, 16, 96, 8, 128
    prompt_len = 45
    plan = beam_schedule(7, width, steps, prompt_len)
    kc = torch.zeros((NB, H, B, D), dtype=torch.float16, device=cuda_device)
    vc = torch.zeros_like(kc)
    alloc = pkv.BlockAllocator(NB, B)
    pk, pv = W.new_tokens(70, prompt_len, H, D, "fp16")
    alloc.add_seq(0, prompt_len)
    pkv.kv_append(pk.to(cuda_device), pv.to(cuda_device), kc, vc,
                  torch.from_numpy(alloc.seq_slots(0, 0, prompt_len)).to(cuda_device))
    hist = {0: (pk.double().numpy(), pv.double().numpy())}
    beams = [0]
    for j in range(1, width):
        alloc.fork(0, j)
        hist[j] = hist[0]
        beams.append(j)
    next_id = width
    pkv.device_status(clear=True)
    for step, parents in enumerate(plan):
        new_beams = []
        for p in parents:
            alloc.fork(beams[p], next_id)
            hist[next_id] = hist[beams[p]]
            new_beams.append(next_id)
            next_id += 1
        for b in beams:
            alloc.free_seq(b)
            del hist[b]
        beams = new_beams
        slots, pairs = alloc.append_slots(beams)
        if len(pairs):
            pkv.block_copy(kc, vc, torch.from_numpy(pairs).to(cuda_device))
        k, v = W.new_tokens(1000 + step, width, H, D, "fp16")
        pkv.kv_append(k.to(cuda_device), v.to(cuda_device), kc, vc,
                      torch.from_numpy(slots).to(cuda_device))
        for i, b in enumerate(beams):
            hist[b] = (np.concatenate([hist[b][0], k[i:i + 1].double().numpy()]),
                       np.concatenate([hist[b][1], v[i:i + 1].double().numpy()]))
        lens = np.array([len(hist[b][0]) for b in beams], dtype=np.int32)
        tables = alloc.block_table(beams, -(-int(lens.max()) // B))
        q = torch.randn((width, 2 * H, D), generator=torch.Generator().manual_seed(step)).half()
        out = torch.empty_like(q, device=cuda_device)
        pkv.paged_attn_decode(out, q.to(cuda_device), kc, vc, torch.from_numpy(tables).to(cuda_device),
                              torch.from_numpy(lens).to(cuda_device), D ** -0.5, int(lens.max()))
        if step % 10 == 9:
            # oracle over each beam's own history, laid out contiguously
            nb = [-(-int(n) // B) for n in lens]
            pool_k = np.zeros((sum(nb), H, B, D))
            pool_v = np.zeros_like(pool_k)
            tab = np.full((width, max(nb)), -1)
            cur = 0
            for i, b in enumerate(beams):
                for t in range(lens[i]):
                    if t % B == 0:
                        tab[i, t // B] = cur
                        cur += 1
                    pool_k[tab[i, t // B], :, t % B] = hist[b][0][t]
                    pool_v[tab[i, t // B], :, t % B] = hist[b][1][t]
            ref = oracle.paged_decode_attention(q.double().numpy(), pool_k, pool_v, tab, lens,
                                                D ** -0.5)
            assert_within_tol(out, ref, torch.float16, f"beam step {step}")
    assert pkv.device_status(clear=True) == 0
    for b in beams:
        alloc.free_seq(b)
    assert alloc.stats()["free_blocks"] == NB
