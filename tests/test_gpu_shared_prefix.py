"""Shared-prefix parallel sampling end to end on the GPU, and a lifecycle
stress of branching, cancellation and immediate block reuse on one stream.

Parallel sampling: 16 prompts (lengths uniform in [100, 700]) x 8 samples,
40 heads of 128, fp16, blocks of 16.  The samples of a prompt share its
physical blocks by reference count; the first divergent token copies the
partially filled last block (copy-on-write); then every step appends one
token per sample and runs decode.  Outputs must equal, bit for bit, those of
unshared per-sample caches holding the same tokens, and match the oracle on
sampled sequences, whose inputs are rebuilt on the host from the generated
tokens (never read back from the device cache)."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_247_gb300 as pkv
from paged_kv_cache_247_gb300 import workloads as W
from _gpu_util import TOL, assert_within_tol, raw_bytes

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status(lib, cuda_device):
    pkv.device_status(clear=True)
    yield
    assert pkv.device_status(clear=True) == 0


def _oracle_for(histories, q_rows, B, scale):
    """Oracle decode for sequences given by their logical K/V histories
    ([n, Hkv, D] fp64 each), laid into a fresh pool left to right."""
    counts = [-(-len(k) // B) for k, _ in histories]
    hkv, D = histories[0][0].shape[1:]
    nb = max(1, sum(counts))
    kc = np.zeros((nb, hkv, B, D))
    vc = np.zeros((nb, hkv, B, D))
    tables = np.full((len(histories), max(counts + [1])), -1, dtype=np.int64)
    cur = 0
    for s, (k, v) in enumerate(histories):
        for t in range(len(k)):
            if t % B == 0:
                tables[s, t // B] = cur
                cur += 1
            kc[tables[s, t // B], :, t % B] = k[t]
            vc[tables[s, t // B], :, t % B] = v[t]
    lens = [len(k) for k, _ in histories]
    return oracle.paged_decode_attention(np.stack(q_rows), kc, vc, tables, lens, scale)


def test_parallel_sampling_shared_prefix(cuda_device):
    w = W.SHARED_PREFIX
    H, D, B, n = w["num_kv_heads"], w["head_dim"], w["block_size"], w["samples"]
    steps = w["steps"]
    prompts = W.shared_prefix_prompts()
    num_seqs = len(prompts) * n
    seq_ids = np.arange(num_seqs, dtype=np.int64)  # prompt i, sample j -> i * n + j
    per_seq_growth = -(-steps // B) + 2
    nb_shared = int(sum(-(-int(p) // B) for p in prompts) + num_seqs * per_seq_growth)
    nb_unshared = int(sum(n * (-(-int(p) // B)) for p in prompts) + num_seqs * per_seq_growth)
    dt = W.DTYPES[w["dtype"]]
    kc = torch.zeros((nb_shared, H, B, D), dtype=dt, device=cuda_device)
    vc = torch.zeros_like(kc)
    ku = torch.zeros((nb_unshared, H, B, D), dtype=dt, device=cuda_device)
    vu = torch.zeros_like(ku)
    shared = pkv.BlockAllocator(nb_shared, B)
    model = oracle.OracleAllocator(nb_shared, B)  # the policy, checked id for id
    unshared = pkv.BlockAllocator(nb_unshared, B)

    watch = [0, 1, 7, 8 * 5 + 3, num_seqs - 1]  # sampled sequences checked by the oracle
    hist = {s: [[], []] for s in watch}
    for i, p in enumerate(prompts.tolist()):
        pk, pv = W.new_tokens(1000 + i, p, H, D, w["dtype"], device=cuda_device)
        shared.add_seq(i * n, p)
        model.add_seq(i * n, p)
        slots = torch.from_numpy(shared.seq_slots(i * n, 0, p)).to(cuda_device)
        pkv.kv_append(pk, pv, kc, vc, slots)
        for j in range(1, n):
            shared.fork(i * n, i * n + j)
            model.fork(i * n, i * n + j)
        for j in range(n):
            unshared.add_seq(i * n + j, p)
            slots_u = torch.from_numpy(unshared.seq_slots(i * n + j, 0, p)).to(cuda_device)
            pkv.kv_append(pk, pv, ku, vu, slots_u)
            if i * n + j in watch:
                hist[i * n + j][0].append(pk.double().cpu().numpy())
                hist[i * n + j][1].append(pv.double().cpu().numpy())
    st = shared.stats()
    assert st["shared_blocks"] == sum(-(-int(p) // B) for p in prompts)

    lens = prompts.repeat(n).astype(np.int64)
    q_gen = torch.Generator(device=cuda_device).manual_seed(7)
    total_copies = 0
    max_blocks = -(-int(lens.max() + steps) // B)
    for step in range(steps):
        slots, pairs = shared.append_slots(seq_ids)
        want_pairs = []
        for s, slot in zip(seq_ids.tolist(), slots.tolist()):
            want_slot, cs, cd = model.append_slot(s)
            assert slot == want_slot
            if cs >= 0:
                want_pairs.append([cs, cd])
        assert pairs.tolist() == want_pairs
        slots_u, pairs_u = unshared.append_slots(seq_ids)
        assert len(pairs_u) == 0
        if len(pairs):
            assert step == 0  # only the first divergent token copies
            total_copies += len(pairs)
            pkv.block_copy(kc, vc, torch.from_numpy(pairs).to(cuda_device))
        k_new, v_new = W.new_tokens(5000 + step, num_seqs, H, D, w["dtype"], device=cuda_device)
        pkv.kv_append(k_new, v_new, kc, vc, torch.from_numpy(slots).to(cuda_device))
        pkv.kv_append(k_new, v_new, ku, vu, torch.from_numpy(slots_u).to(cuda_device))
        lens += 1
        q = torch.randn((num_seqs, H, D), generator=q_gen, device=cuda_device).to(dt)
        t_sh = torch.from_numpy(shared.block_table(seq_ids, max_blocks)).to(cuda_device)
        t_un = torch.from_numpy(unshared.block_table(seq_ids, max_blocks)).to(cuda_device)
        ctx = torch.from_numpy(lens.astype(np.int32)).to(cuda_device)
        out_sh = torch.empty_like(q)
        out_un = torch.empty_like(q)
        mctx = int(lens.max())
        pkv.paged_attn_decode(out_sh, q, kc, vc, t_sh, ctx, D ** -0.5, mctx)
        pkv.paged_attn_decode(out_un, q, ku, vu, t_un, ctx, D ** -0.5, mctx)
        for s in watch:
            hist[s][0].append(k_new[s:s + 1].double().cpu().numpy())
            hist[s][1].append(v_new[s:s + 1].double().cpu().numpy())
        assert torch.equal(out_sh, out_un), f"shared != unshared at step {step}"
        if step in (0, 1, steps // 2, steps - 1):
            histories = [(np.concatenate(hist[s][0]), np.concatenate(hist[s][1])) for s in watch]
            ref = _oracle_for(histories, [q[s].double().cpu().numpy() for s in watch], B, D ** -0.5)
            assert_within_tol(out_sh[watch], ref, dt, f"step {step}")
        if step == 0:
            # cache bytes of the watched sequences, read through their tables,
            # equal the generated tokens exactly (prompt + first new token)
            tab = t_sh.cpu().numpy()
            kb = raw_bytes(kc)
            for s in watch:
                L = int(lens[s])
                rows = np.stack([kb[tab[s, t // B], :, t % B] for t in range(L)])
                want = np.concatenate(hist[s][0]).astype(np.float16).view(np.int16)
                assert np.array_equal(rows, want)
    expect = sum(n - 1 for p in prompts.tolist() if p % B)
    assert total_copies == expect
    assert shared.stats()["cow_copies"] == expect
    for s in seq_ids.tolist():
        shared.free_seq(s)
        unshared.free_seq(s)
    assert shared.stats()["free_blocks"] == nb_shared
    assert unshared.stats()["free_blocks"] == nb_unshared


def test_branch_cancel_reuse_on_one_stream(cuda_device):
    """Forks, appends, cancellations and immediate reuse of freed blocks, all
    enqueued on one stream with no host synchronisation; outputs are checked
    against the oracle afterwards."""
    H, D, B, NB = 4, 64, 8, 96
    rng = np.random.default_rng(11)
    torch.manual_seed(11)
    kc = torch.zeros((NB, H, B, D), dtype=torch.bfloat16, device=cuda_device)
    vc = torch.zeros_like(kc)
    alloc = pkv.BlockAllocator(NB, B)
    hist = {}
    keep = []   # host buffers that must outlive their async copies
    checks = []
    next_id, tok_seed = 0, 0

    def h2d(arr):
        t = arr if isinstance(arr, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(arr))
        t = t.contiguous().pin_memory()
        keep.append(t)
        return t.to(cuda_device, non_blocking=True)

    for step in range(150):
        op = rng.choice(["add", "fork", "free", "decode", "decode"])
        if op == "add" or not hist:
            n = int(rng.integers(1, 40))
            try:
                alloc.add_seq(next_id, n)
            except pkv.OutOfBlocks:
                continue
            k, v = W.new_tokens(tok_seed, n, H, D, "bf16")  # host tensors
            tok_seed += 1
            pkv.kv_append(h2d(k), h2d(v), kc, vc, h2d(alloc.seq_slots(next_id, 0, n)))
            hist[next_id] = [k.double().numpy(), v.double().numpy()]
            next_id += 1
        elif op == "fork":
            parent = int(rng.choice(list(hist)))
            alloc.fork(parent, next_id)
            hist[next_id] = [hist[parent][0].copy(), hist[parent][1].copy()]
            next_id += 1
        elif op == "free":
            s = int(rng.choice(list(hist)))
            alloc.free_seq(s)  # blocks may be handed out by the very next op
            del hist[s]
        else:
            seqs = sorted(hist)
            try:
                slots, pairs = alloc.append_slots(seqs)
            except pkv.OutOfBlocks:
                continue
            if len(pairs):
                pkv.block_copy(kc, vc, h2d(pairs))
            k, v = W.new_tokens(tok_seed, len(seqs), H, D, "bf16")
            tok_seed += 1
            pkv.kv_append(h2d(k), h2d(v), kc, vc, h2d(slots))
            kh, vh = k.double().numpy(), v.double().numpy()
            for i, s in enumerate(seqs):
                hist[s][0] = np.concatenate([hist[s][0], kh[i:i + 1]])
                hist[s][1] = np.concatenate([hist[s][1], vh[i:i + 1]])
            lens = np.array([len(hist[s][0]) for s in seqs], dtype=np.int32)
            mb = int(-(-lens.max() // B))
            tables = alloc.block_table(seqs, mb)
            q_host = torch.randn((len(seqs), 2 * H, D)).to(torch.bfloat16)
            q = h2d(q_host)
            out = torch.empty_like(q)
            pkv.paged_attn_decode(out, q, kc, vc, h2d(tables), h2d(lens), 0.125, int(lens.max()),
                                  partition_size=32)
            checks.append((out, q_host, [(hist[s][0].copy(), hist[s][1].copy()) for s in seqs]))
    torch.cuda.synchronize()
    assert len(checks) > 20
    for out, q, histories in checks:
        ref = _oracle_for(histories, list(q.double().numpy()), B, 0.125)
        assert_within_tol(out, ref, torch.bfloat16, "lifecycle")
    for s in list(hist):
        alloc.free_seq(s)
    assert alloc.stats()["free_blocks"] == NB
