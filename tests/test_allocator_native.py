"""The native block allocator against the oracle's pure-Python model: the
same random mix of prompts, forks, appends, cancellations and reuse must give
the same ids, slots, copy-on-write pairs, tables, counts and errors."""

import numpy as np
import pytest

from oracle import OracleAllocator, OracleOutOfBlocks


@pytest.fixture
def native(lib):
    from paged_kv_cache_247_gb300 import BlockAllocator, OutOfBlocks
    return BlockAllocator, OutOfBlocks


def _same_state(nat, ora, live):
    for s in live:
        n, b = nat.seq_info(s)
        assert n == ora.lengths[s] and b == len(ora.tables[s])
    if live:
        mb = max(len(ora.tables[s]) for s in live) + 1
        assert nat.block_table(sorted(live), mb).tolist() == ora.block_table(sorted(live), mb)
    for blk in range(ora.num_blocks):
        assert nat.refcount(blk) == ora.refcount[blk]
    assert nat.stats() == ora.stats()


def test_thirty_three_tokens(native):
    BlockAllocator, _ = native
    a = BlockAllocator(16, 16)
    a.add_seq(7, 33)
    st = a.stats()
    assert st["used_blocks"] == 3 and st["used_blocks"] * 16 - st["filled_slots"] == 15
    assert a.seq_slots(7, 0, 33).tolist() == [t for t in range(33)]  # ids 0,1,2 in order


@pytest.mark.parametrize("seed", range(5))
def test_matches_oracle_model(native, seed):
    BlockAllocator, OutOfBlocks = native
    rng = np.random.default_rng(100 + seed)
    NB, B = 40, 8
    nat, ora = BlockAllocator(NB, B), OracleAllocator(NB, B)
    live, next_id = [], 0
    for step in range(500):
        op = rng.choice(["add", "fork", "append", "append", "batch", "free"])
        if op == "add" or not live:
            n = int(rng.integers(0, 4 * B))
            try:
                ora.add_seq(next_id, n)
                ok = True
            except OracleOutOfBlocks:
                ok = False
            if ok:
                nat.add_seq(next_id, n)
                live.append(next_id)
            else:
                with pytest.raises(OutOfBlocks):
                    nat.add_seq(next_id, n)
            next_id += 1
        elif op == "fork":
            parent = int(rng.choice(live))
            ora.fork(parent, next_id)
            nat.fork(parent, next_id)
            live.append(next_id)
            next_id += 1
        elif op == "append":
            s = int(rng.choice(live))
            try:
                want = ora.append_slot(s)
            except OracleOutOfBlocks:
                want = None
            if want is None:
                with pytest.raises(OutOfBlocks):
                    nat.append_slot(s)
            else:
                assert nat.append_slot(s) == want
        elif op == "batch":
            seqs = [int(x) for x in rng.choice(live, size=min(len(live), 4), replace=False)]
            try:
                want_slots, want_pairs = ora.append_slots(seqs)
                failed = False
            except OracleOutOfBlocks:
                failed = True
            if failed:
                with pytest.raises(OutOfBlocks):
                    nat.append_slots(seqs)
            else:
                slots, pairs = nat.append_slots(seqs)
                assert slots.tolist() == want_slots
                assert pairs.tolist() == want_pairs
        else:
            s = int(rng.choice(live))
            ora.free_seq(s)
            nat.free_seq(s)
            live.remove(s)
        if step % 25 == 0:
            _same_state(nat, ora, live)
    _same_state(nat, ora, live)
    for s in live:
        nat.free_seq(s)
    st = nat.stats()
    assert st["free_blocks"] == NB and st["used_blocks"] == 0  # everything reclaimed


def test_errors(native, lib):
    BlockAllocator, OutOfBlocks = native
    from paged_kv_cache_247_gb300 import PagedKVError
    a = BlockAllocator(4, 16)
    a.add_seq(1, 10)
    with pytest.raises(PagedKVError):
        a.add_seq(1, 3)     # exists
    with pytest.raises(PagedKVError):
        a.fork(9, 10)       # unknown parent
    with pytest.raises(PagedKVError):
        a.free_seq(42)
    with pytest.raises(PagedKVError):
        a.block_table([1], 0)  # row too small
    with pytest.raises(OutOfBlocks):
        a.add_seq(2, 100)
    assert a.stats()["used_blocks"] == 1
