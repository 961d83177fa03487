"""Pins for the pure-Python allocator model (CPU).

The strongest pin is a content model: every physical slot holds the token id
last written to it, copy-on-write copies a block's slots, and after any mix of
prompts, forks, appends, cancellations and reuse, reading each live sequence
through its block table must give back exactly that sequence's own token
history.  That is the pages' safety claim for sharing ("sharing is safe while
the shared region remains immutable"), checked without trusting the model's
own bookkeeping."""

import json
import os

import numpy as np
import pytest

from oracle import OracleAllocator, OracleOutOfBlocks, blocks_for_tokens

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


class ContentPool:
    """Slot contents of a physical pool, driven by what the allocator returns."""

    def __init__(self, num_blocks, block_size):
        self.B = block_size
        self.slots = [[None] * block_size for _ in range(num_blocks)]

    def write(self, slot, token):
        self.slots[slot // self.B][slot % self.B] = token

    def copy(self, src, dst):
        self.slots[dst] = list(self.slots[src])

    def read(self, table, n):
        return [self.slots[table[t // self.B]][t % self.B] for t in range(n)]


def _check_invariants(a: OracleAllocator):
    refs = [0] * a.num_blocks
    for table in a.tables.values():
        for b in table:
            refs[b] += 1
    assert refs == a.refcount
    assert sorted(a.free) == [b for b in range(a.num_blocks) if refs[b] == 0]
    for s, table in a.tables.items():
        assert len(table) == blocks_for_tokens(a.lengths[s], a.block_size)


def test_thirty_three_tokens_three_blocks():
    with open(GOLDEN) as f:
        fact = json.load(f)["thirty_three_token_sequence"]
    a = OracleAllocator(10, fact["block_size"])
    a.add_seq(0, fact["tokens"])
    st = a.stats()
    assert st["used_blocks"] == fact["printed_blocks"]
    assert st["used_blocks"] * 16 - st["filled_slots"] == fact["printed_unused_positions"]


def test_blocks_taken_only_when_full():
    a = OracleAllocator(64, 16)
    a.add_seq(0, 0)
    for n in range(1, 300):
        before = len(a.tables[0])
        slot, cs, cd = a.append_slot(0)
        grew = len(a.tables[0]) - before
        assert grew == (1 if (n - 1) % 16 == 0 else 0)
        assert (cs, cd) == (-1, -1)
        assert slot == a.slot_of(0, n - 1)
        assert len(a.tables[0]) == -(-n // 16)
    _check_invariants(a)


@pytest.mark.parametrize("prompt,expect_copies", [(100, 7), (96, 0), (1, 7), (16, 0)])
def test_parallel_sampling_copy_on_write(prompt, expect_copies):
    a = OracleAllocator(256, 16)
    pool = ContentPool(256, 16)
    a.add_seq(0, prompt)
    hist = {0: list(range(prompt))}
    for t in range(prompt):
        pool.write(a.slot_of(0, t), t)
    for j in range(1, 8):
        a.fork(0, j)
        hist[j] = list(hist[0])
    copies = 0
    for j in range(8):  # first divergent token of each sample, in sample order
        slot, cs, cd = a.append_slot(j)
        if cs >= 0:
            copies += 1
            pool.copy(cs, cd)
        tok = 10_000 + j
        pool.write(slot, tok)
        hist[j].append(tok)
    assert copies == expect_copies
    for j in range(8):
        assert pool.read(a.tables[j], a.lengths[j]) == hist[j]
    _check_invariants(a)
    for j in range(8):
        a.free_seq(j)
    assert len(a.free) == 256 and not any(a.refcount)


def test_out_of_blocks_leaves_state_unchanged():
    a = OracleAllocator(4, 16)
    a.add_seq(0, 40)  # 3 blocks
    snapshot = (list(a.free), list(a.refcount), {k: list(v) for k, v in a.tables.items()})
    with pytest.raises(OracleOutOfBlocks):
        a.add_seq(1, 17)  # needs 2, 1 free
    assert (list(a.free), list(a.refcount), {k: list(v) for k, v in a.tables.items()}) == snapshot
    a.fork(0, 2)
    for _ in range(8):
        a.append_slot(0)  # 40 -> 48, fills block 3 in place? shared: copy first
    with pytest.raises(OracleOutOfBlocks):
        for _ in range(100):
            a.append_slot(0)
    _check_invariants(a)


def test_free_list_reuse_order():
    a = OracleAllocator(8, 4)
    a.add_seq(0, 9)   # ids 0,1,2
    a.add_seq(1, 4)   # id 3
    a.free_seq(0)     # releases 2,1,0 -> stack top is 0
    a.add_seq(2, 5)
    assert a.tables[2] == [0, 1]


@pytest.mark.parametrize("seed", range(6))
def test_random_branching_cancellation_reuse(seed):
    """Forks, appends, cancellations and immediate reuse interleaved at random."""
    rng = np.random.default_rng(seed)
    NB, B = 48, 4
    a = OracleAllocator(NB, B)
    pool = ContentPool(NB, B)
    hist = {}
    next_id, next_tok = 0, 0
    for _ in range(600):
        op = rng.choice(["add", "fork", "append", "append", "append", "free"])
        try:
            if op == "add" or not hist:
                n = int(rng.integers(0, 3 * B))
                a.add_seq(next_id, n)
                hist[next_id] = []
                for t in range(n):
                    pool.write(a.slot_of(next_id, t), next_tok)
                    hist[next_id].append(next_tok)
                    next_tok += 1
                next_id += 1
            elif op == "fork":
                parent = int(rng.choice(list(hist)))
                a.fork(parent, next_id)
                hist[next_id] = list(hist[parent])
                next_id += 1
            elif op == "append":
                s = int(rng.choice(list(hist)))
                slot, cs, cd = a.append_slot(s)
                if cs >= 0:
                    pool.copy(cs, cd)
                # the written block is never shared at write time
                assert a.refcount[slot // B] == 1
                pool.write(slot, next_tok)
                hist[s].append(next_tok)
                next_tok += 1
            else:
                s = int(rng.choice(list(hist)))
                a.free_seq(s)
                del hist[s]
        except OracleOutOfBlocks:
            pass
        _check_invariants(a)
        for s, h in hist.items():
            assert pool.read(a.tables[s], a.lengths[s]) == h
    for s in list(hist):
        a.free_seq(s)
    assert len(a.free) == NB and not any(a.refcount)
