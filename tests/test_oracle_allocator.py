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


# ------------------------------------------- batched, all-or-nothing appends --
#
# append_slots is the batched form of append_slot ("Only 20.4% of your KV
# cache held actual tokens", section "The part everyone forgets: pages enable
# sharing, not just packing": a step reserves each sequence's next slot and
# copies a shared partial block first; "The KV cache is a systems problem",
# section "Shared prefixes need ownership rules").  Its pins do not trust its
# own snapshot: a successful batch must act exactly like the same appends made
# one at a time (state compared field by field, contents through the slot
# model), and a failed batch must leave every field equal to a deep copy taken
# before the call.

import copy
import inspect
import types

import oracle.allocator as oracle_allocator_module


def _state(a):
    return (list(a.free), list(a.refcount), {k: list(v) for k, v in a.tables.items()},
            dict(a.lengths), a.cow_copies)


def _shared_setup(cls, num_blocks=64, block_size=4):
    """Two prompts, each forked, with partly filled last blocks (copy-on-write
    pending) and one prompt that ends on a block boundary."""
    a = cls(num_blocks, block_size)
    pool = ContentPool(num_blocks, block_size)
    hist = {}
    tok = 0
    for sid, n in ((0, 6), (2, 8), (4, 3)):
        a.add_seq(sid, n)
        hist[sid] = []
        for t in range(n):
            pool.write(a.slot_of(sid, t), tok)
            hist[sid].append(tok)
            tok += 1
    for parent, child in ((0, 1), (2, 3), (4, 5), (4, 6)):
        a.fork(parent, child)
        hist[child] = list(hist[parent])
    return a, pool, hist


def _batch_matches_single_appends(cls):
    """A batch equals the same append_slot calls one by one, and its slots and
    pairs keep every sequence's history intact in the slot model."""
    a, pool, hist = _shared_setup(cls)
    b = copy.deepcopy(a)
    order = [1, 0, 5, 3, 2, 6, 4]
    tok = 1000
    for rnd in range(6):  # crosses block boundaries and later copy-on-writes
        slots, pairs = a.append_slots(order)
        single_slots, single_pairs = [], []
        for s in order:
            slot, cs, cd = oracle_allocator_module.OracleAllocator.append_slot(b, s)
            single_slots.append(slot)
            if cs >= 0:
                single_pairs.append([cs, cd])
        if list(slots) != single_slots or [list(p) for p in pairs] != single_pairs:
            return False
        if _state(a) != _state(b):
            return False
        for src, dst in pairs:  # copies first, then the step's writes
            pool.copy(src, dst)
        for s, slot in zip(order, slots):
            pool.write(slot, tok)
            hist[s].append(tok)
            tok += 1
        for s, h in hist.items():
            if pool.read(a.tables[s], a.lengths[s]) != h:
                return False
        if rnd == 0 and len(pairs) != 3:  # 0/1 and 4/5/6 share partial blocks
            return False
    return True


def _failed_batch_restores(cls):
    """Pool exhausted at the k-th sequence, and an unknown id last: the error
    is raised and every field equals a deep copy taken before the call."""
    # (1) exhausted: two free blocks, the third sequence needs one more
    a = cls(6, 4)
    for sid in range(4):
        a.add_seq(sid, 4)  # blocks 0..3, each full
    a.free_seq(1)
    a.free_seq(3)          # free stack [5, 4, 1, 3]: pops 3, 1, 4, 5
    a.add_seq(4, 5)        # blocks 3, 1, the last one partly filled ...
    a.fork(4, 5)           # ... and shared, so seq 4 copies on its next write
    snap = copy.deepcopy(_state(a))
    if snap[0] != [5, 4] or snap[4] != 0:
        return False
    try:
        a.append_slots([4, 0, 2])  # 4 copies (takes 4), 0 takes 5, 2 finds none
        return False
    except OracleOutOfBlocks:
        pass
    if _state(a) != snap:
        return False
    # (2) a larger pool: copy-on-write and fresh blocks happen, then an
    # unknown sequence id ends the batch
    a, _, _ = _shared_setup(cls, num_blocks=12)
    for s in (0, 1, 4):  # consume and return a few blocks so the stack is out of order
        a.append_slots([s])
    a.free_seq(6)
    a.add_seq(7, 4)
    a.free_seq(7)
    snap = copy.deepcopy(_state(a))
    try:
        a.append_slots([5, 2, 3, 0, 99])
        return False
    except KeyError:
        pass
    if _state(a) != snap:
        return False
    # (3) exhausted by a copy-on-write: nothing changes, not even the count
    a = cls(3, 4)
    a.add_seq(0, 5)
    a.fork(0, 1)
    a.add_seq(2, 1)
    snap = copy.deepcopy(_state(a))
    try:
        a.append_slots([2, 0])  # 2 writes in place, 0 needs a copy: none free
        return False
    except OracleOutOfBlocks:
        pass
    return _state(a) == snap


def _batch_pins_pass(cls):
    # each planted mistake must make a pin return False, not crash it
    return _batch_matches_single_appends(cls) and _failed_batch_restores(cls)


def test_batch_pins_hold_for_the_oracle():
    assert _batch_matches_single_appends(OracleAllocator)
    assert _failed_batch_restores(OracleAllocator)


def test_failed_batch_stack_is_out_of_order():
    """The second failure case starts from a free stack of several distinct
    ids, so a restore in the wrong order changes it."""
    a, _, _ = _shared_setup(OracleAllocator, num_blocks=12)
    for s in (0, 1, 4):
        a.append_slots([s])
    a.free_seq(6)
    a.add_seq(7, 4)
    a.free_seq(7)
    assert len(a.free) >= 2 and a.free != list(reversed(a.free))


def _mutated_allocator(old, new):
    src = inspect.getsource(oracle_allocator_module)
    assert old in src, old
    mod = types.ModuleType("mutated_allocator")
    exec(compile(src.replace(old, new), "mutated_allocator", "exec"), mod.__dict__)
    # raise the same exception class as the real model, so that the pins see
    # the mutant's errors exactly as they see the oracle's
    mod.OracleOutOfBlocks = OracleOutOfBlocks
    return mod.OracleAllocator


@pytest.mark.parametrize("old,new", [
    # the copy-on-write count is not restored
    ("(self.free, self.refcount, self.tables, self.lengths, self.cow_copies) = saved",
     "(self.free, self.refcount, self.tables, self.lengths, _) = saved"),
    # the free stack comes back in the wrong order
    ("saved = (list(self.free),", "saved = (list(reversed(self.free)),"),
    # the tables are saved by reference, so appended blocks survive the restore
    ("{k: list(v) for k, v in self.tables.items()}, dict(self.lengths)",
     "dict(self.tables), dict(self.lengths)"),
    # not all or nothing: the appends before the failure stay
    ("(self.free, self.refcount, self.tables, self.lengths, self.cow_copies) = saved\n",
     "pass\n"),
    # copy pairs reported backwards
    ("pairs.append([src, dst])", "pairs.append([dst, src])"),
    # a batch that skips the copy-on-write bookkeeping of the last sequence
    ("for s in seq_ids:", "for s in list(seq_ids)[:-1]:"),
])
def test_batch_planted_mistake_is_caught(old, new):
    assert not _batch_pins_pass(_mutated_allocator(old, new))
