"""Pure-Python model of the refcounted block allocator (oracle, test infrastructure).

The mechanism, as the pages describe it:

* fixed-size blocks, a per-sequence block table from logical to physical
  blocks, allocation on demand: a new physical block is taken only when all
  earlier blocks are full ("Only 20.4% of your KV cache held actual tokens",
  section "The page table, relocated into attention"; "800 kilobytes per
  token", section "The old answer, imported honestly");
* sharing by reference count: forked samples map their prompt blocks to the
  same physical blocks; when a sequence writes into a shared, partially
  filled block it gets a fresh block, one block of data is copied and the
  old block's count drops by one (copy-on-write); dead sequences just drop
  their counts and blocks that reach zero return to the pool ("Only 20.4%
  ...", section "The part everyone forgets: pages enable sharing, not just
  packing"; "The KV cache is a systems problem", section "Shared prefixes
  need ownership rules").

Policy details the pages leave open, fixed here so that the native allocator
can be compared with this model id for id:

* the free list is a LIFO stack that initially hands out ids 0, 1, 2, ...;
* a sequence's blocks are released from its last logical block to its first;
* copy-on-write happens iff the write position is inside the last block
  (position % B != 0) and that block's count is above one; a write at a block
  boundary takes a fresh block and copies nothing;
* running out of blocks raises and leaves the state unchanged; a batch of
  appends is all or nothing.
"""


class OracleOutOfBlocks(RuntimeError):
    pass


class OracleAllocator:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(range(num_blocks - 1, -1, -1))  # pop() yields 0 first
        self.refcount = [0] * num_blocks
        self.tables = {}   # seq_id -> list of physical ids
        self.lengths = {}  # seq_id -> tokens held
        self.cow_copies = 0

    # -- helpers ---------------------------------------------------------
    def _take(self):
        block = self.free.pop()
        assert self.refcount[block] == 0
        self.refcount[block] = 1
        return block

    # -- operations ------------------------------------------------------
    def add_seq(self, seq_id: int, num_tokens: int):
        """Admit a sequence holding ``num_tokens`` positions (a prompt)."""
        if seq_id in self.tables:
            raise KeyError(f"sequence {seq_id} exists")
        need = -(-num_tokens // self.block_size)
        if need > len(self.free):
            raise OracleOutOfBlocks(need)
        self.tables[seq_id] = [self._take() for _ in range(need)]
        self.lengths[seq_id] = num_tokens

    def fork(self, parent: int, child: int):
        """Child shares every block of the parent (refcount + 1 each)."""
        if child in self.tables:
            raise KeyError(f"sequence {child} exists")
        table = list(self.tables[parent])
        for block in table:
            self.refcount[block] += 1
        self.tables[child] = table
        self.lengths[child] = self.lengths[parent]

    def append_slot(self, seq_id: int):
        """Reserve the slot of the sequence's next token.

        Returns ``(slot, cow_src, cow_dst)`` with ``cow_src = cow_dst = -1``
        when no block has to be copied.
        """
        table = self.tables[seq_id]
        pos = self.lengths[seq_id]
        offset = pos % self.block_size
        cow_src = cow_dst = -1
        if offset == 0:
            if not self.free:
                raise OracleOutOfBlocks(1)
            table.append(self._take())
        else:
            last = table[-1]
            if self.refcount[last] > 1:
                if not self.free:
                    raise OracleOutOfBlocks(1)
                fresh = self._take()
                self.refcount[last] -= 1
                table[-1] = fresh
                cow_src, cow_dst = last, fresh
                self.cow_copies += 1
        self.lengths[seq_id] = pos + 1
        return table[-1] * self.block_size + offset, cow_src, cow_dst

    def append_slots(self, seq_ids):
        """append_slot for each sequence in order, all or nothing.

        Returns ``(slots, pairs)``; if any append fails the allocator is
        restored to its state before the call and the error is raised.
        """
        saved = (list(self.free), list(self.refcount),
                 {k: list(v) for k, v in self.tables.items()}, dict(self.lengths),
                 self.cow_copies)
        slots, pairs = [], []
        try:
            for s in seq_ids:
                slot, src, dst = self.append_slot(s)
                slots.append(slot)
                if src >= 0:
                    pairs.append([src, dst])
        except Exception:
            (self.free, self.refcount, self.tables, self.lengths, self.cow_copies) = saved
            raise
        return slots, pairs

    def free_seq(self, seq_id: int):
        """Drop the sequence; blocks whose count reaches zero are reusable."""
        table = self.tables.pop(seq_id)
        del self.lengths[seq_id]
        for block in reversed(table):
            self.refcount[block] -= 1
            assert self.refcount[block] >= 0
            if self.refcount[block] == 0:
                self.free.append(block)

    # -- queries ---------------------------------------------------------
    def slot_of(self, seq_id: int, position: int) -> int:
        table = self.tables[seq_id]
        return table[position // self.block_size] * self.block_size + position % self.block_size

    def block_table(self, seq_ids, max_blocks: int):
        rows = []
        for s in seq_ids:
            table = self.tables[s]
            if len(table) > max_blocks:
                raise ValueError("table longer than max_blocks")
            rows.append(table + [-1] * (max_blocks - len(table)))
        return rows

    def stats(self):
        used = [b for b in range(self.num_blocks) if self.refcount[b] > 0]
        fill = {}
        for s, table in self.tables.items():
            n = self.lengths[s]
            for i, block in enumerate(table):
                filled = min(self.block_size, n - i * self.block_size)
                fill[block] = max(fill.get(block, 0), filled)
        filled_slots = sum(fill.values())
        return {
            "num_blocks": self.num_blocks,
            "free_blocks": len(self.free),
            "used_blocks": len(used),
            "shared_blocks": sum(1 for b in used if self.refcount[b] > 1),
            "num_seqs": len(self.tables),
            "logical_tokens": sum(self.lengths.values()),
            "filled_slots": filled_slots,
            "cow_copies": self.cow_copies,
        }
