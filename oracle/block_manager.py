"""Oracle: the host-side block manager that produces block tables.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The rules, as the pages state them:

* Pool and free list.  [P1] "How PagedAttention works" step 1 and step 5,
  [P2] "Concrete example: serving a chat workload": physical blocks are handed
  out from a free list and go back to it when a request finishes.  The [P1]
  practice block manager takes the block at the FRONT of the free list; the
  order in which released blocks re-enter the list is not stated.  Reading
  adopted: FIFO -- take from the front, return to the back, in table order.
  The creator may give the initial order explicitly, which is how both of
  [P1]'s worked examples (the practice run, which starts from 0..7, and the
  paged_vs_contiguous.py run, which pops from the end of a permutation) are
  reproduced.
* Reference counts.  [P1] "Memory sharing across requests": every block counts
  the sequences that use it.
* Append one token.  [P1] "How PagedAttention works" steps 1-3 and the
  practice listing: if the sequence has no block yet, or its last block is
  full, take a fresh block; otherwise, if the last block is shared (count > 1),
  copy-on-write: take a fresh block, give it the old block's fill, repoint the
  table, lower the old block's count; then the token takes the next slot of
  the last block.  A full shared block is never written again ([P1] "Memory
  sharing across requests": full prompt blocks are never written), so it never
  needs a copy.
* Fork.  [P1] practice listing and "Memory sharing across requests": the child
  gets a copy of the parent's table, partial last block included, and every
  block's count goes up by one.  ([P2]'s fork_block_table sketch shares only
  the full blocks and drops the partial tail's tokens; it is garbled and not
  followed -- see the design doc.)
* Release.  [P1] practice exercise 3 and the "Fifty chats" question: every
  block's count goes down by one; blocks reaching zero go back on the free
  list, others stay.

Failure: when the free list cannot supply every block an operation needs, the
operation raises OutOfBlocks and changes nothing ([P1] "Worked example": memory
can run out in the middle of generation; what to do then is the scheduler's
policy, outside this component).

Slots: a token's slot is physical_block * block_size + offset, offset being its
position inside the block.
"""

from collections import deque


class OutOfBlocks(RuntimeError):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks, block_size, initial_free_order=None):
        if initial_free_order is None:
            initial_free_order = range(num_blocks)
        order = [int(b) for b in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("initial free order must be a permutation of the pool")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = deque(order)
        self.refs = [0] * num_blocks      # sequences using each block
        self.fill = [0] * num_blocks      # token slots written in each block
        self.tables = {}                  # seq id -> list of physical blocks
        self.next_seq = 0

    # -- queries -----------------------------------------------------------
    def num_free(self):
        return len(self.free)

    def seq_len(self, seq):
        table = self.tables[seq]
        if not table:
            return 0
        return (len(table) - 1) * self.block_size + self.fill[table[-1]]

    def blocks_in_use(self):
        return sum(1 for r in self.refs if r > 0)

    # -- operations ----------------------------------------------------------
    def new_seq(self):
        seq = self.next_seq
        self.next_seq += 1
        self.tables[seq] = []
        return seq

    def _take_free_block(self):
        blk = self.free.popleft()
        self.refs[blk] = 1
        self.fill[blk] = 0
        return blk

    def _blocks_needed(self, seq, n):
        """Fresh blocks that appending n tokens to seq will take."""
        table = self.tables[seq]
        need = 0
        room = 0
        if table:
            last = table[-1]
            room = self.block_size - self.fill[last]
            if room > 0 and self.refs[last] > 1 and n > 0:
                need += 1                      # copy-on-write of the last block
        overflow = max(0, n - room)
        need += -(-overflow // self.block_size)
        return need

    def append_token(self, seq):
        """Append one token; returns (slot, cow) with cow = (src, dst) or None."""
        if self._blocks_needed(seq, 1) > len(self.free):
            raise OutOfBlocks(f"seq {seq}: no free block")
        table = self.tables[seq]
        cow = None
        if not table or self.fill[table[-1]] == self.block_size:
            table.append(self._take_free_block())
        elif self.refs[table[-1]] > 1:
            old = table[-1]
            new = self._take_free_block()
            self.fill[new] = self.fill[old]
            self.refs[old] -= 1
            table[-1] = new
            cow = (old, new)
        last = table[-1]
        offset = self.fill[last]
        self.fill[last] += 1
        return last * self.block_size + offset, cow

    def append_tokens(self, seq, n):
        """Append n tokens; returns (slots, cows). All or nothing."""
        if self._blocks_needed(seq, n) > len(self.free):
            raise OutOfBlocks(f"seq {seq}: {n} tokens do not fit")
        slots, cows = [], []
        for _ in range(n):
            slot, cow = self.append_token(seq)
            slots.append(slot)
            if cow is not None:
                cows.append(cow)
        return slots, cows

    def fork(self, parent):
        child = self.new_seq()
        self.tables[child] = list(self.tables[parent])
        for blk in self.tables[child]:
            self.refs[blk] += 1
        return child

    def release(self, seq):
        """Drop seq; returns the blocks that went back on the free list."""
        freed = []
        for blk in self.tables.pop(seq):
            self.refs[blk] -= 1
            if self.refs[blk] == 0:
                self.fill[blk] = 0
                self.free.append(blk)
                freed.append(blk)
        return freed

    # -- export ----------------------------------------------------------------
    def export(self, seqs, max_blocks_per_seq):
        """(tables [n][MB] padded with -1, context_lens [n]) as Python lists."""
        tables, lens = [], []
        for seq in seqs:
            table = self.tables[seq]
            if len(table) > max_blocks_per_seq:
                raise ValueError(f"seq {seq} has {len(table)} blocks > {max_blocks_per_seq}")
            tables.append(list(table) + [-1] * (max_blocks_per_seq - len(table)))
            lens.append(self.seq_len(seq))
        return tables, lens
