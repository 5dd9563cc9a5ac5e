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
  followed.)
* Release.  [P1] practice exercise 3 and the "Fifty chats" question: every
  block's count goes down by one; blocks reaching zero go back on the free
  list, others stay.
* Swap out / swap in.  [P1] "Common misconceptions": paging alone does not
  move the cache to CPU memory; swapping is a separate technique by which
  blocks are moved out under memory pressure.  [P2] "Why it matters for KV
  cache", "Swapping and preemption": blocks are evicted to CPU memory when GPU
  memory runs short and fetched back when the request resumes.  The pages give
  no further rule; the plainest reading, taken here: a second pool of host
  blocks with its own FIFO free list, counts and fills.  Swapping out a group
  of resident sequences gives every distinct device block the group holds one
  host block (in order of first appearance: sequences in the given order, each
  table in logical order), with the count of group members that hold it and
  the block's fill; the device block's count drops by that many and, at zero,
  the block returns to the device free list (same order).  The sequences'
  tables then name host blocks and the sequences are "swapped": they can be
  released, not appended to, forked or exported.  Swap in is the mirror image
  (host -> fresh device blocks).  Sharing inside the group survives the round
  trip; sharing with a sequence outside the group does not (each side keeps
  its own copy).  Each call returns the (source, destination) block pairs
  whose data must move, in allocation order.

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


class SwappedOut(RuntimeError):
    """The operation needs a resident sequence and this one is swapped out."""


class BlockManagerModel:
    def __init__(self, num_blocks, block_size, initial_free_order=None,
                 num_host_blocks=0, host_free_order=None):
        order = _permutation(initial_free_order, num_blocks)
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = deque(order)
        self.refs = [0] * num_blocks      # sequences using each block
        self.fill = [0] * num_blocks      # token slots written in each block
        self.tables = {}                  # seq id -> list of physical blocks
        self.next_seq = 0
        # host pool for swapped-out sequences
        self.num_host_blocks = num_host_blocks
        self.host_free = deque(_permutation(host_free_order, num_host_blocks))
        self.host_refs = [0] * num_host_blocks
        self.host_fill = [0] * num_host_blocks
        self.swapped = set()              # seq ids whose tables name host blocks

    # -- queries -----------------------------------------------------------
    def num_free(self):
        return len(self.free)

    def seq_len(self, seq):
        table = self.tables[seq]
        if not table:
            return 0
        fill = self.host_fill if seq in self.swapped else self.fill
        return (len(table) - 1) * self.block_size + fill[table[-1]]

    def is_swapped(self, seq):
        return seq in self.swapped

    def _resident(self, seq):
        if seq in self.swapped:
            raise SwappedOut(f"seq {seq} is swapped out")
        return self.tables[seq]

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
        table = self._resident(seq)
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
        self._resident(parent)
        child = self.new_seq()
        self.tables[child] = list(self.tables[parent])
        for blk in self.tables[child]:
            self.refs[blk] += 1
        return child

    def release(self, seq):
        """Drop seq; returns the blocks that went back on their pool's free
        list (host blocks if seq was swapped out)."""
        if seq in self.swapped:
            self.swapped.discard(seq)
            refs, fill, free = self.host_refs, self.host_fill, self.host_free
        else:
            refs, fill, free = self.refs, self.fill, self.free
        freed = []
        for blk in self.tables.pop(seq):
            refs[blk] -= 1
            if refs[blk] == 0:
                fill[blk] = 0
                free.append(blk)
                freed.append(blk)
        return freed

    # -- swapping ----------------------------------------------------------
    def _move(self, seqs, want_swapped, src, dst):
        """Move the group's blocks from pool src to pool dst.

        src, dst: (refs, fill, free) of the two pools.  Returns the
        (source block, destination block) pairs in allocation order.
        """
        seqs = [int(x) for x in seqs]
        if len(set(seqs)) != len(seqs):
            raise ValueError("sequences must be distinct")
        for seq in seqs:
            if seq not in self.tables:
                raise KeyError(seq)
            if (seq in self.swapped) != want_swapped:
                raise SwappedOut(f"seq {seq}: wrong residency for this swap")
        holders = {}                          # block -> group members holding it
        for seq in seqs:
            for blk in self.tables[seq]:
                holders[blk] = holders.get(blk, 0) + 1
        src_refs, src_fill, src_free = src
        dst_refs, dst_fill, dst_free = dst
        if len(holders) > len(dst_free):
            raise OutOfBlocks(f"{len(holders)} blocks to move, {len(dst_free)} free")
        moved = {}
        for blk, count in holders.items():    # dicts keep first-appearance order
            new = dst_free.popleft()
            dst_refs[new] = count
            dst_fill[new] = src_fill[blk]
            moved[blk] = new
        for blk, count in holders.items():
            src_refs[blk] -= count
            if src_refs[blk] == 0:
                src_fill[blk] = 0
                src_free.append(blk)
        for seq in seqs:
            self.tables[seq] = [moved[b] for b in self.tables[seq]]
        return list(moved.items())

    def swap_out(self, seqs):
        """Move resident seqs to the host pool; returns (device, host) pairs."""
        pairs = self._move(seqs, False, (self.refs, self.fill, self.free),
                           (self.host_refs, self.host_fill, self.host_free))
        self.swapped.update(int(x) for x in seqs)
        return pairs

    def swap_in(self, seqs):
        """Bring swapped seqs back to device blocks; returns (host, device) pairs."""
        pairs = self._move(seqs, True, (self.host_refs, self.host_fill, self.host_free),
                           (self.refs, self.fill, self.free))
        self.swapped.difference_update(int(x) for x in seqs)
        return pairs

    # -- export ----------------------------------------------------------------
    def export(self, seqs, max_blocks_per_seq):
        """(tables [n][MB] padded with -1, context_lens [n]) as Python lists."""
        tables, lens = [], []
        for seq in seqs:
            table = self._resident(seq)
            if len(table) > max_blocks_per_seq:
                raise ValueError(f"seq {seq} has {len(table)} blocks > {max_blocks_per_seq}")
            tables.append(list(table) + [-1] * (max_blocks_per_seq - len(table)))
            lens.append(self.seq_len(seq))
        return tables, lens


def _permutation(order, n):
    if order is None:
        return list(range(n))
    order = [int(b) for b in order]
    if sorted(order) != list(range(n)):
        raise ValueError("a free order must be a permutation of its pool")
    return order
