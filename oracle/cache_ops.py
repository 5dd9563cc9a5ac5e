"""Oracle: the slot-mapped cache write and the copy-on-write block copy.

TEST INFRASTRUCTURE ONLY (see the package docstring).

reshape_and_cache.  [P1] "How PagedAttention works", steps 2-3: each new token
goes into the next free slot of the request's last block.  A slot number names
one token position in the pool: slot = physical_block * block_size + offset,
the same (block, offset) split the paged_vs_contiguous.py example on [P1] uses
for token 37.  The write copies the new token's key and value rows, for every
KV head, to that position.  A negative slot means "no write" (padding).

copy_blocks.  [P1] "Memory sharing across requests": copy-on-write copies the
shared block to a fresh block before the writer's token goes in.  The oracle
copies every byte of the block (all heads, all slots) in both caches; the
copied fill count travels with the block ([P1] practice listing).

swap_blocks.  [P2] "Why it matters for KV cache", "Swapping and preemption":
blocks are evicted to CPU memory and fetched back.  The oracle copies every
byte of each listed block from one pool to the other (both caches); the block
manager decides which blocks move where.

valid_slot_mask.  The token positions a batch of sequences actually uses; the
tests poison every other slot of the pool with NaN so that any read outside a
sequence's context shows up in the output.
"""

import numpy as np


def slot_location(slot, block_size):
    """(physical block, offset) of a slot number."""
    return slot // block_size, slot % block_size


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping):
    """Write key[t], value[t] ([H_kv][D] each) to slot_mapping[t], in place.

    key, value: [T][H_kv][D]; caches: [NB][H_kv][bs][D] (same dtype as key);
    slot_mapping: [T] integers, negative = skip.  Raises on a slot outside the
    pool.  Plain element copies: bit-exact by construction.
    """
    num_blocks, _, block_size, _ = key_cache.shape
    for t in range(key.shape[0]):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        blk, off = slot_location(slot, block_size)
        if blk >= num_blocks:
            raise ValueError(f"slot {slot} outside the pool")
        key_cache[blk, :, off, :] = key[t]
        value_cache[blk, :, off, :] = value[t]


def copy_blocks(key_cache, value_cache, pairs):
    """For each (src, dst) pair copy physical block src over block dst, in place.

    Pairs are applied in order.  Plain block copies: bit-exact by construction.
    """
    num_blocks = key_cache.shape[0]
    for src, dst in pairs:
        src, dst = int(src), int(dst)
        if not (0 <= src < num_blocks and 0 <= dst < num_blocks):
            raise ValueError(f"pair ({src}, {dst}) outside the pool")
        key_cache[dst] = key_cache[src]
        value_cache[dst] = value_cache[src]


def swap_blocks(src_key, src_value, dst_key, dst_value, pairs):
    """For each (src, dst) pair copy block src of the source pool over block
    dst of the destination pool, in place, in order.  Bit-exact copies."""
    for src, dst in pairs:
        src, dst = int(src), int(dst)
        if not (0 <= src < src_key.shape[0] and 0 <= dst < dst_key.shape[0]):
            raise ValueError(f"pair ({src}, {dst}) outside a pool")
        dst_key[dst] = src_key[src]
        dst_value[dst] = src_value[src]


def valid_slot_mask(block_tables, context_lens, num_blocks, block_size):
    """[NB][bs] bool: True where some sequence's token t < context_len lives."""
    mask = np.zeros((num_blocks, block_size), dtype=bool)
    for s in range(len(context_lens)):
        for t in range(int(context_lens[s])):
            blk = int(block_tables[s][t // block_size])
            mask[blk, t % block_size] = True
    return mask
