"""Oracle: single-query decode attention read through a block table (fp64).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it computes.  [P1] "How PagedAttention works", step 4: each decode step
the kernel walks the request's block table, loads each block's keys and values
and computes attention exactly as if they were contiguous.  [P1] "Key
takeaways" and "Common misconceptions": paging changes the memory layout, not
the model's outputs.  So the oracle is the plain definition of attention over
the tokens gathered in logical order:

    x_t   = scale * sum_i q[i] * k_t[i]           for t = 0 .. L-1
    out   = sum_t exp(x_t - max x) * v_t / sum_t exp(x_t - max x)

Token -> location.  [P1] "What PagedAttention is": logical block i holds tokens
i*bs .. i*bs+bs-1, and the block table maps logical block i to a physical block.
So token t lives in physical block table[t // bs] at offset t % bs (the
paged_vs_contiguous.py example on [P1] maps token 37 to logical block 2,
offset 5).  [P2] "How PagedAttention works": within a block, tokens are laid
out contiguously.

Readings where the pages are silent:
* cache layout [num_blocks][num_kv_heads][block_size][head_dim];
* grouped-query attention: query head h reads KV head h // (H / H_kv);
* context_len == 0 gives an all-zero output row;
* table entries past ceil(L / bs) are never read (they may hold -1, the
  "unassigned" marker of [P2]'s BlockTable sketch).
"""

import math

import numpy as np


def token_location(table_row, t, block_size):
    """Physical (block, offset) of logical token ``t`` of one sequence."""
    logical_block = t // block_size
    offset = t % block_size
    return int(table_row[logical_block]), offset


def gather_sequence(cache, table_row, context_len, block_size):
    """All ``context_len`` tokens of one sequence, in logical order, as fp64.

    ``cache`` is [num_blocks][num_kv_heads][block_size][head_dim] (any float
    dtype); returns [context_len][num_kv_heads][head_dim] float64.
    """
    num_blocks, num_kv_heads, bs, head_dim = cache.shape
    assert bs == block_size
    out = np.empty((context_len, num_kv_heads, head_dim), dtype=np.float64)
    for t in range(context_len):
        blk, off = token_location(table_row, t, block_size)
        if not 0 <= blk < num_blocks:
            raise ValueError(f"token {t}: physical block {blk} outside the pool")
        out[t] = cache[blk, :, off, :].astype(np.float64)
    return out


def attention_one_head(q, keys, values, scale):
    """softmax(scale * q . k_t) weighted sum of v_t, for one head (fp64).

    q: [D]; keys, values: [L][D]; returns [D].  L == 0 returns zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    if keys.shape[0] == 0:
        return np.zeros(q.shape[0], dtype=np.float64)
    x = scale * (keys @ q)
    w = np.exp(x - x.max())
    return (w @ values) / w.sum()


def paged_decode_attention_one(query_seq, key_cache, value_cache, table_row,
                               context_len, scale):
    """Decode attention for one sequence: query_seq [H][D] -> [H][D] fp64."""
    num_heads = query_seq.shape[0]
    num_kv_heads = key_cache.shape[1]
    block_size = key_cache.shape[2]
    if num_heads % num_kv_heads:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    group = num_heads // num_kv_heads
    keys = gather_sequence(key_cache, table_row, context_len, block_size)
    values = gather_sequence(value_cache, table_row, context_len, block_size)
    out = np.zeros((num_heads, query_seq.shape[1]), dtype=np.float64)
    for h in range(num_heads):
        kvh = h // group
        out[h] = attention_one_head(query_seq[h], keys[:, kvh, :],
                                    values[:, kvh, :], scale)
    return out


def paged_decode_attention(query, key_cache, value_cache, block_tables,
                           context_lens, scale, seqs=None):
    """Decode attention for a batch.

    query [N][H][D]; caches [NB][H_kv][bs][D]; block_tables [N][MB] int;
    context_lens [N] int.  Returns float64 [N][H][D] (rows not in ``seqs``,
    when given, are left as NaN so that a caller cannot mistake them for
    checked values).
    """
    n = query.shape[0]
    out = np.full(query.shape, np.nan, dtype=np.float64)
    rows = range(n) if seqs is None else seqs
    for s in rows:
        out[s] = paged_decode_attention_one(query[s], key_cache, value_cache,
                                            block_tables[s], int(context_lens[s]),
                                            scale)
    return out


def default_scale(head_dim):
    """1/sqrt(head_dim), the scale every workload here uses."""
    return 1.0 / math.sqrt(head_dim)
