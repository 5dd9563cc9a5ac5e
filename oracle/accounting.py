"""Oracle: block counts, slot waste and KV bytes per token.

TEST INFRASTRUCTURE ONLY (see the package docstring).

* blocks_for_tokens: a sequence of n tokens needs ceil(n / block_size) blocks
  ([P1] "How PagedAttention works" step 1: 40 tokens -> 3 blocks of 16).
* paged waste: allocated slots minus used slots, allocated = blocks * bs
  ([P1] "Worked example, step by step"; [P1] paged_vs_contiguous.py output).
* contiguous waste: every request reserves max_len slots up front
  ([P1] "The problem: memory waste in the KV cache").
* kv_bytes_per_token: one key and one value vector per KV head per layer
  ([P1] "Quick recap: the KV cache": 32 layers, 32 KV heads of 128, fp16 ->
  512 KiB per token).
"""


def blocks_for_tokens(n_tokens, block_size):
    return -(-int(n_tokens) // int(block_size))


def paged_slots(lengths, block_size):
    return sum(blocks_for_tokens(n, block_size) for n in lengths) * block_size


def paged_waste_fraction(lengths, block_size):
    used = sum(int(n) for n in lengths)
    alloc = paged_slots(lengths, block_size)
    return 1.0 - used / alloc


def contiguous_waste_fraction(lengths, max_len):
    used = sum(int(n) for n in lengths)
    reserved = max_len * len(lengths)
    return 1.0 - used / reserved


def empty_slots(n_tokens, block_size):
    return blocks_for_tokens(n_tokens, block_size) * block_size - int(n_tokens)


def kv_bytes_per_token(num_layers, num_kv_heads, head_dim, bytes_per_elem):
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_elem
