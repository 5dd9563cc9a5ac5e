"""Pins for the oracle block manager and accounting (CPU only).

Each test checks the oracle against values the pages print (fixtures under
tests/golden/, each with its source) or against consequences of the pages'
rules that the pages state in words.
"""

import numpy as np
import pytest

from oracle import accounting
from oracle.block_manager import BlockManagerModel, OutOfBlocks


def _refs_dict(m):
    return {str(b): r for b, r in enumerate(m.refs) if r > 0}


def test_practice_run_printed_output(golden):
    g = golden("practice_block_manager.json")
    m = BlockManagerModel(g["setup"]["pool"], g["setup"]["block_size"],
                          g["setup"]["free_order"])
    a = m.new_seq()
    m.append_tokens(a, g["setup"]["prompt_tokens"])
    b = m.fork(a)
    assert m.tables[a] == g["after_fork"]["A"]
    assert m.tables[b] == g["after_fork"]["B"]
    assert _refs_dict(m) == g["after_fork"]["refs"]
    m.append_token(a)
    assert m.tables[a] == g["after_A_writes"]["A"]
    assert m.tables[b] == g["after_A_writes"]["B"]
    assert _refs_dict(m) == g["after_A_writes"]["refs"]
    m.append_token(b)
    assert m.tables[a] == g["after_B_writes"]["A"]
    assert m.tables[b] == g["after_B_writes"]["B"]
    assert _refs_dict(m) == g["after_B_writes"]["refs"]
    assert m.blocks_in_use() == g["blocks_in_use"]
    # two private copies of a 7-token sequence at 4 tokens per block
    assert 2 * accounting.blocks_for_tokens(7, 4) == g["with_two_full_copies"]


def test_practice_run_slots_and_cow_pair():
    m = BlockManagerModel(8, 4)
    a = m.new_seq()
    slots, cows = m.append_tokens(a, 6)
    assert slots == [0, 1, 2, 3, 4, 5] and cows == []
    b = m.fork(a)
    slot, cow = m.append_token(a)
    # A's 7th token: offset 2 of its private copy (block 2) of block 1
    assert cow == (1, 2) and slot == 2 * 4 + 2
    assert m.fill[2] == 3 and m.fill[1] == 2
    slot, cow = m.append_token(b)
    assert cow is None and slot == 1 * 4 + 2


def test_paged_vs_contiguous_printed_output(golden):
    g = golden("paged_vs_contiguous.json")
    rng = np.random.default_rng(g["setup"]["numpy_seed"])
    lengths = rng.integers(50, 900, size=8)
    assert lengths.tolist() == g["final_lengths"]
    bs, max_len = g["setup"]["block_size"], g["setup"]["max_len"]
    assert max_len * len(lengths) == g["contiguous"]["reserved_slots"]
    assert int(lengths.sum()) == g["contiguous"]["used_slots"]
    assert round(100 * accounting.contiguous_waste_fraction(lengths, max_len), 1) == \
        g["contiguous"]["waste_percent_1dp"]
    assert accounting.paged_slots(lengths, bs) == g["paged"]["allocated_slots"]
    assert round(100 * accounting.paged_waste_fraction(lengths, bs), 1) == \
        g["paged"]["waste_percent_1dp"]

    perm = rng.permutation(400)
    # the page takes blocks from the end of the permutation; a FIFO free list
    # holding the permutation reversed hands them out in the same order
    m = BlockManagerModel(400, bs, perm[::-1])
    s = m.new_seq()
    slots, _ = m.append_tokens(s, int(lengths[0]))
    table = m.tables[s]
    assert len(table) == g["request0"]["blocks"]
    assert table[:6] == g["request0"]["table_head"]
    t = 37
    assert t // bs == g["token37"]["logical_block"] and t % bs == g["token37"]["offset"]
    assert table[t // bs] == g["token37"]["physical_block"]
    assert slots[t] == g["token37"]["physical_block"] * bs + g["token37"]["offset"]


def test_request_lifecycle(golden):
    g = golden("lifecycle.json")
    bs = g["block_size"]
    order = g["free_blocks_in_order"] + [b for b in range(16) if b not in g["free_blocks_in_order"]]
    m = BlockManagerModel(16, bs, order)
    s = m.new_seq()
    slots, _ = m.append_tokens(s, g["prompt_tokens"])
    assert m.tables[s] == g["blocks_after_prompt"]
    lo, hi = g["last_block_holds_tokens"]
    assert all(sl // bs == g["blocks_after_prompt"][-1] for sl in slots[lo:hi + 1])
    assert accounting.empty_slots(g["prompt_tokens"], bs) == g["empty_slots_in_last_block"]
    free_before = m.num_free()
    lo, hi = g["tokens_without_allocation"]
    for _ in range(lo, hi + 1):
        m.append_token(s)
    assert m.num_free() == free_before and m.tables[s] == g["blocks_after_prompt"]
    assert m.seq_len(s) == g["token_that_allocates"]
    slot, cow = m.append_token(s)           # token 48
    assert cow is None
    assert m.tables[s] == g["blocks_after_token_48"]
    assert slot == g["blocks_after_token_48"][-1] * bs + 0
    # step 5: on finish all blocks return to the free list
    m.release(s)
    assert m.num_free() == 16 and m.blocks_in_use() == 0


def test_four_samples_share_partial_block(golden):
    g = golden("qa_sharing.json")["four_samples"]
    bs = g["block_size"]
    m = BlockManagerModel(64, bs)
    a = m.new_seq()
    m.append_tokens(a, 3 * bs + g["tokens_in_shared_last_block"])
    others = [m.fork(a) for _ in range(g["sharers"] - 1)]
    shared_tail = m.tables[a][-1]
    full = m.tables[a][:-1]
    slot, cow = m.append_token(a)
    assert (cow is not None) == g["writer_copies"]
    assert cow[0] == shared_tail and m.tables[a][-1] == cow[1]
    assert slot == cow[1] * bs + g["writer_slot_offset_in_copy"]
    assert m.refs[shared_tail] == g["original_refs_after"]
    assert m.tables[a][:-1] == full and all(m.refs[b] == g["sharers"] for b in full)
    assert all(m.tables[o][-1] == shared_tail for o in others)


def test_second_writer_does_not_copy(golden):
    g = golden("qa_sharing.json")["second_writer_after_copy"]
    m = BlockManagerModel(16, 16)
    a = m.new_seq()
    m.append_tokens(a, 20)
    b = m.fork(a)
    assert g["sharers"] == 2
    _, cow_a = m.append_token(a)
    _, cow_b = m.append_token(b)
    assert cow_a is not None and (cow_b is not None) == g["second_writer_copies"]


def test_fifty_chats_release(golden):
    g = golden("qa_sharing.json")["fifty_chats"]
    m = BlockManagerModel(g["shared_blocks"] + 10, 16)
    root = m.new_seq()
    m.append_tokens(root, 16 * g["shared_blocks"])
    chats = [root] + [m.fork(root) for _ in range(g["sharers"] - 1)]
    prompt = list(m.tables[root])
    freed = m.release(chats[7])
    assert len(freed) == g["blocks_freed_when_one_ends"]
    assert all(m.refs[b] == g["refs_after"] for b in prompt)


def test_block_size_tradeoff(golden):
    g = golden("block_size_tradeoff.json")
    for case in g["cases"]:
        bs = case["block_size"]
        assert accounting.blocks_for_tokens(g["tokens"], bs) == case["blocks"]
        assert accounting.paged_slots([g["tokens"]], bs) == case["slots"]
        assert accounting.empty_slots(g["tokens"], bs) == case["empty"]
        if "empty_percent_of_allocated" in case:
            assert round(100 * case["empty"] / case["slots"]) == case["empty_percent_of_allocated"]
    mdl = g["bytes_per_token_model"]
    bpt = accounting.kv_bytes_per_token(mdl["layers"], mdl["kv_heads"], mdl["head_dim"],
                                        mdl["bytes_per_elem"])
    assert bpt == g["bytes_per_token"]
    assert 8 * bpt == g["empty_8_slots_MiB"] * 2**20
    assert 168 * bpt == g["empty_168_slots_MiB"] * 2**20


def test_chat_sizing(golden):
    g = golden("chat_sizing.json")
    bs = g["block_size"]
    assert accounting.blocks_for_tokens(g["average_prompt_tokens"], bs) == g["average_prompt_blocks"]
    assert accounting.blocks_for_tokens(g["average_generation_tokens"], bs) == \
        g["average_generation_blocks"]
    per_req = g["average_prompt_blocks"] + g["average_generation_blocks"]
    assert g["concurrent_requests"] * per_req == g["peak_blocks"]
    assert accounting.blocks_for_tokens(g["shared_prefix_tokens"], bs) == g["shared_prefix_blocks"]


# -- consequences of the stated rules (answers not printed on the pages) ------

def test_exercise_full_last_block_needs_no_copy():
    # 8-token prompt at 4 tokens per block: the shared last block is full,
    # so A's first write takes a fresh block instead of copying.
    m = BlockManagerModel(8, 4)
    a = m.new_seq()
    m.append_tokens(a, 8)
    m.fork(a)
    slot, cow = m.append_token(a)
    assert cow is None and m.tables[a] == [0, 1, 2] and slot == 8


def test_exercise_third_sample_writes_last():
    m = BlockManagerModel(8, 4)
    a = m.new_seq()
    m.append_tokens(a, 6)
    b = m.fork(a)
    c = m.fork(a)
    copies = 0
    for s in (a, b, c):
        copies += m.append_token(s)[1] is not None
    assert m.tables[a] == [0, 2] and m.tables[b] == [0, 3] and m.tables[c] == [0, 1]
    assert _refs_dict(m) == {"0": 3, "1": 1, "2": 1, "3": 1}
    assert copies == 2
    freed = m.release(a)
    assert freed == [2] and m.refs[0] == 2


def test_out_of_blocks_leaves_state_unchanged():
    m = BlockManagerModel(4, 4)
    a = m.new_seq()
    m.append_tokens(a, 14)            # 4 blocks, the last one holding 2
    snap = (list(m.free), list(m.refs), list(m.fill), {k: list(v) for k, v in m.tables.items()})
    with pytest.raises(OutOfBlocks):
        m.append_tokens(a, 3)         # needs a 5th block
    assert snap == (list(m.free), list(m.refs), list(m.fill),
                    {k: list(v) for k, v in m.tables.items()})
    b = m.fork(a)
    with pytest.raises(OutOfBlocks):
        m.append_token(b)             # copy-on-write needs a free block
    with pytest.raises(OutOfBlocks):
        m.append_tokens(a, 2)         # a's last block is shared too
    m.release(b)
    m.append_tokens(a, 2)             # sole owner again: fills in place
    assert m.tables[a] == [0, 1, 2, 3] and m.fill[3] == 4


def test_free_list_is_fifo():
    m = BlockManagerModel(6, 2, [5, 4, 3, 2, 1, 0])
    a = m.new_seq()
    m.append_tokens(a, 4)             # blocks 5, 4
    b = m.new_seq()
    m.append_tokens(b, 2)             # block 3
    assert m.release(a) == [5, 4]
    assert list(m.free) == [2, 1, 0, 5, 4]
    c = m.new_seq()
    m.append_tokens(c, 2)
    assert m.tables[c] == [2]
