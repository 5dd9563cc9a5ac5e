"""Pins for the oracle's swap out / swap in (CPU only).

[P1] "Common misconceptions" and [P2] "Why it matters for KV cache",
"Swapping and preemption" say only that blocks go to CPU memory under memory
pressure and come back when the request resumes.  The expected values below
are worked by hand from the reading the oracle states (host pool with its own
FIFO free list; distinct blocks of the group in order of first appearance;
counts = group members holding the block).  The invariants (block
conservation, data round trip, unchanged attention) hold under any reading in
which a swap moves data without changing it.
"""

import copy

import numpy as np
import pytest

from oracle import attention, cache_ops
from oracle.block_manager import BlockManagerModel, OutOfBlocks, SwappedOut


def _state(m):
    return (list(m.free), list(m.refs), list(m.fill), list(m.host_free), list(m.host_refs),
            list(m.host_fill), {k: list(v) for k, v in m.tables.items()}, set(m.swapped))


def test_group_swap_keeps_sharing_worked_by_hand():
    m = BlockManagerModel(8, 4, num_host_blocks=4)
    a = m.new_seq()
    m.append_tokens(a, 6)                       # blocks 0 (full), 1 (2 tokens)
    b = m.fork(a)
    assert m.swap_out([a, b]) == [(0, 0), (1, 1)]
    assert m.host_refs == [2, 2, 0, 0] and m.host_fill == [4, 2, 0, 0]
    assert list(m.free) == [2, 3, 4, 5, 6, 7, 0, 1] and m.refs == [0] * 8
    assert m.tables[a] == m.tables[b] == [0, 1] and m.seq_len(a) == m.seq_len(b) == 6
    assert m.is_swapped(a) and m.is_swapped(b)
    # b alone comes back: fresh device blocks from the front; the host copies
    # stay for a
    assert m.swap_in([b]) == [(0, 2), (1, 3)]
    assert m.tables[b] == [2, 3] and m.refs[2] == m.refs[3] == 1 and m.fill[3] == 2
    assert m.host_refs == [1, 1, 0, 0]
    slot, cow = m.append_token(b)               # sole owner: in place
    assert (slot, cow) == (3 * 4 + 2, None)
    assert m.swap_in([a]) == [(0, 4), (1, 5)]
    assert list(m.host_free) == [2, 3, 0, 1] and m.host_refs == [0] * 4
    assert m.tables[a] == [4, 5] and m.seq_len(a) == 6 and m.seq_len(b) == 7


def test_swap_out_one_sharer_copies_shared_blocks():
    m = BlockManagerModel(6, 4, num_host_blocks=6, host_free_order=[5, 4, 3, 2, 1, 0])
    a = m.new_seq()
    m.append_tokens(a, 9)                       # blocks 0, 1 full; 2 holds 1
    b = m.fork(a)
    c = m.new_seq()
    m.append_tokens(c, 3)                       # block 3
    assert m.swap_out([b, c]) == [(0, 5), (1, 4), (2, 3), (3, 2)]
    assert m.refs[:4] == [1, 1, 1, 0]           # a keeps its blocks; 3 is free
    assert list(m.free) == [4, 5, 3]
    assert m.host_refs == [0, 0, 1, 1, 1, 1]
    # a writes into block 2, no longer shared: no copy-on-write
    assert m.append_token(a) == (2 * 4 + 1, None)
    assert m.release(b) == [5, 4, 3]            # host blocks back on the host list
    assert list(m.host_free) == [1, 0, 5, 4, 3]


def test_swapped_sequence_refuses_resident_operations():
    m = BlockManagerModel(4, 2, num_host_blocks=4)
    a = m.new_seq()
    m.append_tokens(a, 3)
    m.swap_out([a])
    snap = _state(m)
    for op in (lambda: m.append_token(a), lambda: m.append_tokens(a, 2), lambda: m.fork(a),
               lambda: m.export([a], 4), lambda: m.swap_out([a])):
        with pytest.raises(SwappedOut):
            op()
    b = m.new_seq()
    with pytest.raises(SwappedOut):
        m.swap_in([a, b])                       # b is resident
    with pytest.raises(ValueError):
        m.swap_in([a, a])
    snap_b = _state(m)
    assert snap_b[:6] == snap[:6]


def test_swap_out_of_blocks_changes_nothing():
    m = BlockManagerModel(8, 2, num_host_blocks=3)
    a, b = m.new_seq(), m.new_seq()
    m.append_tokens(a, 4)                       # blocks 0, 1
    m.append_tokens(b, 4)                       # blocks 2, 3
    snap = _state(m)
    with pytest.raises(OutOfBlocks):
        m.swap_out([a, b])                      # 4 distinct blocks, 3 host blocks
    assert _state(m) == snap
    assert m.swap_out([a]) == [(0, 0), (1, 1)]
    snap = _state(m)
    with pytest.raises(OutOfBlocks):
        m.swap_out([b])                         # 2 blocks, 1 host block left
    assert _state(m) == snap
    c = m.new_seq()
    m.append_tokens(c, 12)                      # takes the 6 free device blocks
    snap = _state(m)
    with pytest.raises(OutOfBlocks):
        m.swap_in([a])
    assert _state(m) == snap
    m.release(c)
    assert m.swap_in([a]) == [(0, 4), (1, 5)]


def _invariants(m):
    res = [s for s in m.tables if s not in m.swapped]
    swp = [s for s in m.tables if s in m.swapped]
    for pool_refs, pool_free, seqs, n in ((m.refs, m.free, res, m.num_blocks),
                                          (m.host_refs, m.host_free, swp, m.num_host_blocks)):
        held = {}
        for s in seqs:
            for blk in m.tables[s]:
                held[blk] = held.get(blk, 0) + 1
        assert all(pool_refs[b] == held.get(b, 0) for b in range(n))
        assert sorted(list(pool_free) + list(held)) == list(range(n))


@pytest.mark.parametrize("seed", range(6))
def test_random_traces_conserve_blocks_and_data(seed):
    """Brute force: blocks are conserved in both pools, and every sequence's
    gathered K/V is unchanged by any mix of swaps, whatever else happens."""
    rng = np.random.default_rng(4000 + seed)
    nb, nh, bs, hkv, d = 24, 20, 4, 2, 8
    m = BlockManagerModel(nb, bs, rng.permutation(nb), nh, rng.permutation(nh))
    kc = np.full((nb, hkv, bs, d), np.nan)
    vc = np.full_like(kc, np.nan)
    hk = np.full((nh, hkv, bs, d), np.nan)
    hv = np.full_like(hk, np.nan)
    truth = {}                                  # seq -> list of (k, v) rows written
    for _ in range(300):
        live = list(m.tables)
        resident = [s for s in live if not m.is_swapped(s)]
        swapped = [s for s in live if m.is_swapped(s)]
        op = int(rng.integers(0, 8))
        if op == 0 or not live:
            truth[m.new_seq()] = []
        elif op <= 2 and resident:
            s = int(rng.choice(resident))
            try:
                slot, cow = m.append_token(s)
            except OutOfBlocks:
                continue
            if cow is not None:
                cache_ops.copy_blocks(kc, vc, [cow])
            k, v = rng.standard_normal((1, hkv, d)), rng.standard_normal((1, hkv, d))
            cache_ops.reshape_and_cache(k, v, kc, vc, [slot])
            truth[s].append((k[0], v[0]))
        elif op == 3 and resident:
            s = int(rng.choice(resident))
            truth[m.fork(s)] = list(truth[s])
        elif op == 4 and resident:
            group = [int(x) for x in rng.permutation(resident)[: int(rng.integers(1, len(resident) + 1))]]
            try:
                pairs = m.swap_out(group)
            except OutOfBlocks:
                continue
            cache_ops.swap_blocks(kc, vc, hk, hv, pairs)
            for src, _ in pairs:                # freed device blocks lose their data
                if m.refs[src] == 0:
                    kc[src] = vc[src] = np.nan
        elif op == 5 and swapped:
            group = [int(x) for x in rng.permutation(swapped)[: int(rng.integers(1, len(swapped) + 1))]]
            try:
                pairs = m.swap_in(group)
            except OutOfBlocks:
                continue
            cache_ops.swap_blocks(hk, hv, kc, vc, pairs)
            for src, _ in pairs:
                if m.host_refs[src] == 0:
                    hk[src] = hv[src] = np.nan
        elif op == 6 and live:
            s = int(rng.choice(live))
            m.release(s)
            del truth[s]
        _invariants(m)
        for s in live:
            if s not in m.tables:
                continue
            table, n = m.tables[s], len(truth[s])
            assert m.seq_len(s) == n
            pool_k, pool_v = (hk, hv) if m.is_swapped(s) else (kc, vc)
            for t, (k, v) in enumerate(truth[s]):
                blk = table[t // bs]
                assert np.array_equal(pool_k[blk, :, t % bs], k)
                assert np.array_equal(pool_v[blk, :, t % bs], v)


def test_attention_unchanged_by_round_trip():
    rng = np.random.default_rng(7)
    nb, bs, hkv, g, d = 32, 4, 2, 2, 8
    m = BlockManagerModel(nb, bs, rng.permutation(nb), num_host_blocks=16)
    kc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    vc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    seqs = [m.new_seq() for _ in range(3)]
    for s, n in zip(seqs, (7, 13, 4)):
        m.append_tokens(s, n)
    seqs.append(m.fork(seqs[1]))
    q = rng.standard_normal((4, hkv * g, d)).astype(np.float16)
    tables, lens = m.export(seqs, 8)
    before = attention.paged_decode_attention(q, kc, vc, np.array(tables), np.array(lens), d ** -0.5)
    hk = np.zeros((16, hkv, bs, d), np.float16)
    hv = np.zeros_like(hk)
    cache_ops.swap_blocks(kc, vc, hk, hv, m.swap_out([seqs[1], seqs[3]]))
    kc2, vc2 = kc.copy(), vc.copy()
    m.append_tokens(m.new_seq(), 20)            # reuse the freed device blocks
    kc2[:] = vc2[:] = np.float16(np.nan)
    for s in (seqs[0], seqs[2]):                # keep only what resident seqs own
        for blk in m.tables[s]:
            kc2[blk], vc2[blk] = kc[blk], vc[blk]
    cache_ops.swap_blocks(hk, hv, kc2, vc2, m.swap_in([seqs[3], seqs[1]]))
    tables2, lens2 = m.export(seqs, 8)
    assert lens2 == lens and tables2 != tables
    after = attention.paged_decode_attention(q, kc2, vc2, np.array(tables2), np.array(lens2), d ** -0.5)
    assert np.array_equal(before, after)
