"""The seeded workloads replay through the oracle block manager as described."""

import numpy as np
import pytest

import workloads as W
from oracle.block_manager import BlockManagerModel


@pytest.mark.parametrize("name", W.NAMES)
def test_trace_reaches_stated_context_lengths(name):
    wl = W.make(name)
    m = BlockManagerModel(wl.num_blocks, wl.block_size, wl.free_order)
    W.replay(m, wl.ops)
    for s in wl.batch:
        m.append_token(s)
    assert [m.seq_len(s) for s in wl.batch] == wl.context_lens
    tables, lens = m.export(wl.batch, wl.max_blocks_per_seq())
    used = {b for row in tables for b in row if b >= 0}
    assert all(0 <= b < wl.num_blocks for b in used)


def test_shapes_of_the_five_workloads():
    t = W.make("tiny")
    assert t.context_lens == [40, 17, 100, 5] and t.num_blocks == 64 and t.head_dim == 64
    s = W.make("7b")
    assert s.num_seqs == 64 and min(s.context_lens) >= 50 and max(s.context_lens) <= 900
    c = W.make("chat")
    assert c.num_seqs == 128 and min(c.context_lens) >= 150 and max(c.context_lens) <= 2500
    g = W.make("gqa")
    assert g.group == 4 and g.block_size == 32
    assert min(g.context_lens) >= 256 and max(g.context_lens) <= 4096
    p = W.make("prefix")
    assert p.num_seqs == 128 and min(p.context_lens) >= 550 and max(p.context_lens) <= 1000


def test_prefix_divergence_makes_127_copies():
    wl = W.make("prefix")
    m = BlockManagerModel(wl.num_blocks, wl.block_size, wl.free_order)
    W.replay(m, wl.ops, 0, wl.marks["divergence"])
    tail = m.tables[0][-1]
    assert m.refs[tail] == 128 and m.fill[tail] == 4 and len(m.tables[0]) == 32
    res = W.replay(m, wl.ops, wl.marks["divergence"], wl.marks["after_divergence"])
    cows = [c for _, cs in res for c in cs]
    assert len(cows) == 127 and all(src == tail for src, _ in cows)
    assert m.refs[tail] == 1 and m.tables[127][-1] == tail


def test_chat_reuses_freed_blocks():
    wl = W.make("chat")
    releases = [op for op in wl.ops if op[0] == "release"]
    assert len(releases) == 64
    first_release = next(i for i, op in enumerate(wl.ops) if op[0] == "release")
    assert any(op[0] == "new" for op in wl.ops[first_release:])


def test_tensors_are_seeded():
    wl = W.make("tiny")
    a = W.tensors(wl)
    b = W.tensors(wl)
    for k in a:
        assert a[k].dtype.itemsize == 2 and (a[k] == b[k]).all()
    assert tuple(a["key_cache"].shape) == (64, 8, 16, 64)


def test_base_seed_default_and_override():
    """`base` defaults to BASE_SEED (the inputs every test and record use) and
    a different base draws different lengths and free orders."""
    for name in ("7b", "chat", "gqa", "prefix"):
        a, b, c = W.make(name), W.make(name, base=W.BASE_SEED), W.make(name, base=W.BASE_SEED + 1000)
        assert a.context_lens == b.context_lens and a.seed == b.seed
        assert np.array_equal(a.free_order, b.free_order)
        assert a.context_lens != c.context_lens and c.seed == a.seed + 1000
