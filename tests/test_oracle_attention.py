"""Pins for the oracle decode attention and cache ops (CPU only).

The oracle is pinned to things other than itself: closed forms, the pages'
invariants (paging does not change outputs; forked tables that share a prefix
give the same outputs), torch's scaled_dot_product_attention on the gathered
tokens (a library routine), and the request lifecycle the lesson walks through.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import cache_ops as C
from oracle.block_manager import BlockManagerModel


def _rand_pool(rng, nb, hkv, bs, d):
    k = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    v = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    return k, v


def _sdpa(q, k, v, scale):
    """torch SDPA in fp64 on CPU: q [H][D], k/v [L][Hkv][D] -> [H][D]."""
    h, d = q.shape
    hkv = k.shape[1]
    qt = torch.from_numpy(np.asarray(q, np.float64)).view(1, h, 1, d)
    kt = torch.from_numpy(np.asarray(k, np.float64)).permute(1, 0, 2).unsqueeze(0)
    vt = torch.from_numpy(np.asarray(v, np.float64)).permute(1, 0, 2).unsqueeze(0)
    kt = kt.repeat_interleave(h // hkv, dim=1)
    vt = vt.repeat_interleave(h // hkv, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o.view(h, d).numpy()


def _contiguous_table(nblk, start=0):
    return np.arange(start, start + nblk, dtype=np.int32)


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_matches_sdpa_on_gathered_tokens(bs, group):
    rng = np.random.default_rng(100 + bs + group)
    hkv, d = 2, 64
    h = hkv * group
    L = 3 * bs + 5
    nb = 16
    kc, vc = _rand_pool(rng, nb, hkv, bs, d)
    table = rng.permutation(nb)[: -(-L // bs)].astype(np.int32)
    q = rng.standard_normal((h, d)).astype(np.float16)
    scale = 0.125
    out = A.paged_decode_attention_one(q, kc, vc, table, L, scale)
    # gather with explicit (block, offset) arithmetic written out here
    ks = np.stack([kc[table[t // bs], :, t % bs, :] for t in range(L)])
    vs = np.stack([vc[table[t // bs], :, t % bs, :] for t in range(L)])
    ref = _sdpa(q, ks, vs, scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    kc, vc = _rand_pool(rng, 4, 2, 16, 64)
    q = rng.standard_normal((2, 64)).astype(np.float16)
    out = A.paged_decode_attention_one(q, kc, vc, np.array([3, -1], np.int32), 1, 0.125)
    np.testing.assert_array_equal(out, vc[3, :, 0, :].astype(np.float64))


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(2)
    kc, vc = _rand_pool(rng, 8, 1, 16, 64)
    L = 37
    table = np.array([5, 1, 6], np.int32)
    q = np.zeros((1, 64), np.float16)
    out = A.paged_decode_attention_one(q, kc, vc, table, L, 0.125)
    vals = [vc[table[t // 16], 0, t % 16].astype(np.float64) for t in range(L)]
    np.testing.assert_allclose(out[0], np.mean(vals, axis=0), rtol=0, atol=1e-13)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    kc, vc = _rand_pool(rng, 8, 1, 16, 64)
    kc[:] = kc[0, 0, 0]
    L = 20
    table = np.array([2, 4], np.int32)
    q = rng.standard_normal((1, 64)).astype(np.float16)
    out = A.paged_decode_attention_one(q, kc, vc, table, L, 0.125)
    vals = [vc[table[t // 16], 0, t % 16].astype(np.float64) for t in range(L)]
    np.testing.assert_allclose(out[0], np.mean(vals, axis=0), rtol=0, atol=1e-13)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(4)
    kc, vc = _rand_pool(rng, 8, 1, 16, 64)
    L, j = 40, 23
    table = np.array([7, 2, 5], np.int32)
    kj = kc[table[j // 16], 0, j % 16].astype(np.float64)
    q = (kj / np.linalg.norm(kj) * 200.0).astype(np.float16)[None, :]
    out = A.paged_decode_attention_one(q, kc, vc, table, L, 1.0)
    np.testing.assert_allclose(out[0], vc[table[j // 16], 0, j % 16], rtol=0, atol=1e-6)


def test_block_permutation_does_not_change_output():
    """Paging changes the layout, not the output: permute the pool and remap."""
    rng = np.random.default_rng(5)
    nb, hkv, bs, d, h = 24, 4, 16, 64, 8
    kc, vc = _rand_pool(rng, nb, hkv, bs, d)
    q = rng.standard_normal((3, h, d)).astype(np.float16)
    lens = np.array([70, 16, 33], np.int32)
    tables = np.full((3, 5), -1, np.int32)
    perm0 = rng.permutation(nb)
    k = 0
    for s, L in enumerate(lens):
        n = -(-L // bs)
        tables[s, :n] = perm0[k:k + n]
        k += n
    out = A.paged_decode_attention(q, kc, vc, tables, lens, 0.125)
    sigma = rng.permutation(nb)                  # block b moves to sigma[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[sigma], vc2[sigma] = kc, vc
    t2 = np.where(tables >= 0, sigma[np.maximum(tables, 0)], -1).astype(np.int32)
    out2 = A.paged_decode_attention(q, kc2, vc2, t2, lens, 0.125)
    np.testing.assert_array_equal(out, out2)


def test_lifecycle_table_reads_as_contiguous(golden):
    """The walk 7 -> 2 -> 9 -> 4 reads the same tokens a contiguous cache holds."""
    g = golden("lifecycle.json")
    rng = np.random.default_rng(6)
    bs, d, hkv = g["block_size"], 64, 2
    L = g["token_that_allocates"] + 1
    contig_k = rng.standard_normal((L, hkv, d)).astype(np.float16)
    contig_v = rng.standard_normal((L, hkv, d)).astype(np.float16)
    order = g["free_blocks_in_order"] + [b for b in range(16) if b not in g["free_blocks_in_order"]]
    m = BlockManagerModel(16, bs, order)
    s = m.new_seq()
    slots, _ = m.append_tokens(s, L)
    assert m.tables[s] == g["blocks_after_token_48"]
    kc = np.full((16, hkv, bs, d), np.nan, np.float16)
    vc = np.full((16, hkv, bs, d), np.nan, np.float16)
    C.reshape_and_cache(contig_k, contig_v, kc, vc, np.array(slots))
    table = np.array(m.tables[s], np.int32)
    np.testing.assert_array_equal(A.gather_sequence(kc, table, L, bs), contig_k.astype(np.float64))
    q = rng.standard_normal((4, d)).astype(np.float16)
    out = A.paged_decode_attention_one(q, kc, vc, table, L, 0.125)
    np.testing.assert_allclose(out, _sdpa(q, contig_k, contig_v, 0.125), rtol=0, atol=1e-12)


def test_forked_tables_give_identical_outputs():
    rng = np.random.default_rng(7)
    bs, d, hkv, h = 16, 64, 2, 4
    m = BlockManagerModel(32, bs, rng.permutation(32))
    kc, vc = _rand_pool(rng, 32, hkv, bs, d)
    a = m.new_seq()
    m.append_tokens(a, 45)
    b = m.fork(a)
    c = m.fork(a)
    q = rng.standard_normal((h, d)).astype(np.float16)
    tables, lens = m.export([a, b, c], 4)
    outs = [A.paged_decode_attention_one(q, kc, vc, np.array(tables[i]), lens[i], 0.1)
            for i in range(3)]
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    # after b diverges (copy-on-write, then a different token), a and c still agree
    slot, cow = m.append_token(b)
    assert cow is not None and cow[0] == tables[1][2]   # b's shared partial last block is copied
    C.copy_blocks(kc, vc, [cow])
    C.reshape_and_cache(rng.standard_normal((1, hkv, d)).astype(np.float16),
                        rng.standard_normal((1, hkv, d)).astype(np.float16), kc, vc, [slot])
    tables, lens = m.export([a, b, c], 4)
    o_a = A.paged_decode_attention_one(q, kc, vc, np.array(tables[0]), lens[0], 0.1)
    o_c = A.paged_decode_attention_one(q, kc, vc, np.array(tables[2]), lens[2], 0.1)
    np.testing.assert_array_equal(o_a, outs[0])
    np.testing.assert_array_equal(o_c, outs[0])
    # b's first 45 tokens are still the shared prefix
    np.testing.assert_array_equal(A.gather_sequence(kc, np.array(tables[1]), 45, bs),
                                  A.gather_sequence(kc, np.array(tables[0]), 45, bs))


def test_gqa_head_mapping_is_consecutive_groups():
    rng = np.random.default_rng(8)
    bs, d, hkv, group = 16, 64, 2, 4
    kc, vc = _rand_pool(rng, 4, hkv, bs, d)
    kc[:, 1] = np.nan
    vc[:, 1] = np.nan                       # poison KV head 1
    q = rng.standard_normal((hkv * group, d)).astype(np.float16)
    out = A.paged_decode_attention_one(q, kc, vc, np.array([2, 0], np.int32), 20, 0.125)
    assert np.isfinite(out[:group]).all()       # heads 0..3 read KV head 0 only
    assert np.isnan(out[group:]).all()          # heads 4..7 read KV head 1


def test_reads_nothing_past_context():
    rng = np.random.default_rng(9)
    bs, d = 16, 64
    kc, vc = _rand_pool(rng, 8, 1, bs, d)
    table = np.array([6, 3, -1, -1], np.int32)
    L = 21
    mask = C.valid_slot_mask(table[None, :], [L], 8, bs)
    kc.transpose(0, 2, 1, 3)[~mask] = np.nan      # [NB][bs][Hkv][D] view
    vc.transpose(0, 2, 1, 3)[~mask] = np.nan
    assert np.isnan(kc[3, 0, 5:]).all() and np.isfinite(kc[3, 0, :5]).all()
    q = rng.standard_normal((1, d)).astype(np.float16)
    out = A.paged_decode_attention_one(q, kc, vc, table, L, 0.125)
    assert np.isfinite(out).all()
    assert mask.sum() == L and mask[6].all() and mask[3, :5].all() and not mask[3, 5:].any()


def test_empty_context_gives_zeros():
    rng = np.random.default_rng(10)
    kc, vc = _rand_pool(rng, 2, 1, 16, 64)
    q = rng.standard_normal((1, 64)).astype(np.float16)
    out = A.paged_decode_attention_one(q, kc, vc, np.array([-1], np.int32), 0, 0.125)
    assert (out == 0).all()


def test_cache_layout_offsets():
    """A slot's row sits at flat element ((blk*Hkv + h)*bs + off)*D + i."""
    nb, hkv, bs, d = 5, 3, 16, 64
    kc = np.zeros((nb, hkv, bs, d), np.float16)
    vc = np.zeros((nb, hkv, bs, d), np.float16)
    key = np.arange(hkv * d, dtype=np.float16).reshape(1, hkv, d) + 1
    slot = 3 * bs + 7
    C.reshape_and_cache(key, -key, kc, vc, [slot])
    flat = kc.reshape(-1)
    for h in range(hkv):
        base = ((3 * hkv + h) * bs + 7) * d
        np.testing.assert_array_equal(flat[base:base + d], key[0, h])
    assert np.count_nonzero(kc) == hkv * d and np.count_nonzero(vc) == hkv * d


def test_reshape_and_cache_skips_negative_slots():
    kc = np.zeros((2, 1, 4, 8), np.float16)
    vc = np.zeros_like(kc)
    key = np.ones((2, 1, 8), np.float16)
    C.reshape_and_cache(key, key, kc, vc, [-1, 5])
    assert np.count_nonzero(kc) == 8 and (kc[1, 0, 1] == 1).all()


def test_copy_blocks_copies_every_byte_and_nothing_else():
    rng = np.random.default_rng(11)
    kc, vc = _rand_pool(rng, 6, 2, 16, 64)
    k0, v0 = kc.copy(), vc.copy()
    C.copy_blocks(kc, vc, [(1, 4), (2, 0)])
    assert kc[4].tobytes() == k0[1].tobytes() and vc[4].tobytes() == v0[1].tobytes()
    assert kc[0].tobytes() == k0[2].tobytes() and vc[0].tobytes() == v0[2].tobytes()
    for b in (1, 2, 3, 5):
        assert kc[b].tobytes() == k0[b].tobytes() and vc[b].tobytes() == v0[b].tobytes()
