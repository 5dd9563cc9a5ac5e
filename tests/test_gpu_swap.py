"""Swapping on the GPU: the block manager's swap out / swap in against the
oracle model, and pkv_swap_blocks moving the blocks between the device pool
and a page-locked host pool, bit-exact against the oracle's block copies.

[P2] "Why it matters for KV cache", "Swapping and preemption": blocks go to
CPU memory under memory pressure and come back when the request resumes;
[P1] "Common misconceptions": paging does not change the numbers, so a
sequence's attention output after the round trip must be what it was.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import cache_ops as OC
from oracle.block_manager import BlockManagerModel
from pkv_testlib import TOL, Case, bits16, max_abs_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from paged_kv_cache_152_gb300 import build
    build.build()
    import paged_kv_cache_152_gb300 as m
    m.load()
    return m


def _model_at_decode_step(wl, num_host_blocks):
    model = BlockManagerModel(wl.num_blocks, wl.block_size, wl.free_order, num_host_blocks)
    W.replay(model, wl.ops)
    for s in wl.batch:
        model.append_token(s)
    return model


def _pinned_pool_like(t, num_blocks):
    pool = torch.empty((num_blocks,) + tuple(t.shape[1:]), dtype=t.dtype, pin_memory=True)
    pool.fill_(float("nan"))
    return pool


@pytest.mark.parametrize("name,kw,group", [
    ("prefix", dict(num_seqs=16, prefix_len=100), list(range(0, 16, 2))),   # shares the prefix
    ("7b", dict(num_seqs=12), [3, 0, 7, 11]),
    ("chat", dict(num_main=6, num_transient=5), [1, 2]),
])
def test_swap_round_trip_bit_exact(pkv, name, kw, group):
    wl = W.make(name, **kw)
    case = Case(wl)
    case.write_new_tokens()
    before = case.decode().clone()
    nh = wl.num_blocks
    model = _model_at_decode_step(wl, nh)
    case.alloc.host_pool(nh)
    kc, vc = case.t["key_cache"], case.t["value_cache"]
    hk, hv = _pinned_pool_like(kc, nh), _pinned_pool_like(vc, nh)
    torch.cuda.synchronize()
    o_kc, o_vc = kc.cpu().numpy(), vc.cpu().numpy()
    o_hk, o_hv = hk.numpy().copy(), hv.numpy().copy()
    st = case.status

    # swap out: the group's blocks go to the host pool
    seqs = [wl.batch[i] for i in group]
    out_pairs = case.alloc.swap_out(seqs)
    assert [tuple(p) for p in out_pairs.tolist()] == model.swap_out(seqs)
    pkv.swap_blocks(kc, vc, hk, hv, torch.from_numpy(out_pairs.astype(np.int64)).cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    OC.swap_blocks(o_kc, o_vc, o_hk, o_hv, out_pairs)
    assert np.array_equal(bits16(hk), bits16(o_hk)) and np.array_equal(bits16(hv), bits16(o_hv))

    # the freed device blocks are reused by someone else meanwhile
    free = torch.tensor(case.alloc.free_list(), dtype=torch.int64, device="cuda")
    kc[free] = float("nan")
    vc[free] = float("nan")
    o_kc[free.cpu().numpy()] = np.float16(np.nan)
    o_vc[free.cpu().numpy()] = np.float16(np.nan)

    # swap in (another order): fresh device blocks
    back = list(reversed(seqs))
    in_pairs = case.alloc.swap_in(back)
    assert [tuple(p) for p in in_pairs.tolist()] == model.swap_in(back)
    pkv.swap_blocks(hk, hv, kc, vc, torch.from_numpy(in_pairs.astype(np.int64)).cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    OC.swap_blocks(o_hk, o_hv, o_kc, o_vc, in_pairs)
    assert np.array_equal(bits16(kc), bits16(o_kc)) and np.array_equal(bits16(vc), bits16(o_vc))

    # same attention, bit for bit, through the new tables
    tables, lens = case.alloc.export(wl.batch, case.mb)
    mt, ml = model.export(wl.batch, case.mb)
    assert tables.tolist() == mt and lens.tolist() == ml
    assert tables.tolist() != case.tables.cpu().tolist()
    case.tables = torch.from_numpy(tables).cuda()
    after = case.decode(out=torch.empty_like(before))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))
    case.oracle_write_new_tokens()
    assert max_abs_err(after, case.oracle_decode(None), None) <= TOL


def test_swap_blocks_layers_bit_exact(pkv):
    rng = np.random.default_rng(21)
    L, nb, nh, hkv, bs, d = 4, 14, 9, 8, 16, 128
    dev_k = [rng.standard_normal((nb, hkv, bs, d)).astype(np.float16) for _ in range(L)]
    dev_v = [rng.standard_normal((nb, hkv, bs, d)).astype(np.float16) for _ in range(L)]
    host_k = [np.full((nh, hkv, bs, d), np.nan, np.float16) for _ in range(L)]
    host_v = [np.full((nh, hkv, bs, d), np.nan, np.float16) for _ in range(L)]
    g_k = [torch.from_numpy(x).cuda() for x in dev_k]
    g_v = [torch.from_numpy(x).cuda() for x in dev_v]
    p_k = [torch.from_numpy(x).pin_memory() for x in host_k]
    p_v = [torch.from_numpy(x).pin_memory() for x in host_v]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_pairs = [(13, 0), (2, 8), (5, 3), (0, 1)]
    pkv.swap_blocks_layers(g_k, g_v, p_k, p_v, torch.tensor(out_pairs, dtype=torch.int64, device="cuda"),
                           status=st)
    in_pairs = [(8, 6), (0, 12), (3, 7)]
    pkv.swap_blocks_layers(p_k, p_v, g_k, g_v, torch.tensor(in_pairs, dtype=torch.int64, device="cuda"),
                           status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for layer in range(L):
        OC.swap_blocks(dev_k[layer], dev_v[layer], host_k[layer], host_v[layer], out_pairs)
        OC.swap_blocks(host_k[layer], host_v[layer], dev_k[layer], dev_v[layer], in_pairs)
        assert np.array_equal(bits16(p_k[layer]), bits16(host_k[layer]))
        assert np.array_equal(bits16(p_v[layer]), bits16(host_v[layer]))
        assert np.array_equal(bits16(g_k[layer]), bits16(dev_k[layer]))
        assert np.array_equal(bits16(g_v[layer]), bits16(dev_v[layer]))


@pytest.mark.parametrize("shape", [(5, 1, 16, 64), (7, 3, 8, 64), (6, 8, 128, 128)])
def test_swap_blocks_odd_block_sizes(pkv, shape):
    """Blocks of 2 KiB (less than one 16 KiB tile), 6 KiB (a ragged tile) and
    256 KiB (16 tiles) move exactly."""
    rng = np.random.default_rng(22)
    src = rng.standard_normal(shape).astype(np.float16)
    src_v = rng.standard_normal(shape).astype(np.float16)
    g_k, g_v = torch.from_numpy(src).cuda(), torch.from_numpy(src_v).cuda()
    h_k = torch.zeros(shape, dtype=torch.float16).pin_memory()
    h_v = torch.zeros(shape, dtype=torch.float16).pin_memory()
    pairs = [(i, shape[0] - 1 - i) for i in range(shape[0])]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.swap_blocks(g_k, g_v, h_k, h_v, torch.tensor(pairs, dtype=torch.int64, device="cuda"), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(h_k.numpy(), src[::-1]) and np.array_equal(h_v.numpy(), src_v[::-1])


def test_swap_bad_pair_reports_and_skips(pkv):
    kc = torch.arange(4 * 2 * 8 * 64, dtype=torch.float16, device="cuda").view(4, 2, 8, 64)
    vc = kc.clone()
    hk = torch.zeros((3, 2, 8, 64), dtype=torch.float16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    pairs = torch.tensor([[0, 3], [4, 0], [2, 1]], dtype=torch.int64, device="cuda")  # dst 3, src 4 outside
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.swap_blocks(kc, vc, hk, hv, pairs, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == pkv.PKV_ERR_OUT_OF_RANGE
    assert torch.equal(hk[1], kc[2].cpu()) and torch.equal(hv[1], vc[2].cpu())
    assert not hk[0].any() and not hk[2].any()


def test_swap_refuses_pageable_host_memory(pkv):
    """Pageable host memory is refused on the host, before any launch."""
    import ctypes
    lib = pkv.load()
    kc = torch.zeros((4, 2, 8, 64), dtype=torch.float16, device="cuda")
    pageable = np.zeros((4, 2, 8, 64), np.float16)
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    hp = ctypes.c_void_p(pageable.ctypes.data)
    rc = lib.pkv_swap_blocks(vp(kc), vp(kc), hp, hp, vp(pairs), 1, 2 * 8 * 64 * 2, 4, 4, None,
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == pkv.PKV_ERR_INVALID_ARG
    assert not pageable.any()
    with pytest.raises(ValueError):
        pkv.swap_blocks(kc, kc, torch.zeros_like(kc, device="cpu"), torch.zeros_like(kc, device="cpu"), pairs)
