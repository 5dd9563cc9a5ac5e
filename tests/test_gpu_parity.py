"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

* decode attention: max abs error <= 2e-3 (fp16 output, fp32 accumulation);
* reshape_and_cache, copy_blocks: bit-exact;
* every pool slot a sequence does not use holds NaN, so any read past a
  context shows up in the output.

Sizes: the five workloads at full size with every output row checked,
shrunken versions of them on several grids, a brute-force sweep over small
shapes, and edge cases.
"""

import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import cache_ops as OC
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


def _status(case):
    torch.cuda.synchronize()
    return int(case.status.item())


def _full_check(case, seqs, num_ctas=0):
    case.write_new_tokens()
    case.oracle_write_new_tokens()
    torch.cuda.synchronize()
    # the write is bit-exact over the whole pool (NaN poison included)
    assert np.array_equal(bits16(case.t["key_cache"]), bits16(case.o_kc))
    assert np.array_equal(bits16(case.t["value_cache"]), bits16(case.o_vc))
    out = case.decode(num_ctas)
    assert _status(case) == 0
    assert torch.isfinite(out).all()
    ref = case.oracle_decode(seqs)
    err = max_abs_err(out, ref, seqs)
    assert err <= TOL, err
    return out, err


# -- the five workloads ---------------------------------------------------------

def test_tiny_all_rows(pkv):
    case = Case(W.make("tiny"))
    _full_check(case, None)


@pytest.mark.parametrize("name", ["7b", "chat", "gqa", "prefix"])
def test_full_size_all_rows(pkv, name):
    """Every output row of the full-size workload, on the default grid (the
    launch the bench times), against the fp64 oracle."""
    wl = W.make(name)
    case = Case(wl)
    out, _ = _full_check(case, None)
    # deterministic: the same launch gives the same bits
    out2 = case.decode(0, out=torch.empty_like(out))
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


@pytest.mark.parametrize("name,kw", [("7b", dict(num_seqs=9)), ("chat", dict(num_main=6, num_transient=5)),
                                     ("gqa", dict(num_seqs=7)), ("prefix", dict(num_seqs=5))])
@pytest.mark.parametrize("num_ctas", [0, 1, 3, 200])
def test_small_all_rows_any_grid(pkv, name, kw, num_ctas):
    """Every row, and the same answer whatever the grid cuts the work into."""
    case = Case(W.make(name, **kw))
    _full_check(case, None, num_ctas)


def test_single_pass_and_split_agree(pkv):
    case = Case(W.make("gqa", num_seqs=16))
    case.write_new_tokens()
    a = case.decode(1, out=torch.empty_like(case.out)).clone()
    b = case.decode(0, out=torch.empty_like(case.out)).clone()
    c = case.decode(997, out=torch.empty_like(case.out)).clone()
    torch.cuda.synchronize()
    assert (a.float() - b.float()).abs().max().item() <= TOL
    assert (a.float() - c.float()).abs().max().item() <= TOL
    assert _status(case) == 0


# -- brute force over shapes ------------------------------------------------------

def _random_case(rng, n, h, hkv, d, bs, lens, device="cuda", poison=True):
    """Tables from a shuffled pool, tokens written by the oracle side only."""
    nblk = [-(-int(L) // bs) for L in lens]
    nb = max(1, sum(nblk) + 3)
    mb = max(1, max(nblk))
    perm = rng.permutation(nb)
    tables = np.full((n, mb), -1, np.int32)
    k = 0
    for s in range(n):
        tables[s, :nblk[s]] = perm[k:k + nblk[s]]
        k += nblk[s]
    kc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    vc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    if poison:
        mask = OC.valid_slot_mask(tables, lens, nb, bs)
        kc.transpose(0, 2, 1, 3)[~mask] = np.nan
        vc.transpose(0, 2, 1, 3)[~mask] = np.nan
    q = rng.standard_normal((n, h, d)).astype(np.float16)
    return q, kc, vc, tables, np.asarray(lens, np.int32)


def _run_gpu(pkv, q, kc, vc, tables, lens, scale, num_ctas=0):
    dev = "cuda"
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_attention_decode(out, torch.from_numpy(q).to(dev), torch.from_numpy(kc).to(dev),
                               torch.from_numpy(vc).to(dev), torch.from_numpy(tables).to(dev),
                               torch.from_numpy(lens).to(dev), scale, num_ctas=num_ctas, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), int(st.item())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_brute_force_shapes(pkv, d, bs, group):
    rng = np.random.default_rng(d * 1000 + bs * 10 + group)
    hkv = 2
    h = hkv * group
    lens = [1, bs - 1 if bs > 1 else 1, bs, bs + 1, 3 * bs + 5, 70, 0, 2 * bs]
    n = len(lens)
    q, kc, vc, tables, lens = _random_case(rng, n, h, hkv, d, bs, lens)
    scale = 1.0 / math.sqrt(d)
    ref = OA.paged_decode_attention(q, kc, vc, tables, lens, scale)
    for num_ctas in (0, 1, 2, 7):
        out, st = _run_gpu(pkv, q, kc, vc, tables, lens, scale, num_ctas)
        assert st == 0
        assert np.isfinite(out).all()
        assert np.max(np.abs(out - ref)) <= TOL, (num_ctas, np.max(np.abs(out - ref)))
        assert (out[lens == 0] == 0).all()


@pytest.mark.parametrize("d,bs,group,hkv,max_len", [(128, 16, 8, 1, 24), (64, 128, 2, 1, 24)])
def test_maximum_batch(pkv, d, bs, group, hkv, max_len):
    """num_seqs at its limit (4096): the per-sequence arrays take the most
    shared memory there; short contexts (some empty) plus one long one that is
    cut across workers; every row against the oracle, on the default grid and
    on a single CTA."""
    rng = np.random.default_rng(4096 + d + bs)
    n = 4096
    lens = rng.integers(0, max_len + 1, n)
    lens[rng.random(n) < 0.05] = 0
    lens[1234] = 3000
    q, kc, vc, tables, lens = _random_case(rng, n, hkv * group, hkv, d, bs, lens)
    scale = 1.0 / math.sqrt(d)
    ref = OA.paged_decode_attention(q, kc, vc, tables, lens, scale)
    for num_ctas in (0, 1):
        out, st = _run_gpu(pkv, q, kc, vc, tables, lens, scale, num_ctas)
        assert st == 0
        assert np.isfinite(out).all()
        assert np.max(np.abs(out - ref)) <= TOL, (num_ctas, np.max(np.abs(out - ref)))
        assert (out[lens == 0] == 0).all()


def test_long_context_and_many_pieces(pkv):
    """One 32k-token sequence among short ones: cut across many workers."""
    rng = np.random.default_rng(5)
    lens = [32768, 3, 700, 1]
    q, kc, vc, tables, lens = _random_case(rng, 4, 8, 2, 128, 32, lens)
    ref = OA.paged_decode_attention(q, kc, vc, tables, lens, 0.08)
    out, st = _run_gpu(pkv, q, kc, vc, tables, lens, 0.08)
    assert st == 0 and np.max(np.abs(out - ref)) <= TOL


def test_large_scores_stay_finite(pkv):
    """Scores of several hundred: the online softmax must rescale, not overflow."""
    rng = np.random.default_rng(6)
    lens = [300, 45]
    q, kc, vc, tables, lens = _random_case(rng, 2, 4, 4, 128, 16, lens)
    q = (q.astype(np.float32) * 8).astype(np.float16)
    ref = OA.paged_decode_attention(q, kc, vc, tables, lens, 1.0)
    out, st = _run_gpu(pkv, q, kc, vc, tables, lens, 1.0)
    assert st == 0 and np.isfinite(out).all() and np.max(np.abs(out - ref)) <= TOL


def test_block_permutation_and_identity_tables_agree(pkv):
    """Paging is exact: shuffled and contiguous placements give the same answer."""
    rng = np.random.default_rng(7)
    lens = [100, 257, 33]
    q, kc, vc, tables, lens = _random_case(rng, 3, 8, 8, 128, 16, lens, poison=False)
    out_a, _ = _run_gpu(pkv, q, kc, vc, tables, lens, 0.1, num_ctas=1)
    sigma = rng.permutation(kc.shape[0])
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[sigma], vc2[sigma] = kc, vc
    t2 = np.where(tables >= 0, sigma[np.maximum(tables, 0)], -1).astype(np.int32)
    out_b, _ = _run_gpu(pkv, q, kc2, vc2, t2, lens, 0.1, num_ctas=1)
    # a single worker walks every sequence whole: identical arithmetic, identical bits
    assert np.array_equal(out_a, out_b)


def test_forked_prefix_rows_identical_single_pass(pkv):
    """Two forks with the same prefix and query give the same bits (one worker)."""
    import paged_kv_cache_152_gb300 as m
    a = m.BlockAllocator(64, 16, np.random.default_rng(8).permutation(64))
    root = a.new_seq()
    a.append_tokens(root, 77)
    kids = [a.fork(root) for _ in range(3)]
    tables, lens = a.export([root] + kids, 8)
    rng = np.random.default_rng(9)
    kc = rng.standard_normal((64, 4, 16, 128)).astype(np.float16)
    vc = rng.standard_normal((64, 4, 16, 128)).astype(np.float16)
    q1 = rng.standard_normal((1, 8, 128)).astype(np.float16)
    q = np.repeat(q1, 4, axis=0)
    out, st = _run_gpu(pkv, q, kc, vc, tables, lens, 0.1, num_ctas=1)
    assert st == 0
    for i in range(1, 4):
        assert np.array_equal(out[0], out[i])
    ref = OA.paged_decode_attention(q, kc, vc, tables, lens, 0.1)
    assert np.max(np.abs(out - ref)) <= TOL


# -- cache ops ------------------------------------------------------------------

def test_reshape_and_cache_bit_exact_with_skips(pkv):
    rng = np.random.default_rng(10)
    nb, hkv, bs, d, t = 20, 4, 16, 128, 37
    kc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    vc = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    key = rng.standard_normal((t, hkv, d)).astype(np.float16)
    val = rng.standard_normal((t, hkv, d)).astype(np.float16)
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[[3, 11]] = -1
    dev = "cuda"
    gk, gv = torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.reshape_and_cache(torch.from_numpy(key).to(dev), torch.from_numpy(val).to(dev), gk, gv,
                          torch.from_numpy(slots).to(dev), status=st)
    OC.reshape_and_cache(key, val, kc, vc, slots)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(bits16(gk), bits16(kc)) and np.array_equal(bits16(gv), bits16(vc))


def test_reshape_and_cache_out_of_range_slot_reports(pkv):
    dev = "cuda"
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)
    key = torch.ones((2, 2, 64), dtype=torch.float16, device=dev)
    slots = torch.tensor([5, 4 * 16], dtype=torch.int64, device=dev)   # second one is past the pool
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.reshape_and_cache(key, key, kc, vc, slots, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == pkv.PKV_ERR_OUT_OF_RANGE
    assert int((kc != 0).sum().item()) == 2 * 64          # only the valid token landed


def test_copy_blocks_prefix_divergence_bit_exact(pkv):
    """The prefix workload's first divergent step: 127 copy-on-write copies."""
    import paged_kv_cache_152_gb300 as m
    from oracle.block_manager import BlockManagerModel
    wl = W.make("prefix")
    alloc = m.BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
    model = BlockManagerModel(wl.num_blocks, wl.block_size, wl.free_order)
    stop = wl.marks["divergence"]
    W.replay(alloc, wl.ops, 0, stop)
    W.replay(model, wl.ops, 0, stop)
    step = [op[1] for op in wl.ops[stop:wl.marks["after_divergence"]]]
    slots, pairs = alloc.append_batch(step)
    exp = [model.append_token(s) for s in step]
    assert slots.tolist() == [e[0] for e in exp]
    assert [tuple(p) for p in pairs.tolist()] == [e[1] for e in exp if e[1] is not None]
    assert len(pairs) == 127 and m.validate_block_pairs(pairs, wl.num_blocks)
    t = W.tensors(wl, "cuda")
    o_kc, o_vc = t["key_cache"].cpu().numpy(), t["value_cache"].cpu().numpy()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dpairs = torch.from_numpy(pairs.astype(np.int64)).cuda()
    m.copy_blocks(t["key_cache"], t["value_cache"], dpairs, status=st)
    key = t["key"][:len(step)].contiguous()
    val = t["value"][:len(step)].contiguous()
    m.reshape_and_cache(key, val, t["key_cache"], t["value_cache"],
                        torch.from_numpy(slots.astype(np.int64)).cuda(), status=st)
    OC.copy_blocks(o_kc, o_vc, [e[1] for e in exp if e[1] is not None])
    OC.reshape_and_cache(key.cpu().numpy(), val.cpu().numpy(), o_kc, o_vc, slots)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(bits16(t["key_cache"]), bits16(o_kc))
    assert np.array_equal(bits16(t["value_cache"]), bits16(o_vc))


def test_copy_blocks_bad_pair_reports_and_skips(pkv):
    dev = "cuda"
    kc = torch.arange(4 * 2 * 8 * 64, dtype=torch.float16, device=dev).view(4, 2, 8, 64)
    vc = kc.clone()
    before = kc.clone()
    pairs = torch.tensor([[0, 9], [1, 2]], dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.copy_blocks(kc, vc, pairs, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == pkv.PKV_ERR_OUT_OF_RANGE
    assert torch.equal(kc[2], before[1]) and torch.equal(kc[0], before[0]) and torch.equal(kc[3], before[3])


# -- device-side error reporting ----------------------------------------------------

def test_bad_table_entry_and_long_context_report(pkv):
    rng = np.random.default_rng(11)
    lens = [40, 20]
    q, kc, vc, tables, lens_a = _random_case(rng, 2, 4, 4, 64, 16, lens, poison=False)
    bad = tables.copy()
    bad[0, 1] = kc.shape[0] + 5                       # outside the pool
    _, st = _run_gpu(pkv, q, kc, vc, bad, lens_a, 0.1)
    assert st == pkv.PKV_ERR_OUT_OF_RANGE
    long = lens_a.copy()
    long[1] = tables.shape[1] * 16 + 1                # longer than its table row
    _, st = _run_gpu(pkv, q, kc, vc, tables, long, 0.1)
    assert st == pkv.PKV_ERR_OUT_OF_RANGE
    out, st = _run_gpu(pkv, q, kc, vc, tables, lens_a, 0.1)   # the context is still usable
    assert st == 0 and np.isfinite(out).all()


def test_bounded_wait_gives_up_and_context_survives(pkv):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.selftest_wait_timeout(st, 2_000_000)          # 2 ms on a barrier nothing completes
    torch.cuda.synchronize()
    assert int(st.item()) == pkv.PKV_ERR_DEVICE_TIMEOUT
    case = Case(W.make("tiny"))
    case.write_new_tokens()
    case.decode()
    torch.cuda.synchronize()
    assert int(case.status.item()) == 0 and torch.isfinite(case.out).all()


def test_workspace_contents_do_not_matter(pkv):
    """One workspace, pre-filled with garbage, reused by calls with different grids."""
    case = Case(W.make("gqa", num_seqs=20))
    case.write_new_tokens()
    case.oracle_write_new_tokens()
    ref = case.oracle_decode()
    wl = case.wl
    grids = [37, 37, 5, 200, 37, 1]
    size = max(pkv.decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                         wl.block_size, g) for g in grids)
    ws = torch.full((size,), 0xFF, dtype=torch.uint8, device="cuda")
    for i, g in enumerate(grids):
        if i == 3:
            ws.random_(0, 256)
        out = torch.full_like(case.out, float("nan"))
        pkv.paged_attention_decode(out, case.t["query"], case.t["key_cache"], case.t["value_cache"],
                                   case.tables, case.lens, wl.scale, num_ctas=g, workspace=ws,
                                   status=case.status)
        torch.cuda.synchronize()
        assert int(case.status.item()) == 0
        assert max_abs_err(out, ref) <= TOL, (g, max_abs_err(out, ref))


@pytest.mark.parametrize("bs", [8, 32, 64, 128])
def test_block_size_sweep_full_size(pkv, bs):
    """The 7B-class workload at every supported block size ([P1] 'Worked
    example': the block-size trade-off), every row against the oracle."""
    wl = W.make("7b", block_size=bs)
    case = Case(wl)
    _full_check(case, None)


def test_reshape_and_cache_layers_bit_exact(pkv):
    """One launch writes every layer's new tokens ([P2]: a block spans all layers)."""
    rng = np.random.default_rng(12)
    L, nb, hkv, bs, d, t = 5, 12, 4, 16, 128, 21
    dev = "cuda"
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[4] = -1
    kcs = [rng.standard_normal((nb, hkv, bs, d)).astype(np.float16) for _ in range(L)]
    vcs = [rng.standard_normal((nb, hkv, bs, d)).astype(np.float16) for _ in range(L)]
    keys = [rng.standard_normal((t, hkv, d)).astype(np.float16) for _ in range(L)]
    vals = [rng.standard_normal((t, hkv, d)).astype(np.float16) for _ in range(L)]
    g_kc = [torch.from_numpy(x).to(dev) for x in kcs]
    g_vc = [torch.from_numpy(x).to(dev) for x in vcs]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.reshape_and_cache_layers([torch.from_numpy(x).to(dev) for x in keys],
                                 [torch.from_numpy(x).to(dev) for x in vals], g_kc, g_vc,
                                 torch.from_numpy(slots).to(dev), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for layer in range(L):
        OC.reshape_and_cache(keys[layer], vals[layer], kcs[layer], vcs[layer], slots)
        assert np.array_equal(bits16(g_kc[layer]), bits16(kcs[layer]))
        assert np.array_equal(bits16(g_vc[layer]), bits16(vcs[layer]))


def test_copy_blocks_layers_bit_exact(pkv):
    rng = np.random.default_rng(13)
    L, nb, hkv, bs, d = 3, 10, 2, 16, 64
    dev = "cuda"
    kcs = [rng.standard_normal((nb, hkv, bs, d)).astype(np.float16) for _ in range(L)]
    vcs = [rng.standard_normal((nb, hkv, bs, d)).astype(np.float16) for _ in range(L)]
    pairs = [(1, 7), (3, 0), (5, 9)]
    assert pkv.validate_block_pairs(pairs, nb)
    g_kc = [torch.from_numpy(x).to(dev) for x in kcs]
    g_vc = [torch.from_numpy(x).to(dev) for x in vcs]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.copy_blocks_layers(g_kc, g_vc, torch.tensor(pairs, dtype=torch.int64, device=dev), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for layer in range(L):
        OC.copy_blocks(kcs[layer], vcs[layer], pairs)
        assert np.array_equal(bits16(g_kc[layer]), bits16(kcs[layer]))
        assert np.array_equal(bits16(g_vc[layer]), bits16(vcs[layer]))


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("7b", dict(num_seqs=11)), ("gqa", dict(num_seqs=9)),
                                     ("chat", dict(num_main=5, num_transient=4)), ("7b", {}),
                                     ("7b", dict(num_seqs=11, block_size=8)), ("tiny", dict(block_size=8)),
                                     ("gqa", dict(num_seqs=9, block_size=8))])
@pytest.mark.parametrize("num_ctas", [0, 3])
def test_decode_append_equals_write_then_decode(pkv, name, kw, num_ctas):
    """The fused append + attend launch gives the same cache bits and the same
    output bits as reshape_and_cache followed by decode, and matches the oracle."""
    wl = W.make(name, **kw)
    fused, split = Case(wl), Case(wl)
    pkv.paged_attention_decode_append(fused.out, fused.t["query"], fused.t["key"], fused.t["value"],
                                      fused.t["key_cache"], fused.t["value_cache"], fused.tables, fused.lens,
                                      wl.scale, num_ctas=num_ctas, status=fused.status)
    split.write_new_tokens()
    split.decode(num_ctas)
    torch.cuda.synchronize()
    assert int(fused.status.item()) == 0 and int(split.status.item()) == 0
    assert torch.equal(fused.t["key_cache"].view(torch.int16), split.t["key_cache"].view(torch.int16))
    assert torch.equal(fused.t["value_cache"].view(torch.int16), split.t["value_cache"].view(torch.int16))
    assert torch.equal(fused.out.view(torch.int16), split.out.view(torch.int16))
    fused.oracle_write_new_tokens()
    assert max_abs_err(fused.out, fused.oracle_decode()) <= TOL


@pytest.mark.parametrize("name,kw", [("7b", dict(num_seqs=11)), ("gqa", dict(num_seqs=9)), ("tiny", {})])
def test_decode_plan_equals_direct_calls(pkv, name, kw):
    """A DecodePlan launch gives the bits of the direct call it was built from,
    launch after launch, with the buffers' contents changing in between."""
    wl = W.make(name, **kw)
    direct, planned = Case(wl), Case(wl)
    plan = pkv.DecodePlan(planned.out, planned.t["query"], planned.t["key_cache"], planned.t["value_cache"],
                          planned.tables, planned.lens, wl.scale, key=planned.t["key"], value=planned.t["value"],
                          status=planned.status)
    read_only = pkv.DecodePlan(torch.empty_like(planned.out), planned.t["query"], planned.t["key_cache"],
                               planned.t["value_cache"], planned.tables, planned.lens, wl.scale,
                               status=planned.status)
    for step in range(3):
        if step:
            # new queries for both sides (same values), same tables
            q = torch.randn_like(direct.t["query"].float()).half()
            direct.t["query"].copy_(q)
            planned.t["query"].copy_(q)
        pkv.paged_attention_decode_append(direct.out, direct.t["query"], direct.t["key"], direct.t["value"],
                                          direct.t["key_cache"], direct.t["value_cache"], direct.tables,
                                          direct.lens, wl.scale, status=direct.status)
        plan.launch()
        ro = read_only.launch()
        torch.cuda.synchronize()
        assert int(direct.status.item()) == 0 and int(planned.status.item()) == 0
        assert torch.equal(planned.out.view(torch.int16), direct.out.view(torch.int16))
        assert torch.equal(ro.view(torch.int16), direct.out.view(torch.int16))
        assert torch.equal(planned.t["key_cache"].view(torch.int16), direct.t["key_cache"].view(torch.int16))
    plan.close()
    read_only.close()


@pytest.mark.gpu
def test_decode_plan_step_stages_inputs_and_output(pkv):
    """pkv_decode_plan_step: the step's inputs staged in one host region go in
    with one copy, the plan runs, the output comes back to the host; the same
    bits as the direct call on the same inputs, step after step."""
    wl = W.make("tiny")
    direct = Case(wl)
    n, h, d = direct.t["query"].shape
    hkv = direct.t["key"].shape[1]
    mb = direct.tables.shape[1]
    # staging layout: query | key | value | tables | lengths, each 256-byte aligned
    parts = [("q", n * h * d * 2), ("k", n * hkv * d * 2), ("v", n * hkv * d * 2), ("tab", n * mb * 4), ("len", n * 4)]
    offs, off = {}, 0
    for nm, nb in parts:
        offs[nm] = (off, nb)
        off += -(-nb // 256) * 256
    dev = torch.empty(off, dtype=torch.uint8, device="cuda")
    host = torch.zeros(off, dtype=torch.uint8).pin_memory()

    def view(buf, nm, dtype, shape):
        o, nb = offs[nm]
        return buf[o:o + nb].view(dtype).view(*shape)

    staged = Case(wl)  # its caches; inputs come from the staging region
    out = torch.empty_like(direct.out)
    plan = pkv.DecodePlan(out, view(dev, "q", torch.float16, (n, h, d)), staged.t["key_cache"],
                          staged.t["value_cache"], view(dev, "tab", torch.int32, (n, mb)),
                          view(dev, "len", torch.int32, (n,)), wl.scale, key=view(dev, "k", torch.float16, (n, hkv, d)),
                          value=view(dev, "v", torch.float16, (n, hkv, d)), status=staged.status)
    host_out = torch.empty(out.shape, dtype=torch.float16).pin_memory()
    view(host, "tab", torch.int32, (n, mb)).copy_(direct.tables.cpu())
    view(host, "len", torch.int32, (n,)).copy_(direct.lens.cpu())
    for step in range(3):
        q = torch.randn_like(direct.t["query"].float()).half()
        k = torch.randn_like(direct.t["key"].float()).half()
        v = torch.randn_like(direct.t["value"].float()).half()
        direct.t["query"].copy_(q)
        direct.t["key"].copy_(k)
        direct.t["value"].copy_(v)
        view(host, "q", torch.float16, (n, h, d)).copy_(q.cpu())
        view(host, "k", torch.float16, (n, hkv, d)).copy_(k.cpu())
        view(host, "v", torch.float16, (n, hkv, d)).copy_(v.cpu())
        pkv.paged_attention_decode_append(direct.out, direct.t["query"], direct.t["key"], direct.t["value"],
                                          direct.t["key_cache"], direct.t["value_cache"], direct.tables,
                                          direct.lens, wl.scale, status=direct.status)
        plan.step(dev, host, host_out)
        torch.cuda.synchronize()
        assert int(direct.status.item()) == 0 and int(staged.status.item()) == 0
        assert torch.equal(host_out.view(torch.int16), direct.out.cpu().view(torch.int16))
        assert torch.equal(staged.t["key_cache"].view(torch.int16), direct.t["key_cache"].view(torch.int16))
    # no input copy, no output copy: a plain launch
    plan.step()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), direct.out.view(torch.int16))
    with pytest.raises(ValueError):
        plan.step(dev[:16], host)
    plan.close()


def test_decode_plan_writes_mapped_host_output(pkv):
    """A plan whose out is pinned host memory: the kernel writes the output
    over the CPU-GPU link, with the bits of the device-output plan; host
    memory the device cannot reach (pageable) is refused before any launch."""
    import ctypes
    wl = W.make("7b", num_seqs=11)
    dev_case, host_case = Case(wl), Case(wl)
    host_out = torch.full(tuple(dev_case.out.shape), float("nan"), dtype=torch.float16).pin_memory()
    plans = []
    for case, out in ((dev_case, dev_case.out), (host_case, host_out)):
        plans.append(pkv.DecodePlan(out, case.t["query"], case.t["key_cache"], case.t["value_cache"], case.tables,
                                    case.lens, wl.scale, key=case.t["key"], value=case.t["value"],
                                    status=case.status))
    for step in range(3):
        for pl in plans:
            pl.launch()
        torch.cuda.synchronize()
        assert int(dev_case.status.item()) == 0 and int(host_case.status.item()) == 0
        assert torch.equal(host_out.view(torch.int16), dev_case.out.cpu().view(torch.int16))
        assert torch.equal(host_case.t["key_cache"].view(torch.int16), dev_case.t["key_cache"].view(torch.int16))
    for pl in plans:
        pl.close()
    host_case.oracle_write_new_tokens()
    assert max_abs_err(host_out, host_case.oracle_decode()) <= TOL
    # pageable host memory: refused by the library's pointer check
    pageable = np.zeros(host_out.numel(), dtype=np.float16)
    t = host_case.t
    h = ctypes.c_void_p()
    p = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    ws = pkv.new_workspace(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, 0)
    rc = pkv.load().pkv_decode_plan_create(
        ctypes.c_void_p(pageable.ctypes.data), p(t["query"]), None, None, p(t["key_cache"]), p(t["value_cache"]),
        p(host_case.tables), host_case.tables.shape[1], p(host_case.lens), wl.num_seqs, wl.num_heads,
        wl.num_kv_heads, wl.head_dim, wl.block_size, t["key_cache"].shape[0], ctypes.c_float(wl.scale), 0, p(ws),
        ws.numel(), None, ctypes.byref(h))
    assert rc == pkv.PKV_ERR_INVALID_ARG and h.value is None
    with pytest.raises(ValueError):
        pkv.DecodePlan(torch.empty_like(host_out), t["query"], t["key_cache"], t["value_cache"], host_case.tables,
                       host_case.lens, wl.scale)


@pytest.mark.parametrize("d,h,hkv,bs,lens", [
    (128, 4, 4, 16, [16384]),           # group 1: 1,024-chunk segments over many CTAs, partials in shared memory
    (128, 16, 4, 32, [9000, 40, 5000]),  # group 4
    (128, 16, 2, 16, [12000, 7]),        # group 8 at head_dim 128: partials in the workspace
    (64, 8, 2, 16, [20000]),             # head_dim 64
])
@pytest.mark.parametrize("num_ctas", [0, 37, 300])
def test_segments_spanning_many_ctas(pkv, d, h, hkv, bs, lens, num_ctas):
    """Long segments cut over many workers and CTAs: pieces merge within each
    CTA, then the CTAs' parts merge; same result as the oracle, and the same
    bits from launch to launch."""
    rng = np.random.default_rng(77 + d + h + len(lens))
    q, kc, vc, tables, lens_a = _random_case(rng, len(lens), h, hkv, d, bs, lens)
    scale = d ** -0.5
    ref = OA.paged_decode_attention(q, kc, vc, tables, lens_a, scale)
    out, st = _run_gpu(pkv, q, kc, vc, tables, lens_a, scale, num_ctas)
    assert st == 0 and np.max(np.abs(out - ref)) <= TOL
    out2, st2 = _run_gpu(pkv, q, kc, vc, tables, lens_a, scale, num_ctas)
    assert st2 == 0 and np.array_equal(out, out2)
