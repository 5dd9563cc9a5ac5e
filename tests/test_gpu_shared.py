"""Decode with prefix sharing (the grouped kernel) against the fp64 oracle.

pkv_paged_attention_decode_shared reads the blocks that consecutive
sequences of a batch share (forks of one prompt, until copy-on-write) once
for up to 8 of them, with their queries as the rows of one tensor-core tile,
and merges each sequence's shared and own parts.  Paging and sharing do not
change the result ([P1] "Memory sharing across requests": forked requests
read the same physical blocks), so every row is checked against the plain
definition, on every pool slot the batch does not use poisoned with NaN.
"""

import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from pkv_testlib import TOL, Case, max_abs_err

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


def _shared(case):
    return torch.from_numpy(case.alloc.shared_prefix(case.wl.batch)).to("cuda")


def _decode_shared(pkv, case, shared, num_ctas=0, append=True, out=None):
    out = case.out if out is None else out
    kw = dict(key=case.t["key"], value=case.t["value"]) if append else {}
    pkv.paged_attention_decode_shared(out, case.t["query"], case.t["key_cache"], case.t["value_cache"],
                                      case.tables, case.lens, shared, case.wl.scale, num_ctas=num_ctas,
                                      status=case.status, **kw)
    return out


def _check_rows(case, out):
    torch.cuda.synchronize()
    assert int(case.status.item()) == 0
    assert torch.isfinite(out).all()
    case.oracle_write_new_tokens()
    err = max_abs_err(out, case.oracle_decode())
    assert err <= TOL, err
    return err


def forked_workload(seed, head_dim=128, block_size=16, roots=((500, 12),), singles=0, heads=4):
    """Roots with a prompt each, forked into children that each append a
    private suffix (at least one token, so that every copy-on-write happens
    before the decode step); the batch lists each root followed by its
    children, then sequences that share nothing."""
    rng = np.random.default_rng(seed)
    ops, batch, lens = [], [], {}
    nseq = 0

    def new(n):
        nonlocal nseq
        s = nseq
        nseq += 1
        ops.append(("new",))
        if n:
            ops.append(("append", s, n))
        lens[s] = n
        return s

    for prompt, kids in roots:
        r = new(prompt)
        batch.append(r)
        children = []
        for _ in range(kids):
            ops.append(("fork", r))
            c = nseq
            nseq += 1
            lens[c] = prompt
            children.append(c)
        for c in children:
            k = int(rng.integers(1, 3 * block_size))
            ops.append(("append", c, k))
            lens[c] += k
        batch += children
    for _ in range(singles):
        batch.append(new(int(rng.integers(1, 300))))
    ctx = [lens[s] + 1 for s in batch]          # the decode step appends one token each
    need = sum(-(-lens[s] // block_size) + 1 for s in range(nseq)) + 8
    free = rng.permutation(need).astype(np.int32)
    return W.Workload("forked", 9, heads, heads, head_dim, block_size, need, free, ops, batch, ctx,
                      1.0 / math.sqrt(head_dim), 9000 + seed)


@pytest.mark.parametrize("num_ctas", [0, 1, 3, 200])
def test_prefix_workload_every_row(pkv, num_ctas):
    """The prefix workload: 128 forks of a 500-token prompt (31 shared full
    blocks each), one decode step that also writes every new token."""
    case = Case(W.make("prefix"))
    shared = _shared(case)
    assert int(shared[1:].min()) >= 31
    out = _decode_shared(pkv, case, shared, num_ctas)
    _check_rows(case, out)


@pytest.mark.parametrize("kw", [dict(num_seqs=2), dict(num_seqs=9), dict(num_seqs=17, prefix_len=40)])
@pytest.mark.parametrize("num_ctas", [0, 1, 5])
def test_small_prefix_batches(pkv, kw, num_ctas):
    case = Case(W.make("prefix", **kw))
    out = _decode_shared(pkv, case, _shared(case), num_ctas)
    _check_rows(case, out)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [16, 32, 64, 128])
@pytest.mark.parametrize("append", [True, False])
def test_random_forks(pkv, d, bs, append):
    """Several roots (groups longer and shorter than 8, a root with one
    child, one with none), sequences that share nothing, every grid."""
    wl = forked_workload(d + bs, d, bs, roots=((3 * bs + 5, 11), (bs, 1), (5 * bs, 0), (2 * bs + 1, 7)),
                         singles=3)
    for num_ctas in (0, 1, 2, 37):
        case = Case(wl)
        if not append:
            case.write_new_tokens()
        out = _decode_shared(pkv, case, _shared(case), num_ctas, append=append)
        _check_rows(case, out)


def test_zero_hints_and_plans(pkv):
    """All-zero hints read every sequence on its own (same answer within
    rounding); a plan built with the hints gives the bits of the direct call,
    launch after launch; the same launch gives the same bits twice."""
    wl = forked_workload(5, roots=((300, 9),), singles=2)
    a, b = Case(wl), Case(wl)
    out_a = _decode_shared(pkv, a, _shared(a))
    zeros = torch.zeros(wl.num_seqs, dtype=torch.int32, device="cuda")
    out_b = _decode_shared(pkv, b, zeros)
    torch.cuda.synchronize()
    assert (out_a.float() - out_b.float()).abs().max().item() <= TOL
    _check_rows(a, out_a)
    # plans, and determinism
    c = Case(wl)
    shared = _shared(c)
    plan = pkv.DecodePlan(c.out, c.t["query"], c.t["key_cache"], c.t["value_cache"], c.tables, c.lens, wl.scale,
                          key=c.t["key"], value=c.t["value"], status=c.status, shared_blocks=shared)
    d = Case(wl)
    for _ in range(3):
        plan.launch()
        _decode_shared(pkv, d, shared)
        torch.cuda.synchronize()
        assert torch.equal(c.out.view(torch.int16), d.out.view(torch.int16))
        assert torch.equal(c.t["key_cache"].view(torch.int16), d.t["key_cache"].view(torch.int16))
    plan.close()
    assert int(c.status.item()) == 0 and int(d.status.item()) == 0


def test_shapes_outside_the_grouped_kernel_run_the_plain_one(pkv):
    """Group 4 (the gqa workload): the hints are not used; the bits are the
    plain decode's."""
    case, plain = Case(W.make("gqa", num_seqs=12)), Case(W.make("gqa", num_seqs=12))
    shared = torch.ones(12, dtype=torch.int32, device="cuda")   # would be wrong if it were used
    out = _decode_shared(pkv, case, shared)
    pkv.paged_attention_decode_append(plain.out, plain.t["query"], plain.t["key"], plain.t["value"],
                                      plain.t["key_cache"], plain.t["value_cache"], plain.tables, plain.lens,
                                      plain.wl.scale, status=plain.status)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), plain.out.view(torch.int16))
    _check_rows(case, out)
