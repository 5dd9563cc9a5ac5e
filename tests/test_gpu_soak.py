"""Thousands of decode launches on one workspace keep their bits.

A segment cut across CTAs is counted in device-wide on counters tagged with
an epoch kept in the workspace: every call counts on its epoch's parity and
prepares the other parity for the next call, and the last CTA out advances
the epoch.  These tests run that machinery far past a few calls -- launches
back to back, a CUDA graph of launches captured once and replayed, and calls
of two shapes taking turns on the no-allocation entry point's one scratch --
and check that every launch gives the first launch's bits with a clean status
word.  The steps append the same new tokens each time, so each launch
computes the same result.
"""

import pytest
import torch

import workloads as W
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


def _plan(pkv, case, num_ctas=0, workspace=None, shared=None):
    t = case.t
    return pkv.DecodePlan(case.out, t["query"], t["key_cache"], t["value_cache"], case.tables, case.lens,
                          case.wl.scale, key=t["key"], value=t["value"], num_ctas=num_ctas, workspace=workspace,
                          status=case.status, shared_blocks=shared)


def _bits(x):
    return x.view(torch.int16).clone()


@pytest.mark.parametrize("name,kw,num_ctas,shared", [
    ("7b", dict(num_seqs=16), 0, False),
    ("7b", dict(num_seqs=16), 37, False),     # segments cut across CTAs: device-wide counts every launch
    ("gqa", dict(num_seqs=10), 23, False),
    ("prefix", dict(num_seqs=17, prefix_len=120), 29, True),   # the grouped kernel
])
def test_thousands_of_launches_keep_their_bits(pkv, name, kw, num_ctas, shared):
    case = Case(W.make(name, **kw))
    hints = torch.from_numpy(case.alloc.shared_prefix(case.wl.batch)).to("cuda") if shared else None
    plan = _plan(pkv, case, num_ctas, shared=hints)
    sh = torch.cuda.current_stream().cuda_stream
    plan.launch_raw(sh)
    torch.cuda.synchronize()
    first = _bits(case.out)
    for block in range(6):
        for _ in range(499):
            plan.launch_raw(sh)
        plan.launch_raw(sh)
        torch.cuda.synchronize()
        assert int(case.status.item()) == 0, block
        assert torch.equal(_bits(case.out), first), block
    case.oracle_write_new_tokens()
    assert max_abs_err(case.out, case.oracle_decode()) <= TOL
    plan.close()


def test_graph_of_launches_replayed_keeps_its_bits(pkv):
    """Eight launches captured once as a CUDA graph and replayed 300 times:
    each replay reads the epoch the previous launch left, as a launch does."""
    case = Case(W.make("7b", num_seqs=12))
    plan = _plan(pkv, case, num_ctas=19)
    plan.launch()
    torch.cuda.synchronize()
    first = _bits(case.out)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        for _ in range(8):
            plan.launch()
    for r in range(300):
        g.replay()
        if r % 100 == 99:
            torch.cuda.synchronize()
            assert int(case.status.item()) == 0, r
            assert torch.equal(_bits(case.out), first), r
    plan.launch()   # a plain launch after the replays
    torch.cuda.synchronize()
    assert int(case.status.item()) == 0 and torch.equal(_bits(case.out), first)
    plan.close()


def test_two_shapes_take_turns_on_the_noalloc_scratch(pkv):
    """The no-allocation entry point keeps one scratch for every call, so
    calls of different shapes (group 1 and group 4, different counts of
    sequences and CTAs) find the counters and partials the other left there;
    400 alternations, and each shape still gives its own first bits."""
    import ctypes
    a, b = Case(W.make("7b", num_seqs=20)), Case(W.make("gqa", num_seqs=9))
    a.write_new_tokens()
    b.write_new_tokens()
    lib = pkv.load()
    sh = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(case, num_ctas):
        t, wl = case.t, case.wl
        p = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
        rc = lib.pkv_paged_attention_decode_noalloc(
            p(case.out), p(t["query"]), p(t["key_cache"]), p(t["value_cache"]), p(case.tables),
            case.tables.shape[1], p(case.lens), wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim,
            wl.block_size, t["key_cache"].shape[0], ctypes.c_float(wl.scale), num_ctas, p(case.status), sh)
        assert rc == pkv.PKV_OK

    call(a, 31)
    call(b, 0)
    torch.cuda.synchronize()
    fa, fb = _bits(a.out), _bits(b.out)
    for r in range(400):
        call(a, 31)
        call(b, 0)
        if r % 100 == 99:
            torch.cuda.synchronize()
            assert int(a.status.item()) == 0 and int(b.status.item()) == 0, r
            assert torch.equal(_bits(a.out), fa) and torch.equal(_bits(b.out), fb), r
    a.oracle_write_new_tokens()
    assert max_abs_err(a.out, a.oracle_decode()) <= TOL
