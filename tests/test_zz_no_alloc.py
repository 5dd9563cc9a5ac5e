"""The decode entry point that allocates nothing.

Some users of this library cannot allocate device memory: an engine that has
given almost all GPU memory to its own KV pool and caching allocator, a
plug-in without allocation rights, or a hot loop that must not pay for a
cudaMalloc.  pkv_paged_attention_decode_noalloc serves them: it takes no
workspace and uses a fixed 16 MiB scratch array inside the library instead.

This file checks, through the C ABI, that two calls in a row (different
shapes, so the second one runs over whatever the first left in the shared
scratch) each match the regular entry point on the same inputs, within the
tolerance of the other decode tests, and that a call needing more scratch than
the array holds is refused before any launch.  It is named so that pytest runs
it last, and it builds everything it needs, so it also passes on its own in a
fresh process.
"""

import ctypes

import pytest
import torch

import workloads as W
from pkv_testlib import TOL, Case

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


def _noalloc(pkv, case, out, num_ctas=0):
    t, wl = case.t, case.wl
    p = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    return pkv.load().pkv_paged_attention_decode_noalloc(
        p(out), p(t["query"]), p(t["key_cache"]), p(t["value_cache"]), p(case.tables), case.tables.shape[1],
        p(case.lens), wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
        t["key_cache"].shape[0], ctypes.c_float(wl.scale), num_ctas, p(case.status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_regular_entry_point_twice(pkv):
    cases = [Case(W.make("gqa", num_seqs=24)), Case(W.make("7b", num_seqs=40))]
    for case in cases:
        case.write_new_tokens()
        expect = case.decode().clone()                    # regular entry, caller-owned workspace
        got = torch.full_like(expect, float("nan"))
        assert _noalloc(pkv, case, got) == pkv.PKV_OK
        torch.cuda.synchronize()
        assert int(case.status.item()) == 0
        assert torch.isfinite(got).all()
        assert (got.float() - expect.float()).abs().max().item() <= TOL


def test_noalloc_refuses_calls_beyond_its_scratch(pkv):
    case = Case(W.make("gqa", num_seqs=4))
    out = torch.empty_like(case.out)
    wl = case.wl
    huge = 4096      # CTAs (the most a call may ask for): partial results far beyond 16 MiB
    need = pkv.decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                     wl.block_size, huge)
    assert need > 16 * 1024 * 1024
    assert _noalloc(pkv, case, out, num_ctas=huge) == pkv.PKV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(case.status.item()) == 0
