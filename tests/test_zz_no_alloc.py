"""The decode entry point that allocates nothing.

Some users of this library cannot allocate device memory: an engine that has
given almost all GPU memory to its own KV pool and caching allocator, a
plug-in without allocation rights, or a hot loop that must not pay for a
cudaMalloc.  pkv_paged_attention_decode_noalloc serves them: it takes no
workspace and uses a fixed 16 MiB scratch array inside the library instead.

This file checks, through the C ABI:
* four calls in a row whose num_seqs * num_kv_heads grows, shrinks, grows and
  shrinks again (so later calls run over counters and partial results that
  calls of other shapes left in the shared scratch, and one comes back to the
  counter parity an earlier call used): each gives the same bits as the
  regular entry point on the same inputs and the same grid (the same kernel
  runs; only where its scratch lives differs), and one is also checked
  against the fp64 oracle within the tolerance of the other decode tests;
* a call needing more scratch than the array holds is refused before any
  launch;
* the limits stated in the header hold on a 152-SM GB300.
It is named so that pytest runs it last, and it builds everything it needs,
so it also passes on its own in a fresh process.
"""

import ctypes

import pytest
import torch

import workloads as W
from pkv_testlib import TOL, Case, max_abs_err

pytestmark = pytest.mark.gpu

SCRATCH = 16 * 1024 * 1024


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


def test_noalloc_matches_regular_entry_point_over_changing_shapes(pkv):
    # num_seqs * num_kv_heads: 192 -> 1280 -> 1600 -> 256
    shapes = [("gqa", 24), ("7b", 40), ("gqa", 200), ("7b", 8)]
    for k, (name, n) in enumerate(shapes):
        case = Case(W.make(name, num_seqs=n))
        case.write_new_tokens()
        expect = case.decode().clone()                    # regular entry, caller-owned workspace
        got = torch.full_like(expect, float("nan"))
        assert _noalloc(pkv, case, got) == pkv.PKV_OK
        torch.cuda.synchronize()
        assert int(case.status.item()) == 0, (name, n)
        # same kernel, same grid: the same bits
        assert torch.equal(got.view(torch.int16), expect.view(torch.int16)), (name, n)
        if k == len(shapes) - 1:
            # and directly against the oracle
            case.oracle_write_new_tokens()
            err = max_abs_err(got, case.oracle_decode())
            assert err <= TOL, err


def test_noalloc_refuses_calls_beyond_its_scratch(pkv):
    case = Case(W.make("gqa", num_seqs=4))
    out = torch.empty_like(case.out)
    wl = case.wl
    huge = 4096      # CTAs (the most a call may ask for): partial results far beyond 16 MiB
    need = pkv.decode_workspace_size(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                     wl.block_size, huge)
    assert need > SCRATCH
    assert _noalloc(pkv, case, out, num_ctas=huge) == pkv.PKV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(case.status.item()) == 0


@pytest.mark.parametrize("d,g,limit", [(64, 1, 1003408), (64, 8, 687408), (128, 1, 959632), (128, 8, 337200)])
def test_noalloc_limits_in_the_header(pkv, d, g, limit):
    """The header's table of the largest num_seqs * num_kv_heads that fits at
    the default grid (one CTA per SM on 152 SMs)."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the table is stated for 152 SMs")
    n = 4096
    hkv = limit // n
    size = lambda kv: pkv.decode_workspace_size(n, kv * g, kv, d, 16, 0)  # noqa: E731
    assert 0 < size(hkv) <= SCRATCH
    assert size(hkv + 1) > SCRATCH       # n * (hkv + 1) is past the limit
