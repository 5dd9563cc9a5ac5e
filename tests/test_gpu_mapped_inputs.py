"""Serving steps whose inputs the kernel reads straight from page-locked host
memory (pkv_decode_plan_step_mapped) against the same step on inputs in
device memory.

The step's queries, new K/V rows, block tables and context lengths (and the
prefix-sharing hints) sit in one pinned host region; the plan is created on
a device region of the same layout, which the mapped step only uses as an
address.  The kernel then copies each piece's query and each new row with
16-byte lane copies over the CPU-GPU link instead of bulk copies from device
memory: the arithmetic is the same, so the outputs and the cache rows the
step writes must be the same bits as the direct call's, and within the fp64
oracle's tolerance.
"""

import ctypes

import numpy as np
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


def _region(tensors):
    """A pinned host region and a device region of the same layout (each part
    256-byte aligned), the parts copied into the host one; returns both and
    the device views the plan is created on."""
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off += -(-(t.numel() * t.element_size()) // 256) * 256
    host = torch.zeros(off, dtype=torch.uint8).pin_memory()
    dev = torch.full((off,), 0xFF, dtype=torch.uint8, device="cuda")  # never read by a mapped step
    views = []
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        host[o:o + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        views.append(dev[o:o + n].view(t.dtype).view(t.shape))
    return host, dev, views


def _step_pair(pkv, wl, append, shared, num_ctas=0):
    direct, mapped = Case(wl), Case(wl)
    hints = [torch.from_numpy(c.alloc.shared_prefix(wl.batch)).to("cuda") for c in (direct, mapped)] \
        if shared else [None, None]
    kv = dict(key=direct.t["key"], value=direct.t["value"]) if append else {}
    if not append:
        direct.write_new_tokens()
        mapped.write_new_tokens()
    plan_d = pkv.DecodePlan(direct.out, direct.t["query"], direct.t["key_cache"], direct.t["value_cache"],
                            direct.tables, direct.lens, wl.scale, status=direct.status, shared_blocks=hints[0],
                            num_ctas=num_ctas, **kv)
    parts = [mapped.t["query"]] + ([mapped.t["key"], mapped.t["value"]] if append else []) + \
        [mapped.tables, mapped.lens] + ([hints[1]] if shared else [])
    host, dev, views = _region(parts)
    q = views[0]
    k, v = (views[1], views[2]) if append else (None, None)
    tables, lens = views[3 if append else 1], views[4 if append else 2]
    sh = views[-1] if shared else None
    host_out = torch.full(tuple(mapped.out.shape), float("nan"), dtype=torch.float16).pin_memory()
    plan_h = pkv.DecodePlan(host_out, q, mapped.t["key_cache"], mapped.t["value_cache"], tables, lens, wl.scale,
                            key=k, value=v, status=mapped.status, shared_blocks=sh, num_ctas=num_ctas)
    return direct, mapped, plan_d, plan_h, host, dev, host_out


@pytest.mark.parametrize("name,kw,append,shared", [
    ("7b", dict(num_seqs=11), True, False),
    ("7b", dict(num_seqs=11), False, False),
    ("7b", dict(num_seqs=5, block_size=8), True, False),    # a chunk spans two blocks
    ("7b", dict(num_seqs=5, block_size=128), True, False),
    ("gqa", dict(num_seqs=12), True, False),                # group 4
    ("gqa", dict(num_seqs=6, block_size=64), False, False),
    ("tiny", {}, True, False),                              # head_dim 64
    ("tiny", dict(block_size=32), False, False),
    ("prefix", dict(num_seqs=17, prefix_len=40), True, True),   # the grouped kernel
    ("prefix", dict(num_seqs=9, prefix_len=40, block_size=32), False, True),
    ("forked64", {}, True, True),                           # the grouped kernel at head_dim 64
])
def test_mapped_step_matches_device_inputs(pkv, name, kw, append, shared):
    if name == "forked64":
        from test_gpu_shared import forked_workload
        wl = forked_workload(64, 64, 16, roots=((70, 9),), singles=2)
    else:
        wl = W.make(name, **kw)
    direct, mapped, plan_d, plan_h, host, dev, host_out = _step_pair(pkv, wl, append, shared)
    for _ in range(3):  # the same step again: the same bits
        plan_d.launch()
        plan_h.step_mapped(dev, host)
        torch.cuda.synchronize()
        assert int(direct.status.item()) == 0 and int(mapped.status.item()) == 0
        assert torch.equal(host_out.view(torch.int16), direct.out.cpu().view(torch.int16))
        assert torch.equal(mapped.t["key_cache"].view(torch.int16), direct.t["key_cache"].view(torch.int16))
        assert torch.equal(mapped.t["value_cache"].view(torch.int16), direct.t["value_cache"].view(torch.int16))
    assert torch.all(dev == 0xFF)  # the device region was never written
    mapped.oracle_write_new_tokens()  # by the step itself, or by reshape_and_cache before it
    assert max_abs_err(host_out, mapped.oracle_decode()) <= TOL
    plan_d.close()
    plan_h.close()


@pytest.mark.parametrize("name,kw,shared", [("7b", dict(num_seqs=6), False), ("gqa", dict(num_seqs=5), False),
                                            ("prefix", dict(num_seqs=12, prefix_len=300), True)])
@pytest.mark.parametrize("num_ctas", [1, 3, 37])
def test_mapped_step_small_grids(pkv, name, kw, shared, num_ctas):
    """Few CTAs: segments cut between workers and CTAs, merged in shared
    memory and device-wide, with the inputs read from host memory."""
    wl = W.make(name, **kw)
    direct, mapped, plan_d, plan_h, host, dev, host_out = _step_pair(pkv, wl, True, shared, num_ctas)
    for _ in range(2):
        plan_d.launch()
        plan_h.step_mapped(dev, host)
        torch.cuda.synchronize()
        assert int(direct.status.item()) == 0 and int(mapped.status.item()) == 0
        assert torch.equal(host_out.view(torch.int16), direct.out.cpu().view(torch.int16))
    mapped.oracle_write_new_tokens()
    assert max_abs_err(host_out, mapped.oracle_decode()) <= TOL
    plan_d.close()
    plan_h.close()


def test_mapped_step_moves_only_the_inputs_inside_the_region(pkv):
    """Queries and new rows in the host region, tables and lengths left in
    device memory outside it: only the inputs inside the region are read from
    host memory; the same bits as the direct call."""
    wl = W.make("7b", num_seqs=7)
    direct, mapped = Case(wl), Case(wl)
    plan_d = pkv.DecodePlan(direct.out, direct.t["query"], direct.t["key_cache"], direct.t["value_cache"],
                            direct.tables, direct.lens, wl.scale, key=direct.t["key"], value=direct.t["value"],
                            status=direct.status)
    host, dev, (q, k, v) = _region([mapped.t["query"], mapped.t["key"], mapped.t["value"]])
    host_out = torch.full(tuple(mapped.out.shape), float("nan"), dtype=torch.float16).pin_memory()
    plan_h = pkv.DecodePlan(host_out, q, mapped.t["key_cache"], mapped.t["value_cache"], mapped.tables, mapped.lens,
                            wl.scale, key=k, value=v, status=mapped.status)
    plan_d.launch()
    plan_h.step_mapped(dev, host)
    torch.cuda.synchronize()
    assert int(direct.status.item()) == 0 and int(mapped.status.item()) == 0
    assert torch.equal(host_out.view(torch.int16), direct.out.cpu().view(torch.int16))
    assert torch.equal(mapped.t["key_cache"].view(torch.int16), direct.t["key_cache"].view(torch.int16))
    plan_d.close()
    plan_h.close()


def test_mapped_step_refuses_unmapped_or_misaligned_inputs(pkv):
    """Pageable host memory and a region whose query would be misaligned are
    refused before anything is enqueued."""
    wl = W.make("7b", num_seqs=3)
    direct, mapped, plan_d, plan_h, host, dev, host_out = _step_pair(pkv, wl, True, False)
    lib = pkv.load()
    h = plan_h._h
    pageable = np.zeros(host.numel() + 64, dtype=np.uint8)
    rc = lib.pkv_decode_plan_step_mapped(h, ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(pageable.ctypes.data),
                                         host.numel(), None, None)
    assert rc == pkv.PKV_ERR_INVALID_ARG
    rc = lib.pkv_decode_plan_step_mapped(h, ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(host.data_ptr() + 8),
                                         host.numel() - 8, None, None)
    assert rc == pkv.PKV_ERR_INVALID_ARG
    rc = lib.pkv_decode_plan_step_mapped(h, ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(host.data_ptr()), 0,
                                         None, None)
    assert rc == pkv.PKV_ERR_INVALID_ARG
    # a region that ends inside its last input (the lengths): the kernel would
    # read past the host memory given, so the call is refused
    rc = lib.pkv_decode_plan_step_mapped(h, ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(host.data_ptr()),
                                         host.numel() - 256 + 4, None, None)
    assert rc == pkv.PKV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(mapped.status.item()) == 0
    assert torch.isnan(host_out).all()  # nothing ran
    plan_d.close()
    plan_h.close()
