"""Argument checks of the Python binding that need no GPU: every device call
refuses host tensors, wrong element types, non-contiguous views and
inconsistent shapes before it reaches the library, and the block manager's
batch calls refuse output arrays they could overrun."""

import numpy as np
import pytest
import torch

import paged_kv_cache_152_gb300 as pkv


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_152_gb300 import build
    build.build()


def decode_args(n=2, h=4, hkv=2, d=64, nb=6, bs=16, mb=3):
    f16 = dict(dtype=torch.float16)
    return dict(out=torch.zeros(n, h, d, **f16), query=torch.zeros(n, h, d, **f16),
                key_cache=torch.zeros(nb, hkv, bs, d, **f16), value_cache=torch.zeros(nb, hkv, bs, d, **f16),
                block_tables=torch.zeros(n, mb, dtype=torch.int32), context_lens=torch.ones(n, dtype=torch.int32),
                scale=d ** -0.5)


def test_decode_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA"):
        pkv.paged_attention_decode(**decode_args())
    a = decode_args()
    with pytest.raises(ValueError, match="CUDA"):
        pkv.paged_attention_decode_append(key=torch.zeros(2, 2, 64, dtype=torch.float16),
                                          value=torch.zeros(2, 2, 64, dtype=torch.float16), **a)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.DecodePlan(**decode_args())


@pytest.mark.parametrize("name,bad", [
    ("query", torch.zeros(2, 4, 64, dtype=torch.float32)),
    ("key_cache", torch.zeros(6, 2, 16, 64, dtype=torch.bfloat16)),
    ("block_tables", torch.zeros(2, 3, dtype=torch.int64)),
    ("context_lens", torch.ones(2, dtype=torch.int64)),
])
def test_decode_refuses_wrong_element_types(name, bad):
    a = decode_args()
    a[name] = bad
    with pytest.raises(TypeError, match=name):
        pkv.paged_attention_decode(**a)


def test_decode_refuses_views_and_wrong_ranks():
    a = decode_args()
    a["query"] = torch.zeros(4, 2, 64, dtype=torch.float16).transpose(0, 1)   # [2][4][64], not contiguous
    with pytest.raises(ValueError, match="contiguous"):
        pkv.paged_attention_decode(**a)
    a = decode_args()
    a["block_tables"] = torch.zeros(6, dtype=torch.int32)
    with pytest.raises(ValueError, match="dims"):
        pkv.paged_attention_decode(**a)


def test_cache_ops_refuse_host_tensors_and_types():
    f16 = dict(dtype=torch.float16)
    k = torch.zeros(3, 2, 64, **f16)
    kc = torch.zeros(4, 2, 16, 64, **f16)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.reshape_and_cache(k, k, kc, kc, torch.zeros(3, dtype=torch.int64))
    with pytest.raises(TypeError, match="slot_mapping"):
        pkv.reshape_and_cache(k, k, kc, kc, torch.zeros(3, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA"):
        pkv.copy_blocks(kc, kc, torch.zeros(1, 2, dtype=torch.int64))
    with pytest.raises(TypeError, match="block_pairs"):
        pkv.copy_blocks(kc, kc, torch.zeros(1, 2, dtype=torch.int32))
    with pytest.raises(ValueError, match="per layer"):
        pkv.reshape_and_cache_layers([k], [k, k], [kc], [kc], torch.zeros(3, dtype=torch.int64))
    with pytest.raises(ValueError, match="per layer"):
        pkv.copy_blocks_layers([], [], torch.zeros(1, 2, dtype=torch.int64))


def test_swap_refuses_pageable_host_pools():
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="page-locked"):
        pkv.swap_blocks(kc, kc, kc, kc, torch.zeros(1, 2, dtype=torch.int64))


def test_selftest_needs_a_status_word():
    with pytest.raises(ValueError, match="status"):
        pkv.selftest_wait_timeout(None, 10 ** 6)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.selftest_wait_timeout(torch.zeros(1, dtype=torch.int32), 10 ** 6)


def test_allocator_batch_calls_refuse_short_or_mistyped_outputs():
    a = pkv.BlockAllocator(8, 4)
    seqs = [a.new_seq() for _ in range(3)]
    with pytest.raises(ValueError):
        a.append_batch(seqs, slots_out=np.zeros(2, dtype=np.int64))                 # one slot short
    with pytest.raises(ValueError):
        a.append_batch(seqs, slots_out=np.zeros(3, dtype=np.int32))                 # wrong type
    with pytest.raises(ValueError):
        a.export(seqs, 2, tables_out=np.zeros((3, 2), dtype=np.int32)[:, :1])      # a strided view
    assert a.num_free() == 8                                                        # nothing was allocated
    slots, _ = a.append_batch(seqs)
    assert len(slots) == 3 and a.num_free() == 5


def test_one_call_one_device():
    """Device tensors of one call on two GPUs, or a stream on another GPU, are
    refused before anything launches (stand-ins carry only a device)."""
    from types import SimpleNamespace as NS
    on = lambda i: NS(device=torch.device("cuda", i))  # noqa: E731
    host = NS(device=torch.device("cpu"))
    with pytest.raises(ValueError, match="same CUDA device"):
        pkv._one_device((on(0), on(1), None))
    with pytest.raises(ValueError, match="same CUDA device"):
        pkv._one_device((host, None))
    with pytest.raises(ValueError, match="stream"):
        pkv._one_device((on(1), host, on(1)), stream=on(0))


@pytest.mark.gpu
def test_status_word_and_workspace_are_checked():
    """With every other argument valid on the GPU: a status word that is not
    an int32 CUDA tensor with one element, or a host workspace, is refused
    before the call reaches the library (nothing launches)."""
    a = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in decode_args().items()}
    with pytest.raises(TypeError, match="status"):
        pkv.paged_attention_decode(status=torch.zeros(1, dtype=torch.int64, device="cuda"), **a)
    with pytest.raises(ValueError, match="status must be a CUDA"):
        pkv.paged_attention_decode(status=torch.zeros(1, dtype=torch.int32), **a)
    with pytest.raises(ValueError, match="workspace"):
        pkv.paged_attention_decode(workspace=torch.zeros(1 << 20, dtype=torch.uint8), **a)
    k = torch.zeros(2, 2, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError, match="status"):
        pkv.reshape_and_cache(k, k, a["key_cache"], a["value_cache"],
                              torch.zeros(2, dtype=torch.int64, device="cuda"),
                              status=torch.zeros(0, dtype=torch.int32, device="cuda"))


def test_nvtx_ranges_are_opt_in():
    """PKV_NVTX=1 wraps every device call in an NVTX range (a refused call
    still raises through it); without it the calls are the plain functions."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    probe = ("import torch, paged_kv_cache_152_gb300 as pkv\n"
             "fns = [pkv.paged_attention_decode, pkv.reshape_and_cache, pkv.copy_blocks, pkv.swap_blocks,\n"
             "       pkv.DecodePlan.launch, pkv.DecodePlan.step]\n"
             "print(pkv.NVTX, all(hasattr(f, '__wrapped__') for f in fns))\n"
             "try:\n"
             "    pkv.copy_blocks(torch.zeros(2, 1, 16, 64, dtype=torch.float16),\n"
             "                    torch.zeros(2, 1, 16, 64, dtype=torch.float16), torch.zeros(1, 2, dtype=torch.int64))\n"
             "except ValueError:\n"
             "    print('refused')\n")
    for flag, expect in (("1", "True True\nrefused"), ("0", "False False\nrefused")):
        r = subprocess.run([sys.executable, "-c", probe], cwd=root, capture_output=True, text=True,
                           env=dict(os.environ, PKV_NVTX=flag))
        assert r.returncode == 0, r.stderr
        assert r.stdout.strip() == expect
