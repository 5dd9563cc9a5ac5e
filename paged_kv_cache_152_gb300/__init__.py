"""Python binding of libpkv.so, the paged KV cache library for GB300 (sm_103a).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels or its C++ block manager.  Functions take torch tensors (device
memory and streams are torch's) and pass raw pointers, sizes and the current
CUDA stream to the C ABI declared in include/pkv.h.  If the shared library is
missing or fails to load, every call raises -- there is no fallback.  The
library launches on the current CUDA device, so each call runs with the device
its tensors live on made current (they must all share one).

Names mirror the C ABI without its ``pkv_`` prefix:

* paged_attention_decode(out, query, key_cache, value_cache, block_tables,
  context_lens, scale, ...)
* reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, ...)
* copy_blocks(key_cache, value_cache, block_pairs, ...)
* swap_blocks(src_key, src_value, dst_key, dst_value, block_pairs, ...)
* DecodePlan: pkv_decode_plan_* (validate once, launch every step)
* the *_layers variants, one launch for every layer's pool
* BlockAllocator: pkv_alloc_* / pkv_seq_* / pkv_append_* / pkv_fork /
  pkv_release / pkv_export_tables / pkv_swap_out / pkv_swap_in.
"""

import contextlib
import ctypes
import functools
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_OUT_OF_BLOCKS = 2
PKV_ERR_CUDA = 3
PKV_ERR_DEVICE_TIMEOUT = 4
PKV_ERR_OUT_OF_RANGE = 5
PKV_ERR_NOT_FOUND = 6
PKV_ERR_UNSUPPORTED = 7
PKV_ERR_SWAPPED = 8

# Every symbol include/pkv.h declares, with (restype, argtypes).
_c_int, _c_size, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_intp = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [_c_int]),
    "pkv_version": (_c_int, []),
    "pkv_paged_attention_decode": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int,
                                            _c_int, _c_int, _c_int, ctypes.c_float, _c_int, _vp, _c_size,
                                            _vp, _vp]),
    "pkv_paged_attention_decode_append": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int,
                                                   _c_int, _c_int, _c_int, _c_int, _c_int, ctypes.c_float,
                                                   _c_int, _vp, _c_size, _vp, _vp]),
    "pkv_decode_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "pkv_paged_attention_decode_shared": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _vp, _c_int,
                                                   _c_int, _c_int, _c_int, _c_int, _c_int, ctypes.c_float,
                                                   _c_int, _vp, _c_size, _vp, _vp]),
    "pkv_decode_workspace_size_shared": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "pkv_paged_attention_decode_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int,
                                                    _c_int, _c_int, _c_int, _c_int, ctypes.c_float, _c_int,
                                                    _vp, _vp]),
    "pkv_decode_default_ctas": (_c_int, [_c_int, _c_int, _c_int, _c_int]),
    "pkv_reshape_and_cache": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                       _vp, _vp]),
    "pkv_copy_blocks": (_c_int, [_vp, _vp, _vp, _c_int, _c_size, _c_int, _vp, _vp]),
    "pkv_validate_block_pairs": (_c_int, [_i64p, _c_int, _c_int]),
    "pkv_reshape_and_cache_layers": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int,
                                              _c_int, _vp, _vp]),
    "pkv_copy_blocks_layers": (_c_int, [_vp, _vp, _c_int, _vp, _c_int, _c_size, _c_int, _vp, _vp]),
    "pkv_alloc_create": (_c_int, [_c_int, _c_int, _i32p, ctypes.POINTER(_vp)]),
    "pkv_alloc_destroy": (None, [_vp]),
    "pkv_alloc_save": (_c_int, [_vp, _vp, _c_size, ctypes.POINTER(_c_size)]),
    "pkv_alloc_load": (_c_int, [_vp, _c_size, ctypes.POINTER(_vp)]),
    "pkv_seq_new": (_c_int, [_vp, _intp]),
    "pkv_append_token": (_c_int, [_vp, _c_int, _i64p, _i32p]),
    "pkv_append_tokens": (_c_int, [_vp, _c_int, _c_int, _i64p, _i32p, _intp]),
    "pkv_append_batch": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _vp]),  # (void*: raw addresses are cheapest)
    "pkv_fork": (_c_int, [_vp, _c_int, _intp]),
    "pkv_release": (_c_int, [_vp, _c_int, _intp]),
    "pkv_export_tables": (_c_int, [_vp, _vp, _c_int, _vp, _c_int, _vp]),
    "pkv_export_shared_prefix": (_c_int, [_vp, _vp, _c_int, _vp]),
    "pkv_seq_length": (_c_int, [_vp, _c_int, _intp]),
    "pkv_seq_num_blocks": (_c_int, [_vp, _c_int, _intp]),
    "pkv_seq_table": (_c_int, [_vp, _c_int, _i32p, _c_int, _intp]),
    "pkv_block_refcount": (_c_int, [_vp, _c_int, _intp]),
    "pkv_block_fill": (_c_int, [_vp, _c_int, _intp]),
    "pkv_num_free": (_c_int, [_vp, _intp]),
    "pkv_free_list": (_c_int, [_vp, _i32p, _c_int, _intp]),
    "pkv_selftest_wait_timeout": (_c_int, [_vp, ctypes.c_uint64, _vp]),
    "pkv_swap_blocks": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_size, _c_int, _c_int, _vp, _vp]),
    "pkv_swap_blocks_layers": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_size, _c_int, _c_int,
                                        _vp, _vp]),
    "pkv_decode_plan_create": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int,
                                        _c_int, _c_int, _c_int, ctypes.c_float, _c_int, _vp, _c_size, _vp,
                                        ctypes.POINTER(_vp)]),
    "pkv_decode_plan_create_shared": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _vp, _c_int,
                                               _c_int, _c_int, _c_int, _c_int, _c_int, ctypes.c_float, _c_int,
                                               _vp, _c_size, _vp, ctypes.POINTER(_vp)]),
    "pkv_decode_plan_launch": (_c_int, [_vp, _vp]),
    "pkv_decode_plan_step": (_c_int, [_vp, _vp, _vp, _c_size, _vp, _vp]),
    "pkv_decode_plan_step_mapped": (_c_int, [_vp, _vp, _vp, _c_size, _vp, _vp]),
    "pkv_decode_plan_destroy": (None, [_vp]),
    "pkv_alloc_host_pool": (_c_int, [_vp, _c_int, _i32p]),
    "pkv_swap_out": (_c_int, [_vp, _i32p, _c_int, _i32p, _c_int, _intp]),
    "pkv_swap_in": (_c_int, [_vp, _i32p, _c_int, _i32p, _c_int, _intp]),
    "pkv_seq_swapped": (_c_int, [_vp, _c_int, _intp]),
    "pkv_host_block_refcount": (_c_int, [_vp, _c_int, _intp]),
    "pkv_host_block_fill": (_c_int, [_vp, _c_int, _intp]),
    "pkv_num_free_host": (_c_int, [_vp, _intp]),
    "pkv_host_free_list": (_c_int, [_vp, _i32p, _c_int, _intp]),
}

_lib = None


class PkvError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class OutOfBlocks(PkvError):
    pass


class SwappedOut(PkvError):
    pass


def load(path=None):
    """Load libpkv.so (once) and attach the C signatures.  Raises if missing.

    The in-tree build is used unless PKV_LIBRARY names another build of the
    same sources (tuning variants)."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = os.environ.get("PKV_LIBRARY", LIB_PATH)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run paged_kv_cache_152_gb300.build.build() "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


_load_library = load

# PKV_NVTX=1 (read at import): every device call is an NVTX range named after
# it, for profilers that filter or group by range (ncu --nvtx).  Off by
# default; the functions are then the plain ones.
NVTX = os.environ.get("PKV_NVTX") == "1"


def _traced(fn):
    if not NVTX:
        return fn
    import torch
    name = "pkv." + fn.__qualname__

    @functools.wraps(fn)
    def ranged(*args, **kwargs):
        torch.cuda.nvtx.range_push(name)
        try:
            return fn(*args, **kwargs)
        finally:
            torch.cuda.nvtx.range_pop()
    return ranged


def status_string(status):
    return load().pkv_status_string(int(status)).decode()


def _check(status, what):
    if status == PKV_ERR_OUT_OF_BLOCKS:
        raise OutOfBlocks(status, what)
    if status == PKV_ERR_SWAPPED:
        raise SwappedOut(status, what)
    if status != PKV_OK:
        raise PkvError(status, what)


# ---------------------------------------------------------------------------
# device calls

def _out_array(a, dtype, min_items, name):
    """Output arrays handed to the library by address: C-contiguous, of the
    element type the call writes, and large enough."""
    if a.dtype != dtype or not a.flags["C_CONTIGUOUS"] or a.size < min_items:
        raise ValueError(f"{name}: need a C-contiguous {np.dtype(dtype).name} array of >= {min_items} items")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name, ndim=None, device=True):
    import torch
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {tuple(t.shape)}")
    return torch


def _need_all(*specs):
    """_need over (tensor, dtype, name, ndim) specs: every element type,
    layout and rank first, then that every tensor is on a CUDA device."""
    for t, dtype, name, ndim in specs:
        _need(t, dtype, name, ndim, device=False)
    for t, _, name, _ in specs:
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor")


def _status_ptr(status):
    """The caller's device status word: None, or an int32 CUDA tensor."""
    if status is None:
        return None
    _need(status, __import__("torch").int32, "status")
    if status.numel() < 1:
        raise ValueError("status must hold at least one int32")
    return _ptr(status)


def _workspace(ws):
    """A caller-given decode workspace: contiguous device memory (its size
    and alignment are checked by the library)."""
    if ws.device.type != "cuda" or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return _ptr(ws), ws.numel() * ws.element_size()


def _device_guard(index):
    """Make CUDA device `index` current for one library call."""
    import torch
    return contextlib.nullcontext() if torch.cuda.current_device() == index else torch.cuda.device(index)


def _one_device(tensors, stream=None):
    """The device guard for a call on `tensors` (host tensors and None are
    skipped): all CUDA tensors, and the stream if given, on one device."""
    devs = {t.device.index for t in tensors if t is not None and t.device.type == "cuda"}
    if len(devs) != 1:
        raise ValueError("the device tensors of one call must all be on the same CUDA device")
    index = devs.pop()
    if stream is not None and stream.device.index != index:
        raise ValueError(f"stream is on {stream.device}, the tensors on cuda:{index}")
    return _device_guard(index)


def decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas=0):
    return int(load().pkv_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                num_ctas))


def decode_default_ctas(num_heads, num_kv_heads, head_dim, block_size):
    return int(load().pkv_decode_default_ctas(num_heads, num_kv_heads, head_dim, block_size))


def decode_workspace_size_shared(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas=0):
    return int(load().pkv_decode_workspace_size_shared(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                       num_ctas))


def new_workspace(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas=0, device="cuda",
                  shared=False):
    """A device workspace of the size pkv_decode_workspace_size (shared:
    pkv_decode_workspace_size_shared) asks for."""
    import torch
    size = decode_workspace_size_shared if shared else decode_workspace_size
    n = size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_ctas)
    if n == 0:
        raise PkvError(PKV_ERR_UNSUPPORTED, "decode_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


@_traced
def paged_attention_decode(out, query, key_cache, value_cache, block_tables, context_lens, scale,
                           num_ctas=0, workspace=None, status=None, stream=None):
    """pkv_paged_attention_decode on torch tensors (see include/pkv.h).

    out, query: fp16 [N][H][D]; key_cache, value_cache: fp16 [NB][Hkv][bs][D];
    block_tables: int32 [N][MB]; context_lens: int32 [N]; status: int32 [1]
    device tensor or None.  A workspace is allocated (by torch) when None.
    """
    import torch
    _need_all((query, torch.float16, "query", 3), (out, torch.float16, "out", 3),
              (key_cache, torch.float16, "key_cache", 4), (value_cache, torch.float16, "value_cache", 4),
              (block_tables, torch.int32, "block_tables", 2), (context_lens, torch.int32, "context_lens", 1))
    n, h, d = query.shape
    nb, hkv, bs, d2 = key_cache.shape
    if tuple(out.shape) != (n, h, d) or d2 != d or tuple(value_cache.shape) != tuple(key_cache.shape) \
            or block_tables.shape[0] != n or context_lens.shape[0] != n:
        raise ValueError("inconsistent shapes")
    with _one_device((out, query, key_cache, value_cache, block_tables, context_lens, workspace, status), stream):
        if workspace is None:
            workspace = new_workspace(n, h, hkv, d, bs, num_ctas, query.device)
        ws, ws_bytes = _workspace(workspace)
        rc = load().pkv_paged_attention_decode(
            _ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
            block_tables.shape[1], _ptr(context_lens), n, h, hkv, d, bs, nb, float(scale), int(num_ctas),
            ws, ws_bytes, _status_ptr(status), _stream(stream))
    _check(rc, "pkv_paged_attention_decode")
    return out


@_traced
def paged_attention_decode_append(out, query, key, value, key_cache, value_cache, block_tables, context_lens,
                                  scale, num_ctas=0, workspace=None, status=None, stream=None):
    """pkv_paged_attention_decode_append: write each sequence's new token
    (key/value fp16 [N][Hkv][D], position context_len - 1) and attend, in one
    launch."""
    import torch
    _need_all((query, torch.float16, "query", 3), (key, torch.float16, "key", 3),
              (value, torch.float16, "value", 3), (out, torch.float16, "out", 3),
              (key_cache, torch.float16, "key_cache", 4), (value_cache, torch.float16, "value_cache", 4),
              (block_tables, torch.int32, "block_tables", 2), (context_lens, torch.int32, "context_lens", 1))
    n, h, d = query.shape
    nb, hkv, bs, d2 = key_cache.shape
    if tuple(out.shape) != (n, h, d) or d2 != d or tuple(value_cache.shape) != tuple(key_cache.shape) \
            or tuple(key.shape) != (n, hkv, d) or tuple(value.shape) != (n, hkv, d) \
            or block_tables.shape[0] != n or context_lens.shape[0] != n:
        raise ValueError("inconsistent shapes")
    with _one_device((out, query, key, value, key_cache, value_cache, block_tables, context_lens, workspace,
                      status), stream):
        if workspace is None:
            workspace = new_workspace(n, h, hkv, d, bs, num_ctas, query.device)
        ws, ws_bytes = _workspace(workspace)
        rc = load().pkv_paged_attention_decode_append(
            _ptr(out), _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
            _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), n, h, hkv, d, bs, nb, float(scale),
            int(num_ctas), ws, ws_bytes, _status_ptr(status), _stream(stream))
    _check(rc, "pkv_paged_attention_decode_append")
    return out


@_traced
def paged_attention_decode_shared(out, query, key_cache, value_cache, block_tables, context_lens, shared_blocks,
                                  scale, key=None, value=None, num_ctas=0, workspace=None, status=None,
                                  stream=None):
    """pkv_paged_attention_decode_shared: decode (with key/value: append the
    new tokens and attend) reading blocks that consecutive sequences share
    once for all of them.  shared_blocks: int32 [N] CUDA tensor, entry s the
    leading blocks sequence s shares with s - 1 (BlockAllocator.shared_prefix).
    A workspace (shared layout) is allocated when None."""
    import torch
    if (key is None) != (value is None):
        raise ValueError("key and value go together")
    specs = [(query, torch.float16, "query", 3), (out, torch.float16, "out", 3),
             (key_cache, torch.float16, "key_cache", 4), (value_cache, torch.float16, "value_cache", 4),
             (block_tables, torch.int32, "block_tables", 2), (context_lens, torch.int32, "context_lens", 1),
             (shared_blocks, torch.int32, "shared_blocks", 1)]
    if key is not None:
        specs += [(key, torch.float16, "key", 3), (value, torch.float16, "value", 3)]
    _need_all(*specs)
    n, h, d = query.shape
    nb, hkv, bs, d2 = key_cache.shape
    if key is not None and (tuple(key.shape) != (n, hkv, d) or tuple(value.shape) != (n, hkv, d)):
        raise ValueError("inconsistent shapes")
    if tuple(out.shape) != (n, h, d) or d2 != d or tuple(value_cache.shape) != tuple(key_cache.shape) \
            or block_tables.shape[0] != n or context_lens.shape[0] != n or shared_blocks.shape[0] != n:
        raise ValueError("inconsistent shapes")
    with _one_device((out, query, key, value, key_cache, value_cache, block_tables, context_lens, shared_blocks,
                      workspace, status), stream):
        if workspace is None:
            workspace = new_workspace(n, h, hkv, d, bs, num_ctas, query.device, shared=True)
        ws, ws_bytes = _workspace(workspace)
        rc = load().pkv_paged_attention_decode_shared(
            _ptr(out), _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
            _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), _ptr(shared_blocks), n, h, hkv, d, bs,
            nb, float(scale), int(num_ctas), ws, ws_bytes, _status_ptr(status), _stream(stream))
    _check(rc, "pkv_paged_attention_decode_shared")
    return out


class DecodePlan:
    """pkv_decode_plan_*: a decode call validated once and launched many
    times with the same tensors (their contents may change between launches).
    With key/value given, each launch appends the new tokens and attends
    (paged_attention_decode_append); without, it only attends.  The plan keeps
    references to every tensor it was built from, and launch() and step() run
    on their device; launch_raw() and step_raw() expect it to be current.

    out may also be a pinned (page-locked) host tensor: the kernel then writes
    the output over the CPU-GPU link as rows become final, and a serving step
    needs no copy back (step() without host_out); read it once the stream has
    passed the launch."""

    def __init__(self, out, query, key_cache, value_cache, block_tables, context_lens, scale, key=None,
                 value=None, num_ctas=0, workspace=None, status=None, shared_blocks=None):
        import torch
        if (key is None) != (value is None):
            raise ValueError("key and value go together")
        if shared_blocks is not None:
            _need(shared_blocks, torch.int32, "shared_blocks", 1)
            if shared_blocks.shape[0] != query.shape[0]:
                raise ValueError("inconsistent shapes")
        specs = [(query, torch.float16, "query", 3),
                 (key_cache, torch.float16, "key_cache", 4), (value_cache, torch.float16, "value_cache", 4),
                 (block_tables, torch.int32, "block_tables", 2), (context_lens, torch.int32, "context_lens", 1)]
        if key is not None:
            specs += [(key, torch.float16, "key", 3), (value, torch.float16, "value", 3)]
        _need(out, torch.float16, "out", 3, device=False)
        if out.device.type != "cuda" and not out.is_pinned():
            raise ValueError("out must be a CUDA tensor or a pinned host tensor")
        _need_all(*specs)
        n, h, d = query.shape
        nb, hkv, bs, d2 = key_cache.shape
        if key is not None:
            if tuple(key.shape) != (n, hkv, d) or tuple(value.shape) != (n, hkv, d):
                raise ValueError("inconsistent shapes")
        if tuple(out.shape) != (n, h, d) or d2 != d or tuple(value_cache.shape) != tuple(key_cache.shape) \
                or block_tables.shape[0] != n or context_lens.shape[0] != n:
            raise ValueError("inconsistent shapes")
        self._lib = load()
        handle = ctypes.c_void_p()
        with _one_device((out, query, key, value, key_cache, value_cache, block_tables, context_lens, workspace,
                          status, shared_blocks)):
            if workspace is None:
                workspace = new_workspace(n, h, hkv, d, bs, num_ctas, query.device, shared=shared_blocks is not None)
            ws, ws_bytes = _workspace(workspace)
            if shared_blocks is None:
                rc = self._lib.pkv_decode_plan_create(
                    _ptr(out), _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                    _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), n, h, hkv, d, bs, nb,
                    float(scale), int(num_ctas), ws, ws_bytes, _status_ptr(status), ctypes.byref(handle))
            else:
                rc = self._lib.pkv_decode_plan_create_shared(
                    _ptr(out), _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                    _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), _ptr(shared_blocks), n, h, hkv,
                    d, bs, nb, float(scale), int(num_ctas), ws, ws_bytes, _status_ptr(status),
                    ctypes.byref(handle))
        _check(rc, "pkv_decode_plan_create")
        self._keep = (out, query, key, value, key_cache, value_cache, block_tables, context_lens, workspace,
                      status, shared_blocks)
        self._device = query.device.index
        self._h = handle
        self.out = out

    def _guard(self, stream):
        if stream is not None and stream.device.index != self._device:
            raise ValueError(f"stream is on {stream.device}, the plan on cuda:{self._device}")
        return _device_guard(self._device)

    @_traced
    def launch(self, stream=None):
        with self._guard(stream):
            _check(self._lib.pkv_decode_plan_launch(self._h, _stream(stream)), "pkv_decode_plan_launch")
        return self.out

    def launch_raw(self, stream_handle):
        """launch() on a stream given as its raw handle (an int), for loops
        that look the stream up once."""
        _check(self._lib.pkv_decode_plan_launch(self._h, stream_handle), "pkv_decode_plan_launch")

    @_traced
    def step(self, dev_in=None, host_in=None, host_out=None, stream=None):
        """One serving step (pkv_decode_plan_step): host_in -> dev_in (same
        byte size; the region the plan's inputs live in), the launch, then
        out -> host_out.  Host tensors should be pinned; the caller
        synchronises the stream before reading host_out."""
        nbytes = 0
        if host_in is not None:
            if dev_in is None or host_in.numel() * host_in.element_size() != dev_in.numel() * dev_in.element_size():
                raise ValueError("host_in and dev_in must have the same byte size")
            if host_in.is_cuda or not dev_in.is_cuda or not host_in.is_contiguous() or not dev_in.is_contiguous():
                raise ValueError("host_in must be a contiguous host tensor and dev_in a contiguous CUDA tensor")
            nbytes = host_in.numel() * host_in.element_size()
        if host_out is not None:
            if host_out.is_cuda or not host_out.is_contiguous() or \
                    host_out.numel() * host_out.element_size() != self.out.numel() * self.out.element_size():
                raise ValueError("host_out must be a contiguous host tensor the size of out")
        if nbytes and dev_in.device.index != self._device:
            raise ValueError(f"dev_in is on {dev_in.device}, the plan on cuda:{self._device}")
        with self._guard(stream):
            _check(self._lib.pkv_decode_plan_step(self._h, _ptr(dev_in) if nbytes else None,
                                                  _ptr(host_in) if nbytes else None, nbytes,
                                                  _ptr(host_out), _stream(stream)), "pkv_decode_plan_step")
        return host_out

    def step_mapped(self, dev_base, host_in, host_out=None, stream=None):
        """One serving step whose inputs the kernel reads straight from the
        pinned host tensor host_in (pkv_decode_plan_step_mapped): each plan
        input inside dev_base (the device region the plan was created on,
        same byte size, not touched) is read at the same offset of host_in.
        Then out -> host_out as in step().  The caller must not write host_in
        until the stream has passed the launch."""
        nbytes = host_in.numel() * host_in.element_size()
        if host_in.is_cuda or not host_in.is_contiguous() or not dev_base.is_cuda or \
                nbytes != dev_base.numel() * dev_base.element_size():
            raise ValueError("host_in must be a contiguous pinned host tensor the byte size of dev_base")
        if host_out is not None and (host_out.is_cuda or not host_out.is_contiguous() or
                                     host_out.numel() * host_out.element_size() !=
                                     self.out.numel() * self.out.element_size()):
            raise ValueError("host_out must be a contiguous host tensor the size of out")
        with self._guard(stream):
            _check(self._lib.pkv_decode_plan_step_mapped(self._h, _ptr(dev_base), _ptr(host_in), nbytes,
                                                         _ptr(host_out), _stream(stream)),
                   "pkv_decode_plan_step_mapped")
        return host_out

    def step_mapped_raw(self, dev_base_ptr, host_in_ptr, nbytes, host_out_ptr, stream_handle):
        """step_mapped() with raw pointers (ints) and a raw stream handle."""
        _check(self._lib.pkv_decode_plan_step_mapped(self._h, dev_base_ptr, host_in_ptr, nbytes, host_out_ptr,
                                                     stream_handle), "pkv_decode_plan_step_mapped")

    def step_raw(self, dev_in_ptr, host_in_ptr, nbytes, host_out_ptr, stream_handle):
        """step() with raw pointers (ints) and a raw stream handle, unchecked
        beyond what the library checks, for loops that resolve them once."""
        _check(self._lib.pkv_decode_plan_step(self._h, dev_in_ptr, host_in_ptr, nbytes, host_out_ptr,
                                              stream_handle), "pkv_decode_plan_step")

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_decode_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


@_traced
def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, status=None, stream=None):
    """pkv_reshape_and_cache: key/value fp16 [T][Hkv][D], slot_mapping int64 [T]."""
    import torch
    _need_all((key, torch.float16, "key", 3), (value, torch.float16, "value", 3),
              (key_cache, torch.float16, "key_cache", 4), (value_cache, torch.float16, "value_cache", 4),
              (slot_mapping, torch.int64, "slot_mapping", 1))
    t, hkv, d = key.shape
    nb, hkv2, bs, d2 = key_cache.shape
    if hkv2 != hkv or d2 != d or tuple(value.shape) != tuple(key.shape) or slot_mapping.shape[0] != t:
        raise ValueError("inconsistent shapes")
    with _one_device((key, value, key_cache, value_cache, slot_mapping, status), stream):
        rc = load().pkv_reshape_and_cache(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                          _ptr(slot_mapping), t, hkv, d, bs, nb, _status_ptr(status),
                                          _stream(stream))
    _check(rc, "pkv_reshape_and_cache")


@_traced
def copy_blocks(key_cache, value_cache, block_pairs, status=None, stream=None):
    """pkv_copy_blocks: block_pairs int64 [n][2] (src, dst) on the device."""
    import torch
    _need_all((key_cache, torch.float16, "key_cache", 4), (value_cache, torch.float16, "value_cache", 4),
              (block_pairs, torch.int64, "block_pairs", 2))
    nb = key_cache.shape[0]
    block_bytes = key_cache[0].numel() * key_cache.element_size()
    with _one_device((key_cache, value_cache, block_pairs, status), stream):
        rc = load().pkv_copy_blocks(_ptr(key_cache), _ptr(value_cache), _ptr(block_pairs),
                                    block_pairs.shape[0], block_bytes, nb, _status_ptr(status), _stream(stream))
    _check(rc, "pkv_copy_blocks")


def _ptr_array(tensors):
    arr = (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])
    return arr


@_traced
def reshape_and_cache_layers(keys, values, key_caches, value_caches, slot_mapping, status=None, stream=None):
    """pkv_reshape_and_cache_layers: lists (one entry per layer) of key/value
    fp16 [T][Hkv][D] and pools fp16 [NB][Hkv][bs][D]; one slot mapping."""
    torch = __import__("torch")
    n = len(keys)
    if not (len(values) == len(key_caches) == len(value_caches) == n) or n == 0:
        raise ValueError("one key, value, key_cache and value_cache per layer")
    for t in list(keys) + list(values):
        _need(t, torch.float16, "key/value", 3)
    for t in list(key_caches) + list(value_caches):
        _need(t, torch.float16, "cache", 4)
        if tuple(t.shape) != tuple(key_caches[0].shape):
            raise ValueError("every layer's pool must have the same shape")
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    t_, hkv, d = keys[0].shape
    nb, _, bs, _ = key_caches[0].shape
    ka, va, kca, vca = _ptr_array(keys), _ptr_array(values), _ptr_array(key_caches), _ptr_array(value_caches)
    with _one_device(list(keys) + list(values) + list(key_caches) + list(value_caches) + [slot_mapping, status],
                     stream):
        rc = load().pkv_reshape_and_cache_layers(ka, va, kca, vca, n, _ptr(slot_mapping), t_, hkv, d, bs, nb,
                                                 _status_ptr(status), _stream(stream))
    _check(rc, "pkv_reshape_and_cache_layers")


@_traced
def copy_blocks_layers(key_caches, value_caches, block_pairs, status=None, stream=None):
    """pkv_copy_blocks_layers: the same (src, dst) pairs in every layer's pool."""
    torch = __import__("torch")
    n = len(key_caches)
    if len(value_caches) != n or n == 0:
        raise ValueError("one key_cache and value_cache per layer")
    for t in list(key_caches) + list(value_caches):
        _need(t, torch.float16, "cache", 4)
    _need(block_pairs, torch.int64, "block_pairs", 2)
    nb = key_caches[0].shape[0]
    block_bytes = key_caches[0][0].numel() * key_caches[0].element_size()
    with _one_device(list(key_caches) + list(value_caches) + [block_pairs, status], stream):
        rc = load().pkv_copy_blocks_layers(_ptr_array(key_caches), _ptr_array(value_caches), n,
                                           _ptr(block_pairs), block_pairs.shape[0], block_bytes, nb,
                                           _status_ptr(status), _stream(stream))
    _check(rc, "pkv_copy_blocks_layers")


def _pool(t, name):
    """A swap pool: fp16 [NB][Hkv][bs][D], contiguous, on the GPU or in
    page-locked host memory (the library checks the pointer as well)."""
    torch = _need(t, __import__("torch").float16, name, 4, device=False)
    if t.device.type == "cpu" and not t.is_pinned():
        raise ValueError(f"{name}: a host pool must be page-locked (pin_memory)")
    return torch


@_traced
def swap_blocks(src_key, src_value, dst_key, dst_value, block_pairs, status=None, stream=None):
    """pkv_swap_blocks: copy block src of the source pools over block dst of
    the destination pools for each (src, dst) in block_pairs (int64 [n][2],
    device).  One side is normally a pinned host pool."""
    torch = _pool(src_key, "src_key")
    for t, name in ((src_value, "src_value"), (dst_key, "dst_key"), (dst_value, "dst_value")):
        _pool(t, name)
    if tuple(src_key.shape[1:]) != tuple(dst_key.shape[1:]) or src_key.shape != src_value.shape \
            or dst_key.shape != dst_value.shape:
        raise ValueError("source and destination pools must have the same block shape")
    _need(block_pairs, torch.int64, "block_pairs", 2)
    block_bytes = src_key[0].numel() * src_key.element_size()
    with _one_device((src_key, src_value, dst_key, dst_value, block_pairs, status), stream):
        rc = load().pkv_swap_blocks(_ptr(src_key), _ptr(src_value), _ptr(dst_key), _ptr(dst_value),
                                    _ptr(block_pairs), block_pairs.shape[0], block_bytes, src_key.shape[0],
                                    dst_key.shape[0], _status_ptr(status), _stream(stream))
    _check(rc, "pkv_swap_blocks")


@_traced
def swap_blocks_layers(src_keys, src_values, dst_keys, dst_values, block_pairs, status=None, stream=None):
    """pkv_swap_blocks_layers: swap_blocks for every layer in one launch."""
    torch = __import__("torch")
    n = len(src_keys)
    if not (len(src_values) == len(dst_keys) == len(dst_values) == n) or n == 0:
        raise ValueError("one source and one destination pool pair per layer")
    for t in list(src_keys) + list(src_values):
        _pool(t, "source pool")
        if tuple(t.shape) != tuple(src_keys[0].shape):
            raise ValueError("every layer's source pool must have the same shape")
    for t in list(dst_keys) + list(dst_values):
        _pool(t, "destination pool")
        if tuple(t.shape) != tuple(dst_keys[0].shape):
            raise ValueError("every layer's destination pool must have the same shape")
    if tuple(src_keys[0].shape[1:]) != tuple(dst_keys[0].shape[1:]):
        raise ValueError("source and destination pools must have the same block shape")
    _need(block_pairs, torch.int64, "block_pairs", 2)
    block_bytes = src_keys[0][0].numel() * src_keys[0].element_size()
    with _one_device(list(src_keys) + list(src_values) + list(dst_keys) + list(dst_values) +
                     [block_pairs, status], stream):
        rc = load().pkv_swap_blocks_layers(_ptr_array(src_keys), _ptr_array(src_values), _ptr_array(dst_keys),
                                           _ptr_array(dst_values), n, _ptr(block_pairs), block_pairs.shape[0],
                                           block_bytes, src_keys[0].shape[0], dst_keys[0].shape[0],
                                           _status_ptr(status), _stream(stream))
    _check(rc, "pkv_swap_blocks_layers")


def validate_block_pairs(pairs, num_blocks):
    """Host check of (src, dst) pairs for copy_blocks; True if valid."""
    a = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    return load().pkv_validate_block_pairs(a.ctypes.data_as(_i64p), a.shape[0], num_blocks) == PKV_OK


@_traced
def selftest_wait_timeout(status, limit_ns, stream=None):
    """pkv_selftest_wait_timeout: a bounded device wait that gives up and
    reports PKV_ERR_DEVICE_TIMEOUT in status (int32 CUDA tensor)."""
    if status is None:
        raise ValueError("status is required")
    with _one_device((status,), stream):
        rc = load().pkv_selftest_wait_timeout(_status_ptr(status), int(limit_ns), _stream(stream))
    _check(rc, "pkv_selftest_wait_timeout")


# ---------------------------------------------------------------------------
# host block manager

class BlockAllocator:
    """The C++ block manager (pkv_alloc_*).  Same method names as the rules
    describe: new_seq, append_token, append_tokens, append_batch, fork,
    release, export.  Not thread-safe (like the C object): one thread, or the
    caller's lock, per allocator."""

    def __init__(self, num_blocks, block_size, initial_free_order=None):
        lib = load()
        self._lib = lib
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        handle = ctypes.c_void_p()
        order = None
        if initial_free_order is not None:
            self._order = np.ascontiguousarray(np.asarray(initial_free_order, dtype=np.int32))
            if self._order.shape != (self.num_blocks,):
                raise ValueError("initial_free_order must hold num_blocks entries")
            order = self._order.ctypes.data_as(_i32p)
        _check(lib.pkv_alloc_create(self.num_blocks, self.block_size, order, ctypes.byref(handle)),
               "pkv_alloc_create")
        self._h = handle
        self._i = ctypes.c_int()

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_seq(self):
        _check(self._lib.pkv_seq_new(self._h, ctypes.byref(self._i)), "pkv_seq_new")
        return self._i.value

    def append_token(self, seq):
        """-> (slot, cow) with cow = (src, dst) or None."""
        slot = ctypes.c_int64()
        pair = (ctypes.c_int32 * 2)()
        _check(self._lib.pkv_append_token(self._h, seq, ctypes.byref(slot), pair), "pkv_append_token")
        return slot.value, ((pair[0], pair[1]) if pair[0] >= 0 else None)

    def append_tokens(self, seq, n):
        """-> (slots list, cows list); all or nothing."""
        slots = np.empty(max(n, 1), dtype=np.int64)
        pair = (ctypes.c_int32 * 2)()
        ncow = ctypes.c_int()
        _check(self._lib.pkv_append_tokens(self._h, seq, n, slots.ctypes.data_as(_i64p), pair,
                                           ctypes.byref(ncow)), "pkv_append_tokens")
        return slots[:n].tolist(), ([(pair[0], pair[1])] if ncow.value else [])

    def append_batch(self, seqs, slots_out=None, pairs_out=None):
        """One token for each distinct seq, in order.

        -> (slots int64 array [n], cow pairs int32 array [k][2]).  Optional
        preallocated outputs (e.g. pinned host tensors' numpy views) avoid
        allocation in a serving loop.
        """
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        n = s.shape[0]
        slots = slots_out if slots_out is not None else np.empty(max(n, 1), dtype=np.int64)
        pairs = pairs_out if pairs_out is not None else np.empty((max(n, 1), 2), dtype=np.int32)
        _out_array(slots, np.int64, n, "slots_out")
        _out_array(pairs, np.int32, 2 * n, "pairs_out")
        _check(self._lib.pkv_append_batch(self._h, s.ctypes.data, n, slots.ctypes.data, pairs.ctypes.data,
                                          ctypes.byref(self._i)), "pkv_append_batch")
        return slots[:n], pairs[:self._i.value]

    def fork(self, parent):
        _check(self._lib.pkv_fork(self._h, parent, ctypes.byref(self._i)), "pkv_fork")
        return self._i.value

    def release(self, seq):
        """-> number of blocks returned to the free list."""
        _check(self._lib.pkv_release(self._h, seq, ctypes.byref(self._i)), "pkv_release")
        return self._i.value

    def export(self, seqs, max_blocks_per_seq, tables_out=None, lens_out=None):
        """-> (tables int32 [n][MB] padded with -1, context_lens int32 [n])."""
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        n = s.shape[0]
        tables = tables_out if tables_out is not None else np.empty((n, max_blocks_per_seq), np.int32)
        lens = lens_out if lens_out is not None else np.empty(n, np.int32)
        _out_array(tables, np.int32, n * max_blocks_per_seq, "tables_out")
        _out_array(lens, np.int32, n, "lens_out")
        _check(self._lib.pkv_export_tables(self._h, s.ctypes.data, n, tables.ctypes.data, max_blocks_per_seq,
                                           lens.ctypes.data), "pkv_export_tables")
        return tables, lens

    def shared_prefix(self, seqs, out=None):
        """-> int32 [n]: entry i the leading blocks seqs[i] shares with
        seqs[i - 1] (0 for i = 0): the hint of paged_attention_decode_shared."""
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        n = s.shape[0]
        res = out if out is not None else np.empty(n, np.int32)
        _out_array(res, np.int32, n, "out")
        _check(self._lib.pkv_export_shared_prefix(self._h, s.ctypes.data, n, res.ctypes.data),
               "pkv_export_shared_prefix")
        return res

    def seq_len(self, seq):
        _check(self._lib.pkv_seq_length(self._h, seq, ctypes.byref(self._i)), "pkv_seq_length")
        return self._i.value

    def table(self, seq):
        _check(self._lib.pkv_seq_num_blocks(self._h, seq, ctypes.byref(self._i)), "pkv_seq_num_blocks")
        n = self._i.value
        out = np.empty(max(n, 1), np.int32)
        _check(self._lib.pkv_seq_table(self._h, seq, out.ctypes.data_as(_i32p), n, None), "pkv_seq_table")
        return out[:n].tolist()

    def refcount(self, block):
        _check(self._lib.pkv_block_refcount(self._h, block, ctypes.byref(self._i)), "pkv_block_refcount")
        return self._i.value

    def fill(self, block):
        _check(self._lib.pkv_block_fill(self._h, block, ctypes.byref(self._i)), "pkv_block_fill")
        return self._i.value

    def num_free(self):
        _check(self._lib.pkv_num_free(self._h, ctypes.byref(self._i)), "pkv_num_free")
        return self._i.value

    def free_list(self):
        out = np.empty(max(self.num_blocks, 1), np.int32)
        _check(self._lib.pkv_free_list(self._h, out.ctypes.data_as(_i32p), self.num_blocks,
                                       ctypes.byref(self._i)), "pkv_free_list")
        return out[:self._i.value].tolist()

    # -- checkpoint ------------------------------------------------------------
    def save(self):
        """The whole block-manager state as bytes (pkv_alloc_save)."""
        n = ctypes.c_size_t()
        _check(self._lib.pkv_alloc_save(self._h, None, 0, ctypes.byref(n)), "pkv_alloc_save")
        buf = ctypes.create_string_buffer(max(n.value, 1))
        _check(self._lib.pkv_alloc_save(self._h, buf, n.value, ctypes.byref(n)), "pkv_alloc_save")
        return buf.raw[:n.value]

    @classmethod
    def load(cls, blob):
        """A block manager restored from save()'s bytes (pkv_alloc_load);
        refuses (PkvError) any blob that is not a reachable state."""
        blob = bytes(blob)
        self = cls.__new__(cls)
        self._lib = _load_library()
        handle = ctypes.c_void_p()
        _check(self._lib.pkv_alloc_load(blob, len(blob), ctypes.byref(handle)), "pkv_alloc_load")
        self._h = handle
        self._i = ctypes.c_int()
        self.num_blocks, self.block_size, self.num_host_blocks = (
            int(v) for v in np.frombuffer(blob, dtype="<i4", count=3, offset=8))
        return self

    # -- swapping ------------------------------------------------------------
    def host_pool(self, num_host_blocks, host_free_order=None):
        """Give the manager a pool of host blocks for swapped-out sequences."""
        order = None
        if host_free_order is not None:
            self._host_order = np.ascontiguousarray(np.asarray(host_free_order, dtype=np.int32))
            if self._host_order.shape != (int(num_host_blocks),):
                raise ValueError("host_free_order must hold num_host_blocks entries")
            order = self._host_order.ctypes.data_as(_i32p)
        _check(self._lib.pkv_alloc_host_pool(self._h, int(num_host_blocks), order), "pkv_alloc_host_pool")
        self.num_host_blocks = int(num_host_blocks)

    def _move(self, fn, what, seqs):
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        cap = 0
        for q in s.tolist():
            _check(self._lib.pkv_seq_num_blocks(self._h, q, ctypes.byref(self._i)), "pkv_seq_num_blocks")
            cap += self._i.value
        pairs = np.empty((max(cap, 1), 2), dtype=np.int32)
        _check(fn(self._h, s.ctypes.data_as(_i32p), s.shape[0], pairs.ctypes.data_as(_i32p), cap,
                  ctypes.byref(self._i)), what)
        return pairs[:self._i.value]

    def swap_out(self, seqs):
        """-> int32 [k][2] (device block, host block) pairs to copy."""
        return self._move(self._lib.pkv_swap_out, "pkv_swap_out", seqs)

    def swap_in(self, seqs):
        """-> int32 [k][2] (host block, device block) pairs to copy."""
        return self._move(self._lib.pkv_swap_in, "pkv_swap_in", seqs)

    def is_swapped(self, seq):
        _check(self._lib.pkv_seq_swapped(self._h, seq, ctypes.byref(self._i)), "pkv_seq_swapped")
        return bool(self._i.value)

    def host_refcount(self, block):
        _check(self._lib.pkv_host_block_refcount(self._h, block, ctypes.byref(self._i)),
               "pkv_host_block_refcount")
        return self._i.value

    def host_fill(self, block):
        _check(self._lib.pkv_host_block_fill(self._h, block, ctypes.byref(self._i)), "pkv_host_block_fill")
        return self._i.value

    def num_free_host(self):
        _check(self._lib.pkv_num_free_host(self._h, ctypes.byref(self._i)), "pkv_num_free_host")
        return self._i.value

    def host_free_list(self):
        n = getattr(self, "num_host_blocks", 0)
        out = np.empty(max(n, 1), np.int32)
        _check(self._lib.pkv_host_free_list(self._h, out.ctypes.data_as(_i32p), n, ctypes.byref(self._i)),
               "pkv_host_free_list")
        return out[:self._i.value].tolist()
