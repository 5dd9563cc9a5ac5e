"""Host-side checks of the native library (no GPU needed).

* libpkv.so builds, loads and exports every function include/pkv.h declares;
* the decode kernel's work split (pkv_schedule.h) passes its exhaustive CPU
  check;
* host argument validation rejects bad calls before any launch;
* the block manager survives a sanitized fuzz (tests/cpp/test_alloc_fuzz.cpp);
* the header is plain C99 and usable from C (tests/c/test_header_c99.c).
"""

import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_152_gb300 import build
    build.build()
    import paged_kv_cache_152_gb300 as pkv
    return pkv.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 25
    for name in names:
        assert hasattr(lib, name), name
    import paged_kv_cache_152_gb300 as pkv
    assert sorted(pkv.SIGNATURES) == names


def test_exported_symbols_via_nm(lib):
    from paged_kv_cache_152_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pkv_[a-z0-9_]+)", out))
    assert set(declared_functions()) <= exported


def test_library_version_and_status_strings(lib):
    import paged_kv_cache_152_gb300 as pkv
    assert lib.pkv_version() >= 100
    assert pkv.status_string(pkv.PKV_ERR_OUT_OF_BLOCKS) == "PKV_ERR_OUT_OF_BLOCKS"
    assert pkv.status_string(99) == "PKV_UNKNOWN_STATUS"


def test_schedule_exhaustive(tmp_path):
    exe = tmp_path / "test_schedule"
    subprocess.run(["g++", "-O2", "-std=c++17", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "paged_kv_cache_152_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "cpp", "test_schedule.cpp"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "schedule ok" in r.stdout


def test_alloc_fuzz_sanitized(tmp_path):
    """Random block-manager calls through the C ABI under ASan/UBSan:
    conservation, reference counts, table lengths, and failed calls leave the
    state untouched."""
    exe = tmp_path / "test_alloc_fuzz"
    subprocess.run(["g++", "-O1", "-g", "-std=c++17", "-Wall", "-Werror",
                    "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
                    "-fno-omit-frame-pointer", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "cpp", "test_alloc_fuzz.cpp"),
                    os.path.join(ROOT, "paged_kv_cache_152_gb300", "csrc", "pkv_alloc.cpp"),
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "alloc fuzz ok" in r.stdout


def test_header_is_c99_and_usable_from_c(lib, tmp_path):
    """pkv.h compiles as pedantic C99 and a C program drives the block manager
    (and its checkpoint) through libpkv.so."""
    from paged_kv_cache_152_gb300 import LIB_PATH
    libdir = os.path.dirname(LIB_PATH)
    exe = tmp_path / "test_header_c99"
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "test_header_c99.c"),
                    "-L", libdir, "-lpkv", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c99 header ok" in r.stdout


@pytest.fixture
def no_gpu():
    """Host-validation tests pass fake device pointers that must be rejected
    before any launch; never run them where a launch could reach a GPU."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake-pointer host checks run on GPU-less hosts only")


def test_decode_rejects_bad_arguments_on_host(lib, no_gpu):
    import ctypes
    vp = ctypes.c_void_p(256)    # never dereferenced: validation fails first
    call = lambda **kw: lib.pkv_paged_attention_decode(  # noqa: E731
        kw.get("out", vp), vp, vp, vp, vp, kw.get("mb", 4), vp, kw.get("n", 2), kw.get("h", 8),
        kw.get("hkv", 8), kw.get("d", 64), kw.get("bs", 16), kw.get("nb", 10),
        ctypes.c_float(kw.get("scale", 0.125)), 0, kw.get("ws", vp), 1 << 20, None, None)
    import paged_kv_cache_152_gb300 as pkv
    assert call(n=0) == pkv.PKV_OK                       # empty batch: nothing to do
    assert call(out=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(ws=None) == pkv.PKV_ERR_INVALID_ARG
    assert call(h=6, hkv=4) == pkv.PKV_ERR_INVALID_ARG   # heads not a multiple of KV heads
    assert call(scale=-1.0) == pkv.PKV_ERR_INVALID_ARG
    assert call(n=5000) == pkv.PKV_ERR_INVALID_ARG
    assert call(d=96) == pkv.PKV_ERR_UNSUPPORTED
    assert call(bs=24) == pkv.PKV_ERR_UNSUPPORTED
    assert call(h=48, hkv=3) == pkv.PKV_ERR_UNSUPPORTED  # group 16
    assert call(out=ctypes.c_void_p(258)) == pkv.PKV_ERR_INVALID_ARG  # misaligned
    # cache rows (blocks x KV heads x block size) must stay below 2^31
    assert call(nb=(1 << 31) // (8 * 16)) == pkv.PKV_ERR_INVALID_ARG
    assert call(mb=(1 << 26) + 1) == pkv.PKV_ERR_INVALID_ARG    # 2^30 tokens per table row


def test_cache_ops_reject_bad_arguments_on_host(lib, no_gpu):
    import ctypes
    import paged_kv_cache_152_gb300 as pkv
    vp = ctypes.c_void_p(256)
    assert lib.pkv_reshape_and_cache(vp, vp, vp, vp, vp, 0, 8, 64, 16, 4, None, None) == pkv.PKV_OK
    assert lib.pkv_reshape_and_cache(vp, vp, vp, vp, vp, 3, 8, 60, 16, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_reshape_and_cache(None, vp, vp, vp, vp, 3, 8, 64, 16, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy_blocks(vp, vp, vp, 0, 4096, 4, None, None) == pkv.PKV_OK
    assert lib.pkv_copy_blocks(vp, vp, vp, 2, 4001, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_selftest_wait_timeout(None, 10**6, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_selftest_wait_timeout(vp, 10, None) == pkv.PKV_ERR_INVALID_ARG


def test_validate_block_pairs(lib):
    import paged_kv_cache_152_gb300 as pkv
    assert pkv.validate_block_pairs([(1, 2), (3, 4)], 8)
    assert pkv.validate_block_pairs([], 8)
    assert not pkv.validate_block_pairs([(1, 2), (3, 2)], 8)   # same destination twice
    assert not pkv.validate_block_pairs([(1, 2), (2, 4)], 8)   # destination is also a source
    assert not pkv.validate_block_pairs([(1, 8)], 8)           # outside the pool
    assert not pkv.validate_block_pairs([(-1, 3)], 8)


def test_multi_layer_ops_reject_bad_arguments_on_host(lib, no_gpu):
    import ctypes
    import paged_kv_cache_152_gb300 as pkv
    vp = ctypes.c_void_p(256)
    good = (ctypes.c_void_p * 2)(256, 512)
    bad = (ctypes.c_void_p * 2)(256, None)
    odd = (ctypes.c_void_p * 2)(256, 520)
    f = lib.pkv_reshape_and_cache_layers
    assert f(good, good, good, good, 2, vp, 0, 8, 64, 16, 4, None, None) == pkv.PKV_OK   # no tokens
    assert f(good, good, good, good, 0, vp, 3, 8, 64, 16, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(good, good, good, good, 129, vp, 3, 8, 64, 16, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(good, bad, good, good, 2, vp, 3, 8, 64, 16, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(good, good, odd, good, 2, vp, 3, 8, 64, 16, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    g = lib.pkv_copy_blocks_layers
    assert g(good, good, 2, vp, 0, 4096, 4, None, None) == pkv.PKV_OK
    assert g(good, bad, 2, vp, 1, 4096, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert g(good, good, 2, vp, 1, 4001, 4, None, None) == pkv.PKV_ERR_INVALID_ARG


def test_swap_blocks_reject_bad_arguments_on_host(lib, no_gpu):
    import ctypes
    import paged_kv_cache_152_gb300 as pkv
    vp = ctypes.c_void_p(256)
    f = lib.pkv_swap_blocks
    assert f(vp, vp, vp, vp, vp, 0, 4096, 4, 4, None, None) == pkv.PKV_OK           # nothing to move
    assert f(vp, vp, vp, vp, vp, -1, 4096, 4, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(vp, vp, vp, vp, vp, 2, 4001, 4, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(vp, vp, vp, vp, vp, 2, 4096, 0, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(vp, vp, None, vp, vp, 2, 4096, 4, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(vp, vp, vp, ctypes.c_void_p(264), vp, 2, 4096, 4, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(vp, vp, vp, vp, None, 2, 4096, 4, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    # well-formed arguments reach the pointer-attribute query, which has no
    # device to ask here: an error status, never a launch
    assert f(vp, vp, vp, vp, vp, 2, 4096, 4, 4, None, None) == pkv.PKV_ERR_CUDA
    good = (ctypes.c_void_p * 2)(256, 512)
    bad = (ctypes.c_void_p * 2)(256, None)
    g = lib.pkv_swap_blocks_layers
    assert g(good, good, good, good, 2, vp, 0, 4096, 4, 4, None, None) == pkv.PKV_OK
    assert g(good, good, good, good, 0, vp, 1, 4096, 4, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert g(good, good, good, good, 129, vp, 1, 4096, 4, 4, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert g(good, good, bad, good, 2, vp, 1, 4096, 4, 4, None, None) == pkv.PKV_ERR_INVALID_ARG


def test_decode_plan_rejects_bad_arguments_on_host(lib, no_gpu):
    import ctypes
    import paged_kv_cache_152_gb300 as pkv
    vp = ctypes.c_void_p(256)
    h = ctypes.c_void_p(1)

    def create(**kw):
        return lib.pkv_decode_plan_create(
            vp, vp, kw.get("k", None), kw.get("v", None), vp, vp, vp, 4, vp, kw.get("n", 2), 8, 8, 64, 16, 10,
            ctypes.c_float(0.125), 0, kw.get("ws", vp), 1 << 20, None, kw.get("out", ctypes.byref(h)))
    assert create(out=None) == pkv.PKV_ERR_INVALID_ARG
    assert create(k=vp) == pkv.PKV_ERR_INVALID_ARG and h.value is None    # key without value
    assert create(ws=None) == pkv.PKV_ERR_INVALID_ARG and h.value is None
    assert create(n=0) == pkv.PKV_OK and h.value is not None               # empty: launches nothing
    assert lib.pkv_decode_plan_launch(h, None) == pkv.PKV_OK
    # a step of the empty plan without copies enqueues nothing; missing pointers are refused
    assert lib.pkv_decode_plan_step(h, None, None, 0, None, None) == pkv.PKV_OK
    assert lib.pkv_decode_plan_step(h, None, vp, 64, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_plan_step(h, vp, None, 64, None, None) == pkv.PKV_ERR_INVALID_ARG
    lib.pkv_decode_plan_destroy(h)
    assert lib.pkv_decode_plan_launch(None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_plan_step(None, None, None, 0, None, None) == pkv.PKV_ERR_INVALID_ARG
