"""The group-1 CUDA-core form of the decode kernel (an opt-in build,
PKV_DECODE_G1_CUDACORE=1) against the fp64 oracle.

The default build runs Q.K^T and P.V on the tensor cores at every group size;
the CUDA-core form is kept so that the two can be compared on the same ring,
schedule and merges.  This test builds it into a library of its own and runs
the checks in a child process that loads that library (PKV_LIBRARY), so the
rest of the suite keeps using the default build.
"""

import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(ROOT, "paged_kv_cache_152_gb300", "_build", "cudacore", "libpkv.so")


def _child_checks():
    """Run in the child: group-1 shapes and workloads, several grids."""
    import math
    import numpy as np
    import paged_kv_cache_152_gb300 as pkv
    import workloads as W
    from oracle import attention as OA
    from pkv_testlib import TOL, Case, max_abs_err
    from test_gpu_parity import _random_case, _run_gpu
    assert os.path.samefile(pkv.load()._name, LIB)
    for d in (64, 128):
        for bs in (8, 16, 32, 128):
            rng = np.random.default_rng(d + bs)
            lens = [1, bs - 1, bs, bs + 1, 3 * bs + 5, 70, 0, 2 * bs, 1000]
            q, kc, vc, tables, lens = _random_case(rng, len(lens), 4, 4, d, bs, lens)
            ref = OA.paged_decode_attention(q, kc, vc, tables, lens, 1.0 / math.sqrt(d))
            for num_ctas in (0, 1, 3, 37):
                out, st = _run_gpu(pkv, q, kc, vc, tables, lens, 1.0 / math.sqrt(d), num_ctas)
                assert st == 0 and np.isfinite(out).all(), (d, bs, num_ctas)
                err = float(np.max(np.abs(out - ref)))
                assert err <= TOL, (d, bs, num_ctas, err)
    for name, kw in (("7b", {}), ("prefix", {}), ("tiny", {}), ("chat", dict(num_main=6, num_transient=5))):
        case = Case(W.make(name, **kw))
        pkv.paged_attention_decode_append(case.out, case.t["query"], case.t["key"], case.t["value"],
                                          case.t["key_cache"], case.t["value_cache"], case.tables, case.lens,
                                          case.wl.scale, status=case.status)
        torch.cuda.synchronize()
        assert int(case.status.item()) == 0
        case.oracle_write_new_tokens()
        err = max_abs_err(case.out, case.oracle_decode())
        assert err <= TOL, (name, err)
    # the mapped serving step (inputs read from host memory) in this build
    from test_gpu_mapped_inputs import _step_pair
    direct, mapped, plan_d, plan_h, host, dev, host_out = _step_pair(pkv, W.make("7b", num_seqs=9), True, False)
    plan_d.launch()
    plan_h.step_mapped(dev, host)
    torch.cuda.synchronize()
    assert int(direct.status.item()) == 0 and int(mapped.status.item()) == 0
    assert torch.equal(host_out.view(torch.int16), direct.out.cpu().view(torch.int16))
    plan_d.close()
    plan_h.close()
    print("cudacore ok")


def test_cudacore_form_matches_oracle():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    sys.path.insert(0, ROOT)
    from paged_kv_cache_152_gb300 import build
    build.build(defines=["PKV_DECODE_G1_CUDACORE=1"], lib_path=LIB)
    env = dict(os.environ, PKV_LIBRARY=LIB, PYTHONPATH=os.pathsep.join([ROOT, HERE]))
    r = subprocess.run([sys.executable, "-c", "import test_gpu_cudacore as t; t._child_checks()"],
                       cwd=HERE, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "cudacore ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
