"""The tensor-pipe rates the attention and matmul kernels are designed
around, measured on the GPU by tests/probes/tensor_pipe_probe.cu (cycles per
tcgen05.mma, M = 128 or 256, K = 16, bf16):

  * one CTA: N = 64 and N = 128 take about the same time per instruction,
    N = 256 about twice that -- so score products use N = 128 and the
    matmuls N = 256 (CTA pairs);
  * FFMA-heavy warps on the issuing thread's scheduler slow the MMA stream
    several-fold, the same work on the other schedulers does not, and packed
    f32x2 FMA chains slow it far less -- so the elementwise warps use f32x2.

The probe compiles with nvcc for sm_103a; run with -s to see the numbers.
"""
import json
import os
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def test_tensor_pipe_rates():
    src = os.path.join(HERE, "probes", "tensor_pipe_probe.cu")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "probe")
        subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", exe, src],
                       check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=120).stdout
    r = json.loads(out)
    print(json.dumps(r))
    assert r["wait_error"] == 0
    assert all(v > 0 for k, v in r.items() if k != "wait_error")
    # N = 64 costs about what N = 128 costs; N = 256 about twice
    assert r["cg1_ss_n64"] > 0.6 * r["cg1_ss_n128"]
    assert r["cg1_ss_n256"] > 1.5 * r["cg1_ss_n128"]
    # FFMA chains on the issuer's scheduler slow the stream; elsewhere not
    assert r["ts_n64_ffma_same_scheduler"] > 1.5 * r["ts_n64_ffma_other_schedulers"]
    assert r["ts_n64_f32x2_same_scheduler"] < r["ts_n64_ffma_same_scheduler"]
