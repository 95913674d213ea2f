"""The bf16 matmul on the fifteen products of one GPT-2 124M step (B=16,
T=1024), each with the epilogue it has in the step, timed alone by
tests/probes/gemm_shapes_probe.cu (which compiles the library's matmul
source with nvcc for sm_103a), next to torch.matmul (cuBLAS) on the same
shapes and layouts.  Run with -s to see the numbers; the assertions only
check that every launch ran clean and that no shape fell off a cliff.
"""
import json
import os
import subprocess
import tempfile
import time

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
CSRC = os.path.join(ROOT, "transformer_lm_step_gpt_b300", "csrc")


def _cublas(shapes):
    import torch
    out = {}
    for name, (m, n, k) in shapes.items():
        if "wgrad" in name:      # out[m, n] = A^T B, both stored [k][.]
            a = torch.randn(k, m, device="cuda", dtype=torch.bfloat16)
            b = torch.randn(k, n, device="cuda", dtype=torch.bfloat16)
            f = lambda: a.t() @ b
        elif "dgrad" in name:    # out = A B, B stored [k][n]
            a = torch.randn(m, k, device="cuda", dtype=torch.bfloat16)
            b = torch.randn(k, n, device="cuda", dtype=torch.bfloat16)
            f = lambda: a @ b
        else:                    # out = A B^T, B stored [n][k]
            a = torch.randn(m, k, device="cuda", dtype=torch.bfloat16)
            b = torch.randn(n, k, device="cuda", dtype=torch.bfloat16)
            f = lambda: a @ b.t()
        for _ in range(5):
            f()
        torch.cuda.synchronize()
        time.sleep(0.5)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(20):
            f()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 20
        out[name] = dict(us=round(ms * 1e3, 1), tflops=round(2.0 * m * n * k / ms / 1e9))
        del a, b
    return out


def test_step_matmul_shapes():
    src = os.path.join(HERE, "probes", "gemm_shapes_probe.cu")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "probe")
        subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "--expt-relaxed-constexpr", "-I" + CSRC, "-I" + os.path.join(ROOT, "include"), "-o", exe,
                        src, os.path.join(CSRC, "k_gemm_tc.cu"), "-lcuda"], check=True, capture_output=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=300).stdout
    r = json.loads(out)
    assert r["err"] == 0 and r["host_fail"] == 0 and r["cuda"] == "no error", r
    shapes = {k: (v["M"], v["N"], v["K"]) for k, v in r.items() if isinstance(v, dict)}
    assert len(shapes) == 15
    ref = _cublas(shapes)
    print(json.dumps({"library": r, "cublas": ref}))
    for k, v in r.items():
        if isinstance(v, dict):
            assert v["tflops"] > 200, (k, v)
