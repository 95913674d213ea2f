"""GPU parity of the FP8 (E4M3) entry points against the oracle, through the
C ABI: quantisation codes and scales bit for bit (both sides form x * s in
fp32 and round it to the nearest code, ties to even), and the scaled
matmul element by element within fp32 accumulation rounding."""
import numpy as np
import pytest
import torch

import oracle
from transformer_lm_step_gpt_b300 import GPT2Error, fp8_check, fp8_matmul, fp8_quantize
from parity_util import rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("n", [1, 7, 8, 1000, 4099, 1 << 20])
def test_quantize_bit_exact(n, bf16):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * rng.choice([1e-3, 1.0, 50.0], n)).astype(np.float32)
    if n > 10:
        x[5] = np.nan      # left out of the maximum, coded as NaN
        x[6] = 0.0
    xt = torch.from_numpy(x).cuda()
    if bf16:
        xt = xt.to(torch.bfloat16)
        x = xt.float().cpu().numpy()   # the values the kernel sees
    q, s = fp8_quantize(xt)
    fp8_check()
    q_ref, s_ref = oracle.fp8_quantize(x)
    assert s.cpu().numpy()[0] == np.float32(s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quantize_all_zero_and_extremes():
    x = np.zeros(64, np.float32)
    q, s = fp8_quantize(torch.from_numpy(x).cuda())
    assert s.cpu().numpy()[0] == 1.0 and not q.cpu().numpy().any()
    x[3], x[9] = -7.0, 7.0   # two maxima of opposite sign
    q, s = fp8_quantize(torch.from_numpy(x).cuda())
    qn = q.cpu().numpy()
    assert qn[3] == 0xFE and qn[9] == 0x7E


def quantized(shape, seed, scale):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    q, s = fp8_quantize(torch.from_numpy(x).cuda())
    return x, q, s


@pytest.mark.parametrize("out_bf16", [False, True])
@pytest.mark.parametrize("M,N,K", [(300, 200, 208), (1, 256, 128), (257, 520, 96), (128, 1000, 768)])
def test_matmul_matches_oracle(M, N, K, out_bf16):
    _, qa, sa = quantized((M, K), 1, 2.0)
    _, qb, sb = quantized((N, K), 2, 0.05)
    bias = torch.from_numpy(np.random.default_rng(3).normal(0, 1, N).astype(np.float32)).cuda()
    out = fp8_matmul(qa, sa, qb, sb, bias=bias, out_dtype=torch.bfloat16 if out_bf16 else torch.float32)
    fp8_check()
    ref = oracle.fp8_matmul(qa.cpu().numpy(), float(sa[0]), qb.cpu().numpy(), float(sb[0]),
                            bias=bias.cpu().numpy().astype(np.float64))
    got = out.float().cpu().numpy()
    assert rel_l2(got, ref) <= (4e-3 if out_bf16 else 1e-5)
    if not out_bf16:
        assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()


def test_matmul_strided_operands():
    # row strides larger than K (a padded buffer), K not a multiple of 128
    M, N, K, ld = 130, 300, 200, 256
    _, qa_full, sa = quantized((M, ld), 4, 1.0)
    _, qb_full, sb = quantized((N, ld), 5, 1.0)
    qa, qb = qa_full[:, :K], qb_full[:, :K]
    out = fp8_matmul(qa, sa, qb, sb)
    fp8_check()
    ref = oracle.fp8_matmul(np.ascontiguousarray(qa.cpu().numpy()), float(sa[0]),
                            np.ascontiguousarray(qb.cpu().numpy()), float(sb[0]))
    assert rel_l2(out.cpu().numpy(), ref) <= 1e-5


def test_matmul_gpt2_fc_shape_sampled_rows():
    # the fc forward of GPT-2 124M at B=16, T=1024: rows sampled for the oracle
    M, N, K = 16384, 3072, 768
    _, qa, sa = quantized((M, K), 6, 1.0)
    _, qb, sb = quantized((N, K), 7, 0.02)
    out = fp8_matmul(qa, sa, qb, sb, out_dtype=torch.bfloat16)
    fp8_check()
    rows = np.random.default_rng(8).choice(M, 24, replace=False)
    ref = oracle.fp8_matmul(qa[rows].cpu().numpy(), float(sa[0]), qb.cpu().numpy(), float(sb[0]))
    assert rel_l2(out[rows].float().cpu().numpy(), ref) <= 4e-3


def test_matmul_argument_errors():
    q = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    s = torch.ones(2, dtype=torch.float32, device="cuda")
    with pytest.raises(GPT2Error) as e:   # ldb = 40 bytes: not a multiple of 16
        fp8_matmul(q[:, :40], s, torch.zeros((64, 40), dtype=torch.uint8, device="cuda"), s)
    assert e.value.code == -1
    with pytest.raises(GPT2Error) as e:   # a NULL scale
        from transformer_lm_step_gpt_b300 import load_library
        lib = load_library()
        rc = lib.gpt2_fp8_matmul(q.data_ptr(), 64, None, q.data_ptr(), 64, s.data_ptr(), 64, 64, 64, None,
                                 s.data_ptr(), 64, 0, None)
        from transformer_lm_step_gpt_b300 import _check_global
        _check_global(rc)
    assert e.value.code == -1
