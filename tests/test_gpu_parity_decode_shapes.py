"""GPU parity of generation with the key/value cache on shapes beyond
test_gpu_decode.py's, against the oracle's incremental forward, through the
C ABI.

- Head sizes 32 and 128 run the generic decode attention (the TMA-staged
  one serves bf16 at head size 64 only) with the keys split over a cluster:
  T = 130 gives a cluster of 3 CTAs, T = 70 one of 2, so the ranks' (max,
  sum, output) combine is exercised outside head size 64.
- 20 sequences in bf16: more rows than the few-row matmul takes (16), so
  the step runs without its CUDA graph, with the host's position, through
  the tiled matmuls writing the new cache row at a row stride of T rows.
The checks are those of test_gpu_decode.py: every step's scores within the
training tolerances and each drawn token valid against the oracle's CDF
(equal to the oracle's wherever the draw is unique)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, cuda_ids, rel_l2
from test_gpu_decode import CDF_TOL, check_draw, setup

pytestmark = pytest.mark.gpu

#        L  C    NH  V    Vp   maxT B  T
HS32 = (1, 64, 2, 97, 104, 130, 2, 130)    # head size 32, keys over 3 CTAs
HS128 = (1, 128, 1, 120, 128, 70, 2, 70)   # head size 128, one head, keys over 2 CTAs
B20 = (1, 128, 2, 97, 104, 100, 20, 100)   # 20 sequences, head size 64, keys over 2 CTAs


@pytest.mark.parametrize("shape,prec", [(HS32, "fp32"), (HS32, "bf16"), (HS128, "fp32"), (HS128, "bf16"),
                                        (B20, "bf16")])
def test_teacher_forced_decode(shape, prec):
    L, C, NH, V, Vp, maxT, B, T = shape
    m, p = setup(shape, prec, seed=17)
    cfg = oracle.cfg8(*shape)
    rng = np.random.default_rng(23)
    T0, temp = 5, 0.8
    n_new = T - T0 + 1                      # up to the last cache row, T - 1
    prompt = rng.integers(0, V, (B, T0)).astype(np.int32)
    u = rng.random((n_new, B))
    toks_ref, lg_ref = oracle.generate(cfg, p.astype(np.float64), prompt, n_new, temp, u)
    padded = np.zeros((B, T), np.int32)
    padded[:, :T0] = prompt
    m.forward(cuda_ids(padded), None)
    u_d = torch.from_numpy(u.astype(np.float32)).cuda()
    tol = TOL[prec]["rel"]
    for i in range(n_new):
        pos = T0 - 1 + i
        nxt = m.decode_step(cuda_ids(toks_ref[:, pos]), pos, temp, u_d[i])
        lg = m.decode_logits()
        assert np.all(lg[:, V:] == 0)
        assert rel_l2(lg[:, :V], lg_ref[i]) <= tol, (i, rel_l2(lg[:, :V], lg_ref[i]))
        g = nxt.cpu().numpy()
        for b in range(B):
            check_draw(int(g[b]), lg_ref[i, b], temp, float(np.float32(u[i, b])), CDF_TOL[prec])
