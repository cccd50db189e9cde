"""fp16 forward (fa_forward_f16) against the float64 oracle.

Inputs are N(0,1) draws rounded to fp16; the oracle widens the same fp16 values
exactly.  The kernel rounds the softmax weights to fp16 before PV and the output
to fp16, each a relative error of at most 2^-11; with |v| below ~5 for these
draws the output error stays under 2^-11 * (sum_j p_j |v_j| + |o|) < 5e-3.  The
LSE comes from fp32 sums of unrounded weights: 2e-3 is ample.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL_O, TOL_LSE = 5e-3, 2e-3


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 128, 64, False),
    (2, 3, 333, 128, True),      # ragged tail, several heads
    (1, 2, 1000, 128, False),
    (1, 4, 256, 64, True),
    (1, 1, 1, 128, True),        # a single row
])
def test_f16_forward_matches_oracle(B, H, N, d, causal):
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.float16, seed=N + d)
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    assert o.dtype == torch.float16
    ro, rl = oracle.attention_forward(q, k, v, d ** -0.5, causal)
    assert np.abs(o.float().cpu().numpy() - ro).max() <= TOL_O
    assert np.abs(lse.cpu().numpy() - rl).max() <= TOL_LSE


def test_f16_forward_benchmark_shape_sampled_rows():
    """2 x 16 x 4096 x 128 causal, the benchmark's forward shape, in fp16;
    64 sampled rows per head plus the first and last are checked."""
    B, H, N, d = 2, 16, 4096, 128
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.float16, seed=3)
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    rows = sorted(set(inputs.sample_rows(N, 64, seed=N).tolist()) | {0, N - 1})
    ro, rl = oracle.attention_forward_rows(q, k, v, rows, d ** -0.5, True)
    assert np.abs(o[:, :, rows].float().cpu().numpy() - ro).max() <= TOL_O
    assert np.abs(lse[:, :, rows].cpu().numpy() - rl).max() <= TOL_LSE
    assert fa.fa_device_status() == 0


def test_f16_more_precise_than_bf16():
    """The same real-valued inputs through both 16-bit paths: fp16 keeps three
    more mantissa bits, so its error against the oracle is smaller."""
    B, H, N, d = 1, 2, 512, 128
    q32, k32, v32 = inputs.forward_inputs(B, H, N, d, torch.float32, seed=21)
    errs = {}
    for dt in (torch.float16, torch.bfloat16):
        q, k, v = (t.to(dt) for t in (q32, k32, v32))
        o, _ = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
        torch.cuda.synchronize()
        ro, _ = oracle.attention_forward(q, k, v, d ** -0.5, True)
        errs[dt] = np.abs(o.float().cpu().numpy() - ro).max()
    assert errs[torch.float16] < errs[torch.bfloat16]
