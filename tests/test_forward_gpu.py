"""Parity of fa_forward / fa_forward_fp32 (CUDA) with the float64 oracle.

Tolerances: max |O - O_ref| <= 2e-2 and max |LSE - LSE_ref| <= 1e-2 for bf16
inputs (fp32 accumulation, bf16 output), and <= 1e-5 for both in fp32.
Inputs come from exact_attention_11_gb300.inputs; the oracle sees the same
bf16/fp32 values widened to float64.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu

BF16_TOL_O, BF16_TOL_LSE = 2e-2, 1e-2
F32_TOL = 1e-5


def gpu_forward(q, k, v, causal, scale=None):
    dev = torch.device("cuda:0")
    o, lse = fa.forward(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(o, lse, ro, rl, tol_o, tol_l, what):
    eo = float(np.abs(o - ro).max()) if o.size else 0.0
    el = float(np.abs(lse - rl).max()) if lse.size else 0.0
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    assert eo <= tol_o, f"{what}: max|dO| = {eo:.3e} > {tol_o}"
    assert el <= tol_l, f"{what}: max|dLSE| = {el:.3e} > {tol_l}"
    return eo, el


FP32_CASES = [  # (B, H, N, d, causal)
    (1, 1, 64, 64, False),    # the fp32 reference workload: 1 x 1 x 64 x 64
    (1, 1, 64, 64, True),
    (2, 3, 100, 128, True),
    (1, 2, 65, 64, False),
    (1, 1, 1, 128, False),
    (1, 1, 1000, 64, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", FP32_CASES)
def test_fp32_forward_matches_oracle(B, H, N, d, causal):
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.float32, seed=N + d)
    o, lse = gpu_forward(q, k, v, causal)
    ro, rl = oracle.attention_forward(q, k, v, d ** -0.5, causal)
    check(o, lse, ro, rl, F32_TOL, F32_TOL, f"fp32 {B}x{H}x{N}x{d} causal={causal}")


BF16_CASES = [  # (B, H, N, d, causal): tails, single tiles, several tiles
    (1, 1, 128, 128, False),
    (1, 1, 128, 64, True),
    (1, 2, 200, 128, True),
    (2, 2, 1000, 64, False),
    (1, 1, 1, 128, False),
    (1, 1, 1, 64, True),
    (1, 1, 63, 64, True),
    (1, 1, 129, 128, True),
    (1, 3, 257, 64, True),
    (1, 2, 384, 128, False),
    (2, 1, 700, 128, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", BF16_CASES)
def test_bf16_forward_matches_oracle(B, H, N, d, causal):
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=3 * N + d)
    o, lse = gpu_forward(q, k, v, causal)
    ro, rl = oracle.attention_forward(q, k, v, d ** -0.5, causal)
    check(o, lse, ro, rl, BF16_TOL_O, BF16_TOL_LSE, f"bf16 {B}x{H}x{N}x{d} causal={causal}")


def test_bf16_workload_b4_h16_n1024_d64_full():
    """Every output of the 4 x 16 x 1024 x 64 non-causal workload."""
    q, k, v = inputs.forward_inputs(4, 16, 1024, 64, torch.bfloat16, seed=2)
    o, lse = gpu_forward(q, k, v, False)
    ro, rl = oracle.attention_forward(q, k, v, 1 / 8, False)
    check(o, lse, ro, rl, BF16_TOL_O, BF16_TOL_LSE, "4x16x1024x64")


def test_bf16_workload_b2_h16_n4096_d128_causal_full():
    """Every output (all 4096 rows of all 32 heads, O and LSE) of the
    2 x 16 x 4096 x 128 causal workload, in the launch the benchmark times."""
    q, k, v = inputs.forward_inputs(2, 16, 4096, 128, torch.bfloat16, seed=3)
    o, lse = gpu_forward(q, k, v, True)
    ro, rl = oracle.attention_forward(q, k, v, 128 ** -0.5, True)
    check(o, lse, ro, rl, BF16_TOL_O, BF16_TOL_LSE, "2x16x4096x128 causal")


def test_bf16_workload_b1_h8_n16384_d128_causal_full():
    """Every output (all 16384 rows of all 8 heads, O and LSE) of the
    1 x 8 x 16384 x 128 causal workload with inputs N(0,1) * 0.5 (the oracle
    takes some seconds on the host cores)."""
    q, k, v = inputs.forward_inputs(1, 8, 16384, 128, torch.bfloat16, seed=4, amp=0.5)
    o, lse = gpu_forward(q, k, v, True)
    ro, rl = oracle.attention_forward(q, k, v, 128 ** -0.5, True)
    check(o, lse, ro, rl, BF16_TOL_O, BF16_TOL_LSE, "1x8x16384x128 causal")


@pytest.mark.parametrize("B,H,N,d,amp,nrows,seed", [
    (1, 8, 16384, 128, 0.5, 256, 4),    # 1 x 8 x 16384 x 128 causal, inputs * 0.5
])
def test_bf16_large_causal_sampled_rows(B, H, N, d, amp, nrows, seed):
    """The 16K causal workload on the seeded sample of 256 query rows per head
    (plus the first, second and last rows) that the workload's parity
    statement names; the full comparison is the test above."""
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=seed, amp=amp)
    o, lse = gpu_forward(q, k, v, True)
    rows = sorted(set(inputs.sample_rows(N, nrows, seed=seed + 100).tolist()) | {0, 1, N - 1})
    ro, rl = oracle.attention_forward_rows(q, k, v, rows, d ** -0.5, True)
    check(o[:, :, rows], lse[:, :, rows], ro, rl, BF16_TOL_O, BF16_TOL_LSE,
          f"{B}x{H}x{N}x{d} causal sampled")


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_special_cases(d):
    """Cases fixed by the definition: causal row 0 is exactly V[0]; Q = 0
    gives the mean of the visible V rows and LSE = ln(count)."""
    N = 300
    q, k, v = inputs.forward_inputs(1, 2, N, d, torch.bfloat16, seed=9)
    o, lse = gpu_forward(q, k, v, True)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0].float().numpy())
    z = torch.zeros_like(q)
    o, lse = gpu_forward(z, k, v, True)
    vv = v.double().numpy()
    prefix = np.cumsum(vv, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    assert np.abs(o - prefix).max() <= BF16_TOL_O
    assert np.abs(lse - np.log(np.arange(1, N + 1))).max() <= 1e-4
    o, lse = gpu_forward(z, k, v, False)
    assert np.abs(o - vv.mean(axis=2, keepdims=True)).max() <= BF16_TOL_O
    assert np.abs(lse - np.log(N)).max() <= 1e-4


def test_bf16_large_logits_stay_finite():
    """Scores of magnitude ~100s need the running max (safe softmax).  Q and K
    are multiplied by 4 (exact in bf16); V keeps unit scale."""
    q, k, v = inputs.forward_inputs(1, 2, 260, 128, torch.bfloat16, seed=12)
    q, k = q * 4, k * 4
    o, lse = gpu_forward(q, k, v, True, scale=1.0)
    ro, rl = oracle.attention_forward(q, k, v, 1.0, True)
    assert np.isfinite(o).all()
    # LSE is ~hundreds here: allow the fp32 relative error of the scores.
    check(o, lse, ro, rl, BF16_TOL_O, 1e-2 * max(1.0, float(np.abs(rl).max()) / 100),
          "large logits")


def test_bf16_repeat_is_bitwise_deterministic():
    q, k, v = inputs.forward_inputs(2, 4, 777, 128, torch.bfloat16, seed=5)
    a = gpu_forward(q, k, v, True)
    b = gpu_forward(q, k, v, True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_lse_may_be_null():
    q, k, v = inputs.forward_inputs(1, 1, 130, 64, torch.bfloat16, seed=6)
    dev = torch.device("cuda:0")
    o, lse = fa.forward(q.to(dev), k.to(dev), v.to(dev), causal=True, want_lse=False)
    torch.cuda.synchronize()
    assert lse is None
    ro, _ = oracle.attention_forward(q, k, v, 64 ** -0.5, True)
    assert np.abs(o.float().cpu().numpy() - ro).max() <= BF16_TOL_O


def test_device_status_clean_after_forward():
    assert fa.fa_device_status() == 0
