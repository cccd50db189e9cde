"""Forward with a boolean attention mask (fa_forward_masked) against the
float64 oracle ("FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화 분석",
youngju.dev, section 11.3).  Tolerances are the bf16 forward's: 2e-2 on O,
1e-2 on LSE; rows with no visible key must give exactly O = 0, LSE = -inf.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL_O, TOL_LSE = 2e-2, 1e-2


def _run(B, H, N, d, mask, seed, rows=None):
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=seed)
    o, lse = fa.forward_masked(q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(mask).to(DEV))
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ro, rl = oracle.attention_forward_masked(q, k, v, mask, d ** -0.5, rows)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    if rows is not None:
        o, lse = o[:, :, rows], lse[:, :, rows]
    return o, lse, ro, rl


def _close(o, lse, ro, rl):
    fin = np.isfinite(rl)
    assert np.abs(o - ro).max() <= TOL_O
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl))
    assert np.abs(lse[fin] - rl[fin]).max() <= TOL_LSE


@pytest.mark.parametrize("N,d", [(256, 128), (336, 64)])
def test_tril_mask_equals_causal(N, d):
    mask = np.tril(np.ones((N, N), dtype=np.uint8))
    o, lse, ro, rl = _run(1, 2, N, d, mask, seed=N)
    _close(o, lse, ro, rl)
    q, k, v = inputs.forward_inputs(1, 2, N, d, torch.bfloat16, seed=N)
    oc, lc = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    assert np.abs(o - oc.float().cpu().numpy()).max() <= TOL_O


@pytest.mark.parametrize("N,d,density", [(256, 128, 0.5), (512, 64, 0.1), (160, 128, 0.9)])
def test_random_shared_mask(N, d, density):
    r = np.random.default_rng(N)
    mask = (r.random((N, N)) < density).astype(np.uint8)
    o, lse, ro, rl = _run(2, 2, N, d, mask, seed=N + 1)
    _close(o, lse, ro, rl)


def test_per_head_masks_and_empty_rows():
    B, H, N, d = 2, 3, 192, 128
    r = np.random.default_rng(5)
    mask = (r.random((B, H, N, N)) < 0.3).astype(np.uint8)
    mask[0, 1, 17] = 0                 # a row that sees nothing
    mask[1, 2, :40] = 0                # forty of them
    o, lse, ro, rl = _run(B, H, N, d, mask, seed=9)
    _close(o, lse, ro, rl)
    assert np.all(o[0, 1, 17] == 0) and np.isneginf(lse[0, 1, 17])
    assert np.all(o[1, 2, :40] == 0) and np.all(np.isneginf(lse[1, 2, :40]))


def test_sliding_window_mask_sampled_rows():
    """A banded mask (each query sees the 300 keys up to itself) at N = 2048:
    many key tiles fully masked, others partly."""
    B, H, N, d = 1, 4, 2048, 128
    i = np.arange(N)
    mask = ((i[None, :] <= i[:, None]) & (i[None, :] > i[:, None] - 300)).astype(np.uint8)
    rows = sorted(set(inputs.sample_rows(N, 48, seed=2).tolist()) | {0, 299, 300, N - 1})
    o, lse, ro, rl = _run(B, H, N, d, mask, seed=2, rows=rows)
    _close(o, lse, ro, rl)
