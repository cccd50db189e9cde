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


def test_block_sparse_mask_skips_tiles():
    """A mask made of whole 128 x 128 blocks (on or off, per head) plus a
    ragged N: key tiles that no row of an item sees are skipped, fully visible
    tiles read no mask bytes, partial ones (the ragged edge) are masked."""
    B, H, N, d = 1, 3, 720, 128
    r = np.random.default_rng(11)
    nt = (N + 127) // 128
    blocks = r.random((B, H, nt, nt)) < 0.4
    mask = np.repeat(np.repeat(blocks, 128, axis=2), 128, axis=3)[:, :, :N, :N].astype(np.uint8)
    mask[0, 2, 300:310] = 0                     # a few rows with nothing visible
    o, lse, ro, rl = _run(B, H, N, d, mask, seed=12)
    _close(o, lse, ro, rl)


def test_mask_hiding_whole_items():
    """Rows 0-511 see no key at all (two whole work items of 256 rows): they
    must still be written as O = 0, LSE = -inf; the other rows see a band."""
    N, d = 1024, 64
    i = np.arange(N)
    mask = ((i[None, :] <= i[:, None]) & (i[None, :] > i[:, None] - 200)).astype(np.uint8)
    mask[:512] = 0
    o, lse, ro, rl = _run(2, 2, N, d, mask, seed=13)
    _close(o, lse, ro, rl)
    assert np.all(o[:, :, :512] == 0) and np.all(np.isneginf(lse[:, :, :512]))


def test_dense_mask_equals_unmasked_forward():
    """An all-ones mask (every tile fully visible: no mask bytes are read) gives
    the unmasked non-causal forward."""
    B, H, N, d = 1, 2, 384, 128
    mask = np.ones((N, N), dtype=np.uint8)
    o, lse, ro, rl = _run(B, H, N, d, mask, seed=14)
    _close(o, lse, ro, rl)
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=14)
    ou, lu = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=False)
    torch.cuda.synchronize()
    assert np.array_equal(o, ou.float().cpu().numpy())
