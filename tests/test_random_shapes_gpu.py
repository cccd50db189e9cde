"""Seeded random shapes against the float64 oracle: every entry point on
problem sizes, head counts, context lengths and masks drawn at random (a
fixed generator, so the cases are the same on every run), each compared in
full.  The fixed-shape tests pin the edges one at a time; these mix them.

Tolerances are those of the dedicated tests: bf16 O 2e-2 / LSE 1e-2, fp16
5e-3 / 2e-3, fp32 1e-5, the decode 2e-2, the backward R14's, FP8 R20's.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs
from test_backward_gpu import _compare
from test_fp8_gpu import _check_forward

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = {torch.bfloat16: (2e-2, 1e-2), torch.float16: (5e-3, 2e-3), torch.float32: (1e-5, 1e-5)}
_rng = np.random.default_rng(20261202)


def _forward_cases(n):
    out = []
    for _ in range(n):
        dtype = [torch.bfloat16, torch.float16, torch.float32][_rng.integers(3)]
        d = int(_rng.choice([64, 128] if dtype == torch.float32 else [64, 128, 256]))
        N = int(_rng.integers(1, 700 if d < 256 else 400))
        out.append((int(_rng.integers(1, 3)), int(_rng.integers(1, 5)), N, d,
                    bool(_rng.random() < 0.5), dtype))
    return out


FWD = _forward_cases(24)


@pytest.mark.parametrize("B,H,N,d,causal,dtype", FWD,
                         ids=[f"{c[5]}-{c[0]}x{c[1]}x{c[2]}x{c[3]}-{'c' if c[4] else 'nc'}"
                              for c in FWD])
def test_random_forward(B, H, N, d, causal, dtype):
    q, k, v = inputs.forward_inputs(B, H, N, d, dtype, seed=N * 7 + d + H)
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ro, rl = oracle.attention_forward(q, k, v, d ** -0.5, causal)
    tol_o, tol_l = TOL[dtype]
    assert np.abs(o.float().cpu().numpy() - ro).max() <= tol_o
    assert np.abs(lse.cpu().numpy() - rl).max() <= tol_l


BWD = [(int(_rng.integers(1, 3)), int(_rng.integers(1, 4)), int(_rng.integers(1, 500)),
        int(_rng.choice([64, 128])), bool(_rng.random() < 0.5)) for _ in range(10)]


@pytest.mark.parametrize("B,H,N,d,causal", BWD,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{'c' if c[4] else 'nc'}" for c in BWD])
def test_random_backward(B, H, N, d, causal):
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=N + d)
    do = inputs.grad_output(B, H, N, d, torch.bfloat16, seed=N + d)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal)
    grads = fa.backward(qd, kd, vd, o, lse, dod, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ref = oracle.attention_backward(q, k, v, do, d ** -0.5, causal)
    for name, got, want in zip(("dQ", "dK", "dV"), grads, ref):
        _compare(got.float().cpu().numpy(), want, name)


def _decode_cases(n):
    out = []
    for _ in range(n):
        H = int(_rng.choice([4, 8, 12, 16, 32]))
        Hk = int(_rng.choice([h for h in (1, 2, 4, H) if H % h == 0]))
        S = int(_rng.integers(1, 11))
        max_ctx = int(_rng.integers(16, 3000))
        ctx = [0 if _rng.random() < 0.1 else int(_rng.integers(1, max_ctx + 1)) for _ in range(S)]
        out.append((S, H, Hk, max_ctx, ctx))
    return out


DEC = _decode_cases(12)


@pytest.mark.parametrize("S,H,Hk,max_ctx,ctx", DEC,
                         ids=[f"{c[0]}seq-{c[1]}h-{c[2]}kv-{c[3]}" for c in DEC])
def test_random_decode(S, H, Hk, max_ctx, ctx):
    di = inputs.decode_inputs(S, H, 128, 16, max_ctx, seed=S * 31 + H + max_ctx, device=DEV,
                              num_kv_heads=Hk)
    di.context_lens.copy_(torch.tensor(ctx, dtype=torch.int32, device=DEV))
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                          di.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ref, _ = oracle.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables,
                                 di.context_lens, di.scale)
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 2e-2
    for s, c in enumerate(ctx):
        if c == 0:
            assert (got[s] == 0).all()


MSK = [(int(_rng.integers(1, 3)), int(_rng.integers(1, 4)), 16 * int(_rng.integers(1, 33)),
        int(_rng.choice([64, 128])), density, bool(_rng.random() < 0.5))
       for density in (0.05, 0.5, 0.95, 0.05, 0.5, 0.95)]


@pytest.mark.parametrize("B,H,N,d,density,per_head", MSK,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}x{c[3]}-{c[4]}-{'ph' if c[5] else 'sh'}"
                              for c in MSK])
def test_random_mask(B, H, N, d, density, per_head):
    g = np.random.default_rng(N * 13 + d)
    shape = (B, H, N, N) if per_head else (N, N)
    mask = (g.random(shape) < density).astype(np.uint8)
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=N + 3 * d)
    o, lse = fa.forward_masked(q.to(DEV), k.to(DEV), v.to(DEV), torch.as_tensor(mask).to(DEV))
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ro, rl = oracle.attention_forward_masked(q, k, v, mask, d ** -0.5)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.abs(o - ro).max() <= 2e-2
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl))
    assert np.abs(lse[fin] - rl[fin]).max() <= 1e-2


FP8 = [(int(_rng.integers(1, 3)), int(_rng.integers(1, 4)), int(_rng.integers(1, 600)),
        bool(_rng.random() < 0.5), bool(_rng.random() < 0.5)) for _ in range(4)]


@pytest.mark.parametrize("B,H,N,causal,rot", FP8,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}-{'c' if c[3] else 'nc'}-{'rot' if c[4] else 'plain'}"
                              for c in FP8])
def test_random_fp8(B, H, N, causal, rot):
    q, k, v = inputs.forward_inputs(B, H, N, 128, torch.bfloat16, seed=N + 5)
    signs = inputs.rotation_signs(128, seed=N) if rot else None
    _check_forward(q, k, v, causal, signs)
