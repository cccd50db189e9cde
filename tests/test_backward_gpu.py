"""Backward pass (dQ, dK, dV) of the bf16 CUDA path against the float64 oracle.

The kernel rebuilds P from Q, K and the forward's LSE, rounds P and dS to bf16
before they multiply dO, Q and K, and rounds dQ, dK, dV to bf16 at the end
(recomputation scheme of section 7 of "FlashAttention: GPU 메모리 계층을 활용한
어텐션 최적화 분석", youngju.dev).  Each of those roundings has relative error
at most 2^-9, so the error of a gradient is a small multiple of 2^-9 times the
size of the terms it sums.  The test bounds, per gradient tensor G:
    max |G - G_ref| <= 1e-2 * max |G_ref|   and
    rms (G - G_ref) <= 5e-3 * rms (G_ref),
about 5x and 2.5x the errors three bf16 roundings give; a dropped term, a
missing scale or a wrong index is off by far more.  Both bounds also allow an
absolute 1e-5: dS = P (dP - D) cancels exactly when one key is visible (then
O = V and dP = D), and fp32 sums of terms of size |dO| |V| ~ 10 leave about
2^-24 * 10 * sqrt(d) there.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL_MAX, TOL_RMS, ATOL = 1e-2, 5e-3, 1e-5


def _run(B, H, N, d, causal, seed):
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=seed)
    do = inputs.grad_output(B, H, N, d, torch.bfloat16, seed=seed)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return (q, k, v, do), (dq.float().cpu().numpy(), dk.float().cpu().numpy(),
                           dv.float().cpu().numpy())


def _compare(got, ref, name):
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    scale_max = np.abs(ref).max()
    rms_ref = np.sqrt(np.mean(ref ** 2))
    assert err.max() <= TOL_MAX * scale_max + ATOL, \
        f"{name}: max err {err.max():.3e} vs max|ref| {scale_max:.3e}"
    assert np.sqrt(np.mean(err ** 2)) <= TOL_RMS * rms_ref + ATOL, \
        f"{name}: rms err {np.sqrt(np.mean(err ** 2)):.3e} vs rms ref {rms_ref:.3e}"


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 128, 64, False),     # one tile
    (1, 2, 256, 128, True),     # two tiles, diagonal blocks
    (2, 3, 333, 128, True),     # ragged tail, several heads
    (1, 2, 200, 64, True),      # ragged, d = 64
    (1, 1, 130, 64, False),     # two-row tail past one tile
    (1, 2, 1000, 128, False),   # eight key blocks, non-causal
    (1, 1, 1, 128, True),       # a single row
    (2, 3, 333, 64, True),      # d = 64: ragged tail, several heads
    (1, 2, 1000, 64, False),    # d = 64: eight key blocks, non-causal
    (1, 1, 1, 64, True),        # d = 64: a single row
    (1, 1, 65, 64, True),       # d = 64: one key block, second sub-tile empty
])
def test_backward_matches_oracle(B, H, N, d, causal):
    (q, k, v, do), (dq, dk, dv) = _run(B, H, N, d, causal, seed=N + d)
    rq, rk, rv = oracle.attention_backward(q, k, v, do, d ** -0.5, causal)
    _compare(dq, rq, "dQ")
    _compare(dk, rk, "dK")
    _compare(dv, rv, "dV")


def _check_heads(q, k, v, do, grads, heads, d, causal):
    """Oracle gradients of the listed (b, h) heads (each head's gradients
    depend only on that head's inputs), computed in one oracle call."""
    H = q.shape[1]
    flat = [b * H + h for b, h in heads]
    sel = [t.reshape(-1, *t.shape[2:])[flat].unsqueeze(0) for t in (q, k, v, do)]
    ref = oracle.attention_backward(*sel, d ** -0.5, causal)
    for name, got, want in zip(("dQ", "dK", "dV"), grads, ref):
        g = got.reshape(-1, *got.shape[2:])[flat][None]
        _compare(g, want, f"{name} of heads {heads}")


@pytest.mark.parametrize("d", [128, 64])
def test_backward_full_size_all_heads(d):
    """The benchmark's backward workloads, 2 x 16 x 4096 x d causal, in the
    launch the benchmark times; every one of the 32 heads is checked against
    the oracle (eight heads per oracle call)."""
    B, H, N = 2, 16, 4096
    (q, k, v, do), grads = _run(B, H, N, d, True, seed=3)
    every = [(b, h) for b in range(B) for h in range(H)]
    for i in range(0, len(every), 8):
        _check_heads(q, k, v, do, grads, every[i:i + 8], d, True)


@pytest.mark.parametrize("d,causal", [(128, False), (64, False), (128, True), (64, True)])
def test_backward_several_items_per_cta(d, causal):
    """4 x 16 x 1024: 512 (key block, head) items on at most one CTA per SM, so
    each persistent CTA takes several in turn (items of different heads and
    lengths back to back); 12 heads, from both ends of the item order, are
    checked against the oracle."""
    B, H, N = 4, 16, 1024
    (q, k, v, do), grads = _run(B, H, N, d, causal, seed=11 + d)
    heads = [(0, 0), (0, 1), (0, 15), (1, 3), (1, 8), (2, 0), (2, 9), (2, 14), (3, 2), (3, 7),
             (3, 14), (3, 15)]
    _check_heads(q, k, v, do, grads, heads, d, causal)


def test_backward_two_streams_at_once():
    """Two backward calls in flight at once on two streams (separate work
    counters and workspaces), with no wait between the launches; both match
    the oracle."""
    cases = [(1, 3, 700, 128, True, 21), (2, 2, 900, 64, False, 22)]
    prepared = []
    for B, H, N, d, causal, seed in cases:
        q, k, v = (t.to(DEV) for t in inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=seed))
        do = inputs.grad_output(B, H, N, d, torch.bfloat16, seed=seed).to(DEV)
        o, lse = fa.forward(q, k, v, causal=causal)
        prepared.append((q, k, v, do, o, lse, d, causal))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for (q, k, v, do, o, lse, d, causal), st in zip(prepared, streams):
        with torch.cuda.stream(st):
            outs.append(fa.backward(q, k, v, o, lse, do, causal=causal))
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for (q, k, v, do, o, lse, d, causal), grads in zip(prepared, outs):
        ref = oracle.attention_backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), d ** -0.5, causal)
        for name, got, want in zip(("dQ", "dK", "dV"), grads, ref):
            _compare(got.float().cpu().numpy(), want, name)


def test_backward_writes_stay_inside_outputs():
    B, H, N, d = 1, 3, 333, 128
    q, k, v = (t.to(DEV) for t in inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=9))
    do = inputs.grad_output(B, H, N, d, torch.bfloat16, seed=9).to(DEV)
    o, lse = fa.forward(q, k, v, causal=True)
    n = B * H * N * d
    guard = 4096
    bufs = [torch.full((n + guard,), 7.0, dtype=torch.bfloat16, device=DEV) for _ in range(3)]
    dq, dk, dv = (b[:n].view(B, H, N, d) for b in bufs)
    ws = torch.empty((fa.fa_backward_workspace_bytes(B, H, N, d),), dtype=torch.uint8,
                     device=DEV)
    fa.fa_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                   lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                   d ** -0.5, True, ws.data_ptr(), ws.numel(),
                   torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    for b in bufs:
        assert (b[n:] == 7.0).all()
    ref = fa.backward(q, k, v, o, lse, do, causal=True)
    for got, want in zip((dk, dv), ref[1:]):
        assert torch.equal(got, want)   # no atomics in dK, dV: bit-identical


def test_backward_repeatable_and_workspace_reuse():
    """dK and dV are bit-identical across calls; dQ (fp32 atomic sums) agrees
    to bf16 rounding; a reused, dirty workspace gives the same answers."""
    B, H, N, d = 1, 4, 777, 64
    q, k, v = (t.to(DEV) for t in inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=5))
    do = inputs.grad_output(B, H, N, d, torch.bfloat16, seed=5).to(DEV)
    o, lse = fa.forward(q, k, v, causal=False)
    ws = torch.full((fa.fa_backward_workspace_bytes(B, H, N, d) + 64,), 0xAB, dtype=torch.uint8,
                    device=DEV)
    a = fa.backward(q, k, v, o, lse, do, causal=False, workspace=ws)
    b = fa.backward(q, k, v, o, lse, do, causal=False, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    diff = (a[0].float() - b[0].float()).abs().max().item()
    assert diff <= 2 ** -7 * a[0].float().abs().max().item()


def test_backward_rejects_small_workspace():
    q, k, v = (t.to(DEV) for t in inputs.forward_inputs(1, 1, 64, 64, torch.bfloat16, seed=1))
    o, lse = fa.forward(q, k, v)
    small = torch.empty((16,), dtype=torch.uint8, device=DEV)
    with pytest.raises(fa.FattnError):
        fa.backward(q, k, v, o, lse, q, workspace=small)
