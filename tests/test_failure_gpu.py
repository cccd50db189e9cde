"""Device-side failure detection without a GPU fault.

fa_debug_inject_fault(1) makes one CTA of the next forward (bf16, fp16,
masked or E4M3) lose its key-tile copies (its producer stops after the query
tiles); mode 2 does the same to
the next backward (its K and V copies).  The MMA warp's bounded
wait for them runs out after about 2 s, the CTA unwinds, and the host reads
FA_ERR_TIMEOUT from fa_device_status().  Nothing traps, faults or hangs: the
context stays usable and the next forward is correct.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_lost_copy_times_out_and_context_survives():
    dev = torch.device("cuda:0")
    q, k, v = inputs.forward_inputs(1, 4, 640, 128, torch.bfloat16, seed=31)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    assert fa.fa_device_status() == 0
    fa.fa_debug_inject_fault(1)
    t0 = time.perf_counter()
    fa.forward(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert fa.fa_device_status() == -5          # FA_ERR_TIMEOUT, reported once
    assert fa.fa_device_status() == 0
    assert 1.0 < waited < 30.0                  # the 2 s limit ran out, nothing hung
    # The armed fault was consumed: the next call is clean and correct.
    o, lse = fa.forward(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ro, rl = oracle.attention_forward(q, k, v, 128 ** -0.5, True)
    assert np.abs(o.float().cpu().numpy() - ro).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-2


def test_fp8_forward_lost_copy_times_out_and_context_survives():
    """The same failure path in the E4M3 forward, which keeps P in shared
    memory with its own MMA issue order and barriers: mode 1 arms it too;
    the wait runs out, every role unwinds, and the next call gives the same
    bits as a clean call before the fault."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in inputs.forward_inputs(1, 4, 640, 128, torch.bfloat16, seed=33))
    x = fa.quantize_fp8(q, k, v)
    clean, clean_lse = fa.forward_fp8(x, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    fa.fa_debug_inject_fault(1)
    t0 = time.perf_counter()
    fa.forward_fp8(x, causal=True)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert fa.fa_device_status() == -5          # FA_ERR_TIMEOUT, reported once
    assert fa.fa_device_status() == 0
    assert 1.0 < waited < 30.0
    o, lse = fa.forward_fp8(x, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.equal(o, clean) and torch.equal(lse, clean_lse)


@pytest.mark.parametrize("d", [128, 64])
def test_backward_lost_copy_times_out_and_context_survives(d):
    """The same on the persistent backward: one CTA loses the K and V copies
    of its first item, its MMA warp's wait runs out, it unwinds while the
    other CTAs finish their items, and the next backward is correct."""
    dev = torch.device("cuda:0")
    B, H, N = 1, 2, 640
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=33)
    do = inputs.grad_output(B, H, N, d, torch.bfloat16, seed=33)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = fa.forward(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    fa.fa_debug_inject_fault(2)
    t0 = time.perf_counter()
    fa.backward(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert fa.fa_device_status() == -5          # FA_ERR_TIMEOUT, reported once
    assert fa.fa_device_status() == 0
    assert 1.0 < waited < 30.0
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ref = oracle.attention_backward(q, k, v, do, d ** -0.5, True)
    for got, want in zip((dq, dk, dv), ref):
        g = got.float().cpu().numpy()
        assert np.abs(g - want).max() <= 1e-2 * np.abs(want).max() + 1e-5


def test_inject_rejects_unknown_mode():
    with pytest.raises(fa.FattnError):
        fa.fa_debug_inject_fault(7)
    with pytest.raises(fa.FattnError):
        fa.fa_debug_inject_fault(3)
    fa.fa_debug_inject_fault(0)
