"""Paged decode with grouped key/value heads against the float64 oracle.

Query head h reads key/value head h // (H // Hk) ("PagedAttention",
data-sketchers.com, section "Inputs": the caches' num_kv_heads axis).  The
tolerance is the decode's: max |out - ref| <= 2e-2 (bf16 output rounding of
values of size <= ~4, plus bf16 rounding of P-weighted sums in fp32).
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = 2e-2


def _check(di, ctx=None):
    if ctx is not None:
        di.context_lens.copy_(torch.tensor(ctx, dtype=torch.int32, device=DEV))
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                          di.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ref, _ = oracle.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables,
                                 di.context_lens, di.scale)
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= TOL
    return got


@pytest.mark.parametrize("S,H,Hk,max_ctx", [
    (4, 8, 2, 700),      # group 4, two partitions at most
    (5, 8, 4, 1100),     # group 2
    (3, 8, 1, 1000),     # group 8 = two sub-groups of 4, one key/value head
    (2, 64, 1, 600),     # multi-query, 16 sub-groups
    (3, 8, 8, 500),      # group 1: the one-head kernel
    (6, 16, 4, 17),      # two-block contexts
])
def test_gqa_decode_matches_oracle(S, H, Hk, max_ctx):
    di = inputs.decode_inputs(S, H, 128, 16, max_ctx, seed=S * 100 + H + Hk, device=DEV,
                              num_kv_heads=Hk)
    _check(di)


def test_gqa_decode_ragged_and_empty_contexts():
    di = inputs.decode_inputs(5, 16, 128, 16, 2000, seed=7, device=DEV, num_kv_heads=4)
    got = _check(di, ctx=[2000, 0, 1, 513, 1999])
    assert (got[1] == 0).all()       # context 0: zero output rows


def test_gqa_decode_benchmark_workload():
    """64 sequences x 32 query heads x 8 key/value heads, contexts U[1, 4096]:
    the shape the benchmark times; 8 sequences are checked against the oracle."""
    di = inputs.decode_inputs(64, 32, 128, 16, 4096, seed=5, device=DEV, num_kv_heads=8)
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                          di.scale)
    torch.cuda.synchronize()
    rows = [0, 7, 19, 31, 40, 52, 60, 63]
    sel = torch.tensor(rows, device=DEV)
    ref, _ = oracle.paged_decode(di.q[sel], di.k_cache, di.v_cache, di.block_tables[sel],
                                 di.context_lens[sel], di.scale)
    assert np.abs(out[sel].float().cpu().numpy() - ref).max() <= TOL


def test_gqa_decode_equals_replicated_one_head_decode():
    """The grouped kernel and the one-head kernel on caches whose key/value heads
    are repeated for their query heads give the same outputs up to the order of
    their fp32 sums (the grouped kernel adds even and odd terms in separate
    packed lanes): at most one bf16 step apart, and mostly bit-equal."""
    S, H, Hk = 4, 8, 2
    di = inputs.decode_inputs(S, H, 128, 16, 900, seed=11, device=DEV, num_kv_heads=Hk)
    g = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens, di.scale)
    kc = di.k_cache.repeat_interleave(H // Hk, dim=1).contiguous()
    vc = di.v_cache.repeat_interleave(H // Hk, dim=1).contiguous()
    m = fa.paged_decode(di.q, kc, vc, di.block_tables, di.context_lens, di.scale)
    torch.cuda.synchronize()
    gf, mf = g.float(), m.float()
    assert ((gf - mf).abs() <= mf.abs() * 2.0 ** -7 + 1e-6).all()
    assert (gf == mf).float().mean().item() > 0.8
