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
from test_decode_gpu import poisoned_caches

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = 2e-2
TC_ONLY = (3, 5, 6, 7, 16, 32)      # group sizes only the tensor-core kernel takes


@pytest.fixture(params=[2, 1], ids=["tensor_cores", "cuda_cores"])
def impl(request):
    """Runs a test once per grouped-decode kernel (fa_decode_gqa_select)."""
    fa.fa_decode_gqa_select(request.param)
    yield request.param
    fa.fa_decode_gqa_select(0)


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
    (3, 8, 1, 1000),     # group 8, one key/value head
    (2, 64, 1, 600),     # multi-query: 4 slices of 16 / 16 sub-groups of 4
    (3, 8, 8, 500),      # group 1: the one-head kernel
    (6, 16, 4, 17),      # two-block contexts
    (3, 12, 4, 900),     # group 3
    (2, 24, 4, 1300),    # group 6
    (3, 7, 1, 700),      # group 7
    (2, 32, 2, 1500),    # group 16: every MMA column
    (2, 64, 2, 800),     # group 32: two slices of 16
    (2, 96, 2, 700),     # group 48: three slices of 16 / twelve sub-groups of 4
])
def test_gqa_decode_matches_oracle(impl, S, H, Hk, max_ctx):
    if impl == 1 and H // Hk in TC_ONLY:
        pytest.skip("group size served by the tensor-core kernel only")
    di = inputs.decode_inputs(S, H, 128, 16, max_ctx, seed=S * 100 + H + Hk, device=DEV,
                              num_kv_heads=Hk)
    _check(di)


def test_gqa_decode_ragged_and_empty_contexts(impl):
    di = inputs.decode_inputs(5, 16, 128, 16, 2000, seed=7, device=DEV, num_kv_heads=4)
    got = _check(di, ctx=[2000, 0, 1, 513, 1999])
    assert (got[1] == 0).all()       # context 0: zero output rows


def test_gqa_decode_tile_boundaries(impl):
    """Contexts at and next to the block (16), step (128) and partition (512)
    boundaries."""
    ctx = [1, 15, 16, 17, 127, 128, 129, 511, 512, 513, 1024, 1025]
    di = inputs.decode_inputs(len(ctx), 16, 128, 16, 1100, seed=23, device=DEV, num_kv_heads=2)
    _check(di, ctx=ctx)


def test_gqa_decode_many_partitions(impl):
    """Contexts of up to four 1024-token partitions of the tensor-core kernel
    (merged from registers loaded in one round trip) and of five to nine
    (merged by the general loop), at and next to the four-partition edge."""
    ctx = [3072, 4095, 4096, 4097, 5121, 9000]
    di = inputs.decode_inputs(len(ctx), 8, 128, 16, 9000, seed=31, device=DEV, num_kv_heads=2)
    _check(di, ctx=ctx)


def test_gqa_decode_tails_of_every_length(impl):
    """Contexts whose last 1024-token partition holds each of 1 .. 8 steps of
    128 tokens, or none (whole partitions only), and empty ones, in an order
    not sorted by length: the tensor-core kernel hands out the whole
    partitions first and then these ragged tails, longest first."""
    ctx = []
    for full in range(3):
        for steps in (8, 1, 5, 3, 7, 2, 6, 4):
            ctx.append(1024 * full + 128 * (steps - 1) + 1 + (37 * steps + 11 * full) % 127)
    ctx += [1024, 0, 2048, 3072, 0]
    di = inputs.decode_inputs(len(ctx), 32, 128, 16, 3100, seed=47, device=DEV, num_kv_heads=8)
    got = _check(di, ctx=ctx)
    assert (got[[25, 28]] == 0).all()


def test_gqa_decode_dense_numbering_limit(impl):
    """1024 sequences, the most the tensor-core kernel numbers from its
    shared-memory prefix sums (one ragged tail each, of every length), some
    empty: 16 sampled sequences against the oracle, all against the other
    kernel."""
    S = 1024
    di = inputs.decode_inputs(S, 8, 128, 16, 1000, seed=53, device=DEV, num_kv_heads=2)
    di.context_lens[::89] = 0
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                          di.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert (out[::89] == 0).all()
    sel = torch.tensor(list(range(3, S, 67)), device=DEV)
    ref, _ = oracle.paged_decode(di.q[sel], di.k_cache, di.v_cache, di.block_tables[sel],
                                 di.context_lens[sel], di.scale)
    assert np.abs(out[sel].float().cpu().numpy() - ref).max() <= TOL
    fa.fa_decode_gqa_select(3 - impl)
    other = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                            di.scale)
    fa.fa_decode_gqa_select(impl)
    torch.cuda.synchronize()
    assert (out.float() - other.float()).abs().max().item() <= TOL


def test_gqa_decode_ignores_cache_slots_past_the_context(impl):
    """Slots past a sequence's context (the tail of its last block, and blocks
    it does not use) may hold anything: NaN there changes no output bit."""
    di = inputs.decode_inputs(6, 32, 128, 16, 1000, seed=31, device=DEV, num_kv_heads=4)
    ctx = [1000, 3, 130, 515, 17, 999]
    clean = _check(di, ctx=ctx)
    kc, vc = poisoned_caches(di)
    out = fa.paged_decode(di.q, kc, vc, di.block_tables, di.context_lens, di.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.equal(out.float().cpu(), torch.from_numpy(clean))


def test_gqa_decode_many_sequences(impl):
    """More sequences than the tensor-core kernel numbers densely (1024): its
    (partition, sequence) numbering with empty units.  16 sampled sequences
    against the oracle, and every output against the other kernel."""
    S = 1100
    di = inputs.decode_inputs(S, 8, 128, 16, 700, seed=43, device=DEV, num_kv_heads=2)
    di.context_lens[::97] = 0                      # a few sequences with no context
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                          di.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert (out[::97] == 0).all()
    rows = list(range(0, S, 71))
    sel = torch.tensor(rows, device=DEV)
    ref, _ = oracle.paged_decode(di.q[sel], di.k_cache, di.v_cache, di.block_tables[sel],
                                 di.context_lens[sel], di.scale)
    assert np.abs(out[sel].float().cpu().numpy() - ref).max() <= TOL
    fa.fa_decode_gqa_select(3 - impl)
    other = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                            di.scale)
    fa.fa_decode_gqa_select(impl)
    torch.cuda.synchronize()
    assert (out.float() - other.float()).abs().max().item() <= TOL


def test_gqa_decode_shared_prefix_blocks(impl):
    """Sequences whose block tables share physical blocks (a cached common
    prefix) each read them as their own."""
    di = inputs.decode_inputs(4, 16, 128, 16, 900, seed=51, device=DEV, num_kv_heads=4)
    bt = di.block_tables.clone()
    bt[1:, :5] = bt[0, :5]
    di.block_tables.copy_(bt)
    _check(di, ctx=[900, 700, 333, 81])


def test_gqa_decode_repeat_calls_are_identical(impl):
    """The split-K counters are left at zero: a second call gives the same bits."""
    di = inputs.decode_inputs(8, 32, 128, 16, 3000, seed=41, device=DEV, num_kv_heads=8)
    a = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens, di.scale)
    b = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens, di.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_gqa_decode_benchmark_workload(impl):
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
    """The CUDA-core grouped kernel and the one-head kernel on caches whose
    key/value heads are repeated for their query heads give the same outputs up
    to the order of their fp32 sums (the grouped kernel adds even and odd terms
    in separate packed lanes): at most one bf16 step apart, and mostly
    bit-equal."""
    S, H, Hk = 4, 8, 2
    di = inputs.decode_inputs(S, H, 128, 16, 900, seed=11, device=DEV, num_kv_heads=Hk)
    fa.fa_decode_gqa_select(1)
    try:
        g = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                            di.scale)
    finally:
        fa.fa_decode_gqa_select(0)
    kc = di.k_cache.repeat_interleave(H // Hk, dim=1).contiguous()
    vc = di.v_cache.repeat_interleave(H // Hk, dim=1).contiguous()
    m = fa.paged_decode(di.q, kc, vc, di.block_tables, di.context_lens, di.scale)
    torch.cuda.synchronize()
    gf, mf = g.float(), m.float()
    assert ((gf - mf).abs() <= mf.abs() * 2.0 ** -7 + 1e-6).all()
    assert (gf == mf).float().mean().item() > 0.8


def test_gqa_decode_in_cuda_graph():
    """The tensor-core decode (its dependent launches included) captured in a
    CUDA graph replays to the eager result, bit for bit."""
    di = inputs.decode_inputs(8, 32, 128, 16, 2000, seed=61, device=DEV, num_kv_heads=8)
    fa.fa_decode_gqa_select(2)
    try:
        out = torch.empty_like(di.q)
        fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                        di.scale, out=out)          # workspace and cache views set up
        torch.cuda.synchronize()
        eager = out.clone()
        graph = torch.cuda.CUDAGraph()
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables,
                                di.context_lens, di.scale, out=out)
        torch.cuda.synchronize()
        for _ in range(3):
            out.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, eager)
        assert fa.fa_device_status() == 0
    finally:
        fa.fa_decode_gqa_select(0)
