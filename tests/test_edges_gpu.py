"""Edge cases of the CUDA path against the float64 oracle: writes stay inside
the outputs, concurrent calls on two streams, many small work items, long
non-causal rows, and decode shapes with ragged block tables."""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL_O, TOL_L = 2e-2, 1e-2


def _ref(q, k, v, causal, rows=None):
    d = q.shape[-1]
    if rows is None:
        return oracle.attention_forward(q, k, v, d ** -0.5, causal)
    return oracle.attention_forward_rows(q, k, v, rows, d ** -0.5, causal)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("N,d,causal", [(333, 128, True), (97, 64, False), (1, 128, True)])
def test_outputs_do_not_spill_past_their_end(dtype, N, d, causal):
    B, H = 1, 3
    q, k, v = inputs.forward_inputs(B, H, N, d, dtype, seed=N)
    guard = 4096
    o_buf = torch.full((B * H * N * d + guard,), 7.0, dtype=dtype, device=DEV)
    l_buf = torch.full((B * H * N + guard,), 7.0, dtype=torch.float32, device=DEV)
    o = o_buf[:B * H * N * d].view(B, H, N, d)
    lse = l_buf[:B * H * N].view(B, H, N)
    fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, out=o, lse=lse)
    torch.cuda.synchronize()
    assert (o_buf[B * H * N * d:] == 7.0).all()
    assert (l_buf[B * H * N:] == 7.0).all()
    ro, rl = _ref(q, k, v, causal)
    tol = (TOL_O, TOL_L) if dtype == torch.bfloat16 else (1e-5, 1e-5)
    assert np.abs(o.float().cpu().numpy() - ro).max() <= tol[0]
    assert np.abs(lse.cpu().numpy() - rl).max() <= tol[1]


def test_two_streams_at_once():
    """Two forwards in flight together on different streams (separate work
    counters) both match the oracle."""
    qa, ka, va = (t.to(DEV) for t in inputs.forward_inputs(2, 8, 1536, 128, torch.bfloat16, seed=41))
    qb, kb, vb = (t.to(DEV) for t in inputs.forward_inputs(1, 16, 1024, 64, torch.bfloat16, seed=42))
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(sa):
            oa, la = fa.forward(qa, ka, va, causal=True)
        with torch.cuda.stream(sb):
            ob, lb = fa.forward(qb, kb, vb, causal=False)
    torch.cuda.synchronize()
    rows = [0, 511, 1024, 1535]
    ro, rl = _ref(qa.cpu(), ka.cpu(), va.cpu(), True, rows)
    assert np.abs(oa[:, :, rows].float().cpu().numpy() - ro).max() <= TOL_O
    assert np.abs(la[:, :, rows].cpu().numpy() - rl).max() <= TOL_L
    ro, rl = _ref(qb.cpu(), kb.cpu(), vb.cpu(), False)
    assert np.abs(ob.float().cpu().numpy() - ro).max() <= TOL_O
    assert np.abs(lb.cpu().numpy() - rl).max() <= TOL_L
    assert fa.fa_device_status() == 0


@pytest.mark.parametrize("B,H,N,d,causal", [
    (8, 64, 256, 64, True),      # 512 small items: more items than SMs, several rounds
    (3, 5, 2300, 128, False),    # long non-causal rows with a ragged tail
    (1, 2, 2048, 64, True),      # d = 64 with many key tiles
])
def test_more_forward_shapes(B, H, N, d, causal):
    q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=B * H + N)
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    rows = sorted(set(inputs.sample_rows(N, 64, seed=N).tolist()) | {0, N - 1})
    ro, rl = _ref(q, k, v, causal, rows)
    assert np.abs(o[:, :, rows].float().cpu().numpy() - ro).max() <= TOL_O
    assert np.abs(lse[:, :, rows].cpu().numpy() - rl).max() <= TOL_L


def test_fp32_longer_causal():
    q, k, v = inputs.forward_inputs(1, 2, 2048, 128, torch.float32, seed=77)
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    rows = [0, 1, 700, 2047]
    ro, rl = _ref(q, k, v, True, rows)
    assert np.abs(o[:, :, rows].cpu().numpy() - ro).max() <= 1e-5
    assert np.abs(lse[:, :, rows].cpu().numpy() - rl).max() <= 1e-5


@pytest.mark.parametrize("S,H,max_ctx,ctx", [
    (3, 1, 1000, [1000, 999, 17]),        # one head, 63-block tables
    (4, 7, 33, [33, 32, 16, 1]),          # tables of 3 blocks
    (2, 2, 5000, [5000, 4097]),           # more partitions than the benchmark workload
])
def test_decode_shapes(S, H, max_ctx, ctx):
    di = inputs.decode_inputs(S, H, 128, 16, max_ctx, seed=S * H, device=DEV)
    di.context_lens.copy_(torch.tensor(ctx, dtype=torch.int32, device=DEV))
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens, di.scale)
    torch.cuda.synchronize()
    ro, _ = oracle.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                                di.scale)
    assert np.abs(out.float().cpu().numpy() - ro).max() <= TOL_O


def test_decode_workspace_grows_on_a_second_stream_while_a_forward_runs():
    """A small decode on one stream, then (ordered after it by an event) a
    larger decode on a second stream whose split-K workspace must grow, in
    stream order, while a forward runs on a third stream.  Nothing waits for
    the device in between; all three results match the oracle."""
    fa.fa_release()   # start from an empty workspace, so the second decode grows it
    small = inputs.decode_inputs(2, 2, 128, 16, 600, seed=51, device=DEV)
    large = inputs.decode_inputs(24, 8, 128, 16, 3000, seed=52, device=DEV)
    q, k, v = (t.to(DEV) for t in inputs.forward_inputs(2, 8, 2048, 128, torch.bfloat16, seed=53))
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s3):
        o, lse = fa.forward(q, k, v, causal=True)
    with torch.cuda.stream(s1):
        out_small = fa.paged_decode(small.q, small.k_cache, small.v_cache, small.block_tables,
                                    small.context_lens, small.scale)
        done = torch.cuda.Event()
        done.record(s1)
    s2.wait_event(done)
    with torch.cuda.stream(s2):
        out_large = fa.paged_decode(large.q, large.k_cache, large.v_cache, large.block_tables,
                                    large.context_lens, large.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for di, out in ((small, out_small), (large, out_large)):
        ro, _ = oracle.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables,
                                    di.context_lens, di.scale)
        assert np.abs(out.float().cpu().numpy() - ro).max() <= TOL_O
    rows = [0, 1000, 2047]
    ro, rl = _ref(q.cpu(), k.cpu(), v.cpu(), True, rows)
    assert np.abs(o[:, :, rows].float().cpu().numpy() - ro).max() <= TOL_O
    assert np.abs(lse[:, :, rows].cpu().numpy() - rl).max() <= TOL_L


def test_decode_workspace_cannot_grow_during_capture():
    """A call being captured into a graph may not allocate: with a workspace
    too small for it, the decode returns FA_ERR_UNSUPPORTED and the capture
    can still be ended."""
    fa.fa_release()
    small = inputs.decode_inputs(1, 1, 128, 16, 100, seed=54, device=DEV)
    large = inputs.decode_inputs(8, 8, 128, 16, 2000, seed=55, device=DEV)
    fa.paged_decode(small.q, small.k_cache, small.v_cache, small.block_tables,
                    small.context_lens, small.scale)
    torch.cuda.synchronize()
    out = torch.empty_like(large.q)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    err = None
    with torch.cuda.stream(s):
        g.capture_begin()
        try:
            fa.fa_paged_decode(large.q.data_ptr(), large.k_cache.data_ptr(),
                               large.v_cache.data_ptr(), large.block_tables.data_ptr(),
                               large.context_lens.data_ptr(), out.data_ptr(), 8, 8, 128, 16,
                               large.max_blocks, large.scale, s.cuda_stream)
        except fa.FattnError as e:
            err = e
        finally:
            g.capture_end()
    assert err is not None and err.status == -2   # FA_ERR_UNSUPPORTED
    torch.cuda.synchronize()


def test_forwards_and_backward_in_one_cuda_graph():
    """The bf16 forward, the masked forward (mask summary and forward, chained
    by dependent launches), the E4M3 forward and the backward captured into
    one CUDA graph replay to the eager results: bit for bit, except dQ, whose
    fp32 sums over key blocks may add in another order (as between two eager
    calls).  Each captured launch keeps its own work-counter slot."""
    B, H, N, d = 1, 4, 640, 128
    q, k, v = (t.to(DEV) for t in inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=71))
    do = inputs.grad_output(B, H, N, d, torch.bfloat16, seed=71).to(DEV)
    g = torch.Generator().manual_seed(71)
    mask = (torch.rand((N, N), generator=g) < 0.5).to(torch.uint8).to(DEV)
    x = fa.quantize_fp8(q, k, v)
    ws = torch.empty((fa.fa_backward_workspace_bytes(B, H, N, d),), dtype=torch.uint8,
                     device=DEV)
    o, om, o8 = (torch.empty_like(q) for _ in range(3))
    lse, lm, l8 = (torch.empty((B, H, N), dtype=torch.float32, device=DEV) for _ in range(3))

    def work():
        fa.forward(q, k, v, causal=True, out=o, lse=lse)
        fa.forward_masked(q, k, v, mask, out=om, lse=lm)
        fa.forward_fp8(x, causal=True, out=o8, lse=l8)
        return fa.backward(q, k, v, o, lse, do, causal=True, workspace=ws)

    eager_grads = work()   # also sizes the library's mask summary buffer
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, om, lm, o8, l8)]
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            grads = work()
    torch.cuda.synchronize()
    for _ in range(3):
        for t in (o, lse, om, lm, o8, l8) + tuple(grads):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert fa.fa_device_status() == 0
        for got, want in zip((o, lse, om, lm, o8, l8), eager):
            assert torch.equal(got, want)
        assert torch.equal(grads[1], eager_grads[1]) and torch.equal(grads[2], eager_grads[2])
        dq, dq0 = grads[0].float(), eager_grads[0].float()
        assert (dq - dq0).abs().max().item() <= 2 ** -7 * dq0.abs().max().item()
