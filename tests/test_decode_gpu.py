"""Parity of fa_paged_decode (CUDA) with the float64 oracle.

Tolerance: max |out - out_ref| <= 2e-2 (bf16 inputs, fp32 accumulation,
bf16 output).  Context lengths cover the edges of the 16-token cache block
and the 512-token partition, a single token, and an empty context.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 2e-2
DEV = "cuda:0"


def compact(di, seqs):
    """The listed sequences' inputs with only the cache blocks they use,
    renumbered, copied to the host (test plumbing: no attention arithmetic)."""
    bs = di.block_size
    bt = di.block_tables[seqs].cpu()
    cl = di.context_lens[seqs].cpu()
    used = sorted({int(bt[i, b]) for i in range(len(seqs))
                   for b in range((int(cl[i]) + bs - 1) // bs)})
    remap = {pb: n for n, pb in enumerate(used)}
    bt2 = torch.zeros_like(bt)
    for i in range(len(seqs)):
        for b in range((int(cl[i]) + bs - 1) // bs):
            bt2[i, b] = remap[int(bt[i, b])]
    idx = torch.tensor(used if used else [0], dtype=torch.int64, device=di.k_cache.device)
    kc = di.k_cache.index_select(0, idx).cpu()
    vc = di.v_cache.index_select(0, idx).cpu()
    return di.q[seqs].cpu(), kc, vc, bt2, cl


def run_and_check(di, seqs=None):
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens, di.scale)
    torch.cuda.synchronize()
    S = di.q.shape[0]
    seqs = list(range(S)) if seqs is None else list(seqs)
    q, kc, vc, bt, cl = compact(di, seqs)
    ro, _ = oracle.paged_decode(q, kc, vc, bt, cl, di.scale)
    got = out[seqs].float().cpu().numpy()
    err = float(np.abs(got - ro).max())
    assert np.isfinite(got).all()
    assert err <= TOL, f"max|d out| = {err:.3e}"
    return out


def test_decode_small_random():
    di = inputs.decode_inputs(6, 4, 128, 16, 700, seed=11, device=DEV)
    run_and_check(di)


def test_decode_context_edges():
    di = inputs.decode_inputs(12, 3, 128, 16, 1100, seed=12, device=DEV)
    edges = [1, 15, 16, 17, 511, 512, 513, 1024, 1025, 1100, 2, 33]
    di.context_lens.copy_(torch.tensor(edges, dtype=torch.int32, device=DEV))
    run_and_check(di)


def test_decode_empty_context_gives_zeros():
    di = inputs.decode_inputs(3, 2, 128, 16, 64, seed=13, device=DEV)
    di.context_lens.copy_(torch.tensor([0, 5, 0], dtype=torch.int32, device=DEV))
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens, di.scale)
    torch.cuda.synchronize()
    assert (out[0] == 0).all() and (out[2] == 0).all()
    run_and_check(di, seqs=[1])


def test_decode_single_token_returns_its_value():
    """With one context token the softmax weight is exactly 1."""
    di = inputs.decode_inputs(2, 2, 128, 16, 16, seed=14, device=DEV)
    di.context_lens.fill_(1)
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens, di.scale)
    torch.cuda.synchronize()
    for s in range(2):
        pb = int(di.block_tables[s, 0])
        want = di.v_cache[pb, :, :, 0]          # [H, D]: token 0 of the block
        assert torch.equal(out[s], want)


def test_decode_workload_64seq_32head_full():
    """Every output of the 64-sequence, 32-head, 4096-token-max workload
    (caches of 16384 blocks): the oracle runs over all 64 sequences, four at a
    time, so that only the cache blocks of four sequences are widened to
    float64 at once."""
    di = inputs.decode_inputs(64, 32, 128, 16, 4096, seed=5, device=DEV)
    out = fa.paged_decode(di.q, di.k_cache, di.v_cache, di.block_tables, di.context_lens,
                          di.scale)
    torch.cuda.synchronize()
    got_all = out.float().cpu().numpy()
    assert np.isfinite(got_all).all()
    worst = 0.0
    for s0 in range(0, 64, 4):
        seqs = list(range(s0, s0 + 4))
        q, kc, vc, bt, cl = compact(di, seqs)
        ro, _ = oracle.paged_decode(q, kc, vc, bt, cl, di.scale)
        worst = max(worst, float(np.abs(got_all[seqs] - ro).max()))
        del kc, vc
    assert worst <= TOL, f"max|d out| = {worst:.3e}"


def test_decode_repeat_is_deterministic_and_counters_reset():
    di = inputs.decode_inputs(5, 4, 128, 16, 2000, seed=15, device=DEV)
    a = run_and_check(di).clone()
    b = run_and_check(di)
    assert torch.equal(a, b)
    assert fa.fa_device_status() == 0


def poisoned_caches(di):
    """Copies of the caches with NaN in every slot past each sequence's
    context: the tail of its last block and the blocks it does not use."""
    kc, vc = di.k_cache.clone(), di.v_cache.clone()
    bs = di.block_size
    ctx = di.context_lens.cpu().tolist()
    bt = di.block_tables.cpu()
    for s, c in enumerate(ctx):
        for j in range(bt.shape[1]):
            first = c - bs * j                   # first unused slot of this block
            if first >= bs:
                continue
            blk = int(bt[s, j])
            kc[blk, :, :, max(first, 0):, :] = float("nan")
            vc[blk, :, :, max(first, 0):] = float("nan")
    return kc, vc


def test_decode_ignores_cache_slots_past_the_context():
    """Slots past a sequence's context may hold anything: with NaN there the
    output is bit-equal to the clean run, for the allocating and the
    fixed-scratch decode."""
    di = inputs.decode_inputs(6, 4, 128, 16, 1000, seed=16, device=DEV)
    di.context_lens.copy_(torch.tensor([1000, 3, 130, 515, 17, 999], dtype=torch.int32,
                                       device=DEV))
    clean = run_and_check(di).clone()
    kc, vc = poisoned_caches(di)
    out = fa.paged_decode(di.q, kc, vc, di.block_tables, di.context_lens, di.scale)
    out2 = torch.empty_like(out)
    S, H, D = di.q.shape
    fa.fa_paged_decode_noalloc(di.q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                               di.block_tables.data_ptr(), di.context_lens.data_ptr(),
                               out2.data_ptr(), S, H, D, di.block_size, di.block_tables.shape[1],
                               di.scale, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.equal(out, clean)
    assert torch.equal(out2, clean)


def test_decode_shared_prefix_blocks():
    """Sequences sharing physical cache blocks (a common prefix) read them
    independently."""
    di = inputs.decode_inputs(4, 4, 128, 16, 900, seed=17, device=DEV)
    bt = di.block_tables.clone()
    bt[1:, :5] = bt[0, :5]
    di.block_tables.copy_(bt)
    di.context_lens.copy_(torch.tensor([900, 700, 333, 81], dtype=torch.int32, device=DEV))
    run_and_check(di)
