"""fa_paged_decode_noalloc: the paged decode for callers that may not
allocate device memory while they run -- a server whose memory pool claimed
all of HBM at start-up, a latency-bound loop that cannot accept the device
synchronisation cudaMalloc/cudaFree may cause, a plug-in whose host
framework owns every allocation.  Its split-K scratch is a fixed device
array inside the library.  It runs the same kernel with the same split as
fa_paged_decode, so its output must be bit-identical to that call's, call
after call, although every call reuses (and leaves behind) the same scratch
contents; and once the library is loaded, a call must not change the
device's free memory.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import pytest
import torch

import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _call(fn, di, out, stream):
    S, H, D = di.q.shape
    fn(di.q.data_ptr(), di.k_cache.data_ptr(), di.v_cache.data_ptr(),
       di.block_tables.data_ptr(), di.context_lens.data_ptr(), out.data_ptr(), S, H, D,
       di.block_size, di.max_blocks, di.scale, stream)


@pytest.mark.parametrize("num_seqs,num_heads,max_ctx,seed", [
    (64, 32, 4096, 5),    # the benchmark's decode workload (~8.5 MB of scratch)
    (7, 3, 1500, 21),     # ragged contexts spanning 1-3 partitions
])
def test_noalloc_matches_allocating_decode_twice(num_seqs, num_heads, max_ctx, seed):
    di = inputs.decode_inputs(num_seqs, num_heads, 128, 16, max_ctx, seed=seed, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    ref = torch.empty_like(di.q)
    _call(fa.fa_paged_decode, di, ref, stream)
    outs = [torch.full_like(di.q, float("nan")) for _ in range(2)]
    for got in outs:  # the second call starts from the first call's leftovers
        _call(fa.fa_paged_decode_noalloc, di, got, stream)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for got in outs:
        assert torch.equal(got, ref), \
            f"max |noalloc - decode| = {(got.float() - ref.float()).abs().max().item():.3e}"


def test_noalloc_calls_leave_free_device_memory_unchanged():
    """With the library's own decode workspace released, one warm-up call and
    then two calls on a problem that fa_paged_decode would need to grow that
    workspace for leave the device's free memory unchanged; the allocating
    decode, run afterwards, gives the same bits."""
    warm = inputs.decode_inputs(2, 2, 128, 16, 100, seed=31, device=DEV)
    big = inputs.decode_inputs(48, 32, 128, 16, 4096, seed=32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    w_out = torch.empty_like(warm.q)
    outs = [torch.empty_like(big.q) for _ in range(2)]
    ref = torch.empty_like(big.q)
    fa.fa_release()
    _call(fa.fa_paged_decode_noalloc, warm, w_out, stream)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for got in outs:
        _call(fa.fa_paged_decode_noalloc, big, got, stream)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, f"free memory moved by {free_before - free_after} bytes"
    _call(fa.fa_paged_decode, big, ref, stream)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for got in outs:
        assert torch.equal(got, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    di = inputs.decode_inputs(2, 2, 128, 16, 64, seed=3, device=DEV)
    out = torch.empty_like(di.q)
    stream = torch.cuda.current_stream().cuda_stream
    # 4096 sequences x 64 heads x 256 blocks would need ~545 MB of scratch.
    with pytest.raises(fa.FattnError) as exc:
        fa.fa_paged_decode_noalloc(di.q.data_ptr(), di.k_cache.data_ptr(),
                                   di.v_cache.data_ptr(), di.block_tables.data_ptr(),
                                   di.context_lens.data_ptr(), out.data_ptr(), 4096, 64, 128, 16,
                                   256, di.scale, stream)
    assert exc.value.status == -2  # FA_ERR_UNSUPPORTED
