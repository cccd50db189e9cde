"""fa_paged_decode_noalloc: the paged decode for callers that cannot allocate
device memory during a call (for example a server whose memory pool owns all
of HBM, or a loop that cannot afford cudaMalloc's synchronisation).  Its
split-K scratch is a fixed device array inside the library, so it must give
the same result as fa_paged_decode, call after call, even though every call
reuses (and leaves behind) the same scratch contents.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import pytest
import torch

import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 2e-2  # the decode parity tolerance used throughout the suite
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
    for _ in range(2):  # the second call starts from the first call's leftovers
        got = torch.full_like(di.q, float("nan"))
        _call(fa.fa_paged_decode_noalloc, di, got, stream)
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all()
        err = (got.float() - ref.float()).abs().max().item()
        assert err <= TOL, f"max |noalloc - decode| = {err:.3e}"


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
