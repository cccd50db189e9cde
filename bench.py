"""Benchmark of libfattn's hot path on GB300.

One step = one exact attention forward over the 2 x 16 x 4096 x 128 causal
bf16 workload (fa_forward) + one paged decode over the 64-sequence x 32-head
x head 128 workload with contexts uniform in [1, 4096] (fa_paged_decode):
every row of the hot path.  Inputs are seeded synthetic draws, resident in
device memory before timing starts.  Each kernel launch is bracketed by CUDA
events on the stream it runs on.  L2 is flushed (a 512 MiB write) before each
forward and backward launch, outside the events; the decodes read more than L2
holds (2.2 GB and 0.55 GB per launch) and are not flushed.

Printed JSON line (rank 0):
  value          forward TFLOP/s, FLOPs = 4*B*H*N^2*d/2 (causal)
  decode         decode GB/s over the algorithmic bytes (K/V of every context
                 token, q, block table entries read, out)
  roofline       the forward (dominant kernel) against the measured bf16 peak
  fwd_f16        fa_forward_f16 on the forward workload in fp16 (same FLOPs)
  fwd_masked     fa_forward_masked with the tril mask on the forward workload
  fwd_d256       fa_forward on 2 x 8 x 4096 x 256 causal (head dimension 256)
  fwd_fp8        fa_forward_fp8 on the forward workload quantized to E4M3 by
                 fa_quantize_fp8 (timed separately), against 2x the bf16 peak
  backward       fa_backward (dQ, dK, dV) of the forward workload, TFLOP/s with
                 FLOPs = 2.5 x the forward's, and its own roofline
  decode_gqa     fa_paged_decode_gqa on the decode's sequences with 8 key/value
                 heads for the 32 query heads, GB/s and HBM roofline
  e2e            the same metrics through the C ABI with pinned host buffers,
                 host<->device copies inside the timed region (copy-in, compute
                 and copy-out of consecutive steps overlap on three streams)
  cpu_baseline   the float64 CPU oracle on the host cores, on a sample
--impl reference times that oracle alone (the reference arm of this build).
Multi-GPU (torchrun): each rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FWD = dict(B=2, H=16, N=4096, d=128, causal=True, seed=3)
# The long-sequence forward, timed separately and reported nested.
FWD_LONG = dict(B=1, H=8, N=16384, d=128, causal=True, seed=4, amp=0.5)
DEC = dict(num_seqs=64, num_heads=32, head_size=128, block_size=16, max_ctx=4096, seed=5)
# Head dimension 256, timed separately and reported nested.
FWD_D256 = dict(B=2, H=8, N=4096, d=256, causal=True, seed=6)
# Grouped key/value heads: the same sequences and contexts, 8 cached heads.
DEC_GQA = dict(DEC, num_kv_heads=8)
L2_FLUSH_BYTES = 512 << 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "fwd attention TFLOPS & % of BF16 tensor peak; paged-decode HBM GB/s"


def fwd_flops(B, H, N, d, causal, **_):
    """Algorithmic FLOPs of one forward: QK^T and PV, 2*N*N*d each per head,
    halved under the causal mask."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def bwd_flops_of(B, H, N, d, causal, **_):
    """Algorithmic FLOPs of one backward: the S recomputation and dP = dO V^T,
    dV, dK and dQ products, 2*N*N*d each per head (five against the forward's
    two), halved under the causal mask."""
    return 2.5 * fwd_flops(B, H, N, d, causal)


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu record, or None when the
    kernel's sources changed since that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    for src, digest in rec["sources"].items():
        try:
            with open(os.path.join(ROOT, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest()[:16] != digest:
                    return None
        except OSError:
            return None
    return rec["dram_read_bytes"] + rec["dram_write_bytes"]


def reduce_over_ranks(times, status, device):
    """The job's figures across ranks: every time is the slowest rank's (max)
    and the status is the worst one (min: error codes are negative)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(times), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    st = torch.tensor([int(status)], device=device, dtype=torch.int32)
    dist.all_reduce(st, op=dist.ReduceOp.MIN)
    return t.tolist(), int(st.item())


def weak_scaling_rate(units_per_rank, world_size, max_ms, unit_scale):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (each rank runs its own replica of the workload)."""
    return world_size * units_per_rank / (max_ms * 1e-3) / unit_scale


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# The GPU arm

def gpu_arm(args):
    import torch
    import torch.distributed as dist

    import exact_attention_11_gb300 as fa
    from exact_attention_11_gb300 import _build, inputs

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    fa.load()

    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    B, H, N, d, causal = FWD["B"], FWD["H"], FWD["N"], FWD["d"], FWD["causal"]
    # Each rank draws its own replica (weak scaling): seed offset by rank.
    q, k, v = (t.to(dev) for t in inputs.forward_inputs(B, H, N, d, torch.bfloat16,
                                                         seed=FWD["seed"] + 1000 * rank))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    di = inputs.decode_inputs(DEC["num_seqs"], DEC["num_heads"], DEC["head_size"],
                              DEC["block_size"], DEC["max_ctx"], seed=DEC["seed"] + 1000 * rank,
                              device=dev)
    out = torch.empty_like(di.q)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    scale = d ** -0.5

    def run_fwd():
        fa.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, H, N, d, scale, causal, sptr)

    S, Hd, D = di.q.shape

    def run_dec():
        fa.fa_paged_decode(di.q.data_ptr(), di.k_cache.data_ptr(), di.v_cache.data_ptr(),
                           di.block_tables.data_ptr(), di.context_lens.data_ptr(),
                           out.data_ptr(), S, Hd, D, di.block_size, di.max_blocks, di.scale, sptr)

    flops = fwd_flops(**FWD)
    bwd_flops = bwd_flops_of(**FWD)
    ctx = di.context_lens.to(torch.int64)
    n_blk = int(((ctx + di.block_size - 1) // di.block_size).sum())
    dec_bytes = (di.kv_bytes_read() + di.q.numel() * 2 + out.numel() * 2 + n_blk * 4
                 + S * 4)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            run_fwd()
            run_dec()
    stream.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the load
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush.zero_()   # the forward's inputs (100 MB) fit in L2
            evs[i][0].record(stream)
            run_fwd()
            evs[i][1].record(stream)
            # the decode reads 2.2 GB per launch, far more than L2 holds: no flush
            # (a flush write would leave 126 MB of dirty lines for it to evict)
            evs[i][2].record(stream)
            run_dec()
            evs[i][3].record(stream)
    stream.synchronize()
    wall = time.perf_counter() - t0
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    dec_ms = sum(e[2].elapsed_time(e[3]) for e in evs) / K
    status = fa.fa_device_status()

    peaks, peak_kind = read_peaks()

    # The long-sequence forward: timed the same way, reported as "fwd_long".
    LB, LH, LN, Ld = FWD_LONG["B"], FWD_LONG["H"], FWD_LONG["N"], FWD_LONG["d"]
    lq, lk, lv = (t.to(dev) for t in inputs.forward_inputs(
        LB, LH, LN, Ld, torch.bfloat16, seed=FWD_LONG["seed"] + 1000 * rank, amp=FWD_LONG["amp"]))
    lo = torch.empty_like(lq)
    llse = torch.empty((LB, LH, LN), dtype=torch.float32, device=dev)

    def run_long():
        fa.fa_forward(lq.data_ptr(), lk.data_ptr(), lv.data_ptr(), lo.data_ptr(), llse.data_ptr(),
                      LB, LH, LN, Ld, Ld ** -0.5, True, sptr)

    kl = max(3, min(K // 4, 100))
    lev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(kl)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush.zero_()
            run_long()
        for i in range(kl):
            flush.zero_()
            lev[i][0].record(stream)
            run_long()
            lev[i][1].record(stream)
    stream.synchronize()
    long_ms = sum(e[0].elapsed_time(e[1]) for e in lev) / kl
    del lq, lk, lv, lo, llse

    # The fp16 forward on the same workload, timed the same way, as "fwd_f16".
    hq16, hk16, hv16 = (t.to(torch.float16) for t in inputs.forward_inputs(
        B, H, N, d, torch.float32, seed=FWD["seed"] + 1000 * rank))
    q16, k16, v16 = (t.to(dev) for t in (hq16, hk16, hv16))
    o16 = torch.empty_like(q16)

    def run_f16():
        fa.fa_forward_f16(q16.data_ptr(), k16.data_ptr(), v16.data_ptr(), o16.data_ptr(),
                          lse.data_ptr(), B, H, N, d, scale, causal, sptr)

    kf = max(3, min(K // 4, 100))
    fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(kf)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush.zero_()
            run_f16()
        for i in range(kf):
            flush.zero_()
            fev[i][0].record(stream)
            run_f16()
            fev[i][1].record(stream)
    stream.synchronize()
    f16_ms = sum(e[0].elapsed_time(e[1]) for e in fev) / kf
    del q16, k16, v16, o16, hq16, hk16, hv16

    # The forward with a boolean mask (tril, the causal pattern as an explicit
    # [N, N] mask), timed the same way, as "fwd_masked".
    tril = torch.tril(torch.ones(N, N, dtype=torch.uint8, device=dev))

    def run_masked():
        fa.fa_forward_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), tril.data_ptr(), 0, B, H, N, d, scale, sptr)

    km = max(3, min(K // 4, 100))
    mev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(km)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush.zero_()
            run_masked()
        for i in range(km):
            flush.zero_()
            mev[i][0].record(stream)
            run_masked()
            mev[i][1].record(stream)
    stream.synchronize()
    masked_ms = sum(e[0].elapsed_time(e[1]) for e in mev) / km
    del tril

    # Head dimension 256 (2 x 8 x 4096 x 256 causal), timed the same way, as
    # "fwd_d256".
    DB, DH, DN, Dd = FWD_D256["B"], FWD_D256["H"], FWD_D256["N"], FWD_D256["d"]
    dq_, dk_, dv_ = (t.to(dev) for t in inputs.forward_inputs(
        DB, DH, DN, Dd, torch.bfloat16, seed=FWD_D256["seed"] + 1000 * rank))
    do_ = torch.empty_like(dq_)
    dlse = torch.empty((DB, DH, DN), dtype=torch.float32, device=dev)

    def run_d256():
        fa.fa_forward(dq_.data_ptr(), dk_.data_ptr(), dv_.data_ptr(), do_.data_ptr(),
                      dlse.data_ptr(), DB, DH, DN, Dd, Dd ** -0.5, FWD_D256["causal"], sptr)

    kd = max(3, min(K // 4, 100))
    dev_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(kd)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush.zero_()
            run_d256()
        for i in range(kd):
            flush.zero_()
            dev_ev[i][0].record(stream)
            run_d256()
            dev_ev[i][1].record(stream)
    stream.synchronize()
    d256_ms = sum(e[0].elapsed_time(e[1]) for e in dev_ev) / kd
    del dq_, dk_, dv_, do_, dlse

    # The FP8 forward on the same workload: the inputs are block-quantized to
    # E4M3 once (fa_quantize_fp8), then fa_forward_fp8 is timed the same way,
    # and the quantization on its own; reported as "fwd_fp8".
    x8 = fa.quantize_fp8(q, k, v)
    qws = torch.empty((max(fa.fa_quantize_fp8_workspace_bytes(B, H, N, d), 16),),
                      dtype=torch.uint8, device=dev)

    def run_fp8():
        fa.fa_forward_fp8(x8.q8.data_ptr(), x8.k8.data_ptr(), x8.vt8.data_ptr(),
                          x8.q_scale.data_ptr(), x8.k_scale.data_ptr(), x8.v_scale.data_ptr(),
                          o.data_ptr(), lse.data_ptr(), B, H, N, d, scale, causal, sptr)

    def run_quant():
        fa.fa_quantize_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), None, x8.q8.data_ptr(),
                           x8.k8.data_ptr(), x8.vt8.data_ptr(), x8.q_scale.data_ptr(),
                           x8.k_scale.data_ptr(), x8.v_scale.data_ptr(), B, H, N, d,
                           qws.data_ptr(), qws.numel(), sptr)

    kq = max(3, min(K // 4, 100))
    qev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(kq)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush.zero_()
            run_quant()
            flush.zero_()
            run_fp8()
        for i in range(kq):
            flush.zero_()
            qev[i][0].record(stream)
            run_fp8()
            qev[i][1].record(stream)
            flush.zero_()
            qev[i][2].record(stream)
            run_quant()
            qev[i][3].record(stream)
    stream.synchronize()
    fp8_ms = sum(e[0].elapsed_time(e[1]) for e in qev) / kq
    quant_ms = sum(e[2].elapsed_time(e[3]) for e in qev) / kq
    del x8, qws
    with torch.cuda.stream(stream):
        run_fwd()   # o, lse of the causal forward again (the backward uses them)

    # The backward (dQ, dK, dV) of the main forward workload, timed the same
    # way on the forward's own O and LSE, reported as "backward".
    g_out = inputs.grad_output(B, H, N, d, torch.bfloat16, seed=FWD["seed"] + 1000 * rank).to(dev)
    gq, gk, gv = (torch.empty_like(q) for _ in range(3))
    bws_bytes = fa.fa_backward_workspace_bytes(B, H, N, d)
    bws = torch.empty((bws_bytes,), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        run_fwd()

    def run_bwd():
        fa.fa_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), g_out.data_ptr(),
                       lse.data_ptr(), gq.data_ptr(), gk.data_ptr(), gv.data_ptr(), B, H, N, d,
                       scale, causal, bws.data_ptr(), bws_bytes, sptr)

    kb = max(3, min(K // 4, 100))
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(kb)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush.zero_()
            run_bwd()
        for i in range(kb):
            flush.zero_()
            bev[i][0].record(stream)
            run_bwd()
            bev[i][1].record(stream)
    stream.synchronize()
    bwd_ms = sum(e[0].elapsed_time(e[1]) for e in bev) / kb
    del g_out, gq, gk, gv, bws

    # The grouped-head decode (4 query heads per cached head), timed the same
    # way, reported as "decode_gqa".  The automatic choice runs the
    # tensor-core kernel here, then its partition-merge kernel: two launches.
    dg = inputs.decode_inputs(DEC_GQA["num_seqs"], DEC_GQA["num_heads"], DEC_GQA["head_size"],
                              DEC_GQA["block_size"], DEC_GQA["max_ctx"],
                              seed=DEC_GQA["seed"] + 1000 * rank, device=dev,
                              num_kv_heads=DEC_GQA["num_kv_heads"])
    gout = torch.empty_like(dg.q)
    Sg, Hg, Dg = dg.q.shape

    def run_gqa():
        fa.fa_paged_decode_gqa(dg.q.data_ptr(), dg.k_cache.data_ptr(), dg.v_cache.data_ptr(),
                               dg.block_tables.data_ptr(), dg.context_lens.data_ptr(),
                               gout.data_ptr(), Sg, Hg, dg.num_kv_heads, Dg, dg.block_size,
                               dg.max_blocks, dg.scale, sptr)

    gctx = dg.context_lens.to(torch.int64)
    g_blk = int(((gctx + dg.block_size - 1) // dg.block_size).sum())
    gqa_bytes = (dg.kv_bytes_read() + dg.q.numel() * 2 + gout.numel() * 2
                 + g_blk * 4 + Sg * 4)
    kg = max(3, min(K // 4, 100))
    gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(kg)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            run_gqa()
        for i in range(kg):   # 0.55 GB read per launch, larger than L2: no flush
            gev[i][0].record(stream)
            run_gqa()
            gev[i][1].record(stream)
    stream.synchronize()
    gqa_ms = sum(e[0].elapsed_time(e[1]) for e in gev) / kg
    del dg, gout

    # End to end through the C ABI with pinned host buffers: every step copies
    # its inputs host -> device, runs the call and copies its results back.
    # The three stages run on their own streams over two device slots, as a
    # serving loop overlaps them (step i+1's inputs arrive while step i
    # computes); the timed region runs from the first copy in to the last copy
    # out, so every step's transfers are inside it.
    ke = max(3, min(K, 50))

    def pipeline(h2d, compute, d2h):
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def run(n, first):
            for i in range(first, first + n):
                sl = i % 2
                if i >= 2:
                    s_in.wait_event(ev_out[sl])      # the slot's previous results are out
                with torch.cuda.stream(s_in):
                    h2d(sl)
                ev_in[sl].record(s_in)
                stream.wait_event(ev_in[sl])
                compute(sl)
                ev_comp[sl].record(stream)
                s_out.wait_event(ev_comp[sl])
                with torch.cuda.stream(s_out):
                    d2h(sl)
                ev_out[sl].record(s_out)

        run(2, 0)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        run(ke, 2)
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / ke

    hq, hk, hv = (torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(3))
    for h, t in zip((hq, hk, hv), (q, k, v)):
        h.copy_(t)
    ho = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True) for _ in range(2)]
    dqkv = [[torch.empty_like(q) for _ in range(3)] for _ in range(2)]
    do_ = [torch.empty_like(o) for _ in range(2)]
    dl = [torch.empty_like(lse) for _ in range(2)]

    def fwd_h2d(sl):
        for dst, src in zip(dqkv[sl], (hq, hk, hv)):
            dst.copy_(src, non_blocking=True)

    def fwd_compute(sl):
        a, b_, c = dqkv[sl]
        fa.fa_forward(a.data_ptr(), b_.data_ptr(), c.data_ptr(), do_[sl].data_ptr(),
                      dl[sl].data_ptr(), B, H, N, d, scale, causal, sptr)

    def fwd_d2h(sl):
        ho[sl].copy_(do_[sl], non_blocking=True)
        hl[sl].copy_(dl[sl], non_blocking=True)

    e2e_fwd_ms = pipeline(fwd_h2d, fwd_compute, fwd_d2h)
    del dqkv, do_, dl

    hdq = torch.empty(di.q.shape, dtype=di.q.dtype, pin_memory=True)
    hdq.copy_(di.q)
    hbt = torch.empty(di.block_tables.shape, dtype=torch.int32, pin_memory=True)
    hbt.copy_(di.block_tables)
    hcl = torch.empty(di.context_lens.shape, dtype=torch.int32, pin_memory=True)
    hcl.copy_(di.context_lens)
    hout = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    ddec = [(torch.empty_like(di.q), torch.empty_like(di.block_tables),
             torch.empty_like(di.context_lens), torch.empty_like(out)) for _ in range(2)]

    def dec_h2d(sl):
        ddq, dbt, dcl, _ = ddec[sl]
        ddq.copy_(hdq, non_blocking=True)
        dbt.copy_(hbt, non_blocking=True)
        dcl.copy_(hcl, non_blocking=True)

    def dec_compute(sl):
        ddq, dbt, dcl, dout_ = ddec[sl]
        fa.fa_paged_decode(ddq.data_ptr(), di.k_cache.data_ptr(), di.v_cache.data_ptr(),
                           dbt.data_ptr(), dcl.data_ptr(), dout_.data_ptr(), S, Hd, D,
                           di.block_size, di.max_blocks, di.scale, sptr)

    def dec_d2h(sl):
        hout[sl].copy_(ddec[sl][3], non_blocking=True)

    e2e_dec_ms = pipeline(dec_h2d, dec_compute, dec_d2h)
    del ddec
    h2d = 3 * q.numel() * 2 + di.q.numel() * 2 + di.block_tables.numel() * 4 + S * 4
    d2h = o.numel() * 2 + lse.numel() * 4 + out.numel() * 2

    if ws > 1:
        (fwd_ms, dec_ms, e2e_fwd_ms, e2e_dec_ms, wall, long_ms, bwd_ms, gqa_ms,
         f16_ms, masked_ms), status = reduce_over_ranks(
            [fwd_ms, dec_ms, e2e_fwd_ms, e2e_dec_ms, wall, long_ms, bwd_ms, gqa_ms, f16_ms,
             masked_ms], status, dev)

    tflops = weak_scaling_rate(flops, ws, fwd_ms, 1e12)
    per_gpu_tflops = weak_scaling_rate(flops, 1, fwd_ms, 1e12)
    gbs = weak_scaling_rate(dec_bytes, ws, dec_ms, 1e9)
    per_gpu_gbs = weak_scaling_rate(dec_bytes, 1, dec_ms, 1e9)
    peak_t = peaks["bf16_tflops"]
    peak_h = peaks["hbm_gbs"]
    result = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(fwd_ms + dec_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs; no dataset)",
        "config": {
            "workload": "fa_forward bf16 B=2 H=16 N=4096 d=128 causal + fa_paged_decode bf16 "
                        "64 seqs x 32 heads x head 128, block 16, ctx U[1,4096]",
            "fwd": {k_: v_ for k_, v_ in FWD.items() if k_ != "seed"},
            "decode": {k_: v_ for k_, v_ in DEC.items() if k_ != "seed"},
            "decode_sum_ctx": int(ctx.sum()),
            "l2": "forward, 16K, fp16, masked, d256 and FP8 forwards, FP8 quantization and "
                  "backward: flushed (512 MiB write) before every timed launch; decode "
                  "(2.2 GB read per launch) and grouped decode (0.55 GB): inputs larger than "
                  "L2, not flushed",
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "sms": torch.cuda.get_device_properties(dev).multi_processor_count,
        },
        "fwd_ms": round(fwd_ms, 4),
        "fwd_long": {
            "workload": "fa_forward bf16 B=1 H=8 N=16384 d=128 causal, inputs N(0,1)*0.5",
            "ms": round(long_ms, 4),
            "value": round(weak_scaling_rate(fwd_flops(**FWD_LONG), ws, long_ms, 1e12), 2),
            "unit": "TFLOP/s",
            "frac_of_bf16_peak": round(fwd_flops(**FWD_LONG) / (long_ms * 1e-3) / 1e12
                                       / peaks["bf16_tflops"], 4),
        },
        "fwd_f16": {
            "workload": "fa_forward_f16 fp16 B=2 H=16 N=4096 d=128 causal (the forward's inputs "
                        "rounded to fp16)",
            "ms": round(f16_ms, 4),
            "value": round(weak_scaling_rate(flops, ws, f16_ms, 1e12), 2),
            "unit": "TFLOP/s",
            "frac_of_bf16_peak": round(flops / (f16_ms * 1e-3) / 1e12 / peak_t, 4),
        },
        "fwd_masked": {
            "workload": "fa_forward_masked bf16 B=2 H=16 N=4096 d=128 with the [N,N] tril mask "
                        "(key tiles no row of a work item sees are skipped; FLOPs counted for the "
                        "visible half; the mask's tile summary is inside the timed call)",
            "ms": round(masked_ms, 4),
            "value": round(weak_scaling_rate(flops, ws, masked_ms, 1e12), 2),
            "unit": "TFLOP/s",
            "frac_of_bf16_peak": round(flops / (masked_ms * 1e-3) / 1e12 / peak_t, 4),
            "traffic_forward_kernel": recorded_traffic("fwd_bf16_tc_kernel<128,0,1,0>"),
        },
        "fwd_d256": {
            "workload": "fa_forward bf16 B=2 H=8 N=4096 d=256 causal",
            "ms": round(d256_ms, 4),
            "value": round(weak_scaling_rate(fwd_flops(**FWD_D256), ws, d256_ms, 1e12), 2),
            "unit": "TFLOP/s",
            "frac_of_bf16_peak": round(fwd_flops(**FWD_D256) / (d256_ms * 1e-3) / 1e12 / peak_t,
                                       4),
            "roofline": {"bound": "tensor",
                         "achieved": round(weak_scaling_rate(fwd_flops(**FWD_D256), 1, d256_ms,
                                                             1e12), 2),
                         "peak": peak_t, "unit": "TFLOP/s",
                         "frac": round(weak_scaling_rate(fwd_flops(**FWD_D256), 1, d256_ms, 1e12)
                                       / peak_t, 4),
                         "traffic": recorded_traffic("fwd_d256_kernel<0>"),
                         "peak_kind": f"{peak_kind} bf16 burst", "kernel": "fwd_d256_kernel<0>"},
        },
        "fwd_fp8": {
            "workload": "fa_forward_fp8 on the forward workload block-quantized to E4M3 "
                        "(fa_quantize_fp8: 128-row blocks for Q and K, per-head V; no "
                        "transform), bf16 output",
            "ms": round(fp8_ms, 4),
            "value": round(weak_scaling_rate(flops, ws, fp8_ms, 1e12), 2),
            "unit": "TFLOP/s",
            "quantize_ms": round(quant_ms, 4),
            "value_with_quantize": round(weak_scaling_rate(flops, ws, fp8_ms + quant_ms, 1e12), 2),
            "roofline": {"bound": "tensor",
                         "achieved": round(weak_scaling_rate(flops, 1, fp8_ms, 1e12), 2),
                         "peak": round(2 * peak_t, 1), "unit": "TFLOP/s",
                         "frac": round(weak_scaling_rate(flops, 1, fp8_ms, 1e12) / (2 * peak_t), 4),
                         "traffic": recorded_traffic("fwd_bf16_tc_kernel<128,0,0,1>"),
                         "peak_kind": f"{peak_kind} bf16 burst x 2 (nominal fp8/bf16 ratio)",
                         "kernel": "fwd_bf16_tc_kernel<128,0,0,1> (E4M3)"},
        },
        "backward": {
            "workload": "fa_backward bf16 B=2 H=16 N=4096 d=128 causal (dQ, dK, dV of the "
                        "forward workload, upstream gradient N(0,1))",
            "ms": round(bwd_ms, 4),
            "value": round(weak_scaling_rate(bwd_flops, ws, bwd_ms, 1e12), 2),
            "unit": "TFLOP/s",
            "flops_per_launch": bwd_flops,
            "roofline": {"bound": "tensor",
                         "achieved": round(weak_scaling_rate(bwd_flops, 1, bwd_ms, 1e12), 2),
                         "peak": peak_t, "unit": "TFLOP/s",
                         "frac": round(weak_scaling_rate(bwd_flops, 1, bwd_ms, 1e12) / peak_t, 4),
                         "traffic": recorded_traffic("bwd_pipe_kernel"),
                         "peak_kind": f"{peak_kind} bf16 burst",
                         "kernel": "bwd_prep_kernel + bwd_pipe_kernel + bwd_dq_kernel"},
        },
        "fwd_frac_of_bf16_peak": round(per_gpu_tflops / peak_t, 4),
        "decode": {
            "value": round(gbs, 1), "unit": "GB/s", "ms": round(dec_ms, 4),
            "bytes_per_launch": dec_bytes,
            "roofline": {"bound": "hbm", "achieved": round(per_gpu_gbs, 1), "peak": peak_h,
                         "unit": "GB/s", "frac": round(per_gpu_gbs / peak_h, 4),
                         "traffic": recorded_traffic("paged_decode_kernel"),
                         "peak_kind": peak_kind},
        },
        "decode_gqa": {
            "workload": "fa_paged_decode_gqa bf16 64 seqs x 32 query heads x 8 key/value heads x "
                        "head 128, block 16, ctx U[1,4096] (the decode's contexts); "
                        "tensor-core kernel + partition merge",
            "value": round(weak_scaling_rate(gqa_bytes, ws, gqa_ms, 1e9), 1), "unit": "GB/s",
            "ms": round(gqa_ms, 4), "bytes_per_launch": gqa_bytes,
            "roofline": {"bound": "hbm",
                         "achieved": round(weak_scaling_rate(gqa_bytes, 1, gqa_ms, 1e9), 1),
                         "peak": peak_h, "unit": "GB/s",
                         "frac": round(weak_scaling_rate(gqa_bytes, 1, gqa_ms, 1e9) / peak_h, 4),
                         "traffic": recorded_traffic("paged_decode_gqa_tc_kernel<4>"),
                         "peak_kind": peak_kind},
        },
        "roofline": {"bound": "tensor", "achieved": round(per_gpu_tflops, 2), "peak": peak_t,
                     "unit": "TFLOP/s", "frac": round(per_gpu_tflops / peak_t, 4),
                     "traffic": recorded_traffic("fwd_bf16_tc_kernel<128>"),
                     "peak_kind": f"{peak_kind} bf16 burst",
                     "kernel": "fwd_bf16_tc_kernel<128>", "flops_per_launch": flops},
        "e2e": {"value": round(weak_scaling_rate(flops, ws, e2e_fwd_ms, 1e12), 2), "unit": "TFLOP/s",
                "decode_gbs": round(weak_scaling_rate(dec_bytes, ws, e2e_dec_ms, 1e9), 1),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "KV cache resident (serving state); q, K, V, q_decode, block table, "
                        "context lens copied in and O, LSE, out copied back every step; copies "
                        "in, compute and copies out on three streams over two device slots "
                        "(step i+1's inputs arrive while step i computes)"},
        # library kernels inside timed regions (a backward is three launches)
        # fwd_fp8: kq forwards + kq quantizations of two launches each
        "gpu_launches": 2 * K + kl + kf + km + kd + 3 * kq + 3 * kb + 2 * kg + 2 * ke,
        "clocks": clk,
        "device_status": status,
        "wall_s": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if ws > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


# ---------------------------------------------------------------------------
# The float64 CPU oracle, timed on the host cores

class OracleSampler:
    """Times the float64 oracle on the forward workload, in units of 256
    consecutive query rows of one head (causal), visited in a fixed order, until
    a time budget is spent.  Inputs are drawn once, like the GPU arm's."""

    ROWS = 256

    def __init__(self):
        import torch

        import oracle
        from exact_attention_11_gb300 import inputs
        oracle.build()
        self.oracle = oracle
        B, H, N, d = FWD["B"], FWD["H"], FWD["N"], FWD["d"]
        q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=FWD["seed"])
        self.q, self.k, self.v = (t.double().reshape(B * H, N, d).numpy() for t in (q, k, v))
        self.N, self.d, self.BH = N, d, B * H
        self.units = [(h, r0) for r0 in range(0, N, self.ROWS) for h in range(B * H)]
        self.next = 0
        self.cores = oracle.max_threads()

    def unit_flops(self, r0):
        r1 = min(self.N, r0 + self.ROWS)
        # causal: row i sees i + 1 keys; QK^T and PV cost 2 * (i + 1) * d each
        return 4.0 * self.d * sum(i + 1 for i in range(r0, r1))

    def run(self, budget_s):
        flops, secs, n = 0.0, 0.0, 0
        while n == 0 or secs < budget_s:
            h, r0 = self.units[self.next % len(self.units)]
            self.next += 1
            rows = list(range(r0, min(self.N, r0 + self.ROWS)))
            sl = slice(h, h + 1)
            t0 = time.perf_counter()
            self.oracle.attention_forward_rows(self.q[sl][None], self.k[sl][None],
                                               self.v[sl][None], rows, self.d ** -0.5, True)
            secs += time.perf_counter() - t0
            flops += self.unit_flops(r0)
            n += 1
        return flops, secs, n


def cpu_baseline(target_s: float):
    smp = OracleSampler()
    flops, secs, n = smp.run(target_s)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": smp.cores, "kind": "oracle",
            "sample": f"{n} blocks of 256 causal query rows (of the 512 blocks of the "
                      f"2x16x4096x128 forward), float64, {secs:.1f} s"}


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    smp = OracleSampler()
    # Each step is a bounded sample, sized so the whole run stays near 150 s.
    budget = max(0.02, min(0.5, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        smp.run(budget)
    flops, secs, units = 0.0, 0.0, 0
    for _ in range(args.steps):
        f, s_, n = smp.run(budget)
        flops, secs, units = flops + f, secs + s_, units + n
    value = flops / secs / 1e12
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) inputs; no dataset)",
        "config": {"workload": "fa_forward bf16 B=2 H=16 N=4096 d=128 causal (oracle: blocks "
                               "of 256 query rows per step)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": smp.cores, "kind": "oracle",
                         "sample": f"{units} blocks of 256 causal query rows over "
                                   f"{args.steps} steps, float64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="approximate CPU time for the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        ap.error("--warmup must be >= 3")
    res = reference_arm(args) if args.impl == "reference" else gpu_arm(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
