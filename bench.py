"""Benchmark of libfattn's hot path on GB300.

One step = one exact attention forward over the 2 x 16 x 4096 x 128 causal
bf16 workload (fa_forward) + one paged decode over the 64-sequence x 32-head
x head 128 workload with contexts uniform in [1, 4096] (fa_paged_decode):
every row of the hot path.  Inputs are seeded synthetic draws, resident in
device memory before timing starts.  Each kernel launch is bracketed by CUDA
events on the stream it runs on.  L2 is flushed (a 512 MiB write) before each
launch of a workload whose inputs L2 could hold, outside the events; the
decodes read more than L2 holds (2.2 GB and 0.55 GB per launch) and are not
flushed (a separate decode figure is taken after a flush too).

The main loop times exactly --steps steps; `value` (forward TFLOP/s) and the
decode figure come from it.  Every other leg -- the five reference workloads
and the extensions -- runs until its launches have taken at least
--min-seconds of device time (and at least --steps launches), and reports
the median, p10 and p90 of its per-launch times.

Printed JSON line (rank 0), in this order:
  value          forward TFLOP/s (median over the main loop), FLOPs =
                 4*B*H*N^2*d/2 (causal)
  summary        one compact line per reference workload (fp32 64x64;
                 4x16x1024x64; 2x16x4096x128 causal; 1x8x16384x128 causal;
                 the paged decode): rate, fraction of its roofline, median ms
  roofline       the forward (dominant kernel) against the measured bf16 peak
  decode         decode GB/s over the algorithmic bytes (K/V of every context
                 token, q, block table entries read, out), q and out rotated
                 over four buffers; also after an L2 flush
  fwd_f16 / fwd_masked / fwd_d256 / fwd_fp8 / backward / backward_d64 /
  decode_gqa     the extensions, each with its own roofline
  e2e            the same metrics through the C ABI with pinned host buffers,
                 host<->device copies inside the timed region (copy-in, compute
                 and copy-out of consecutive steps overlap on three streams)
  cpu_baseline   the float64 CPU oracle on the host cores, on bounded samples
--impl reference times that oracle alone, as the comparison arm: the same
metric and workload, computed by the float64 CPU implementation.
--only LEG[,LEG] runs only the named legs (no main loop, e2e, CPU baseline or
hashing), allocating only their workloads: the entry used for profiling.
Multi-GPU (torchrun): each rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The five reference workloads.
FWD_F32 = dict(B=1, H=1, N=64, d=64, causal=False, seed=1)
FWD_D64 = dict(B=4, H=16, N=1024, d=64, causal=False, seed=2)
FWD = dict(B=2, H=16, N=4096, d=128, causal=True, seed=3)
FWD_LONG = dict(B=1, H=8, N=16384, d=128, causal=True, seed=4, amp=0.5)
DEC = dict(num_seqs=64, num_heads=32, head_size=128, block_size=16, max_ctx=4096, seed=5)
# Extensions.
FWD_D256 = dict(B=2, H=8, N=4096, d=256, causal=True, seed=6)
BWD_D64 = dict(B=2, H=16, N=4096, d=64, causal=True, seed=3)
DEC_GQA = dict(DEC, num_kv_heads=8)
L2_FLUSH_BYTES = 512 << 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "fwd attention TFLOPS & % of BF16 tensor peak; paged-decode HBM GB/s"
LEGS = ("fwd", "decode", "fwd_f32", "fwd_d64", "fwd_long", "fwd_f16", "fwd_masked", "fwd_d256",
        "fwd_fp8", "backward", "backward_d64", "decode_gqa")


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


def percentiles(ms):
    """median, p10 and p90 of a list of per-launch times (ms)."""
    s = sorted(ms)
    if len(s) == 1:
        return s[0], s[0], s[0]

    def q(f):
        x = f * (len(s) - 1)
        i = int(math.floor(x))
        j = min(i + 1, len(s) - 1)
        return s[i] + (s[j] - s[i]) * (x - i)
    return q(0.5), q(0.1), q(0.9)


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
        # "under load": samples drawing more than a third of the peak power seen
        loaded = [c for c, p in zip(sm, power) if p >= max(power) / 3] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "samples_under_load": len(loaded),
                "reasons": sorted(reasons)}


def tensor_sha256(t, chunk_bytes=256 << 20):
    """sha256 of a tensor's bytes (device tensors copied to the host in chunks)."""
    import torch
    flat = t.reshape(-1).view(torch.uint8)
    h = hashlib.sha256()
    for i in range(0, flat.numel(), chunk_bytes):
        h.update(flat[i:i + chunk_bytes].cpu().numpy().tobytes())
    return h.hexdigest()


# ---------------------------------------------------------------------------
# The GPU arm

class LegTimer:
    """Times one call repeatedly on `stream`, each launch (or, for calls too
    short to time alone and that need no L2 flush, each group of launches)
    between two CUDA events, until the timed launches have taken at least
    `min_s` of device time and there are at least `min_iters` of them."""

    def __init__(self, torch, stream, flush, min_s, min_iters, max_iters=60000):
        self.torch, self.stream, self.flush = torch, stream, flush
        self.min_s, self.min_iters, self.max_iters = min_s, min_iters, max_iters

    def _probe(self, fn, flush):
        torch, s = self.torch, self.stream
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            for _ in range(3):
                if flush:
                    self.flush.zero_()
                fn(0)
            if flush:
                self.flush.zero_()
            a.record(s)
            fn(0)
            b.record(s)
        s.synchronize()
        return max(a.elapsed_time(b), 1e-3)

    def run(self, fn, flush, launches_per_call=1):
        """fn(i) enqueues call i.  Returns the leg's timing record."""
        torch, s = self.torch, self.stream
        est = self._probe(fn, flush)
        group = 1 if flush else max(1, int(math.ceil(0.2 / est)))
        n_groups = max(int(math.ceil(self.min_iters / group)),
                       int(math.ceil(self.min_s * 1e3 / (est * group))))
        n_groups = min(n_groups, max(1, self.max_iters // group))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_groups)]
        i = 0
        with torch.cuda.stream(s):
            for a, b in evs:
                if flush:
                    self.flush.zero_()
                a.record(s)
                for _ in range(group):
                    fn(i)
                    i += 1
                b.record(s)
        s.synchronize()
        per = [a.elapsed_time(b) / group for a, b in evs]
        med, p10, p90 = percentiles(per)
        return {"ms": round(med, 5), "p10_ms": round(p10, 5), "p90_ms": round(p90, 5),
                "calls": i, "device_s": round(sum(per) * group / 1e3, 3),
                "launches": i * launches_per_call}


def _rate_record(units, ms, ws, unit_scale, unit, peak, peak_kind, bound, kernel, traffic,
                 extra=None):
    achieved = weak_scaling_rate(units, 1, ms, unit_scale)
    r = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4), "traffic": traffic, "peak_kind": peak_kind,
         "kernel": kernel}
    if extra:
        r.update(extra)
    return round(weak_scaling_rate(units, ws, ms, unit_scale), 2), r


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

    only = None if not args.only else [x.strip() for x in args.only.split(",") if x.strip()]
    if only:
        bad = [x for x in only if x not in LEGS]
        if bad:
            raise SystemExit(f"unknown legs {bad}; known: {', '.join(LEGS)}")

    def want(leg):
        return only is None or leg in only

    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    timer = LegTimer(torch, stream, flush, args.min_seconds, max(args.steps, 3))
    peaks, peak_kind = read_peaks()
    peak_t, peak_h = peaks["bf16_tflops"], peaks["hbm_gbs"]
    tensor_kind, hbm_kind = f"{peak_kind} bf16 burst", f"{peak_kind} copy"
    legs, times, hashes = {}, {}, {}
    launches = 0
    seed_off = 1000 * rank   # each rank draws its own replica (weak scaling)

    def fwd_inputs(cfg, dtype=torch.bfloat16):
        return tuple(t.to(dev) for t in inputs.forward_inputs(
            cfg["B"], cfg["H"], cfg["N"], cfg["d"], dtype, seed=cfg["seed"] + seed_off,
            amp=cfg.get("amp", 1.0)))

    def decode_workload(cfg, num_seqs):
        return inputs.decode_inputs(num_seqs, cfg["num_heads"], cfg["head_size"],
                                    cfg["block_size"], cfg["max_ctx"], seed=cfg["seed"] + seed_off,
                                    device=dev, num_kv_heads=cfg.get("num_kv_heads"))

    def decode_bytes(di):
        ctx = di.context_lens.to(torch.int64)
        n_blk = int(((ctx + di.block_size - 1) // di.block_size).sum())
        return di.kv_bytes_read() + 2 * di.q.numel() * 2 + n_blk * 4 + di.q.shape[0] * 4

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)   # let the sampler start before the load

    # ---- the main loop: exactly K steps of (forward, decode) ----------------
    main = None
    B, H, N, d, causal = FWD["B"], FWD["H"], FWD["N"], FWD["d"], FWD["causal"]
    scale = d ** -0.5
    need_main_inputs = only is None or "fwd" in only or "fwd_masked" in only
    if need_main_inputs:
        q, k, v = fwd_inputs(FWD)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)

        def run_fwd(_i=0):
            fa.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                          lse.data_ptr(), B, H, N, d, scale, causal, sptr)
    if only is None or "decode" in only:
        di = decode_workload(DEC, args.decode_seqs)
        S, Hd, D = di.q.shape
        # q and out rotate over four buffers, so consecutive launches do not
        # find the previous launch's small tensors in L2.
        dqs = [di.q] + [di.q.clone() for _ in range(3)]
        outs = [torch.empty_like(di.q) for _ in range(4)]
        dec_bytes = decode_bytes(di)

        def run_dec(i=0):
            fa.fa_paged_decode(dqs[i % 4].data_ptr(), di.k_cache.data_ptr(),
                               di.v_cache.data_ptr(), di.block_tables.data_ptr(),
                               di.context_lens.data_ptr(), outs[i % 4].data_ptr(), S, Hd, D,
                               di.block_size, di.max_blocks, di.scale, sptr)
    flops = fwd_flops(**FWD)

    if only is None:
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                flush.zero_()
                run_fwd()
                run_dec(i)
        stream.synchronize()
        K = args.steps
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(K):
                flush.zero_()   # the forward's inputs (100 MB) fit in L2
                evs[i][0].record(stream)
                run_fwd()
                evs[i][1].record(stream)
                # the decode reads 2.2 GB per launch, far more than L2 holds: no flush
                evs[i][2].record(stream)
                run_dec(i)
                evs[i][3].record(stream)
        stream.synchronize()
        wall = time.perf_counter() - t0
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        f_ms = [e[0].elapsed_time(e[1]) for e in evs]
        d_ms = [e[2].elapsed_time(e[3]) for e in evs]
        main = {"fwd": percentiles(f_ms), "dec": percentiles(d_ms),
                "fwd_mean": sum(f_ms) / K, "dec_mean": sum(d_ms) / K, "wall": wall}
        launches += 2 * K
        times["main_fwd"] = main["fwd"][0]
        times["main_dec"] = main["dec"][0]
        if rank == 0 and not args.no_hash:
            for name, t in (("fwd_q", q), ("fwd_k", k), ("fwd_v", v), ("decode_q", di.q),
                            ("decode_block_tables", di.block_tables),
                            ("decode_context_lens", di.context_lens),
                            ("decode_k_cache", di.k_cache), ("decode_v_cache", di.v_cache)):
                hashes[name] = tensor_sha256(t)

    # ---- the 2 x 16 x 4096 x 128 causal forward, >= min_s of launches ------
    if want("fwd"):
        rec = timer.run(run_fwd, True)
        launches += rec["launches"]
        times["fwd"] = rec["ms"]
        legs["fwd"] = rec
    if only is None:
        hq, hk, hv = (torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(3))
        for h, t in zip((hq, hk, hv), (q, k, v)):
            h.copy_(t)

    # ---- the paged decode: rotated buffers, and after an L2 flush ----------
    if want("decode"):
        rec = timer.run(run_dec, False)
        launches += rec["launches"]
        times["decode"] = rec["ms"]
        legs["decode"] = rec
        recf = timer.run(run_dec, True)
        launches += recf["launches"]
        times["decode_flushed"] = recf["ms"]
        legs["decode_flushed"] = recf

    # ---- end to end through the C ABI with pinned host buffers --------------
    # Every step copies its inputs host -> device, runs the call and copies its
    # results back; the three stages run on their own streams over two device
    # slots, as a serving loop overlaps them (step i+1's inputs arrive while
    # step i computes); the timed region runs from the first copy in to the
    # last copy out, so every step's transfers are inside it.
    ke = max(3, min(args.steps, 50))

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

    e2e = None
    if only is None:
        hdq = torch.empty(di.q.shape, dtype=di.q.dtype, pin_memory=True)
        hdq.copy_(di.q)
        hbt = torch.empty(di.block_tables.shape, dtype=torch.int32, pin_memory=True)
        hbt.copy_(di.block_tables)
        hcl = torch.empty(di.context_lens.shape, dtype=torch.int32, pin_memory=True)
        hcl.copy_(di.context_lens)
        hout = [torch.empty(di.q.shape, dtype=di.q.dtype, pin_memory=True) for _ in range(2)]
        ddec = [(torch.empty_like(di.q), torch.empty_like(di.block_tables),
                 torch.empty_like(di.context_lens), torch.empty_like(di.q)) for _ in range(2)]

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
        launches += ke
        dec_h2d_bytes = di.q.numel() * 2 + di.block_tables.numel() * 4 + S * 4
        dec_d2h_bytes = di.q.numel() * 2
        dec_sum_ctx = int(di.context_lens.to(torch.int64).sum())
    if only is None or "decode" in only:
        del di, dqs, outs

    # ---- fp32 forward, 1 x 1 x 64 x 64 --------------------------------------
    if want("fwd_f32"):
        c = FWD_F32
        a, b_, c_ = fwd_inputs(c, torch.float32)
        of = torch.empty_like(a)
        lf = torch.empty((c["B"], c["H"], c["N"]), dtype=torch.float32, device=dev)

        def run_f32(_i=0):
            fa.fa_forward_fp32(a.data_ptr(), b_.data_ptr(), c_.data_ptr(), of.data_ptr(),
                               lf.data_ptr(), c["B"], c["H"], c["N"], c["d"], c["d"] ** -0.5,
                               c["causal"], sptr)
        rec = timer.run(run_f32, False)
        launches += rec["launches"]
        times["fwd_f32"] = rec["ms"]
        legs["fwd_f32"] = rec
        del a, b_, c_, of, lf

    # ---- 4 x 16 x 1024 x 64 non-causal --------------------------------------
    def plain_forward_leg(name, cfg, dtype=torch.bfloat16, fn=None):
        a, b_, c_ = fwd_inputs(cfg, dtype)
        oo = torch.empty_like(a)
        ll = torch.empty((cfg["B"], cfg["H"], cfg["N"]), dtype=torch.float32, device=dev)
        call = fn or fa.fa_forward

        def run(_i=0):
            call(a.data_ptr(), b_.data_ptr(), c_.data_ptr(), oo.data_ptr(), ll.data_ptr(),
                 cfg["B"], cfg["H"], cfg["N"], cfg["d"], cfg["d"] ** -0.5, cfg["causal"], sptr)
        rec = timer.run(run, True)
        times[name] = rec["ms"]
        legs[name] = rec
        return rec

    if want("fwd_d64"):
        launches += plain_forward_leg("fwd_d64", FWD_D64)["launches"]
    if want("fwd_long"):
        launches += plain_forward_leg("fwd_long", FWD_LONG)["launches"]
    if want("fwd_f16"):
        launches += plain_forward_leg("fwd_f16", FWD, torch.float16, fa.fa_forward_f16)["launches"]
    if want("fwd_d256"):
        launches += plain_forward_leg("fwd_d256", FWD_D256)["launches"]

    # ---- the forward with a boolean mask (tril: the causal pattern) --------
    if want("fwd_masked"):
        tril = torch.tril(torch.ones(N, N, dtype=torch.uint8, device=dev))

        def run_masked(_i=0):
            fa.fa_forward_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), tril.data_ptr(), 0, B, H, N, d, scale, sptr)
        if not need_main_inputs:
            raise SystemExit("fwd_masked needs the forward workload")
        rec = timer.run(run_masked, True, launches_per_call=3)
        launches += rec["launches"]
        times["fwd_masked"] = rec["ms"]
        legs["fwd_masked"] = rec
        del tril

    # ---- FP8: quantization, then the forward on resident E4M3 codes --------
    if want("fwd_fp8"):
        qq, kk, vv = (q, k, v) if need_main_inputs else fwd_inputs(FWD)
        x8 = fa.quantize_fp8(qq, kk, vv)
        o8 = torch.empty_like(qq)
        l8 = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        qws = torch.empty((max(fa.fa_quantize_fp8_workspace_bytes(B, H, N, d), 16),),
                          dtype=torch.uint8, device=dev)

        def run_fp8(_i=0):
            fa.fa_forward_fp8(x8.q8.data_ptr(), x8.k8.data_ptr(), x8.vt8.data_ptr(),
                              x8.q_scale.data_ptr(), x8.k_scale.data_ptr(), x8.v_scale.data_ptr(),
                              o8.data_ptr(), l8.data_ptr(), B, H, N, d, scale, causal, sptr)

        def run_quant(_i=0):
            fa.fa_quantize_fp8(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), None,
                               x8.q8.data_ptr(), x8.k8.data_ptr(), x8.vt8.data_ptr(),
                               x8.q_scale.data_ptr(), x8.k_scale.data_ptr(),
                               x8.v_scale.data_ptr(), B, H, N, d, qws.data_ptr(), qws.numel(),
                               sptr)
        rec = timer.run(run_fp8, True)
        recq = timer.run(run_quant, True, launches_per_call=2)
        # context for the quantization's rate: a plain device copy moving the
        # same number of bytes (half read, half written), timed the same way
        # (L2 flushed before each call, so both pay for its dirty lines)
        csrc = torch.empty((3 * B * H * N * d * 3) // 2, dtype=torch.uint8, device=dev)
        cdst = torch.empty_like(csrc)
        recc = timer.run(lambda _i=0: cdst.copy_(csrc), True, launches_per_call=0)
        del csrc, cdst
        launches += rec["launches"] + recq["launches"]
        times["fwd_fp8"], times["fp8_quant"] = rec["ms"], recq["ms"]
        times["copy_same_bytes"] = recc["ms"]
        legs["fwd_fp8"], legs["fp8_quant"] = rec, recq
        del x8, o8, l8, qws, qq, kk, vv

    # ---- backward, d = 128 and d = 64 ----------------------------------------
    def backward_leg(name, cfg):
        a, b_, c_ = fwd_inputs(cfg)
        Bb, Hb, Nb, db = cfg["B"], cfg["H"], cfg["N"], cfg["d"]
        g_out = inputs.grad_output(Bb, Hb, Nb, db, torch.bfloat16, seed=cfg["seed"] + seed_off)
        g_out = g_out.to(dev)
        oo = torch.empty_like(a)
        ll = torch.empty((Bb, Hb, Nb), dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            fa.fa_forward(a.data_ptr(), b_.data_ptr(), c_.data_ptr(), oo.data_ptr(),
                          ll.data_ptr(), Bb, Hb, Nb, db, db ** -0.5, cfg["causal"], sptr)
        gq, gk, gv = (torch.empty_like(a) for _ in range(3))
        nbytes = fa.fa_backward_workspace_bytes(Bb, Hb, Nb, db)
        bws = torch.empty((nbytes,), dtype=torch.uint8, device=dev)

        def run(_i=0):
            fa.fa_backward(a.data_ptr(), b_.data_ptr(), c_.data_ptr(), oo.data_ptr(),
                           g_out.data_ptr(), ll.data_ptr(), gq.data_ptr(), gk.data_ptr(),
                           gv.data_ptr(), Bb, Hb, Nb, db, db ** -0.5, cfg["causal"],
                           bws.data_ptr(), nbytes, sptr)
        rec = timer.run(run, True, launches_per_call=3)
        times[name] = rec["ms"]
        legs[name] = rec
        return rec

    if want("backward"):
        launches += backward_leg("backward", FWD)["launches"]
    if want("backward_d64"):
        launches += backward_leg("backward_d64", BWD_D64)["launches"]

    # ---- grouped-head decode (4 query heads per cached head) ---------------
    if want("decode_gqa"):
        fa.fa_decode_gqa_select(args.gqa_impl)
        dg = decode_workload(DEC_GQA, args.decode_seqs)
        Sg, Hg, Dg = dg.q.shape
        gqs = [dg.q] + [dg.q.clone() for _ in range(3)]
        gouts = [torch.empty_like(dg.q) for _ in range(4)]
        gqa_bytes = decode_bytes(dg)

        def run_gqa(i=0):
            fa.fa_paged_decode_gqa(gqs[i % 4].data_ptr(), dg.k_cache.data_ptr(),
                                   dg.v_cache.data_ptr(), dg.block_tables.data_ptr(),
                                   dg.context_lens.data_ptr(), gouts[i % 4].data_ptr(), Sg, Hg,
                                   dg.num_kv_heads, Dg, dg.block_size, dg.max_blocks, dg.scale,
                                   sptr)
        rec = timer.run(run_gqa, False, launches_per_call=1 if args.gqa_impl == 1 else 2)
        fa.fa_decode_gqa_select(0)
        launches += rec["launches"]
        times["decode_gqa"] = rec["ms"]
        legs["decode_gqa"] = rec
        del dg, gqs, gouts

    # ---- end to end, forward --------------------------------------------------
    if only is None:
        ho = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
        hl = [torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True) for _ in range(2)]
        dqkv = [[torch.empty_like(q) for _ in range(3)] for _ in range(2)]
        do_ = [torch.empty_like(o) for _ in range(2)]
        dl = [torch.empty_like(lse) for _ in range(2)]

        def fwd_h2d(sl):
            for dst, src in zip(dqkv[sl], (hq, hk, hv)):
                dst.copy_(src, non_blocking=True)

        def fwd_compute(sl):
            a, b_, c_ = dqkv[sl]
            fa.fa_forward(a.data_ptr(), b_.data_ptr(), c_.data_ptr(), do_[sl].data_ptr(),
                          dl[sl].data_ptr(), B, H, N, d, scale, causal, sptr)

        def fwd_d2h(sl):
            ho[sl].copy_(do_[sl], non_blocking=True)
            hl[sl].copy_(dl[sl], non_blocking=True)

        e2e_fwd_ms = pipeline(fwd_h2d, fwd_compute, fwd_d2h)
        launches += ke
        del dqkv, do_, dl
        e2e = {"fwd_ms": e2e_fwd_ms, "dec_ms": e2e_dec_ms,
               "h2d": 3 * q.numel() * 2 + dec_h2d_bytes,
               "d2h": o.numel() * 2 + lse.numel() * 4 + dec_d2h_bytes}

    torch.cuda.synchronize()
    clk = clocks.stop()
    status = fa.fa_device_status()

    # ---- the job's figures ------------------------------------------------------
    names = sorted(times)
    if ws > 1:
        extra = [main["fwd_mean"], main["dec_mean"], main["wall"]] if main else []
        if e2e:
            extra += [e2e["fwd_ms"], e2e["dec_ms"]]
        vals, status = reduce_over_ranks([times[n] for n in names] + extra, status, dev)
        for n, val in zip(names, vals):
            times[n] = val
        rest = vals[len(names):]
        if main:
            main["fwd_mean"], main["dec_mean"], main["wall"] = rest[:3]
            rest = rest[3:]
        if e2e:
            e2e["fwd_ms"], e2e["dec_ms"] = rest[:2]

    def leg_out(name, units, unit_scale, unit, peak, kind, bound, kernel, workload,
                traffic=None, extra=None):
        rec = legs[name]
        ms = times[name]
        value, roof = _rate_record(units, ms, ws, unit_scale, unit, peak, kind, bound, kernel,
                                   traffic)
        out = {"workload": workload, "value": value, "unit": unit, "ms": round(ms, 5),
               "p10_ms": rec["p10_ms"], "p90_ms": rec["p90_ms"], "calls": rec["calls"],
               "device_s": rec["device_s"], "roofline": roof}
        if extra:
            out.update(extra)
        return out

    res = {}
    if "fwd_f32" in legs:
        c = FWD_F32
        # fp32 FMA rate: SMs x 128 lanes x 2 FLOP x the maximum SM clock
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peak_f32 = round(sms * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12, 1)
        res["fwd_f32"] = leg_out("fwd_f32", fwd_flops(**c), 1e12, "TFLOP/s", peak_f32,
                                 "fp32 FMA rate from SM count and maximum clock", "alu",
                                 "fwd_f32_kernel<64>",
                                 "fa_forward_fp32 fp32 B=1 H=1 N=64 d=64 non-causal (timed in "
                                 "groups of launches: one launch is a few microseconds)",
                                 recorded_traffic("fwd_f32_kernel<64>"))
        res["fwd_f32"]["roofline"]["note"] = ("exact fp32 FMAs on the CUDA cores; one 64-row "
                                              "head is two small CTAs, so the figure is launch "
                                              "latency, not a use of the device")
    if "fwd_d64" in legs:
        res["fwd_d64"] = leg_out("fwd_d64", fwd_flops(**FWD_D64), 1e12, "TFLOP/s", peak_t,
                                 tensor_kind, "tensor", "fwd_bf16_tc_kernel<64>",
                                 "fa_forward bf16 B=4 H=16 N=1024 d=64 non-causal",
                                 recorded_traffic("fwd_bf16_tc_kernel<64>"))
    if "fwd" in legs:
        res["fwd"] = leg_out("fwd", flops, 1e12, "TFLOP/s", peak_t, tensor_kind, "tensor",
                             "fwd_bf16_tc_kernel<128>",
                             "fa_forward bf16 B=2 H=16 N=4096 d=128 causal",
                             recorded_traffic("fwd_bf16_tc_kernel<128>"))
    if "fwd_long" in legs:
        res["fwd_long"] = leg_out("fwd_long", fwd_flops(**FWD_LONG), 1e12, "TFLOP/s", peak_t,
                                  tensor_kind, "tensor", "fwd_bf16_tc_kernel<128>",
                                  "fa_forward bf16 B=1 H=8 N=16384 d=128 causal, inputs "
                                  "N(0,1)*0.5",
                                  recorded_traffic("fwd_bf16_tc_kernel<128> 1x8x16384"))
    if "decode" in legs:
        res["decode"] = leg_out("decode", dec_bytes, 1e9, "GB/s", peak_h, hbm_kind, "hbm",
                                "paged_decode_kernel",
                                f"fa_paged_decode bf16 {args.decode_seqs} seqs x 32 heads x head "
                                "128, block 16, ctx U[1,4096]; q and out rotated over 4 buffers",
                                recorded_traffic("paged_decode_kernel"),
                                {"bytes_per_launch": dec_bytes})
        fl = leg_out("decode_flushed", dec_bytes, 1e9, "GB/s", peak_h, hbm_kind, "hbm",
                     "paged_decode_kernel", "the same decode, each launch after a 512 MiB write")
        res["decode"]["after_l2_flush"] = {k_: fl[k_] for k_ in ("value", "ms", "p10_ms",
                                                                "p90_ms", "calls")}
        res["decode"]["after_l2_flush"]["frac"] = fl["roofline"]["frac"]
    if "fwd_f16" in legs:
        res["fwd_f16"] = leg_out("fwd_f16", flops, 1e12, "TFLOP/s", peak_t, tensor_kind,
                                 "tensor", "fwd_bf16_tc_kernel<128,1>",
                                 "fa_forward_f16 fp16 B=2 H=16 N=4096 d=128 causal (the forward's "
                                 "inputs rounded to fp16)")
    if "fwd_masked" in legs:
        res["fwd_masked"] = leg_out("fwd_masked", flops, 1e12, "TFLOP/s", peak_t, tensor_kind,
                                    "tensor", "mask summary (2 kernels) + "
                                    "fwd_bf16_tc_kernel<128,0,1,0>",
                                    "fa_forward_masked bf16 B=2 H=16 N=4096 d=128 with the [N,N] "
                                    "tril mask (FLOPs of the visible half; the mask's tile summary "
                                    "is inside the timed call)",
                                    recorded_traffic("fwd_bf16_tc_kernel<128,0,1,0>"))
    if "fwd_d256" in legs:
        res["fwd_d256"] = leg_out("fwd_d256", fwd_flops(**FWD_D256), 1e12, "TFLOP/s", peak_t,
                                  tensor_kind, "tensor", "fwd_d256_kernel<0>",
                                  "fa_forward bf16 B=2 H=8 N=4096 d=256 causal",
                                  recorded_traffic("fwd_d256_kernel<0>"))
    if "fwd_fp8" in legs:
        res["fwd_fp8"] = leg_out("fwd_fp8", flops, 1e12, "TFLOP/s", round(2 * peak_t, 1),
                                 f"{peak_kind} bf16 burst x 2 (nominal fp8/bf16 ratio)", "tensor",
                                 "fwd_bf16_tc_kernel<128,0,0,1> (E4M3)",
                                 "fa_forward_fp8 on the forward workload block-quantized to E4M3 "
                                 "(fa_quantize_fp8: 128-row blocks for Q and K, per-head V; no "
                                 "transform), bf16 output",
                                 recorded_traffic("fwd_bf16_tc_kernel<128,0,0,1>"))
        # algorithmic: each bf16 input read once, each E4M3 code written once
        quant_bytes = 3 * B * H * N * d * 3
        res["fwd_fp8"]["quantize"] = leg_out(
            "fp8_quant", quant_bytes, 1e9, "GB/s", peak_h, hbm_kind, "hbm",
            "fp8_quant_rows_kernel + fp8_quant_v_kernel",
            "fa_quantize_fp8 of the forward workload (algorithmic bytes: 2 B read + 1 B "
            "written per element of Q, K and V; the kernels read V twice)")
        res["fwd_fp8"]["quantize"]["same_bytes_copy"] = {
            "what": f"torch device copy of {quant_bytes / 2e6:.1f} MB ({quant_bytes / 1e6:.0f} MB "
                    "moved), timed like the quantization",
            "ms": times["copy_same_bytes"],
            "GB/s": round(quant_bytes / (times["copy_same_bytes"] * 1e-3) / 1e9, 1),
            "quantize_rate_over_copy_rate": round(times["copy_same_bytes"] / times["fp8_quant"], 3)}
        res["fwd_fp8"]["value_with_quantize"] = round(
            weak_scaling_rate(flops, ws, times["fwd_fp8"] + times["fp8_quant"], 1e12), 2)
    if "backward" in legs:
        bf = bwd_flops_of(**FWD)
        res["backward"] = leg_out("backward", bf, 1e12, "TFLOP/s", peak_t, tensor_kind, "tensor",
                                  "bwd_prep_kernel + bwd_pipe_kernel + bwd_dq_kernel",
                                  "fa_backward bf16 B=2 H=16 N=4096 d=128 causal (dQ, dK, dV of "
                                  "the forward workload, upstream gradient N(0,1))",
                                  recorded_traffic("bwd_pipe_kernel"),
                                  {"flops_per_launch": bf})
    if "backward_d64" in legs:
        bf = bwd_flops_of(**BWD_D64)
        res["backward_d64"] = leg_out("backward_d64", bf, 1e12, "TFLOP/s", peak_t, tensor_kind,
                                      "tensor", "bwd_prep_kernel + bwd_pipe64_kernel + "
                                      "bwd_dq_kernel",
                                      "fa_backward bf16 B=2 H=16 N=4096 d=64 causal",
                                      recorded_traffic("bwd_pipe64_kernel"),
                                      {"flops_per_launch": bf})
    if "decode_gqa" in legs:
        gk = ("paged_decode_gqa_kernel<4>" if args.gqa_impl == 1 else
              "paged_decode_gqa_tc_kernel<4> + paged_decode_merge_kernel")
        res["decode_gqa"] = leg_out("decode_gqa", gqa_bytes, 1e9, "GB/s", peak_h, hbm_kind,
                                    "hbm", gk,
                                    f"fa_paged_decode_gqa bf16 {args.decode_seqs} seqs x 32 query "
                                    "heads x 8 key/value heads x head 128, block 16, ctx "
                                    "U[1,4096]; q and out rotated over 4 buffers",
                                    recorded_traffic(gk.split(" ")[0]),
                                    {"bytes_per_launch": gqa_bytes})

    if only is not None:
        if ws > 1:
            dist.destroy_process_group()
        if rank != 0:
            return None
        return {"only": only, "n_gpus": ws, "clocks": clk, "device_status": status,
                "gpu_launches": launches, **res}

    # The K-step main loop: `value` and the dominant kernel's roofline.
    fwd_med, fwd_p10, fwd_p90 = main["fwd"]
    dec_med, dec_p10, dec_p90 = main["dec"]
    if ws > 1:
        fwd_med, dec_med = times["main_fwd"], times["main_dec"]
    tflops = weak_scaling_rate(flops, ws, fwd_med, 1e12)
    per_gpu_tflops = weak_scaling_rate(flops, 1, fwd_med, 1e12)
    per_gpu_gbs = weak_scaling_rate(dec_bytes, 1, dec_med, 1e9)

    def brief(name, key="value"):
        r = res[name]
        return {"value": r[key], "unit": r["unit"], "frac": r["roofline"]["frac"],
                "ms": r["ms"]}

    summary = {
        "c1 fp32 1x1x64x64": brief("fwd_f32"),
        "c2 bf16 4x16x1024x64": brief("fwd_d64"),
        "c3 bf16 2x16x4096x128 causal": {"value": round(tflops, 2), "unit": "TFLOP/s",
                                         "frac": round(per_gpu_tflops / peak_t, 4),
                                         "ms": round(fwd_med, 5), "of_1s_leg": brief("fwd")},
        "c4 bf16 1x8x16384x128 causal": brief("fwd_long"),
        "c5 decode 64x32x128": {"value": round(weak_scaling_rate(dec_bytes, ws, dec_med, 1e9), 1),
                                "unit": "GB/s", "frac": round(per_gpu_gbs / peak_h, 4),
                                "ms": round(dec_med, 5), "of_1s_leg": brief("decode")},
    }
    result = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "summary": summary,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(main["fwd_mean"] + main["dec_mean"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs; no dataset)",
        "roofline": {"bound": "tensor", "achieved": round(per_gpu_tflops, 2), "peak": peak_t,
                     "unit": "TFLOP/s", "frac": round(per_gpu_tflops / peak_t, 4),
                     "traffic": recorded_traffic("fwd_bf16_tc_kernel<128>"),
                     "peak_kind": tensor_kind, "kernel": "fwd_bf16_tc_kernel<128>",
                     "flops_per_launch": flops},
        "main_loop": {"fwd_ms_median": round(fwd_med, 5), "fwd_ms_p10": round(fwd_p10, 5),
                      "fwd_ms_p90": round(fwd_p90, 5), "fwd_ms_mean": round(main["fwd_mean"], 5),
                      "decode_ms_median": round(dec_med, 5), "decode_ms_p10": round(dec_p10, 5),
                      "decode_ms_p90": round(dec_p90, 5),
                      "decode_ms_mean": round(main["dec_mean"], 5)},
        "config": {
            "workload": "fa_forward bf16 B=2 H=16 N=4096 d=128 causal + fa_paged_decode bf16 "
                        "64 seqs x 32 heads x head 128, block 16, ctx U[1,4096]",
            "fwd": {k_: v_ for k_, v_ in FWD.items() if k_ != "seed"},
            "decode": {k_: v_ for k_, v_ in DEC.items() if k_ != "seed"},
            "decode_sum_ctx": dec_sum_ctx,
            "l2": "forwards, FP8 quantization and backwards: flushed (512 MiB write) before "
                  "every timed launch; decodes (2.2 GB and 0.55 GB read per launch): inputs "
                  "larger than L2, not flushed (q and out rotated), plus a flushed decode figure",
            "timing": f"main loop: exactly {args.steps} steps; other legs: at least "
                      f"{args.min_seconds} s of device time and {max(args.steps, 3)} launches "
                      "each, median/p10/p90 of per-launch CUDA-event times",
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "sms": torch.cuda.get_device_properties(dev).multi_processor_count,
            "input_sha256": hashes,
        },
        "decode": res["decode"],
        **{k_: res[k_] for k_ in ("fwd_f32", "fwd_d64", "fwd", "fwd_long", "fwd_f16",
                                   "fwd_masked", "fwd_d256", "fwd_fp8", "backward",
                                   "backward_d64", "decode_gqa")},
        "e2e": {"value": round(weak_scaling_rate(flops, ws, e2e["fwd_ms"], 1e12), 2),
                "unit": "TFLOP/s",
                "decode_gbs": round(weak_scaling_rate(dec_bytes, ws, e2e["dec_ms"], 1e9), 1),
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "note": "KV cache resident (serving state); q, K, V, q_decode, block table, "
                        "context lens copied in and O, LSE, out copied back every step; copies "
                        "in, compute and copies out on three streams over two device slots "
                        "(step i+1's inputs arrive while step i computes)"},
        "gpu_launches": launches,
        "clocks": clk,
        "device_status": status,
        "wall_s": round(main["wall"], 4),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if ws > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


# ---------------------------------------------------------------------------
# The float64 CPU oracle, timed on the host cores

class OracleSampler:
    """Times the float64 oracle on a forward workload (the 2 x 16 x 4096 x 128
    causal one by default), in units of 256 consecutive query rows of one
    head, visited in a fixed order, until a time budget is spent.  Inputs are
    drawn once, like the GPU arm's."""

    ROWS = 256

    def __init__(self, cfg=None, nthreads=0):
        import torch

        import oracle
        from exact_attention_11_gb300 import inputs
        oracle.build()
        self.oracle = oracle
        cfg = cfg or FWD
        B, H, N, d = cfg["B"], cfg["H"], cfg["N"], cfg["d"]
        q, k, v = inputs.forward_inputs(B, H, N, d, torch.bfloat16, seed=cfg["seed"],
                                        amp=cfg.get("amp", 1.0))
        self.q, self.k, self.v = (t.double().reshape(B * H, N, d).numpy() for t in (q, k, v))
        self.N, self.d, self.BH, self.causal = N, d, B * H, cfg["causal"]
        self.units = [(h, r0) for r0 in range(0, N, self.ROWS) for h in range(B * H)]
        self.next = 0
        self.nthreads = nthreads
        self.cores = nthreads or oracle.max_threads()

    def unit_flops(self, r0):
        r1 = min(self.N, r0 + self.ROWS)
        if not self.causal:
            return 4.0 * self.d * self.N * (r1 - r0)
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
                                               self.v[sl][None], rows, self.d ** -0.5,
                                               self.causal, self.nthreads)
            secs += time.perf_counter() - t0
            flops += self.unit_flops(r0)
            n += 1
        return flops, secs, n


def _time_full_forward(cfg, dtype_name="bf16"):
    """The oracle over a whole (small) forward workload, timed once."""
    import torch

    import oracle
    from exact_attention_11_gb300 import inputs
    dtype = torch.float32 if dtype_name == "fp32" else torch.bfloat16
    q, k, v = (t.double().numpy() for t in inputs.forward_inputs(
        cfg["B"], cfg["H"], cfg["N"], cfg["d"], dtype, seed=cfg["seed"]))
    t0 = time.perf_counter()
    oracle.attention_forward(q, k, v, cfg["d"] ** -0.5, cfg["causal"])
    secs = time.perf_counter() - t0
    return {"value": fwd_flops(**cfg) / secs / 1e12, "unit": "TFLOP/s", "s": round(secs, 4),
            "sample": "the whole workload"}


def _time_long_forward_extrapolated():
    """The 1 x 8 x 16384 x 128 causal forward: 256 seeded query rows of every
    head timed, the full pass extrapolated from the time per unit of work."""
    import numpy as np
    import torch

    import oracle
    from exact_attention_11_gb300 import inputs
    c = FWD_LONG
    q, k, v = (t.double().numpy() for t in inputs.forward_inputs(
        c["B"], c["H"], c["N"], c["d"], torch.bfloat16, seed=c["seed"], amp=c["amp"]))
    rows = inputs.sample_rows(c["N"], 256, seed=c["seed"] + 100).numpy()
    t0 = time.perf_counter()
    oracle.attention_forward_rows(q, k, v, rows, c["d"] ** -0.5, True)
    secs = time.perf_counter() - t0
    flops = 4.0 * c["d"] * float(np.sum(rows + 1)) * c["B"] * c["H"]
    rate = flops / secs
    return {"value": rate / 1e12, "unit": "TFLOP/s", "s": round(secs, 4),
            "full_pass_s_extrapolated": round(fwd_flops(**c) / rate, 2),
            "sample": "256 seeded query rows of each of the 8 heads; the full-pass time is "
                      "extrapolated (labelled), not measured"}


def _time_decode_sample(budget_s):
    """The decode oracle on 4 sequences drawn like the 64-sequence workload
    (same head count, block size and context distribution), on the host."""
    import torch

    import oracle
    from exact_attention_11_gb300 import inputs
    di = inputs.decode_inputs(4, DEC["num_heads"], DEC["head_size"], DEC["block_size"],
                              DEC["max_ctx"], seed=DEC["seed"], device="cpu")
    q, kc, vc = (t.double().numpy() for t in (di.q, di.k_cache, di.v_cache))
    bt, cl = di.block_tables.numpy(), di.context_lens.numpy()
    nbytes = di.kv_bytes_read()
    secs, n = 0.0, 0
    while n == 0 or secs < budget_s:
        t0 = time.perf_counter()
        oracle.paged_decode(q, kc, vc, bt, cl, di.scale)
        secs += time.perf_counter() - t0
        n += 1
    return {"value": n * nbytes / secs / 1e9, "unit": "GB/s", "s": round(secs, 3),
            "sample": f"{n} passes over 4 sequences x 32 heads (sum of contexts "
                      f"{int(torch.as_tensor(cl).sum())}) drawn like the 64-sequence workload; "
                      "bytes = the K/V bytes the GPU decode counts"}


def cpu_baseline(target_s: float):
    smp = OracleSampler()
    flops, secs, n = smp.run(target_s * 0.5)
    one = OracleSampler(nthreads=1)
    f1, s1, n1 = one.run(target_s * 0.2)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": smp.cores, "kind": "oracle",
            "sample": f"{n} blocks of 256 causal query rows (of the 512 blocks of the "
                      f"2x16x4096x128 forward), float64, {secs:.1f} s",
            "one_thread": {"value": f1 / s1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                           "sample": f"{n1} blocks of 256 rows, {s1:.1f} s"},
            "configs": {"c1 fp32 1x1x64x64": _time_full_forward(FWD_F32, "fp32"),
                        "c2 bf16 4x16x1024x64": _time_full_forward(FWD_D64),
                        "c4 bf16 1x8x16384x128 causal": _time_long_forward_extrapolated(),
                        "c5 decode": _time_decode_sample(target_s * 0.25)}}


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
    ap.add_argument("--cpu-seconds", type=float, default=16.0,
                    help="approximate CPU time for the oracle baseline samples")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-hash", action="store_true", help="skip the inputs' sha256")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="device time each secondary leg runs for (0: just --steps launches)")
    ap.add_argument("--only", default="",
                    help=f"comma-separated legs to run alone ({', '.join(LEGS)})")
    ap.add_argument("--decode-seqs", type=int, default=DEC["num_seqs"],
                    help="sequences of the decode workloads (smaller for profiling)")
    ap.add_argument("--gqa-impl", type=int, default=0, choices=[0, 1, 2],
                    help="grouped-decode kernel (fa_decode_gqa_select): 0 automatic, 1 CUDA "
                         "cores, 2 tensor cores")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        ap.error("--warmup must be >= 3")
    res = reference_arm(args) if args.impl == "reference" else gpu_arm(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
