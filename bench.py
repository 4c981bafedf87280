"""Benchmark of the masked / biased attention hot path on GB300.

One step = block classification + forward (O, lse) + backward (dQ, dK, dV,
dBias) of one batch of a synthetic workload; by default the N=16384 workload
(B=1, Hq=16, Hkv=4, d=128, causal, per-row top-2048 mask built from an N(0,1)
bias).  The metric is effective fwd+bwd TFLOP/s counted over non-skipped
128x128 tiles: (4 + 10) * d * 128^2 * (active tiles) * (Hq / Hkv) per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME]

--workload selects one of the other measured problems (n4096_hq32_hkv8,
n65536_hq16_hkv2, docmask_b2_n32768: the FlashMask causal document mask given as
column ranges, no bias).  With N > 1 (torchrun, one process per GPU) every rank
runs its own copy of the workload (weak scaling, no collective on the data path)
and rank 0 prints the aggregate.  --impl reference times the fp64 CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "n16384_hq16_hkv4"
BENCH_WORKLOADS = ("n16384_hq16_hkv4", "n4096_hq32_hkv8", "n65536_hq16_hkv2", "docmask_b2_n32768")
METRIC = "effective fwd+bwd TFLOP/s (non-skipped tiles) and % of roofline, 1 GB300"
TILE = 128
KERNELS_PER_STEP = 5  # classify, fwd, bwd_pre, bwd, dq_convert
# DRAM bytes (read + write) of one bwd_kernel launch, per workload, from an ncu capture of
# the current kernel; a workload without an entry reports null.  n16384_hq16_hkv4: one kv
# group of the workload (Hq=4, Hkv=1) is captured; the four kv groups are independent CTAs
# with the same work, so the full launch moves 4x that: 373,442,048 read and 533,421,056
# written per kv group.
BWD_TRAFFIC_BYTES = {"n16384_hq16_hkv4": 4 * (373199104 + 532822272)}
E2E_MAX_HOST_BYTES = 24e9  # larger workloads report no end-to-end number (pinned host copies)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe is None:
            return self
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        self.fh = open(self.path, "w")
        self.proc = subprocess.Popen([exe, "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                                     stderr=subprocess.DEVNULL)
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def replica_seed(base_seed: int, rank: int) -> int:
    """Each replica draws its own copy of the workload (weak scaling)."""
    return base_seed + rank


def max_over_ranks(values, dist=None, device=None):
    """Element-wise max of per-rank timings (the slowest rank sets the time)."""
    import torch

    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Aggregate throughput: the units all ranks processed / the (max) step time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def algorithmic_bytes(wl, bm):
    """Minimum bytes the path must move (a dense mask once over causally allowed
    tiles, or the column ranges once; bias in fwd and bwd over active tiles; dBias
    over all of N^2; Q K V O dO dQ dK dV and lse once each)."""
    tile_elems = TILE * TILE
    nq_t, nk_t = bm.shape[2], bm.shape[3]
    active = int((bm != 0).sum())
    if wl.mask_kind == "dense":
        causal_tiles = sum(1 for qt in range(nq_t) for kt in range(nk_t) if kt <= qt) * wl.B * wl.Hkv
        mask_b = causal_tiles * tile_elems * 2
    elif wl.mask_kind == "colranges":
        mask_b = wl.B * wl.Hkv * wl.Nk * 2 * 4
    else:
        mask_b = 0
    has_bias = wl.has_bias or wl.mask_kind == "dense"
    bias_b = 2 * active * tile_elems * 2 if has_bias else 0
    dbias_b = wl.B * wl.Hkv * wl.Nq * wl.Nk * 2 if has_bias else 0
    io = 2 * (4 * wl.B * wl.Nq * wl.Hq * wl.d + 4 * wl.B * wl.Nk * wl.Hkv * wl.d) + 4 * wl.B * wl.Hq * wl.Nq
    return {"mask": mask_b, "bias": bias_b, "dbias": dbias_b, "io": io, "total": mask_b + bias_b + dbias_b + io,
            "bwd_kernel": bias_b // 2 + dbias_b + 2 * (3 * wl.B * wl.Nq * wl.Hq * wl.d +
                                                       2 * wl.B * wl.Nk * wl.Hkv * wl.d)}


def select_peak(peaks, clocks):
    """The bf16 peak a kernel is held against: the burst figure (a cuBLAS GEMM timed
    alone, at full clock) unless this run's own clock samples saw the power cap, in
    which case the sustained figure (the same GEMM in a seconds-long loop)."""
    if "sw_power_cap" in (clocks.get("reasons") or []):
        return peaks["bf16_tflops_sustained"], peaks["source"] + " bf16_tflops_sustained (sw_power_cap seen in this run)"
    return peaks["bf16_tflops"], peaks["source"] + " bf16_tflops (burst; no power cap seen in this run)"


def run_gpu(args):
    import torch

    from block_sparse_masked_02_gb300 import fdma, workloads as W

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    fdma.load()
    wl = W.WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    inp = W.make_inputs(wl, device=dev, seed=replica_seed(wl.seed, rank))
    q, k, v, do = (inp[n] for n in ("q", "k", "v", "dout"))
    bias, mask, cr = inp["bias"], inp["mask"], inp["colranges"]
    kw = dict(mask=mask, colranges=cr, bias=bias, causal=wl.causal, scale=wl.scale)
    a = fdma.make_args(q, k, v, **kw)
    wsp = fdma.alloc_workspace(a, True, dev)
    bm = fdma.classify_blocks(q, k, v, mask=mask, colranges=cr, causal=wl.causal, workspace=wsp)
    active = int((bm != 0).sum().item())
    partial = int((bm == 1).sum().item())
    full = int((bm == 2).sum().item())
    flops_fwd = 4.0 * wl.d * TILE * TILE * active * wl.G
    flops_bwd = 10.0 * wl.d * TILE * TILE * active * wl.G
    flops = flops_fwd + flops_bwd
    out = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.Hq, wl.Nq), dtype=torch.float32, device=dev)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
             torch.empty_like(bias) if bias is not None else None)
    stream = torch.cuda.current_stream()
    R = fdma.FDMA_FLAG_REUSE_CLASSIFICATION

    def step():
        fdma.classify_blocks(q, k, v, mask=mask, colranges=cr, causal=wl.causal, workspace=wsp)
        fdma.fwd(q, k, v, workspace=wsp, flags=R, out=out, lse=lse, **kw)
        fdma.bwd(q, k, v, out, do, lse, workspace=wsp, flags=R, grads=grads, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fdma.device_error() != 0:
        raise RuntimeError("kernel-side error during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local] if ws > 1 else \
        os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(args.steps):
            e = ev[i]
            e[0].record(stream)
            fdma.classify_blocks(q, k, v, mask=mask, colranges=cr, causal=wl.causal, workspace=wsp)
            e[1].record(stream)
            fdma.fwd(q, k, v, workspace=wsp, flags=R, out=out, lse=lse, **kw)
            e[2].record(stream)
            fdma.bwd(q, k, v, out, do, lse, workspace=wsp, flags=R, grads=grads, **kw)
            e[3].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ms_total = t0.elapsed_time(t1)
    ms_cls = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    ms_fwd = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    ms_bwd = sum(e[2].elapsed_time(e[3]) for e in ev) / args.steps
    err = fdma.device_error()

    # ---- end to end: pinned host inputs in, results out, through the same C-ABI calls.  Every
    # step copies its own inputs in and its results out; the copies are pipelined across steps
    # (two device slots; host->device on one stream, device->host on another), so step i+1's
    # inputs arrive and step i-1's results leave while step i computes.
    names_in = [n for n in ("q", "k", "v", "dout", "mask", "colranges", "bias") if inp[n] is not None]
    dev_out = [t for t in (out, lse, *grads) if t is not None]
    h2d = sum(inp[n].numel() * inp[n].element_size() for n in names_in)
    d2h = sum(t.numel() * t.element_size() for t in dev_out)
    e2e = None
    if h2d + d2h <= E2E_MAX_HOST_BYTES:
        host_in = {n: inp[n].cpu().pin_memory() for n in names_in}
        slots = 2
        dev_in = [{n: torch.empty_like(inp[n]) for n in host_in} for _ in range(slots)]
        dev_res = [(torch.empty_like(out), torch.empty_like(lse), tuple(None if g is None else torch.empty_like(g)
                                                                         for g in grads)) for _ in range(slots)]
        host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_out] for _ in range(slots)]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(slots)]
        ev_done = [torch.cuda.Event() for _ in range(slots)]
        ev_out = [torch.cuda.Event() for _ in range(slots)]
        e2e_steps = max(2, min(args.steps, 6))

        def e2e_step(i):
            sl = i % slots
            din, (o_, l_, g_), hout = dev_in[sl], dev_res[sl], host_out[sl]
            with torch.cuda.stream(s_in):
                if i >= slots:
                    s_in.wait_event(ev_done[sl])  # step i-2's compute has finished with this slot
                for n, t in host_in.items():
                    din[n].copy_(t, non_blocking=True)
                ev_in[sl].record(s_in)
            stream.wait_event(ev_in[sl])
            if i >= slots:
                stream.wait_event(ev_out[sl])  # step i-2's results have been copied out
            ekw = dict(mask=din.get("mask"), colranges=din.get("colranges"), bias=din.get("bias"),
                       causal=wl.causal, scale=wl.scale)
            fdma.classify_blocks(din["q"], din["k"], din["v"], mask=ekw["mask"], colranges=ekw["colranges"],
                                 causal=wl.causal, workspace=wsp, stream=stream)
            fdma.fwd(din["q"], din["k"], din["v"], workspace=wsp, flags=R, out=o_, lse=l_, stream=stream, **ekw)
            fdma.bwd(din["q"], din["k"], din["v"], o_, din["dout"], l_, workspace=wsp, flags=R, grads=g_,
                     stream=stream, **ekw)
            ev_done[sl].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[sl])
                for h, d in zip(hout, [t for t in (o_, l_, *g_) if t is not None]):
                    h.copy_(d, non_blocking=True)
                ev_out[sl].record(s_out)

        for i in range(slots):
            e2e_step(i)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        s_in.wait_event(s0)
        for i in range(e2e_steps):
            e2e_step(i)
        for ev in ev_out:
            stream.wait_event(ev)  # every step's results are on the host
        s1.record(stream)
        torch.cuda.synchronize()
        e2e = s0.elapsed_time(s1) / e2e_steps
        assert fdma.device_error() == 0
    ms_e2e = e2e if e2e is not None else -1.0

    ms_total, ms_e2e, ms_bwd, ms_fwd, ms_cls = max_over_ranks([ms_total, ms_e2e, ms_bwd, ms_fwd, ms_cls], dist, dev)
    if rank != 0:
        dist.destroy_process_group()
        return None

    peaks = _peaks()
    clocks = clk.summary()
    peak, peak_source = select_peak(peaks, clocks)
    ms_step = ms_total / args.steps
    value = whole_job_tflops(flops, ws, ms_step)
    bw = algorithmic_bytes(wl, bm.cpu().numpy())
    roof_ms = max(flops / (peak * 1e12), bw["total"] / (peaks["hbm_gbs"] * 1e9)) * 1e3
    bwd_achieved = flops_bwd / (ms_bwd * 1e-3) / 1e12
    traffic = BWD_TRAFFIC_BYTES.get(args.workload)
    if wl.mask_kind == "dense":
        mask_desc = f"causal and per-row top-{wl.keep_window} of an N(0,1) bias"
    else:
        mask_desc = f"causal document mask as column ranges, document lengths U[{wl.doc_lo},{wl.doc_hi}], no bias"
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": wl.B, "N": wl.Nq, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                   "mask": mask_desc, "dbias": bias is not None,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "inputs larger than L2" if bw["total"] > 2 * 129e6 else "inputs may fit in L2",
                   "tiles": {"active": active, "partial": partial, "full": full, "total": int(bm.numel()),
                             "skip_ratio": round(1 - active / bm.numel(), 4)}},
        "pct_of_roofline": round(100.0 * roof_ms / ms_step, 2),
        "roofline_ms": round(roof_ms, 4),
        "breakdown_ms": {"classify": round(ms_cls, 4), "fwd": round(ms_fwd, 4), "bwd": round(ms_bwd, 4)},
        "phase_tflops": {"fwd": round(flops_fwd / (ms_fwd * 1e-3) / 1e12, 2), "bwd": round(bwd_achieved, 2)},
        "roofline": {"kernel": "bwd (fdma_bwd: bwd_pre + bwd_kernel + dq_convert)", "bound": "tensor",
                     "achieved": round(bwd_achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "peak_source": peak_source, "frac": round(bwd_achieved / peak, 4),
                     "traffic": traffic,
                     "traffic_note": ("ncu dram bytes of one bwd_kernel launch (profiles/)" if traffic is not None
                                      else "null: no ncu capture of the current bwd_kernel on this workload")},
        "e2e": ({"value": round(whole_job_tflops(flops, ws, ms_e2e), 3), "unit": "TFLOP/s",
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 3),
                 "copies": "pinned host buffers; each step's copies in and out, pipelined across steps (two "
                           "device slots: step i+1's host->device and step i-1's device->host copies overlap "
                           "step i's compute)"}
                if e2e is not None else
                {"value": None, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                 "note": "not measured: pinned host copies of this workload exceed the bench's host budget"}),
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clocks,
        "device_error": err,
    }
    if not args.no_cpu_baseline:
        prob, r0 = _cpu_problem(inp, wl, tiles=64)
        line["cpu_baseline"] = cpu_baseline(prob, wl, r0, seconds=args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    return line


class _RowWindow:
    """Host copy of rows [r0, r0 + R) of (batch 0, kv head 0) of a (B,Hkv,Nq,Nk)
    tensor; the oracle only indexes inside that window."""

    def __init__(self, rows, r0, shape):
        self.shape = tuple(shape)
        self.r0 = r0
        self.data = rows

    def __getitem__(self, idx):
        b, g, rs, cs = idx
        assert b == 0 and g == 0 and rs.start >= self.r0
        return self.data[rs.start - self.r0:rs.stop - self.r0, cs]


def cpu_baseline(prob, wl, r0, seconds=15.0, max_tiles=None):
    """Times the fp64 oracle (as written, no tuning) on whole 128-row query tiles of
    (batch 0, kv group 0), all its query heads, last (longest causal) tiles first, down
    to row r0, until about `seconds` of CPU time or `max_tiles`.  The forward (O and lse
    of every head) and the backward (which recomputes them, as the kernels do) are timed
    separately; the rate counts the sample's non-skipped tiles exactly like the GPU metric."""
    from oracle import attention as orc

    nqt = -(-wl.Nq // TILE)
    nkt = -(-wl.Nk // TILE)
    done = active = 0
    t_fwd = t_bwd = 0.0
    qt = nqt - 1
    while qt >= 0 and qt * TILE >= r0 and (t_fwd + t_bwd < seconds or done == 0):
        if max_tiles is not None and done >= max_tiles:
            break
        q0, q1 = qt * TILE, min((qt + 1) * TILE, wl.Nq)
        t0 = time.perf_counter()
        kv = orc._kv(prob, 0, 0)
        keep = orc.keep_rows(prob, 0, 0, q0, q1)
        for h in range(wl.G):
            orc.forward_rows(prob, 0, h, q0, q1, kv, keep)
        t1 = time.perf_counter()
        orc.backward_rows(prob, 0, 0, q0, q1, kv, keep)
        t2 = time.perf_counter()
        t_fwd += t1 - t0
        t_bwd += t2 - t1
        active += sum(int(keep[:, kt * TILE:(kt + 1) * TILE].any()) for kt in range(nkt))
        done += 1
        qt -= 1
    units = TILE * TILE * active * wl.G * wl.d
    t_used = t_fwd + t_bwd
    return {"value": round(14.0 * units / t_used / 1e12, 6), "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"{done} query tile(s) x {wl.G} heads of kv group 0 ({active} active tiles), fwd+bwd, "
                      f"{t_used:.2f} s; numpy float64 (BLAS threads = host cores)",
            "seconds": round(t_used, 3), "fwd_seconds": round(t_fwd, 3), "bwd_seconds": round(t_bwd, 3),
            "fwd_tflops": round(4.0 * units / t_fwd / 1e12, 6), "bwd_tflops": round(10.0 * units / t_bwd / 1e12, 6)}


def _cpu_problem(inp, wl, tiles):
    """The oracle's view of the GPU inputs for the last `tiles` query tiles of (batch 0,
    kv group 0): host copies of Q, K, V, dO and only those rows of the bias and mask."""
    from oracle import attention as orc

    r0 = max(0, wl.Nq - tiles * TILE)
    host = {n: inp[n].cpu() for n in ("q", "k", "v", "dout")}
    bw = mw = cr = None
    if inp["bias"] is not None:
        bw = _RowWindow(inp["bias"][0, 0, r0:].cpu(), r0, inp["bias"].shape)
    if inp["mask"] is not None:
        mw = _RowWindow(inp["mask"][0, 0, r0:].cpu(), r0, inp["mask"].shape)
    if inp["colranges"] is not None:
        cr = inp["colranges"].cpu()
    prob = orc.Problem(host["q"], host["k"], host["v"], bias=bw, mask=mw, colranges=cr, causal=wl.causal,
                       scale=wl.scale, dout=host["dout"])
    return prob, r0


def _host_problem(wl, tiles):
    """The workload's recipe drawn on the host for the sampled rows only: Q, K, V, dO,
    the column ranges, and the last `tiles` query tiles of kv group 0's bias / mask."""
    import torch

    from block_sparse_masked_02_gb300 import workloads as W
    from oracle import attention as orc

    if wl.mask_kind != "dense":
        inp = W.make_inputs(wl, device="cpu")
        return _cpu_problem(inp, wl, tiles)
    g = torch.Generator().manual_seed(wl.seed)
    host = {
        "q": torch.randn((wl.B, wl.Nq, wl.Hq, wl.d), generator=g).to(torch.bfloat16),
        "k": torch.randn((wl.B, wl.Nk, wl.Hkv, wl.d), generator=g).to(torch.bfloat16),
        "v": torch.randn((wl.B, wl.Nk, wl.Hkv, wl.d), generator=g).to(torch.bfloat16),
        "dout": torch.randn((wl.B, wl.Nq, wl.Hq, wl.d), generator=g).to(torch.bfloat16),
    }
    r0 = max(0, wl.Nq - tiles * TILE)
    bias = torch.randn((1, 1, wl.Nq - r0, wl.Nk), generator=g).to(torch.bfloat16)
    mask = W.topk_mask_from_bias(bias, wl.keep_window)
    bias.masked_fill_(mask == 0, W.BF16_MIN)
    shape = (wl.B, wl.Hkv, wl.Nq, wl.Nk)
    prob = orc.Problem(host["q"], host["k"], host["v"], bias=_RowWindow(bias[0, 0], r0, shape),
                       mask=_RowWindow(mask[0, 0], r0, shape), causal=wl.causal, scale=wl.scale, dout=host["dout"])
    return prob, r0


def run_reference(args):
    """--impl reference: the fp64 CPU oracle, as written, is the reference arm."""
    ws, rank, _ = _dist()
    if rank != 0:
        return None
    from block_sparse_masked_02_gb300 import workloads as W

    wl = W.WORKLOADS[args.workload]
    prob, r0 = _host_problem(wl, tiles=1)
    for _ in range(args.warmup):
        cpu_baseline(prob, wl, r0, seconds=0.0, max_tiles=1)
    rates, secs, fwd_s, bwd_s = [], [], [], []
    for _ in range(args.steps):
        r = cpu_baseline(prob, wl, r0, seconds=0.0, max_tiles=1)
        rates.append(r["value"])
        secs.append(r["seconds"])
        fwd_s.append(r["fwd_seconds"])
        bwd_s.append(r["bwd_seconds"])
    value = statistics.median(rates)
    ms_step = 1e3 * statistics.median(secs)
    if wl.mask_kind == "dense":
        mask_desc = f"causal and per-row top-{wl.keep_window} of an N(0,1) bias"
    else:
        mask_desc = f"causal document mask as column ranges, document lengths U[{wl.doc_lo},{wl.doc_hi}], no bias"
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": args.workload, "B": wl.B, "N": wl.Nq, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                   "mask": mask_desc, "dbias": wl.has_bias or wl.mask_kind == "dense"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                         "sample": f"each step: the last query tile x {wl.G} heads of kv group 0 (fwd+bwd), "
                                   "rows drawn on the host with the workload's recipe",
                         "fwd_seconds": round(statistics.median(fwd_s), 3),
                         "bwd_seconds": round(statistics.median(bwd_s), 3)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=BENCH_WORKLOADS)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
