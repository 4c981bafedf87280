"""Runs one named workload through the library once (classify, forward and
optionally backward) on cuda:0: the command to put under a profiler.

    python -m block_sparse_masked_02_gb300.run_case --workload n4096_hq32_hkv8 [--fwd-only] [--repeat R]
        [--Hq H --Hkv G] [--d D --dv DV] [--time]

--Hq / --Hkv run the named workload with fewer heads (the same recipe and sizes
otherwise), e.g. one kv group of a problem too large to capture whole.  --d / --dv
change the head dims (q/k and v), e.g. --d 256 or --d 192 --dv 128.  --time reports
the median forward and backward call times (CUDA events, after two untimed calls) and
their effective TFLOP/s over the active tiles: 2 * 128^2 * (d + dv) flops per active
(tile, query head) forward, 2 * 128^2 * (3d + 2dv) backward (S, dP, dV, dQ, dK).
"""
import argparse
import statistics

import torch

from . import fdma, workloads as W


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="n4096_hq32_hkv8", choices=sorted(W.WORKLOADS))
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--repeat", type=int, default=1)
    ap.add_argument("--Hq", type=int, default=0)
    ap.add_argument("--Hkv", type=int, default=0)
    ap.add_argument("--d", type=int, default=0)
    ap.add_argument("--dv", type=int, default=0)
    ap.add_argument("--time", action="store_true")
    a = ap.parse_args()
    fdma.load()
    wl = W.WORKLOADS[a.workload]
    if a.Hq or a.Hkv:
        wl = W.scaled(wl, Hq=a.Hq or wl.Hq, Hkv=a.Hkv or wl.Hkv)
    if a.d:
        wl = W.scaled(wl, d=a.d, scale=a.d ** -0.5)
    dv = a.dv or wl.d
    t = W.make_inputs(wl, device="cuda")
    if dv != wl.d:
        g = torch.Generator(device="cuda").manual_seed(wl.seed + 7)
        t["v"] = torch.randn(wl.B, wl.Nk, wl.Hkv, dv, generator=g, device="cuda").bfloat16()
        t["dout"] = torch.randn(wl.B, wl.Nq, wl.Hq, dv, generator=g, device="cuda").bfloat16()
    kw = dict(mask=t["mask"], colranges=t["colranges"], bias=t["bias"], causal=wl.causal, scale=wl.scale)
    tf, tb = [], []
    for it in range(a.repeat + (2 if a.time else 0)):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        out, lse = fdma.fwd(t["q"], t["k"], t["v"], **kw)
        e[1].record()
        if not a.fwd_only:
            fdma.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, **kw)
        e[2].record()
        if a.time and it >= 2:
            torch.cuda.synchronize()
            tf.append(e[0].elapsed_time(e[1]))
            tb.append(e[1].elapsed_time(e[2]))
    torch.cuda.synchronize()
    err = fdma.device_error()
    msg = f"{a.workload} d={wl.d} dv={dv}: done, device error {err}"
    if a.time and tf:
        bm = fdma.classify_blocks(t["q"], t["k"], t["v"], mask=t["mask"], colranges=t["colranges"],
                                  causal=wl.causal)
        units = int((bm != 0).sum().item()) * wl.G  # active (tile, query head) pairs
        ff = 2 * 128 * 128 * (wl.d + dv) * units
        fb = 2 * 128 * 128 * (3 * wl.d + 2 * dv) * units
        mf, mb = statistics.median(tf), statistics.median(tb)
        msg += f"; fwd {mf:.3f} ms ({ff / mf / 1e9:.1f} TFLOP/s)"
        if not a.fwd_only:
            msg += f", bwd {mb:.3f} ms ({fb / mb / 1e9:.1f} TFLOP/s)"
    print(msg)
    raise SystemExit(1 if err else 0)


if __name__ == "__main__":
    main()
