"""Runs one named workload through the library once (classify, forward and
optionally backward) on cuda:0: the command to put under a profiler.

    python -m block_sparse_masked_02_gb300.run_case --workload n4096_hq32_hkv8 [--fwd-only] [--repeat R]
        [--Hq H --Hkv G]

--Hq / --Hkv run the named workload with fewer heads (the same recipe and sizes
otherwise), e.g. one kv group of a problem too large to capture whole.
"""
import argparse

import torch

from . import fdma, workloads as W


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="n4096_hq32_hkv8", choices=sorted(W.WORKLOADS))
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--repeat", type=int, default=1)
    ap.add_argument("--Hq", type=int, default=0)
    ap.add_argument("--Hkv", type=int, default=0)
    a = ap.parse_args()
    fdma.load()
    wl = W.WORKLOADS[a.workload]
    if a.Hq or a.Hkv:
        wl = W.scaled(wl, Hq=a.Hq or wl.Hq, Hkv=a.Hkv or wl.Hkv)
    t = W.make_inputs(wl, device="cuda")
    kw = dict(mask=t["mask"], colranges=t["colranges"], bias=t["bias"], causal=wl.causal, scale=wl.scale)
    for _ in range(a.repeat):
        out, lse = fdma.fwd(t["q"], t["k"], t["v"], **kw)
        if not a.fwd_only:
            fdma.bwd(t["q"], t["k"], t["v"], out, t["dout"], lse, **kw)
    torch.cuda.synchronize()
    err = fdma.device_error()
    print(f"{a.workload}: done, device error {err}")
    raise SystemExit(1 if err else 0)


if __name__ == "__main__":
    main()
