"""Context-parallel split on one GPU: every rank of a planned split is run in turn through the
library (its runs of query rows against the keys it would receive, with the causal row offset
of fdma_args.is_causal = 2), the exchange done by indexing.  Key tiles a rank does not need are
zero in its K/V, so a read of one would show.  Put together, the ranks' O, lse and dBias equal
the unsplit call's bit for bit (the same tiles in the same order), and O, dQ, dK, dV and dBias
match the oracle of the unsplit problem (FlashMask README, "CPB" and "Overlap")."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as orc
from block_sparse_masked_02_gb300 import cp
from block_sparse_masked_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAXABS, O_RELL2, G_RELL2 = 1e-2, 5e-3, 1e-2


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_masked_02_gb300 import fdma

    fdma.load()
    return fdma


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300)


def _c(t):
    return None if t is None else t.cuda()


@pytest.mark.parametrize("case", ["topk_bias_d128", "topk_bias_d64", "docmask_d128"])
@pytest.mark.parametrize("world", [2, 3])
def test_split_equals_unsplit(F, case, world):
    N = 10 * cp.TILE + 72  # a ragged last tile
    if case.startswith("topk"):
        d = 128 if case.endswith("128") else 64
        wl = W.scaled(W.WORKLOADS["n4096_hq32_hkv8"], Nq=N, Nk=N, Hq=4, Hkv=2, d=d, keep_window=300,
                      scale=1 / math.sqrt(d), seed=500 + d + world)
    else:
        wl = W.Workload("doc_cp", 1, N, N, 4, 2, 128, True, 1 / math.sqrt(128), "colranges", 0, False,
                        doc_lo=150, doc_hi=500, seed=600 + world)
    inp = W.make_inputs(wl)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "dout"))
    mask, cr, bias = _c(inp.get("mask")), _c(inp.get("colranges")), _c(inp.get("bias"))
    kw = dict(mask=mask, colranges=cr, bias=bias, scale=wl.scale)
    out_f, lse_f = F.fwd(q, k, v, causal=True, **kw)
    dq_f, dk_f, dv_f, db_f = F.bwd(q, k, v, out_f, do, lse_f, causal=True, **kw)
    bm = F.classify_blocks(q, k, v, mask=mask, colranges=cr, causal=True)
    plan = cp.balance(cp.tile_work(bm), world)
    assert plan.loads.max() <= plan.loads.sum() / world + cp.tile_work(bm).max()

    out = torch.zeros_like(out_f)
    lse = torch.full_like(lse_f, float("nan"))
    dq = torch.zeros_like(dq_f)
    db = None if db_f is None else torch.zeros_like(db_f)
    dk = torch.zeros(k.shape, dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    for rank in range(world):
        own = plan.tiles_of(rank)
        need = cp.needed_key_tiles(bm[:, :, own, :])
        # the K/V this rank would hold after the gather: needed (or own) tiles only
        kr, vr = torch.zeros_like(k), torch.zeros_like(v)
        for t in range(len(need)):
            if need[t] or t in own:
                sl = slice(t * cp.TILE, (t + 1) * cp.TILE)
                kr[:, sl], vr[:, sl] = k[:, sl], v[:, sl]
        runs = plan.runs_of(rank)
        fw = cp.forward_runs(F, runs, q=q, k=kr, v=vr, mask=mask, colranges=cr, bias=bias, scale=wl.scale)
        per_run, dkp, dvp = cp.backward_runs(F, runs, fw, q=q, k=kr, v=vr, dout=do, mask=mask, colranges=cr,
                                             bias=bias, scale=wl.scale)
        for (r0, r1, o, l), (_, _, dqr, dbr) in zip(fw, per_run):
            out[:, r0:r1] = o
            lse[:, :, r0:r1] = l
            dq[:, r0:r1] = dqr
            if db is not None:
                db[:, :, r0:r1] = dbr
        dk += dkp
        dv += dvp
    assert F.device_error() == 0
    assert torch.equal(out, out_f)
    assert torch.equal(lse.isneginf(), lse_f.isneginf())
    fin = torch.isfinite(lse_f)
    assert torch.equal(lse[fin], lse_f[fin])
    if db is not None:
        assert torch.equal(db, db_f)
    p = orc.Problem(inp["q"], inp["k"], inp["v"], bias=inp.get("bias"), mask=inp.get("mask"),
                    colranges=inp.get("colranges"), causal=True, scale=wl.scale, dout=inp["dout"])
    O, _ = orc.forward(p)
    rq, rk, rv, rb = orc.backward(p, want_dbias=db is not None)
    o = out.float().cpu().numpy()
    assert np.abs(o - O).max() <= O_MAXABS and rel_l2(o, O) <= O_RELL2
    for x, ref in ((dq, rq), (dk, rk), (dv, rv)) + (((db, rb),) if db is not None else ()):
        assert rel_l2(x.float().cpu().numpy(), ref) <= G_RELL2


def test_causal_offset_rows_see_the_global_keys(F):
    """is_causal = 2: rows [r0, r1) of a causal problem with q_offset = r0, alone, give the
    unsplit call's rows bit for bit (forward and the tile classes)."""
    N = 6 * cp.TILE
    wl = W.scaled(W.WORKLOADS["n4096_hq32_hkv8"], Nq=N, Nk=N, Hq=2, Hkv=1, d=64, keep_window=200,
                  scale=0.125, seed=77)
    inp = W.make_inputs(wl)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    mask, bias = inp["mask"].cuda(), inp["bias"].cuda()
    out_f, lse_f = F.fwd(q, k, v, mask=mask, bias=bias, causal=True, scale=wl.scale)
    bm_f = F.classify_blocks(q, k, v, mask=mask, causal=True)
    r0, r1 = 2 * cp.TILE, 4 * cp.TILE + 40
    o, l = F.fwd(q[:, r0:r1], k, v, mask=mask[:, :, r0:r1], bias=bias[:, :, r0:r1], scale=wl.scale,
                 causal_offset=r0)
    bm = F.classify_blocks(q[:, r0:r1], k, v, mask=mask[:, :, r0:r1], causal_offset=r0)
    assert F.device_error() == 0
    assert torch.equal(o, out_f[:, r0:r1]) and torch.equal(l, lse_f[:, :, r0:r1])
    assert torch.equal(bm[:, :, :2], bm_f[:, :, 2:4])  # (the third local tile holds 40 rows only)
