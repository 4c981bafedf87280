"""Parity at the full workload sizes, in the launch configuration bench.py
times (classify, then forward and backward reusing the classification).

N=4096 is compared element by element.  At N=16384, N=65536 and the
document-mask workload the oracle recomputes sampled query rows one by one
(O, lse, dQ for every head of the group, dBias, block-map rows, bit-exact);
the same recipe at N = 15896 with odd group sizes and MHA (the forward's paired
query tiles, an odd tile count and a ragged tail) is checked the same way.
dK and dV are compared element by element on the whole of kv group 0 at
N=16384, and at N=65536 and on the document mask on the last 256 key columns of
one kv group: under the causal mask (and, for the document mask, inside the key's
document) key j receives gradient only from query rows i >= j, so the oracle's
backward over the last 256 query rows gives those columns exactly.  They are also
checked everywhere through identities that hold at any size:

    sum_j dK[b, j, g] = scale * sum_i sum_{h in g} q_i * (sum_j dS_ij) = 0
    sum_j dV[b, j, g] = sum_{h in g} sum_{i: row not empty} dO[b, i, h]
    sum_j dBias[b, g, i, j] = 0      (since sum_j P_ij dP_ij = delta_i)
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as orc
from block_sparse_masked_02_gb300 import workloads as W
from parity_report import record

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

O_MAXABS, O_RELL2, G_RELL2, LSE_ABS = 1e-2, 5e-3, 1e-2, 4e-3


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_masked_02_gb300 import fdma

    fdma.load()
    return fdma


def rel_l2(x, ref):
    den = np.linalg.norm(ref)
    return np.linalg.norm(np.asarray(x, np.float64) - ref) / (den if den > 0 else 1.0)


def run_bench_config(F, wl, inp):
    q, k, v, do = inp["q"], inp["k"], inp["v"], inp["dout"]
    bias, mask, cr = inp["bias"], inp["mask"], inp["colranges"]
    args = F.make_args(q, k, v, mask=mask, colranges=cr, bias=bias, causal=wl.causal, scale=wl.scale)
    ws = F.alloc_workspace(args, True, q.device)
    bm = F.classify_blocks(q, k, v, mask=mask, colranges=cr, causal=wl.causal, workspace=ws)
    R = F.FDMA_FLAG_REUSE_CLASSIFICATION
    out, lse = F.fwd(q, k, v, mask=mask, colranges=cr, bias=bias, causal=wl.causal, scale=wl.scale, workspace=ws,
                     flags=R)
    dq, dk, dv, db = F.bwd(q, k, v, out, do, lse, mask=mask, colranges=cr, bias=bias, causal=wl.causal,
                           scale=wl.scale, workspace=ws, flags=R)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    del ws
    return bm, out, lse, dq, dk, dv, db


def sample_rows(N, n, seed):
    rng = np.random.default_rng(seed)
    rows = set([0, 1, 127, 128, N - 1]) | set(rng.integers(0, N, n).tolist())
    return sorted(r for r in rows if r < N)


def check_rows(p, wl, bm, out, lse, dq, db, b, g, rows):
    """Oracle rows one by one (each row as its own 1-row block).  Returns the largest
    errors seen (O max-abs, lse, per-row dQ and dBias relative L2)."""
    kv = orc._kv(p, b, g)
    nkt = bm.shape[3]
    worst = {"o_maxabs": 0.0, "lse_maxabs": 0.0, "dq_row_rel_l2_max": 0.0, "dbias_row_rel_l2_max": 0.0}
    for i in rows:
        keep = orc.keep_rows(p, b, g, i, i + 1)
        # block-map row of this query tile is checked on its first sampled row
        for h in range(g * wl.G, (g + 1) * wl.G):
            O, L, _ = orc.forward_rows(p, b, h, i, i + 1, kv, keep)
            o = out[b, i, h].float().cpu().numpy()
            lg = float(lse[b, h, i])
            if np.isneginf(L[0]):
                assert lg == -math.inf and np.all(o == 0.0)
            else:
                worst["lse_maxabs"] = max(worst["lse_maxabs"], abs(lg - L[0]))
                worst["o_maxabs"] = max(worst["o_maxabs"], np.abs(o - O[0]).max())
                assert abs(lg - L[0]) <= LSE_ABS
                assert np.abs(o - O[0]).max() <= O_MAXABS
        dq_r, _, _, db_r = orc.backward_rows(p, b, g, i, i + 1, kv, keep)
        got = dq[b, i, g * wl.G:(g + 1) * wl.G].float().cpu().numpy()
        if np.abs(dq_r[0]).max() > 1e-3:
            worst["dq_row_rel_l2_max"] = max(worst["dq_row_rel_l2_max"], rel_l2(got, dq_r[0]))
        assert rel_l2(got, dq_r[0]) <= G_RELL2 or np.abs(got - dq_r[0]).max() <= 1e-3
        if db is not None:
            drow = db[b, g, i].float().cpu().numpy()
            if np.abs(db_r[0]).max() > 1e-3:
                worst["dbias_row_rel_l2_max"] = max(worst["dbias_row_rel_l2_max"], rel_l2(drow, db_r[0]))
            assert rel_l2(drow, db_r[0]) <= G_RELL2 or np.abs(drow - db_r[0]).max() <= 1e-3
            assert np.all(drow[~keep[0]] == 0.0)
            assert abs(drow.astype(np.float64).sum()) <= 1e-2 * max(1.0, np.abs(drow).sum())
    # bit-exact block-map rows for the sampled query tiles
    for qt in sorted(set(r // 128 for r in rows)):
        r0, r1 = qt * 128, min(qt * 128 + 128, wl.Nq)
        keep = orc.keep_rows(p, b, g, r0, r1)
        for kt in range(nkt):
            blk = keep[:, kt * 128:(kt + 1) * 128]
            ref = 0 if not blk.any() else (2 if blk.all() else 1)
            assert int(bm[b, g, qt, kt]) == ref
    return worst


def check_last_key_columns(p, wl, dk, dv, b, g, ncols=256):
    """dK / dV of the last `ncols` keys of (b, g) element by element: with a causal
    square problem (and a document mask that never reaches back across documents) those
    keys receive gradient only from the last `ncols` query rows, whose oracle backward is
    therefore the exact reference.  Returns the relative L2 errors."""
    assert wl.causal and wl.Nq == wl.Nk
    kv = orc._kv(p, b, g)
    _, dk_part, dv_part, _ = orc.backward_rows(p, b, g, wl.Nq - ncols, wl.Nq, kv)
    got_k = dk[b, wl.Nk - ncols:, g].float().cpu().numpy()
    got_v = dv[b, wl.Nk - ncols:, g].float().cpu().numpy()
    ek = rel_l2(got_k, dk_part[wl.Nk - ncols:])
    ev = rel_l2(got_v, dv_part[wl.Nk - ncols:])
    assert ek <= G_RELL2, ("dk", ek)
    assert ev <= G_RELL2, ("dv", ev)
    return ek, ev


def check_dk_dv_identities(p, wl, lse, dk, dv, do):
    for b in range(wl.B):
        for g in range(wl.Hkv):
            sk = dk[b, :, g].double().sum(0).cpu().numpy()
            scale_k = dk[b, :, g].double().abs().sum(0).cpu().numpy().max()
            assert np.abs(sk).max() <= 2e-2 * max(scale_k, 1e-6)
            heads = range(g * wl.G, (g + 1) * wl.G)
            expect = np.zeros(wl.d)
            for h in heads:
                nonempty = torch.isfinite(lse[b, h]).cpu()
                expect += do[b, :, h].double().cpu()[nonempty].sum(0).numpy()
            sv = dv[b, :, g].double().sum(0).cpu().numpy()
            assert np.abs(sv - expect).max() <= 2e-2 * max(np.abs(expect).max(), 1.0) + 1e-2 * np.sqrt(wl.Nq)


def test_n4096_full_elementwise(F):
    wl = W.WORKLOADS["n4096_hq32_hkv8"]
    inp = W.make_inputs(wl, device="cuda")
    bm, out, lse, dq, dk, dv, db = run_bench_config(F, wl, inp)
    host = {k: (v.cpu() if v is not None else None) for k, v in inp.items()}
    p = orc.Problem(host["q"], host["k"], host["v"], bias=host["bias"], mask=host["mask"], causal=True,
                    scale=wl.scale, dout=host["dout"])
    assert np.array_equal(bm.cpu().numpy(), orc.classify_blocks(p))
    O, L = orc.forward(p)
    o = out.float().cpu().numpy()
    assert np.abs(o - O).max() <= O_MAXABS and rel_l2(o, O) <= O_RELL2
    fin = np.isfinite(L)
    assert np.array_equal(np.isfinite(lse.cpu().numpy()), fin)
    lse_err = np.abs(lse.cpu().numpy()[fin] - L[fin]).max()
    assert lse_err <= LSE_ABS
    case = "n4096_hq32_hkv8 (element-wise)"
    record(case, o_maxabs=np.abs(o - O).max(), o_rel_l2=rel_l2(o, O), lse_maxabs=lse_err)
    rq, rk, rv, rb = orc.backward(p)
    for name, x, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv), ("dbias", db, rb)):
        e = rel_l2(x.float().cpu().numpy(), ref)
        record(case, **{name + "_rel_l2": e})
        assert e <= G_RELL2, name


def test_n16384_sampled_rows_and_columns(F):
    wl = W.WORKLOADS["n16384_hq16_hkv4"]
    inp = W.make_inputs(wl, device="cuda")
    bm, out, lse, dq, dk, dv, db = run_bench_config(F, wl, inp)
    p = orc.Problem(inp["q"], inp["k"], inp["v"], bias=inp["bias"], mask=inp["mask"], causal=True,
                    scale=wl.scale, dout=inp["dout"])
    case = "n16384_hq16_hkv4 (sampled rows; dK/dV of kv group 0 element-wise)"
    for g in (0, wl.Hkv - 1):
        record(case, **check_rows(p, wl, bm, out, lse, dq, db, 0, g, sample_rows(wl.Nq, 12, 5 + g)))
    check_dk_dv_identities(p, wl, lse, dk, dv, inp["dout"])
    # dK / dV columns of kv group 0 against the oracle (whole group, row blocks of 2048)
    cols = [0, 5, 4096, 9999, wl.Nk - 1]
    kv = orc._kv(p, 0, 0)
    dk_ref = np.zeros((wl.Nk, wl.d))
    dv_ref = np.zeros((wl.Nk, wl.d))
    for r0 in range(0, wl.Nq, 2048):
        _, dk_part, dv_part, _ = orc.backward_rows(p, 0, 0, r0, min(r0 + 2048, wl.Nq), kv)
        dk_ref += dk_part
        dv_ref += dv_part
    for j in cols:
        for got, ref in ((dk[0, j, 0], dk_ref[j]), (dv[0, j, 0], dv_ref[j])):
            g_ = got.float().cpu().numpy()
            assert rel_l2(g_, ref) <= 2e-2 or np.abs(g_ - ref).max() <= 2e-3
    ek = rel_l2(dk[0, :, 0].float().cpu().numpy(), dk_ref)
    ev = rel_l2(dv[0, :, 0].float().cpu().numpy(), dv_ref)
    record(case, dk_rel_l2=ek, dv_rel_l2=ev)
    assert ek <= G_RELL2
    assert ev <= G_RELL2


def test_n65536_sampled_rows(F):
    wl = W.WORKLOADS["n65536_hq16_hkv2"]
    inp = W.make_inputs(wl, device="cuda")
    bm, out, lse, dq, dk, dv, db = run_bench_config(F, wl, inp)
    p = orc.Problem(inp["q"], inp["k"], inp["v"], bias=inp["bias"], mask=inp["mask"], causal=True,
                    scale=wl.scale, dout=inp["dout"])
    case = "n65536_hq16_hkv2 (sampled rows; dK/dV of the last 256 keys of kv group 1 element-wise)"
    record(case, **check_rows(p, wl, bm, out, lse, dq, db, 0, 1, sample_rows(wl.Nq, 6, 11)))
    ek, ev = check_last_key_columns(p, wl, dk, dv, 0, 1)
    record(case, dk_rel_l2=ek, dv_rel_l2=ev)
    check_dk_dv_identities(p, wl, lse, dk, dv, inp["dout"])
    # skip ratio: the causal half of the tiles, and top-4096 of 65536 leaves essentially no empty tile
    bmn = bm.cpu().numpy()
    assert abs((bmn == 0).mean() - 0.499) < 0.01


def test_docmask_sampled_rows(F):
    wl = W.WORKLOADS["docmask_b2_n32768"]
    inp = W.make_inputs(wl, device="cuda")
    bm, out, lse, dq, dk, dv, db = run_bench_config(F, wl, inp)
    assert db is None
    p = orc.Problem(inp["q"], inp["k"], inp["v"], colranges=inp["colranges"], causal=True, scale=wl.scale,
                    dout=inp["dout"])
    case = "docmask_b2_n32768 (sampled rows; dK/dV of the last 256 keys of batch 1, kv group 3 element-wise)"
    record(case, **check_rows(p, wl, bm, out, lse, dq, None, 1, 3, sample_rows(wl.Nq, 8, 17)))
    ek, ev = check_last_key_columns(p, wl, dk, dv, 1, 3)
    record(case, dk_rel_l2=ek, dv_rel_l2=ev)
    check_dk_dv_identities(p, wl, lse, dk, dv, inp["dout"])
    # document masks skip most tiles
    assert (bm.cpu().numpy() == 0).mean() > 0.8


@pytest.mark.parametrize("Hq,Hkv", [(6, 2), (3, 3)])
def test_odd_groups_sampled_rows(F, Hq, Hkv):
    """Odd group sizes and MHA at full length on the bench recipe (causal top-2048 with a bias),
    N = 15896: the forward pairs the query tiles of one head (125 tiles, so the last pair has no
    second tile; a ragged tail of 24 rows).  Sampled rows (O, lse, dQ, dBias, block-map rows),
    dK / dV of the last 256 keys element by element, and the identities."""
    wl = W.scaled(W.WORKLOADS["n16384_hq16_hkv4"], Nq=15896, Nk=15896, Hq=Hq, Hkv=Hkv, seed=1010 + Hq)
    inp = W.make_inputs(wl, device="cuda")
    bm, out, lse, dq, dk, dv, db = run_bench_config(F, wl, inp)
    p = orc.Problem(inp["q"], inp["k"], inp["v"], bias=inp["bias"], mask=inp["mask"], causal=True,
                    scale=wl.scale, dout=inp["dout"])
    case = f"N=15896 Hq{Hq} Hkv{Hkv} (sampled rows; dK/dV of the last 256 keys element-wise)"
    rows = sample_rows(wl.Nq, 10, 40 + Hq) + [wl.Nq - 24, wl.Nq - 25, 124 * 128 - 1]
    record(case, **check_rows(p, wl, bm, out, lse, dq, db, 0, Hkv - 1, sorted(set(rows))))
    ek, ev = check_last_key_columns(p, wl, dk, dv, 0, Hkv - 1)
    record(case, dk_rel_l2=ek, dv_rel_l2=ev)
    check_dk_dv_identities(p, wl, lse, dk, dv, inp["dout"])
