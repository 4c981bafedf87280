"""Context-parallel host logic (block_sparse_masked_02_gb300.cp) on the CPU: the balance of
query tiles over ranks, the localization of one run of rows (masks, column ranges and the
causal rule), and a world-size-2 gloo run of the K/V gather and the dK/dV reduction in which
the oracle is each rank's local attention: the ranks' results put together equal the unsplit
problem's (FlashMask README, "CPB" and "Overlap")."""
import itertools
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import attention as orc
from block_sparse_masked_02_gb300 import cp

T = cp.TILE


# ----------------------------------------------------------------------------- balance
def _pair_can_improve(work, owner, a, b):
    la = work[owner == a].sum()
    lb = work[owner == b].sum()
    cur = max(la, lb)
    ta, tb = np.flatnonzero(owner == a), np.flatnonzero(owner == b)
    for t in ta:
        if max(la - work[t], lb + work[t]) < cur:
            return True
    for t, u in itertools.product(ta, tb):
        d = work[t] - work[u]
        if max(la - d, lb + d) < cur:
            return True
    return False


@pytest.mark.parametrize("seed,n,world", [(1, 40, 3), (2, 128, 8), (3, 7, 4), (4, 5, 8), (5, 64, 2)])
def test_balance_assigns_each_tile_once_and_no_pair_step_helps(seed, n, world):
    work = np.random.default_rng(seed).integers(0, 60, n)
    plan = cp.balance(work, world)
    assert plan.owner.shape == (n,) and plan.owner.min() >= 0 and plan.owner.max() < world
    assert np.array_equal(plan.loads, np.bincount(plan.owner, weights=work, minlength=world).astype(np.int64))
    a, b = int(np.argmax(plan.loads)), int(np.argmin(plan.loads))
    assert a == b or not _pair_can_improve(work, plan.owner, a, b)
    # never worse than the classic bound of largest-first placement
    assert plan.loads.max() <= work.sum() / world + work.max()
    again = cp.balance(work, world)
    assert np.array_equal(again.owner, plan.owner)  # deterministic


def test_balance_of_a_causal_profile():
    """Query tile t of a causal problem has nT - t active tiles: equal-length contiguous chunks
    give rank 0 about twice the mean; the balanced split is within 1 %."""
    nT, world = 128, 8
    work = nT - np.arange(nT)
    plan = cp.balance(work, world)
    assert plan.loads.max() / plan.loads.mean() < 1.01
    chunk = work.reshape(world, -1).sum(axis=1)
    assert chunk.max() / chunk.mean() > 1.8


def test_runs_and_row_spans():
    assert cp.runs([5, 1, 2, 3, 7, 8]) == [(1, 4), (5, 6), (7, 9)]
    assert cp.runs([]) == []
    assert cp.row_span((3, 5), 600) == (384, 600)  # ragged last tile


def test_tile_work_and_needed_key_tiles():
    bm = np.random.default_rng(3).integers(0, 3, (2, 3, 5, 6)).astype(np.int8)
    assert np.array_equal(cp.tile_work(bm), np.array([(bm[:, :, t, :] != 0).sum() for t in range(5)]))
    rows = bm[:, :, [1, 3], :]
    want = np.array([(rows[:, :, :, j] != 0).any() for j in range(6)])
    assert np.array_equal(cp.needed_key_tiles(rows), want)
    assert np.array_equal(cp.tile_work(torch.from_numpy(bm)), cp.tile_work(bm))


def _full_problem(seed, N, kind, Hq=2, Hkv=1, d=8):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(1, N, Hq, d, generator=g, dtype=torch.float64)
    k = torch.randn(1, N, Hkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(1, N, Hkv, d, generator=g, dtype=torch.float64)
    do = torch.randn(1, N, Hq, d, generator=g, dtype=torch.float64)
    bias = torch.randn(1, Hkv, N, N, generator=g, dtype=torch.float64)
    mask = cr = None
    if kind == "dense":
        mask = (torch.rand(1, Hkv, N, N, generator=g) < 0.4).to(torch.float64)
    elif kind in ("colranges", "colranges2"):
        s = torch.randint(-5, N + 5, (1, Hkv, N), generator=g)
        ln = torch.randint(-3, N // 2, (1, Hkv, N), generator=g)
        cr = torch.stack([s, s + ln], dim=-1)
        if kind == "colranges2":
            s2 = torch.randint(-5, N + 5, (1, Hkv, N), generator=g)
            cr = torch.cat([cr, torch.stack([s2, s2 + 7], dim=-1)], dim=-1)
        cr = cr.to(torch.int32)
    return q, k, v, do, bias, mask, cr


@pytest.mark.parametrize("kind", ["dense", "colranges", "colranges2", "none"])
@pytest.mark.parametrize("causal", [True, False])
def test_localized_run_keeps_exactly_the_global_rows(kind, causal):
    """A run's own problem (rows [r0, r1) against all keys, shifted column ranges, causal row
    offset r0) keeps exactly the keys the unsplit problem keeps on those rows."""
    N = 3 * T + 44
    q, k, v, do, bias, mask, cr = _full_problem(5, N, kind)
    full = orc.Problem(q, k, v, bias=bias, mask=mask, colranges=cr, causal=causal)
    for run in [(0, 1), (1, 3), (2, 4), (3, 4), (0, 4)]:
        li = cp.localize(run, q=q, dout=do, mask=mask, colranges=cr, bias=bias, causal=causal)
        loc = orc.Problem(li.q, k, v, bias=li.bias, mask=li.mask, colranges=li.colranges, causal=causal,
                          causal_offset=li.causal_offset)
        assert (li.r0, li.r1) == cp.row_span(run, N)
        assert np.array_equal(orc.keep_rows(loc, 0, 0, 0, li.r1 - li.r0), orc.keep_rows(full, 0, 0, li.r0, li.r1))


# ----------------------------------------------------------------------------- two ranks (gloo)
def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _doc_problem(N):
    """Self-attention over two documents (tiles 0-1 and 2-4) plus a bias, as a dense mask:
    a rank whose queries lie in one document needs no key tile of the other."""
    q, k, v, do, bias, _, _ = _full_problem(11, N, "none", Hq=2, Hkv=1, d=8)
    cut = 2 * T
    doc = torch.zeros(N, N, dtype=torch.float64)
    doc[:cut, :cut] = 1
    doc[cut:, cut:] = 1
    mask = (doc * (torch.rand(N, N, generator=torch.Generator().manual_seed(12)) < 0.7)).reshape(1, 1, N, N)
    return q, k, v, do, bias, mask


def _cp_worker(rank, world, port, N, out):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import attention as orc_
    from block_sparse_masked_02_gb300 import cp as cp_

    q, k, v, do, bias, mask = _doc_problem(N)
    bm = orc_.classify_blocks(orc_.Problem(q, k, v, bias=bias, mask=mask, causal=True))
    plan = cp_.balance(cp_.tile_work(bm), world)
    own = plan.tiles_of(rank)
    needs = cp_.exchange_needs(cp_.needed_key_tiles(bm[:, :, own, :]))
    # this rank holds only its own tiles of K and V
    rows = torch.zeros(N, dtype=torch.bool)
    for t in own:
        rows[t * T:(t + 1) * T] = True
    k_own = k * rows[None, :, None, None]
    v_own = v * rows[None, :, None, None]
    kf, vf = cp_.gather_kv(k_own, v_own, plan, needs, N)
    res = {"own": own.tolist(), "needs": needs.tolist(), "runs": []}
    dk_part = np.zeros(k.shape)
    dv_part = np.zeros(v.shape)
    for run in plan.runs_of(rank):
        li = cp_.localize(run, q=q, dout=do, mask=mask, bias=bias, causal=True)
        p = orc_.Problem(li.q, kf, vf, bias=li.bias, mask=li.mask, causal=True, causal_offset=li.causal_offset,
                         dout=li.dout)
        O, lse = orc_.forward(p)
        dq, dk, dv, db = orc_.backward(p)
        dk_part += dk
        dv_part += dv
        res["runs"].append((li.r0, li.r1, O, lse, dq, db))
    dkr, dvr = cp_.reduce_dkdv(torch.from_numpy(dk_part), torch.from_numpy(dv_part), plan, needs, N)
    res["dk"], res["dv"] = dkr.numpy(), dvr.numpy()
    res["kf"], res["vf"] = kf.numpy(), vf.numpy()
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gather_attend_reduce_equal_the_unsplit_problem():
    world, port, N = 2, _free_port(), 5 * T
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_cp_worker, args=(world, port, N, out), nprocs=world, join=True, start_method="spawn")
    q, k, v, do, bias, mask = _doc_problem(N)
    full = orc.Problem(q, k, v, bias=bias, mask=mask, causal=True, dout=do)
    O, lse = orc.forward(full)
    dq, dk, dv, db = orc.backward(full)
    owned = sorted(t for r in range(world) for t in out[r]["own"])
    assert owned == list(range(N // T))  # every tile owned exactly once
    kn, vn = k.numpy(), v.numpy()
    pruned = 0
    for r in range(world):
        res = out[r]
        needs = np.array(res["needs"])
        for t in range(N // T):
            sl = slice(t * T, (t + 1) * T)
            if needs[r, t] or t in res["own"]:
                assert np.array_equal(res["kf"][:, sl], kn[:, sl]) and np.array_equal(res["vf"][:, sl], vn[:, sl])
            else:
                pruned += 1
                assert not res["kf"][:, sl].any()  # never sent
            if t in res["own"]:
                assert np.abs(res["dk"][:, sl] - dk[:, sl]).max() < 1e-5 * np.abs(dk).max()
                assert np.abs(res["dv"][:, sl] - dv[:, sl]).max() < 1e-5 * np.abs(dv).max()
        for r0, r1, Or, lser, dqr, dbr in res["runs"]:
            assert np.abs(Or - O[:, r0:r1]).max() < 1e-12
            ref = lse[:, :, r0:r1]
            assert np.array_equal(np.isneginf(lser), np.isneginf(ref))  # rows that see no key
            fin = np.isfinite(ref)
            assert np.abs(lser[fin] - ref[fin]).max() < 1e-12
            assert np.abs(dqr - dq[:, r0:r1]).max() < 1e-12
            assert np.abs(dbr - db[:, :, r0:r1]).max() < 1e-12
    assert pruned > 0  # the document split leaves key tiles some rank never receives
