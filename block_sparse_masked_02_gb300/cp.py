"""Context-parallel split of self-attention over the sequence (FlashMask README, "CPB:
mask-aware load balancing" and "Overlap: mask-aware communication/computation overlap").

Every rank owns a set of 128-token tiles of the sequence: their queries, keys, values and
output gradients, and the mask and bias rows of its queries (built where they are used, so no
mask is ever communicated: the "localized transformation" of the pages).  Forward: each rank
receives, from their owners, the K/V tiles that its own query rows need (a key tile none of
its rows reaches is never sent: the pages' mask-aware pruning of the KV transfer), then runs
the attention of its query rows against the keys.  Backward: each rank's dK/dV partial sums
over all keys go back to the owners of those key tiles, which add them up (a reduce-scatter
restricted to the tiles that were sent).  dQ, dBias, O and lse stay with the rows' owner.

Balance (reading of the pages' HCC-IPO, which they do not spell out): the cost of a query tile
is its count of active tiles (non-skipped tiles of its block-map row, summed over batch and kv
heads).  Tiles are first placed largest first on the least loaded rank, then the most and the
least loaded ranks repeatedly exchange the one tile move or tile swap that most lowers the
larger of their two loads, until no move or swap lowers it (pairwise optimal, iterated).  The
pages' hierarchical (intra/inter-node) level does not arise on one node and is not modelled.

A contiguous run of owned tiles is one attention call: rows [r0, r1) of the sequence against
all keys, with the causal rule kept global through the row offset (is_causal 2, q_offset = r0).

Host logic only.  The collectives are torch.distributed point-to-point calls (NCCL between
GPUs, gloo on the CPU); GPU tensors are exchanged tile by tile into local HBM (no multicast, no
peer access from kernels).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

TILE = 128


# ----------------------------------------------------------------------------- planning
def tile_work(block_map) -> np.ndarray:
    """Cost of each query tile: its active (non-skipped) tiles summed over batch and kv heads.
    block_map: int8 (B, Hkv, nTq, nTk) tile classes (0 skip, 1 partial, 2 full)."""
    bm = block_map.cpu().numpy() if hasattr(block_map, "cpu") else np.asarray(block_map)
    return (bm != 0).sum(axis=(0, 1, 3)).astype(np.int64)


@dataclasses.dataclass
class Plan:
    world: int
    owner: np.ndarray  # (nT,) rank owning each tile
    loads: np.ndarray  # (world,) summed work

    def tiles_of(self, rank: int) -> np.ndarray:
        return np.flatnonzero(self.owner == rank)

    def runs_of(self, rank: int) -> List[Tuple[int, int]]:
        return runs(self.tiles_of(rank))


def _best_pair_step(work, owner, a, b, la, lb):
    """Best single move (a -> b) or swap (a <-> b) by the larger of the two new loads."""
    ta = np.flatnonzero(owner == a)
    tb = np.flatnonzero(owner == b)
    best = (max(la, lb), None)
    for t in ta:  # move t from a to b
        m = max(la - work[t], lb + work[t])
        if m < best[0]:
            best = (m, ("move", t))
    if len(ta) and len(tb):
        wa, wb = work[ta], work[tb]
        # swap t (a) and u (b): loads la - wa + wb, lb + wa - wb
        d = wa[:, None] - wb[None, :]
        m = np.maximum(la - d, lb + d)
        i, j = np.unravel_index(np.argmin(m), m.shape)
        if m[i, j] < best[0]:
            best = (int(m[i, j]), ("swap", ta[i], tb[j]))
    return best[1]


def balance(work: Sequence[int], world: int, max_steps: int = 10000) -> Plan:
    """Assign query tiles to `world` ranks: largest first onto the least loaded rank, then
    iterated pairwise improvement between the most and the least loaded rank (see module
    docstring).  Deterministic: ties go to the lower tile index and the lower rank."""
    work = np.asarray(work, dtype=np.int64)
    if world < 1:
        raise ValueError("world must be >= 1")
    n = len(work)
    owner = np.zeros(n, dtype=np.int64)
    loads = np.zeros(world, dtype=np.int64)
    for t in sorted(range(n), key=lambda t: (-work[t], t)):
        r = int(np.argmin(loads))
        owner[t] = r
        loads[r] += work[t]
    for _ in range(max_steps):
        a, b = int(np.argmax(loads)), int(np.argmin(loads))
        if a == b:
            break
        step = _best_pair_step(work, owner, a, b, loads[a], loads[b])
        if step is None:
            break
        if step[0] == "move":
            t = step[1]
            owner[t] = b
            loads[a] -= work[t]
            loads[b] += work[t]
        else:
            t, u = step[1], step[2]
            owner[t], owner[u] = b, a
            loads[a] += work[u] - work[t]
            loads[b] += work[t] - work[u]
    return Plan(world, owner, loads)


def runs(tiles: Sequence[int]) -> List[Tuple[int, int]]:
    """Sorted tile indices as maximal contiguous runs [t0, t1)."""
    out: List[Tuple[int, int]] = []
    for t in sorted(int(x) for x in tiles):
        if out and out[-1][1] == t:
            out[-1] = (out[-1][0], t + 1)
        else:
            out.append((t, t + 1))
    return out


def needed_key_tiles(block_map_rows) -> np.ndarray:
    """bool (nTk,): key tiles that some query tile of these block-map rows does not skip.
    block_map_rows: int8 (B, Hkv, n_rows, nTk)."""
    bm = block_map_rows.cpu().numpy() if hasattr(block_map_rows, "cpu") else np.asarray(block_map_rows)
    return (bm != 0).any(axis=(0, 1, 2))


# ----------------------------------------------------------------------------- localization
def row_span(run: Tuple[int, int], N: int) -> Tuple[int, int]:
    """Sequence rows [r0, r1) of a run of tiles (the last tile may be ragged)."""
    return run[0] * TILE, min(run[1] * TILE, N)


def local_colranges(colranges: torch.Tensor, r0: int) -> torch.Tensor:
    """Column ranges in the run's own row numbering: every masked row range moves down by r0
    (the kernels clamp the ranges to the run's rows)."""
    return colranges - r0


@dataclasses.dataclass
class LocalInputs:
    """Inputs of one run: rows [r0, r1) of q / dout / mask / bias against all keys."""
    r0: int
    r1: int
    q: torch.Tensor
    dout: Optional[torch.Tensor]
    mask: Optional[torch.Tensor]
    colranges: Optional[torch.Tensor]
    bias: Optional[torch.Tensor]
    causal_offset: Optional[int]


def localize(run, *, q, dout=None, mask=None, colranges=None, bias=None, causal=True, Nk=None) -> LocalInputs:
    """Slice one run's rows out of sequence-length tensors (views where the kernels accept
    them).  q / dout (B, N, Hq, d); mask / bias (B, Hkv, N, Nk); colranges (B, Hkv, Nk, 2|4)."""
    N = q.shape[1]
    Nk = N if Nk is None else Nk
    r0, r1 = row_span(run, N)
    return LocalInputs(
        r0, r1,
        q[:, r0:r1],
        None if dout is None else dout[:, r0:r1].contiguous(),
        None if mask is None else mask[:, :, r0:r1, :],
        None if colranges is None else local_colranges(colranges, r0),
        None if bias is None else bias[:, :, r0:r1, :],
        (r0 + (Nk - N)) if causal else None,
    )


# ----------------------------------------------------------------------------- exchange
def _tile(x: torch.Tensor, t: int, N: int) -> torch.Tensor:
    """Rows of tile t along dim 1 of a (B, N, H, d) tensor."""
    return x[:, t * TILE:min((t + 1) * TILE, N)]


def exchange_needs(needed: np.ndarray, group=None) -> np.ndarray:
    """All ranks' needed-key-tile bitmaps, (world, nT) bool, by one all-gather."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    mine = torch.from_numpy(needed.astype(np.uint8))
    dev = _comm_device(group)
    mine = mine.to(dev)
    allv = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(allv, mine, group=group)
    return np.stack([a.cpu().numpy().astype(bool) for a in allv])


def _comm_device(group=None):
    import torch.distributed as dist

    return torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" else torch.device("cpu")


def gather_kv(k_own: torch.Tensor, v_own: torch.Tensor, plan: Plan, needs: np.ndarray, N: int, group=None):
    """Full-length K and V for this rank: its own tiles, plus the tiles it needs from their
    owners (point-to-point).  k_own / v_own: (B, N, Hkv, d) tensors of which only the owned
    tiles are read.  Tiles this rank does not need stay zero (no kernel reads them: every
    tile of those key columns is skipped in this rank's rows)."""
    import torch.distributed as dist

    rank = dist.get_rank(group)
    k = torch.zeros_like(k_own)
    v = torch.zeros_like(v_own)
    for t in plan.tiles_of(rank):
        _tile(k, t, N).copy_(_tile(k_own, t, N))
        _tile(v, t, N).copy_(_tile(v_own, t, N))
    ops, recv, keep = [], [], []
    for t in range(len(plan.owner)):
        src = int(plan.owner[t])
        for dst in range(plan.world):
            if dst == src or not needs[dst, t]:
                continue
            if src == rank:
                for x in (k_own, v_own):
                    buf = _tile(x, t, N).contiguous()
                    keep.append(buf)  # alive until the sends complete
                    ops.append(dist.isend(buf, dst, group=group))
            elif dst == rank:
                bk = torch.empty_like(_tile(k, t, N).contiguous())
                bv = torch.empty_like(bk)
                ops.append(dist.irecv(bk, src, group=group))
                ops.append(dist.irecv(bv, src, group=group))
                recv.append((t, bk, bv))
    for op in ops:
        op.wait()
    for t, bk, bv in recv:
        _tile(k, t, N).copy_(bk)
        _tile(v, t, N).copy_(bv)
    return k, v


def reduce_dkdv(dk_part: torch.Tensor, dv_part: torch.Tensor, plan: Plan, needs: np.ndarray, N: int, group=None):
    """Sum the ranks' dK/dV partials into the owners' tiles: a rank sends the partial of every
    key tile it needed but does not own to that tile's owner; an owner adds what it receives
    (in fp32) to its own partial.  Returns fp32 (B, N, Hkv, d) tensors holding this rank's
    tiles (zero elsewhere)."""
    import torch.distributed as dist

    rank = dist.get_rank(group)
    dk = torch.zeros(dk_part.shape, dtype=torch.float32, device=dk_part.device)
    dv = torch.zeros_like(dk)
    for t in plan.tiles_of(rank):
        _tile(dk, t, N).copy_(_tile(dk_part, t, N).float())
        _tile(dv, t, N).copy_(_tile(dv_part, t, N).float())
    ops, recv, keep = [], [], []
    for t in range(len(plan.owner)):
        dst = int(plan.owner[t])
        for src in range(plan.world):
            if src == dst or not needs[src, t]:
                continue
            if src == rank:
                for x in (dk_part, dv_part):
                    buf = _tile(x, t, N).contiguous()
                    keep.append(buf)  # alive until the sends complete
                    ops.append(dist.isend(buf, dst, group=group))
            elif dst == rank:
                bk = torch.empty(_tile(dk_part, t, N).shape, dtype=dk_part.dtype, device=dk_part.device)
                bv = torch.empty_like(bk)
                ops.append(dist.irecv(bk, src, group=group))
                ops.append(dist.irecv(bv, src, group=group))
                recv.append((t, bk, bv))
    for op in ops:
        op.wait()
    for t, bk, bv in recv:
        _tile(dk, t, N).add_(bk.float())
        _tile(dv, t, N).add_(bv.float())
    return dk, dv


# ----------------------------------------------------------------------------- attention
def forward_runs(fdma, runs_, *, q, k, v, mask=None, colranges=None, bias=None, causal=True, scale=None):
    """The forward of every run of this rank through the library (k / v full length, with at
    least the needed tiles present).  Returns [(r0, r1, out, lse)]."""
    res = []
    for run in runs_:
        li = localize(run, q=q, mask=mask, colranges=colranges, bias=bias, causal=causal, Nk=k.shape[1])
        out, lse = fdma.fwd(li.q, k, v, mask=li.mask, colranges=li.colranges, bias=li.bias, scale=scale,
                            causal_offset=li.causal_offset, causal=causal)
        res.append((li.r0, li.r1, out, lse))
    return res


def backward_runs(fdma, runs_, fwd_res, *, q, k, v, dout, mask=None, colranges=None, bias=None, causal=True,
                  scale=None, want_dbias=True):
    """The backward of every run.  Returns ([(r0, r1, dq, dbias)], dk_part, dv_part): dQ and
    dBias of the run's rows, and this rank's dK/dV partial sums over all keys (fp32)."""
    per_run = []
    dk = torch.zeros(k.shape, dtype=torch.float32, device=k.device)
    dv = torch.zeros_like(dk)
    for run, (r0, r1, out, lse) in zip(runs_, fwd_res):
        li = localize(run, q=q, dout=dout, mask=mask, colranges=colranges, bias=bias, causal=causal, Nk=k.shape[1])
        dq, dkr, dvr, db = fdma.bwd(li.q, k, v, out, li.dout, lse, mask=li.mask, colranges=li.colranges,
                                    bias=li.bias, scale=scale, want_dbias=want_dbias,
                                    causal_offset=li.causal_offset, causal=causal)
        dk += dkr.float()
        dv += dvr.float()
        per_run.append((r0, r1, dq, db))
    return per_run, dk, dv
