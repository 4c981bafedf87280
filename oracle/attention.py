"""fp64 CPU oracle for masked, biased softmax attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
the benchmark's CPU-baseline leg may import this module; the product path
never does.  It shares no code with the CUDA path: it is the plain definition
written out with numpy in float64, one (batch, head) and one block of query
rows at a time (the row blocks only bound memory; every row is still the full
dense definition and no tile is ever skipped).

Definition followed (Flash-DMA README, "Quick Start" example and
"Key Features"; Flash-DMA issue #73, "Project Progress"; FlashMask README,
"Formulation"):

    keep(b,g,i,j) = mask[b,g,i,j] != 0            (dense 4D mask, per kv head; bf16, uint8 or bool;
                                                   or bit-packed: bit j % 8 of byte j // 8 of row i)
                  | not (start[b,g,j] <= i < end[b,g,j])   (column ranges: one masked
                                                            row range per key column,
                                                            or two, masked as a union)
                  | True                                    (no mask)
                  and (j <= i + c if causal)                (c = Nk - Nq: bottom-right
                                                            aligned, j <= i for square
                                                            problems; or a given row offset
                                                            c: the rows are rows c - (Nk - N) ..
                                                            of a longer causal problem over the
                                                            same keys, as one rank of a
                                                            context-parallel split holds them,
                                                            FlashMask README, "CPB")
    s_ij = scale * q_i . k_j + bias[b,g,i,j]   if keep, else -inf
    P    = softmax_j(s),  O_i = sum_j P_ij v_j,  lse_i = max_j s_ij + ln sum_j exp(s_ij - max)

Query head h reads kv head g = h // (Hq / Hkv).  v (and so O, dO, dV) may have a
head dim dv other than the d of q and k (FlashMask README, "Performance": the SM100
head-dim table lists d = 192 with dv = 128).  A row with no kept key has
O_i = 0, lse_i = -inf and contributes nothing to any gradient.  The scale
multiplies Q K^T only; the bias is added unscaled.

Backward (closed-form gradients of L = sum(O * dO)):

    D_i  = dO_i . O_i
    dP   = dO V^T,   dS = P * (dP - D)
    dV_j = sum_{h in g, i} P_ij dO_i
    dQ_i = scale * sum_j dS_ij k_j
    dK_j = scale * sum_{h in g, i} dS_ij q_i
    dBias[b,g,i,j] = sum_{h in g} dS_ij     (zero wherever keep is false)

Block classification (Flash-DMA "Key Features": OR-reduction of each mask
block; FlashMask "Sparse computation": fully masked / partially masked /
unmasked): for a tile of tile_m x tile_n positions, count the kept in-bounds
elements k and the in-bounds elements n: k == 0 -> 0 (skip), k == n -> 2
(full), otherwise 1 (partial).
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

SKIP, PARTIAL, FULL = 0, 1, 2


def _f64(x) -> np.ndarray:
    """float64 numpy copy of a torch tensor (any dtype) or array."""
    if hasattr(x, "detach"):
        import torch

        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        import torch

        return x.detach().to("cpu", torch.int64).numpy()
    return np.asarray(x, dtype=np.int64)


class Problem:
    """Inputs of one attention call, as given to both implementations.

    q (B,Nq,Hq,d), k/v (B,Nk,Hkv,d), dout like q; bias and mask (B,Hkv,Nq,Nk)
    or None; colranges (B,Hkv,Nk,2) or (B,Hkv,Nk,4) int or None; causal_offset: the causal
    rule's row offset (default Nk - Nq); mask_bits: the mask
    bit-packed, uint8 (B,Hkv,Nq,ceil(Nk/8)), key j of a row = bit j % 8 of byte j // 8.
    Tensors may be torch (any dtype, any device) or numpy; slices are converted to float64
    on demand.
    """

    def __init__(self, q, k, v, *, bias=None, mask=None, colranges=None, causal=False, scale=None, dout=None,
                 mask_bits=None, causal_offset=None):
        self.q, self.k, self.v = q, k, v
        self.bias, self.mask, self.colranges, self.mask_bits = bias, mask, colranges, mask_bits
        self.causal = bool(causal)
        self.B, self.Nq, self.Hq, self.d = (int(s) for s in q.shape)
        self.Nk, self.Hkv = int(k.shape[1]), int(k.shape[2])
        self.dv = int(v.shape[3])  # head dim of v, O and dO (d for q and k)
        # key j is visible from query row i when j <= i + causal_offset (if causal)
        self.causal_offset = self.Nk - self.Nq if causal_offset is None else int(causal_offset)
        assert self.Hq % self.Hkv == 0
        self.G = self.Hq // self.Hkv
        self.scale = 1.0 / math.sqrt(self.d) if scale is None else float(scale)
        self.dout = dout
        if sum(x is not None for x in (mask, colranges, mask_bits)) > 1:
            raise ValueError("give one of a dense mask, a bit-packed mask or column ranges")


def keep_rows(p: Problem, b: int, g: int, r0: int, r1: int) -> np.ndarray:
    """bool (r1-r0, Nk): keep(b, g, i, j) for query rows i in [r0, r1)."""
    i = np.arange(r0, r1)[:, None]
    j = np.arange(p.Nk)[None, :]
    if p.mask is not None:
        keep = _f64(p.mask[b, g, r0:r1, :]) != 0.0
    elif p.mask_bits is not None:
        raw = _i64(p.mask_bits[b, g, r0:r1, :])  # (R, ceil(Nk/8)) byte values
        bit = (raw[:, :, None] >> np.arange(8)[None, None, :]) & 1  # bit e of byte c = key 8c+e
        keep = bit.reshape(r1 - r0, -1)[:, :p.Nk] != 0
    elif p.colranges is not None:
        cr = _i64(p.colranges[b, g])  # (Nk, 2) or (Nk, 4)
        masked = (cr[:, 0][None, :] <= i) & (i < cr[:, 1][None, :])
        if cr.shape[1] == 4:
            masked |= (cr[:, 2][None, :] <= i) & (i < cr[:, 3][None, :])
        keep = ~masked
    else:
        keep = np.ones((r1 - r0, p.Nk), dtype=bool)
    if p.causal:
        keep = keep & (j <= i + p.causal_offset)
    return keep


def _kv(p: Problem, b: int, g: int):
    return _f64(p.k[b, :, g, :]), _f64(p.v[b, :, g, :])


def forward_rows(p: Problem, b: int, h: int, r0: int, r1: int, kv=None, keep=None):
    """O (R,dv), lse (R,), P (R,Nk) for query head h, rows [r0, r1)."""
    g = h // p.G
    K, V = _kv(p, b, g) if kv is None else kv
    if keep is None:
        keep = keep_rows(p, b, g, r0, r1)
    Q = _f64(p.q[b, r0:r1, h, :])
    s = p.scale * (Q @ K.T)
    if p.bias is not None:
        s = s + _f64(p.bias[b, g, r0:r1, :])
    s = np.where(keep, s, -np.inf)
    m = s.max(axis=1)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.where(keep, np.exp(s - m_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    l_safe = np.where(empty, 1.0, l)
    P = e / l_safe[:, None]
    O = P @ V
    O[empty] = 0.0
    lse = np.where(empty, -np.inf, m_safe + np.log(l_safe))
    return O, lse, P


def forward(p: Problem, row_block: int = 1024):
    """Full O (B,Nq,Hq,dv) and lse (B,Hq,Nq), float64."""
    O = np.zeros((p.B, p.Nq, p.Hq, p.dv))
    lse = np.zeros((p.B, p.Hq, p.Nq))
    for b in range(p.B):
        for g in range(p.Hkv):
            kv = _kv(p, b, g)
            for r0 in range(0, p.Nq, row_block):
                r1 = min(r0 + row_block, p.Nq)
                keep = keep_rows(p, b, g, r0, r1)
                for h in range(g * p.G, (g + 1) * p.G):
                    O[b, r0:r1, h], lse[b, h, r0:r1], _ = forward_rows(p, b, h, r0, r1, kv, keep)
    return O, lse


def backward_rows(p: Problem, b: int, g: int, r0: int, r1: int, kv=None, keep=None):
    """Gradient pieces produced by query rows [r0, r1) of kv group g.

    Returns dq (R,G,d) for those rows, the rows' additive contributions
    dk_part (Nk,d) / dv_part (Nk,dv), and dbias rows (R,Nk) (sum over the group's heads).
    """
    K, V = _kv(p, b, g) if kv is None else kv
    if keep is None:
        keep = keep_rows(p, b, g, r0, r1)
    R = r1 - r0
    dq = np.zeros((R, p.G, p.d))
    dk = np.zeros((p.Nk, p.d))
    dv = np.zeros((p.Nk, p.dv))
    dbias = np.zeros((R, p.Nk))
    for hh in range(p.G):
        h = g * p.G + hh
        O, _, P = forward_rows(p, b, h, r0, r1, (K, V), keep)
        dO = _f64(p.dout[b, r0:r1, h, :])
        Q = _f64(p.q[b, r0:r1, h, :])
        D = (dO * O).sum(axis=1)
        dP = dO @ V.T
        dS = P * (dP - D[:, None])
        dv += P.T @ dO
        dq[:, hh, :] = p.scale * (dS @ K)
        dk += p.scale * (dS.T @ Q)
        dbias += dS
    return dq, dk, dv, dbias


def backward(p: Problem, row_block: int = 1024, want_dbias: bool = True):
    """Full dq (B,Nq,Hq,d), dk (B,Nk,Hkv,d), dv (B,Nk,Hkv,dv), dbias (B,Hkv,Nq,Nk) or None."""
    assert p.dout is not None
    dq = np.zeros((p.B, p.Nq, p.Hq, p.d))
    dk = np.zeros((p.B, p.Nk, p.Hkv, p.d))
    dv = np.zeros((p.B, p.Nk, p.Hkv, p.dv))
    dbias = np.zeros((p.B, p.Hkv, p.Nq, p.Nk)) if want_dbias else None
    for b in range(p.B):
        for g in range(p.Hkv):
            kv = _kv(p, b, g)
            for r0 in range(0, p.Nq, row_block):
                r1 = min(r0 + row_block, p.Nq)
                q_, k_, v_, db_ = backward_rows(p, b, g, r0, r1, kv)
                dq[b, r0:r1, g * p.G:(g + 1) * p.G, :] = q_
                dk[b, :, g, :] += k_
                dv[b, :, g, :] += v_
                if want_dbias:
                    dbias[b, g, r0:r1, :] = db_
    return dq, dk, dv, dbias


def classify_blocks(p: Problem, tile_m: int = 128, tile_n: int = 128) -> np.ndarray:
    """int8 (B, Hkv, ceil(Nq/tile_m), ceil(Nk/tile_n)) in {0 skip, 1 partial, 2 full}."""
    nqt = -(-p.Nq // tile_m)
    nkt = -(-p.Nk // tile_n)
    out = np.zeros((p.B, p.Hkv, nqt, nkt), dtype=np.int8)
    pad = nkt * tile_n - p.Nk
    for b in range(p.B):
        for g in range(p.Hkv):
            for qt in range(nqt):
                r0, r1 = qt * tile_m, min((qt + 1) * tile_m, p.Nq)
                keep = keep_rows(p, b, g, r0, r1)
                kept = np.pad(keep, ((0, 0), (0, pad))).reshape(r1 - r0, nkt, tile_n).sum(axis=(0, 2))
                inb = np.full(nkt, (r1 - r0) * tile_n)
                inb[-1] = (r1 - r0) * (p.Nk - (nkt - 1) * tile_n)
                out[b, g, qt] = np.where(kept == 0, SKIP, np.where(kept == inb, FULL, PARTIAL))
    return out


def effective_flops(block_map: np.ndarray, Hq: int, Hkv: int, d: int, tile: int = 128) -> dict:
    """Effective FLOPs counted over non-skipped tiles: 4*d*tile^2 per tile and
    query head for the forward (QK^T, PV), 10*d*tile^2 for the backward (the
    recomputed QK^T plus dP, dV, dK, dQ)."""
    active = int((block_map != SKIP).sum()) * (Hq // Hkv)
    return {"fwd": 4.0 * d * tile * tile * active, "bwd": 10.0 * d * tile * tile * active}
