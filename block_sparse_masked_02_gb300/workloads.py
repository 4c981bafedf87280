"""Seeded synthetic inputs shared by the oracle-side tests and the GPU path.

This module only draws inputs.  It holds none of the attention arithmetic, so
both the CUDA path and the CPU oracle can consume the same tensors without
sharing any of the method's code.

Recipes (Flash-DMA README, "Quick Start" example; FlashMask README,
"Overview" / column-wise sparse representation):

* Q, K, V, dO and the bias are N(0, 1) drawn in fp32 from a seeded
  ``torch.Generator`` and rounded to bf16.
* Dynamic mask: for every query row, keep the ``keep_window`` keys with the
  largest bias (the example's ``torch.topk`` over the last dim), write 1 there
  and 0 elsewhere in the input dtype, then overwrite the bias with the dtype's
  minimum wherever the mask is 0.  When the row is no longer than the window,
  every key is kept.  Ties between equal bf16 bias values are broken by the
  smaller key index, through a unique integer key, so the mask is the same on
  every device and with every top-k implementation.
* Column ranges (FlashMask): per (batch, kv-head, key column j) one half-open
  range ``[start, end)`` of query rows that are MASKED for key j.  The causal
  document mask used here gives key j the range ``[end of j's document, N)``;
  the causal part inside the document comes from ``is_causal``.  Document
  lengths are uniform integers in [lo, hi], drawn per batch element until the
  sequence is covered; the last document is cut at N.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

BF16_MIN = torch.finfo(torch.bfloat16).min


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and mask recipe of one attention problem."""

    name: str
    B: int
    Nq: int
    Nk: int
    Hq: int
    Hkv: int
    d: int
    causal: bool
    scale: float
    mask_kind: str  # "none" | "dense" | "colranges"
    keep_window: int = 0  # dense top-k window (0: keep every key)
    has_bias: bool = True
    doc_lo: int = 512
    doc_hi: int = 8192
    seed: int = 1000

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


def _wl(name, B, N, Hq, Hkv, d, causal, mask_kind, keep_window=0, has_bias=True, seed=1000, scale=None):
    return Workload(name, B, N, N, Hq, Hkv, d, causal, scale if scale is not None else 1.0 / math.sqrt(d),
                    mask_kind, keep_window, has_bias, seed=seed)


# The five problems the method is measured on (dynamic top-k mask + bias, and the
# FlashMask causal document mask).  Seeds are 1000 + index.
WORKLOADS = {
    "tiny_n256_d64": _wl("tiny_n256_d64", 1, 256, 2, 1, 64, True, "dense", 128, seed=1000, scale=1.0 / 8.0),
    "n4096_hq32_hkv8": _wl("n4096_hq32_hkv8", 1, 4096, 32, 8, 128, True, "dense", 2048, seed=1001),
    "n16384_hq16_hkv4": _wl("n16384_hq16_hkv4", 1, 16384, 16, 4, 128, True, "dense", 2048, seed=1002),
    "n65536_hq16_hkv2": _wl("n65536_hq16_hkv2", 1, 65536, 16, 2, 128, True, "dense", 4096, seed=1003),
    "docmask_b2_n32768": Workload("docmask_b2_n32768", 2, 32768, 32768, 32, 8, 128, True, 1.0 / math.sqrt(128),
                                  "colranges", 0, False, seed=1004),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, gen, device, chunk_rows: int = 0) -> torch.Tensor:
    """N(0,1) in fp32 rounded to bf16.  With chunk_rows > 0 the leading dims are
    flattened and drawn in row chunks (bounds the fp32 temporary)."""
    if chunk_rows <= 0:
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    out = torch.empty(shape, device=device, dtype=torch.bfloat16)
    flat = out.view(-1, shape[-1])
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(r0 + chunk_rows, flat.shape[0])
        flat[r0:r1] = torch.randn((r1 - r0, shape[-1]), generator=gen, device=device,
                                  dtype=torch.float32).to(torch.bfloat16)
    return out


def _topk_keys(bias_rows: torch.Tensor) -> torch.Tensor:
    """Unique int32 ordering key per element: larger bias first, then smaller
    column index.  bias_rows is bf16 (..., Nk) with Nk <= 65536."""
    nk = bias_rows.shape[-1]
    assert nk <= 65536
    bits = bias_rows.contiguous().view(torch.int16).to(torch.int64) & 0xFFFF
    ordered = torch.where((bits & 0x8000) != 0, (~bits) & 0xFFFF, bits | 0x8000)
    col = torch.arange(nk, device=bias_rows.device, dtype=torch.int64)
    key = ordered * 65536 + (65535 - col) - (1 << 31)
    return key.to(torch.int32)


def topk_mask_from_bias(bias: torch.Tensor, keep_window: int, chunk_rows: int = 256) -> torch.Tensor:
    """Return the bf16 0/1 keep-mask (same shape as bias) selecting, per query
    row, the keep_window largest bias entries (ties: smaller key index)."""
    nk = bias.shape[-1]
    mask = torch.zeros_like(bias)
    if keep_window <= 0 or nk <= keep_window:
        mask.fill_(1.0)
        return mask
    flat_b = bias.view(-1, nk)
    flat_m = mask.view(-1, nk)
    for r0 in range(0, flat_b.shape[0], chunk_rows):
        r1 = min(r0 + chunk_rows, flat_b.shape[0])
        rows = flat_b[r0:r1]
        idx = torch.topk(_topk_keys(rows), keep_window, dim=-1, largest=True, sorted=False).indices
        vals = torch.gather(rows, -1, idx)
        valid = (vals != BF16_MIN).to(torch.bfloat16)
        flat_m[r0:r1].scatter_(-1, idx, valid)
    return mask


def doc_colranges(B: int, Hkv: int, N: int, lo: int, hi: int, seed: int, device="cpu") -> torch.Tensor:
    """int32 (B, Hkv, N, 2): key j's masked query rows [end of its document, N)."""
    g = _gen("cpu", seed)
    out = torch.empty((B, Hkv, N, 2), dtype=torch.int32)
    for b in range(B):
        ends = torch.empty(N, dtype=torch.int32)
        pos = 0
        while pos < N:
            length = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
            e = min(pos + length, N)
            ends[pos:e] = e
            pos = e
        out[b, :, :, 0] = ends
        out[b, :, :, 1] = N
    return out.to(device)


def make_inputs(wl: Workload, device="cpu", seed: Optional[int] = None, dout_ones: bool = False) -> dict:
    """Draw every input of workload `wl` on `device`.

    Returns q, k, v, dout (bf16, BSHD), bias (bf16 (B,Hkv,Nq,Nk) or None),
    mask (bf16 (B,Hkv,Nq,Nk) or None), colranges (int32 (B,Hkv,Nk,2) or None).
    """
    seed = wl.seed if seed is None else seed
    g = _gen(device, seed)
    q = _randn_bf16((wl.B, wl.Nq, wl.Hq, wl.d), g, device)
    k = _randn_bf16((wl.B, wl.Nk, wl.Hkv, wl.d), g, device)
    v = _randn_bf16((wl.B, wl.Nk, wl.Hkv, wl.d), g, device)
    dout = torch.ones_like(q) if dout_ones else _randn_bf16((wl.B, wl.Nq, wl.Hq, wl.d), g, device)
    bias = mask = colranges = None
    need_bias = wl.has_bias or wl.mask_kind == "dense"
    if need_bias:
        bias = _randn_bf16((wl.B, wl.Hkv, wl.Nq, wl.Nk), g, device, chunk_rows=4096)
    if wl.mask_kind == "dense":
        mask = topk_mask_from_bias(bias, wl.keep_window)
        bias.masked_fill_(mask == 0, BF16_MIN)
    elif wl.mask_kind == "colranges":
        colranges = doc_colranges(wl.B, wl.Hkv, wl.Nk, wl.doc_lo, wl.doc_hi, seed, device)
    if not wl.has_bias:
        bias = None
    return dict(q=q, k=k, v=v, dout=dout, bias=bias, mask=mask, colranges=colranges)


def scaled(wl: Workload, **kw) -> Workload:
    """Copy of `wl` with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(wl, **kw)
