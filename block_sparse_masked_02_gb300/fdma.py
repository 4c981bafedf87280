"""ctypes binding of libfdma (include/fdma.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libfdma.so.  Tensors are torch CUDA tensors used as plain device
buffers; there is no CPU or PyTorch fallback, and calling these functions
without the compiled library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

FDMA_OK = 0
FDMA_ERR_INVALID = 1
FDMA_ERR_UNSUPPORTED = 2
FDMA_ERR_CUDA = 3
FDMA_ERR_TIMEOUT = 4
FDMA_ERR_WORKSPACE = 5

FDMA_MASK_NONE = 0
FDMA_MASK_DENSE = 1
FDMA_MASK_COLRANGES = 2
FDMA_MASK_DENSE_U8 = 3
FDMA_MASK_COLRANGES2 = 4
FDMA_MASK_BITS = 5

FDMA_FLAG_REUSE_CLASSIFICATION = 1
FDMA_FLAG_NO_SKIP = 2
FDMA_FLAG_TEST_SHORT_WAIT = 4

TILE = 128

EXPORTED = ("fdma_workspace_size", "fdma_classify_blocks", "fdma_fwd", "fdma_bwd", "fdma_get_device_error",
            "fdma_status_string", "fdma_fwd_noalloc", "fdma_topk_mask")


class FdmaArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Nq", ctypes.c_int32), ("Nk", ctypes.c_int32),
        ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("q_stride", ctypes.c_int64 * 3),
        ("k", ctypes.c_void_p), ("k_stride", ctypes.c_int64 * 3),
        ("v", ctypes.c_void_p), ("v_stride", ctypes.c_int64 * 3),
        ("mask_kind", ctypes.c_int32),
        ("mask", ctypes.c_void_p), ("mask_stride", ctypes.c_int64 * 3),
        ("colranges", ctypes.c_void_p), ("cr_stride", ctypes.c_int64 * 2),
        ("bias", ctypes.c_void_p), ("bias_stride", ctypes.c_int64 * 3),
        ("is_causal", ctypes.c_int32), ("scale", ctypes.c_float), ("flags", ctypes.c_uint32),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("q_offset", ctypes.c_int32), ("dv", ctypes.c_int32),
    ]


class FdmaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_LIB = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libfdma.so (built by __graft_entry__.build() or build.py)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libfdma.so not built ({path}); run block_sparse_masked_02_gb300/build.py")
        _build.build()
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(FdmaArgs)
    lib.fdma_workspace_size.argtypes = [P, ctypes.c_int]
    lib.fdma_workspace_size.restype = ctypes.c_size_t
    lib.fdma_classify_blocks.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.fdma_classify_blocks.restype = ctypes.c_int
    lib.fdma_fwd.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.fdma_fwd.restype = ctypes.c_int
    lib.fdma_bwd.argtypes = [P] + [ctypes.c_void_p] * 8
    lib.fdma_bwd.restype = ctypes.c_int
    lib.fdma_get_device_error.argtypes = [ctypes.c_void_p]
    lib.fdma_get_device_error.restype = ctypes.c_int
    lib.fdma_status_string.argtypes = [ctypes.c_int]
    lib.fdma_status_string.restype = ctypes.c_char_p
    lib.fdma_fwd_noalloc.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.fdma_fwd_noalloc.restype = ctypes.c_int
    lib.fdma_topk_mask.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64)] + [ctypes.c_int] * 6 + \
        [ctypes.c_void_p] * 3
    lib.fdma_topk_mask.restype = ctypes.c_int
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    return load().fdma_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libfdma takes CUDA tensors only (no CPU path)")


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


class PackedMask:
    """A bit-packed keep mask: uint8 (B, Hkv, Nq, ceil(Nk/8)), key j of a row is bit j & 7 of
    byte j >> 3 (least significant bit first), with a contiguous last dimension.  Pass it as
    `mask=` to classify_blocks / fwd / bwd."""

    def __init__(self, bits: torch.Tensor, nk: int):
        if bits.dtype != torch.uint8 or bits.dim() != 4 or bits.stride(3) != 1:
            raise ValueError("packed mask must be uint8 (B, Hkv, Nq, ceil(Nk/8)) with a contiguous last dim")
        if bits.shape[3] != -(-nk // 8):
            raise ValueError("packed mask has ceil(Nk/8) bytes per row")
        self.bits, self.nk = bits, int(nk)
        self.is_cuda = bits.is_cuda


def pack_mask(mask: torch.Tensor) -> PackedMask:
    """Bit-pack a (B, Hkv, Nq, Nk) mask (nonzero = keep) on its device."""
    B, H, Nq, Nk = mask.shape
    nb = -(-Nk // 8)
    keep = torch.zeros((B, H, Nq, nb * 8), dtype=torch.uint8, device=mask.device)
    keep[..., :Nk] = (mask != 0).to(torch.uint8)
    weights = (1 << torch.arange(8, device=mask.device, dtype=torch.int32)).to(torch.uint8)
    bits = (keep.view(B, H, Nq, nb, 8) * weights).sum(dim=-1, dtype=torch.int32).to(torch.uint8)
    return PackedMask(bits.contiguous(), Nk)


def make_args(q, k, v, *, mask=None, colranges=None, bias=None, causal=False, scale=None, workspace=None,
              flags=0, causal_offset=None) -> FdmaArgs:
    """Fill fdma_args from tensors: q (B,Nq,Hq,d), k (B,Nk,Hkv,d), v (B,Nk,Hkv,dv) with a
    contiguous head dim (dv = d, or the forward-only pairs 192 / 128 and 256 / 256); mask (B,Hkv,Nq,Nk) bf16, uint8 or bool and bias (B,Hkv,Nq,Nk) bf16 with
    contiguous columns (stride 0 broadcasts a batch or head axis); colranges int32
    (B,Hkv,Nk,2) (one masked row range per key) or (B,Hkv,Nk,4) (two).  causal=True keeps
    keys j <= i + (Nk - Nq); with causal_offset=c (an int) keys j <= i + c instead, i.e. the
    query rows are rows c - (Nk - Nq_full) ... of a longer causal problem (is_causal 2)."""
    a = FdmaArgs()
    a.B, a.Nq, a.Hq, a.d = (int(x) for x in q.shape)
    a.Nk, a.Hkv = int(k.shape[1]), int(k.shape[2])
    a.dv = int(v.shape[3])
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.stride(3) != 1:
            raise ValueError(f"{name} must be bf16 with a contiguous head dim")
        setattr(a, name, t.data_ptr())
        getattr(a, name + "_stride")[:] = [t.stride(0), t.stride(1), t.stride(2)]
    if mask is not None and colranges is not None:
        raise ValueError("pass either mask or colranges")
    if isinstance(mask, PackedMask):
        if mask.nk != a.Nk:
            raise ValueError("packed mask was built for another key length")
        a.mask_kind = FDMA_MASK_BITS
        a.mask = mask.bits.data_ptr()
        a.mask_stride[:] = [mask.bits.stride(0), mask.bits.stride(1), mask.bits.stride(2)]
    elif mask is not None:
        if mask.dtype not in (torch.bfloat16, torch.uint8, torch.bool) or mask.stride(3) != 1:
            raise ValueError("mask must be bf16, uint8 or bool with contiguous columns")
        a.mask_kind = FDMA_MASK_DENSE if mask.dtype == torch.bfloat16 else FDMA_MASK_DENSE_U8
        a.mask = mask.data_ptr()
        a.mask_stride[:] = [mask.stride(0), mask.stride(1), mask.stride(2)]
    elif colranges is not None:
        per = int(colranges.shape[3])
        if colranges.dtype != torch.int32 or per not in (2, 4) or colranges.stride(3) != 1 or \
                colranges.stride(2) != per:
            raise ValueError("colranges must be int32 with a contiguous (Nk, 2) or (Nk, 4) block per head")
        a.mask_kind = FDMA_MASK_COLRANGES if per == 2 else FDMA_MASK_COLRANGES2
        a.colranges = colranges.data_ptr()
        a.cr_stride[:] = [colranges.stride(0), colranges.stride(1)]
    else:
        a.mask_kind = FDMA_MASK_NONE
    if bias is not None:
        if bias.dtype != torch.bfloat16 or bias.stride(3) != 1:
            raise ValueError("bias must be bf16 with contiguous columns")
        a.bias = bias.data_ptr()
        a.bias_stride[:] = [bias.stride(0), bias.stride(1), bias.stride(2)]
    if causal_offset is not None:
        a.is_causal = 2
        a.q_offset = int(causal_offset)
    else:
        a.is_causal = 1 if causal else 0
    a.scale = float(scale) if scale is not None else float(a.d) ** -0.5
    a.flags = int(flags)
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def workspace_size(args: FdmaArgs, for_bwd: bool) -> int:
    return int(load().fdma_workspace_size(ctypes.byref(args), 1 if for_bwd else 0))


def alloc_workspace(args: FdmaArgs, for_bwd: bool, device) -> torch.Tensor:
    n = workspace_size(args, for_bwd)
    if n == 0:
        # invalid shape: let the entry point name the problem (no workspace attached)
        lib = load()
        st = lib.fdma_bwd(ctypes.byref(args), None, None, None, None, None, None, None, None) if for_bwd else \
            lib.fdma_fwd(ctypes.byref(args), None, None, None)
        raise FdmaError(st if st != FDMA_OK else FDMA_ERR_INVALID, "fdma_workspace_size")
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def _attach(args: FdmaArgs, ws: torch.Tensor):
    args.workspace = ws.data_ptr()
    args.workspace_bytes = ws.numel()


def _raise(status: int, where: str):
    if status != FDMA_OK:
        raise FdmaError(status, where)


def classify_blocks(q, k, v, *, mask=None, colranges=None, causal=False, workspace=None, flags=0, stream=None,
                    causal_offset=None):
    """Tile classes int8 (B, Hkv, ceil(Nq/128), ceil(Nk/128)): 0 skip, 1 partial, 2 full."""
    _check_cuda(q, k, v, mask, colranges, workspace)
    args = make_args(q, k, v, mask=mask, colranges=colranges, causal=causal, flags=flags, causal_offset=causal_offset)
    ws = workspace if workspace is not None else alloc_workspace(args, False, q.device)
    _attach(args, ws)
    B, Nq, Hkv, Nk = q.shape[0], q.shape[1], k.shape[2], k.shape[1]
    bm = torch.empty((B, Hkv, -(-Nq // TILE), -(-Nk // TILE)), dtype=torch.int8, device=q.device)
    _raise(load().fdma_classify_blocks(ctypes.byref(args), TILE, TILE, bm.data_ptr(), _stream_ptr(stream)),
           "fdma_classify_blocks")
    return bm


def topk_mask(bias, keep_window, *, mask_dtype=torch.bfloat16, fill_bias=True, inplace=False, mask=None,
              stream=None):
    """Dynamic top-k mask of a bf16 bias (B, Hkv, Nq, Nk): returns (mask, bias_out).

    mask is 1 at the keep_window largest bias entries of each row (ties: smaller key
    index; selected entries equal to the bf16 minimum are not kept), 0 elsewhere, all
    ones when Nk <= keep_window; dtype bf16 or uint8.  bias_out is the bias with the
    bf16 minimum where the mask is 0 (the bias itself when inplace, a new tensor of the
    same strides otherwise, None without fill_bias)."""
    _check_cuda(bias, mask)
    if bias.dtype != torch.bfloat16 or bias.dim() != 4 or bias.stride(3) != 1:
        raise ValueError("bias must be bf16 (B, Hkv, Nq, Nk) with a contiguous last dimension")
    if mask_dtype not in (torch.bfloat16, torch.uint8):
        raise ValueError("mask_dtype must be torch.bfloat16 or torch.uint8")
    B, Hkv, Nq, Nk = bias.shape
    if mask is None:
        mask = torch.empty((B, Hkv, Nq, Nk), dtype=mask_dtype, device=bias.device)
    elif mask.dtype != mask_dtype or tuple(mask.shape) != (B, Hkv, Nq, Nk) or not mask.is_contiguous():
        raise ValueError("mask must be a contiguous (B, Hkv, Nq, Nk) tensor of mask_dtype")
    bias_out = None
    if fill_bias:
        bias_out = bias if inplace else torch.empty_strided(bias.shape, bias.stride(), dtype=bias.dtype,
                                                             device=bias.device)
    strides = (ctypes.c_int64 * 3)(*bias.stride()[:3])
    kind = FDMA_MASK_DENSE if mask_dtype == torch.bfloat16 else FDMA_MASK_DENSE_U8
    _raise(load().fdma_topk_mask(bias.data_ptr(), strides, B, Hkv, Nq, Nk, int(keep_window), kind, mask.data_ptr(),
                                 bias_out.data_ptr() if bias_out is not None else None, _stream_ptr(stream)),
           "fdma_topk_mask")
    return mask, bias_out


def fwd(q, k, v, *, mask=None, colranges=None, bias=None, causal=False, scale=None, workspace=None, flags=0,
        out=None, lse=None, stream=None, causal_offset=None):
    """Returns (out (B,Nq,Hq,dv) bf16, lse (B,Hq,Nq) fp32)."""
    _check_cuda(q, k, v, mask, colranges, bias, workspace)
    args = make_args(q, k, v, mask=mask, colranges=colranges, bias=bias, causal=causal, scale=scale, flags=flags,
                     causal_offset=causal_offset)
    ws = workspace if workspace is not None else alloc_workspace(args, False, q.device)
    _attach(args, ws)
    B, Nq, Hq, _ = q.shape
    if out is None:
        out = torch.empty((B, Nq, Hq, v.shape[3]), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _raise(load().fdma_fwd(ctypes.byref(args), out.data_ptr(), lse.data_ptr(), _stream_ptr(stream)), "fdma_fwd")
    return out, lse


def bwd(q, k, v, out, dout, lse, *, mask=None, colranges=None, bias=None, causal=False, scale=None,
        want_dbias=True, workspace=None, flags=0, grads=None, stream=None, causal_offset=None):
    """Returns (dq, dk, dv, dbias-or-None)."""
    _check_cuda(q, k, v, out, dout, lse, mask, colranges, bias, workspace)
    for name, t in (("out", out), ("dout", dout), ("lse", lse)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    args = make_args(q, k, v, mask=mask, colranges=colranges, bias=bias, causal=causal, scale=scale, flags=flags,
                     causal_offset=causal_offset)
    ws = workspace if workspace is not None else alloc_workspace(args, True, q.device)
    _attach(args, ws)
    if grads is None:
        dq = torch.empty_like(q, memory_format=torch.contiguous_format)
        dk = torch.empty(k.shape, dtype=torch.bfloat16, device=q.device)
        dv = torch.empty(v.shape, dtype=torch.bfloat16, device=q.device)
        db = torch.empty(bias.shape, dtype=torch.bfloat16, device=q.device) if (want_dbias and bias is not None) \
            else None
    else:
        dq, dk, dv, db = grads
    _raise(load().fdma_bwd(ctypes.byref(args), out.data_ptr(), dout.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                           dk.data_ptr(), dv.data_ptr(), _ptr(db), _stream_ptr(stream)), "fdma_bwd")
    return dq, dk, dv, db


def device_error(stream=None) -> int:
    """Synchronize and return (then clear) the first kernel-side error status."""
    return int(load().fdma_get_device_error(_stream_ptr(stream)))


def fwd_noalloc(q, k, v, *, mask=None, colranges=None, bias=None, causal=False, scale=None, flags=0, out=None,
                lse=None, stream=None, causal_offset=None):
    """Forward through fdma_fwd_noalloc: the library's fixed 16 MiB device array serves as
    the workspace, so nothing is allocated for it (out and lse are allocated here only when
    not given).  Returns (out, lse)."""
    _check_cuda(q, k, v, mask, colranges, bias)
    args = make_args(q, k, v, mask=mask, colranges=colranges, bias=bias, causal=causal, scale=scale, flags=flags,
                     causal_offset=causal_offset)
    B, Nq, Hq, _ = q.shape
    if out is None:
        out = torch.empty((B, Nq, Hq, v.shape[3]), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _raise(load().fdma_fwd_noalloc(ctypes.byref(args), out.data_ptr(), lse.data_ptr(), _stream_ptr(stream)),
           "fdma_fwd_noalloc")
    return out, lse
