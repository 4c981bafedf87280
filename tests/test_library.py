"""Host-side checks of the C-ABI library that need no GPU: it builds, loads,
exports every entry point include/fdma.h declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re
import shutil

import pytest

from block_sparse_masked_02_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fdma.h")


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"FDMA_API\s+[\w\s\*]+?\b(fdma_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def F():
    if not os.path.exists(B.LIB) and shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no nvcc to build libfdma")
    B.build()
    from block_sparse_masked_02_gb300 import fdma

    return fdma


def test_header_declares_the_entry_points():
    assert _declared() == sorted(["fdma_workspace_size", "fdma_classify_blocks", "fdma_fwd", "fdma_bwd",
                                  "fdma_get_device_error", "fdma_status_string", "fdma_fwd_noalloc",
                                  "fdma_topk_mask"])


def test_library_exports_every_declared_symbol(F):
    lib = ctypes.CDLL(B.LIB)
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(F.EXPORTED) == set(_declared())


def test_status_strings(F):
    assert F.status_string(0) == "ok"
    assert "workspace" in F.status_string(F.FDMA_ERR_WORKSPACE)
    assert F.status_string(99) == "unknown status"


def _args(F, **kw):
    a = F.FdmaArgs()
    a.B, a.Nq, a.Nk, a.Hq, a.Hkv, a.d = 1, 256, 256, 4, 2, 128
    fake = 1 << 20  # never dereferenced: validation fails first or the size is pure arithmetic
    a.q = a.k = a.v = fake
    a.q_stride[:] = [256 * 4 * 128, 4 * 128, 128]
    a.k_stride[:] = [256 * 2 * 128, 2 * 128, 128]
    a.v_stride[:] = [256 * 2 * 128, 2 * 128, 128]
    a.scale = 0.088
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_workspace_size_arithmetic(F):
    a = _args(F)
    lib = F.load()
    fwd = lib.fdma_workspace_size(ctypes.byref(a), 0)
    bwd = lib.fdma_workspace_size(ctypes.byref(a), 1)
    tiles = 1 * 2 * 2 * 2
    assert fwd >= tiles + 2 * tiles * 128 * 16
    assert bwd >= fwd + 2 * (4 * 256 * 4) + 256 * 4 * 128 * 4
    assert lib.fdma_workspace_size(ctypes.byref(_args(F, d=100)), 0) == 0
    # d = 96 runs on the 128-wide kernels: its dQ accumulator rows are 128 floats wide
    assert lib.fdma_workspace_size(ctypes.byref(_args(F, d=96)), 1) == bwd
    assert lib.fdma_workspace_size(ctypes.byref(_args(F, Hq=3)), 0) == 0


@pytest.mark.parametrize("field,value,status", [
    ("scale", float("nan"), 1), ("scale", -1.0, 1), ("Hq", 3, 1), ("d", 100, 2), ("d", 136, 2), ("d", 36, 2), ("d", 0, 2),
    ("Nk", 0, 1), ("is_causal", 3, 1), ("is_causal", -1, 1),
    ("mask_kind", 7, 1), ("mask_kind", 1, 1), ("mask_kind", 3, 1), ("mask_kind", 4, 1), ("Hkv", 0, 1),
])
def test_argument_validation_before_any_cuda_call(F, field, value, status):
    a = _args(F, **{field: value})
    lib = F.load()
    rc = lib.fdma_fwd(ctypes.byref(a), 1 << 20, 1 << 20, None)
    assert rc == status


@pytest.mark.parametrize("d,dv,ok", [(192, 128, True), (256, 0, True), (256, 256, True), (128, 64, False),
                                     (192, 0, False), (192, 192, False), (256, 128, False), (64, 128, False)])
def test_head_dim_pairs(F, d, dv, ok):
    """(d, dv) = (192, 128) and (256, 256) have forward and backward workspace sizes (the
    backward's fp32 dQ accumulator is d wide); other unequal pairs and other widths above 128
    are refused by both entry points before any CUDA call."""
    a = _args(F, d=d, dv=dv)
    lib = F.load()
    fw, bw = lib.fdma_workspace_size(ctypes.byref(a), 0), lib.fdma_workspace_size(ctypes.byref(a), 1)
    assert (fw > 0) == ok and (bw > 0) == ok
    if ok:
        nqpad, Hq = 256, 4
        assert bw - fw >= nqpad * Hq * d * 4  # the accumulator rows are d floats
    else:
        fake = 1 << 20  # never dereferenced: the head dims are refused first
        assert lib.fdma_fwd(ctypes.byref(a), fake, fake, None) == F.FDMA_ERR_UNSUPPORTED
        assert lib.fdma_bwd(ctypes.byref(a), fake, fake, fake, fake, fake, fake, None, None) == F.FDMA_ERR_UNSUPPORTED


def test_negative_v_head_dim_is_invalid(F):
    a = _args(F, dv=-8)
    lib = F.load()
    assert lib.fdma_fwd(ctypes.byref(a), 1 << 20, 1 << 20, None) == F.FDMA_ERR_INVALID
    assert lib.fdma_workspace_size(ctypes.byref(a), 0) == 0


def test_missing_workspace_is_reported(F):
    a = _args(F)
    lib = F.load()
    assert lib.fdma_fwd(ctypes.byref(a), 1 << 20, 1 << 20, None) == F.FDMA_ERR_WORKSPACE
    assert lib.fdma_classify_blocks(ctypes.byref(a), 128, 128, None, None) == F.FDMA_ERR_WORKSPACE


@pytest.mark.parametrize("Nk,keep,kind,stride_row,status", [
    (64, 0, 1, 64, 1),        # keep_window must be >= 1
    (60, 8, 1, 64, 2),        # Nk not a multiple of 8
    (65544, 8, 1, 65544, 2),  # row longer than one CTA's shared memory
    (64, 8, 2, 64, 1),        # mask kind must be dense bf16 or uint8
    (64, 8, 1, 12, 2),        # row stride not a multiple of 8
    (64, 8, 1, 56, 1),        # rows overlap while the bias is rewritten
])
def test_topk_argument_validation_before_any_cuda_call(F, Nk, keep, kind, stride_row, status):
    lib = F.load()
    strides = (ctypes.c_int64 * 3)(4 * stride_row, 2 * stride_row, stride_row)
    rc = lib.fdma_topk_mask(1 << 20, strides, 1, 2, 2, Nk, keep, kind, 1 << 21, 1 << 20, None)
    assert rc == status


def test_pack_mask_matches_numpy_packbits(F):
    import numpy as np
    import torch
    g = torch.Generator().manual_seed(4)
    for nk in (16, 21, 130):
        m = (torch.rand(2, 3, 5, nk, generator=g) < 0.4).to(torch.bfloat16)
        pm = F.pack_mask(m)
        ref = np.packbits((m != 0).numpy(), axis=-1, bitorder="little")
        assert pm.nk == nk and np.array_equal(pm.bits.numpy(), ref)


def test_binding_refuses_cpu_tensors_and_bad_packed_masks(F):
    import torch
    bias = torch.zeros(1, 1, 4, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        F.topk_mask(bias, 4)
    q = torch.zeros(1, 128, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        F.fwd(q, q[:, :, :1], q[:, :, :1])
    with pytest.raises(ValueError):
        F.PackedMask(torch.zeros(1, 1, 4, 2, dtype=torch.int32), 16)  # not uint8
    with pytest.raises(ValueError):
        F.PackedMask(torch.zeros(1, 1, 4, 3, dtype=torch.uint8), 16)  # ceil(16/8) = 2 bytes per row
    pm = F.PackedMask(torch.zeros(1, 1, 4, 3, dtype=torch.uint8), 17)
    assert pm.nk == 17 and not pm.is_cuda


def test_causal_row_offset_is_range_checked_before_any_cuda_call(F):
    lib = F.load()
    for off, want in (((1 << 30) + 1, 1), (-(1 << 30) - 1, 1)):
        a = _args(F, is_causal=2)
        a.q_offset = off
        assert lib.fdma_fwd(ctypes.byref(a), 1 << 20, 1 << 20, None) == want
    a = _args(F, is_causal=1)
    a.q_offset = 1 << 31 - 1  # ignored unless is_causal == 2
    assert lib.fdma_workspace_size(ctypes.byref(a), 1) > 0
