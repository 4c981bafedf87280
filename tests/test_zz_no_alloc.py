"""fdma_fwd_noalloc: the forward for callers that cannot allocate device
memory when they call it.  Its workspace is the library's own fixed device
array, so these tests check, through the C ABI, that two calls in a row give
the same result as fdma_fwd with a caller-allocated workspace, and that a
problem too large for the array is refused before anything runs.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes
import math

import numpy as np
import pytest
import torch

from block_sparse_masked_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_MAXABS, O_RELL2, LSE_ABS = 1e-2, 5e-3, 4e-3


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_masked_02_gb300 import fdma

    fdma.load()
    return fdma


def _case(seed, N, Hq, Hkv, d, keep):
    wl = W.scaled(W.WORKLOADS["n4096_hq32_hkv8"], Nq=N, Nk=N, Hq=Hq, Hkv=Hkv, d=d, keep_window=keep,
                  scale=1 / math.sqrt(d), seed=seed)
    t = W.make_inputs(wl, device="cuda")
    return wl, t


def _noalloc_via_cabi(F, wl, t):
    """Calls fdma_fwd_noalloc directly through ctypes (no workspace attached)."""
    args = F.make_args(t["q"], t["k"], t["v"], mask=t["mask"], bias=t["bias"], causal=True, scale=wl.scale)
    assert args.workspace is None and args.workspace_bytes == 0
    out = torch.empty_like(t["q"])
    lse = torch.empty((wl.B, wl.Hq, wl.Nq), dtype=torch.float32, device="cuda")
    st = F.load().fdma_fwd_noalloc(ctypes.byref(args), out.data_ptr(), lse.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == F.FDMA_OK, F.status_string(st)
    return out, lse


def _close(a, b):
    x = a.float().cpu().numpy()
    y = b.float().cpu().numpy()
    assert np.abs(x - y).max() <= O_MAXABS
    assert np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-30) <= O_RELL2


@pytest.mark.parametrize("order", ["first", "second"])
def test_noalloc_forward_matches_fdma_fwd_on_two_calls_in_a_row(F, order):
    cases = [_case(301, 512, 8, 2, 128, 128), _case(302, 384, 4, 4, 64, 96)]
    if order == "second":
        cases = cases[::-1]
    for wl, t in cases:  # two calls in a row on the shared array, different problems
        o1, l1 = _noalloc_via_cabi(F, wl, t)
        o2, l2 = F.fwd(t["q"], t["k"], t["v"], mask=t["mask"], bias=t["bias"], causal=True, scale=wl.scale)
        torch.cuda.synchronize()
        assert F.device_error() == 0
        _close(o1, o2)
        fin = torch.isfinite(l2)
        assert torch.equal(fin, torch.isfinite(l1))
        assert (l1[fin] - l2[fin]).abs().max().item() <= LSE_ABS


def test_noalloc_refuses_a_problem_larger_than_its_array(F):
    # B * Hkv * 64 * 64 tiles = 8192 tiles -> about 33.6 MB of forward workspace > 16 MiB
    q = torch.zeros(1, 8192, 4, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 8192, 2, 64, dtype=torch.bfloat16, device="cuda")
    args = F.make_args(q, k, k, causal=True)
    assert F.workspace_size(args, False) > 16 << 20
    out = torch.empty_like(q)
    lse = torch.empty((1, 4, 8192), dtype=torch.float32, device="cuda")
    st = F.load().fdma_fwd_noalloc(ctypes.byref(args), out.data_ptr(), lse.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == F.FDMA_ERR_WORKSPACE
