"""A whole attention step (classify, forward, backward) captured in one CUDA graph and
replayed: the library's calls only enqueue work on the caller's stream, so the replay gives the
eager results (dK, dV, dBias, O and lse bit for bit; dQ within the reordering of its fp32
atomics), and a replay after the inputs change in place follows the new inputs."""
import numpy as np
import pytest
import torch

from block_sparse_masked_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_masked_02_gb300 import fdma

    fdma.load()
    return fdma


def _rel(x, ref):
    x, ref = x.double(), ref.double()
    return float((x - ref).norm() / max(float(ref.norm()), 1e-30))


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 4, 2), (64, 3, 1)])
def test_step_replays_from_a_cuda_graph(F, d, Hq, Hkv):
    wl = W.scaled(W.WORKLOADS["n4096_hq32_hkv8"], Nq=640, Nk=640, Hq=Hq, Hkv=Hkv, d=d, keep_window=200,
                  scale=d ** -0.5, seed=900 + d)
    inp = W.make_inputs(wl, device="cuda")
    q, k, v, do, bias, mask = (inp[n] for n in ("q", "k", "v", "dout", "bias", "mask"))
    a = F.make_args(q, k, v, mask=mask, bias=bias, causal=True, scale=wl.scale)
    ws = F.alloc_workspace(a, True, q.device)
    out = torch.empty_like(q)
    lse = torch.empty((1, Hq, 640), dtype=torch.float32, device="cuda")
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(bias))
    R = F.FDMA_FLAG_REUSE_CLASSIFICATION
    kw = dict(mask=mask, bias=bias, causal=True, scale=wl.scale, workspace=ws)

    def step():
        F.classify_blocks(q, k, v, mask=mask, causal=True, workspace=ws)
        F.fwd(q, k, v, flags=R, out=out, lse=lse, **kw)
        F.bwd(q, k, v, out, do, lse, flags=R, grads=grads, **kw)

    def snapshot():
        return [t.clone() for t in (out, lse) + grads]

    step()
    assert F.device_error() == 0
    eager = snapshot()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on a side stream before the capture
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in (out, lse) + grads:
        t.fill_(7)
    graph.replay()
    torch.cuda.synchronize()
    assert F.device_error() == 0
    got = snapshot()
    for i in (0, 1, 3, 4, 5):  # out, lse, dk, dv, dbias
        assert torch.equal(got[i], eager[i])
    assert _rel(got[2], eager[2]) < 1e-3  # dq
    # new inputs in place: the replay follows them
    q.copy_(q.flip(1))
    step()
    torch.cuda.synchronize()
    eager2 = snapshot()
    graph.replay()
    torch.cuda.synchronize()
    assert F.device_error() == 0
    got2 = snapshot()
    assert not torch.equal(eager2[0], eager[0])
    for i in (0, 1, 3, 4, 5):
        assert torch.equal(got2[i], eager2[i])
    assert np.isfinite(_rel(got2[2], eager2[2])) and _rel(got2[2], eager2[2]) < 1e-3
