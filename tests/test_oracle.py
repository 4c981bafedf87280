"""Pins for the fp64 oracle: each test ties it to something other than itself
(finite differences, torch's SDPA library routine, brute-force loops, closed
forms, invariants and the shapes the Flash-DMA README prints)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as orc
from block_sparse_masked_02_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(seed, B=1, Nq=40, Nk=40, Hq=2, Hkv=1, d=8, causal=True, mask="dense", bias=True, density=0.5,
             scale=None, keep_diag=False, dv=None):
    g = torch.Generator().manual_seed(seed)
    dv = d if dv is None else dv
    q = torch.randn(B, Nq, Hq, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Nk, Hkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Nk, Hkv, dv, generator=g, dtype=torch.float64)
    do = torch.randn(B, Nq, Hq, dv, generator=g, dtype=torch.float64)
    bb = torch.randn(B, Hkv, Nq, Nk, generator=g, dtype=torch.float64) if bias else None
    m = cr = None
    if mask == "dense":
        m = (torch.rand(B, Hkv, Nq, Nk, generator=g) < density).to(torch.float64)
        if keep_diag:
            n = min(Nq, Nk)
            m[:, :, torch.arange(n), torch.arange(n)] = 1.0
    elif mask == "colranges":
        s = torch.randint(-3, Nq + 3, (B, Hkv, Nk), generator=g)
        ln = torch.randint(-2, Nq // 2, (B, Hkv, Nk), generator=g)
        cr = torch.stack([s, s + ln], dim=-1).to(torch.int32)
    return orc.Problem(q, k, v, bias=bb, mask=m, colranges=cr, causal=causal, scale=scale, dout=do)


def _loss(p):
    O, _ = orc.forward(p)
    return float((O * orc._f64(p.dout)).sum())


# ----------------------------------------------------------------- finite differences
@pytest.mark.parametrize("causal,mask", [(True, "dense"), (False, "dense"), (True, "colranges"), (False, None)])
def test_gradients_match_central_differences(causal, mask):
    p = _problem(7, Nq=24, Nk=20 if not causal else 24, Hq=2, Hkv=1, d=4, causal=causal, mask=mask)
    dq, dk, dv, dbias = orc.backward(p)
    h = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv), ("bias", dbias)):
        t = getattr(p, name)
        fd = np.zeros(grad.shape)
        flat = t.view(-1)
        for idx in range(flat.numel()):
            old = float(flat[idx])
            flat[idx] = old + h
            lp = _loss(p)
            flat[idx] = old - h
            lm = _loss(p)
            flat[idx] = old
            fd.reshape(-1)[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - grad).max() / max(np.abs(grad).max(), 1e-30)
        assert err < 1e-6, (name, err)


# ----------------------------------------------------------------- library routine
def _sdpa(p):
    """torch SDPA (CPU, fp64) with the mask folded into an additive float mask."""
    G = p.G
    q = p.q.permute(0, 2, 1, 3).clone().requires_grad_(True)
    k = p.k.permute(0, 2, 1, 3).clone().requires_grad_(True)
    v = p.v.permute(0, 2, 1, 3).clone().requires_grad_(True)
    bias = (p.bias if p.bias is not None else torch.zeros(p.B, p.Hkv, p.Nq, p.Nk, dtype=torch.float64))
    bias = bias.clone().requires_grad_(True)
    keep = torch.ones(p.B, p.Hkv, p.Nq, p.Nk, dtype=torch.bool)
    if p.mask is not None:
        keep = p.mask != 0
    if p.causal:
        keep = keep & torch.tril(torch.ones(p.Nq, p.Nk, dtype=torch.bool))
    am = bias.masked_fill(~keep, float("-inf")).repeat_interleave(G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1), attn_mask=am, scale=p.scale)
    (out * p.dout.permute(0, 2, 1, 3)).sum().backward()
    return (out.detach().permute(0, 2, 1, 3).numpy(), q.grad.permute(0, 2, 1, 3).numpy(),
            k.grad.permute(0, 2, 1, 3).numpy(), v.grad.permute(0, 2, 1, 3).numpy(), bias.grad.numpy())


@pytest.mark.parametrize("Hq,Hkv,causal,with_mask,dv", [(2, 1, True, True, 16), (4, 2, False, True, 16),
                                                        (4, 4, True, False, 16), (6, 2, True, True, 16),
                                                        (4, 2, True, True, 24), (2, 1, False, True, 8)])
def test_matches_torch_sdpa(Hq, Hkv, causal, with_mask, dv):
    """Against torch's SDPA, also with a V head dim other than the Q/K one (dv = 24 and 8 with
    d = 16, as the 192 / 128 configuration of the FlashMask README head-dim table)."""
    p = _problem(11, B=2, Nq=70, Nk=70, Hq=Hq, Hkv=Hkv, d=16, causal=causal,
                 mask="dense" if with_mask else None, density=0.6, keep_diag=True, scale=0.3, dv=dv)
    O, _ = orc.forward(p)
    dq, dk, dv, dbias = orc.backward(p)
    rO, rdq, rdk, rdv, rdb = _sdpa(p)
    for a, b in ((O, rO), (dq, rdq), (dk, rdk), (dv, rdv), (dbias, rdb)):
        assert np.abs(a - b).max() < 1e-10 * max(1.0, np.abs(b).max())


@pytest.mark.parametrize("Nq,Nk,offset", [(37, 70, 0), (37, 70, 20), (37, 70, -4), (40, 40, 17), (70, 37, -50)])
def test_causal_row_offset_matches_torch_tril(Nq, Nk, offset):
    """causal_offset=c keeps key j for query row i when j <= i + c: the keep set is torch's
    lower triangle with diagonal c (torch.tril), and outputs and gradients equal SDPA's on it.
    With c = Nk - Nq it is the default bottom-right rule; rows [c, c + Nq) of a square causal
    problem of length Nk see exactly these keys (one rank's rows in a context-parallel split)."""
    p = _problem(43 + offset, B=1, Nq=Nq, Nk=Nk, Hq=2, Hkv=1, d=8, causal=True, mask="dense", density=0.8, scale=0.5)
    p.causal_offset = offset
    O, lse = orc.forward(p)
    dq, dk, dv, dbias = orc.backward(p)
    keep = (p.mask != 0) & torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=offset)
    live = keep.any(dim=-1)
    q = p.q.permute(0, 2, 1, 3).clone().requires_grad_(True)
    k = p.k.permute(0, 2, 1, 3).clone().requires_grad_(True)
    v = p.v.permute(0, 2, 1, 3).clone().requires_grad_(True)
    bias = p.bias.clone().requires_grad_(True)
    am = bias.masked_fill(~keep, float("-inf")).masked_fill(~live[..., None], 0.0).repeat_interleave(p.G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(p.G, dim=1), v.repeat_interleave(p.G, dim=1), attn_mask=am, scale=p.scale)
    live_h = live.repeat_interleave(p.G, dim=1)
    (out * (p.dout.permute(0, 2, 1, 3) * live_h[..., None])).sum().backward()
    lv = live_h.permute(0, 2, 1).numpy()
    assert np.abs(O[lv] - out.detach().permute(0, 2, 1, 3).numpy()[lv]).max() < 1e-10
    assert np.all(O[~lv] == 0.0) and np.all(np.isneginf(lse.transpose(0, 2, 1)[~lv]))
    for a, b in ((dq, q.grad), (dk, k.grad), (dv, v.grad)):
        b = b.permute(0, 2, 1, 3).numpy()
        assert np.abs(a - b).max() < 1e-10 * max(1.0, np.abs(b).max())
    rdb = bias.grad.masked_fill(~live[..., None], 0.0).numpy()
    assert np.abs(dbias - rdb).max() < 1e-10 * max(1.0, np.abs(rdb).max())
    if offset == Nk - Nq:
        p.causal_offset = None
        assert np.array_equal(orc.forward(orc.Problem(p.q, p.k, p.v, bias=p.bias, mask=p.mask, causal=True,
                                                      scale=p.scale))[0], O)
    if Nq + offset <= Nk and offset >= 0:
        # the same rows inside the square problem of length Nk (rows offset .. offset + Nq)
        g = torch.Generator().manual_seed(7)
        qf = torch.randn(1, Nk, 2, 8, generator=g, dtype=torch.float64)
        qf[:, offset:offset + Nq] = p.q
        mf = torch.ones(1, 1, Nk, Nk, dtype=torch.float64)
        mf[:, :, offset:offset + Nq] = p.mask
        bf = torch.zeros(1, 1, Nk, Nk, dtype=torch.float64)
        bf[:, :, offset:offset + Nq] = p.bias
        Of, _ = orc.forward(orc.Problem(qf, p.k, p.v, bias=bf, mask=mf, causal=True, scale=p.scale))
        assert np.abs(Of[:, offset:offset + Nq] - O).max() < 1e-12


@pytest.mark.parametrize("Nq,Nk", [(37, 70), (70, 37), (64, 64)])
def test_bottom_right_causal_matches_torch_lower_right_bias(Nq, Nk):
    """Causal alignment when Nq != Nk: torch's own lower-right causal bias
    (torch.nn.attention.bias.causal_lower_right) decides which keys a row sees."""
    from torch.nn.attention.bias import causal_lower_right

    p = _problem(41, B=2, Nq=Nq, Nk=Nk, Hq=4, Hkv=2, d=8, causal=True, mask="dense", density=0.8, scale=0.4)
    O, lse = orc.forward(p)
    dq, dk, dv, dbias = orc.backward(p)
    G = p.G
    q = p.q.permute(0, 2, 1, 3).clone().requires_grad_(True)
    k = p.k.permute(0, 2, 1, 3).clone().requires_grad_(True)
    v = p.v.permute(0, 2, 1, 3).clone().requires_grad_(True)
    bias = p.bias.clone().requires_grad_(True)
    keep = (p.mask != 0) & causal_lower_right(Nq, Nk)._materialize()
    # rows with no kept key are O = 0 / no gradient in the oracle; SDPA makes them NaN, so
    # they are compared separately and their dO is zeroed for the library run
    live = keep.any(dim=-1)  # (B, Hkv, Nq)
    am = bias.masked_fill(~keep, float("-inf"))
    am = am.masked_fill(~live[..., None], 0.0).repeat_interleave(G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1), attn_mask=am, scale=p.scale)
    live_h = live.repeat_interleave(G, dim=1)  # (B, Hq, Nq)
    do = p.dout.permute(0, 2, 1, 3) * live_h[..., None]
    (out * do).sum().backward()
    rO = out.detach().permute(0, 2, 1, 3).numpy()
    lv = live_h.permute(0, 2, 1).numpy()  # (B, Nq, Hq)
    assert np.abs(O[lv] - rO[lv]).max() < 1e-10
    assert np.all(O[~lv] == 0.0) and np.all(np.isneginf(lse.transpose(0, 2, 1)[~lv]))
    if Nq > Nk:
        assert (~lv).any()  # the first Nq - Nk rows see no key
    for a, b in ((dq, q.grad.permute(0, 2, 1, 3).numpy()), (dk, k.grad.permute(0, 2, 1, 3).numpy()),
                 (dv, v.grad.permute(0, 2, 1, 3).numpy())):
        assert np.abs(a - b).max() < 1e-10 * max(1.0, np.abs(b).max())
    rdb = bias.grad.masked_fill(~live[..., None], 0.0).numpy()
    assert np.abs(dbias - rdb).max() < 1e-10 * max(1.0, np.abs(rdb).max())


def test_all_ones_mask_zero_bias_is_plain_softmax_attention():
    p = _problem(3, B=1, Nq=50, Nk=50, Hq=2, Hkv=2, d=8, causal=False, mask=None, bias=False)
    O, lse = orc.forward(p)
    q = p.q.permute(0, 2, 1, 3)
    k = p.k.permute(0, 2, 1, 3)
    v = p.v.permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=p.scale).permute(0, 2, 1, 3).numpy()
    assert np.abs(O - ref).max() < 1e-12
    ref_lse = torch.logsumexp(p.scale * q @ k.transpose(-1, -2), dim=-1).numpy()
    assert np.abs(lse - ref_lse).max() < 1e-12


# ----------------------------------------------------------------- brute force
def test_brute_force_loops():
    p = _problem(5, B=1, Nq=13, Nk=13, Hq=2, Hkv=1, d=3, causal=True, mask="dense", density=0.7, scale=0.7)
    O, lse = orc.forward(p)
    q, k, v, bias, mask = (orc._f64(x) for x in (p.q, p.k, p.v, p.bias, p.mask))
    for h in range(p.Hq):
        for i in range(p.Nq):
            scores = {}
            for j in range(p.Nk):
                if mask[0, 0, i, j] != 0 and j <= i:
                    dot = sum(q[0, i, h, t] * k[0, j, 0, t] for t in range(p.d))
                    scores[j] = p.scale * dot + bias[0, 0, i, j]
            if not scores:
                assert np.all(O[0, i, h] == 0.0) and lse[0, h, i] == -np.inf
                continue
            mx = max(scores.values())
            z = sum(math.exp(s - mx) for s in scores.values())
            for t in range(p.d):
                ref = sum(math.exp(s - mx) / z * v[0, j, 0, t] for j, s in scores.items())
                assert abs(O[0, i, h, t] - ref) < 1e-12
            assert abs(lse[0, h, i] - (mx + math.log(z))) < 1e-12


def test_top_k_mask_matches_brute_force_selection():
    g = torch.Generator().manual_seed(2)
    # coarse values force many ties; the tie-break prefers the smaller column
    bias = (torch.randint(-4, 5, (2, 3, 9, 37), generator=g).float() / 2).to(torch.bfloat16)
    mask = W.topk_mask_from_bias(bias, 10)
    for idx in np.ndindex(2, 3, 9):
        row = [float(x) for x in bias[idx]]
        order = sorted(range(37), key=lambda j: (-row[j], j))[:10]
        ref = np.zeros(37)
        ref[order] = 1.0
        assert np.array_equal(mask[idx].float().numpy(), ref)


def test_causal_topk_workload_matches_brute_force():
    wl = W.scaled(W.WORKLOADS["tiny_n256_d64"], Nq=40, Nk=40, keep_window=12, d=8, scale=0.25)
    t = W.make_inputs(wl)
    p = orc.Problem(t["q"], t["k"], t["v"], bias=t["bias"], mask=t["mask"], causal=True, scale=wl.scale)
    O, _ = orc.forward(p)
    q, k, v, bias = (orc._f64(x) for x in (t["q"], t["k"], t["v"], t["bias"]))
    raw = bias.copy()
    for h in range(wl.Hq):
        for i in range(wl.Nq):
            # keys kept: the 12 largest biases of the row (smaller index on ties), then causal
            kept = [j for j in range(wl.Nk) if t["mask"][0, 0, i, j] != 0 and j <= i]
            assert (t["mask"][0, 0, i] != 0).sum() == 12
            if not kept:
                assert np.all(O[0, i, h] == 0)
                continue
            s = np.array([wl.scale * q[0, i, h] @ k[0, j, 0] + raw[0, 0, i, j] for j in kept])
            w = np.exp(s - s.max())
            w /= w.sum()
            ref = sum(wj * v[0, j, 0] for wj, j in zip(w, kept))
            assert np.abs(O[0, i, h] - ref).max() < 1e-12


# ----------------------------------------------------------------- closed forms and conventions
def test_uniform_scores_closed_form():
    p = _problem(1, B=1, Nq=30, Nk=30, Hq=1, Hkv=1, d=5, causal=True, mask=None, bias=False)
    p.q = torch.zeros_like(p.q)
    O, lse = orc.forward(p)
    v = orc._f64(p.v)[0, :, 0]
    for i in range(30):
        assert np.abs(O[0, i, 0] - v[: i + 1].mean(axis=0)).max() < 1e-13
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-13


def test_fully_masked_and_single_key_rows():
    p = _problem(9, B=1, Nq=16, Nk=16, Hq=2, Hkv=1, d=4, causal=False, mask="dense", density=0.5)
    p.mask[0, 0, 3, :] = 0.0  # row 3: no key
    p.mask[0, 0, 5, :] = 0.0
    p.mask[0, 0, 5, 9] = 1.0  # row 5: only key 9
    O, lse = orc.forward(p)
    dq, dk, dv, dbias = orc.backward(p)
    assert np.all(O[0, 3] == 0.0) and np.all(lse[0, :, 3] == -np.inf)
    assert np.all(dq[0, 3] == 0.0) and np.all(dbias[0, 0, 3] == 0.0)
    v = orc._f64(p.v)
    for h in range(2):
        assert np.abs(O[0, 5, h] - v[0, 9, 0]).max() < 1e-15
    assert np.abs(dbias[0, 0, 5]).max() < 1e-14
    assert np.abs(dq[0, 5]).max() < 1e-14


def test_dbias_rows_sum_to_zero_and_dq_identity():
    p = _problem(4, B=2, Nq=33, Nk=33, Hq=4, Hkv=2, d=6, causal=True, mask="dense", density=0.6)
    dq, dk, dv, dbias = orc.backward(p)
    assert np.abs(dbias.sum(axis=-1)).max() < 1e-12
    # dQ_h = scale * dS_h K, and the group's dS sum is dbias: sum_h dQ_h = scale * dbias K
    k = orc._f64(p.k)
    for b in range(2):
        for g in range(2):
            lhs = dq[b, :, 2 * g:2 * g + 2].sum(axis=1)
            rhs = p.scale * dbias[b, g] @ k[b, :, g]
            assert np.abs(lhs - rhs).max() < 1e-12


def test_gqa_equals_repeated_mha():
    p = _problem(6, B=1, Nq=28, Nk=28, Hq=6, Hkv=2, d=4, causal=True, mask="dense", density=0.6)
    G = p.G
    m = orc.Problem(p.q, p.k.repeat_interleave(G, dim=2), p.v.repeat_interleave(G, dim=2),
                    bias=p.bias.repeat_interleave(G, dim=1), mask=p.mask.repeat_interleave(G, dim=1),
                    causal=True, scale=p.scale, dout=p.dout)
    O1, l1 = orc.forward(p)
    O2, l2 = orc.forward(m)
    assert np.abs(O1 - O2).max() < 1e-14 and np.array_equal(l1 == -np.inf, l2 == -np.inf)
    g1 = orc.backward(p)
    g2 = orc.backward(m)
    assert np.abs(g1[0] - g2[0]).max() < 1e-13
    for a, b, axis in ((g1[1], g2[1], 2), (g1[2], g2[2], 2)):
        summed = b.reshape(b.shape[0], b.shape[1], p.Hkv, G, b.shape[3]).sum(axis=3)
        assert np.abs(a - summed).max() < 1e-12
    db2 = g2[3].reshape(1, p.Hkv, G, 28, 28).sum(axis=2)
    assert np.abs(g1[3] - db2).max() < 1e-12


def test_colranges_equal_dense_expansion():
    p = _problem(8, B=2, Nq=45, Nk=45, Hq=2, Hkv=2, d=4, causal=True, mask="colranges")
    cr = p.colranges.long()
    i = torch.arange(p.Nq)[None, None, :, None]
    dense = (~((cr[..., 0][:, :, None, :] <= i) & (i < cr[..., 1][:, :, None, :]))).to(torch.float64)
    d = orc.Problem(p.q, p.k, p.v, bias=p.bias, mask=dense, causal=True, scale=p.scale, dout=p.dout)
    a, b = orc.forward(p), orc.forward(d)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    ga, gb = orc.backward(p), orc.backward(d)
    for x, y in zip(ga, gb):
        assert np.array_equal(x, y)
    assert np.array_equal(orc.classify_blocks(p, 8, 8), orc.classify_blocks(d, 8, 8))


def test_two_column_ranges_are_the_intersection_of_single_ranges():
    """Two masked row ranges per key column keep exactly what both single-range
    masks keep (the union of the masked ranges), and an empty second range changes
    nothing."""
    g = torch.Generator().manual_seed(17)
    B, N, Hkv = 2, 41, 2
    base = _problem(19, B=B, Nq=N, Nk=N, Hq=4, Hkv=Hkv, d=4, causal=True, mask=None)
    r = []
    for _ in range(2):
        s0 = torch.randint(-3, N + 3, (B, Hkv, N), generator=g)
        r.append(torch.stack([s0, s0 + torch.randint(-2, N // 2, (B, Hkv, N), generator=g)], dim=-1))
    cr2 = torch.cat(r, dim=-1).to(torch.int32)

    def with_cr(cr):
        return orc.Problem(base.q, base.k, base.v, bias=base.bias, colranges=cr, causal=True, scale=base.scale,
                           dout=base.dout)

    k1 = np.stack([np.stack([orc.keep_rows(with_cr(r[0].to(torch.int32)), b, h, 0, N) for h in range(Hkv)])
                   for b in range(B)])
    k2 = np.stack([np.stack([orc.keep_rows(with_cr(r[1].to(torch.int32)), b, h, 0, N) for h in range(Hkv)])
                   for b in range(B)])
    dense = orc.Problem(base.q, base.k, base.v, bias=base.bias, mask=torch.from_numpy((k1 & k2).astype(np.float64)),
                        causal=True, scale=base.scale, dout=base.dout)
    two = with_cr(cr2)
    a, b = orc.forward(two), orc.forward(dense)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    for x, y in zip(orc.backward(two), orc.backward(dense)):
        assert np.array_equal(x, y)
    assert np.array_equal(orc.classify_blocks(two, 8, 8), orc.classify_blocks(dense, 8, 8))
    empty2 = torch.cat([r[0], torch.zeros_like(r[0])], dim=-1).to(torch.int32)
    assert np.array_equal(orc.forward(with_cr(empty2))[0], orc.forward(with_cr(r[0].to(torch.int32)))[0])


def test_uint8_and_bool_masks_equal_the_bf16_mask():
    p = _problem(23, B=1, Nq=33, Nk=33, Hq=2, Hkv=1, d=4, causal=True, mask="dense", density=0.4)
    ref = orc.forward(p)
    for m in (p.mask.to(torch.uint8) * 7, p.mask != 0):
        o = orc.forward(orc.Problem(p.q, p.k, p.v, bias=p.bias, mask=m, causal=True, scale=p.scale))
        assert np.array_equal(o[0], ref[0]) and np.array_equal(o[1], ref[1])


def test_broadcast_bias_equals_the_materialised_bias():
    p = _problem(29, B=2, Nq=24, Nk=24, Hq=4, Hkv=2, d=4, causal=True, mask="dense", density=0.7)
    bb = torch.randn(1, 1, 24, 24, generator=torch.Generator().manual_seed(5), dtype=torch.float64)
    exp = bb.expand(2, 2, 24, 24)  # stride 0 over batch and heads
    a = orc.Problem(p.q, p.k, p.v, bias=exp, mask=p.mask, causal=True, scale=p.scale, dout=p.dout)
    b = orc.Problem(p.q, p.k, p.v, bias=exp.contiguous(), mask=p.mask, causal=True, scale=p.scale, dout=p.dout)
    for x, y in zip(orc.forward(a) + orc.backward(a), orc.forward(b) + orc.backward(b)):
        assert np.array_equal(x, y)


# ----------------------------------------------------------------- block map
@pytest.mark.parametrize("Nq,Nk,tm,tn,causal", [(13, 11, 4, 5, True), (17, 17, 8, 8, False), (20, 9, 3, 4, False),
                                                 (9, 20, 4, 3, True), (17, 17, 8, 8, True)])
def test_block_map_brute_force(Nq, Nk, tm, tn, causal):
    p = _problem(12, B=1, Nq=Nq, Nk=Nk, Hq=2, Hkv=2, d=2, causal=causal, mask="dense", density=0.15)
    p.mask[0, 1, :tm, :] = 1.0  # a band of full tiles
    bm = orc.classify_blocks(p, tm, tn)
    mask = orc._f64(p.mask)
    for g in range(2):
        for qt in range(bm.shape[2]):
            for kt in range(bm.shape[3]):
                kept = n = 0
                for i in range(qt * tm, min((qt + 1) * tm, Nq)):
                    for j in range(kt * tn, min((kt + 1) * tn, Nk)):
                        n += 1
                        kept += int(mask[0, g, i, j] != 0 and (not p.causal or j <= i + Nk - Nq))
                ref = 0 if kept == 0 else (2 if kept == n else 1)
                assert bm[0, g, qt, kt] == ref


def test_skipping_blocks_changes_nothing():
    """Dropping every key column that lies in a skipped tile of the row block
    gives the same output (skipped tiles contribute exactly nothing)."""
    p = _problem(13, B=1, Nq=64, Nk=64, Hq=2, Hkv=1, d=4, causal=True, mask="dense", density=0.05)
    p.mask[0, 0, :, 40:56] = 0.0
    tile = 8
    bm = orc.classify_blocks(p, tile, tile)
    assert (bm == 0).sum() > (bm.size // 2)
    O, lse = orc.forward(p)
    for qt in range(bm.shape[2]):
        cols = np.concatenate([np.arange(kt * tile, (kt + 1) * tile) for kt in range(bm.shape[3])
                               if bm[0, 0, qt, kt] != 0] or [np.zeros(0, dtype=np.int64)])
        r0, r1 = qt * tile, (qt + 1) * tile
        if cols.size == 0:
            assert np.all(O[0, r0:r1] == 0) and np.all(lse[0, :, r0:r1] == -np.inf)
            continue
        sub = orc.Problem(p.q[:, r0:r1], p.k[:, cols], p.v[:, cols], bias=p.bias[:, :, r0:r1][..., cols],
                          mask=(p.mask[:, :, r0:r1][..., cols] != 0) & (torch.from_numpy(cols)[None, :] <=
                                                                      torch.arange(r0, r1)[:, None]),
                          causal=False, scale=p.scale)
        Os, ls = orc.forward(sub)
        assert np.abs(Os - O[0:1, r0:r1]).max() < 1e-13
        assert np.array_equal(np.isneginf(ls), np.isneginf(lse[:, :, r0:r1]))


# ----------------------------------------------------------------- printed shapes
def test_quickstart_shapes_golden():
    gold = json.load(open(os.path.join(GOLDEN, "quickstart_shapes.json")))
    wl = W.WORKLOADS["tiny_n256_d64"]
    assert [wl.B, wl.Nq, wl.Hq, wl.d] == gold["output_shape"] and wl.Hkv == gold["setup"]["num_kv_heads"]
    t = W.make_inputs(wl, dout_ones=True)
    p = orc.Problem(t["q"], t["k"], t["v"], bias=t["bias"], mask=t["mask"], causal=True, scale=wl.scale,
                    dout=t["dout"])
    O, lse = orc.forward(p)
    assert list(O.shape) == gold["output_shape"]
    dq, dk, dv, dbias = orc.backward(p)
    gs = gold["grad_shapes"]
    assert [list(dq.shape), list(dk.shape), list(dv.shape), list(dbias.shape)] == \
        [gs["query"], gs["key"], gs["value"], gs["bias"]]
    assert np.isfinite(O).all()
    # the top-128 window leaves each row with exactly 128 kept keys before the causal cut
    assert bool(((t["mask"] != 0).sum(-1) == 128).all())


def test_effective_flops_counts_active_tiles():
    bm = np.array([[[[2, 0], [1, 2]]]], dtype=np.int8)
    f = orc.effective_flops(bm, Hq=4, Hkv=1, d=128)
    assert f["fwd"] == 4 * 128 * 128 * 128 * 3 * 4 and f["bwd"] == 10 * 128 * 128 * 128 * 3 * 4


def test_bit_packed_mask_equals_the_dense_mask():
    # bits packed by numpy (least significant bit first) give the same keep set, also for
    # a key length that is not a multiple of 8
    for nk in (33, 40):
        p = _problem(41, B=1, Nq=29, Nk=nk, Hq=2, Hkv=1, d=4, causal=True, mask="dense", density=0.5)
        packed = np.packbits((p.mask != 0).numpy(), axis=-1, bitorder="little")
        alt = orc.Problem(p.q, p.k, p.v, bias=p.bias, mask_bits=packed, causal=True, scale=p.scale, dout=p.dout)
        assert np.array_equal(orc.keep_rows(alt, 0, 0, 0, 29), orc.keep_rows(p, 0, 0, 0, 29))
        o, ref = orc.forward(alt), orc.forward(p)
        assert np.array_equal(o[0], ref[0]) and np.array_equal(o[1], ref[1])
