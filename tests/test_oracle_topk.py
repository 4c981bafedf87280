"""Pins of the top-k mask oracle (oracle/topk.py) against brute force and the
example's own construction; CPU only."""
import numpy as np
import torch

from oracle import topk as otk
from block_sparse_masked_02_gb300 import workloads as W


def _brute(row, k):
    """Selection by repeated scans: take the largest remaining value, the
    smallest index among equal ones, k times; drop picks equal to the minimum."""
    n = len(row)
    if n <= k:
        return [True] * n
    left = list(range(n))
    keep = [False] * n
    for _ in range(k):
        best = left[0]
        for j in left[1:]:
            if row[j] > row[best]:
                best = j
        left.remove(best)
        keep[best] = row[best] != otk.BF16_MIN
    return keep


def test_bf16_min_constant():
    assert otk.BF16_MIN == float(torch.finfo(torch.bfloat16).min)


def test_matches_brute_force_with_many_ties():
    g = torch.Generator().manual_seed(5)
    vals = (torch.randint(-3, 4, (3, 2, 6, 24), generator=g).float() / 2).to(torch.bfloat16).double().numpy()
    for k in (1, 5, 11, 23):
        keep, out = otk.topk_mask(vals, k)
        for idx in np.ndindex(3, 2, 6):
            assert keep[idx].tolist() == _brute(vals[idx].tolist(), k)
            assert np.array_equal(out[idx], np.where(keep[idx], vals[idx], otk.BF16_MIN))


def test_positive_and_negative_zero_are_equal():
    row = np.array([1.0, -0.0, 0.0, -0.0, 0.0, -1.0])
    assert otk.topk_row(row, 3).tolist() == [True, True, True, False, False, False]
    row2 = np.array([0.0, -0.0, 0.0, -0.0])
    assert otk.topk_row(row2, 2).tolist() == [True, True, False, False]


def test_selected_minimum_values_are_not_kept():
    m = otk.BF16_MIN
    row = np.array([m, 2.0, m, m, 1.0, m, m, m])
    # three largest: 2.0, 1.0 and the first minimum (index 0); the minimum is not kept
    assert otk.topk_row(row, 3).tolist() == [False, True, False, False, True, False, False, False]


def test_short_rows_keep_everything_and_leave_the_bias():
    vals = np.array([[[[otk.BF16_MIN, 0.5, -2.0, 1.0]]]])
    keep, out = otk.topk_mask(vals, 4)
    assert keep.all() and np.array_equal(out, vals)
    keep, out = otk.topk_mask(vals, 9)
    assert keep.all() and np.array_equal(out, vals)


def test_kept_values_dominate_dropped_values():
    g = torch.Generator().manual_seed(8)
    vals = torch.randn((2, 64, 200), generator=g).to(torch.bfloat16).double().numpy()
    keep, _ = otk.topk_mask(vals, 37)
    for idx in np.ndindex(2, 64):
        kv, dv = vals[idx][keep[idx]], vals[idx][~keep[idx]]
        assert keep[idx].sum() == 37
        assert kv.min() >= dv.max()
        t = kv.min()  # at the threshold value the kept indices precede the dropped ones
        ki = np.flatnonzero(keep[idx] & (vals[idx] == t))
        di = np.flatnonzero(~keep[idx] & (vals[idx] == t))
        assert di.size == 0 or ki.max() < di.min()


def test_matches_the_example_construction_of_the_input_generator():
    # the generator follows the example with torch.topk on unique integer keys
    g = torch.Generator().manual_seed(11)
    bias = torch.randn((1, 2, 48, 256), generator=g).to(torch.bfloat16)
    mask = W.topk_mask_from_bias(bias, 128)
    keep, out = otk.topk_mask(bias.double().numpy(), 128)
    assert np.array_equal((mask != 0).numpy(), keep)
    filled = bias.masked_fill(mask == 0, W.BF16_MIN)
    assert np.array_equal(filled.double().numpy(), out)
