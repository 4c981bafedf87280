"""CPU oracle for the dynamic top-k mask built from the bias.

TEST INFRASTRUCTURE ONLY.  Only the test suite may import this module; the
product path never does.  It shares no code with the CUDA path.

Definition followed (Flash-DMA README, "Quick Start" example, the block that
builds the sparse mask from the bias before the attention call): for every
query row of a bias of shape (B, Hkv, Nq, Nk)

  * when the row is no longer than the window (Nk <= k) the mask is all ones
    and the bias is left as it is;
  * otherwise the k keys of largest bias are selected, a selected key whose
    bias equals the dtype minimum is not kept, the mask is 1 at the kept keys
    and 0 elsewhere, and the bias is replaced by the dtype minimum wherever
    the mask is 0.

The example leaves the choice among equal bias values to the top-k routine;
here equal values go to the smaller key index first, and +0 and -0 are equal
(they are equal numbers).  Values are compared as the float64 numbers the
bf16 inputs represent.
"""
from __future__ import annotations

import numpy as np

# smallest finite bf16: -(2 - 2**-7) * 2**127
BF16_MIN = -(2.0 - 2.0 ** -7) * 2.0 ** 127


def topk_row(values: np.ndarray, k: int) -> np.ndarray:
    """Boolean keep flags of one row (float64 values of the bf16 bias)."""
    n = values.shape[0]
    if n <= k:
        return np.ones(n, dtype=bool)
    # primary key: value, largest first; secondary key: key index, smallest first
    order = np.lexsort((np.arange(n), -values))
    keep = np.zeros(n, dtype=bool)
    chosen = order[:k]
    keep[chosen] = values[chosen] != BF16_MIN
    return keep


def topk_mask(bias: np.ndarray, k: int):
    """bias: float64 array (B, Hkv, Nq, Nk) of bf16 values.  Returns (keep flags
    bool (B, Hkv, Nq, Nk), bias with BF16_MIN wherever the flag is False; the
    bias unchanged when Nk <= k)."""
    bias = np.asarray(bias, dtype=np.float64)
    keep = np.empty(bias.shape, dtype=bool)
    for idx in np.ndindex(*bias.shape[:-1]):
        keep[idx] = topk_row(bias[idx], k)
    if bias.shape[-1] <= k:
        return keep, bias.copy()
    return keep, np.where(keep, bias, BF16_MIN)
