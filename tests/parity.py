"""Helpers shared by the GPU parity tests: run the oracle stage by stage and
compare index sets modulo ties and outputs within the stated tolerances.

Tolerances:
* index sets: exact, except elements whose oracle value lies within
  TIE_REL * max(|theta|, TIE_FLOOR) of the k-th threshold theta (cosines are
  bounded by 1, so the magnitude of theta is floored at 1e-2: an absolute
  band of 1e-6 around thresholds that fall near zero).  The set size is exact.
* scores: SCORE_ATOL absolute.  A cosine of fp32-accumulated products of unit
  rows has at most about d * 2^-24 ~ 8e-6 of rounding for d = 128; the bf16
  hi/lo split of the pre-aggregated rows adds about 2^-17.
* attention output: max-abs 2e-2 for bf16 inputs, 1e-4 for fp32 inputs,
  against the oracle run on the GPU's own selected set.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import quoka_oracle as qo

TIE_REL = 1e-4
TIE_FLOOR = 1e-2
SCORE_ATOL = 2e-5
O_ATOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def check_index_rows(gpu_idx: np.ndarray, values: np.ndarray, k: int, largest: bool, what: str):
    """gpu_idx [rows, k'] against the oracle's `values` [rows, n]: same size, ascending, unique, in range,
    and equal to the oracle's top/bottom-k set except within the tie band of the k-th value."""
    rows, n = values.shape
    k_eff = min(k, n)
    assert gpu_idx.shape == (rows, k_eff), (what, gpu_idx.shape, (rows, k_eff))
    for r in range(rows):
        g = gpu_idx[r].astype(np.int64)
        assert np.all(np.diff(g) > 0), f"{what} row {r}: not strictly ascending"
        assert g.min() >= 0 and g.max() < n, f"{what} row {r}: out of range"
        v = values[r]
        order = np.argsort(-v if largest else v, kind="stable")
        ref = set(order[:k_eff].tolist())
        got = set(g.tolist())
        if got == ref:
            continue
        theta = v[order[k_eff - 1]]
        band = TIE_REL * max(abs(theta), TIE_FLOOR)
        diff = got.symmetric_difference(ref)
        bad = [i for i in diff if abs(v[i] - theta) > band]
        assert not bad, (f"{what} row {r}: {len(diff)} differing, {len(bad)} outside the tie band "
                         f"(theta={theta}, band={band}); e.g. {[(i, v[i]) for i in bad[:5]]}")


def oracle_query_values(Q: np.ndarray, H_kv: int, gqa: str) -> np.ndarray:
    """The value query selection ranks: per-head cosine (max) or group-averaged cosine (mean)."""
    cos = qo.query_cosines(Q)
    if gqa == "max":
        return cos
    return cos.reshape(H_kv, Q.shape[0] // H_kv, -1).mean(axis=1)


def check_output(O_gpu: torch.Tensor, O_ref: np.ndarray, what: str):
    tol = O_ATOL[O_gpu.dtype]
    err = np.max(np.abs(f64(O_gpu) - O_ref)) if O_ref.size else 0.0
    assert err <= tol, f"{what}: max-abs error {err} > {tol}"
    return err
