"""Helpers that compare the CUDA library's results with the CPU oracle.

Selection rule (per unit): let s_k and s_{k+1} be the oracle's k-th and
(k+1)-th candidate scores. If s_k - s_{k+1} >= 1e-3 * max(|s_k|, 1e-30) the GPU
set must equal the oracle set exactly. Otherwise the unit is a near-tie: the
GPU set must hold every candidate scoring above s_k + band, only candidates
scoring at least s_k - band, the forced block, and exactly as many scored
blocks as the oracle.

Attention outputs are compared with the oracle attending over the GPU's own
(validated) selection: bf16 max-abs <= 2e-2, fp32 |d| <= 1e-3 * max(1, |ref|).

Pooled summaries: the oracle sums a block's 64 keys in double and rounds the
mean once into the storage type; the library sums in fp32. bf16 summaries must
be within one bf16 step of the oracle's (the count of one-step differences is
reported); fp32 summaries within the error bound of a 64-term fp32 sum
(63 * 2^-24 * mean|K|) plus one rounding of the result.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import msa_oracle as O

REL_GAP = 1e-3
BF16_ABS = 2e-2
BF16_REL_RMS = 1e-2
F32_REL = 1e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


class SelectionStats:
    def __init__(self):
        self.units = 0
        self.near_ties = 0

    def __repr__(self):
        return f"SelectionStats(units={self.units}, near_ties={self.near_ties})"


# Parity counts of the full-size cases (near-ties at the selection boundary,
# summary elements one bf16 step from the oracle's), printed at the end of the
# pytest session by tests/conftest.py.
REPORT: list = []


def record(name: str, **counts) -> None:
    REPORT.append((name, counts))


class PoolStats:
    """Summary elements compared and how many differ from the oracle's (by at
    most one bf16 step, or within the fp32 summation bound)."""

    def __init__(self):
        self.elements = 0
        self.differ = 0

    def __repr__(self):
        return f"PoolStats(elements={self.elements}, differ={self.differ})"


def bf16_step(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 values at |x| (8 significant bits; 2^-133 below the
    normal range)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    step = np.exp2(e - 7)
    return np.where(a >= 2.0 ** -126, step, 2.0 ** -133)


def check_pooled(got: np.ndarray, stored: np.ndarray, exact: np.ndarray, store: str, k_rows=None,
                 stats: PoolStats | None = None, what: str = "pooled keys") -> int:
    """Compare the library's summaries of one unit ([n, D]) with the oracle's
    (stored and exact). Returns the number of elements that differ."""
    got = np.asarray(got, dtype=np.float64)
    stored = np.asarray(stored, dtype=np.float64)
    assert got.shape == stored.shape, f"{what}: shape {got.shape} vs {stored.shape}"
    d = np.abs(got - stored)
    if store == "bf16":
        assert (d <= bf16_step(stored)).all(), f"{what}: more than one bf16 step from the oracle"
    else:
        n = stored.shape[0]
        kr = np.asarray(k_rows[: n * 64], dtype=np.float64).reshape(n, 64, -1)
        bound = 63 * 2.0 ** -24 * np.abs(kr).mean(axis=1) + 2.0 ** -24 * np.abs(exact)
        assert (np.abs(got - exact) <= bound).all(), f"{what}: beyond the fp32 summation bound"
    differ = int((d > 0).sum())
    if stats is not None:
        stats.elements += int(d.size)
        stats.differ += differ
    return differ


def check_selection(gpu_row: np.ndarray, scores: np.ndarray, k_scored: int, forced, k_total: int,
                    stats: SelectionStats | None = None, needles=()) -> bool:
    """Validate one unit's GPU index row against the oracle scores. Returns
    True when the unit was a near-tie."""
    gpu_row = np.asarray(gpu_row).astype(np.int64)
    n = scores.shape[0]
    k = min(k_scored, n)
    want_len = k + (1 if forced is not None else 0)
    got = [int(b) for b in gpu_row if b >= 0]
    assert all(b == -1 for b in gpu_row[len(got):]), f"padding must be trailing -1: {gpu_row}"
    assert len(got) == want_len, f"expected {want_len} blocks, got {len(got)}: {gpu_row}"
    assert got == sorted(got) and len(set(got)) == len(got), f"not sorted/unique: {got}"
    scored = [b for b in got if b != forced] if forced is not None else list(got)
    if forced is not None:
        assert forced in got, f"forced block {forced} missing"
    assert len(scored) == k, f"{len(scored)} scored blocks, expected {k}"
    assert all(0 <= b < n for b in scored), f"non-candidate selected: {scored} (n={n})"
    for b in needles:
        assert b in got, f"needle block {b} not selected"
    if stats is not None:
        stats.units += 1
    oracle_sel = O.select_blocks(scores, k_scored, forced, k_total)
    gap = O.boundary_gap(scores, k_scored)
    if gap is None:
        assert list(gpu_row) == list(oracle_sel)
        return False
    s_k, s_k1 = gap
    band = REL_GAP * max(abs(s_k), 1e-30)
    if s_k - s_k1 >= band:
        assert list(gpu_row) == list(oracle_sel), f"selection differs:\n gpu {list(gpu_row)}\n ora {list(oracle_sel)}"
        return False
    sc = np.asarray(scores)
    must = set(np.nonzero(sc > s_k + band)[0].tolist())
    assert must <= set(scored), "a block clearly above the k-th score is missing"
    assert all(sc[b] >= s_k - band for b in scored), "a block clearly below the k-th score was kept"
    if stats is not None:
        stats.near_ties += 1
    return True


def check_output(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "output") -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    info = dict(max_abs=float(d.max()) if d.size else 0.0, rms_ref=rms)
    if dtype == "bf16":
        assert info["max_abs"] <= BF16_ABS, f"{what}: max-abs {info['max_abs']:.3e} > {BF16_ABS}"
        if rms > 0:
            assert info["max_abs"] / rms <= BF16_REL_RMS * 10, f"{what}: max-abs/rms {info['max_abs'] / rms:.3e}"
            info["rel_rms_err"] = float(np.sqrt(np.mean(d ** 2))) / rms
            assert info["rel_rms_err"] <= BF16_REL_RMS, f"{what}: rms error {info['rel_rms_err']:.3e} of rms(ref)"
    else:
        lim = F32_REL * np.maximum(1.0, np.abs(ref))
        bad = d > lim
        assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond 1e-3 relative (max {d.max():.3e})"
    return info


def check_lse(got: np.ndarray, ref: np.ndarray, what="lse") -> None:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got)), f"{what}: finiteness differs"
    d = np.abs(got[fin] - ref[fin])
    assert (d <= 1e-3 * np.maximum(1.0, np.abs(ref[fin]))).all(), f"{what}: max diff {d.max():.3e}"


SCALE = 1.0 / math.sqrt(128)
