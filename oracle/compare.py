"""fp64 oracle for the three-way score comparison.  TEST INFRASTRUCTURE ONLY.

Three score sets for the same saved token ids ("Debugging Logprob Mismatches in
LLM Reinforcement Learning", One Response, Three Scores):

    A = generation, B = rollout prefill replay, C = frozen trainer forward.

Pairs are left minus right: A-B, B-C, A-C (same page, Check Whether the Pattern
Extends Across the Response: "keep the subtraction order explicit").

Per sequence j (rows seq_offsets[j] .. seq_offsets[j+1]-1), over its *active*
tokens (mask == 1) taken in order:

* for each pair (x, y):
  - mismatch_count: tokens whose float32 bit patterns differ (+0.0 vs -0.0
    differ; a value comparison is not a bitwise one) -- "Fault localization and
    mismatch bisect", Compare per-token logprobs;
  - first_div: ordinal (among active tokens) of the first bitwise difference,
    -1 if none -- same section (``first`` of compare_logprobs) and Per-sequence
    observation patterns (first divergence position);
  - longest_run: longest run of consecutive active ordinals that all differ --
    Per-sequence observation patterns (longest run of differences);
  - max_abs_diff = max |fp64(x) - fp64(y)|, signed_mean = mean(x - y),
    mae = mean |x - y| -- Metric measurement basis (logprob_mae) and the
    ``compare`` summary of the Debugging page (signed mean, MAE, maximum);
* with d = C - A (trainer minus rollout, "Debugging ...", What a Logprob
  Difference Means; Metric measurement basis, d = lp_train - lp_rollout):
  - mean_log_ratio = mean(C - A), mean_weight_move = mean(C - B),
    mean_same_version = mean(B - A): the exact split of eq. (1) of
    "Rollout-Training Mismatch in LLM RL" (section 1.2), with B in the role of
    p_v, C of p_k and A of q_v;
  - k3_mean = mean(expm1(d) - d): Schulman k3, exp(d) - 1 - d, evaluated with
    expm1 to avoid cancellation; overflow is flagged, never clipped (Metric
    measurement basis);
  - TIS weight w = min(exp(d), cap) -- "Rollout-Training Mismatch in LLM RL",
    section 2.1 (w_TIS = min(w, C)) and "Diagnosing Training Inference Mismatch
    in LLM Reinforcement Learning", 3. TIS (token TIS = clamp(exp(old -
    rollout), max=C), padding weights set to zero).  The clip decision is taken
    as d > ln(cap), so the integer clip count does not depend on exp();
    tis_mean = mean(w), tis_clipped = number of clipped tokens; per-token
    weights are 0 on inactive tokens.

Error contract ("Debugging ...", the ``compare`` function of Case 1: equal
shapes, binary mask with at least one active token, finite active scores;
"Fault localization ...", Compare per-token logprobs: every sequence needs at
least one valid token):  ``oracle_compare`` raises ``OracleError`` with the
name of the violated rule; ``oracle_compare_lenient`` instead reports per
sequence flags and still computes the statistics of the valid sequences.
"""
from __future__ import annotations

import math
from typing import Dict, List

import numpy as np

FLAG_EMPTY = 1
FLAG_BAD_MASK = 2
FLAG_NONFINITE = 4
FLAG_BAD_OFFSETS = 8
FLAG_K3_OVERFLOW = 16

PAIRS = (("A", "B"), ("B", "C"), ("A", "C"))


class OracleError(ValueError):
    """A violated input rule; ``.code`` names it (SHAPE, EMPTY_SEQUENCE, ...)."""

    def __init__(self, code: str, msg: str):
        super().__init__(f"{code}: {msg}")
        self.code = code


def _bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).view(np.int32)


def _longest_true_run(b: np.ndarray) -> int:
    if b.size == 0 or not b.any():
        return 0
    edges = np.diff(np.concatenate(([0], b.astype(np.int8), [0])))
    starts = np.flatnonzero(edges == 1)
    ends = np.flatnonzero(edges == -1)
    return int(np.max(ends - starts))


def _differ(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """Bitwise inequality of float32 scores (integer views, not values)."""
    return _bits(x) != _bits(y)


def _k3_terms(d: np.ndarray) -> np.ndarray:
    """Schulman k3 per token, exp(d) - 1 - d, evaluated as expm1(d) - d."""
    with np.errstate(over="ignore", invalid="ignore"):
        return np.expm1(d) - d


def _tis_weights(d: np.ndarray, tis_cap: float):
    """Token TIS weight min(exp(d), cap); the clip decision is d > ln(cap)."""
    clipped = d > math.log(tis_cap)
    w = np.full(d.shape, float(tis_cap))
    w[~clipped] = np.exp(d[~clipped])
    return w, clipped


def _pair_stats(x: np.ndarray, y: np.ndarray) -> Dict:
    differ = _differ(x, y)
    delta = x.astype(np.float64) - y.astype(np.float64)
    nz = np.flatnonzero(differ)
    return dict(
        mismatch_count=int(differ.sum()),
        first_div=int(nz[0]) if nz.size else -1,
        longest_run=_longest_true_run(differ),
        max_abs_diff=float(np.max(np.abs(delta))),
        signed_mean=float(np.mean(delta)),
        mae=float(np.mean(np.abs(delta))),
    )


def _zero_stats() -> Dict:
    z = dict(mismatch_count=0, first_div=-1, longest_run=0, max_abs_diff=0.0,
             signed_mean=0.0, mae=0.0)
    return dict(n_valid=0, pair=[dict(z) for _ in PAIRS], mean_log_ratio=0.0,
                mean_weight_move=0.0, mean_same_version=0.0, k3_mean=0.0, tis_mean=0.0,
                tis_clipped=0, flags=0)


def _seq_stats(A, B, C, tis_cap: float):
    """Statistics of one sequence's active tokens (already masked, in order)."""
    sets = dict(A=A, B=B, C=C)
    st = _zero_stats()
    st["n_valid"] = int(A.shape[0])
    st["pair"] = [_pair_stats(sets[l], sets[r]) for l, r in PAIRS]
    a, b, c = (v.astype(np.float64) for v in (A, B, C))
    d = c - a
    st["mean_log_ratio"] = float(np.mean(d))
    st["mean_weight_move"] = float(np.mean(c - b))
    st["mean_same_version"] = float(np.mean(b - a))
    st["k3_mean"] = float(np.mean(_k3_terms(d)))
    if not math.isfinite(st["k3_mean"]):
        st["flags"] |= FLAG_K3_OVERFLOW
    w, clipped = _tis_weights(d, tis_cap)
    st["tis_mean"] = float(np.mean(w))
    st["tis_clipped"] = int(clipped.sum())
    return st, w


def _active_rows(m: np.ndarray, start: int) -> np.ndarray:
    """Rows of one sequence whose mask is 1, in order (their ordinals are 0, 1, ...)."""
    return np.flatnonzero(m == 1) + start


def _check_shapes(A, B, C, seq_offsets, mask):
    for name, v in (("lp_gen", A), ("lp_replay", B), ("lp_train", C), ("mask", mask)):
        if v.ndim != 1 or v.shape != A.shape:
            raise OracleError("SHAPE", f"{name} must be 1-D with the same length as lp_gen")
    if seq_offsets.ndim != 1 or seq_offsets.shape[0] < 2:
        raise OracleError("SHAPE", "seq_offsets needs at least 2 entries")


def oracle_compare_lenient(lp_gen, lp_replay, lp_train, seq_offsets, mask, tis_cap: float):
    """Per-sequence statistics with per-sequence flags instead of exceptions.

    Returns (stats: list of dicts, tis_w: float32 [T] (NaN where no sequence
    covers the token), errors: list of error names in check order).
    """
    A = np.asarray(lp_gen, dtype=np.float32)
    B = np.asarray(lp_replay, dtype=np.float32)
    C = np.asarray(lp_train, dtype=np.float32)
    mask = np.asarray(mask)
    offs = np.asarray(seq_offsets, dtype=np.int64)
    _check_shapes(A, B, C, offs, mask)
    if not (tis_cap > 0 and math.isfinite(tis_cap)):
        raise OracleError("INVALID_ARG", "tis_cap must be positive and finite")
    T = A.shape[0]
    tis_w = np.full(T, np.nan, dtype=np.float32)
    stats: List[Dict] = []
    errors: List[str] = []
    for j in range(offs.shape[0] - 1):
        a, b = int(offs[j]), int(offs[j + 1])
        if not (0 <= a <= b <= T):
            st = _zero_stats()
            st["flags"] = FLAG_BAD_OFFSETS
            stats.append(st)
            errors.append("INVALID_ARG")
            continue
        m = mask[a:b]
        if not np.all((m == 0) | (m == 1)):
            st = _zero_stats()
            st["flags"] = FLAG_BAD_MASK
            stats.append(st)
            errors.append("BAD_MASK")
            continue
        act = _active_rows(m, a)
        if act.size == 0:
            st = _zero_stats()
            st["flags"] = FLAG_EMPTY
            tis_w[a:b] = 0.0
            stats.append(st)
            errors.append("EMPTY_SEQUENCE")
            continue
        xa, xb, xc = A[act], B[act], C[act]
        nonfinite = not (np.all(np.isfinite(xa)) and np.all(np.isfinite(xb))
                         and np.all(np.isfinite(xc)))
        with np.errstate(over="ignore", invalid="ignore"):
            st, w = _seq_stats(xa, xb, xc, tis_cap)
        if nonfinite:
            st["flags"] |= FLAG_NONFINITE
            errors.append("NONFINITE")
        tis_w[a:b] = 0.0
        tis_w[act] = w.astype(np.float32)
        stats.append(st)
    return stats, tis_w, errors


def oracle_compare(lp_gen, lp_replay, lp_train, seq_offsets, mask, tis_cap: float):
    """Strict form: raises ``OracleError`` on the first violated rule."""
    stats, tis_w, errors = oracle_compare_lenient(lp_gen, lp_replay, lp_train, seq_offsets,
                                                  mask, tis_cap)
    if errors:
        raise OracleError(errors[0], "input rule violated")
    return stats, tis_w
