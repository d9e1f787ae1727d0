"""fp64 oracle for the extended per-sequence mismatch diagnostics.  TEST
INFRASTRUCTURE ONLY.

Same roles and masking as ``oracle.compare`` (A generation, B replay, C trainer;
pairs A-B, B-C, A-C left minus right; active tokens only; d = C - A).  Per
valid sequence:

* |left - right| quantiles p50 / p95 / p99 for each pair -- "Diagnosing Training
  Inference Mismatch in LLM Reinforcement Learning", 5. practical indicators
  (abs(delta_logprob) p50 / p95 / p99 / max), and the p95 / p99 of the
  ``compare`` summary of "Debugging Logprob Mismatches ...", Case 1.  Linear
  interpolation between order statistics (Hyndman-Fan type 7):
  h = (n - 1) q,  Q = x[floor h] + (h - floor h) (x[floor h + 1] - x[floor h]),
  x sorted ascending.
* probability MAE per pair: mean |exp(left) - exp(right)| -- "Fault localization
  and mismatch bisect", Metric measurement basis (probability_mae).
* top-1 flips per pair: active tokens whose top-1 ids differ -- 5. practical
  indicators (top-1 token flip rate); -1 when the top-1 ids are not supplied.
* sequence-accumulated mismatch: sum of d, k1_sum = sum of -d (k1 = -log r with
  r = exp(d)), k3_sum = sum of expm1(d) - d -- "Diagnosing ...", 3. TIS (sequence
  rejection by sum_t K1(r_corr) or sum_t K3(r_corr)); reading: K1(r) = -log r,
  K3(r) = r - 1 - log r, the estimators of KL(rollout || trainer) on samples
  from the rollout.
* sequence TIS weight: min(exp(sum d), cap) -- same section (sequence TIS),
  clip decided as sum d > ln(cap).
* ratio error: mean |exp(d) - 1| -- 5. practical indicators (PPO ratio error
  exp(delta_logprob)); evaluated as |expm1(d)|.
* MIS: w = exp(d); kept tokens satisfy lo <= w <= hi (decided as
  ln(lo) <= d <= ln(hi)); mis_mean = mean of w over all active tokens with the
  dropped ones counted as 0 -- "Rollout-Training Mismatch in LLM RL", section
  2.1 (w_MIS = w 1[l <= w <= u]).
* w2_mean = mean exp(2 d): the ratio-only second moment E_q[w^2] = exp D_2(p||q)
  -- "Rollout-Training Mismatch in LLM RL", section 5.3 (eq. 10 context).

Flags follow ``oracle.compare``.  The quantiles are defined, and computed here,
for a sequence of any length.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

from .compare import (FLAG_BAD_MASK, FLAG_BAD_OFFSETS, FLAG_EMPTY, FLAG_K3_OVERFLOW,
                      FLAG_NONFINITE, PAIRS, OracleError, _check_shapes)

QUANTILES = (0.5, 0.95, 0.99)


def quantile_linear(x: np.ndarray, q: float) -> float:
    """Type-7 quantile: linear interpolation between the order statistics of x."""
    xs = np.sort(np.asarray(x, dtype=np.float64))
    n = xs.shape[0]
    h = (n - 1) * q
    lo = int(math.floor(h))
    hi = min(lo + 1, n - 1)
    return float(xs[lo] + (h - lo) * (xs[hi] - xs[lo]))


def _prob_mae(left: np.ndarray, right: np.ndarray) -> float:
    """mean |exp(left) - exp(right)| (fp64)."""
    return float(np.mean(np.abs(np.exp(left) - np.exp(right))))


def _seq_tis(log_ratio_sum: float, tis_cap: float) -> float:
    """Sequence TIS weight min(exp(sum d), cap), clip decided as sum d > ln(cap)."""
    return float(tis_cap) if log_ratio_sum > math.log(tis_cap) else math.exp(log_ratio_sum)


def _mis(d: np.ndarray, lo: float, hi: float):
    """MIS weights w 1[lo <= w <= hi] with w = exp(d); returns (sum of kept w, kept count)."""
    kept = (d >= math.log(lo)) & (d <= math.log(hi))
    return float(np.sum(np.exp(d[kept]))), int(kept.sum())


def _empty_diag(flags: int) -> Dict:
    return dict(n_valid=0, abs_q50=[0.0] * 3, abs_q95=[0.0] * 3, abs_q99=[0.0] * 3,
                prob_mae=[0.0] * 3, top1_flips=[-1] * 3, log_ratio_sum=0.0, k1_sum=0.0,
                k3_sum=0.0, seq_tis=0.0, ratio_err_mean=0.0, mis_mean=0.0, mis_kept=0,
                w2_mean=0.0, flags=flags)


def _seq_diag(sets, tops, tis_cap, mis_lo, mis_hi) -> Dict:
    A, B, C = (sets[k].astype(np.float64) for k in "ABC")
    n = A.shape[0]
    st = _empty_diag(0)
    st["n_valid"] = n
    f64 = dict(A=A, B=B, C=C)
    for p, (l, r) in enumerate(PAIRS):
        a = np.abs(f64[l] - f64[r])
        st["abs_q50"][p], st["abs_q95"][p], st["abs_q99"][p] = (
            quantile_linear(a, q) for q in QUANTILES)
        st["prob_mae"][p] = _prob_mae(f64[l], f64[r])
        if tops[l] is not None and tops[r] is not None:
            st["top1_flips"][p] = int(np.sum(tops[l] != tops[r]))
    d = C - A
    with np.errstate(over="ignore", invalid="ignore"):
        st["log_ratio_sum"] = float(np.sum(d))
        st["k1_sum"] = float(np.sum(-d))
        st["k3_sum"] = float(np.sum(np.expm1(d) - d))
        st["seq_tis"] = _seq_tis(st["log_ratio_sum"], tis_cap)
        st["ratio_err_mean"] = float(np.mean(np.abs(np.expm1(d))))
        kept_sum, st["mis_kept"] = _mis(d, mis_lo, mis_hi)
        st["mis_mean"] = kept_sum / n
        st["w2_mean"] = float(np.mean(np.exp(2.0 * d)))
    if not math.isfinite(st["k3_sum"]):
        st["flags"] |= FLAG_K3_OVERFLOW
    return st


def oracle_diag_lenient(lp_gen, lp_replay, lp_train, seq_offsets, mask, tis_cap: float,
                        mis_lo: float, mis_hi: float,
                        top1: Sequence[Optional[np.ndarray]] = (None, None, None)):
    """Per-sequence diagnostics with per-sequence flags (statistics of flagged
    BAD_OFFSETS / BAD_MASK / EMPTY sequences are zero).  Returns (diags, errors)."""
    A = np.asarray(lp_gen, dtype=np.float32)
    B = np.asarray(lp_replay, dtype=np.float32)
    C = np.asarray(lp_train, dtype=np.float32)
    mask = np.asarray(mask)
    offs = np.asarray(seq_offsets, dtype=np.int64)
    _check_shapes(A, B, C, offs, mask)
    if not (tis_cap > 0 and math.isfinite(tis_cap)):
        raise OracleError("INVALID_ARG", "tis_cap must be positive and finite")
    if not (0 < mis_lo <= mis_hi and math.isfinite(mis_hi)):
        raise OracleError("INVALID_ARG", "need 0 < mis_lo <= mis_hi < inf")
    tops = {k: (None if t is None else np.asarray(t, dtype=np.int64))
            for k, t in zip("ABC", top1)}
    T = A.shape[0]
    out: List[Dict] = []
    errors: List[str] = []
    for j in range(offs.shape[0] - 1):
        a, b = int(offs[j]), int(offs[j + 1])
        if not (0 <= a <= b <= T):
            out.append(_empty_diag(FLAG_BAD_OFFSETS))
            errors.append("INVALID_ARG")
            continue
        m = mask[a:b]
        if not np.all((m == 0) | (m == 1)):
            out.append(_empty_diag(FLAG_BAD_MASK))
            errors.append("BAD_MASK")
            continue
        act = np.flatnonzero(m == 1) + a
        if act.size == 0:
            out.append(_empty_diag(FLAG_EMPTY))
            errors.append("EMPTY_SEQUENCE")
            continue
        sets = dict(A=A[act], B=B[act], C=C[act])
        sub_tops = {k: (None if t is None else t[act]) for k, t in tops.items()}
        st = _seq_diag(sets, sub_tops, tis_cap, mis_lo, mis_hi)
        if not all(np.all(np.isfinite(v)) for v in sets.values()):
            st["flags"] |= FLAG_NONFINITE
            errors.append("NONFINITE")
        out.append(st)
    return out, errors


def oracle_diag(*args, **kw):
    """Strict form: raises ``OracleError`` on the first violated rule."""
    out, errors = oracle_diag_lenient(*args, **kw)
    if errors:
        raise OracleError(errors[0], "input rule violated")
    return out
