"""fp64 oracle for the FP8 (e4m3) variant of the linear logprob.  TEST
INFRASTRUCTURE ONLY.

"Rollout-Training Mismatch in LLM RL", section 3 (Unified FP8 table): forward
fake quantization feeds FP8 quantize-dequantize values to BF16 GEMMs; native
FP8 GEMMs consume FP8 codes and scales.  The pages fix neither the FP8 format
nor the scaling granularity; the readings taken here:

* format e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
  infinities): normal values 2^(e-7) (1 + m/8) for exponent fields 1..15
  (except the all-ones NaN code), subnormals 2^-6 (m/8), largest finite 448;
* quantisation rounds to nearest, ties to even, and saturates to +-448;
* one scale per row: for the activations one per token row of y (after the
  bf16 rounding of the final norm, as a BF16 model holds it), for W one per
  vocabulary row; the scale is the smallest power of two s with
  max|row| / s <= 448 (s = 1 for an all-zero row), so Q(x) = e4m3(x / s) and
  DQ = s * Q(x) exactly;
* logits z = sum_i DQ(y)_i DQ(W)_vi -- the same value native FP8 MMA produces
  from the codes when both scales are applied after accumulation -- then the
  same softmax definition as ``oracle.logprob``.

y is the RMSNorm of ``oracle.logprob``: evaluated in fp64 and rounded once to
bf16 (nearest even).

Admissible results.  An e4m3 code is an integer taken from y's bf16 value, and
that bf16 value is itself a rounding decision.  An implementation that
evaluates the RMSNorm in a narrower format (fp32) gets a value within a small
relative distance ``margin`` of the exact one; where the exact value lies that
close to a bf16 rounding midpoint, either bf16 neighbour is a correct rounding
of a correct fp32 evaluation, and when the two neighbours give different e4m3
codes (or a different row scale) the logits differ by a whole code step.
``oracle_logprob_fp8_admissible`` lists, per row, the result of every such
combination of choices.  Rounding is monotone, so the bf16 values reachable
from the interval [x - margin |x|, x + margin |x|] are exactly the roundings of
its two ends; with margin = 0 the list holds the one result of
``oracle_logprob_fp8``.  The margin is the implementation's error bound, an
input here.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

from .fp32head import rmsnorm_unrounded
from .logprob import lse_stats, rmsnorm, round_to_bf16, widen_bf16, _top2_gap

E4M3_MAX = 448.0


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value (ties to even mantissa), saturated to +-448; fp64 in/out."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # x = f 2^e, 0.5 <= |f| < 1  ->  2^(e-1) <= |x|
    unb = np.maximum(e - 1, -6)              # exponent of the leading bit, subnormal floor
    q = np.ldexp(np.ones_like(x), unb - 3)   # spacing: 3 mantissa bits
    r = np.rint(x / q) * q
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def fp8_scale(amax: float) -> float:
    """Smallest power of two s with amax / s <= 448 (1 for amax = 0)."""
    if amax == 0.0:
        return 1.0
    f, e = math.frexp(amax)                  # amax = f 2^e, 0.5 <= f < 1; 448 = 0.875 2^9
    k = e - 9 if f <= 0.875 else e - 8
    return math.ldexp(1.0, k)


def quantize_rows(x: np.ndarray):
    """Per-row scaled e4m3 values: returns (codes as fp64 values, scales)."""
    x = np.asarray(x, dtype=np.float64)
    scales = np.array([fp8_scale(float(np.max(np.abs(r)))) if r.size else 1.0 for r in x])
    codes = e4m3_round(x / scales[:, None])
    return codes, scales


def dequantized_weights(W_bits, vocab_block: int = 8192) -> np.ndarray:
    """DQ(W) in fp64 [V, d], W quantised once by vocabulary row."""
    V = W_bits.shape[0]
    Wq = np.empty((V, W_bits.shape[1]))
    for v0 in range(0, V, vocab_block):
        c, s = quantize_rows(widen_bf16(W_bits[v0:v0 + vocab_block]))
        Wq[v0:v0 + vocab_block] = c * s[:, None]
    return Wq


def _scores(z: np.ndarray, x: np.ndarray, V: int, temperature: float):
    """(logprob, lse, top1, gap, zmax) of logit rows z for target ids x."""
    s, lse = lse_stats(z, temperature)
    ok = (x >= 0) & (x < V)
    sx = np.full(z.shape[0], np.nan)
    sx[ok] = s[np.flatnonzero(ok), x[ok]]
    return sx - lse, lse, np.argmax(z, axis=1), _top2_gap(z), np.max(z, axis=1)


def oracle_logprob_fp8(hidden_bits, gamma_bits, W_bits, token_ids, temperature: float,
                       eps: float, row_block: int = 128, vocab_block: int = 8192, Wq=None):
    """Scores with FP8-quantised y and W.  Same output dict as oracle_logprob.
    ``Wq``: DQ(W) from ``dequantized_weights``, to reuse across calls."""
    hidden_bits = np.asarray(hidden_bits, dtype=np.uint16)
    T = hidden_bits.shape[0]
    V = W_bits.shape[0]
    ids = np.asarray(token_ids, dtype=np.int64)
    gamma = widen_bf16(gamma_bits)
    if Wq is None:
        Wq = dequantized_weights(W_bits, vocab_block)
    out = dict(logprob=np.empty(T), lse=np.empty(T), top1=np.empty(T, dtype=np.int64),
               gap=np.empty(T), zmax=np.empty(T), bad_token=(ids < 0) | (ids >= V),
               nonfinite=np.zeros(T, dtype=bool))
    for r0 in range(0, T, row_block):
        r1 = min(T, r0 + row_block)
        y = rmsnorm(widen_bf16(hidden_bits[r0:r1]), gamma, eps)
        cy, sy = quantize_rows(y)
        z = (cy * sy[:, None]) @ Wq.T
        res = _scores(z, ids[r0:r1], V, temperature)
        for k, v in zip(("logprob", "lse", "top1", "gap", "zmax"), res):
            out[k][r0:r1] = v
    return out


def bf16_choices(x: np.ndarray, margin: float):
    """The bf16 roundings of every value within relative distance ``margin`` of x:
    (lo, hi) arrays, equal where only one rounding is reachable.  Rounding is
    monotone, so the two ends of the interval give them all (margin < 2^-10, far
    below half a bf16 step, so the interval holds at most one midpoint)."""
    if not 0.0 <= margin < 2.0 ** -10:
        raise ValueError("margin must lie in [0, 2^-10)")
    x = np.asarray(x, dtype=np.float64)
    r = np.abs(x) * margin
    return round_to_bf16(x - r), round_to_bf16(x + r)


def _row_alternatives(x_row: np.ndarray, margin: float):
    """For one row of exact (unrounded) y values: the base bf16 row, and the
    elements whose bf16 choice can change the row's codes or its scale, each with
    its other admissible value."""
    base = round_to_bf16(x_row)
    lo, hi = bf16_choices(x_row, margin)
    amb = np.flatnonzero(lo != hi)
    if amb.size == 0:
        return base, amb, np.empty(0)
    other = np.where(lo[amb] == base[amb], hi[amb], lo[amb])
    fixed = np.ones(base.shape[0], dtype=bool)
    fixed[amb] = False
    amax_fixed = float(np.max(np.abs(base[fixed]))) if fixed.any() else 0.0
    # every row maximum a choice can produce, hence every scale
    cand = [amax_fixed] + [float(v) for v in np.abs(np.concatenate([base[amb], other]))
                           if v > amax_fixed]
    scales = sorted({fp8_scale(a) for a in cand})
    keep = np.zeros(amb.size, dtype=bool)
    for s in scales:
        keep |= e4m3_round(base[amb] / s) != e4m3_round(other / s)
    keep |= np.maximum(np.abs(base[amb]), np.abs(other)) > amax_fixed   # may set the scale
    return base, amb[keep], other[keep]


def oracle_logprob_fp8_admissible(hidden_bits, gamma_bits, W_bits, token_ids,
                                  temperature: float, eps: float, margin: float,
                                  max_choices: int = 8, Wq=None):
    """Every FP8-head result reachable from the exact y by bf16 roundings of
    values within relative distance ``margin`` (module docstring).

    Returns a list with one entry per row: a list of dicts (logprob, lse, top1,
    gap), the first being ``oracle_logprob_fp8``'s own result; or None when more
    than ``max_choices`` elements of the row are ambiguous (2^k alternatives)."""
    hidden_bits = np.asarray(hidden_bits, dtype=np.uint16)
    V = W_bits.shape[0]
    ids = np.asarray(token_ids, dtype=np.int64)
    gamma = widen_bf16(gamma_bits)
    if Wq is None:
        Wq = dequantized_weights(W_bits)
    x_all = rmsnorm_unrounded(widen_bf16(hidden_bits), gamma, eps)
    rows = []
    for t in range(hidden_bits.shape[0]):
        base, idx, other = _row_alternatives(x_all[t], margin)
        if idx.size > max_choices:
            rows.append(None)
            continue
        ys = []
        for pick in itertools.product((False, True), repeat=int(idx.size)):
            y = base.copy()
            sel = np.array(pick, dtype=bool)
            y[idx[sel]] = other[sel]
            ys.append(y)
        Y = np.stack(ys)
        cy, sy = quantize_rows(Y)
        z = (cy * sy[:, None]) @ Wq.T
        lp, lse, top1, gap, _ = _scores(z, np.full(Y.shape[0], ids[t]), V, temperature)
        rows.append([dict(logprob=float(lp[i]), lse=float(lse[i]), top1=int(top1[i]),
                          gap=float(gap[i])) for i in range(Y.shape[0])])
    return rows
