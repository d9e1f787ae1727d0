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

Precision of y.  The e4m3 code of an element of y is an integer decided from
y's bf16 value; one bf16 step of y moves that code across an e4m3 rounding
boundary with probability about 1/16, and one code step moves a logit by up to
~1e-2.  An fp64 RMSNorm and an fp32 one round a few y values per million to
different bf16 neighbours, so the code decision is taken here in fp32, the
precision the scoring kernel takes it in, with the RMSNorm reduction order
fixed and stated ("Training and rollout stop disagreeing: vime and RL-Kernel
...", Interpretation: the strict path pins the RMSNorm reduction domain, and a
fixed order is what makes a reduction batch-invariant):

* 32 partial sums; partial l adds h_i^2 for the 8-element chunks l, l+32,
  l+64, ... of the row in increasing order (each square is exact in fp32: a
  bf16 value has 8 significant bits), every addition rounded to fp32;
* the partials combine by the butterfly s_l <- s_l + s_(l xor o) for
  o = 16, 8, 4, 2, 1, rounded to fp32 (every partial ends equal);
* rstd = 1 / sqrt(s / d + eps) and y = bf16((h * rstd) * gamma), each
  operation rounded to fp32 (round to nearest even), then to bf16.

``rmsnorm_fp32`` is that computation; ``oracle_logprob_fp8(...,
y_precision="fp64")`` uses the fp64 RMSNorm of ``oracle.logprob`` instead.
"""
from __future__ import annotations

import math

import numpy as np

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


def rmsnorm_fp32(h: np.ndarray, gamma: np.ndarray, eps: float, return_rstd: bool = False):
    """y = bf16((h * rstd) * gamma) with every step in fp32 and the reduction order stated
    in the module docstring.  h, gamma: fp64 arrays holding bf16 values.  Returns y as fp64
    (and the fp32 rstd of each row with ``return_rstd``)."""
    f32 = np.float32
    h = np.asarray(h, dtype=np.float64)
    T, d = h.shape
    nvec = -(-d // 8)
    nchunk = -(-nvec // 32)
    hp = np.zeros((T, nchunk * 32 * 8))
    hp[:, :d] = h
    hp = hp.reshape(T, nchunk, 32, 8)            # [row, round, partial, element]
    part = np.zeros((T, 32), dtype=f32)
    for c in range(nchunk):
        for i in range(8):
            sq = hp[:, c, :, i] ** 2                 # exact
            part = (part.astype(np.float64) + sq).astype(f32)
    lanes = np.arange(32)
    for o in (16, 8, 4, 2, 1):
        part = part + part[:, lanes ^ o]             # fp32 additions
    ss = part[:, 0]
    rstd = f32(1.0) / np.sqrt(ss / f32(d) + f32(eps))
    y32 = (h.astype(f32) * rstd[:, None]) * np.asarray(gamma, dtype=np.float64).astype(f32)[None, :]
    y = round_to_bf16(y32.astype(np.float64))
    return (y, rstd) if return_rstd else y


def oracle_logprob_fp8(hidden_bits, gamma_bits, W_bits, token_ids, temperature: float,
                       eps: float, row_block: int = 128, vocab_block: int = 8192,
                       y_precision: str = "fp32"):
    """Scores with FP8-quantised y and W.  Same output dict as oracle_logprob."""
    if y_precision not in ("fp32", "fp64"):
        raise ValueError("y_precision must be 'fp32' or 'fp64'")
    norm = rmsnorm_fp32 if y_precision == "fp32" else rmsnorm
    hidden_bits = np.asarray(hidden_bits, dtype=np.uint16)
    T = hidden_bits.shape[0]
    V = W_bits.shape[0]
    ids = np.asarray(token_ids, dtype=np.int64)
    gamma = widen_bf16(gamma_bits)
    # W quantised once, by vocabulary row
    Wq = np.empty((V, W_bits.shape[1]))
    for v0 in range(0, V, vocab_block):
        c, s = quantize_rows(widen_bf16(W_bits[v0:v0 + vocab_block]))
        Wq[v0:v0 + vocab_block] = c * s[:, None]
    out = dict(logprob=np.empty(T), lse=np.empty(T), top1=np.empty(T, dtype=np.int64),
               gap=np.empty(T), zmax=np.empty(T), bad_token=(ids < 0) | (ids >= V),
               nonfinite=np.zeros(T, dtype=bool))
    for r0 in range(0, T, row_block):
        r1 = min(T, r0 + row_block)
        y = norm(widen_bf16(hidden_bits[r0:r1]), gamma, eps)
        cy, sy = quantize_rows(y)
        z = (cy * sy[:, None]) @ Wq.T
        s, lse = lse_stats(z, temperature)
        x = ids[r0:r1]
        ok = (x >= 0) & (x < V)
        sx = np.full(r1 - r0, np.nan)
        sx[ok] = s[np.flatnonzero(ok), x[ok]]
        out["logprob"][r0:r1] = sx - lse
        out["lse"][r0:r1] = lse
        out["top1"][r0:r1] = np.argmax(z, axis=1)
        out["zmax"][r0:r1] = np.max(z, axis=1)
        out["gap"][r0:r1] = _top2_gap(z)
    return out
