"""fp64 oracle for the selected-token ("linear") logprob.  TEST INFRASTRUCTURE ONLY.

What is computed, per row t (rows are pre-aligned: hidden row t predicts
token_ids[t]):

    rstd_t  = 1 / sqrt( (1/d) sum_i h_ti^2 + eps )                 RMSNorm
    y_ti    = bf16_round_nearest_even( h_ti * rstd_t * gamma_i )    one rounding point
    z_tv    = sum_i y_ti W_vi                                        LM head, fp64
    s_tv    = z_tv / tau                                             temperature
    lse_t   = log sum_v exp(s_tv)                                    natural log, nats
    logprob_t = s_t[x_t] - lse_t
    top1_t  = smallest v with z_tv = max_v z_tv

Sources:
* the selected-token logprob is the chosen token's logit minus the log of the
  sum of exponentiated logits over the whole vocabulary -- "Debugging Logprob
  Mismatches in LLM Reinforcement Learning", Case 2: A and B Stay Close; C
  Changes (the l_t = z_t[x_t] - log sum_v exp z_t[v] equation), and What a
  Logprob Difference Means (natural log, unit nats);
* temperature divides the logits *before* the softmax, so it changes the
  normaliser -- same page, Make Sure Both Scores Describe the Same Probability
  (score-definition table) and "How this differs from a real temperature
  mismatch";
* the normaliser runs over the true vocabulary range, merged across vocabulary
  shards -- same page, "Collect A/B and C in Your Own Run" (vocab-parallel
  normaliser), and "Training and rollout stop disagreeing: vime and RL-Kernel
  ...", Interpretation (linear logprob true vocabulary range and cross-rank LSE
  merge);
* RMSNorm with a stated reduction domain and epsilon -- "Training and rollout
  stop disagreeing ...", Interpretation (RMSNorm reduction domain and epsilon).
  The pages never write the formula; the textbook form above (eps inside the
  square root, mean over the true d) is the reading taken.
* one bf16 rounding point (y), fp32 logits never rounded: bf16 operands with
  fp32 accumulation; logits are cast to fp32 for the log-softmax ("Debugging
  Logprob Mismatches ...", trainer_scores in Collect A/B and C in Your Own Run).

Invalid token ids (outside [0, V)) give a NaN logprob for that row; lse and top1
are still reported.  Non-finite hidden values are reported in ``nonfinite``.
"""
from __future__ import annotations

import numpy as np

BF16_MAX = float.fromhex("0x1.fe00000000000p+127")


def widen_bf16(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Nearest bf16 value (ties to even) of each fp64 value, returned as fp64.

    bf16 keeps 8 significant bits.  For |x| in [2^(e-1), 2^e) the grid spacing
    is 2^(e-8); below 2^-126 (bf16 subnormals) it stays 2^-133.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    q = np.ldexp(np.ones_like(x), e - 8)
    r = np.rint(x / q) * q
    over = np.abs(r) > BF16_MAX
    if np.any(over):
        r = np.where(over, np.copysign(np.inf, x), r)
    return r


def rmsnorm(h: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """y = bf16(h * rstd * gamma), rstd = 1/sqrt(mean(h^2) + eps), all in fp64."""
    ms = np.mean(h * h, axis=1)
    rstd = 1.0 / np.sqrt(ms + eps)
    return round_to_bf16(h * rstd[:, None] * gamma[None, :])


def logits(y: np.ndarray, W_bits: np.ndarray, vocab_block: int = 8192) -> np.ndarray:
    """z = y . W^T in fp64 (W widened exactly), computed in vocabulary column blocks."""
    V = W_bits.shape[0]
    z = np.empty((y.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, vocab_block):
        v1 = min(V, v0 + vocab_block)
        z[:, v0:v1] = y @ widen_bf16(W_bits[v0:v1]).T
    return z


def lse_stats(z: np.ndarray, temperature: float):
    """s = z / tau and lse = log sum exp(s) per row (max-shifted), natural log."""
    s = z / temperature
    m = np.max(s, axis=1)
    lse = m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))
    return s, lse


def _top2_gap(z: np.ndarray) -> np.ndarray:
    if z.shape[1] < 2:
        return np.full(z.shape[0], np.inf)
    p = np.partition(z, z.shape[1] - 2, axis=1)
    return p[:, -1] - p[:, -2]


def oracle_logprob(hidden_bits, gamma_bits, W_bits, token_ids, temperature: float, eps: float,
                   row_block: int = 128):
    """Score every row.  Returns a dict of fp64 arrays:

    logprob [T], lse [T], top1 [T] (int64), gap [T] (z top-1 minus top-2),
    zmax [T], bad_token [T] (bool), nonfinite [T] (bool).
    """
    hidden_bits = np.asarray(hidden_bits, dtype=np.uint16)
    T, d = hidden_bits.shape
    V = W_bits.shape[0]
    ids = np.asarray(token_ids, dtype=np.int64)
    gamma = widen_bf16(gamma_bits)
    out = dict(logprob=np.empty(T), lse=np.empty(T), top1=np.empty(T, dtype=np.int64),
               gap=np.empty(T), zmax=np.empty(T),
               bad_token=(ids < 0) | (ids >= V), nonfinite=np.zeros(T, dtype=bool))
    for r0 in range(0, T, row_block):
        r1 = min(T, r0 + row_block)
        h = widen_bf16(hidden_bits[r0:r1])
        out["nonfinite"][r0:r1] = ~np.all(np.isfinite(h), axis=1)
        y = rmsnorm(h, gamma, eps)
        z = logits(y, W_bits)
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


def oracle_log_softmax_rows(hidden_bits, gamma_bits, W_bits, temperature: float, eps: float):
    """Full log_softmax(z / tau) rows [T, V] (small cases only; used for sum-exp checks)."""
    h = widen_bf16(hidden_bits)
    y = rmsnorm(h, widen_bf16(gamma_bits), eps)
    z = logits(y, W_bits)
    s, lse = lse_stats(z, temperature)
    return s - lse[:, None]
