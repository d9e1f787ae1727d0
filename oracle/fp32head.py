"""fp64 oracle for the FP32 variant of the linear logprob.  TEST INFRASTRUCTURE
ONLY.

"Rollout-Training Mismatch in LLM RL", section 4.3: one framework enables an
FP32 rollout LM head; section 5.2: wider arithmetic may sit beside the aligned
forward if it is validated on its own.  The pages do not spell the variant out;
the reading taken here:

* y = h * rstd * gamma with rstd = 1 / sqrt(mean(h^2) + eps), as in
  ``oracle.logprob`` but NOT rounded to bf16 (the head consumes fp32
  activations);
* W is an fp32 matrix [V, d] (fp32 master weights, or bf16 weights widened),
  taken exactly;
* z = y . W^T in fp64, then the softmax definition of ``oracle.logprob``
  (s = z / tau, lse, logprob = s_x - lse, top-1 = first arg-max of z).
"""
from __future__ import annotations

import numpy as np

from .logprob import lse_stats, widen_bf16, _top2_gap


def rmsnorm_unrounded(h: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """y = h * rstd * gamma in fp64, rstd = 1/sqrt(mean(h^2) + eps); no rounding."""
    ms = np.mean(h * h, axis=1)
    rstd = 1.0 / np.sqrt(ms + eps)
    return h * rstd[:, None] * gamma[None, :]


def oracle_logprob_fp32(hidden_bits, gamma_bits, W_f32, token_ids, temperature: float,
                        eps: float, row_block: int = 128, vocab_block: int = 8192):
    """Scores of the FP32 head.  W_f32: float32 [V, d].  Same output dict as
    oracle_logprob."""
    hidden_bits = np.asarray(hidden_bits, dtype=np.uint16)
    W = np.asarray(W_f32, dtype=np.float32)
    T = hidden_bits.shape[0]
    V = W.shape[0]
    ids = np.asarray(token_ids, dtype=np.int64)
    gamma = widen_bf16(gamma_bits)
    out = dict(logprob=np.empty(T), lse=np.empty(T), top1=np.empty(T, dtype=np.int64),
               gap=np.empty(T), zmax=np.empty(T), bad_token=(ids < 0) | (ids >= V),
               nonfinite=np.zeros(T, dtype=bool))
    for r0 in range(0, T, row_block):
        r1 = min(T, r0 + row_block)
        y = rmsnorm_unrounded(widen_bf16(hidden_bits[r0:r1]), gamma, eps)
        z = np.empty((r1 - r0, V))
        for v0 in range(0, V, vocab_block):
            z[:, v0:v0 + vocab_block] = y @ W[v0:v0 + vocab_block].astype(np.float64).T
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
