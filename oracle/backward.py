"""fp64 oracle for the backward of the linear logprob.  TEST INFRASTRUCTURE ONLY.

"Rollout-Training Mismatch in LLM RL", section 5.2: the inference kernels
define the forward values and the trainer supplies the backward, through a
custom autograd wrapper around each forward operation, with gradients checked
against an independent reference; the recipe recomputes the forward instead of
saving its intermediates.  For the selected-token logprob of the "linear
logprob" path (logprob_t = s_t[x_t] - lse_t, s = z / tau, z = y . W^T; see
``oracle.logprob``) and an upstream gradient g_t = dL/dlogprob_t:

    dL/dz_tv = (g_t / tau) * (1[v = x_t] - p_tv),   p_tv = exp(s_tv - lse_t)
    dL/dy    = G . W          [T, d]
    dL/dW    = G^T . y        [V, d]

with y the bf16-rounded RMSNorm output of the forward (the GEMM operand).
Readings: a row whose token id is outside [0, V) contributes nothing (its G row
is zero; the forward reports such rows as errors); the gradient is taken with
respect to y as the GEMM consumes it.  ``rmsnorm_backward`` continues it to the
hidden states and gamma, passing the bf16 rounding of y straight through (the
usual reading for a rounding inside a differentiated forward), so a custom
autograd wrapper can return dL/dh, dL/dgamma and dL/dW.
The result dict also carries, for the parity tests, the magnitudes
|G| . |W| and |G|^T . |y| that bound how far bf16 rounding of G can move each
output element.
"""
from __future__ import annotations

import numpy as np

from .logprob import logits, lse_stats, rmsnorm, widen_bf16


def logit_grad(z: np.ndarray, token_ids, grad, temperature: float) -> np.ndarray:
    """G = dL/dz for L = sum_t grad_t * logprob_t (rows with invalid ids give zero rows)."""
    T, V = z.shape
    s, lse = lse_stats(z, temperature)
    p = np.exp(s - lse[:, None])
    ids = np.asarray(token_ids, dtype=np.int64)
    ok = (ids >= 0) & (ids < V)
    onehot = np.zeros((T, V))
    onehot[np.flatnonzero(ok), ids[ok]] = 1.0
    G = (np.asarray(grad, dtype=np.float64) / temperature)[:, None] * (onehot - p)
    G[~ok] = 0.0
    return G


def oracle_logprob_backward(hidden_bits, gamma_bits, W_bits, token_ids, temperature: float,
                            eps: float, grad_logprob, vocab_block: int = 8192, dW_rows=None):
    """Returns dict: dy [T, d], dW [V, d], bound_dy [T, d], bound_dW [V, d], y [T, d].
    With ``dW_rows`` (vocabulary ids) dW and bound_dW hold only those rows, in that order."""
    hidden_bits = np.asarray(hidden_bits, dtype=np.uint16)
    W_bits = np.asarray(W_bits, dtype=np.uint16)
    V, d = W_bits.shape
    y = rmsnorm(widen_bf16(hidden_bits), widen_bf16(gamma_bits), eps)
    z = logits(y, W_bits, vocab_block)
    G = logit_grad(z, token_ids, grad_logprob, temperature)
    del z
    T = y.shape[0]
    dy = np.zeros((T, d))
    bdy = np.zeros((T, d))
    ay = np.abs(y)
    for v0 in range(0, V, vocab_block):
        v1 = min(V, v0 + vocab_block)
        Wb = widen_bf16(W_bits[v0:v1])
        Gb = G[:, v0:v1]
        dy += Gb @ Wb
        bdy += np.abs(Gb) @ np.abs(Wb)
    rows = np.arange(V) if dW_rows is None else np.asarray(dW_rows, dtype=np.int64)
    Gr = G[:, rows]
    dW = Gr.T @ y
    bdW = np.abs(Gr).T @ ay
    return dict(dy=dy, dW=dW, bound_dy=bdy, bound_dW=bdW, y=y)


def rmsnorm_backward(h: np.ndarray, gamma: np.ndarray, eps: float, dy: np.ndarray):
    """Backward of y = h * rstd * gamma (rstd = 1/sqrt(mean(h^2) + eps)) in fp64, taking
    the bf16 rounding of y as the identity (straight through).  Returns (dh [T, d],
    dgamma [d]):

        dh_ti    = rstd_t gamma_i dy_ti - (rstd_t^3 / d) h_ti sum_j gamma_j dy_tj h_tj
        dgamma_i = sum_t dy_ti h_ti rstd_t
    """
    h = np.asarray(h, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    d = h.shape[1]
    rstd = 1.0 / np.sqrt(np.mean(h * h, axis=1) + eps)
    s = np.sum(gamma[None, :] * dy * h, axis=1)
    dh = rstd[:, None] * gamma[None, :] * dy - (rstd ** 3 / d)[:, None] * h * s[:, None]
    dgamma = np.sum(dy * h * rstd[:, None], axis=0)
    return dh, dgamma
