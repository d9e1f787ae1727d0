"""fp64 oracle for the processed (top-k / top-p filtered) selected-token logprob.
TEST INFRASTRUCTURE ONLY.

"Debugging Logprob Mismatches in LLM Reinforcement Learning", Make Sure Both
Scores Describe the Same Probability: the sampling (behaviour) score is taken
on the distribution actually used after filters and processors; top-k with
k = 2 turns (0.50, 0.30, 0.20) into (0.625, 0.375, 0) -- the kept tokens are
renormalised, the others get probability 0.  "Fault localization and mismatch
bisect", Metric measurement basis: processed scores need the same temperature,
truncation and penalty settings on both sides.

Readings (the pages give the top-k example only):
* order: temperature, then top-k, then top-p on the renormalised top-k
  distribution;
* top-k keeps the k tokens with the largest logits; equal logits are ordered
  by the lower token id;
* top-p keeps, in that order, every token whose preceding cumulative
  probability is < p (the smallest prefix with mass >= p; the first token is
  always kept);
* processed logprob = s_x - log sum_{v kept} exp(s_v) for a kept target,
  -inf for a filtered-out target (probability 0), with s = z / tau.

``process_head`` gives the sampler's top-k head of a row (ids and processed
logprobs), the support a sampler-expected score is taken over ("Rollout-Training
Mismatch in LLM RL", section 4.3: the reference implementation of score
centering stores a top-k head).

Per row the oracle also reports the decision margins used by the parity
tests: ``gap_k`` = z_(k) - z_(k+1) (the logit gap at the top-k boundary) and
``margin_p`` = the distance of the top-p cumulative sums next to the cut from p,
``rank_gap`` = the smallest logit gap between neighbours inside the top-k head.
"""
from __future__ import annotations

import math

import numpy as np

from .logprob import logits, rmsnorm, widen_bf16


def process_head(z: np.ndarray, temperature: float, top_k: int, top_p: float):
    """The sampler's top-k head of one row of fp64 logits: the min(top_k, V) token ids in
    top-k order (logit descending, lower id first on ties) and their processed logprobs
    (log of the renormalised top-k / top-p distribution; -inf where top-p removed the
    token).  The support that a sampler-expected score is taken over."""
    V = z.shape[0]
    order = np.lexsort((np.arange(V), -z))
    top = order[:min(top_k, V)]
    s = z[top] / temperature
    m = s[0]
    e = np.exp(s - m)
    q = e / np.sum(e)
    before = np.concatenate(([0.0], np.cumsum(q)[:-1]))
    keep = before < top_p
    keep[0] = True
    lse = m + math.log(float(np.sum(np.exp(s[keep] - m))))
    return top.astype(np.int64), np.where(keep, s - lse, -math.inf)


def process_row(z: np.ndarray, x: int, temperature: float, top_k: int, top_p: float):
    """Processed score of token x for one row of fp64 logits z."""
    V = z.shape[0]
    order = np.lexsort((np.arange(V), -z))          # z descending, then id ascending
    k = min(top_k, V)
    top = order[:k]
    s = z[top] / temperature
    m = s[0]
    e = np.exp(s - m)
    q = e / np.sum(e)                                # renormalised top-k distribution
    before = np.concatenate(([0.0], np.cumsum(q)[:-1]))
    keep = before < top_p
    keep[0] = True
    kept = top[keep]
    sk = s[keep]
    lse = m + math.log(float(np.sum(np.exp(sk - m))))
    gap_k = float(z[order[k - 1]] - z[order[k]]) if k < V else math.inf
    margin_p = float(np.min(np.abs(before - top_p))) if top_p < 1.0 else math.inf
    if x in set(int(v) for v in kept):
        lp = float(z[x] / temperature - lse)
    else:
        lp = -math.inf
    return lp, lse, int(kept.shape[0]), gap_k, margin_p


def oracle_processed_logprob(hidden_bits, gamma_bits, W_bits, token_ids, temperature: float,
                             eps: float, top_k: int, top_p: float, row_block: int = 64):
    """Processed logprob of every row.  Returns dict of arrays: logprob, lse_kept, kept,
    gap_k, margin_p."""
    hidden_bits = np.asarray(hidden_bits, dtype=np.uint16)
    T = hidden_bits.shape[0]
    gamma = widen_bf16(gamma_bits)
    V = np.asarray(W_bits).shape[0]
    kk = min(top_k, V)
    out = dict(logprob=np.empty(T), lse_kept=np.empty(T), kept=np.empty(T, dtype=np.int64),
               gap_k=np.empty(T), margin_p=np.empty(T),
               topk_ids=np.empty((T, kk), dtype=np.int64), topk_logprob=np.empty((T, kk)),
               rank_gap=np.empty(T))
    ids = np.asarray(token_ids, dtype=np.int64)
    for r0 in range(0, T, row_block):
        r1 = min(T, r0 + row_block)
        y = rmsnorm(widen_bf16(hidden_bits[r0:r1]), gamma, eps)
        z = logits(y, W_bits)
        for i in range(r1 - r0):
            res = process_row(z[i], int(ids[r0 + i]), temperature, top_k, top_p)
            (out["logprob"][r0 + i], out["lse_kept"][r0 + i], out["kept"][r0 + i],
             out["gap_k"][r0 + i], out["margin_p"][r0 + i]) = res
            out["topk_ids"][r0 + i], out["topk_logprob"][r0 + i] = process_head(
                z[i], temperature, top_k, top_p)
            zk = z[i][out["topk_ids"][r0 + i]]
            out["rank_gap"][r0 + i] = float(np.min(zk[:-1] - zk[1:])) if kk > 1 else math.inf
    return out
