"""Seeded synthetic inputs for the linear-logprob scorer and the three-way compare.

This module only *generates data*. It holds none of the scoring or comparison
arithmetic: no normalisation, no matrix products, no softmax, no statistics.
Both the fp64 CPU oracle (``oracle/``) and the CUDA path are fed from here, so
that they see byte-identical inputs; neither of them is imported here.

Every tensor is drawn from its own numpy ``PCG64`` stream keyed by
``(seed, workload id, tensor name)``, so a tensor does not change when another
one is added or resized.  bf16 tensors are produced by rounding float32 draws to
nearest-even and are returned as raw ``uint16`` bit patterns.

Shapes and distributions follow the scoring workloads the pages describe:

* head shapes of Qwen3-1.7B (d=2048) and Qwen3-8B (d=4096) with the padded
  vocabulary V=151936 ("Diagnosing Training Inference Mismatch in LLM
  Reinforcement Learning", results 1 and 6);
* one prompt x 8 samples with a shared prompt prefix ("Training and rollout stop
  disagreeing: vime and RL-Kernel ...", Interpretation: 1 prompt times 8
  samples per step), so the same-prefix sibling property can be checked
  ("Fault localization and mismatch bisect", Same-prefix sibling);
* response masks with prompt / response / padding ("Debugging Logprob Mismatches
  in LLM Reinforcement Learning", Save the Inputs Needed for That Replay);
* three score sets: generation (A), replay (B) and trainer (C), where C sees a
  perturbed hidden state or a stale weight version ("Debugging Logprob
  Mismatches ...", One Response, Three Scores; Case 3).

Notation: N(mu, var) names the *variance*, so N(0, 1e-2) has sigma 0.1.
No public dataset, tokenizer or checkpoint is read; these arrays stand in for
them.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, List, Optional, Sequence

import numpy as np

SEED = 0

# workload ids used to key the random streams
WORKLOAD_IDS = {
    "tiny": 0,
    "qwen3_1p7b": 1,
    "qwen3_8b": 2,
    "sweep_8b": 3,
    "long_5120": 4,
    "custom": 9,
}


def stream(workload: str, tensor: str, seed: int = SEED, extra: int = 0) -> np.random.Generator:
    """An independent PCG64 stream for one tensor of one workload."""
    key = [seed, WORKLOAD_IDS.get(workload, 99), zlib.crc32(tensor.encode()), extra]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits.

    Inputs are finite draws; NaN/Inf handling is not needed for generated data.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for building perturbations)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(gen: np.random.Generator, shape, sigma: float = 1.0, mean: float = 0.0,
                chunk_rows: int = 8192) -> np.ndarray:
    """bf16 bits of mean + sigma * N(0,1), drawn row-chunk by row-chunk (bounded memory)."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    if len(shape) == 1 or shape[0] == 0:
        v = gen.standard_normal(shape, dtype=np.float32)
        return f32_to_bf16_bits(v * np.float32(sigma) + np.float32(mean))
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        v = gen.standard_normal((r1 - r0,) + shape[1:], dtype=np.float32)
        out[r0:r1] = f32_to_bf16_bits(v * np.float32(sigma) + np.float32(mean))
    return out


def perturb_bf16(base_bits: np.ndarray, gen: np.random.Generator, sigma: float,
                 chunk_rows: int = 8192) -> np.ndarray:
    """bf16 bits of base + N(0, sigma^2) (base widened exactly, sum rounded to bf16)."""
    out = np.empty_like(base_bits)
    for r0 in range(0, base_bits.shape[0], chunk_rows):
        r1 = min(base_bits.shape[0], r0 + chunk_rows)
        v = gen.standard_normal(base_bits[r0:r1].shape, dtype=np.float32)
        out[r0:r1] = f32_to_bf16_bits(bf16_bits_to_f32(base_bits[r0:r1]) + v * np.float32(sigma))
    return out


def zipf_ids(gen: np.random.Generator, perm: np.ndarray, n: int, s: float = 1.1) -> np.ndarray:
    """n token ids: truncated Zipf(s) ranks 1..V by inverse CDF, mapped through ``perm``."""
    V = perm.shape[0]
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = gen.random(n)
    ranks = np.minimum(np.searchsorted(cdf, u, side="right"), V - 1)
    return perm[ranks].astype(np.int32)


@dataclasses.dataclass
class Head:
    """An LM head: bf16 W [V,d] (nn.Linear layout, K-major) and final-norm gamma [d]."""
    d: int
    V: int
    W: np.ndarray          # uint16 [V, d]
    gamma: np.ndarray      # uint16 [d]
    vocab_perm: np.ndarray  # int64 [V]  (token id of Zipf rank r+1)


def make_head(workload: str, d: int, V: int, seed: int = SEED) -> Head:
    """W ~ N(0, (2/sqrt(d))^2), gamma = 1 + N(0, 0.05), vocabulary permutation."""
    W = normal_bf16(stream(workload, "W", seed), (V, d), sigma=2.0 / np.sqrt(d))
    gamma = normal_bf16(stream(workload, "gamma", seed), (d,), sigma=float(np.sqrt(0.05)), mean=1.0)
    perm = stream(workload, "vocab_perm", seed).permutation(V)
    return Head(d=d, V=V, W=W, gamma=gamma, vocab_perm=perm)


def fp32_weights(head: Head, seed: int = SEED, rel_sigma: float = 1e-3) -> np.ndarray:
    """fp32 [V, d] weights near the head's bf16 W: W * (1 + N(0, rel_sigma^2)) rounded to
    fp32, so that almost no element is a bf16 (or tf32) value (fp32 master weights)."""
    g = stream("fp32w", f"W{head.V}x{head.d}", seed)
    base = bf16_bits_to_f32(head.W).astype(np.float64)
    noise = g.standard_normal(base.shape, dtype=np.float32).astype(np.float64)
    return (base * (1.0 + rel_sigma * noise)).astype(np.float32)


@dataclasses.dataclass
class ScoreBatch:
    """One workload's rows plus the three score-set inputs and the compare layout.

    Rows are *pre-aligned*: hidden row t predicts token_ids[t].
    ``hidden_gen`` feeds both the generation (A) and the replay (B) scores;
    ``hidden_train`` feeds the trainer score (C), together with ``W_train``
    (``None`` means the same W as A/B).
    """
    name: str
    head: Head
    T: int
    temperature: float
    eps: float
    tis_cap: float
    hidden_gen: np.ndarray        # uint16 [T, d]
    hidden_train: np.ndarray      # uint16 [T, d]
    W_train: Optional[np.ndarray]  # uint16 [V, d] or None
    token_ids: np.ndarray         # int32 [T]
    seq_offsets: np.ndarray       # int64 [S+1]
    mask: np.ndarray              # uint8 [T]
    meta: Dict

    @property
    def d(self) -> int:
        return self.head.d

    @property
    def V(self) -> int:
        return self.head.V

    @property
    def n_seq(self) -> int:
        return int(self.seq_offsets.shape[0] - 1)


def _suffix_mask(S: int, L: int, n_resp: int) -> np.ndarray:
    m = np.zeros((S, L), dtype=np.uint8)
    m[:, L - n_resp:] = 1
    return m.reshape(-1)


def make_tiny(seed: int = SEED) -> ScoreBatch:
    """T=64 as 4 sequences of 16, d=128, V=1000, temperature 1, eps 1e-6.

    Response mask = last 12 tokens of each sequence.  Trainer hidden =
    hidden + N(0, 1e-2), and 2 active rows get +0.5 added to every element.
    """
    S, L, d, V = 4, 16, 128, 1000
    T = S * L
    head = make_head("tiny", d, V, seed)
    hidden = normal_bf16(stream("tiny", "hidden", seed), (T, d))
    ids = zipf_ids(stream("tiny", "ids", seed), head.vocab_perm, T)
    mask = _suffix_mask(S, L, 12)
    h_train = perturb_bf16(hidden, stream("tiny", "train_noise", seed), 0.1)
    active = np.flatnonzero(mask)
    shifted = np.sort(stream("tiny", "shift_rows", seed).choice(active, size=2, replace=False))
    h32 = bf16_bits_to_f32(h_train)
    h32[shifted] += np.float32(0.5)
    h_train = f32_to_bf16_bits(h32)
    return ScoreBatch("tiny", head, T, 1.0, 1e-6, 2.0, hidden, h_train, None, ids,
                      np.arange(0, T + 1, L, dtype=np.int64), mask,
                      dict(S=S, L=L, shifted_rows=shifted.tolist()))


def _train_hidden_heavy(workload: str, hidden: np.ndarray, seed: int,
                        share_prefix: Optional[tuple] = None) -> np.ndarray:
    """hidden + N(0, 1e-2) on every row, plus N(0, 0.3) on 1% of rows.

    ``share_prefix=(S, L, P)``: the first P rows of each of the S sequences of
    length L get the *same* perturbation as sequence 0 (siblings share a prompt).
    """
    T, d = hidden.shape
    h_train = perturb_bf16(hidden, stream(workload, "train_noise", seed), 0.1)
    n_heavy = max(1, T // 100)
    rows = np.sort(stream(workload, "heavy_rows", seed).choice(T, size=n_heavy, replace=False))
    g = stream(workload, "heavy_noise", seed)
    h32 = bf16_bits_to_f32(h_train[rows])
    h32 += g.standard_normal(h32.shape, dtype=np.float32) * np.float32(np.sqrt(0.3))
    h_train[rows] = f32_to_bf16_bits(h32)
    if share_prefix is not None:
        S, L, P = share_prefix
        for s in range(1, S):
            h_train[s * L:s * L + P] = h_train[0:P]
    return h_train


def make_qwen3_1p7b(seed: int = SEED, T: int = 8192) -> ScoreBatch:
    """d=2048, V=151936, T=8192 as 16 x 512, temperature 1, last 384 tokens active."""
    L = 512
    S = T // L
    d, V = 2048, 151936
    head = make_head("qwen3_1p7b", d, V, seed)
    hidden = normal_bf16(stream("qwen3_1p7b", "hidden", seed), (T, d))
    ids = zipf_ids(stream("qwen3_1p7b", "ids", seed), head.vocab_perm, T)
    mask = _suffix_mask(S, L, 384)
    h_train = _train_hidden_heavy("qwen3_1p7b", hidden, seed)
    return ScoreBatch("qwen3_1p7b", head, T, 1.0, 1e-6, 2.0, hidden, h_train, None, ids,
                      np.arange(0, T + 1, L, dtype=np.int64), mask, dict(S=S, L=L))


def make_qwen3_8b(seed: int = SEED, samples: int = 8, prefix: int = 1024, response: int = 3072,
                  head: Optional[Head] = None) -> ScoreBatch:
    """One prompt x 8 samples: 1024 shared prompt rows + 3072 response rows each.

    d=4096, V=151936, temperature 0.7, TIS cap 2.0; mask = response rows.
    Prompt rows (hidden, ids and the trainer perturbation) are identical across
    samples, so their scores must be bitwise identical (sibling check).
    """
    L = prefix + response
    S = samples
    T = S * L
    d, V = 4096, 151936
    head = head if head is not None else make_head("qwen3_8b", d, V, seed)
    hp = normal_bf16(stream("qwen3_8b", "hidden_prefix", seed), (prefix, d))
    hr = normal_bf16(stream("qwen3_8b", "hidden_response", seed), (S * response, d))
    idp = zipf_ids(stream("qwen3_8b", "ids_prefix", seed), head.vocab_perm, prefix)
    idr = zipf_ids(stream("qwen3_8b", "ids_response", seed), head.vocab_perm, S * response)
    hidden = np.empty((T, d), dtype=np.uint16)
    ids = np.empty((T,), dtype=np.int32)
    for s in range(S):
        hidden[s * L:s * L + prefix] = hp
        hidden[s * L + prefix:(s + 1) * L] = hr[s * response:(s + 1) * response]
        ids[s * L:s * L + prefix] = idp
        ids[s * L + prefix:(s + 1) * L] = idr[s * response:(s + 1) * response]
    mask = _suffix_mask(S, L, response)
    h_train = _train_hidden_heavy("qwen3_8b", hidden, seed, share_prefix=(S, L, prefix))
    return ScoreBatch("qwen3_8b", head, T, 0.7, 1e-6, 2.0, hidden, h_train, None, ids,
                      np.arange(0, T + 1, L, dtype=np.int64), mask,
                      dict(S=S, L=L, prefix=prefix, response=response))


def make_long_5120(seed: int = SEED, S: int = 64, L: int = 2048, prompt: int = 256,
                   resp_lo: int = 256, resp_hi: int = 1792, head: Optional[Head] = None,
                   with_stale: bool = True) -> ScoreBatch:
    """d=5120, V=151936, T=64 x 2048, temperature 0.7.

    Each 2048-slot sequence: 256 prompt rows, a response of length U[256,1792]
    (mask = response), then padding rows (token id 0, still scored).
    The trainer set uses a stale weight version W' = W + N(0, 1e-3).
    """
    d, V = 5120, 151936
    T = S * L
    head = head if head is not None else make_head("long_5120", d, V, seed)
    hidden = normal_bf16(stream("long_5120", "hidden", seed), (T, d))
    ids = zipf_ids(stream("long_5120", "ids", seed), head.vocab_perm, T)
    lens = stream("long_5120", "resp_len", seed).integers(resp_lo, resp_hi + 1, size=S)
    mask = np.zeros((S, L), dtype=np.uint8)
    ids2 = ids.reshape(S, L)
    for s in range(S):
        mask[s, prompt:prompt + lens[s]] = 1
        ids2[s, prompt + lens[s]:] = 0
    W_train = perturb_bf16(head.W, stream("long_5120", "W_stale", seed), float(np.sqrt(1e-3))) \
        if with_stale else None
    return ScoreBatch("long_5120", head, T, 0.7, 1e-6, 2.0, hidden, hidden, W_train,
                      ids2.reshape(-1).copy(), np.arange(0, T + 1, L, dtype=np.int64),
                      mask.reshape(-1), dict(S=S, L=L, prompt=prompt, resp_len=lens.tolist()))


@dataclasses.dataclass
class SweepPlan:
    """Batch-invariance sweep: fixed target rows scored inside batches of size M."""
    head: Head
    targets_hidden: np.ndarray   # uint16 [N, d]
    targets_ids: np.ndarray      # int32 [N]
    temperature: float
    eps: float
    batches: Dict[int, List[dict]]  # M -> list of {hidden, ids, target_pos, target_idx}


def make_sweep(Ms: Sequence[int] = (1, 7, 64, 513, 4096, 16384), n_targets: int = 4096,
               seed: int = SEED, head: Optional[Head] = None, d: int = 4096,
               V: int = 151936, max_batches_per_M: Optional[int] = None) -> SweepPlan:
    """Targets are seed-permuted, split into batches of M, placed at random positions;
    partial batches (and M > n_targets) are topped up with fresh N(0,1) filler rows.

    ``max_batches_per_M`` limits how many batches of each M are materialised
    (the targets they hold are the ones compared across M).
    """
    head = head if head is not None else make_head("sweep_8b", d, V, seed)
    d = head.d
    th = normal_bf16(stream("sweep_8b", "targets_hidden", seed), (n_targets, d))
    tid = zipf_ids(stream("sweep_8b", "targets_ids", seed), head.vocab_perm, n_targets)
    batches: Dict[int, List[dict]] = {}
    for M in Ms:
        g = stream("sweep_8b", "placement", seed, extra=int(M))
        order = g.permutation(n_targets)
        per = min(M, n_targets)
        out = []
        for b0 in range(0, n_targets, per):
            if max_batches_per_M is not None and len(out) >= max_batches_per_M:
                break
            tix = order[b0:b0 + per]
            pos = np.sort(g.choice(M, size=tix.shape[0], replace=False))
            n_fill = M - tix.shape[0]
            hid = np.empty((M, d), dtype=np.uint16)
            ids = np.empty((M,), dtype=np.int32)
            if n_fill:
                fill_pos = np.setdiff1d(np.arange(M), pos)
                hid[fill_pos] = normal_bf16(g, (n_fill, d))
                ids[fill_pos] = zipf_ids(g, head.vocab_perm, n_fill)
            hid[pos] = th[tix]
            ids[pos] = tid[tix]
            out.append(dict(hidden=hid, ids=ids, target_pos=pos, target_idx=tix))
        batches[M] = out
    return SweepPlan(head, th, tid, 0.7, 1e-6, batches)


def make_custom(T: int, d: int, V: int, temperature: float = 1.0, eps: float = 1e-6,
                seq_len: Optional[int] = None, n_resp: Optional[int] = None,
                seed: int = SEED, tag: str = "") -> ScoreBatch:
    """Small ad-hoc shapes (ragged tails, edge cases) with the same distributions."""
    wl = "custom"
    head = Head(d=d, V=V,
                W=normal_bf16(stream(wl, f"W{tag}{V}x{d}", seed), (V, d), sigma=2.0 / np.sqrt(d)),
                gamma=normal_bf16(stream(wl, f"gamma{tag}{d}", seed), (d,),
                                  sigma=float(np.sqrt(0.05)), mean=1.0),
                vocab_perm=stream(wl, f"perm{tag}{V}", seed).permutation(V))
    hidden = normal_bf16(stream(wl, f"hidden{tag}{T}x{d}", seed), (T, d))
    ids = zipf_ids(stream(wl, f"ids{tag}{T}x{V}", seed), head.vocab_perm, T)
    L = seq_len if seq_len else T
    S = (T + L - 1) // L
    offs = np.minimum(np.arange(0, S + 1, dtype=np.int64) * L, T)
    mask = np.zeros(T, dtype=np.uint8)
    for s in range(S):
        a, b = int(offs[s]), int(offs[s + 1])
        k = (b - a) if n_resp is None else min(n_resp, b - a)
        mask[b - k:b] = 1
    h_train = perturb_bf16(hidden, stream(wl, f"train{tag}{T}x{d}", seed), 0.1)
    return ScoreBatch(f"custom{tag}", head, T, temperature, eps, 2.0, hidden, h_train, None,
                      ids, offs, mask, dict(S=S, L=L))


WORKLOADS = {
    "tiny": make_tiny,
    "qwen3_1p7b": make_qwen3_1p7b,
    "qwen3_8b": make_qwen3_8b,
    "long_5120": make_long_5120,
}
