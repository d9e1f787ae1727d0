"""Shared helpers for the GPU-vs-oracle parity tests (test infrastructure).

Tolerances, as the scoring contract states them:
* logprob and lse: |gpu - oracle| <= 2e-3 nats (bf16 operands, fp32 accumulation
  against the fp64 oracle);
* top-1: exact wherever the oracle's top-2 logit gap exceeds 1e-3;
* compare statistics: counts, first positions, runs and max_abs_diff bit-exact;
  means within 1e-9 relative.  A relative bar needs a floor when a mean is a
  sum of mixed-sign terms that nearly cancels: two fp64 summations of n terms
  in different orders differ by at most ~2 n eps64 * mean|term|, so the bar
  used is 1e-9 * max(|ref|, mean|term|) (mean|term| is the pair's MAE for the
  signed means).  For k3 each side also evaluates expm1 with an error of about
  one ulp of |d|, so its bar adds 4 eps64 * mean|d|.
* per-token TIS weights (float32): within one float32 ulp of the oracle.
"""
from __future__ import annotations

import math

import numpy as np

import oracle

LP_TOL = 2e-3
TOP1_GAP = 1e-3
MEAN_REL = 1e-9
EPS64 = 2.0 ** -52


def bf16_cuda(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def cuda_tensor(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_logprob_parity(gpu, orc, rows=None, what=""):
    """gpu = (lp, lse, top1) numpy arrays (all rows); orc = oracle dict for ``rows``."""
    lp, lse, top1 = gpu
    if rows is not None:
        lp, lse, top1 = lp[rows], lse[rows], top1[rows]
    ok_tok = ~orc["bad_token"]
    dlp = np.abs(lp[ok_tok].astype(np.float64) - orc["logprob"][ok_tok])
    dlse = np.abs(lse.astype(np.float64) - orc["lse"])
    assert np.all(np.isfinite(lp[ok_tok])), f"{what}: non-finite logprob"
    assert dlp.max(initial=0) <= LP_TOL, f"{what}: logprob max err {dlp.max():.3e}"
    assert dlse.max(initial=0) <= LP_TOL, f"{what}: lse max err {dlse.max():.3e}"
    sel = orc["gap"] > TOP1_GAP
    bad = np.flatnonzero(sel & (top1.astype(np.int64) != orc["top1"]))
    assert bad.size == 0, f"{what}: top1 differs on {bad.size} rows with gap > 1e-3, e.g. {bad[:5]}"
    if rows is None or len(rows):
        assert np.all(np.isnan(lp[~ok_tok])), f"{what}: invalid ids must give NaN"
    return dict(lp_max_err=float(dlp.max(initial=0)), lse_max_err=float(dlse.max(initial=0)),
                top1_checked=int(sel.sum()), rows=int(len(lse)))


def fp8_y_margin(d: int) -> float:
    """Relative error bound of y before its bf16 rounding, as the RMSNorm kernel computes
    it in fp32 (u = 2^-24): each lane adds the squares of its 8-element chunks with fused
    multiply-adds, n = 8 ceil(d / 256) rounded additions, then 5 butterfly additions
    ((n + 5) u on the sum, all terms positive); the division by d and the + eps add u
    each; the square root halves the argument's error and adds u; 1 / x adds u; h * rstd
    and * gamma add u each: (n + 7) / 2 + 4 = n / 2 + 7.5 units, rounded up to n / 2 + 8
    for the second-order terms."""
    n = 8 * (-(-d // 256))
    return (n / 2 + 8) * 2.0 ** -24


def assert_fp8_admissible_parity(gpu, adm, ids, V, rows=None, what="", max_exempt=0.01):
    """FP8-head parity: each row's GPU (logprob, lse) within LP_TOL of one of the row's
    admissible oracle results (``oracle.oracle_logprob_fp8_admissible``), and top-1 equal to
    that result's wherever its gap exceeds TOP1_GAP.  Rows with more ambiguous elements than
    the oracle enumerates are exempt; at most ``max_exempt`` of the rows may be.  Returns the
    counts (rows, rows with several admissible results, exempt rows)."""
    lp, lse, top1 = gpu
    if rows is not None:
        lp, lse, top1, ids = lp[rows], lse[rows], top1[rows], np.asarray(ids)[rows]
    multi = exempt = 0
    for i, alts in enumerate(adm):
        if alts is None:
            exempt += 1
            continue
        multi += len(alts) > 1
        bad_id = not (0 <= int(ids[i]) < V)
        ok = False
        for a in alts:
            if abs(float(lse[i]) - a["lse"]) > LP_TOL:
                continue
            if bad_id:
                ok = bool(np.isnan(lp[i]))
            else:
                ok = abs(float(lp[i]) - a["logprob"]) <= LP_TOL and (
                    a["gap"] <= TOP1_GAP or int(top1[i]) == a["top1"])
            if ok:
                break
        assert ok, (f"{what}: row {i} (lp {lp[i]!r}, lse {lse[i]!r}, top1 {top1[i]}) matches none "
                    f"of {len(alts)} admissible results, e.g. {alts[0]}")
    assert exempt <= max_exempt * max(1, len(adm)), f"{what}: {exempt} exempt rows"
    return dict(rows=len(adm), several=multi, exempt=exempt)


def _close(g, r, scale, extra=0.0):
    if g == r:
        return True
    return abs(g - r) <= MEAN_REL * max(abs(r), scale) + extra


def assert_compare_parity(gpu_stats, orc_stats, what=""):
    """gpu_stats: list of dicts (binding.stats_to_dicts); orc_stats: oracle list."""
    assert len(gpu_stats) == len(orc_stats)
    for j, (g, r) in enumerate(zip(gpu_stats, orc_stats)):
        tag = f"{what} seq {j}"
        assert g["flags"] == r["flags"], f"{tag}: flags {g['flags']} vs {r['flags']}"
        assert g["n_valid"] == r["n_valid"], tag
        if r["flags"] & (oracle.FLAG_BAD_MASK | oracle.FLAG_BAD_OFFSETS | oracle.FLAG_EMPTY |
                         oracle.FLAG_NONFINITE):
            continue
        for p in range(3):
            gp, rp = g["pair"][p], r["pair"][p]
            for k in ("mismatch_count", "first_div", "longest_run"):
                assert gp[k] == rp[k], f"{tag} pair {p} {k}: {gp[k]} vs {rp[k]}"
            assert gp["max_abs_diff"] == rp["max_abs_diff"], f"{tag} pair {p} max_abs"
            assert _close(gp["mae"], rp["mae"], rp["mae"]), f"{tag} pair {p} mae"
            assert _close(gp["signed_mean"], rp["signed_mean"], rp["mae"]), f"{tag} pair {p} mean"
        mae = [r["pair"][p]["mae"] for p in range(3)]
        assert _close(g["mean_log_ratio"], r["mean_log_ratio"], mae[2]), f"{tag} log ratio"
        assert _close(g["mean_weight_move"], r["mean_weight_move"], mae[1]), f"{tag} weight move"
        assert _close(g["mean_same_version"], r["mean_same_version"], mae[0]), f"{tag} same ver"
        assert _close(g["k3_mean"], r["k3_mean"], r["k3_mean"], 4 * EPS64 * mae[2]), f"{tag} k3"
        assert _close(g["tis_mean"], r["tis_mean"], r["tis_mean"]), f"{tag} tis"
        assert g["tis_clipped"] == r["tis_clipped"], f"{tag} clipped"


def assert_tis_parity(gpu_w: np.ndarray, orc_w: np.ndarray, covered: np.ndarray):
    g = gpu_w[covered].astype(np.float32)
    r = orc_w[covered].astype(np.float32)
    ulp = np.abs(np.spacing(r))
    assert np.all(np.abs(g.astype(np.float64) - r.astype(np.float64)) <= ulp), "tis_w > 1 ulp"


def covered_rows(seq_offsets, T):
    c = np.zeros(T, dtype=bool)
    for j in range(len(seq_offsets) - 1):
        a, b = int(seq_offsets[j]), int(seq_offsets[j + 1])
        if 0 <= a <= b <= T:
            c[a:b] = True
    return c


def sample_rows(T: int, n: int, seed: int = 1234, must=()) -> np.ndarray:
    g = np.random.default_rng(seed)
    rows = set(int(x) for x in must if 0 <= x < T)
    rows.update(g.choice(T, size=min(n, T), replace=False).tolist())
    rows.update([0, T - 1])
    return np.array(sorted(rows), dtype=np.int64)


ROW_TILE = 128


def raster_group_tiles(d: int) -> int:
    """Row tiles per raster group of the scoring GEMM's one-tile schedule at hidden size d
    (48 up to d = 4096, 36 above)."""
    return 48 if d <= 4096 else 36


def tile_rows(T: int, group_tiles: int, seed: int = 1234, must=()) -> np.ndarray:
    """Rows for a one-by-one oracle check that reach every part of the schedule: one
    seeded row inside every 128-row tile (the ragged last tile included), and the
    first and last row of every raster group of ``group_tiles`` tiles."""
    g = np.random.default_rng(seed)
    rows = set(int(x) for x in must if 0 <= x < T)
    for t0 in range(0, T, ROW_TILE):
        rows.add(int(g.integers(t0, min(T, t0 + ROW_TILE))))
    span = group_tiles * ROW_TILE
    for r0 in range(0, T, span):
        rows.update([r0, min(T, r0 + span) - 1])
    return np.array(sorted(rows), dtype=np.int64)


def finite_close(a, b, tol):
    return math.isfinite(a) and abs(a - b) <= tol
