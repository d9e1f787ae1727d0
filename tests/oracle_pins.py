"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with a
value the pages print, a closed form, an invariant, a library routine the
oracle does not call, or a brute-force evaluation.  ``test_oracle_pins.py``
runs them against the oracle as it stands; ``test_oracle_mutations.py`` plants
plausible mistakes in the oracle and checks that some pin catches each one.
"""
from __future__ import annotations

import json
import math
import struct
import os
from fractions import Fraction

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# bf16 helpers built independently of the oracle (for constructing inputs)

def _all_finite_bf16():
    """Every finite bf16 value as (sorted fp64 values, their uint16 patterns)."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        vals = (pats.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok = np.isfinite(vals)
    pats, vals = pats[ok], vals[ok]
    # keep one zero (+0) so the table is strictly increasing
    keep = ~((vals == 0) & (pats != 0))
    pats, vals = pats[keep], vals[keep]
    order = np.argsort(vals, kind="stable")
    return vals[order], pats[order]


_BF16_TABLE = None


def brute_nearest_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest finite bf16 by exhaustive table search; exact ties go to the even pattern."""
    global _BF16_TABLE
    if _BF16_TABLE is None:
        _BF16_TABLE = _all_finite_bf16()
    vals, pats = _BF16_TABLE
    x = np.asarray(x, dtype=np.float64)
    hi = np.clip(np.searchsorted(vals, x, side="left"), 1, vals.size - 1)
    lo = hi - 1
    dlo = np.abs(x - vals[lo])
    dhi = np.abs(vals[hi] - x)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (pats[hi] % 2 == 0))
    return np.where(pick_hi, vals[hi], vals[lo])


def trunc_bf16_bits(x: float) -> int:
    """bf16 pattern of x truncated toward zero (via float32)."""
    return int(np.float32(x).view(np.uint32) >> np.uint32(16))


def bits_value(b: int) -> float:
    return float(np.uint32(b << 16).view(np.float32))


def exact_logit_head(z_rows, n_limbs: int = 7):
    """A d=8 head whose logits equal the given fp64 targets to ~1e-16.

    hidden = 1 everywhere and eps = 0 give rstd = 1, so y = gamma exactly with
    gamma_i = 2^(-8 i).  Each W row holds the target split into truncated bf16
    limbs: z_v = sum_i W_vi 2^(-8 i).  Returns (hidden_bits [1,8], gamma_bits,
    W_bits [V,8], exact z as Fractions).
    """
    z_rows = [float(v) for v in z_rows]
    V = len(z_rows)
    d = 8
    gamma_bits = np.array([trunc_bf16_bits(2.0 ** (-8 * i)) for i in range(d)], dtype=np.uint16)
    W = np.zeros((V, d), dtype=np.uint16)
    z_exact = []
    for v, target in enumerate(z_rows):
        r = Fraction(target)
        tot = Fraction(0)
        for i in range(n_limbs):
            scaled = r * (2 ** (8 * i))
            b = trunc_bf16_bits(float(scaled))
            W[v, i] = b
            limb = Fraction(bits_value(b)) / (2 ** (8 * i))
            tot += limb
            r -= limb
        z_exact.append(tot)
    hidden = np.full((1, d), trunc_bf16_bits(1.0), dtype=np.uint16)
    return hidden, gamma_bits, W, z_exact


def _score(z_targets, x, tau):
    h, g, W, zx = exact_logit_head(z_targets)
    out = oracle.oracle_logprob(h, g, W, np.array([x], dtype=np.int32), tau, 0.0)
    return out, zx


# ---------------------------------------------------------------------------
# logprob pins

def pin_widen():
    v = oracle.widen_bf16(np.array([0x3F80, 0xC000, 0x7F80, 0x0001, 0x8000], dtype=np.uint16))
    assert v[0] == 1.0 and v[1] == -2.0 and v[2] == np.inf
    assert v[3] == 2.0 ** -133 and v[4] == 0.0 and math.copysign(1, v[4]) < 0


def pin_round_to_bf16_brute():
    g = np.random.default_rng(123)
    x = np.concatenate([
        g.standard_normal(20000) * 3.0,
        g.standard_normal(2000) * 1e-38,           # bf16 subnormal range
        np.ldexp(g.random(2000) + 0.5, g.integers(-120, 120, 2000)),
    ])
    vals, _ = _all_finite_bf16()
    mid = (vals[1000:30000:7] + vals[1001:30001:7]) / 2.0   # exact midpoints -> ties
    x = np.concatenate([x, mid, -mid])
    got = oracle.round_to_bf16(x)
    want = brute_nearest_bf16(x)
    assert np.array_equal(got, want), "round_to_bf16 disagrees with exhaustive nearest-even search"


def pin_v8_uniform():
    """All logits equal: logprob = -ln 8 for every token, top-1 = 0 (lowest id on ties)."""
    for x in (0, 3, 7):
        out, _ = _score([0.0] * 8, x, 1.0)
        assert abs(out["logprob"][0] - (-math.log(8))) < 1e-15
        assert abs(out["logprob"][0] - (-2.0794415416798357)) < 1e-15
        assert out["top1"][0] == 0


def pin_v8_page_probabilities():
    """p = 0.10 vs 0.12 for the scored token (Debugging page, What a Logprob Difference Means)."""
    gd = golden("logprob_difference_example.json")
    p1 = [0.10, 0.30, 0.20, 0.10, 0.10, 0.10, 0.05, 0.05]
    p2 = [0.12, 0.28, 0.20, 0.10, 0.10, 0.10, 0.05, 0.05]
    o1, _ = _score([math.log(p) for p in p1], 0, 1.0)
    o2, _ = _score([math.log(p) for p in p2], 0, 1.0)
    l1, l2 = o1["logprob"][0], o2["logprob"][0]
    assert abs(l1 - math.log(0.10)) < 1e-12 and abs(l2 - math.log(0.12)) < 1e-12
    assert round(l1, 4) == gd["logprob_rollout"] and round(l2, 4) == gd["logprob_train"]
    assert round(l2 - l1, 4) == gd["train_minus_rollout"]
    assert abs((l2 - l1) - 0.1823215568) < 1e-9
    assert round(math.exp(l2 - l1), 2) == gd["ratio"]
    assert o1["top1"][0] == 1 and o2["top1"][0] == 1
    assert abs(o1["gap"][0] - (math.log(0.30) - math.log(0.20))) < 1e-12


def pin_v8_temperature():
    """tau = 0.5 on z = 0..7: log_softmax(z/tau), not log_softmax(z)/tau (Debugging page,
    'How this differs from a real temperature mismatch')."""
    tau = 0.5
    lse_scaled = math.log((math.exp(16) - 1) / (math.exp(2) - 1))      # ln sum_k e^{2k}
    lse_raw = math.log((math.exp(8) - 1) / (math.exp(1) - 1))          # ln sum_k e^{k}
    for x in (0, 5, 7):
        out, _ = _score([float(k) for k in range(8)], x, tau)
        want = 2 * x - lse_scaled
        wrong = (x - lse_raw) / tau
        assert abs(out["logprob"][0] - want) < 1e-12
        assert abs(out["lse"][0] - lse_scaled) < 1e-12
        assert abs(want - wrong) > 0.05
        assert out["top1"][0] == 7


def pin_large_logits():
    """Logits near 800 must not overflow the normaliser (max shift)."""
    z = [800.0 - k for k in range(8)]
    out, _ = _score(z, 2, 1.0)
    want = -2.0 - math.log(sum(math.exp(-k) for k in range(8)))
    assert math.isfinite(out["logprob"][0]) and abs(out["logprob"][0] - want) < 1e-12
    assert abs(out["lse"][0] - (800.0 + math.log(sum(math.exp(-k) for k in range(8))))) < 1e-11


def pin_rmsnorm_closed_form():
    """Constant rows: y = bf16(c / sqrt(c^2 + eps) * gamma); scale invariance at eps = 0."""
    for c, eps in ((2.0, 0.25), (0.5, 1e-6), (3.0, 1.0)):
        h = np.full((1, 16), c)
        gam = np.ones(16)
        y = oracle.rmsnorm(h, gam, eps)
        want = brute_nearest_bf16(np.array([c / math.sqrt(c * c + eps)]))[0]
        assert np.all(y == want), (c, eps, y[0, 0], want)
    g = np.random.default_rng(5)
    hb = synth.f32_to_bf16_bits(g.standard_normal((4, 64)).astype(np.float32))
    h = oracle.widen_bf16(hb)
    gam = oracle.widen_bf16(synth.f32_to_bf16_bits((1 + 0.2 * g.standard_normal(64)).astype(np.float32)))
    assert np.array_equal(oracle.rmsnorm(h, gam, 0.0), oracle.rmsnorm(4.0 * h, gam, 0.0))


def pin_rmsnorm_library():
    """fp64 torch rms_norm (not used by the oracle) then nearest-even bf16 matches."""
    import torch
    b = synth.make_custom(T=16, d=256, V=64, eps=1e-5, tag="rmslib")
    h = oracle.widen_bf16(b.hidden_gen)
    gam = oracle.widen_bf16(b.head.gamma)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h), (h.shape[1],), torch.from_numpy(gam),
                                       eps=b.eps).numpy()
    want = brute_nearest_bf16(ref)
    got = oracle.rmsnorm(h, gam, b.eps)
    diff = got != want
    # fp64 rounding order may move a value across a bf16 rounding midpoint only if it sits
    # within ~1e-15 relative of it: allow at most a handful of such elements, each 1 bf16 step.
    assert diff.sum() <= 2
    if diff.any():
        assert np.all(np.abs(got[diff] - want[diff]) <= np.abs(want[diff]) * 2.0 ** -7)


def pin_library_log_softmax():
    """At tau = 1 torch.log_softmax + gather (the trainer extraction of the Debugging page's
    trainer_scores) reproduces the oracle's lse / logprob / argmax on the same logits;
    at tau != 1 torch.logsumexp(z / tau) does."""
    import torch
    b = synth.make_custom(T=24, d=128, V=333, tag="lsm")
    y = oracle.rmsnorm(oracle.widen_bf16(b.hidden_gen), oracle.widen_bf16(b.head.gamma), b.eps)
    z = oracle.logits(y, b.head.W)
    for tau in (1.0, 0.7):
        out = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, tau, b.eps)
        zt = torch.from_numpy(z)
        ls = torch.log_softmax(zt / tau, dim=-1)
        lp = ls.gather(1, torch.from_numpy(b.token_ids.astype(np.int64))[:, None])[:, 0].numpy()
        assert np.max(np.abs(lp - out["logprob"])) < 1e-12
        lse = torch.logsumexp(zt / tau, dim=-1).numpy()
        assert np.max(np.abs(lse - out["lse"])) < 1e-12
        assert np.array_equal(torch.argmax(zt, dim=-1).numpy(), out["top1"])


def pin_sum_exp_one():
    """exp(log_softmax) sums to 1 within 1e-12 on full rows."""
    b = synth.make_tiny()
    for tau in (1.0, 0.7):
        rows = oracle.oracle_log_softmax_rows(b.hidden_gen, b.head.gamma, b.head.W, tau, b.eps)
        for r in rows:
            assert abs(math.fsum(np.exp(r)) - 1.0) < 1e-12


def pin_invariants():
    """logprob <= 0, lse >= max s, the top-1 token has the highest logprob, gap >= 0."""
    b = synth.make_tiny()
    tau = 0.7
    out = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, tau, b.eps)
    rows = oracle.oracle_log_softmax_rows(b.hidden_gen, b.head.gamma, b.head.W, tau, b.eps)
    assert np.all(out["logprob"] <= 0)
    assert np.all(out["lse"] >= out["zmax"] / tau)
    assert np.array_equal(np.argmax(rows, axis=1), out["top1"])
    assert np.all(out["gap"] >= 0)
    assert np.allclose(rows[np.arange(b.T), b.token_ids], out["logprob"], atol=1e-12, rtol=0)


def _mp_nearest_bf16(x_mp):
    import mpmath
    return brute_nearest_bf16(np.array([float(x_mp)]))[0] if abs(float(x_mp)) > 0 else 0.0


def pin_brute_force_mpmath():
    """Small rows evaluated end to end at 50 digits (mpmath), including the bf16 rounding of y
    by exhaustive search; the oracle must agree to 1e-12."""
    import mpmath
    mpmath.mp.dps = 50
    b = synth.make_custom(T=3, d=16, V=40, temperature=0.7, eps=1e-6, tag="mp")
    out = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 0.7, 1e-6)
    hb = oracle.widen_bf16(b.hidden_gen)  # exact widening (pinned by pin_widen)
    gb = oracle.widen_bf16(b.head.gamma)
    Wb = oracle.widen_bf16(b.head.W)
    for t in range(b.T):
        h = [mpmath.mpf(float(v)) for v in hb[t]]
        ms = mpmath.fsum(v * v for v in h) / len(h)
        rstd = 1 / mpmath.sqrt(ms + mpmath.mpf(1e-6))
        y = []
        for i, v in enumerate(h):
            pre = v * rstd * mpmath.mpf(float(gb[i]))
            # exact nearest bf16 of the 50-digit value: fp64 conversion first is safe unless
            # the value lies within 1e-16 relative of a bf16 midpoint (not the case here)
            y.append(mpmath.mpf(_mp_nearest_bf16(pre)))
        z = [mpmath.fsum(y[i] * mpmath.mpf(float(Wb[v, i])) for i in range(len(y))) for v in range(b.V)]
        s = [zz / mpmath.mpf(0.7) for zz in z]
        lse = mpmath.log(mpmath.fsum(mpmath.exp(v) for v in s))
        x = int(b.token_ids[t])
        lp = s[x] - lse
        assert abs(float(lp) - out["logprob"][t]) < 1e-12
        assert abs(float(lse) - out["lse"][t]) < 1e-12
        zf = [float(v) for v in z]
        assert out["top1"][t] == int(np.argmax(zf))


def pin_bad_token():
    b = synth.make_custom(T=4, d=64, V=50, tag="badtok")
    ids = b.token_ids.copy()
    ids[1] = 50
    ids[2] = -1
    out = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, ids, 1.0, b.eps)
    assert np.isnan(out["logprob"][1]) and np.isnan(out["logprob"][2])
    assert np.all(np.isfinite(out["lse"])) and np.isfinite(out["logprob"][0])
    assert list(out["bad_token"]) == [False, True, True, False]


# ---------------------------------------------------------------------------
# compare pins

def _one_seq(A, B, C, mask=None, cap=2.0):
    A = np.asarray(A, dtype=np.float32)
    n = A.shape[0]
    mask = np.ones(n, dtype=np.uint8) if mask is None else np.asarray(mask, dtype=np.uint8)
    st, w = oracle.oracle_compare(A, np.asarray(B, np.float32), np.asarray(C, np.float32),
                                  np.array([0, n], dtype=np.int64), mask, cap)
    return st[0], w


def pin_recorded_token_summary():
    """The Case 1 outlier token: the per-pair statistics of a one-token sequence reproduce the
    printed differences (signed mean to 6 places, MAE and maximum equal to its size)."""
    gd = golden("recorded_token_case1.json")
    sc = gd["scores"]
    for label, want in gd["signed_differences_6dp"].items():
        l, r = label.split("-")
        st, _ = _one_seq([sc[l]], [sc[r]], [sc[r]])
        pr = st["pair"][0]
        assert st["n_valid"] == 1
        # A is printed with more digits than a float32 holds: the pair sees its float32 value
        want_exact = float(np.float64(np.float32(sc[l])) - np.float64(np.float32(sc[r])))
        assert pr["signed_mean"] == want_exact
        assert round(pr["signed_mean"], 6) == want, (label, pr["signed_mean"], want)
        assert pr["mae"] == pr["max_abs_diff"] == abs(want_exact)


def pin_recorded_token_bitwise():
    """B0, B1, C0, C1 are float32 values: B1 and C0 differ by one float32 step (about
    1.19e-7 nat), C0 and C1 are bitwise equal."""
    gd = golden("recorded_token_case1.json")
    s = {k: np.float32(v) for k, v in gd["scores"].items() if k != "A"}
    for k, v in gd["scores"].items():
        if k != "A":
            assert float(s[k]) == v, "page value is not a float32"
    st, _ = _one_seq([s["B0"]], [s["B1"]], [s["C0"]])
    # pairs: (A,B)=(B0,B1), (B,C)=(B1,C0), (A,C)=(B0,C0)
    assert st["pair"][0]["mismatch_count"] == 1 and st["pair"][0]["first_div"] == 0
    assert st["pair"][1]["max_abs_diff"] == 2.0 ** -23
    assert abs(st["pair"][1]["max_abs_diff"] - gd["B1_minus_C0_about"]) < 0.01e-7
    assert round(st["pair"][0]["signed_mean"], 6) == gd["signed_differences_6dp"]["B0-B1"]
    st2, _ = _one_seq([s["C0"]], [s["C1"]], [s["C1"]])
    assert st2["pair"][0]["mismatch_count"] == 0 and st2["pair"][0]["max_abs_diff"] == 0.0


def pin_case3_outlier():
    gd = golden("case3_stale_outlier.json")
    s = gd["scores"]
    st, _ = _one_seq([s["A"]], [s["B0"]], [s["C0"]])
    assert st["pair"][0]["mismatch_count"] == 0 and st["pair"][0]["max_abs_diff"] == 0.0
    assert abs(st["pair"][1]["max_abs_diff"] - gd["differences_9dp"]["B0-C0"]) < 5e-10
    assert abs(st["pair"][1]["signed_mean"] - gd["differences_9dp"]["B0-C0"]) < 5e-10
    assert st["pair"][1]["first_div"] == 0 and st["pair"][1]["longest_run"] == 1


def pin_fig1_split():
    """Eq. (1) with the Figure 1 numbers: C - A = (C - B) + (B - A); w = 1.05, r = 1.20."""
    gd = golden("fig1_ratio_split.json")
    A = np.float32(math.log(gd["q_v"]))
    B = np.float32(math.log(gd["p_v"]))
    C = np.float32(math.log(gd["p_k"]))
    st, _ = _one_seq([A], [B], [C], cap=2.0)
    tol = 4e-7   # float32 rounding of the three inputs
    assert abs(st["mean_log_ratio"] - gd["log_pk_over_qv"]) < tol
    assert round(math.log(gd["p_k"] / gd["q_v"]), 10) == gd["log_pk_over_qv"]
    assert abs(st["mean_weight_move"] - math.log(gd["r"])) < tol
    assert abs(st["mean_same_version"] - math.log(gd["w"])) < tol
    assert st["mean_log_ratio"] == st["mean_weight_move"] + st["mean_same_version"]
    # token TIS weight with the historical trainer as anchor: w = pi0 / q = 0.21 / 0.20
    st2, w2 = _one_seq([A], [A], [B], cap=2.0)
    assert abs(st2["tis_mean"] - gd["w"]) < 1e-6 and abs(float(w2[0]) - gd["w"]) < 1e-6
    assert st2["tis_clipped"] == 0
    # movement ratio r = p_k / pi0 read through the same statistic
    st3, _ = _one_seq([B], [B], [C], cap=2.0)
    assert abs(st3["tis_mean"] - gd["r"]) < 1e-6


def pin_tii_example():
    gd = golden("tii_weight_example.json")
    A = np.float32(math.log(gd["q_v"]))
    C = np.float32(math.log(gd["p_k"]))
    st, w = _one_seq([A], [A], [C], cap=2.0)
    assert st["pair"][0]["mismatch_count"] == 0 and st["mean_same_version"] == 0.0
    assert abs(st["tis_mean"] - gd["weight"]) < 1e-6


def pin_eq1_exact_per_token():
    """Per token, (C - B) + (B - A) equals C - A exactly (rational arithmetic on float32
    inputs), and the per-sequence means obey the split to 1e-12 relative."""
    g = np.random.default_rng(7)
    A = (g.standard_normal(500) * 3 - 5).astype(np.float32)
    B = (A + g.standard_normal(500).astype(np.float32) * np.float32(0.01)).astype(np.float32)
    C = (B + g.standard_normal(500).astype(np.float32) * np.float32(0.3)).astype(np.float32)
    for a, b, c in zip(A[:50], B[:50], C[:50]):
        fa, fb, fc = Fraction(float(a)), Fraction(float(b)), Fraction(float(c))
        assert (fc - fb) + (fb - fa) == fc - fa
        assert Fraction(float(np.float64(c) - np.float64(a))) == fc - fa
    st, _ = _one_seq(A, B, C)
    lhs = st["mean_log_ratio"]
    rhs = st["mean_weight_move"] + st["mean_same_version"]
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))
    want = float(sum(Fraction(float(c)) - Fraction(float(a)) for a, c in zip(A, C)) / len(A))
    assert abs(lhs - want) <= 1e-12 * abs(want)


def pin_identical_inputs():
    g = np.random.default_rng(3)
    A = (g.standard_normal(300) - 4).astype(np.float32)
    mask = (g.random(300) < 0.7).astype(np.uint8)
    mask[0] = 1
    st, w = _one_seq(A, A.copy(), A.copy(), mask)
    for p in st["pair"]:
        assert p["mismatch_count"] == 0 and p["first_div"] == -1 and p["longest_run"] == 0
        assert p["max_abs_diff"] == 0.0 and p["signed_mean"] == 0.0 and p["mae"] == 0.0
    assert st["k3_mean"] == 0.0 and st["tis_mean"] == 1.0 and st["tis_clipped"] == 0
    assert st["n_valid"] == int(mask.sum())
    assert np.all(w[mask == 1] == 1.0) and np.all(w[mask == 0] == 0.0)


def pin_k3_closed_form():
    """k3 = exp(d) - 1 - d: d = ln 2 gives 1 - ln 2, d = -1 gives 1/e (up to the float32
    rounding of the inputs); tiny d gives d^2/2 + d^3/6 + ... to 1e-8 relative, which an
    evaluation as exp(d) - 1 - d would miss by cancellation."""
    a = np.float32(-3.0)
    for d, closed in ((math.log(2.0), 1 - math.log(2.0)), (-1.0, math.exp(-1.0))):
        c = np.float32(a + np.float32(d))
        dd = float(np.float64(c) - np.float64(a))
        st, _ = _one_seq([a], [a], [c])
        assert abs(st["k3_mean"] - closed) < 1e-6
        assert abs(st["k3_mean"] - (math.exp(dd) - 1 - dd)) < 1e-12
    a = np.float32(-1.0)
    c = np.nextafter(a, np.float32(0))  # d = one float32 step = 2^-24
    dd = float(np.float64(c) - np.float64(a))
    st, _ = _one_seq([a], [a], [c])
    series = dd * dd / 2 + dd ** 3 / 6 + dd ** 4 / 24
    assert abs(st["k3_mean"] - series) <= 1e-8 * series


def pin_k3_overflow_flag():
    st, _ = _one_seq([np.float32(-900.0)], [np.float32(-900.0)], [np.float32(-50.0)])
    assert not math.isfinite(st["k3_mean"])
    assert st["flags"] & oracle.FLAG_K3_OVERFLOW
    assert st["tis_mean"] == 2.0 and st["tis_clipped"] == 1


def pin_tis_clip():
    A = np.float32(-5.0)
    for d, w_want, clip in ((math.log(3.0), 2.0, 1), (math.log(1.5), 1.5, 0), (-1.0, math.exp(-1.0), 0)):
        C = np.float32(A + np.float32(d))
        st, w = _one_seq([A], [A], [C], cap=2.0)
        assert st["tis_clipped"] == clip
        assert abs(st["tis_mean"] - w_want) < 2e-6 * w_want
    st, w = _one_seq([A, A], [A, A], [np.float32(0.0), A], mask=[1, 0], cap=2.0)
    assert w[1] == 0.0 and w[0] == 2.0


def pin_active_ordinals():
    """first divergence and longest run count active tokens only; a masked gap does not break
    a run of differences ("Fault localization ...", Per-sequence observation patterns)."""
    mask = np.array([1, 1, 0, 1, 1, 1, 0, 1], dtype=np.uint8)
    A = np.full(8, -1.0, dtype=np.float32)
    B = A.copy()
    for pos in (1, 3, 4, 7, 6):  # 6 is masked
        B[pos] = np.float32(-1.5)
    st, _ = _one_seq(A, B, B, mask)
    p = st["pair"][0]
    assert p["mismatch_count"] == 4 and p["first_div"] == 1 and p["longest_run"] == 3
    assert st["n_valid"] == 6
    assert abs(p["mae"] - 4 * 0.5 / 6) < 1e-15 and abs(p["signed_mean"] - 4 * 0.5 / 6) < 1e-15
    assert p["max_abs_diff"] == 0.5


def pin_signed_zero_and_nan():
    """+0.0 and -0.0 differ bitwise but not in value; NaN on an active token is an error."""
    st, _ = _one_seq([np.float32(0.0)], [np.float32(-0.0)], [np.float32(0.0)])
    assert st["pair"][0]["mismatch_count"] == 1 and st["pair"][0]["max_abs_diff"] == 0.0
    assert st["pair"][2]["mismatch_count"] == 0
    try:
        _one_seq([np.float32(np.nan), np.float32(-1)], [np.float32(-1)] * 2, [np.float32(-1)] * 2)
    except oracle.OracleError as e:
        assert e.code == "NONFINITE"
    else:
        raise AssertionError("NaN on an active token must raise")
    st, _ = _one_seq([np.float32(np.nan), np.float32(-1)], [np.float32(-1)] * 2,
                     [np.float32(-1)] * 2, mask=[0, 1])
    assert st["n_valid"] == 1


def pin_error_contract():
    ok = np.zeros(8, np.float32)
    offs = np.array([0, 4, 8], dtype=np.int64)
    m = np.ones(8, np.uint8)
    cases = [
        ("SHAPE", (ok, ok[:7], ok, offs, m, 2.0)),
        ("BAD_MASK", (ok, ok, ok, offs, np.array([1, 2, 1, 1, 1, 1, 1, 1], np.uint8), 2.0)),
        ("EMPTY_SEQUENCE", (ok, ok, ok, offs, np.array([1, 1, 1, 1, 0, 0, 0, 0], np.uint8), 2.0)),
        ("INVALID_ARG", (ok, ok, ok, np.array([0, 5, 4], np.int64), m, 2.0)),
        ("INVALID_ARG", (ok, ok, ok, np.array([0, 4, 9], np.int64), m, 2.0)),
        ("INVALID_ARG", (ok, ok, ok, offs, m, 0.0)),
    ]
    for code, args in cases:
        try:
            oracle.oracle_compare(*args)
        except oracle.OracleError as e:
            assert e.code == code, (code, e.code)
        else:
            raise AssertionError(f"expected {code}")


def pin_bitwise_requests():
    """Two responses scored twice, one token changed by 0.5 in the first and a masked
    token changed in the second: per sequence the mismatch count, first divergence
    (active ordinal) and maximum |difference| are the hand-counted values, and a change on
    a masked token is not seen."""
    x = np.array([-1.0, -2.0, -3.0, -0.5, -0.25], np.float32)
    y = x.copy()
    y[1] = -2.5                       # sequence 0, ordinal 1
    y[3] = -7.0                       # sequence 1, masked out
    mask = np.array([1, 1, 1, 0, 1], np.uint8)
    offs = np.array([0, 3, 5], np.int64)
    st, _ = oracle.oracle_compare(x, y, y, offs, mask, 2.0)
    s0, s1 = st[0]["pair"][0], st[1]["pair"][0]
    assert (st[0]["n_valid"], st[1]["n_valid"]) == (3, 1)
    assert (s0["mismatch_count"], s0["first_div"], s0["longest_run"]) == (1, 1, 1)
    assert s0["max_abs_diff"] == 0.5 and s0["signed_mean"] == 0.5 / 3
    assert (s1["mismatch_count"], s1["first_div"], s1["max_abs_diff"]) == (0, -1, 0.0)
    assert sum(q["pair"][0]["mismatch_count"] for q in st) == 1


def pin_shift_fault_detected():
    """Scoring with token ids shifted by one inside each sequence is detected: every active
    token whose shifted id differs mismatches (Fault localization page: +-1 offsets)."""
    b = synth.make_tiny()
    A = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 1.0, b.eps)["logprob"]
    ids_s = b.token_ids.copy()
    for j in range(b.n_seq):
        a0, a1 = b.seq_offsets[j], b.seq_offsets[j + 1]
        ids_s[a0:a1] = np.roll(b.token_ids[a0:a1], -1)
    C = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, ids_s, 1.0, b.eps)["logprob"]
    A32, C32 = A.astype(np.float32), C.astype(np.float32)
    stats, _ = oracle.oracle_compare(A32, A32, C32, b.seq_offsets, b.mask, 2.0)
    for j, st in enumerate(stats):
        a0, a1 = b.seq_offsets[j], b.seq_offsets[j + 1]
        act = np.flatnonzero(b.mask[a0:a1]) + a0
        changed = int(np.sum(ids_s[act] != b.token_ids[act]))
        assert st["pair"][2]["mismatch_count"] == changed
        assert changed >= st["n_valid"] - 2
        assert st["pair"][2]["mae"] > 0.5
        assert st["pair"][0]["mismatch_count"] == 0


def pin_topk_renorm_example():
    """The page's k=2 renormalisation (used as a fixture check of the golden file only)."""
    gd = golden("topk_renormalisation.json")
    p = np.array(gd["probs"])
    keep = np.argsort(-p)[:gd["k"]]
    q = np.zeros_like(p)
    q[keep] = p[keep] / p[keep].sum()
    assert np.allclose(q, gd["renormalised"], atol=1e-15)


# ---------------------------------------------------------------------------
# extended diagnostics pins

def _diag1(A, B, C, mask=None, cap=2.0, lo=0.5, hi=1.5, top1=(None, None, None)):
    A = np.asarray(A, dtype=np.float32)
    n = A.shape[0]
    mask = np.ones(n, dtype=np.uint8) if mask is None else np.asarray(mask, dtype=np.uint8)
    return oracle.oracle_diag(A, np.asarray(B, np.float32), np.asarray(C, np.float32),
                              np.array([0, n], dtype=np.int64), mask, cap, lo, hi, top1)[0]


def pin_quantile_definition():
    """Type-7 quantiles: closed form on 0..99 and numpy's 'linear' method (a library routine
    the oracle does not call) on random data."""
    x = np.arange(100, dtype=np.float64)[::-1].copy()
    assert oracle.quantile_linear(x, 0.5) == 49.5
    assert abs(oracle.quantile_linear(x, 0.95) - 94.05) < 1e-12
    assert abs(oracle.quantile_linear(x, 0.99) - 98.01) < 1e-12
    g = np.random.default_rng(11)
    for n in (1, 2, 3, 7, 100, 1001):
        v = np.abs(g.standard_normal(n)) * 0.3
        for q in oracle.QUANTILES:
            ref = float(np.quantile(v, q, method="linear"))
            assert abs(oracle.quantile_linear(v, q) - ref) <= 1e-15 * max(1.0, abs(ref))


def pin_diag_quantiles_in_sequence():
    """|A - B| = 0.01 k on 101 active tokens (masked tokens interleaved) -> p50 = 0.5, p95 = 0.95,
    p99 = 0.99 (up to float32 rounding of the inputs)."""
    k = np.arange(101)
    A = np.full(202, -2.0, np.float32)
    B = A.copy()
    mask = np.zeros(202, np.uint8)
    mask[::2] = 1
    B[::2] = (A[::2].astype(np.float64) - 0.01 * k).astype(np.float32)
    B[1::2] = np.float32(-50.0)                   # masked: must not count
    st = _diag1(A, B, B, mask)
    assert st["n_valid"] == 101
    assert abs(st["abs_q50"][0] - 0.50) < 1e-6 and abs(st["abs_q95"][0] - 0.95) < 1e-6
    assert abs(st["abs_q99"][0] - 0.99) < 1e-6 and st["abs_q50"][1] == 0.0


def pin_diag_page_probability_mae():
    """p = 0.10 vs 0.12 (Debugging page, What a Logprob Difference Means): probability MAE 0.02
    while the logprob difference is 0.1823."""
    A = np.float32(math.log(0.10))
    C = np.float32(math.log(0.12))
    st = _diag1([A], [A], [C])
    assert abs(st["prob_mae"][2] - 0.02) < 1e-8 and st["prob_mae"][0] == 0.0
    assert abs(st["abs_q99"][2] - 0.1823215568) < 1e-6


def pin_diag_fig1_sequence():
    """Two tokens with the Figure 1 ratio w = 0.21 / 0.20 each: sequence ratio 1.1025, k1 sum
    -2 ln 1.05, k3 sum 2 (0.05 - ln 1.05), ratio error 0.05, mean w^2 1.1025."""
    A = np.float32(math.log(0.20))
    C = np.float32(math.log(0.21))
    st = _diag1([A, A], [A, A], [C, C], cap=2.0)
    d = float(np.float64(C) - np.float64(A))
    assert abs(d - math.log(1.05)) < 4e-7
    assert abs(st["log_ratio_sum"] - 2 * math.log(1.05)) < 1e-6
    assert abs(st["seq_tis"] - 1.1025) < 2e-6
    assert abs(st["k1_sum"] + 2 * math.log(1.05)) < 1e-6
    assert abs(st["k3_sum"] - 2 * (0.05 - math.log(1.05))) < 1e-7
    assert abs(st["ratio_err_mean"] - 0.05) < 1e-6
    assert abs(st["w2_mean"] - 1.1025) < 2e-6
    capped = _diag1([A, A], [A, A], [C, C], cap=1.1)
    assert capped["seq_tis"] == 1.1


def pin_diag_mis_and_flips():
    A = np.full(3, -4.0, np.float32)
    C = np.array([-4.0 + math.log(1.05), -4.0 + math.log(2.0), -4.0 - math.log(4.0)], np.float32)
    t_a = np.array([5, 6, 7])
    t_c = np.array([5, 9, 8])
    st = _diag1(A, A, C, lo=0.5, hi=1.5, top1=(t_a, t_a, t_c))
    assert st["mis_kept"] == 1
    assert abs(st["mis_mean"] - 1.05 / 3) < 1e-6
    assert st["top1_flips"] == [0, 2, 2]
    st2 = _diag1(A, A, C, lo=0.5, hi=1.5)
    assert st2["top1_flips"] == [-1, -1, -1]


def pin_diag_recorded_token():
    """One active token: every quantile equals its |difference| (the page's note that p95, p99
    and the maximum coincide for a single token)."""
    gd = golden("recorded_token_case1.json")
    s = {k: np.float32(v) for k, v in gd["scores"].items() if k != "A"}
    st = _diag1([s["B0"]], [s["B1"]], [s["C0"]])
    want = abs(float(np.float64(s["B0"]) - np.float64(s["B1"])))
    assert st["abs_q50"][0] == st["abs_q95"][0] == st["abs_q99"][0] == want
    assert round(want, 6) == gd["signed_differences_6dp"]["B0-B1"]


def pin_diag_quantiles_long_sequence():
    """Quantiles at any length: |A - B| = float32(k / 1000) for k = 0..40000 in a shuffled
    order with masked tokens between them; type-7 interpolation lands on order statistics
    k = 20000, 38000 and 39600 exactly (h = 40000 q is an integer)."""
    n = 40001
    g = np.random.default_rng(11)
    vals = (np.arange(n) / 1000.0).astype(np.float32)
    g.shuffle(vals)
    A = np.zeros(2 * n, np.float32)
    A[0::2] = vals
    A[1::2] = np.float32(9.0)                      # masked: must not enter the statistics
    mask = np.zeros(2 * n, np.uint8)
    mask[0::2] = 1
    B = np.zeros(2 * n, np.float32)
    out = oracle.oracle_diag(A, B, B, np.array([0, 2 * n], np.int64), mask, 2.0, 0.5, 2.0)
    st = out[0]
    assert st["n_valid"] == n and st["flags"] == 0
    for key, k in (("abs_q50", 20000), ("abs_q95", 38000), ("abs_q99", 39600)):
        assert st[key][0] == float(np.float32(k / 1000.0)), (key, st[key][0])
        assert st[key][1] == 0.0


# ---------------------------------------------------------------------------
# processed (top-k / top-p) logprob pins

def _proc(z_targets, x, tau, k, p):
    h, g, W, _ = exact_logit_head(z_targets)
    return oracle.oracle_processed_logprob(h, g, W, np.array([x], np.int32), tau, 0.0, k, p)


def pin_processed_page_topk():
    """Top-k with k = 2 turns (0.50, 0.30, 0.20) into (0.625, 0.375, 0) (Debugging page,
    Make Sure Both Scores Describe the Same Probability)."""
    gd = golden("topk_renormalisation.json")
    z = [math.log(v) for v in gd["probs"]]
    for x, want in enumerate(gd["renormalised"]):
        out = _proc(z, x, 1.0, gd["k"], 1.0)
        if want == 0.0:
            assert out["logprob"][0] == -math.inf
        else:
            assert abs(out["logprob"][0] - math.log(want)) < 1e-12
        assert out["kept"][0] == 2
    assert abs(_proc(z, 0, 1.0, 2, 1.0)["lse_kept"][0] - math.log(0.8)) < 1e-12


def pin_processed_top_p_boundary():
    """Top-p on (0.5, 0.3, 0.2): p = 0.7 keeps {0, 1} (the prefix reaching 0.8 >= 0.7),
    p = 0.81 keeps all three, p = 0.4 keeps only token 0."""
    z = [math.log(0.5), math.log(0.3), math.log(0.2)]
    o = _proc(z, 1, 1.0, 3, 0.7)
    assert o["kept"][0] == 2 and abs(o["logprob"][0] - math.log(0.375)) < 1e-12
    assert _proc(z, 2, 1.0, 3, 0.7)["logprob"][0] == -math.inf
    o = _proc(z, 2, 1.0, 3, 0.81)
    assert o["kept"][0] == 3 and abs(o["logprob"][0] - math.log(0.2)) < 1e-12
    o = _proc(z, 0, 1.0, 3, 0.4)
    assert o["kept"][0] == 1 and o["logprob"][0] == 0.0


def pin_processed_ties_and_temperature():
    """Equal logits at the top-k cut keep the lower ids; temperature is applied before
    filtering: on z = (0, 1, 2, 3) with tau = 0.5, k = 2 the kept scores are 6 - lse, 4 - lse
    with lse = ln(e^6 + e^4)."""
    o = _proc([1.0, 1.0, 1.0, 0.0], 1, 1.0, 2, 1.0)
    assert abs(o["logprob"][0] - math.log(0.5)) < 1e-12
    assert _proc([1.0, 1.0, 1.0, 0.0], 2, 1.0, 2, 1.0)["logprob"][0] == -math.inf
    lse = math.log(math.exp(6.0) + math.exp(4.0))
    o = _proc([0.0, 1.0, 2.0, 3.0], 2, 0.5, 2, 1.0)
    assert abs(o["logprob"][0] - (4.0 - lse)) < 1e-12
    assert abs(o["lse_kept"][0] - lse) < 1e-12


def pin_processed_reduces_to_raw():
    """k = V and p = 1 keep the whole vocabulary: the processed score is the raw score."""
    b = synth.make_custom(T=12, d=64, V=90, temperature=0.8, tag="proc_raw")
    raw = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 0.8, b.eps)
    pr = oracle.oracle_processed_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 0.8,
                                         b.eps, 90, 1.0)
    assert np.max(np.abs(raw["logprob"] - pr["logprob"])) < 1e-12
    assert np.all(pr["kept"] == 90)


def pin_processed_library_topk():
    """torch.topk + log_softmax on the kept logits (library routines the oracle does not call)."""
    import torch
    b = synth.make_custom(T=10, d=128, V=300, temperature=0.7, tag="proc_lib")
    y = oracle.rmsnorm(oracle.widen_bf16(b.hidden_gen), oracle.widen_bf16(b.head.gamma), b.eps)
    z = torch.from_numpy(oracle.logits(y, b.head.W))
    k = 17
    vals, idx = torch.topk(z, k, dim=1)
    ls = torch.log_softmax(vals / 0.7, dim=1)
    ids = idx[:, 3].numpy().astype(np.int32)              # a kept target in every row
    pr = oracle.oracle_processed_logprob(b.hidden_gen, b.head.gamma, b.head.W, ids, 0.7, b.eps,
                                         k, 1.0)
    assert np.max(np.abs(pr["logprob"] - ls[:, 3].numpy())) < 1e-12


def pin_processed_head():
    """The top-k head: k = 2 on (0.5, 0.3, 0.2) gives ids (0, 1) with ln 0.625, ln 0.375;
    k = 3, p = 0.7 keeps two and reports -inf for the third; torch.topk (a library routine)
    gives the same ids on distinct logits and log_softmax of the top-k values the same
    logprobs when p = 1."""
    import torch
    z = np.log(np.array([0.5, 0.3, 0.2]))
    ids, lp = oracle.process_head(z, 1.0, 2, 1.0)
    assert list(ids) == [0, 1]
    assert np.max(np.abs(lp - np.log([0.625, 0.375]))) < 1e-12
    ids, lp = oracle.process_head(z, 1.0, 3, 0.7)
    assert list(ids) == [0, 1, 2] and lp[2] == -math.inf
    assert np.max(np.abs(lp[:2] - np.log([0.625, 0.375]))) < 1e-12
    ids, lp = oracle.process_head(np.array([1.0, 1.0, 1.0, 0.0]), 1.0, 2, 1.0)
    assert list(ids) == [0, 1]                     # ties keep the lower ids
    b = synth.make_custom(T=6, d=128, V=300, temperature=0.7, tag="proc_head")
    pr = oracle.oracle_processed_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 0.7,
                                         b.eps, 9, 1.0)
    y = oracle.rmsnorm(oracle.widen_bf16(b.hidden_gen), oracle.widen_bf16(b.head.gamma), b.eps)
    vals, idx = torch.topk(torch.from_numpy(oracle.logits(y, b.head.W)), 9, dim=1)
    assert np.array_equal(pr["topk_ids"], idx.numpy())
    ls = torch.log_softmax(vals / 0.7, dim=1).numpy()
    assert np.max(np.abs(pr["topk_logprob"] - ls)) < 1e-12


# ---------------------------------------------------------------------------
# FP8 (e4m3) head pins

def _e4m3_table():
    """All finite e4m3 values decoded from the bit layout (1 sign, 4 exponent bits with
    bias 7, 3 mantissa bits; code 0x7F / 0xFF is NaN), with their codes."""
    vals, codes = [], []
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        vals.append(-v if s else v)
        codes.append(c)
    vals, codes = np.array(vals), np.array(codes)
    keep = ~((vals == 0) & (codes == 0x80))
    vals, codes = vals[keep], codes[keep]
    o = np.argsort(vals, kind="stable")
    return vals[o], codes[o]


def pin_e4m3_rounding_exhaustive():
    """Nearest-even e4m3 rounding against an exhaustive search of the 253 finite values,
    including exact ties; torch's float8_e4m3fn conversion (a library routine) agrees."""
    import torch
    vals, codes = _e4m3_table()
    assert vals.max() == 448.0 and vals[vals > 0].min() == 2.0 ** -9
    g = np.random.default_rng(17)
    x = np.concatenate([g.uniform(-448, 448, 20000), g.standard_normal(5000) * 0.01,
                        (vals[:-1] + vals[1:]) / 2.0])
    hi = np.clip(np.searchsorted(vals, x, side="left"), 1, vals.size - 1)
    lo = hi - 1
    dlo, dhi = np.abs(x - vals[lo]), np.abs(vals[hi] - x)
    pick = (dhi < dlo) | ((dhi == dlo) & (codes[hi] % 2 == 0))
    want = np.where(pick, vals[hi], vals[lo])
    got = oracle.e4m3_round(x)
    assert np.array_equal(got, want)
    tq = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(tq, want)
    assert oracle.e4m3_round(np.array([1.0625]))[0] == 1.0       # tie -> even mantissa
    assert oracle.e4m3_round(np.array([1.1875]))[0] == 1.25


def pin_fp8_scale_rule():
    """The scale is the smallest power of two s with max|row| / s <= 448."""
    for amax, s in ((448.0, 1.0), (449.0, 2.0), (224.0, 0.5), (1.0, 2.0 ** -8), (0.0, 1.0),
                    (448.0 * 2 ** -20, 2.0 ** -20), (900.0, 4.0)):
        assert oracle.fp8_scale(amax) == s, (amax, s)
    g = np.random.default_rng(3)
    for amax in np.abs(g.standard_normal(200)) * 10 ** g.uniform(-3, 3, 200):
        s = oracle.fp8_scale(float(amax))
        assert amax / s <= 448 < amax / (s / 2)
        assert math.frexp(s)[0] == 0.5


def pin_fp8_exact_head():
    """When y and W are already e4m3 values with unit scales, the FP8 oracle equals the bf16
    oracle; a scale applied to a whole W row cancels exactly in the dequantised logits."""
    z = [1.0, 2.0, 0.5, -1.5, 3.0, 0.0, -0.25, 1.75]
    h = np.full((1, 8), trunc_bf16_bits(1.0), dtype=np.uint16)
    g = np.full(8, trunc_bf16_bits(0.0), dtype=np.uint16)
    g[0] = trunc_bf16_bits(1.0)                     # y = (1, 0, ..., 0): an e4m3 value
    W = np.zeros((8, 8), dtype=np.uint16)
    W[:, 0] = [trunc_bf16_bits(v) for v in z]       # every logit is an e4m3 value
    for x in range(8):
        a = oracle.oracle_logprob(h, g, W, np.array([x], np.int32), 0.9, 0.0)
        b = oracle.oracle_logprob_fp8(h, g, W, np.array([x], np.int32), 0.9, 0.0)
        assert a["logprob"][0] == b["logprob"][0] and a["top1"][0] == b["top1"][0]
    W2 = W.copy()
    W2[:, 0] = [trunc_bf16_bits(v * 8.0) for v in z]  # same row, 8x larger: scale absorbs it
    b2 = oracle.oracle_logprob_fp8(h, g, W2, np.array([4], np.int32), 1.0, 0.0)
    lse = math.log(sum(math.exp(8.0 * v) for v in z))
    assert abs(b2["logprob"][0] - (8.0 * 3.0 - lse)) < 1e-12


def pin_fp8_quantized_dot_product():
    """Random rows: z_fp8 = (Q(y) s_y) . (Q(W) s_W) written out term by term in exact rational
    arithmetic matches the oracle's logits to 1e-12."""
    b = synth.make_custom(T=2, d=64, V=12, tag="fp8dot")
    y = oracle.rmsnorm(oracle.widen_bf16(b.hidden_gen), oracle.widen_bf16(b.head.gamma), b.eps)
    Wf = oracle.widen_bf16(b.head.W)
    out = oracle.oracle_logprob_fp8(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 1.0, b.eps)
    for t in range(2):
        sy = oracle.fp8_scale(float(np.max(np.abs(y[t]))))
        qy = [Fraction(float(v)) * Fraction(sy) for v in oracle.e4m3_round(y[t] / sy)]
        zs = []
        for v in range(12):
            sw = oracle.fp8_scale(float(np.max(np.abs(Wf[v]))))
            qw = [Fraction(float(u)) * Fraction(sw) for u in oracle.e4m3_round(Wf[v] / sw)]
            zs.append(float(sum(a * c for a, c in zip(qy, qw))))
        m = max(zs)
        lse = m + math.log(sum(math.exp(v - m) for v in zs))
        assert abs(out["lse"][t] - lse) < 1e-12
        assert abs(out["logprob"][t] - (zs[b.token_ids[t]] - lse)) < 1e-12


def pin_fp8_y_is_the_bf16_heads_y():
    """The FP8 head quantises the y of the bf16 head: fp64 RMSNorm (torch's rms_norm, a
    routine the oracle does not call) rounded once to the nearest bf16 (table search).
    Logits built from that y and the pinned quantiser give the oracle's lse to 1e-12."""
    import torch
    b = synth.make_custom(T=6, d=64, V=20, tag="fp8y")
    h64 = torch.from_numpy(oracle.widen_bf16(b.hidden_gen))
    g64 = torch.from_numpy(oracle.widen_bf16(b.head.gamma))
    y = brute_nearest_bf16(torch.nn.functional.rms_norm(h64, (64,), g64, eps=b.eps).numpy())
    cy, sy = oracle.quantize_rows(y)
    cw, sw = oracle.quantize_rows(oracle.widen_bf16(b.head.W))
    z = (cy * sy[:, None]) @ (cw * sw[:, None]).T
    m = z.max(axis=1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    out = oracle.oracle_logprob_fp8(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 1.0, b.eps)
    assert np.max(np.abs(out["lse"] - lse)) < 1e-12, np.max(np.abs(out["lse"] - lse))


def _f32(x: float) -> float:
    """Round a Python float (fp64) to the nearest fp32 value, ties to even."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def pin_bf16_choices_brute():
    """bf16_choices against brute force: the set of nearest-bf16 roundings (table search)
    of 64 points spread over [x - m|x|, x + m|x|] equals {lo, hi}, on values placed at,
    near and away from rounding midpoints."""
    vals, _ = _all_finite_bf16()
    g = np.random.default_rng(5)
    i = np.flatnonzero((np.abs(vals[:-1]) > 1e-30) & (np.abs(vals[1:]) < 1e30))
    i = g.choice(i, 400)
    a = vals[i]
    mids = (vals[i] + vals[i + 1]) / 2                       # rounding midpoints
    xs = np.concatenate([mids, mids * (1 + 3e-7), mids * (1 - 3e-7), a, g.standard_normal(200)])
    for m in (0.0, 1e-7, 4.3e-6):
        lo, hi = oracle.bf16_choices(xs, m)
        for i, x in enumerate(xs):
            pts = x + np.linspace(-1.0, 1.0, 65) * abs(x) * m
            got = set(brute_nearest_bf16(pts).tolist())
            assert got == {float(lo[i]), float(hi[i])}, (x, m, got, lo[i], hi[i])
    lo, hi = oracle.bf16_choices(mids, 1e-6)
    assert np.all(lo < hi)                                   # a midpoint is always ambiguous


def pin_fp8_admissible_margin_zero():
    """With margin 0 the admissible set is the oracle's own result, alone."""
    b = synth.make_custom(T=5, d=128, V=50, temperature=0.8, tag="adm0")
    out = oracle.oracle_logprob_fp8(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 0.8, b.eps)
    adm = oracle.oracle_logprob_fp8_admissible(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids,
                                               0.8, b.eps, 0.0)
    for t, alts in enumerate(adm):
        assert len(alts) == 1
        assert alts[0]["logprob"] == out["logprob"][t] and alts[0]["top1"] == out["top1"][t]


def pin_fp8_admissible_scale_flip():
    """A row whose maximum lies on a bf16 rounding midpoint (7.015625, between 7.0 and
    7.03125) whose two neighbours give different row scales (2^-6 and 2^-5): the codes of
    the maximum agree, but a tiny element (1.8358e-5, in e4m3's subnormal range) becomes
    2^-15 under one scale and 0 under the other.  The admissible set must hold both
    results, computed here by hand: logits (7 + 64 * 2^-15, 7, 0, 0) and (7, 7, 0, 0)."""
    d = 64
    h = np.zeros(d)
    h[0], h[2] = 7.0, 2.0 ** -16
    g = np.ones(d)
    g[2] = 1.203125
    eps = 1.0 / (7.015625 / 7.0) ** 2 - float(np.mean(h * h))     # rstd = 7.015625 / 7
    W = np.zeros((4, d))
    W[0, 0], W[0, 2], W[1, 0] = 1.0, 64.0, 1.0
    bits = lambda a: np.array([[trunc_bf16_bits(v) for v in r] for r in np.atleast_2d(a)],
                              dtype=np.uint16)
    hb, gb, Wb = bits(h), bits(g)[0], bits(W)
    assert np.array_equal(oracle.widen_bf16(hb)[0], h) and np.array_equal(oracle.widen_bf16(Wb), W)
    adm = oracle.oracle_logprob_fp8_admissible(hb, gb, Wb, np.array([0], np.int32), 1.0, eps,
                                               1e-6)[0]
    assert adm is not None and len(adm) == 2, adm
    want = []
    for z0 in (7.0 + 64 * 2.0 ** -15, 7.0):
        z = np.array([z0, 7.0, 0.0, 0.0])
        lse = math.log(sum(math.exp(v) for v in z))
        want.append((z0 - lse, lse))
    got = sorted((a["logprob"], a["lse"]) for a in adm)
    for (lp_g, lse_g), (lp_w, lse_w) in zip(got, sorted(want)):
        assert abs(lp_g - lp_w) < 1e-12 and abs(lse_g - lse_w) < 1e-12, (got, want)
    # the oracle's own result is one of them (the tie rounds to the even 7.0: scale 2^-6)
    base = oracle.oracle_logprob_fp8(hb, gb, Wb, np.array([0], np.int32), 1.0, eps)
    assert abs(base["lse"][0] - want[0][1]) < 1e-12


def _rmsnorm_fp32_generic(h, g, eps, order):
    """An fp32 RMSNorm in a generic summation order ('fwd': one running sum in element
    order, 'rev': reversed, 'pair': numpy's float32 pairwise sum), every other step in fp32
    as the textbook formula reads.  Not any kernel's order."""
    f32 = np.float32
    sq = (h * h).astype(f32)                                  # exact: 8-bit significands
    if order == "pair":
        ss = np.sum(sq, axis=1, dtype=f32)
    else:
        cols = range(h.shape[1]) if order == "fwd" else range(h.shape[1] - 1, -1, -1)
        ss = np.zeros(h.shape[0], f32)
        for k in cols:
            ss = ss + sq[:, k]
    rstd = f32(1.0) / np.sqrt(ss / f32(h.shape[1]) + f32(eps))
    y32 = (h.astype(f32) * rstd[:, None]) * g.astype(f32)[None, :]
    return oracle.round_to_bf16(y32.astype(np.float64))


def pin_fp8_admissible_covers_fp32_evaluations():
    """fp32 RMSNorms in three generic orders, each followed by the FP8 quantisation and an
    fp64 head, land inside the admissible set taken with their error bound
    ((d + 1) / 2 + 5) 2^-24 (sum of d squares, /d, + eps, sqrt, 1/x, two products), and
    some of them really take the other rounding (so the set is not the base alone)."""
    d, T, V = 512, 12000, 16
    b = synth.make_custom(T=T, d=d, V=V, tag="adm32")
    h = oracle.widen_bf16(b.hidden_gen)
    g = oracle.widen_bf16(b.head.gamma)
    margin = ((d + 1) / 2 + 5) * 2.0 ** -24
    Wq = oracle.dequantized_weights(b.head.W)
    base_y = oracle.rmsnorm(h, g, b.eps)
    ys = {o: _rmsnorm_fp32_generic(h, g, b.eps, o) for o in ("fwd", "rev", "pair")}
    moved = np.zeros(T, dtype=bool)
    for y in ys.values():
        cb, sb = oracle.quantize_rows(base_y)
        cy, sy = oracle.quantize_rows(y)
        moved |= np.any(cb * sb[:, None] != cy * sy[:, None], axis=1)
    rows = np.flatnonzero(moved)
    assert rows.size >= 3, rows.size                         # the pin has teeth
    adm = oracle.oracle_logprob_fp8_admissible(b.hidden_gen[rows], b.head.gamma, b.head.W,
                                               b.token_ids[rows], 1.0, b.eps, margin, Wq=Wq)
    for y in ys.values():
        cy, sy = oracle.quantize_rows(y[rows])
        z = (cy * sy[:, None]) @ Wq.T
        m = z.max(axis=1)
        lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        for i, t in enumerate(rows):
            alts = adm[i]
            assert alts is not None and len(alts) >= 2
            assert min(abs(a["lse"] - lse[i]) for a in alts) < 1e-12, (t, lse[i])


# ---------------------------------------------------------------------------
# FP32 head pins

def pin_fp32_head_mpmath():
    """FP32 head rows evaluated end to end at 50 digits (mpmath) with fp32 weights that are
    not bf16 values and y never rounded; the oracle must agree to 1e-12."""
    import mpmath
    mpmath.mp.dps = 50
    b = synth.make_custom(T=3, d=16, V=40, temperature=0.7, eps=1e-6, tag="mp32")
    W32 = synth.fp32_weights(b.head)
    assert np.mean(oracle.round_to_bf16(W32.astype(np.float64)) != W32) > 0.9
    out = oracle.oracle_logprob_fp32(b.hidden_gen, b.head.gamma, W32, b.token_ids, 0.7, 1e-6)
    hb = oracle.widen_bf16(b.hidden_gen)
    gb = oracle.widen_bf16(b.head.gamma)
    for t in range(b.T):
        h = [mpmath.mpf(float(v)) for v in hb[t]]
        rstd = 1 / mpmath.sqrt(mpmath.fsum(v * v for v in h) / len(h) + mpmath.mpf(1e-6))
        y = [v * rstd * mpmath.mpf(float(gb[i])) for i, v in enumerate(h)]
        z = [mpmath.fsum(y[i] * mpmath.mpf(float(W32[v, i])) for i in range(len(y)))
             for v in range(b.V)]
        s = [zz / mpmath.mpf(0.7) for zz in z]
        lse = mpmath.log(mpmath.fsum(mpmath.exp(v) for v in s))
        x = int(b.token_ids[t])
        assert abs(float(s[x] - lse) - out["logprob"][t]) < 1e-12
        assert abs(float(lse) - out["lse"][t]) < 1e-12
        assert out["top1"][t] == int(np.argmax([float(v) for v in z]))


def pin_fp32_head_reduces_to_bf16():
    """With |h| = 2 everywhere and eps = 0, y = (h / 2) gamma is a bf16 value, so rounding y
    changes nothing; with bf16-valued W the FP32 oracle equals the bf16 oracle exactly.
    With fp32 weights the two differ (the head is not silently rounded)."""
    b = synth.make_custom(T=5, d=64, V=300, tag="r32")
    h = np.where((np.arange(5 * 64).reshape(5, 64) % 5) == 0, 0xC000, 0x4000).astype(np.uint16)
    Wf = oracle.widen_bf16(b.head.W).astype(np.float32)
    a = oracle.oracle_logprob(h, b.head.gamma, b.head.W, b.token_ids, 0.8, 0.0)
    c = oracle.oracle_logprob_fp32(h, b.head.gamma, Wf, b.token_ids, 0.8, 0.0)
    for k in ("logprob", "lse", "top1"):
        assert np.array_equal(a[k], c[k]), k
    c2 = oracle.oracle_logprob_fp32(h, b.head.gamma, synth.fp32_weights(b.head), b.token_ids,
                                    0.8, 0.0)
    assert np.max(np.abs(c2["lse"] - a["lse"])) > 1e-6


def pin_fp32_head_torch():
    """fp64 torch: rms_norm (library routine), matmul, log_softmax and argmax agree with the
    FP32 oracle to 1e-12 on a ragged shape."""
    import torch
    b = synth.make_custom(T=7, d=192, V=777, temperature=1.3, eps=1e-5, tag="t32")
    W32 = synth.fp32_weights(b.head)
    out = oracle.oracle_logprob_fp32(b.hidden_gen, b.head.gamma, W32, b.token_ids, 1.3, 1e-5)
    h = torch.from_numpy(oracle.widen_bf16(b.hidden_gen))
    g = torch.from_numpy(oracle.widen_bf16(b.head.gamma))
    y = torch.nn.functional.rms_norm(h, (192,), weight=g, eps=1e-5)
    z = y @ torch.from_numpy(W32.astype(np.float64)).T
    ls = torch.log_softmax(z / 1.3, dim=1)
    ids = torch.from_numpy(b.token_ids.astype(np.int64))
    assert np.max(np.abs(ls.gather(1, ids[:, None])[:, 0].numpy() - out["logprob"])) < 1e-12
    assert np.array_equal(torch.argmax(z, dim=1).numpy(), out["top1"])


# ---------------------------------------------------------------------------
# Backward pins

def _bwd_case(tag, T=4, d=16, V=40, tau=0.7):
    b = synth.make_custom(T=T, d=d, V=V, temperature=tau, tag=tag)
    g = np.random.default_rng(sum(tag.encode())).standard_normal(T)
    return b, g


def pin_backward_finite_differences():
    """dL/dy and dL/dW against central differences of L = sum_t g_t logprob_t, the forward
    taken through the oracle's lse_stats on z = y W^T (fp64, step 1e-6)."""
    b, g = _bwd_case("bwdfd")
    tau = b.temperature
    out = oracle.oracle_logprob_backward(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, tau,
                                         b.eps, g)
    y = out["y"]
    W = oracle.widen_bf16(b.head.W)
    ids = b.token_ids.astype(np.int64)

    def loss(yy, WW):
        s, lse = oracle.lse_stats(yy @ WW.T, tau)
        return float(np.sum(g * (s[np.arange(len(ids)), ids] - lse)))

    h = 1e-6
    for t, i in ((0, 0), (1, 5), (3, 15), (2, 7)):
        e = np.zeros_like(y)
        e[t, i] = h
        fd = (loss(y + e, W) - loss(y - e, W)) / (2 * h)
        assert abs(fd - out["dy"][t, i]) < 1e-7 * max(1.0, abs(fd)), (t, i)
    for v, i in ((0, 0), (int(ids[0]), 3), (39, 15), (17, 8)):
        e = np.zeros_like(W)
        e[v, i] = h
        fd = (loss(y, W + e) - loss(y, W - e)) / (2 * h)
        assert abs(fd - out["dW"][v, i]) < 1e-7 * max(1.0, abs(fd)), (v, i)


def pin_backward_torch_autograd():
    """torch fp64 autograd of sum_t g_t log_softmax(y W^T / tau)[t, x_t] (a library routine)
    matches dL/dy and dL/dW to 1e-12 on a ragged shape."""
    import torch
    b, g = _bwd_case("bwdtorch", T=9, d=48, V=333, tau=1.3)
    out = oracle.oracle_logprob_backward(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 1.3,
                                         b.eps, g, vocab_block=100)
    y = torch.tensor(out["y"], requires_grad=True)
    W = torch.tensor(oracle.widen_bf16(b.head.W), requires_grad=True)
    lp = torch.log_softmax(y @ W.T / 1.3, dim=1)
    ids = torch.from_numpy(b.token_ids.astype(np.int64))
    (torch.from_numpy(g) * lp.gather(1, ids[:, None])[:, 0]).sum().backward()
    assert np.max(np.abs(y.grad.numpy() - out["dy"])) < 1e-12
    assert np.max(np.abs(W.grad.numpy() - out["dW"])) < 1e-12


def pin_backward_invariants():
    """Each G row sums to zero (the probabilities sum to one), so every column of dW sums to
    zero; g = 0 gives zero gradients; a one-word vocabulary has logprob 0 and no gradient;
    an invalid token id row contributes nothing; the bounds dominate the results."""
    b, g = _bwd_case("bwdinv", T=6, d=32, V=50, tau=0.9)
    ids = b.token_ids.copy()
    ids[2] = 50
    out = oracle.oracle_logprob_backward(b.hidden_gen, b.head.gamma, b.head.W, ids, 0.9, b.eps, g)
    assert np.max(np.abs(out["dW"].sum(axis=0))) < 1e-12
    assert np.all(out["dy"][2] == 0.0)
    assert np.all(np.abs(out["dy"]) <= out["bound_dy"] + 1e-15)
    assert np.all(np.abs(out["dW"]) <= out["bound_dW"] + 1e-15)
    z = oracle.backward.logit_grad(np.random.default_rng(1).standard_normal((3, 7)),
                                   np.array([0, 6, 3]), np.ones(3), 0.5)
    assert np.max(np.abs(z.sum(axis=1))) < 1e-15
    zero = oracle.oracle_logprob_backward(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids,
                                          0.9, b.eps, np.zeros(6))
    assert not np.any(zero["dy"]) and not np.any(zero["dW"])
    one = oracle.oracle_logprob_backward(b.hidden_gen, b.head.gamma, b.head.W[:1],
                                         np.zeros(6, np.int32), 0.9, b.eps, g)
    assert np.max(np.abs(one["dy"])) < 1e-15 and np.max(np.abs(one["dW"])) < 1e-15


def pin_backward_temperature_closed_form():
    """Two-word vocabulary, one row, y = (1), W = (a, b): logprob of word 0 is
    -log(1 + e^((b - a) / tau)), so dL/dy = (a - b) q / tau with q = sigmoid((b - a) / tau)."""
    a, bb, tau = 1.5, -0.25, 0.6
    h = np.array([[0x3F80]], dtype=np.uint16)            # h = 1
    gam = np.array([0x3F80], dtype=np.uint16)            # gamma = 1 -> y = 1 (eps = 0)
    W = np.array([[trunc_bf16_bits(a)], [trunc_bf16_bits(bb)]], dtype=np.uint16)
    out = oracle.oracle_logprob_backward(h, gam, W, np.array([0]), tau, 0.0, np.array([1.0]))
    q = 1.0 / (1.0 + math.exp(-(bb - a) / tau))
    assert abs(out["dy"][0, 0] - (a - bb) * q / tau) < 1e-14
    assert abs(out["dW"][0, 0] - q / tau) < 1e-14 and abs(out["dW"][1, 0] + q / tau) < 1e-14


def pin_rmsnorm_backward_finite_differences():
    """dL/dh and dL/dgamma of L = sum dy * y(h, gamma) (y unrounded) against central
    differences, and torch fp64 autograd of rms_norm (a library routine)."""
    import torch
    b = synth.make_custom(T=5, d=24, V=4, tag="rmsbwd")
    h = oracle.widen_bf16(b.hidden_gen)
    g = oracle.widen_bf16(b.head.gamma)
    dy = np.random.default_rng(9).standard_normal(h.shape)
    eps = 1e-5
    dh, dgam = oracle.rmsnorm_backward(h, g, eps, dy)

    def loss(hh, gg):
        return float(np.sum(dy * oracle.rmsnorm_unrounded(hh, gg, eps)))

    step = 1e-6
    for t, i in ((0, 0), (2, 7), (4, 23)):
        e = np.zeros_like(h)
        e[t, i] = step
        fd = (loss(h + e, g) - loss(h - e, g)) / (2 * step)
        assert abs(fd - dh[t, i]) < 1e-7 * max(1.0, abs(fd)), (t, i)
    for i in (0, 11, 23):
        e = np.zeros_like(g)
        e[i] = step
        fd = (loss(h, g + e) - loss(h, g - e)) / (2 * step)
        assert abs(fd - dgam[i]) < 1e-7 * max(1.0, abs(fd)), i
    ht = torch.tensor(h, requires_grad=True)
    gt = torch.tensor(g, requires_grad=True)
    y = torch.nn.functional.rms_norm(ht, (24,), weight=gt, eps=eps)
    (y * torch.from_numpy(dy)).sum().backward()
    assert np.max(np.abs(ht.grad.numpy() - dh)) < 1e-12
    assert np.max(np.abs(gt.grad.numpy() - dgam)) < 1e-12


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
