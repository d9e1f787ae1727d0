"""tim_compare_diag (through the C ABI) against the fp64 diagnostics oracle run on the
same score arrays."""
import math

import numpy as np
import pytest

import oracle
from parity import cuda_tensor

pytestmark = pytest.mark.gpu

REL = 1e-9
EPS64 = 2.0 ** -52


@pytest.fixture(scope="module")
def tim():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import rollout_logprob_consistency_gb300 as tim
    return tim


def close(g, r, scale, extra=0.0):
    if g == r or (math.isnan(g) and math.isnan(r)):
        return True
    return abs(g - r) <= REL * max(abs(r), scale) + extra


def assert_diag_parity(g_list, r_list, d_abs_sum, what=""):
    """d_abs_sum[j] = sum |d| of sequence j (floor for the signed sums)."""
    assert len(g_list) == len(r_list)
    skip = (oracle.FLAG_BAD_MASK | oracle.FLAG_BAD_OFFSETS | oracle.FLAG_EMPTY |
            oracle.FLAG_NONFINITE)
    for j, (g, r) in enumerate(zip(g_list, r_list)):
        tag = f"{what} seq {j}"
        assert g["flags"] == r["flags"], (tag, g["flags"], r["flags"])
        assert g["n_valid"] == r["n_valid"], tag
        if r["flags"] & skip:
            continue
        # exact order statistics and the interpolation rounded operation by operation
        for k in ("abs_q50", "abs_q95", "abs_q99"):
            for p in range(3):
                a, b = g[k][p], r[k][p]
                assert (math.isnan(a) and math.isnan(b)) or a == b, (tag, k, p, a, b)
        assert g["top1_flips"] == r["top1_flips"], tag
        assert g["mis_kept"] == r["mis_kept"], tag
        for p in range(3):
            assert close(g["prob_mae"][p], r["prob_mae"][p], r["prob_mae"][p]), (tag, "prob", p)
        n = r["n_valid"]
        assert close(g["log_ratio_sum"], r["log_ratio_sum"], d_abs_sum[j]), (tag, "sum d")
        assert close(g["k1_sum"], r["k1_sum"], d_abs_sum[j]), (tag, "k1")
        assert close(g["k3_sum"], r["k3_sum"], r["k3_sum"], 4 * EPS64 * d_abs_sum[j]), (tag, "k3")
        assert close(g["ratio_err_mean"], r["ratio_err_mean"], r["ratio_err_mean"],
                     4 * EPS64 * d_abs_sum[j] / n), (tag, "ratio err")
        assert close(g["mis_mean"], r["mis_mean"], r["mis_mean"]), (tag, "mis")
        assert close(g["w2_mean"], r["w2_mean"], r["w2_mean"]), (tag, "w2")
        # seq_tis = exp(sum d): relative error follows the absolute error of the sum
        assert close(g["seq_tis"], r["seq_tis"], r["seq_tis"],
                     r["seq_tis"] * 2 * REL * max(1.0, d_abs_sum[j])), (tag, "seq tis")


def make_case(T, seed, n_seq=6, heavy=2.0):
    g = np.random.default_rng(seed)
    A = (-np.abs(g.standard_normal(T)) * 4).astype(np.float32)
    B = A.copy()
    flip = g.random(T) < 0.3
    B[flip] = A[flip] + (g.standard_normal(flip.sum()) * 1e-3).astype(np.float32)
    C = (B + (g.standard_normal(T) * 0.05).astype(np.float32)).astype(np.float32)
    k = g.random(T) < 0.02
    C[k] += np.float32(heavy)
    cuts = np.sort(g.choice(np.arange(1, T), size=min(T - 1, n_seq - 1), replace=False))
    offs = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    mask = (g.random(T) < 0.8).astype(np.uint8)
    for j in range(len(offs) - 1):
        if mask[offs[j]:offs[j + 1]].sum() == 0:
            mask[offs[j + 1] - 1] = 1
    tops = [g.integers(0, 50, T).astype(np.int32) for _ in range(3)]
    tops[1] = np.where(g.random(T) < 0.9, tops[0], tops[1]).astype(np.int32)
    return A, B, C, offs, mask, tops


def run(tim, A, B, C, offs, mask, tops, cap=2.0, lo=0.5, hi=1.5, check=True):
    tt = [None if t is None else cuda_tensor(t) for t in tops]
    arr = tim.compare_diag(cuda_tensor(A), cuda_tensor(B), cuda_tensor(C), cuda_tensor(offs),
                           cuda_tensor(mask), cap, lo, hi, top1=tt, check=check)
    return tim.diag_to_dicts(arr)


def d_abs(A, C, offs, mask):
    out = []
    for j in range(len(offs) - 1):
        a, b = int(offs[j]), int(offs[j + 1])
        if not (0 <= a <= b <= len(A)):
            out.append(0.0)
            continue
        act = np.flatnonzero(mask[a:b] == 1) + a
        out.append(float(np.sum(np.abs(C[act].astype(np.float64) - A[act]))))
    return out


@pytest.mark.parametrize("T,seed", [(1, 0), (50, 1), (3000, 2), (40000, 3)])
def test_diag_parity(tim, T, seed):
    A, B, C, offs, mask, tops = make_case(T, seed)
    if T == 1:
        offs, mask = np.array([0, 1]), np.ones(1, np.uint8)
    g = run(tim, A, B, C, offs, mask, tops)
    r, errs = oracle.oracle_diag_lenient(A, B, C, offs, mask, 2.0, 0.5, 1.5, tops)
    assert not errs
    assert_diag_parity(g, r, d_abs(A, C, offs, mask), what=f"T={T}")


# active tokens a quantile CTA holds in shared memory; longer sequences take the
# select over the shared-memory keys plus the rest kept in the workspace
SHARED_KEYS = 16384


def test_diag_without_top1_and_long_sequence(tim):
    """A sequence just past the shared-memory key capacity (16389 active tokens) next to a
    short one: exact quantiles with the keys past the shared-memory ones in the workspace, no flag."""
    n = SHARED_KEYS + 5
    A, B, C, _, _, _ = make_case(n + 100, 7)
    offs = np.array([0, 100, n + 100], dtype=np.int64)
    mask = np.ones(n + 100, np.uint8)
    g = run(tim, A, B, C, offs, mask, (None, None, None), cap=1.5, lo=0.9, hi=1.2)
    r, _ = oracle.oracle_diag_lenient(A, B, C, offs, mask, 1.5, 0.9, 1.2)
    assert g[1]["flags"] == 0 and g[1]["top1_flips"] == [-1, -1, -1]
    assert_diag_parity(g, r, d_abs(A, C, offs, mask), what="long")


def test_diag_exact_quantile_sequence(tim):
    k = np.arange(101)
    A = np.full(202, -2.0, np.float32)
    B = A.copy()
    mask = np.zeros(202, np.uint8)
    mask[::2] = 1
    B[::2] = (A[::2].astype(np.float64) - 0.01 * k).astype(np.float32)
    B[1::2] = np.float32(-50.0)
    g = run(tim, A, B, B, np.array([0, 202]), mask, (None, None, None))
    r, _ = oracle.oracle_diag_lenient(A, B, B, np.array([0, 202]), mask, 2.0, 0.5, 1.5)
    assert g[0]["abs_q50"][0] == r[0]["abs_q50"][0] and g[0]["abs_q99"][0] == r[0]["abs_q99"][0]
    assert abs(g[0]["abs_q95"][0] - 0.95) < 1e-6


@pytest.mark.parametrize("case", ["empty", "bad_mask", "nan_active", "bad_offsets"])
def test_diag_errors(tim, case):
    A, B, C, _, _, tops = make_case(64, 11)
    offs = np.array([0, 16, 32, 48, 64])
    mask = np.ones(64, np.uint8)
    want = {"empty": "TIM_ERR_EMPTY_SEQUENCE", "bad_mask": "TIM_ERR_BAD_MASK",
            "nan_active": "TIM_ERR_NONFINITE", "bad_offsets": "TIM_ERR_INVALID_ARG"}[case]
    if case == "empty":
        mask[16:32] = 0
    elif case == "bad_mask":
        mask[40] = 3
    elif case == "nan_active":
        C[50] = np.inf
    else:
        offs = np.array([0, 16, 12, 48, 64])
    with pytest.raises(tim.TimError) as ei:
        run(tim, A, B, C, offs, mask, tops)
    assert ei.value.name == want
    g = run(tim, A, B, C, offs, mask, tops, check=False)
    r, errs = oracle.oracle_diag_lenient(A, B, C, offs, mask, 2.0, 0.5, 1.5, tops)
    assert errs
    assert_diag_parity(g, r, d_abs(A, C, offs, mask), what=case)


def _same(x, y):
    if isinstance(x, dict):
        return x.keys() == y.keys() and all(_same(x[k], y[k]) for k in x)
    if isinstance(x, (list, tuple)):
        return len(x) == len(y) and all(_same(a, b) for a, b in zip(x, y))
    if isinstance(x, float) and math.isnan(x):
        return isinstance(y, float) and math.isnan(y)
    return x == y


def test_diag_sequence_results_do_not_depend_on_the_batch(tim):
    """Each sequence's diagnostics are the same bits alone or inside any batch."""
    A, B, C, offs, mask, tops = make_case(20000, 21, n_seq=5)
    full = run(tim, A, B, C, offs, mask, tops)
    for j in range(len(offs) - 1):
        a, b = int(offs[j]), int(offs[j + 1])
        one = run(tim, A[a:b], B[a:b], C[a:b], np.array([0, b - a], np.int64), mask[a:b],
                  [t[a:b] for t in tops])
        assert _same(one[0], full[j]), j


def _eighths(g, n, lo, hi):
    return (g.integers(lo, hi, n) / 8.0).astype(np.float32)


def test_diag_quantiles_exact_on_ties_tiny_and_maximal_sequences(tim):
    """The order statistics are selected, not approximated: every quantile equals the
    oracle's sorted-array formula bit for bit, across tie groups that straddle the
    interpolation ranks, all-equal sequences, 1-3 tokens, widely spread magnitudes,
    sequences at and past the shared-memory key capacity, and long sequences (65573 and
    about 68000 active tokens) with keys kept in the workspace."""
    g = np.random.default_rng(31)
    parts = []

    def add(A, B, C, mask=None):
        parts.append((A, B, C, np.ones(len(A), np.uint8) if mask is None else mask))

    for n in (1, 2, 3):
        A = _eighths(g, n, -80, -8)
        add(A, A + _eighths(g, n, 0, 9), A + _eighths(g, n, -9, 9))
    A = _eighths(g, 5000, -80, -8)
    add(A, A.copy(), A.copy())                                    # all |delta| = 0
    A = _eighths(g, 4099, -80, -8)
    B = (A + g.choice([0.0, 0.5, 1.0], 4099)).astype(np.float32)  # three values
    add(A, B, (B + g.choice([0.0, 0.25], 4099)).astype(np.float32))
    for zeros in (101, 150):                                      # rank 100 / 101 at a tie edge
        A = _eighths(g, 202, -80, -8)
        B = A.copy()
        B[zeros:] = A[zeros:] - (np.arange(202 - zeros) + 1) / 64.0
        add(A, B.astype(np.float32), B.astype(np.float32))
    for n in (SHARED_KEYS, SHARED_KEYS + 1, 65536 + 37):         # both selects, spread exponents
        A = (-np.abs(g.standard_normal(n)) * 4 - 1).astype(np.float32)
        B = (A + g.standard_normal(n) * 10.0 ** g.uniform(-6, 1, n)).astype(np.float32)
        add(A, B, (B + g.standard_normal(n) * 1e-3).astype(np.float32))
    A = _eighths(g, 70001, -80, -8)                               # long, three tie groups
    B = (A + g.choice([0.0, 0.5, 1.0], 70001, p=[0.5, 0.45, 0.05])).astype(np.float32)
    add(A, B, B.copy(), (g.random(70001) < 0.97).astype(np.uint8))
    A = _eighths(g, 3000, -80, -8)                                # inactive tokens interleaved
    B = (A - g.integers(0, 4, 3000) / 16.0).astype(np.float32)
    add(A, B, A.copy(), (g.random(3000) < 0.5).astype(np.uint8))

    A, B, C, mask = (np.concatenate([p[i] for p in parts]) for i in range(4))
    offs = np.cumsum([0] + [len(p[0]) for p in parts]).astype(np.int64)
    got = run(tim, A, B, C, offs, mask, (None, None, None))
    ref, errs = oracle.oracle_diag_lenient(A, B, C, offs, mask, 2.0, 0.5, 1.5)
    assert not errs
    for j, (x, y) in enumerate(zip(got, ref)):
        assert x["flags"] == y["flags"] and x["n_valid"] == y["n_valid"], j
        for k in ("abs_q50", "abs_q95", "abs_q99"):
            assert x[k] == y[k], (j, k, x[k], y[k])


def test_diag_and_compare_one_sequence_past_the_part_cap(tim):
    """A 300000-token sequence: its part count is capped at 256, so every part holds
    more than 512 tokens (each thread loops, all warps reduce); its quantiles (about
    270000 active tokens) come from the select over shared-memory and workspace keys, exact."""
    from parity import assert_compare_parity
    T = 300000
    A, B, C, _, _, tops = make_case(T, 41)
    offs = np.array([0, T], np.int64)
    mask = (np.random.default_rng(42).random(T) < 0.9).astype(np.uint8)
    g = run(tim, A, B, C, offs, mask, tops)
    r, errs = oracle.oracle_diag_lenient(A, B, C, offs, mask, 2.0, 0.5, 1.5, tops)
    assert not errs and g[0]["flags"] == 0
    assert_diag_parity(g, r, d_abs(A, C, offs, mask), what="past the cap")
    stats, w = tim.compare(cuda_tensor(A), cuda_tensor(B), cuda_tensor(C), cuda_tensor(offs),
                           cuda_tensor(mask), 2.0)
    ro, rw, errs = oracle.oracle_compare_lenient(A, B, C, offs, mask, 2.0)
    assert not errs
    assert_compare_parity(tim.stats_to_dicts(stats), ro, what="past the cap")
