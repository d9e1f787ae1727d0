"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch each.

A mutation that no pin catches would mean the oracle's correctness rests on
itself for that step.  Each case names the pins expected to fail.
"""
import math

import numpy as np
import pytest

import oracle
import oracle.compare as oc
import oracle.logprob as ol
import oracle_pins as P


def _lse_after_softmax(z, temperature):
    # log_softmax(z) / tau instead of log_softmax(z / tau)
    m = np.max(z, axis=1)
    lse = m + np.log(np.sum(np.exp(z - m[:, None]), axis=1))
    return z / temperature, lse / temperature


def _lse_no_shift(z, temperature):
    s = z / temperature
    with np.errstate(over="ignore"):
        return s, np.log(np.sum(np.exp(s), axis=1))


def _rms_eps_outside(h, gamma, eps):
    ms = np.mean(h * h, axis=1)
    rstd = 1.0 / np.sqrt(ms) + eps
    return ol.round_to_bf16(h * rstd[:, None] * gamma[None, :])


def _rms_no_round(h, gamma, eps):
    ms = np.mean(h * h, axis=1)
    return h * (1.0 / np.sqrt(ms + eps))[:, None] * gamma[None, :]


def _rms_sum_not_mean(h, gamma, eps):
    ms = np.sum(h * h, axis=1) / (h.shape[1] - 1)
    return ol.round_to_bf16(h * (1.0 / np.sqrt(ms + eps))[:, None] * gamma[None, :])


def _logits_reversed_features(y, W_bits, vocab_block=8192):
    return y @ ol.widen_bf16(W_bits[:, ::-1]).T


def _round_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.ldexp(np.ones_like(x), np.maximum(e, -125) - 8)
    return np.trunc(x / q) * q


_orig_oracle_logprob = ol.oracle_logprob


def _gather_next_id(hidden_bits, gamma_bits, W_bits, token_ids, temperature, eps, row_block=128):
    ids = (np.asarray(token_ids, dtype=np.int64) + 1) % W_bits.shape[0]
    return _orig_oracle_logprob(hidden_bits, gamma_bits, W_bits, ids, temperature, eps, row_block)


def _top1_last(hidden_bits, gamma_bits, W_bits, token_ids, temperature, eps, row_block=128):
    out = _orig_oracle_logprob(hidden_bits, gamma_bits, W_bits, token_ids, temperature, eps, row_block)
    rows = ol.oracle_log_softmax_rows(hidden_bits, gamma_bits, W_bits, temperature, eps)
    out["top1"] = rows.shape[1] - 1 - np.argmax(rows[:, ::-1], axis=1)
    return out


_orig_pair = oc._pair_stats


def _pair_reversed(x, y):
    return _orig_pair(y, x)


def _differ_by_value(x, y):
    return x != y


def _run_plus_one(b):
    if b.size == 0 or not b.any():
        return 0
    edges = np.diff(np.concatenate(([0], b.astype(np.int8), [0])))
    return int(np.max(np.flatnonzero(edges == -1) - np.flatnonzero(edges == 1))) + 1


def _active_all_rows(m, start):
    return np.arange(m.shape[0]) + start


def _k3_exp_plus(d):
    with np.errstate(over="ignore", invalid="ignore"):
        return np.exp(d) - 1 + d


def _k3_naive(d):
    with np.errstate(over="ignore", invalid="ignore"):
        return np.exp(d) - 1 - d


_orig_tis = oc._tis_weights


def _tis_reversed(d, cap):
    return _orig_tis(-d, cap)


def _tis_no_clip(d, cap):
    with np.errstate(over="ignore"):
        w = np.exp(d)
    return w, np.zeros(d.shape, dtype=bool)


import oracle.diag as od


def _quantile_nearest(x, q):
    xs = np.sort(np.asarray(x, dtype=np.float64))
    return float(xs[int(round((xs.shape[0] - 1) * q))])


def _quantile_n_not_n_minus_1(x, q):
    xs = np.sort(np.asarray(x, dtype=np.float64))
    h = xs.shape[0] * q
    lo = min(int(math.floor(h)), xs.shape[0] - 1)
    hi = min(lo + 1, xs.shape[0] - 1)
    return float(xs[lo] + (h - lo) * (xs[hi] - xs[lo]))


def _prob_mae_in_logs(left, right):
    return float(np.mean(np.abs(left - right)))


def _seq_tis_mean_not_sum(log_ratio_sum, cap):
    return min(math.exp(log_ratio_sum / 2.0), cap)


def _mis_keeps_everything(d, lo, hi):
    return float(np.sum(np.exp(d))), int(d.shape[0])


import oracle.processed as opr

_orig_process_row = opr.process_row


def _proc_cum_inclusive(z, x, temperature, top_k, top_p):
    V = z.shape[0]
    order = np.lexsort((np.arange(V), -z))
    top = order[:min(top_k, V)]
    s = z[top] / temperature
    q = np.exp(s - s[0]) / np.sum(np.exp(s - s[0]))
    keep = np.cumsum(q) < top_p
    keep[0] = True
    kept = top[keep]
    lse = s[0] + math.log(float(np.sum(np.exp(s[keep] - s[0]))))
    lp = float(z[x] / temperature - lse) if x in set(kept.tolist()) else -math.inf
    return lp, lse, int(kept.shape[0]), 0.0, 0.0


def _proc_no_renorm(z, x, temperature, top_k, top_p):
    lp, lse, kept, g, m = _orig_process_row(z, x, temperature, top_k, top_p)
    s = z / temperature
    full = float(np.max(s) + np.log(np.sum(np.exp(s - np.max(s)))))
    return (lp if lp == -math.inf else float(s[x] - full)), full, kept, g, m


def _proc_ties_high_id(z, x, temperature, top_k, top_p):
    V = z.shape[0]
    zz = z.copy()
    return _orig_process_row(zz[::-1].copy(), V - 1 - x, temperature, top_k, top_p)


_orig_process_head = opr.process_head


def _head_not_renormalised(z, temperature, top_k, top_p):
    ids, lp = _orig_process_head(z, temperature, top_k, top_p)
    s = z / temperature
    full = float(np.max(s) + np.log(np.sum(np.exp(s - np.max(s)))))
    return ids, np.where(np.isfinite(lp), s[ids] - full, lp)


def _head_id_order(z, temperature, top_k, top_p):
    ids, lp = _orig_process_head(z, temperature, top_k, top_p)
    o = np.argsort(ids, kind="stable")
    return ids[o], lp[o]


import oracle.fp8 as of8


def _e4m3_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.ldexp(np.ones_like(x), np.maximum(e - 1, -6) - 3)
    return np.clip(np.trunc(x / q) * q, -448.0, 448.0)


def _e4m3_two_mantissa_bits(x):
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.ldexp(np.ones_like(x), np.maximum(e - 1, -6) - 2)
    return np.clip(np.rint(x / q) * q, -448.0, 448.0)


def _scale_max_over_448(amax):
    return amax / 448.0 if amax else 1.0


def _fp8_y_unrounded(h, gamma, eps):
    return h * (1.0 / np.sqrt(np.mean(h * h, axis=1) + eps))[:, None] * gamma[None, :]


def _choices_none(x, margin):
    r = ol.round_to_bf16(x)
    return r, r


def _choices_one_sided(x, margin):
    x = np.asarray(x, dtype=np.float64)
    return ol.round_to_bf16(x), ol.round_to_bf16(x + np.abs(x) * margin)


_orig_row_alternatives = of8._row_alternatives


def _alternatives_codes_only(x_row, margin):
    # keep only elements whose codes differ under the base scale (ignores the row scale)
    base = ol.round_to_bf16(x_row)
    lo, hi = of8.bf16_choices(x_row, margin)
    amb = np.flatnonzero(lo != hi)
    other = np.where(lo[amb] == base[amb], hi[amb], lo[amb])
    s = of8.fp8_scale(float(np.max(np.abs(base))))
    keep = of8.e4m3_round(base[amb] / s) != of8.e4m3_round(other / s)
    return base, amb[keep], other[keep]


def _alternatives_wrong_other(x_row, margin):
    base, idx, other = _orig_row_alternatives(x_row, margin)
    return base, idx, 2 * base[idx] - other                 # mirrored: not a rounding of x


import oracle.fp32head as of32


def _rms_unrounded_but_rounded(h, gamma, eps):
    return ol.round_to_bf16(h * (1.0 / np.sqrt(np.mean(h * h, axis=1) + eps))[:, None] *
                            gamma[None, :])


def _rms_unrounded_eps_outside(h, gamma, eps):
    return h * (1.0 / (np.sqrt(np.mean(h * h, axis=1)) + eps))[:, None] * gamma[None, :]


import oracle.backward as obw

_orig_logit_grad = obw.logit_grad


def _grad_no_temperature(z, token_ids, grad, temperature):
    return _orig_logit_grad(z, token_ids, grad, temperature) * temperature


def _grad_softmax_of_raw_logits(z, token_ids, grad, temperature):
    return _orig_logit_grad(z * temperature, token_ids, grad, temperature)


def _grad_sign_flipped(z, token_ids, grad, temperature):
    return -_orig_logit_grad(z, token_ids, grad, temperature)


def _grad_next_token(z, token_ids, grad, temperature):
    return _orig_logit_grad(z, (np.asarray(token_ids) + 1) % z.shape[1], grad, temperature)


_orig_rms_bwd = obw.rmsnorm_backward


def _rms_bwd_no_projection(h, gamma, eps, dy):
    h = np.asarray(h, dtype=np.float64)
    rstd = 1.0 / np.sqrt(np.mean(h * h, axis=1) + eps)
    dh = rstd[:, None] * np.asarray(gamma)[None, :] * dy          # drops the rstd' term
    return dh, np.sum(dy * h * rstd[:, None], axis=0)


def _rms_bwd_dgamma_without_rstd(h, gamma, eps, dy):
    dh, _ = _orig_rms_bwd(h, gamma, eps, dy)
    return dh, np.sum(np.asarray(dy) * np.asarray(h), axis=0)


MUTATIONS = [
    ("temperature after softmax", ol, "lse_stats", _lse_after_softmax, ["pin_v8_temperature"]),
    ("no max shift", ol, "lse_stats", _lse_no_shift, ["pin_large_logits"]),
    ("eps outside sqrt", ol, "rmsnorm", _rms_eps_outside, ["pin_rmsnorm_closed_form"]),
    ("y not rounded to bf16", ol, "rmsnorm", _rms_no_round, ["pin_brute_force_mpmath"]),
    ("sum/(d-1) instead of mean", ol, "rmsnorm", _rms_sum_not_mean, ["pin_rmsnorm_closed_form"]),
    ("W features reversed", ol, "logits", _logits_reversed_features, ["pin_brute_force_mpmath"]),
    ("bf16 truncation not nearest-even", ol, "round_to_bf16", _round_truncate,
     ["pin_round_to_bf16_brute"]),
    ("gather the next id", ol, "oracle_logprob", _gather_next_id, ["pin_v8_page_probabilities"]),
    ("top-1 picks last on ties", ol, "oracle_logprob", _top1_last, ["pin_v8_uniform"]),
    ("pair subtraction reversed", oc, "_pair_stats", _pair_reversed, ["pin_recorded_token_summary",
                                                                      "pin_case3_outlier"]),
    ("value compare instead of bitwise", oc, "_differ", _differ_by_value, ["pin_signed_zero_and_nan"]),
    ("longest run off by one", oc, "_longest_true_run", _run_plus_one, ["pin_active_ordinals"]),
    ("mask ignored (positions, not active ordinals)", oc, "_active_rows", _active_all_rows,
     ["pin_active_ordinals"]),
    ("k3 sign of d flipped", oc, "_k3_terms", _k3_exp_plus, ["pin_k3_closed_form"]),
    ("k3 by exp(d)-1-d (cancellation)", oc, "_k3_terms", _k3_naive, ["pin_k3_closed_form"]),
    ("TIS ratio inverted (A - C)", oc, "_tis_weights", _tis_reversed, ["pin_fig1_split"]),
    ("TIS without the cap", oc, "_tis_weights", _tis_no_clip, ["pin_tis_clip"]),
    ("quantile by nearest rank", od, "quantile_linear", _quantile_nearest,
     ["pin_quantile_definition", "pin_diag_quantiles_in_sequence"]),
    ("quantile index n q", od, "quantile_linear", _quantile_n_not_n_minus_1,
     ["pin_quantile_definition"]),
    ("probability MAE on logprobs", od, "_prob_mae", _prob_mae_in_logs,
     ["pin_diag_page_probability_mae"]),
    ("sequence TIS from a mean", od, "_seq_tis", _seq_tis_mean_not_sum, ["pin_diag_fig1_sequence"]),
    ("MIS keeps every token", od, "_mis", _mis_keeps_everything, ["pin_diag_mis_and_flips"]),
    ("top-p cut on inclusive cumulative mass", opr, "process_row", _proc_cum_inclusive,
     ["pin_processed_top_p_boundary"]),
    ("processed score not renormalised", opr, "process_row", _proc_no_renorm,
     ["pin_processed_page_topk"]),
    ("top-k ties keep the higher ids", opr, "process_row", _proc_ties_high_id,
     ["pin_processed_ties_and_temperature"]),
    ("top-k head not renormalised", opr, "process_head", _head_not_renormalised,
     ["pin_processed_head"]),
    ("top-k head in id order", opr, "process_head", _head_id_order, ["pin_processed_head"]),
    ("e4m3 truncation", of8, "e4m3_round", _e4m3_truncate, ["pin_e4m3_rounding_exhaustive"]),
    ("e4m3 with two mantissa bits", of8, "e4m3_round", _e4m3_two_mantissa_bits,
     ["pin_e4m3_rounding_exhaustive"]),
    ("non-power-of-two scale", of8, "fp8_scale", _scale_max_over_448, ["pin_fp8_scale_rule"]),
    ("FP8 y not rounded to bf16", of8, "rmsnorm", _fp8_y_unrounded,
     ["pin_fp8_y_is_the_bf16_heads_y"]),
    ("admissible set without the other rounding", of8, "bf16_choices", _choices_none,
     ["pin_bf16_choices_brute", "pin_fp8_admissible_covers_fp32_evaluations"]),
    ("admissible set rounds one end only", of8, "bf16_choices", _choices_one_sided,
     ["pin_bf16_choices_brute"]),
    ("admissible alternative is not a rounding", of8, "_row_alternatives",
     _alternatives_wrong_other, ["pin_fp8_admissible_covers_fp32_evaluations"]),
    ("admissible set ignores a flip of the row scale", of8, "_row_alternatives",
     _alternatives_codes_only, ["pin_fp8_admissible_scale_flip"]),
    ("FP32 head rounds y to bf16", of32, "rmsnorm_unrounded", _rms_unrounded_but_rounded,
     ["pin_fp32_head_mpmath", "pin_fp32_head_torch"]),
    ("FP32 head eps outside the sqrt", of32, "rmsnorm_unrounded", _rms_unrounded_eps_outside,
     ["pin_fp32_head_mpmath", "pin_fp32_head_torch"]),
    ("backward without 1/tau", obw, "logit_grad", _grad_no_temperature,
     ["pin_backward_finite_differences", "pin_backward_torch_autograd"]),
    ("backward softmax of raw logits", obw, "logit_grad", _grad_softmax_of_raw_logits,
     ["pin_backward_torch_autograd", "pin_backward_temperature_closed_form"]),
    ("backward sign flipped", obw, "logit_grad", _grad_sign_flipped,
     ["pin_backward_finite_differences"]),
    ("backward one-hot on the next id", obw, "logit_grad", _grad_next_token,
     ["pin_backward_torch_autograd"]),
    ("RMSNorm backward without the rstd derivative", obw, "rmsnorm_backward",
     _rms_bwd_no_projection, ["pin_rmsnorm_backward_finite_differences"]),
    ("RMSNorm backward dgamma without rstd", obw, "rmsnorm_backward",
     _rms_bwd_dgamma_without_rstd, ["pin_rmsnorm_backward_finite_differences"]),
]


@pytest.mark.parametrize("name,mod,attr,fn,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(monkeypatch, name, mod, attr, fn, pins):
    monkeypatch.setattr(mod, attr, fn)
    if hasattr(oracle, attr):   # names re-exported by the package
        monkeypatch.setattr(oracle, attr, fn)
    caught = []
    for pin_name in pins:
        try:
            getattr(P, pin_name)()
        except (AssertionError, oracle.OracleError, FloatingPointError):
            caught.append(pin_name)
    assert caught, f"mutation '{name}' passed every pin in {pins}"
