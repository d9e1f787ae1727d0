"""The FP32 head (tim_split_tf32, tim_logprob_fp32) through the C ABI against the
fp64 FP32-head oracle.

Tolerance.  The GEMM forms each product from tf32 parts: big (11 significant
bits) and small = x - big (|small| < 2^-10 |x|, truncated to tf32 by the MMA:
error < 2^-20 |x|); the dropped small*small term is < 2^-20 |a b|; so a product
is off by < 3 * 2^-20 of its size: ~1e-5 on a logit for these shapes
(random-sign errors over d terms of |y W| ~ 0.03).  The tensor-core accumulation
adds a bias: each MMA step can lose up to one ulp of the running fp32 sum, so
the error grows linearly with the number of steps (d/8 for the main sum; the
correction products go to their own accumulator).  Measured on GB300 over 128
rows, V = 8192: mean lse error -3.7e-5, max 4.5e-5 at d = 4096 (-7e-5 / 9.7e-5
at d = 8192), the bf16 head showing the same trend at half the size (d/16
steps).  The bias grows with d (steps) and a logprob divides logit errors by
tau, so logprob and lse are checked to 6e-5 * (d / 1024) / tau: 2.4e-4 at
d = 4096, tau = 1 (3x the measured maximum there; ten times tighter than the bf16
head), 4.3e-4 at d = 5120, tau = 0.7 (measured 2.5e-4); top-1 where the oracle's
logit gap exceeds 1e-4."""
import numpy as np
import pytest

import oracle
import synth
from parity import bf16_cuda, cuda_tensor, sample_rows

pytestmark = pytest.mark.gpu

FP32_TOP1_GAP = 1e-4


def fp32_tol(d, tau):
    return 6e-5 * (d / 1024.0) / tau


@pytest.fixture(scope="module")
def tim():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import rollout_logprob_consistency_gb300 as tim
    return tim


def f32_cuda(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def assert_fp32_parity(got, orc, d, tau, rows=None, what=""):
    tol = fp32_tol(d, tau)
    lp, lse, top1 = got
    if rows is not None:
        lp, lse, top1 = lp[rows], lse[rows], top1[rows]
    ok = ~orc["bad_token"]
    dlp = np.abs(lp[ok].astype(np.float64) - orc["logprob"][ok])
    dlse = np.abs(lse.astype(np.float64) - orc["lse"])
    assert dlp.max(initial=0) <= tol, f"{what}: logprob max err {dlp.max():.3e}"
    assert dlse.max(initial=0) <= tol, f"{what}: lse max err {dlse.max():.3e}"
    sel = orc["gap"] > FP32_TOP1_GAP
    bad = np.flatnonzero(sel & (top1.astype(np.int64) != orc["top1"]))
    assert bad.size == 0, f"{what}: top1 differs on {bad.size} rows"
    return float(max(dlp.max(initial=0), dlse.max(initial=0)))


def test_split_tf32_definition(tim):
    g = np.random.default_rng(8)
    x = np.concatenate([g.standard_normal(4000).astype(np.float32) * 10.0 ** g.integers(-6, 6, 4000),
                        np.array([0.0, -0.0, 1.0, -3.5, 1e-40, 3.0e38], np.float32),
                        np.zeros(2, np.float32)]).astype(np.float32)
    big, small = (t.cpu().numpy() for t in tim.split_tf32(f32_cuda(x)))
    want_big = (x.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    assert np.array_equal(big.view(np.uint32), want_big.view(np.uint32))
    assert np.array_equal(small.view(np.uint32), (x - want_big).view(np.uint32))
    assert np.array_equal((big.astype(np.float64) + small), x.astype(np.float64))   # exact split


@pytest.mark.parametrize("T,d,V,tau", [(1, 64, 300, 1.0), (5, 64, 1, 1.0), (64, 128, 1000, 1.0),
                                       (129, 256, 2049, 0.7), (300, 320, 5000, 1.3),
                                       (77, 5120, 3001, 0.7)])
def test_fp32_parity(tim, T, d, V, tau):
    b = synth.make_custom(T=T, d=d, V=V, temperature=tau, tag=f"f32{T}_{d}_{V}")
    W32 = synth.fp32_weights(b.head)
    Wb, Ws = tim.split_tf32(f32_cuda(W32))
    got = [x.cpu().numpy() for x in tim.logprob_fp32(bf16_cuda(b.hidden_gen),
                                                     bf16_cuda(b.head.gamma), Wb, Ws,
                                                     cuda_tensor(b.token_ids), tau, b.eps)]
    orc = oracle.oracle_logprob_fp32(b.hidden_gen, b.head.gamma, W32, b.token_ids, tau, b.eps)
    assert_fp32_parity(got, orc, d, tau, what=f"fp32 T={T} d={d} V={V}")


def test_fp32_full_head_batch_invariance_and_precision_gain(tim):
    b = synth.make_custom(T=200, d=4096, V=151936, temperature=0.7, tag="f32full")
    W32 = synth.fp32_weights(b.head)
    Wb, Ws = tim.split_tf32(f32_cuda(W32))
    hid, gam, ids = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), cuda_tensor(b.token_ids)
    full = [x.cpu().numpy() for x in tim.logprob_fp32(hid, gam, Wb, Ws, ids, 0.7, b.eps)]
    rows = sample_rows(200, 40)
    orc = oracle.oracle_logprob_fp32(b.hidden_gen[rows], b.head.gamma, W32, b.token_ids[rows],
                                     0.7, b.eps)
    err32 = assert_fp32_parity(full, orc, 4096, 0.7, rows=rows, what="fp32 full head")
    part = [x.cpu().numpy() for x in tim.logprob_fp32(hid[13:77].contiguous(), gam, Wb, Ws,
                                                      cuda_tensor(b.token_ids[13:77]), 0.7, b.eps)]
    for x, y in zip(part, full):
        assert x.tobytes() == y[13:77].tobytes()
    # the bf16 head on the same inputs (W rounded to bf16, y rounded to bf16) is much further
    # from the fp32 definition
    bf = [x.cpu().numpy() for x in tim.logprob(hid, gam, bf16_cuda(b.head.W), ids, 0.7, b.eps)]
    errbf = float(np.max(np.abs(bf[1][rows].astype(np.float64) - orc["lse"])))
    assert err32 < 0.1 * errbf, (err32, errbf)
