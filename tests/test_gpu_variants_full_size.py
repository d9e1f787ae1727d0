"""The next-row paths at the benchmark's full size and launch configuration
(Qwen3-8B-shaped head, T = 32768, d = 4096, V = 151936, trainer hidden states, as
bench.py times them), checked against the fp64 oracle row by row -- one seeded row
inside every 128-row tile and both ends of every raster group (``parity.tile_rows``)
for every path --
with each path's own tolerance (see the per-path test files), and by properties
that hold at any size."""
import math

import numpy as np
import pytest

import oracle
import synth
from parity import (assert_fp8_admissible_parity, bf16_cuda, cuda_tensor, fp8_y_margin,
                    raster_group_tiles, tile_rows)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def tim():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import rollout_logprob_consistency_gb300 as tim
    return tim


@pytest.fixture(scope="module")
def work(tim):
    b = synth.make_qwen3_8b()
    dev = dict(hid=bf16_cuda(b.hidden_train), gam=bf16_cuda(b.head.gamma),
               W=bf16_cuda(b.head.W), ids=cuda_tensor(b.token_ids))
    return b, dev


def test_processed_full_size(tim, work):
    from test_gpu_processed import check
    b, dv = work
    got = [x.cpu().numpy() for x in tim.processed_logprob(dv["hid"], dv["gam"], dv["W"],
                                                          dv["ids"], 0.7, b.eps, 50, 0.95)]
    rows = tile_rows(b.T, raster_group_tiles(b.head.d))
    orc = oracle.oracle_processed_logprob(b.hidden_train[rows], b.head.gamma, b.head.W,
                                          b.token_ids[rows], float(np.float32(0.7)), b.eps, 50,
                                          float(np.float32(0.95)))
    check([g[rows] for g in got], orc, "processed T=32768")
    assert np.all(got[2] >= 1) and np.all(got[2] <= 50)


def test_fp8_head_full_size(tim, work):
    b, dv = work
    W8, sW = tim.quantize_fp8_rows(dv["W"])
    got = [x.cpu().numpy() for x in tim.logprob_fp8(dv["hid"], dv["gam"], W8, sW, dv["ids"], 0.7,
                                                    b.eps)]
    rows = tile_rows(b.T, raster_group_tiles(b.head.d))
    adm = oracle.oracle_logprob_fp8_admissible(b.hidden_train[rows], b.head.gamma, b.head.W,
                                               b.token_ids[rows], 0.7, b.eps, fp8_y_margin(4096))
    res = assert_fp8_admissible_parity(got, adm, b.token_ids, b.V, rows=rows, what="fp8 T=32768")
    print(f"fp8 T=32768: {res}")


def test_fp32_head_full_size(tim, work):
    import torch
    from test_gpu_fp32 import assert_fp32_parity
    b, dv = work
    Wb, Ws = tim.split_tf32(dv["W"].float().contiguous())
    got = [x.cpu().numpy() for x in tim.logprob_fp32(dv["hid"], dv["gam"], Wb, Ws, dv["ids"], 0.7,
                                                     b.eps)]
    del Wb, Ws
    torch.cuda.empty_cache()
    rows = tile_rows(b.T, raster_group_tiles(b.head.d))
    W32 = oracle.widen_bf16(b.head.W).astype(np.float32)
    orc = oracle.oracle_logprob_fp32(b.hidden_train[rows], b.head.gamma, W32, b.token_ids[rows],
                                     0.7, b.eps)
    assert_fp32_parity(got, orc, 4096, 0.7, rows=rows, what="fp32 T=32768")


def test_backward_full_size(tim, work):
    """dy on sampled rows against the oracle (rows are independent); dW by an exact
    property of the gradient: every row of G sums to zero, so every column of dW sums to
    zero up to the bf16 rounding of G (relative error at most 2^-8 per element), which
    moves a row's sum by at most 2^-8 sum_v |G_tv| <= 2^-7 |g_t| / tau; the bound per
    column is therefore 2^-7 sum_t (|g_t| / tau) |y_ti| (the fp32 accumulation adds far
    less)."""
    import torch
    from test_gpu_backward import DELTA
    b, dv = work
    g = np.where(b.mask > 0, 1.0, 0.0).astype(np.float32)       # loss over response tokens
    _, lse, _ = tim.logprob(dv["hid"], dv["gam"], dv["W"], dv["ids"], 0.7, b.eps)
    dy, dW = tim.logprob_backward(dv["hid"], dv["gam"], dv["W"], dv["ids"], lse,
                                  torch.from_numpy(g).cuda(), 0.7, b.eps)
    rows = tile_rows(b.T, raster_group_tiles(b.head.d), must=[b.meta["prefix"] + 3])
    orc = oracle.oracle_logprob_backward(b.hidden_train[rows], b.head.gamma, b.head.W,
                                         b.token_ids[rows], 0.7, b.eps, g[rows], dW_rows=[0])
    dyr = dy.cpu().numpy()[rows].astype(np.float64)
    Wf = oracle.widen_bf16(b.head.W)
    ids = b.token_ids[rows].astype(np.int64)
    tgt = (np.abs(g[rows].astype(np.float64)) / 0.7)[:, None] * np.abs(Wf[ids])
    tol = 2.0 ** -8 * orc["bound_dy"] + DELTA * tgt + 1e-6 * orc["bound_dy"].max()
    assert np.all(np.abs(dyr - orc["dy"]) <= tol), float(np.abs(dyr - orc["dy"]).max())
    colsum = dW.sum(dim=0, dtype=torch.float64).cpu().numpy()
    gam = oracle.widen_bf16(b.head.gamma)
    bound = np.zeros(b.head.d)
    for r0 in range(0, b.T, 4096):
        y = oracle.rmsnorm(oracle.widen_bf16(b.hidden_train[r0:r0 + 4096]), gam, b.eps)
        bound += (np.abs(g[r0:r0 + 4096].astype(np.float64)) / 0.7) @ np.abs(y)
    assert np.all(np.abs(colsum) <= 2.0 ** -7 * bound), float(
        np.max(np.abs(colsum) / bound))
    assert math.isfinite(float(dW.abs().max()))
