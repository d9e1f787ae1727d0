"""tim_processed_logprob (top-k then top-p) through the C ABI against the fp64 oracle.

Kept-set membership is a discrete decision: rows whose top-k boundary gap is
below 1e-3 (logit units) or whose top-p cumulative mass lies within 1e-4 of p
next to the cut are exempt from the membership check (the same rule as top-1
ties); everywhere else the kept count must match exactly and the scores must
agree within 2e-3 nats (or both be -inf)."""
import math

import numpy as np
import pytest

import oracle
import synth
from parity import LP_TOL, bf16_cuda, cuda_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tim():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import rollout_logprob_consistency_gb300 as tim
    return tim


def check(got, orc, what):
    lp, lse, kept = got
    ok = (orc["gap_k"] > 1e-3) & (orc["margin_p"] > 1e-4)
    assert ok.mean() > 0.8, f"{what}: too many exempt rows"
    idx = np.flatnonzero(ok)
    assert np.array_equal(kept[idx], orc["kept"][idx]), f"{what}: kept sets differ"
    for i in idx:
        a, b = float(lp[i]), float(orc["logprob"][i])
        if b == -math.inf:
            assert a == -math.inf, (what, i, a, b)
        else:
            assert abs(a - b) <= LP_TOL, (what, i, a, b)
        assert abs(float(lse[i]) - orc["lse_kept"][i]) <= LP_TOL, (what, i)


def check_head(got_ids, got_lp, orc, what):
    """Rows whose top-k boundary and top-p cut are decided (as in ``check``): the head holds
    the same ids; where the ranks inside the head are decided too (neighbour gaps > 1e-3)
    the order matches; the logprob of every id matches within 2e-3 (or both -inf)."""
    ok = (orc["gap_k"] > 1e-3) & (orc["margin_p"] > 1e-4)
    for i in np.flatnonzero(ok):
        gi, oi = got_ids[i].astype(np.int64), orc["topk_ids"][i]
        assert set(gi.tolist()) == set(oi.tolist()), (what, i)
        if orc["rank_gap"][i] > 1e-3:
            assert np.array_equal(gi, oi), (what, i)
        want = dict(zip(oi.tolist(), orc["topk_logprob"][i].tolist()))
        for v, a in zip(gi.tolist(), got_lp[i].tolist()):
            b = want[v]
            if b == -math.inf:
                assert a == -math.inf, (what, i, v, a)
            else:
                assert abs(a - b) <= LP_TOL, (what, i, v, a, b)


def targets(b, tau):
    """Half the rows target the oracle's top-1 token (kept), half a Zipf draw."""
    raw = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, tau, b.eps)
    ids = b.token_ids.copy()
    ids[::2] = raw["top1"][::2]
    return ids


@pytest.mark.parametrize("T,d,V,tau,k,p", [
    (50, 128, 1000, 1.0, 1, 1.0), (50, 128, 1000, 1.0, 2, 1.0), (50, 128, 1000, 0.7, 17, 0.9),
    (33, 192, 2048, 1.3, 64, 0.5), (40, 256, 20000, 0.8, 40, 0.95), (9, 64, 5000, 1.0, 5, 1.0),
    (256, 128, 3000, 0.9, 10, 0.9),   # two row tiles per W tile, the leader prefetching W
    (384, 128, 3000, 0.9, 10, 0.9),   # three row tiles
    (512, 128, 3000, 0.9, 10, 0.9),   # four row tiles
])
def test_processed_parity(tim, T, d, V, tau, k, p):
    b = synth.make_custom(T=T, d=d, V=V, temperature=tau, tag=f"pr{T}_{d}_{V}")
    ids = targets(b, tau)
    got = [x.cpu().numpy() for x in tim.processed_logprob(
        bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W), cuda_tensor(ids),
        tau, b.eps, k, p)]
    orc = oracle.oracle_processed_logprob(b.hidden_gen, b.head.gamma, b.head.W, ids,
                                          float(np.float32(tau)), b.eps, k, float(np.float32(p)))
    check(got, orc, f"T={T} V={V} k={k} p={p}")
    r = tim.processed_logprob(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma),
                              bf16_cuda(b.head.W), cuda_tensor(ids), tau, b.eps, k, p, head=True)
    assert r[3].shape == (T, min(k, V))
    check_head(r[3].cpu().numpy(), r[4].cpu().numpy(), orc, f"T={T} V={V} k={k} p={p} head")


def test_processed_full_head_and_batch_invariance(tim):
    import torch
    b = synth.make_custom(T=96, d=4096, V=151936, temperature=0.7, tag="pr_full")
    ids = targets(b, 0.7)
    hid, gam, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    for k, p in ((1, 1.0), (20, 0.95), (64, 1.0)):
        full = [x.cpu().numpy() for x in tim.processed_logprob(hid, gam, W, cuda_tensor(ids), 0.7,
                                                               b.eps, k, p)]
        orc = oracle.oracle_processed_logprob(b.hidden_gen, b.head.gamma, b.head.W, ids,
                                              float(np.float32(0.7)), b.eps, k,
                                              float(np.float32(p)))
        check(full, orc, f"full head k={k} p={p}")
        r = tim.processed_logprob(hid, gam, W, cuda_tensor(ids), 0.7, b.eps, k, p, head=True)
        assert all(np.array_equal(r[j].cpu().numpy(), full[j]) for j in range(3))
        check_head(r[3].cpu().numpy(), r[4].cpu().numpy(), orc, f"full head k={k} p={p} head")
        # rows scored in another batch split give the same bits
        part = [x.cpu().numpy() for x in tim.processed_logprob(
            hid[7:40].contiguous(), gam, W, cuda_tensor(ids[7:40]), 0.7, b.eps, k, p)]
        for x, y in zip(part, full):
            assert x.tobytes() == y[7:40].tobytes()
        # and inside a 256-row batch (two row tiles against each W tile)
        fill = synth.make_custom(T=160, d=4096, V=151936, tag="pr_fill")
        big_h = torch.cat([hid, bf16_cuda(fill.hidden_gen)])
        big_ids = cuda_tensor(np.concatenate([ids, fill.token_ids]).astype(np.int32))
        big = [x.cpu().numpy() for x in tim.processed_logprob(big_h, gam, W, big_ids, 0.7, b.eps,
                                                              k, p)]
        for x, y in zip(big, full):
            assert x[:96].tobytes() == y.tobytes()


def test_processed_k1_is_top1(tim):
    """k = 1 keeps only the arg-max: its processed logprob is 0, others -inf."""
    b = synth.make_custom(T=30, d=128, V=3000, tag="pr_k1")
    hid, gam, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    _, _, top1 = tim.logprob(hid, gam, W, cuda_tensor(b.token_ids), 1.0, b.eps)
    ids = top1.cpu().numpy().astype(np.int32)
    ids[1::3] = (ids[1::3] + 1) % 3000
    lp, _, kept = [x.cpu().numpy() for x in tim.processed_logprob(hid, gam, W, cuda_tensor(ids),
                                                                  1.0, b.eps, 1, 1.0)]
    assert np.all(kept == 1)
    assert np.all(lp[0::3] == 0.0) and np.all(lp[1::3] == -np.inf)


def test_processed_fallback_rows(tim):
    """Rows whose top logits crowd one 256-column tile (five copies of the row's arg-max
    W row placed in one tile) cannot be vouched for by the per-tile top-4 lists and are
    rescored over the gathered fallback rows; the result must still match the oracle and
    be identical when the row is scored alone."""
    b = synth.make_custom(T=64, d=256, V=20000, temperature=0.9, tag="pr_fb")
    raw = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 0.9, b.eps)
    W = b.head.W.copy()
    t_fb = [0, 5, 33]
    for r in t_fb:                                  # five ties at the top inside tile 40 + r
        base = (40 + r) * 256
        for c in range(5):
            W[base + 17 * c] = b.head.W[raw["top1"][r]]
    ids = targets(b, 0.9)
    ids[t_fb] = [(40 + r) * 256 + 34 for r in t_fb]  # the third copy of the tie
    hid, gam, Wd = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(W)
    for k, p in ((8, 1.0), (20, 0.9)):
        got = [x.cpu().numpy() for x in tim.processed_logprob(hid, gam, Wd, cuda_tensor(ids), 0.9,
                                                              b.eps, k, p)]
        orc = oracle.oracle_processed_logprob(b.hidden_gen, b.head.gamma, W, ids,
                                              float(np.float32(0.9)), b.eps, k,
                                              float(np.float32(p)))
        check(got, orc, f"fallback k={k} p={p}")
        for r in t_fb:
            assert got[2][r] >= min(5, k) or p < 1.0
            one = [x.cpu().numpy() for x in tim.processed_logprob(
                hid[r:r + 1].contiguous(), gam, Wd, cuda_tensor(ids[r:r + 1]), 0.9, b.eps, k, p)]
            assert all(one[j].tobytes() == got[j][r:r + 1].tobytes() for j in range(3))


def test_processed_capacity_error(tim):
    """Every logit tied: more candidates than the per-row capacity -> TIM_ERR_CAPACITY."""
    b = synth.make_custom(T=8, d=64, V=4096, tag="pr_cap")
    W = np.repeat(b.head.W[:1], 4096, axis=0)
    with pytest.raises(tim.TimError) as ei:
        tim.processed_logprob(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(W),
                              cuda_tensor(b.token_ids), 1.0, b.eps, 8, 1.0)
    assert ei.value.name == "TIM_ERR_CAPACITY"


def test_processed_argument_limits(tim):
    b = synth.make_custom(T=4, d=64, V=5000, tag="pr_arg")
    args = (bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W),
            cuda_tensor(b.token_ids), 1.0, b.eps)
    for k, p in ((0, 1.0), (65, 1.0), (4, 0.0), (4, 1.5)):
        with pytest.raises(tim.TimError):
            tim.processed_logprob(*args, k, p)
    with pytest.raises(tim.TimError) as ei:       # 20 tiles < k = 32 and V > capacity
        tim.processed_logprob(*args, 32, 1.0)
    assert ei.value.name == "TIM_ERR_SHAPE"
