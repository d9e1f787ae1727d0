"""Backward of the linear logprob (tim_logprob_backward) through the C ABI against
the fp64 oracle.

Tolerance, per output element.  The GPU rounds G = dL/dz to bf16 (relative
error <= 2^-9) before the two tensor-core products, so each element of dy = G.W
and dW = G^T.y may move by 2^-9 sum |G||W| (resp. |G||y|), the "bound" the
oracle returns; 2^-8 of it is allowed.  G also inherits the forward's errors
through p = exp(z / tau - lse): relative 1e-4 at most for the shapes here (the
forward's logit and lse errors), inside the bound for every entry except the
target's, where G = (g / tau)(1 - p_x) can be small while its absolute error
is (g / tau) p_x 1e-4; that term is allowed as DELTA * (|g_t| / tau) * |W| (dy)
and DELTA * sum over rows with x_t = v of (|g_t| / tau) |y_t| (dW), DELTA = 1e-3.
fp32 accumulation adds 1e-6 of the largest bound.  dW = G^T.y is also linear in
y, and the GPU's bf16 y and the oracle's differ by one bf16 step (at most 2^-7
relative) on a few elements per hundred thousand (the fp32 and fp64 RMSNorms
round them to different neighbours); a column of dW holding such an element
moves by up to 2^-7 of its bound, so dW is allowed 3 * 2^-8 of the bound."""
import numpy as np
import pytest

import oracle
import synth
from parity import bf16_cuda, cuda_tensor, sample_rows

pytestmark = pytest.mark.gpu

DELTA = 1e-3


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


def upstream(T, seed):
    g = np.random.default_rng(seed).standard_normal(T).astype(np.float32)
    g[3::7] = 0.0                     # masked tokens
    return g


def run(tim, b, g, **kw):
    hid, gam, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    ids = cuda_tensor(b.token_ids)
    _, lse, _ = tim.logprob(hid, gam, W, ids, b.temperature, b.eps)
    dy, dW = tim.logprob_backward(hid, gam, W, ids, lse, f32_cuda(g), b.temperature, b.eps, **kw)
    return dy.cpu().numpy().astype(np.float64), dW.cpu().numpy().astype(np.float64)


def check(b, g, dy, dW, orc, dW_rows=None, what=""):
    tau = b.temperature
    Wf = oracle.widen_bf16(b.head.W)
    ag = np.abs(g.astype(np.float64)) / tau
    ids = b.token_ids.astype(np.int64)
    tgt_dy = ag[:, None] * np.abs(Wf[ids])
    tol_dy = 2.0 ** -8 * orc["bound_dy"] + DELTA * tgt_dy + 1e-6 * orc["bound_dy"].max()
    err = np.abs(dy - orc["dy"])
    bad = np.argwhere(err > tol_dy)
    assert bad.size == 0, f"{what}: dy off at {bad[:3].tolist()}, err {err.max():.3e}"
    rows = np.arange(b.head.V) if dW_rows is None else np.asarray(dW_rows)
    tgt_dW = np.zeros((rows.size, b.head.d))
    pos = {int(v): k for k, v in enumerate(rows)}
    for t, x in enumerate(ids):
        if int(x) in pos:
            tgt_dW[pos[int(x)]] += ag[t] * np.abs(orc["y"][t])
    tol_dW = 3 * 2.0 ** -8 * orc["bound_dW"] + DELTA * tgt_dW + 1e-6 * orc["bound_dW"].max()
    errw = np.abs(dW[rows] - orc["dW"])
    badw = np.argwhere(errw > tol_dW)
    assert badw.size == 0, f"{what}: dW off at {badw[:3].tolist()}, err {errw.max():.3e}"
    if np.linalg.norm(orc["dy"]) > 0:      # (a one-word vocabulary has no gradient at all)
        rel = np.linalg.norm(dy - orc["dy"]) / np.linalg.norm(orc["dy"])
        assert rel < 5e-3, f"{what}: dy relative error {rel:.2e}"


@pytest.mark.parametrize("T,d,V,tau", [(1, 64, 300, 1.0), (5, 64, 1, 1.0), (64, 128, 1000, 1.0),
                                       (129, 256, 2049, 0.7), (300, 320, 5000, 1.3),
                                       (77, 5120, 3001, 0.7)])
def test_backward_parity(tim, T, d, V, tau):
    b = synth.make_custom(T=T, d=d, V=V, temperature=tau, tag=f"bw{T}_{d}_{V}")
    g = upstream(T, T + d)
    dy, dW = run(tim, b, g)
    orc = oracle.oracle_logprob_backward(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, tau,
                                         b.eps, g)
    check(b, g, dy, dW, orc, what=f"T={T} d={d} V={V}")


def test_backward_chunks_and_invariance(tim):
    b = synth.make_custom(T=300, d=256, V=3000, temperature=0.9, tag="bwchunk")
    g = upstream(300, 5)
    dy, dW = run(tim, b, g)
    dy2, dW2 = run(tim, b, g, chunk_rows=70)
    assert dy2.tobytes() == dy.tobytes(), "dy rows must not depend on the batch split"
    assert np.max(np.abs(dW2 - dW)) <= 1e-5 * np.max(np.abs(dW))
    # accumulate_dW adds: two calls on the same rows give twice dW (exact in fp32)
    import torch
    hid, gam, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    ids = cuda_tensor(b.token_ids)
    _, lse, _ = tim.logprob(hid, gam, W, ids, 0.9, b.eps)
    gd = f32_cuda(g)
    out_dW = torch.empty(3000, 256, dtype=torch.float32, device="cuda")
    tim.logprob_backward(hid, gam, W, ids, lse, gd, 0.9, b.eps, out_dW=out_dW)
    first = out_dW.clone()
    ws = tim.Workspace(int(tim.lib().tim_logprob_backward_workspace_size(300, 256, 3000)))
    dy_dev = torch.empty(300, 256, dtype=torch.float32, device="cuda")
    code = tim.lib().tim_logprob_backward(hid.data_ptr(), gam.data_ptr(), W.data_ptr(),
                                          ids.data_ptr(), lse.data_ptr(), gd.data_ptr(), 300, 256,
                                          3000, 0.9, b.eps, dy_dev.data_ptr(), out_dW.data_ptr(),
                                          1, ws.ptr, ws.nbytes, None)
    assert code == 0
    ws.check("accumulate")
    assert torch.equal(out_dW, 2 * first)


def test_backward_invalid_token(tim):
    b = synth.make_custom(T=40, d=128, V=700, tag="bwbad")
    ids = b.token_ids.copy()
    ids[3] = 700
    import torch
    hid, gam, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    lse = torch.zeros(40, dtype=torch.float32, device="cuda")
    ws = tim.Workspace(int(tim.lib().tim_logprob_backward_workspace_size(40, 128, 700)))
    dy, dW = tim.logprob_backward(hid, gam, W, cuda_tensor(ids), lse, f32_cuda(np.ones(40)), 1.0,
                                  b.eps, workspace=ws, check=False)
    torch.cuda.synchronize()
    assert not torch.any(dy[3]).item()
    with pytest.raises(tim.TimError) as ei:
        ws.check("bad token")
    assert ei.value.name == "TIM_ERR_TOKEN_RANGE"


def test_backward_full_head(tim):
    b = synth.make_custom(T=128, d=4096, V=151936, temperature=0.7, tag="bwfull")
    g = upstream(128, 11)
    dy, dW = run(tim, b, g)
    vrows = np.unique(np.concatenate([b.token_ids[:16], sample_rows(151936, 48)]))
    orc = oracle.oracle_logprob_backward(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 0.7,
                                         b.eps, g, dW_rows=vrows)
    check(b, g, dy, dW, orc, dW_rows=vrows, what="full head")
    # dy rows are batch-invariant
    hid, gam, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    sub = slice(13, 77)
    bs = synth.make_custom(T=64, d=4096, V=151936, temperature=0.7, tag="bwfull")
    bs.hidden_gen, bs.token_ids = b.hidden_gen[sub].copy(), b.token_ids[sub].copy()
    dys, _ = run(tim, bs, g[sub])
    assert dys.tobytes() == dy[sub].tobytes()
