"""RMSNorm backward (tim_rmsnorm_backward) and the custom autograd wrapper
(linear_logprob) through the C ABI against the fp64 oracle.

Tolerance of the RMSNorm backward: fp32 arithmetic with sums of d terms (a row's
s_t) and of at most 256 rows plus one fold per chunk (dgamma): each element of
dh may move by 1e-5 of |r gamma dy| + (r^3 / d) |h| sum |gamma dy h|, each dgamma
by 5e-5 of sum_t |dy h r| (both well above the worst-case fp32 rounding of those
sums at these sizes, about 256 + 128 steps of 2^-24)."""
import numpy as np
import pytest

import oracle
import synth
from parity import bf16_cuda, cuda_tensor

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


def f32_cuda(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def check_rms_bwd(h, g, eps, dy, dh, dgam, what):
    want_dh, want_dg = oracle.rmsnorm_backward(h, g, eps, dy)
    r = 1.0 / np.sqrt(np.mean(h * h, axis=1) + eps)
    d = h.shape[1]
    bound_dh = (np.abs(r[:, None] * g[None, :] * dy) +
                (r ** 3 / d)[:, None] * np.abs(h) * np.sum(np.abs(g[None, :] * dy * h), axis=1)[:, None])
    err = np.abs(dh - want_dh)
    assert np.all(err <= 1e-5 * bound_dh + 1e-30), (what, float(err.max()))
    bound_dg = np.sum(np.abs(dy * h * r[:, None]), axis=0)
    errg = np.abs(dgam - want_dg)
    assert np.all(errg <= 5e-5 * bound_dg + 1e-30), (what, float(errg.max()))


@pytest.mark.parametrize("T,d", [(1, 64), (77, 5120), (300, 256), (1000, 4096)])
def test_rmsnorm_backward_parity(tim, T, d):
    b = synth.make_custom(T=T, d=d, V=16, tag=f"rb{T}_{d}")
    dy = np.random.default_rng(T + d).standard_normal((T, d)).astype(np.float32)
    dh, dg = tim.rmsnorm_backward(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), f32_cuda(dy),
                                  b.eps)
    check_rms_bwd(oracle.widen_bf16(b.hidden_gen), oracle.widen_bf16(b.head.gamma), b.eps,
                  dy.astype(np.float64), dh.cpu().numpy().astype(np.float64),
                  dg.cpu().numpy().astype(np.float64), f"T={T} d={d}")
    # rows are independent: a sub-batch gives the same dh bits; dgamma accumulates
    import torch
    dh2, _ = tim.rmsnorm_backward(bf16_cuda(b.hidden_gen[T // 3:]), bf16_cuda(b.head.gamma),
                                  f32_cuda(dy[T // 3:]), b.eps)
    assert dh2.cpu().numpy().tobytes() == dh.cpu().numpy()[T // 3:].tobytes()
    dg2 = dg.clone()
    tim.rmsnorm_backward(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), f32_cuda(dy), b.eps,
                         out_dgamma=dg2, accumulate_dgamma=True)
    assert torch.equal(dg2, 2 * dg)


def test_linear_logprob_autograd(tim):
    """loss = sum_t g_t logprob_t through the autograd wrapper: the forward values equal
    tim_logprob's bits, the gradients equal the direct calls (cast to bf16) and the fp64
    chain oracle (dW and dy from the logprob backward, then the RMSNorm backward)."""
    import torch
    b = synth.make_custom(T=96, d=256, V=3000, temperature=0.8, tag="agrad")
    g = np.random.default_rng(3).standard_normal(96).astype(np.float32)
    hid = bf16_cuda(b.hidden_gen).clone().requires_grad_()
    gam = bf16_cuda(b.head.gamma).clone().requires_grad_()
    W = bf16_cuda(b.head.W).clone().requires_grad_()
    ids = cuda_tensor(b.token_ids)
    lp = tim.linear_logprob(hid, gam, W, ids, 0.8, b.eps)
    ref_lp, lse, _ = tim.logprob(hid.detach(), gam.detach(), W.detach(), ids, 0.8, b.eps)
    assert lp.detach().cpu().numpy().tobytes() == ref_lp.cpu().numpy().tobytes()
    (lp * f32_cuda(g)).sum().backward()
    dy, dW = tim.logprob_backward(hid.detach(), gam.detach(), W.detach(), ids, lse, f32_cuda(g),
                                  0.8, b.eps)
    dh, dg = tim.rmsnorm_backward(hid.detach(), gam.detach(), dy, b.eps)
    assert torch.equal(W.grad, dW.to(torch.bfloat16))
    assert torch.equal(hid.grad, dh.to(torch.bfloat16))
    assert torch.equal(gam.grad, dg.to(torch.bfloat16))
    # chain oracle: dW within the logprob-backward bound, dh / dgamma from the oracle's dy
    orc = oracle.oracle_logprob_backward(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 0.8,
                                         b.eps, g)
    errw = np.abs(dW.cpu().numpy() - orc["dW"])
    assert np.all(errw <= 3 * 2.0 ** -8 * orc["bound_dW"] + 1e-6 * orc["bound_dW"].max() + 1e-3 *
                  np.abs(orc["dW"]).max())
    h64, g64 = oracle.widen_bf16(b.hidden_gen), oracle.widen_bf16(b.head.gamma)
    want_dh, want_dg = oracle.rmsnorm_backward(h64, g64, b.eps, orc["dy"])
    rel = np.linalg.norm(dh.cpu().numpy() - want_dh) / np.linalg.norm(want_dh)
    assert rel < 5e-3, rel
    relg = np.linalg.norm(dg.cpu().numpy() - want_dg) / np.linalg.norm(want_dg)
    assert relg < 5e-3, relg
