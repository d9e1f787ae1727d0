"""The FP8 (e4m3) head (tim_quantize_fp8_rows, tim_logprob_fp8) through the C ABI
against the fp64 FP8 oracle: quantiser codes and scales bit-exact, scores within
2e-3 nats, top-1 exact where the oracle's gap exceeds 1e-3, batch invariance.

y is the fp64 RMSNorm rounded to bf16, as for the bf16 head.  The kernel computes
it in fp32, so where the exact value lies within the kernel's error bound
(``parity.fp8_y_margin``) of a bf16 rounding midpoint it may round the other way,
and when that changes an e4m3 code (or the row scale) the logits move by a code
step.  Each row is therefore checked against its admissible oracle results
(``oracle.oracle_logprob_fp8_admissible``): the oracle's own, plus one per
combination of those roundings."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_fp8_admissible_parity, bf16_cuda, cuda_tensor, fp8_y_margin

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


def e4m3_bits_to_f64(codes):
    import torch
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_quantizer_bit_exact(tim):
    b = synth.make_custom(T=300, d=256, V=500, tag="q8")
    rows = np.concatenate([b.head.W, np.zeros((2, 256), np.uint16)])   # all-zero rows too
    codes, scales = tim.quantize_fp8_rows(bf16_cuda(rows))
    codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
    want_c, want_s = oracle.quantize_rows(oracle.widen_bf16(rows))
    assert np.array_equal(scales.astype(np.float64), want_s)
    assert np.array_equal(e4m3_bits_to_f64(codes), want_c)


@pytest.mark.parametrize("T,d,V,tau", [(1, 128, 300, 1.0), (5, 128, 1, 1.0), (64, 128, 1000, 1.0),
                                       (129, 256, 2049, 0.7), (300, 384, 5000, 1.3),
                                       (77, 5120, 3001, 0.7)])
def test_fp8_parity(tim, T, d, V, tau):
    b = synth.make_custom(T=T, d=d, V=V, temperature=tau, tag=f"f8{T}_{d}_{V}")
    W8, sW = tim.quantize_fp8_rows(bf16_cuda(b.head.W))
    got = [x.cpu().numpy() for x in tim.logprob_fp8(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma),
                                                    W8, sW, cuda_tensor(b.token_ids), tau, b.eps)]
    adm = oracle.oracle_logprob_fp8_admissible(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids,
                                               tau, b.eps, fp8_y_margin(d))
    res = assert_fp8_admissible_parity(got, adm, b.token_ids, V, what=f"fp8 T={T} d={d} V={V}")
    print(f"fp8 T={T} d={d} V={V}: {res}")


def test_fp8_full_head_and_batch_invariance(tim):
    b = synth.make_custom(T=200, d=4096, V=151936, temperature=0.7, tag="f8full")
    W8, sW = tim.quantize_fp8_rows(bf16_cuda(b.head.W))
    hid, gam, ids = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), cuda_tensor(b.token_ids)
    full = [x.cpu().numpy() for x in tim.logprob_fp8(hid, gam, W8, sW, ids, 0.7, b.eps)]
    rows = np.arange(0, 200, 5)
    adm = oracle.oracle_logprob_fp8_admissible(b.hidden_gen[rows], b.head.gamma, b.head.W,
                                               b.token_ids[rows], 0.7, b.eps, fp8_y_margin(4096))
    res = assert_fp8_admissible_parity(full, adm, b.token_ids, 151936, rows=rows,
                                       what="fp8 full head")
    print(f"fp8 full head: {res}")
    part = [x.cpu().numpy() for x in tim.logprob_fp8(hid[13:77].contiguous(), gam, W8, sW,
                                                     cuda_tensor(b.token_ids[13:77]), 0.7, b.eps)]
    for x, y in zip(part, full):
        assert x.tobytes() == y[13:77].tobytes()
    # against the bf16 head: close but not equal (the quantisation moves the logits)
    bf = [x.cpu().numpy() for x in tim.logprob(hid, gam, bf16_cuda(b.head.W), ids, 0.7, b.eps)]
    assert 0 < np.max(np.abs(bf[0] - full[0])) < 0.5


def test_fp8_shape_rules(tim):
    b = synth.make_custom(T=4, d=192, V=300, tag="f8arg")
    W8, sW = tim.quantize_fp8_rows(bf16_cuda(b.head.W))
    with pytest.raises(tim.TimError) as ei:                      # d must be a multiple of 128
        tim.logprob_fp8(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), W8, sW,
                        cuda_tensor(b.token_ids), 1.0, b.eps,
                        workspace=tim.Workspace(1 << 20))
    assert ei.value.name in ("TIM_ERR_SHAPE", "TIM_ERR_WORKSPACE")
