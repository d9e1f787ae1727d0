"""tim_logprob (through the C ABI) against the fp64 oracle: small and ragged shapes,
temperatures, batch invariance, and the data-dependent error paths."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_logprob_parity, bf16_cuda, cuda_tensor

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


def run(tim, hidden_bits, gamma_bits, W_bits, ids, tau, eps, check=True):
    lp, lse, top1 = tim.logprob(bf16_cuda(hidden_bits), bf16_cuda(gamma_bits), bf16_cuda(W_bits),
                                cuda_tensor(np.asarray(ids, dtype=np.int32)), tau, eps,
                                check=check)
    return lp.cpu().numpy(), lse.cpu().numpy(), top1.cpu().numpy()


SHAPES = [
    # (T, d, V, tau): one row, one column, ragged row/vocab tails, several M and N tiles
    (1, 64, 1, 1.0),
    (1, 64, 300, 0.7),
    (7, 64, 257, 1.0),
    (64, 128, 1000, 1.0),
    (129, 128, 1000, 0.5),
    (300, 256, 513, 1.3),
    (257, 192, 2048, 1.0),
    (384, 128, 1000, 1.0),
    (512, 256, 3001, 0.8),
    (513, 320, 4099, 0.9),
    (640, 64, 151936, 0.9),   # five row tiles, one per item, the leader prefetching W
    (1024, 4096, 20000, 0.9), # eight row tiles as four pairs per W tile, with the prefetch
    (1024, 64, 151936, 0.9),  # the same at d < 4096: one row tile per item, with the prefetch
    (256, 5120, 3001, 0.7),   # row-tile pairs at the long-rollout hidden size
]


@pytest.mark.parametrize("T,d,V,tau", SHAPES)
def test_parity_small(tim, T, d, V, tau):
    b = synth.make_custom(T=T, d=d, V=V, temperature=tau, tag=f"p{T}_{d}_{V}")
    gpu = run(tim, b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, tau, b.eps)
    orc = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, tau, b.eps)
    assert_logprob_parity(gpu, orc, what=f"T={T} d={d} V={V}")


def test_concurrent_streams_same_bits(tim):
    """Scoring the same rows on two streams at once, each in its own batch composition
    (the GEMMs then share the SMs and run with fewer resident CTAs each), gives exactly
    the bits of a lone call: no result depends on which CTA or SM computes a tile."""
    import torch
    b = synth.make_custom(T=700, d=512, V=20000, temperature=0.9, tag="streams")
    hid, gam, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    ids = cuda_tensor(b.token_ids)
    ref = [x.cpu().numpy() for x in tim.logprob(hid, gam, W, ids, 0.9, b.eps)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        with torch.cuda.stream(s1):
            a = tim.logprob(hid, gam, W, ids, 0.9, b.eps, stream=s1, check=False)
        with torch.cuda.stream(s2):
            c = tim.logprob(hid[100:600].contiguous(), gam, W, ids[100:600].contiguous(), 0.9,
                            b.eps, stream=s2, check=False)
        outs.append((a, c))
    torch.cuda.synchronize()
    for a, c in outs:
        for x, r in zip(a, ref):
            assert x.cpu().numpy().tobytes() == r.tobytes()
        for x, r in zip(c, ref):
            assert x.cpu().numpy().tobytes() == r[100:600].tobytes()


def test_large_logits(tim):
    """W scaled by 16 (exact in bf16): logits of +-100 and more, logprobs near -200 for
    the tail; the max-shifted merge keeps every row finite and within tolerance."""
    b = synth.make_custom(T=100, d=256, V=3000, temperature=0.8, tag="biglogit")
    W16 = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(b.head.W) * 16.0)
    # hidden = +-2 with eps = 0: y = +-gamma exactly, so no bf16 rounding of y can differ
    # between the fp32 kernel and the fp64 oracle (a one-step difference of y would move
    # these large logits by ~1e-3)
    sign = np.random.default_rng(4).random((100, 256)) < 0.5
    hid = np.where(sign, 0xC000, 0x4000).astype(np.uint16)
    gpu = run(tim, hid, b.head.gamma, W16, b.token_ids, 0.8, 0.0)
    orc = oracle.oracle_logprob(hid, b.head.gamma, W16, b.token_ids, 0.8, 0.0)
    assert orc["zmax"].max() > 50
    assert_logprob_parity(gpu, orc, what="W x 16")


@pytest.mark.parametrize("tau", [0.05, 10.0])
def test_temperature_extremes(tim, tau):
    """tau = 0.05 (scaled logits up to ~200, one token holds almost all mass) and tau = 10
    (nearly flat).  y is made exact (hidden = +-2, eps = 0: y = +-gamma) because a logprob
    divides logit differences by tau, and a one-bf16-step difference of y between the fp32
    kernel and the fp64 oracle would be magnified twentyfold at tau = 0.05."""
    b = synth.make_custom(T=64, d=128, V=1000, temperature=tau, tag="tau_ext")
    sign = np.random.default_rng(5).random((64, 128)) < 0.5
    hid = np.where(sign, 0xC000, 0x4000).astype(np.uint16)
    gpu = run(tim, hid, b.head.gamma, b.head.W, b.token_ids, tau, 0.0)
    orc = oracle.oracle_logprob(hid, b.head.gamma, b.head.W, b.token_ids, tau, 0.0)
    assert_logprob_parity(gpu, orc, what=f"tau={tau}")


def test_tiny_workload_parity_and_replay_split(tim):
    """The 64-row tiny workload: A and C against the oracle; B = the same rows scored in a
    different batch split and order must equal A bitwise."""
    b = synth.make_tiny()
    A = run(tim, b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 1.0, b.eps)
    C = run(tim, b.hidden_train, b.head.gamma, b.head.W, b.token_ids, 1.0, b.eps)
    oA = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 1.0, b.eps)
    oC = oracle.oracle_logprob(b.hidden_train, b.head.gamma, b.head.W, b.token_ids, 1.0, b.eps)
    assert_logprob_parity(A, oA, what="tiny A")
    assert_logprob_parity(C, oC, what="tiny C")
    perm = np.random.default_rng(0).permutation(b.T)
    Bparts = {}
    for lo, hi in ((0, 7), (7, 28), (28, 64)):
        rows = perm[lo:hi]
        out = run(tim, b.hidden_gen[rows], b.head.gamma, b.head.W, b.token_ids[rows], 1.0, b.eps)
        for k, r in enumerate(rows):
            Bparts[int(r)] = (out[0][k], out[1][k], out[2][k])
    for r in range(b.T):
        assert Bparts[r][0].tobytes() == A[0][r].tobytes()
        assert Bparts[r][1].tobytes() == A[1][r].tobytes()
        assert Bparts[r][2] == A[2][r]


def test_eps_and_scale(tim):
    b = synth.make_custom(T=40, d=256, V=700, tag="eps")
    for eps in (0.0, 1e-5, 0.5):
        gpu = run(tim, b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 1.0, eps)
        orc = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, b.token_ids, 1.0, eps)
        assert_logprob_parity(gpu, orc, what=f"eps={eps}")


def test_batch_invariance_small(tim):
    """Targets scored inside batches of different sizes, positions and neighbours give
    bitwise identical (logprob, lse, top1)."""
    head = synth.make_custom(T=1, d=256, V=3000, tag="bi").head
    plan = synth.make_sweep(Ms=(1, 7, 64, 129, 200, 384, 512, 513), n_targets=200, head=head)
    ref = None
    for M, batches in plan.batches.items():
        got = np.zeros((200, 3), dtype=np.uint32)
        for bt in batches:
            lp, lse, top1 = run(tim, bt["hidden"], head.gamma, head.W, bt["ids"], 0.7, 1e-6)
            got[bt["target_idx"], 0] = lp[bt["target_pos"]].view(np.uint32)
            got[bt["target_idx"], 1] = lse[bt["target_pos"]].view(np.uint32)
            got[bt["target_idx"], 2] = top1[bt["target_pos"]].view(np.uint32)
        if ref is None:
            ref = got
            orc = oracle.oracle_logprob(plan.targets_hidden, head.gamma, head.W, plan.targets_ids,
                                        0.7, 1e-6)
            assert_logprob_parity((got[:, 0].view(np.float32), got[:, 1].view(np.float32),
                                   got[:, 2].view(np.int32)), orc, what="sweep")
        else:
            assert np.array_equal(ref, got), f"M={M}: rows differ bitwise"


def test_invalid_token_ids(tim):
    b = synth.make_custom(T=20, d=64, V=500, tag="badid")
    ids = b.token_ids.copy()
    ids[3] = 500
    ids[11] = -2
    lp, lse, top1 = tim.logprob(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma),
                                bf16_cuda(b.head.W), cuda_tensor(ids), 1.0, b.eps, check=False)
    ws_err = None
    try:
        tim.logprob(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W),
                    cuda_tensor(ids), 1.0, b.eps, check=True)
    except tim.TimError as e:
        ws_err = e.name
    assert ws_err == "TIM_ERR_TOKEN_RANGE"
    gpu = (lp.cpu().numpy(), lse.cpu().numpy(), top1.cpu().numpy())
    orc = oracle.oracle_logprob(b.hidden_gen, b.head.gamma, b.head.W, ids, 1.0, b.eps)
    assert_logprob_parity(gpu, orc, what="bad ids")


def test_nonfinite_hidden(tim):
    b = synth.make_custom(T=9, d=64, V=100, tag="nan")
    h = b.hidden_gen.copy()
    h[4, 10] = 0x7FC0  # bf16 NaN
    with pytest.raises(tim.TimError) as ei:
        run(tim, h, b.head.gamma, b.head.W, b.token_ids, 1.0, b.eps)
    assert ei.value.name == "TIM_ERR_NONFINITE"
    # the workspace status is cleared by the sync: a clean call afterwards reports OK
    ws = tim.Workspace(tim.logprob_workspace_size(9, 64, 100))
    tim.logprob(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W),
                cuda_tensor(b.token_ids), 1.0, b.eps, workspace=ws, check=True)


def test_stages_equal_fused_call(tim):
    import torch
    b = synth.make_custom(T=150, d=128, V=1500, tag="stg")
    hidden, gamma, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    ids = cuda_tensor(b.token_ids)
    a = tim.logprob(hidden, gamma, W, ids, 0.8, b.eps)
    ws = tim.Workspace(tim.logprob_workspace_size(150, 128, 1500))
    out = (torch.empty(150, device="cuda"), torch.empty(150, device="cuda"),
           torch.empty(150, dtype=torch.int32, device="cuda"))
    tim.logprob_stages(hidden, gamma, W, ids, 0.8, b.eps, out, ws)
    ws.check()
    for x, y in zip(a, out):
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                           y.view(torch.int32) if y.dtype == torch.float32 else y)


def test_argument_errors_on_device(tim):
    b = synth.make_custom(T=4, d=64, V=10, tag="arg")
    with pytest.raises(tim.TimError) as ei:
        tim.logprob(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W),
                    cuda_tensor(b.token_ids), 0.0, b.eps)
    assert ei.value.name == "TIM_ERR_INVALID_ARG"
    small = tim.Workspace(1024)
    with pytest.raises(tim.TimError) as ei:
        tim.logprob(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W),
                    cuda_tensor(b.token_ids), 1.0, b.eps, workspace=small)
    assert ei.value.name == "TIM_ERR_WORKSPACE"
