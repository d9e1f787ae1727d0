"""The vocabulary-parallel path (G shards run one after another on one GPU, records merged
in rank order) gives bitwise the same logprob / lse / top-1 as tim_logprob, and matches
the oracle."""
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


@pytest.mark.parametrize("T,d,V,tau", [(300, 128, 1000, 1.0), (129, 256, 5000, 0.7),
                                       (70, 192, 4099, 1.3), (64, 4096, 151936, 0.7)])
def test_sharded_equals_unsharded(tim, T, d, V, tau):
    b = synth.make_custom(T=T, d=d, V=V, temperature=tau, tag=f"vp{T}_{d}_{V}")
    ids = b.token_ids.copy()
    ids[3] = V - 1                       # a target in the last (partial) tile
    hid, gam, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    ids_d = cuda_tensor(ids)
    ref = [x.cpu().numpy() for x in tim.logprob(hid, gam, W, ids_d, tau, b.eps)]
    for G in (1, 2, 4, 8, 16):
        got = [x.cpu().numpy() for x in tim.logprob_vocab_parallel_emulated(hid, gam, W, ids_d, G,
                                                                             tau, b.eps)]
        for x, y in zip(got, ref):
            assert x.tobytes() == y.tobytes(), f"G={G}: sharded result differs from unsharded"
    rows = np.arange(min(T, 40))
    orc = oracle.oracle_logprob(b.hidden_gen[rows], b.head.gamma, b.head.W, ids[rows], tau, b.eps)
    assert_logprob_parity(ref, orc, rows=rows, what="vocab-parallel")


def test_merge_reports_token_range(tim):
    b = synth.make_custom(T=20, d=64, V=700, tag="vpbad")
    ids = b.token_ids.copy()
    ids[2] = 700
    with pytest.raises(tim.TimError) as ei:
        tim.logprob_vocab_parallel_emulated(bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma),
                                            bf16_cuda(b.head.W), cuda_tensor(ids), 4, 1.0, b.eps)
    assert ei.value.name == "TIM_ERR_TOKEN_RANGE"
