"""Scoring and the three-way compare captured once in a CUDA graph and replayed.

tim_logprob and tim_compare enqueue only kernel launches on the
caller's stream, allocate nothing and never synchronise when the caller passes its own
output buffers and workspace, so a serving loop can capture them once and replay the
graph on new inputs written into the same buffers.  Each replay must give exactly the
bits of a direct call on the same inputs: the graph changes neither the kernels nor
their order, and the scores are batch-invariant by construction anyway.
"""
import numpy as np
import pytest

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


def _bits(ts):
    return [t.cpu().numpy().tobytes() for t in ts]


@pytest.mark.parametrize("T", [200, 300])  # two row tiles (row-tile pairs), three (one tile each)
def test_logprob_graph_replay_same_bits(tim, T):
    import torch
    b = synth.make_custom(T=T, d=256, V=3000, temperature=0.8, tag=f"graph{T}")
    gam, W, ids = bf16_cuda(b.head.gamma), bf16_cuda(b.head.W), cuda_tensor(b.token_ids)
    hid = bf16_cuda(b.hidden_gen).clone()            # the graph's static input
    out = (torch.empty(T, device="cuda"), torch.empty(T, device="cuda"),
           torch.empty(T, dtype=torch.int32, device="cuda"))
    ws = tim.Workspace(tim.logprob_workspace_size(T, 256, 3000))
    tim.logprob(hid, gam, W, ids, 0.8, b.eps, out=out, workspace=ws)   # warm-up, checked
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tim.logprob(hid, gam, W, ids, 0.8, b.eps, out=out, workspace=ws, check=False)

    for source in (b.hidden_train, b.hidden_gen, b.hidden_train):
        hid.copy_(bf16_cuda(source))
        g.replay()
        torch.cuda.synchronize()
        ws.check("graph replay")
        direct = tim.logprob(bf16_cuda(source), gam, W, ids, 0.8, b.eps)
        assert _bits(out) == _bits(direct)


def test_compare_graph_replay_same_bits(tim):
    import torch
    b = synth.make_custom(T=600, d=64, V=500, seq_len=150, n_resp=100, tag="graphcmp")
    rng = np.random.default_rng(7)
    sets = [rng.normal(-3.0, 1.0, size=(3, 600)).astype(np.float32) for _ in range(3)]
    sets[1][1] = sets[1][0]                           # B == A: no mismatch in pair A-B
    offs, mask = cuda_tensor(b.seq_offsets), cuda_tensor(b.mask)
    lp = [torch.empty(600, device="cuda") for _ in range(3)]   # static inputs
    S = b.seq_offsets.shape[0] - 1
    stats = torch.empty(S * tim.SEQ_STATS_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    tis_w = torch.empty(600, device="cuda")
    ws = tim.Workspace(tim.compare_workspace_size(600, S))
    for x, v in zip(lp, sets[0]):
        x.copy_(torch.from_numpy(v))
    tim.compare(*lp, offs, mask, 2.0, out_stats=stats, out_tis_w=tis_w, workspace=ws,
                to_host=False)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tim.compare(*lp, offs, mask, 2.0, out_stats=stats, out_tis_w=tis_w, workspace=ws,
                    check=False, to_host=False)

    for s in sets:
        for x, v in zip(lp, s):
            x.copy_(torch.from_numpy(v))
        g.replay()
        torch.cuda.synchronize()
        ws.check("graph replay")
        d_stats, d_w = tim.compare(*[torch.from_numpy(v).cuda() for v in s], offs, mask, 2.0,
                                   to_host=False)
        assert _bits([stats, tis_w]) == _bits([d_stats, d_w])
