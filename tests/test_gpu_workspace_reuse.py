"""One workspace reused by tim_compare / tim_compare_diag calls of changing shape.

The per-sequence part counters live at offsets that depend on the sequence
count, so a call with more sequences than the last one finds the previous
call's bases and partials where its counters go.  Each call must still give
the bits of a call on a fresh workspace (the partition kernel of every call
zeroes the counters it uses), also right after a call that failed."""
import math

import numpy as np
import pytest

from parity import cuda_tensor

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


def _same(x, y):
    if isinstance(x, dict):
        return x.keys() == y.keys() and all(_same(x[k], y[k]) for k in x)
    if isinstance(x, (list, tuple)):
        return len(x) == len(y) and all(_same(a, b) for a, b in zip(x, y))
    if isinstance(x, float) and math.isnan(x):
        return isinstance(y, float) and math.isnan(y)
    return x == y


def _case(T, S, seed, bad_offsets=False):
    g = np.random.default_rng(seed)
    A = (-np.abs(g.standard_normal(T)) * 4).astype(np.float32)
    B = np.where(g.random(T) < 0.3, A + np.float32(1e-3) * g.standard_normal(T), A).astype(np.float32)
    C = (B + np.float32(0.05) * g.standard_normal(T)).astype(np.float32)
    cuts = np.sort(g.choice(np.arange(1, T), size=S - 1, replace=False))
    offs = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    if bad_offsets:
        offs[S // 2] = offs[S // 2 + 1] + 1          # one sequence with end < start
    mask = np.ones(T, np.uint8)
    tops = [g.integers(0, 40, T).astype(np.int32) for _ in range(3)]
    return A, B, C, offs, mask, tops


# (T, S, bad offsets): fewer sequences, then many more, one, a failing call, another shape
SHAPES = [(50, 2, False), (30000, 200, False), (5000, 1, False), (30000, 300, True),
          (20000, 250, False), (30000, 300, False)]


def _run_compare(tim, case, ws, check):
    A, B, C, offs, mask, _ = case
    stats, w = tim.compare(cuda_tensor(A), cuda_tensor(B), cuda_tensor(C), cuda_tensor(offs),
                           cuda_tensor(mask), 2.0, workspace=ws, check=check)
    return tim.stats_to_dicts(stats), w.cpu().numpy().tobytes()


def _run_diag(tim, case, ws, check):
    A, B, C, offs, mask, tops = case
    arr = tim.compare_diag(cuda_tensor(A), cuda_tensor(B), cuda_tensor(C), cuda_tensor(offs),
                           cuda_tensor(mask), 2.0, 0.5, 1.5,
                           top1=tuple(cuda_tensor(t) for t in tops), workspace=ws, check=check)
    return tim.diag_to_dicts(arr)


@pytest.mark.parametrize("family", ["compare", "diag"])
def test_workspace_reused_across_shapes(tim, family):
    import torch
    lib = tim.lib()
    size = (lib.tim_compare_workspace_size if family == "compare"
            else lib.tim_compare_diag_workspace_size)
    run = _run_compare if family == "compare" else _run_diag
    shared = tim.Workspace(max(int(size(T, S)) for T, S, _ in SHAPES), torch.device("cuda"))
    for i, (T, S, bad) in enumerate(SHAPES):
        case = _case(T, S, 100 + i, bad)
        fresh = tim.Workspace(int(size(T, S)), torch.device("cuda"))
        if bad:
            with pytest.raises(tim.TimError):
                run(tim, case, shared, True)           # raises and clears the status word
            got, want = run(tim, case, shared, False), run(tim, case, fresh, False)
            fresh.sync_status()
            shared.sync_status()
        else:
            got, want = run(tim, case, shared, True), run(tim, case, fresh, True)
        assert _same(got, want), (family, T, S)
