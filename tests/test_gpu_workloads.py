"""Full-size scoring workloads on the GPU, through the C ABI, in the launch
configuration the benchmark times.  The fp64 oracle checks rows one by one: one
seeded row inside every 128-row tile and both ends of every raster group of the
GEMM's schedule (``parity.tile_rows``); properties that hold at any size
(bitwise replay equality, same-prefix siblings, batch invariance, the eq. (1)
split) are checked on all rows."""
import numpy as np
import pytest

import oracle
import synth
from parity import (assert_compare_parity, assert_logprob_parity, assert_tis_parity,
                    bf16_cuda, covered_rows, cuda_tensor, raster_group_tiles, tile_rows)

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


def score(tim, hidden_dev, gamma_dev, W_dev, ids_dev, tau, eps, splits=None):
    """Score all rows; with ``splits`` (row index arrays) score them in several calls."""
    import torch
    T = hidden_dev.shape[0]
    if splits is None:
        lp, lse, top1 = tim.logprob(hidden_dev, gamma_dev, W_dev, ids_dev, tau, eps)
        return lp.cpu().numpy(), lse.cpu().numpy(), top1.cpu().numpy()
    lp = np.empty(T, np.float32)
    lse = np.empty(T, np.float32)
    top1 = np.empty(T, np.int32)
    for rows in splits:
        r = torch.from_numpy(rows).cuda()
        a, b, c = tim.logprob(hidden_dev[r].contiguous(), gamma_dev, W_dev, ids_dev[r].contiguous(),
                              tau, eps)
        lp[rows], lse[rows], top1[rows] = a.cpu().numpy(), b.cpu().numpy(), c.cpu().numpy()
    return lp, lse, top1


def same_bits(x, y):
    return all(np.array_equal(np.asarray(a).view(np.uint32), np.asarray(b).view(np.uint32))
               for a, b in zip(x, y))


def three_way(tim, b, W_train_bits=None):
    hid = bf16_cuda(b.hidden_gen)
    hid_c = bf16_cuda(b.hidden_train)
    gam = bf16_cuda(b.head.gamma)
    W = bf16_cuda(b.head.W)
    Wc = W if W_train_bits is None else bf16_cuda(W_train_bits)
    ids = cuda_tensor(b.token_ids)
    A = score(tim, hid, gam, W, ids, b.temperature, b.eps)
    perm = np.random.default_rng(5).permutation(b.T)
    cuts = [0, b.T // 3, b.T // 3 + 1, b.T]
    B = score(tim, hid, gam, W, ids, b.temperature, b.eps,
              splits=[np.sort(perm[cuts[i]:cuts[i + 1]]) for i in range(3)])
    C = score(tim, hid_c, gam, Wc, ids, b.temperature, b.eps)
    assert same_bits(A, B), "replay in another batch split must be bitwise identical"
    rows = tile_rows(b.T, raster_group_tiles(b.head.d))
    oA = oracle.oracle_logprob(b.hidden_gen[rows], b.head.gamma, b.head.W, b.token_ids[rows],
                               b.temperature, b.eps)
    assert_logprob_parity(A, oA, rows=rows, what=f"{b.name} A")
    oC = oracle.oracle_logprob(b.hidden_train[rows], b.head.gamma,
                               b.head.W if W_train_bits is None else W_train_bits,
                               b.token_ids[rows], b.temperature, b.eps)
    assert_logprob_parity(C, oC, rows=rows, what=f"{b.name} C")
    g, w = tim.compare(cuda_tensor(A[0]), cuda_tensor(B[0]), cuda_tensor(C[0]),
                       cuda_tensor(b.seq_offsets), cuda_tensor(b.mask), b.tis_cap)
    gs = tim.stats_to_dicts(g)
    r, rw = oracle.oracle_compare(A[0], B[0], C[0], b.seq_offsets, b.mask, b.tis_cap)
    assert_compare_parity(gs, r, what=b.name)
    assert_tis_parity(w.cpu().numpy(), rw, covered_rows(b.seq_offsets, b.T))
    # extended diagnostics on the same arrays, with the top-1 ids of each score set
    from test_gpu_diag import assert_diag_parity, d_abs
    tops = (cuda_tensor(A[2]), cuda_tensor(B[2]), cuda_tensor(C[2]))
    gd = tim.diag_to_dicts(tim.compare_diag(
        cuda_tensor(A[0]), cuda_tensor(B[0]), cuda_tensor(C[0]), cuda_tensor(b.seq_offsets),
        cuda_tensor(b.mask), b.tis_cap, 0.5, 2.0, top1=tops))
    rd = oracle.oracle_diag(A[0], B[0], C[0], b.seq_offsets, b.mask, b.tis_cap, 0.5, 2.0,
                            (A[2], B[2], C[2]))
    assert_diag_parity(gd, rd, d_abs(A[0], C[0], b.seq_offsets, b.mask), what=b.name)
    for st in gs:  # A and B agree bitwise: same-version term is exactly zero
        assert st["pair"][0]["mismatch_count"] == 0 and st["mean_same_version"] == 0.0
        lhs = st["mean_log_ratio"]
        rhs = st["mean_weight_move"] + st["mean_same_version"]
        assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))
    return A, C, gs


def test_qwen3_1p7b_head(tim):
    b = synth.make_qwen3_1p7b()
    three_way(tim, b)


def test_qwen3_8b_head_siblings(tim):
    b = synth.make_qwen3_8b()
    A, C, gs = three_way(tim, b)
    L, P = b.meta["L"], b.meta["prefix"]
    for s in range(1, b.meta["S"]):
        for X in (A, C):
            for arr in X:
                assert np.asarray(arr[s * L:s * L + P]).tobytes() == np.asarray(arr[:P]).tobytes(), \
                    f"sample {s}: shared prefix not bitwise identical"


def test_batch_invariance_sweep_8b_head(tim):
    """The 4096 target rows in batches of M = 1, 7, 64, 513, 4096 and 16384, plus
    M = 200, 256, 384, 512, 768, 1152, 6144 and 6145, covering every schedule form of
    the GEMM: one row tile (M <= 128); a row-tile pair per W tile (200, 256); pairs
    with several items per W tile and the leader's L2 prefetch (512, 768, 4096, and
    6144 = the 48-tile raster group); odd tile counts, one row tile per item with the
    prefetch (384, 513, 1152); and batches of several raster groups, as pairs (16384)
    and one row tile per item (6145, 49 tiles).  Every target keeps its bits."""
    import torch
    plan = synth.make_sweep(Ms=(1, 7, 64, 200, 256, 384, 512, 513, 768, 1152, 4096, 6144, 6145,
                                16384))
    head = plan.head
    gam, W = bf16_cuda(head.gamma), bf16_cuda(head.W)
    ref = None
    for M, batches in plan.batches.items():
        ws = tim.Workspace(tim.logprob_workspace_size(M, head.d, head.V))
        out = (torch.empty(M, device="cuda"), torch.empty(M, device="cuda"),
               torch.empty(M, dtype=torch.int32, device="cuda"))
        got = np.zeros((plan.targets_ids.shape[0], 3), np.uint32)
        for bt in batches:
            lp, lse, top1 = tim.logprob(bf16_cuda(bt["hidden"]), gam, W, cuda_tensor(bt["ids"]),
                                        plan.temperature, plan.eps, out=out, workspace=ws,
                                        check=False)
            pos = bt["target_pos"]
            got[bt["target_idx"], 0] = lp.cpu().numpy()[pos].view(np.uint32)
            got[bt["target_idx"], 1] = lse.cpu().numpy()[pos].view(np.uint32)
            got[bt["target_idx"], 2] = top1.cpu().numpy()[pos].view(np.uint32)
        ws.check(f"M={M}")
        if ref is None:
            ref = got
            rows = tile_rows(got.shape[0], raster_group_tiles(head.d))
            orc = oracle.oracle_logprob(plan.targets_hidden[rows], head.gamma, head.W,
                                        plan.targets_ids[rows], plan.temperature, plan.eps)
            assert_logprob_parity((got[:, 0].view(np.float32), got[:, 1].view(np.float32),
                                   got[:, 2].view(np.int32)), orc, rows=rows, what="sweep")
        else:
            diff = np.flatnonzero(np.any(ref != got, axis=1))
            assert diff.size == 0, f"M={M}: {diff.size} target rows differ bitwise"


def test_long_rollout_5120_stale_weights(tim):
    b = synth.make_long_5120()
    A, C, gs = three_way(tim, b, W_train_bits=b.W_train)
    # a stale weight version moves every active token (Case 3 pattern: A == B, C differs)
    assert all(st["pair"][1]["mismatch_count"] > 0.9 * st["n_valid"] for st in gs)
