"""tim_compare (through the C ABI) against the fp64 oracle run on the same score arrays."""
import math

import numpy as np
import pytest

import oracle
from parity import assert_compare_parity, assert_tis_parity, covered_rows, cuda_tensor

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


def gpu_compare(tim, A, B, C, offs, mask, cap, check=True, offset_elems=0):
    import torch
    def dev(x, dt):
        t = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        if offset_elems:
            pad = torch.zeros(t.shape[0] + offset_elems, dtype=t.dtype, device="cuda")
            pad[offset_elems:] = t
            return pad[offset_elems:]
        return t
    stats, w = tim.compare(dev(A, np.float32), dev(B, np.float32), dev(C, np.float32),
                           cuda_tensor(np.asarray(offs, np.int64)), dev(mask, np.uint8),
                           cap, check=check)
    return tim.stats_to_dicts(stats), w.cpu().numpy()


def scores(n, seed, noise=1e-2, heavy=0.0):
    g = np.random.default_rng(seed)
    A = (-np.abs(g.standard_normal(n)) * 4).astype(np.float32)
    B = A.copy()
    flip = g.random(n) < 0.3
    B[flip] = (A[flip] + g.standard_normal(flip.sum()).astype(np.float32) * np.float32(1e-3))
    C = (B + g.standard_normal(n).astype(np.float32) * np.float32(noise)).astype(np.float32)
    if heavy:
        k = g.random(n) < 0.02
        C[k] += np.float32(heavy)
    return A, B, C


def layouts(T, seed):
    g = np.random.default_rng(seed)
    cuts = np.sort(g.choice(np.arange(1, T), size=min(T - 1, 9), replace=False))
    offs = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    mask = np.zeros(T, np.uint8)
    for j in range(len(offs) - 1):
        a, b = offs[j], offs[j + 1]
        p = a + (b - a) // 3
        mask[p:b] = 1
        mask[a + g.integers(0, max(1, b - a)):b][::5] = 0   # gaps inside the response
        if mask[a:b].sum() == 0:
            mask[b - 1] = 1
    return offs, mask


@pytest.mark.parametrize("T,seed,offset", [(1, 0, 0), (37, 1, 0), (1000, 2, 0), (1000, 3, 1),
                                            (4099, 4, 0), (20000, 5, 3), (70001, 6, 0)])
def test_compare_parity_random(tim, T, seed, offset):
    A, B, C = scores(T, seed, heavy=3.0)
    offs, mask = layouts(T, seed) if T > 1 else (np.array([0, 1]), np.ones(1, np.uint8))
    g, w = gpu_compare(tim, A, B, C, offs, mask, 2.0, offset_elems=offset)
    r, rw, errs = oracle.oracle_compare_lenient(A, B, C, offs, mask, 2.0)
    assert not errs
    assert_compare_parity(g, r, what=f"T={T}")
    assert_tis_parity(w, rw, covered_rows(offs, T))


def test_identical_sets(tim):
    A, _, _ = scores(5000, 9)
    offs = np.array([0, 1000, 2500, 5000])
    mask = np.ones(5000, np.uint8)
    g, w = gpu_compare(tim, A, A, A, offs, mask, 2.0)
    for st in g:
        for p in st["pair"]:
            assert p["mismatch_count"] == 0 and p["first_div"] == -1 and p["longest_run"] == 0
            assert p["max_abs_diff"] == 0.0 and p["signed_mean"] == 0.0
        assert st["k3_mean"] == 0.0 and st["tis_mean"] == 1.0 and st["tis_clipped"] == 0
    assert np.all(w == 1.0)


def test_signed_zero_and_runs(tim):
    mask = np.array([1, 1, 0, 1, 1, 1, 0, 1], np.uint8)
    A = np.full(8, -1.0, np.float32)
    B = A.copy()
    for pos in (1, 3, 4, 7, 6):
        B[pos] = -1.5
    A[0], B[0] = 0.0, -0.0
    g, _ = gpu_compare(tim, A, B, B, [0, 8], mask, 2.0)
    r, _, _ = oracle.oracle_compare_lenient(A, B, B, [0, 8], mask, 2.0)
    assert_compare_parity(g, r)
    assert g[0]["pair"][0]["mismatch_count"] == 5 and g[0]["pair"][0]["longest_run"] == 4


@pytest.mark.parametrize("case", ["empty", "bad_mask", "nan_active", "bad_offsets"])
def test_compare_errors(tim, case):
    A, B, C = scores(64, 11)
    offs = np.array([0, 16, 32, 48, 64])
    mask = np.ones(64, np.uint8)
    want = {"empty": "TIM_ERR_EMPTY_SEQUENCE", "bad_mask": "TIM_ERR_BAD_MASK",
            "nan_active": "TIM_ERR_NONFINITE", "bad_offsets": "TIM_ERR_INVALID_ARG"}[case]
    if case == "empty":
        mask[16:32] = 0
    elif case == "bad_mask":
        mask[40] = 2
    elif case == "nan_active":
        C[50] = np.nan
        A[5] = np.nan
        mask[5] = 0   # NaN on an inactive token is allowed
    else:
        offs = np.array([0, 16, 12, 48, 64])
    with pytest.raises(tim.TimError) as ei:
        gpu_compare(tim, A, B, C, offs, mask, 2.0)
    assert ei.value.name == want
    g, _ = gpu_compare(tim, A, B, C, offs, mask, 2.0, check=False)
    r, _, errs = oracle.oracle_compare_lenient(A, B, C, offs, mask, 2.0)
    assert errs
    assert_compare_parity(g, r, what=case)


def test_k3_overflow_and_tis_clip(tim):
    A = np.array([-900.0, -5.0, -5.0, -5.0], np.float32)
    C = np.array([-50.0, -5.0 + math.log(3.0), -5.0 + math.log(1.5), -6.0], np.float32)
    g, w = gpu_compare(tim, A, A, C, [0, 1, 4], np.ones(4, np.uint8), 2.0)
    r, rw, _ = oracle.oracle_compare_lenient(A, A, C, [0, 1, 4], np.ones(4, np.uint8), 2.0)
    assert g[0]["flags"] & oracle.FLAG_K3_OVERFLOW and math.isinf(g[0]["k3_mean"])
    assert_compare_parity(g, r)
    assert_tis_parity(w, rw, np.ones(4, bool))
    assert g[1]["tis_clipped"] == 1


def test_sequence_stats_do_not_depend_on_the_batch(tim):
    """A sequence's statistics (integers and fp64 sums alike) are the same bits whatever
    batch it is compared in: each sequence is cut into parts by its own length."""
    A, B, C = scores(30000, 11)
    offs = np.array([0, 700, 9000, 9001, 23000, 30000], np.int64)
    mask = np.ones(30000, np.uint8)
    full, wf = gpu_compare(tim, A, B, C, offs, mask, 2.0)
    for j in range(len(offs) - 1):
        a, b = offs[j], offs[j + 1]
        one, w1 = gpu_compare(tim, A[a:b], B[a:b], C[a:b], np.array([0, b - a], np.int64),
                              mask[a:b], 2.0)
        assert one[0] == full[j], j
        assert w1.tobytes() == wf[a:b].tobytes()
    # and inside a differently shaped batch (another sequence in front)
    pre = 5000
    A2 = np.concatenate([A[:pre], A[700:9000]])
    B2 = np.concatenate([B[:pre], B[700:9000]])
    C2 = np.concatenate([C[:pre], C[700:9000]])
    two, _ = gpu_compare(tim, A2, B2, C2, np.array([0, pre, pre + 8300], np.int64),
                         np.ones(pre + 8300, np.uint8), 2.0)
    assert two[1] == full[1]
