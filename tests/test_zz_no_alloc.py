"""tim_logprob_noalloc, the entry point for callers that cannot allocate device
memory (for example a scoring hook inside an engine that has already claimed the
free device memory for its own pools, or code that must not call cudaMalloc /
cudaFree because they can synchronise the device).  It keeps its scratch in a
fixed 8 MiB array inside the library instead of a caller workspace.

Checked through the C ABI against tim_logprob on two calls in a row (the second
call finds the first call's bytes still in the shared array), within the
parity tolerance of the other tests, and for the size limit at its exact edges.
After the first call (the set-up), calls at sizes not seen before take no device
memory: the free device memory reported by cudaMemGetInfo does not move.  This
file is collected last so that a failure here comes after every other test has
run.
"""
import ctypes

import numpy as np
import pytest

import synth
from parity import LP_TOL, bf16_cuda, cuda_tensor

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import rollout_logprob_consistency_gb300 as tim
    L = tim.lib()
    f = L.tim_logprob_noalloc
    vp = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                  ctypes.c_float, vp, vp, vp, vp, vp]
    return torch, tim, f


def call_noalloc(torch, f, hidden, gamma, W, ids, tau, eps):
    T = hidden.shape[0]
    lp = torch.empty(T, dtype=torch.float32, device="cuda")
    lse = torch.empty(T, dtype=torch.float32, device="cuda")
    top1 = torch.empty(T, dtype=torch.int32, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    code = f(hidden.data_ptr(), gamma.data_ptr(), W.data_ptr(), ids.data_ptr(), T,
             hidden.shape[1], W.shape[0], tau, eps, lp.data_ptr(), lse.data_ptr(),
             top1.data_ptr(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return code, (lp.cpu().numpy(), lse.cpu().numpy(), top1.cpu().numpy()), int(st.item())


def call_into(torch, f, hidden, gamma, W, ids, tau, eps, out):
    """The entry point with outputs allocated beforehand (nothing allocated here)."""
    lp, lse, top1, st = out
    T = hidden.shape[0]
    return f(hidden.data_ptr(), gamma.data_ptr(), W.data_ptr(), ids.data_ptr(), T,
             hidden.shape[1], W.shape[0], tau, eps, lp[:T].data_ptr(), lse[:T].data_ptr(),
             top1[:T].data_ptr(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_takes_no_device_memory_after_setup(env):
    """First call (the set-up) at one row and d = 4096, then calls at sizes not seen
    before -- 129, 300 and 416 rows (one-tile and row-tile-pair GEMM forms) and 384 rows
    at d = 5120 -- leave cudaMemGetInfo's free memory exactly where it was, and give the
    bits of tim_logprob."""
    torch, tim, f = env
    b4 = synth.make_custom(T=416, d=4096, V=151936, temperature=0.7, tag="noalloc_mem4")
    b5 = synth.make_custom(T=384, d=5120, V=151936, temperature=0.7, tag="noalloc_mem5")
    dev = {}
    for key, b in (("4", b4), ("5", b5)):
        dev[key] = (bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W),
                    cuda_tensor(b.token_ids))
    out = (torch.empty(416, dtype=torch.float32, device="cuda"),
           torch.empty(416, dtype=torch.float32, device="cuda"),
           torch.empty(416, dtype=torch.int32, device="cuda"),
           torch.full((1,), -1, dtype=torch.int32, device="cuda"))
    h, g, W, ids = dev["4"]
    assert call_into(torch, f, h[:1], g, W, ids[:1], 0.7, b4.eps, out) == 0      # set-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    results = []
    for key, T, eps in (("4", 129, b4.eps), ("4", 300, b4.eps), ("4", 416, b4.eps),
                        ("5", 384, b5.eps)):
        h, g, W, ids = dev[key]
        assert call_into(torch, f, h[:T], g, W, ids[:T], 0.7, eps, out) == 0
        torch.cuda.synchronize()
        assert int(out[3].item()) == 0
        results.append((key, T, [x[:T].cpu().numpy().copy() for x in out[:3]]))
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
    for key, T, got in results:
        h, g, W, ids = dev[key]
        eps = b4.eps if key == "4" else b5.eps
        ref = [x.cpu().numpy() for x in tim.logprob(h[:T], g, W, ids[:T], 0.7, eps)]
        assert all(x.tobytes() == y.tobytes() for x, y in zip(got, ref)), (key, T)


def test_noalloc_size_limit_at_its_edges(env):
    """The header's limits: 416 rows at d = 4096 and 384 rows at d = 5120 (V = 151936) are
    accepted, one row more is rejected with TIM_ERR_WORKSPACE and nothing enqueued; each
    answer agrees with tim_logprob_workspace_size against the 8 MiB array."""
    torch, tim, f = env
    for d, T_max in ((4096, 416), (5120, 384)):
        b = synth.make_custom(T=T_max + 1, d=d, V=151936, temperature=0.7, tag=f"noalloc_edge{d}")
        hid, gam, W = bf16_cuda(b.hidden_gen), bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
        ids = cuda_tensor(b.token_ids)
        assert tim.logprob_workspace_size(T_max, d, 151936) <= SCRATCH_BYTES
        assert tim.logprob_workspace_size(T_max + 1, d, 151936) > SCRATCH_BYTES
        code, got, status = call_noalloc(torch, f, hid[:T_max], gam, W, ids[:T_max], 0.7, b.eps)
        assert code == 0 and status == 0, (d, code, status)
        ref = [x.cpu().numpy() for x in tim.logprob(hid[:T_max], gam, W, ids[:T_max], 0.7, b.eps)]
        assert all(x.tobytes() == y.tobytes() for x, y in zip(got, ref)), d
        code, _, status = call_noalloc(torch, f, hid, gam, W, ids, 0.7, b.eps)
        assert code == tim.STATUS["TIM_ERR_WORKSPACE"] and status == -1, (d, code, status)


def test_noalloc_matches_workspace_path_twice(env):
    torch, tim, f = env
    b = synth.make_custom(T=200, d=4096, V=151936, temperature=0.7, tag="noalloc")
    gam, W = bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    for rows in (slice(0, 64), slice(0, 200)):          # two calls in a row
        hid = bf16_cuda(b.hidden_gen[rows])
        ids = cuda_tensor(b.token_ids[rows])
        assert tim.logprob_workspace_size(hid.shape[0], 4096, 151936) <= SCRATCH_BYTES
        code, got, status = call_noalloc(torch, f, hid, gam, W, ids, 0.7, b.eps)
        assert code == 0 and status == 0
        ref = [x.cpu().numpy() for x in tim.logprob(hid, gam, W, ids, 0.7, b.eps)]
        assert np.max(np.abs(got[0] - ref[0])) <= LP_TOL
        assert np.max(np.abs(got[1] - ref[1])) <= LP_TOL
        assert np.array_equal(got[2], ref[2])
        # the same kernels on the same rows: bitwise identical in fact
        assert got[0].tobytes() == ref[0].tobytes() and got[1].tobytes() == ref[1].tobytes()


def test_noalloc_status_and_limit(env):
    torch, tim, f = env
    b = synth.make_custom(T=40, d=256, V=3000, tag="noalloc_small")
    gam, W = bf16_cuda(b.head.gamma), bf16_cuda(b.head.W)
    ids_np = b.token_ids.copy()
    ids_np[7] = 3000                                   # out of range -> NaN row + status
    hid, ids = bf16_cuda(b.hidden_gen), cuda_tensor(ids_np)
    code, got, status = call_noalloc(torch, f, hid, gam, W, ids, 1.0, b.eps)
    assert code == 0 and status == tim.STATUS["TIM_ERR_TOKEN_RANGE"] and np.isnan(got[0][7])
    ref = [x.cpu().numpy() for x in tim.logprob(hid, gam, W, ids, 1.0, b.eps, check=False)]
    ok = np.arange(40) != 7
    assert np.max(np.abs(got[0][ok] - ref[0][ok])) <= LP_TOL
    # a following clean call reports no error (the status word is cleared per call)
    code, _, status = call_noalloc(torch, f, hid, gam, W, cuda_tensor(b.token_ids), 1.0, b.eps)
    assert code == 0 and status == 0
    # beyond the fixed scratch: rejected with nothing enqueued
    big_T = 20000
    assert tim.logprob_workspace_size(big_T, 256, 3000) > SCRATCH_BYTES
    big = torch.zeros(big_T, 256, dtype=torch.bfloat16, device="cuda")
    big_ids = torch.zeros(big_T, dtype=torch.int32, device="cuda")
    code, _, _ = call_noalloc(torch, f, big, gam, W, big_ids, 1.0, b.eps)
    assert code == tim.STATUS["TIM_ERR_WORKSPACE"]
    # the binding's thin wrapper gives the same bits as the direct call
    ids = cuda_tensor(b.token_ids)
    _, got, _ = call_noalloc(torch, f, hid, gam, W, ids, 1.0, b.eps)
    out = (torch.empty(40, device="cuda"), torch.empty(40, device="cuda"),
           torch.empty(40, dtype=torch.int32, device="cuda"))
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    tim.logprob_noalloc(hid, gam, W, ids, 1.0, b.eps, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert all(x.cpu().numpy().tobytes() == y.tobytes() for x, y in zip(out, got))
