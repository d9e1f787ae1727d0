"""The N > 1 benchmark plumbing on CPU ranks (gloo, world size 2): every rank
scores its own batch (weak scaling), the time reported is the max over ranks,
and the barrier joins; no data-path collective is involved."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), TIM_BENCH_BACKEND="gloo")
    import bench
    r, w, local, dist = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(dist, None)
    t = bench.max_over_ranks(10.0 + rank, dist, None)
    # each rank draws its own batch from a rank-keyed seed (weak scaling)
    import synth
    b = synth.make_custom(T=8, d=64, V=32, seed=rank, tag="mr")
    q.put((rank, t, b.hidden_gen.tobytes()))
    dist.destroy_process_group()


def test_two_ranks_gloo():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[1] for o in out] == [11.0, 11.0]      # max over ranks
    assert out[0][2] != out[1][2]                    # distinct batches per rank


def _failing_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), TIM_BENCH_BACKEND="gloo")
    import bench
    _, _, _, dist = bench.dist_setup(world, timeout_s=5.0)
    if rank == 1:
        q.put((rank, "left"))
        q.close()
        q.join_thread()        # flush the message before the abrupt exit
        os._exit(3)            # this rank fails between steps: it never reaches the barrier
    try:
        bench.barrier(dist, None)
        q.put((rank, "no error"))
    except Exception as e:      # the surviving rank learns of it from the timeout
        q.put((rank, "error: " + type(e).__name__))


def test_rank_failure_is_reported_not_hung():
    """A rank that dies between steps: the other rank's next collective raises within the
    process-group timeout instead of hanging (host-side failure detection, gloo)."""
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_failing_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert out[1] == "left" and procs[1].exitcode == 3
    assert out[0].startswith("error"), out[0]
