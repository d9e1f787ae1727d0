"""Host side of the vocabulary-parallel path (CPU): the shard layout tiles the vocabulary in
whole 256-column tiles along the 16 fixed merge ranges, and the record all-gather returns
every rank's records in rank order (gloo, world size 2)."""
import os
import socket

import pytest


@pytest.fixture(scope="module")
def tim():
    import __graft_entry__
    __graft_entry__.build()
    import rollout_logprob_consistency_gb300 as tim
    return tim


@pytest.mark.parametrize("V", [1, 255, 256, 1000, 4099, 5000, 151936])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_shard_layout(tim, V, G):
    n_tiles = (V + 255) // 256
    per = (n_tiles + 15) // 16
    L = 16 // G
    pos = 0
    for g in range(G):
        v0, n = tim.vocab_shard(V, G, g)
        if n:
            assert v0 == pos and v0 % 256 == 0
            assert v0 == g * L * per * 256                  # aligned to the merge ranges
            pos = v0 + n
        else:
            assert g * L * per >= n_tiles                     # only trailing shards are empty
    assert pos == V


def test_shard_arguments(tim):
    with pytest.raises(tim.TimError):
        tim.vocab_shard(1000, 3, 0)
    with pytest.raises(tim.TimError):
        tim.vocab_shard(1000, 4, 4)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    from rollout_logprob_consistency_gb300 import binding
    dist.init_process_group("gloo", rank=rank, world_size=world)
    T = 5
    rec = torch.full((T, 4), float(rank)) + torch.arange(T, dtype=torch.float32)[:, None]
    tgt = torch.full((T,), 10.0 * rank)
    recs, tgts = binding.gather_shard_records(rec, tgt)
    q.put((rank, recs.numpy().tolist(), tgts.numpy().tolist()))
    dist.destroy_process_group()


def test_gather_in_rank_order():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    outs = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, recs, tgts in outs:
        assert [r[0][0] for r in recs] == [0.0, 1.0]
        assert tgts[0][0] == 0.0 and tgts[1][0] == 10.0
    assert outs[0][1] == outs[1][1]
