"""Multi-rank host logic of the bench, on CPU with two gloo ranks.

Block drafting shards by request: every rank drafts its own batch with no collective on the data
path, so what a multi-GPU run adds is host logic only: disjoint per-rank inputs, the slowest rank's
time and the whole-job throughput. These run here as two processes on the gloo backend.
"""
import multiprocessing as mp
import os
import socket
import sys
import traceback

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out) -> None:
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                          WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
        sys.path.insert(0, ROOT)
        import torch
        import torch.distributed as dist

        import bench
        import dspark_inputs as di
        dist.init_process_group("gloo", rank=rank, world_size=world)
        assert bench.dist_env() == (world, rank, rank)
        nsets = 4
        cids = [bench.set_cid(rank, s, nsets) for s in range(nsets)]
        every = [None] * world
        dist.all_gather_object(every, cids)
        # the rank's first batch really is a different draw of the same shape
        w = di.lattice_workload(cids[0], R=2, B=3, V_d=64, K=8, rank=16, peak=8.0)
        heads = [None] * world
        dist.all_gather_object(heads, (w["logits"][:, :8].tobytes(), w["prev"].tolist()))
        slow = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
        dist.barrier()
        out.put((rank, every, heads, slow, None))
        dist.destroy_process_group()
    except Exception:  # report, do not hang the other rank's queue read
        out.put((rank, None, None, None, traceback.format_exc()))


@pytest.mark.timeout(300)
def test_two_gloo_ranks_disjoint_inputs_and_slowest_rank_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, every, heads, slow, err = q.get(timeout=240)
        res[rank] = (every, heads, slow, err)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r][3] is None, res[r][3]
    every, heads, _, _ = res[0]
    assert every == res[1][0]
    assert every[0][0] == 2                              # rank 0's first set is the named workload
    assert not set(every[0]) & set(every[1])             # no batch drafted twice
    assert heads[0] != heads[1]
    assert res[0][2] == res[1][2] == 15.0                 # both ranks report the slowest time


def test_whole_job_throughput_and_single_rank_defaults():
    sys.path.insert(0, ROOT)
    import bench
    # two ranks x 32 requests x 100 steps in 50 ms
    assert bench.job_blocks_per_s(2, 32, 100, 50.0) == pytest.approx(128000.0)
    assert bench.max_over_ranks(3.5, None) == 3.5        # no process group: the rank's own time
    grid = [bench.set_cid(r, s, 4) for r in range(8) for s in range(4)]
    assert grid[0] == 2 and len(set(grid)) == len(grid)  # eight ranks, four sets each: all distinct


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class A:
        steps, warmup = 1, 3
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
