"""Failure detection without a GPU fault: every wait of a tensor-core tile is bounded, and a wait
that runs out is reported as DSPARK_ETIMEOUT with the tile's results left unwritten. The test hook
sets the first wait's limit to 0 polls, so the timeout path runs at once; the kernel still waits for
its MMAs in flight (with the full limit) before it releases tensor memory, so nothing is left
running on the GPU, and the next call with the default limit succeeds."""
import numpy as np
import pytest
import torch

import dspark_inputs as di
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

ETIMEOUT = 6


@pytest.fixture
def ds():
    import dspark_draft_selection_gb300 as ds
    yield ds
    ds.dspark_test_set_first_wait_polls(0xFFFFFFFF)


def test_lattice_wait_that_runs_out_reports_timeout(ds):
    w = di.lattice_workload(60, R=3, B=4, V_d=5000, K=64, rank=256)
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), w["B"], 64)
    prev, E, W = dev(w["prev"]), dev(w["E"]), dev(w["W"])
    trans = torch.full((3, 4, 64, 64), 7.5, dtype=torch.float32, device="cuda")
    ds.dspark_test_set_first_wait_polls(0)
    _, _, st = ds.dspark_lattice_score(ct, prev, E, W, out=(trans, torch.empty((3, 4), device="cuda")))
    rank_, tgt, score, st2 = ds.dspark_lattice_chain(cv, ct, prev, E, W, "maxsum")
    torch.cuda.synchronize()
    assert ds.read_status(st) == ETIMEOUT and ds.read_status(st2) == ETIMEOUT
    assert torch.all(trans == 7.5)                      # no tile was written
    ds.dspark_test_set_first_wait_polls(0xFFFFFFFF)
    _, _, st = ds.dspark_lattice_score(ct, prev, E, W, out=(trans, torch.empty((3, 4), device="cuda")))
    torch.cuda.synchronize()
    assert ds.read_status(st) == 0 and not torch.all(trans == 7.5)


def test_dense_walk_wait_that_runs_out_reports_timeout(ds):
    w = di.lattice_workload(61, R=3, B=3, V_d=4000, K=0, rank=64, with_seeds=True)
    R, B, V = 3, 3, 4000
    q = ds.dense_record(R * B, V)
    q[0].fill_(-3.25)
    ds.dspark_test_set_first_wait_polls(0)
    tgt, idx, st = ds.dspark_dense_walk(dev(w["logits"]), B, dev(w["prev"]), dev(w["E"]), dev(w["W"]),
                                        temperature=1.0, seed=dev(w["seed"]), step=dev(w["step"]), q=q)
    torch.cuda.synchronize()
    assert ds.read_status(st) == ETIMEOUT
    assert torch.all(q[0] == -3.25)                     # no z row of the record was written
    ds.dspark_test_set_first_wait_polls(0xFFFFFFFF)
    tgt, idx, st = ds.dspark_dense_walk(dev(w["logits"]), B, dev(w["prev"]), dev(w["E"]), dev(w["W"]),
                                        temperature=1.0, seed=dev(w["seed"]), step=dev(w["step"]), q=q)
    torch.cuda.synchronize()
    assert ds.read_status(st) == 0 and not torch.any(q[0] == -3.25)
