"""Every entry point called from two host threads at once on one device (each thread with its own
stream and buffers) gives the same results as a single-threaded run: the library keeps no per-call
state, and its per-device kernel configuration is set up under a lock."""
import threading

import numpy as np
import pytest
import torch

import dspark_inputs as di
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


def _all_entry_points(ds, w, v, stream):
    out = []
    with torch.cuda.stream(stream):
        logits = dev(w["logits"])
        cd, ct, cv, st = ds.dspark_topk(logits, w["B"], w["K"], stream=stream)
        prev, E, W = dev(w["prev"]), dev(w["E"]), dev(w["W"])
        trans, gate, _ = ds.dspark_lattice_score(ct, prev, E, W, stream=stream)
        ch = ds.dspark_chain_select(cv, trans, ct, "maxsum", stream=stream)
        lc = ds.dspark_lattice_chain(cv, ct, prev, E, W, "walk", stream=stream)
        seed, step = dev(v["seed"]), dev(v["step"])
        smp = ds.dspark_sample(dev(v["logits"]), v["B"], temperature=0.9, top_p=0.9, seed=seed, step=step,
                               stream=stream)
        q = ds.dense_record(v["R"] * v["B"], v["V_d"])
        dw = ds.dspark_dense_walk(dev(v["logits"]), v["B"], dev(v["prev"]), dev(v["E"]), dev(v["W"]),
                                  temperature=1.0, seed=seed, step=step, q=q, stream=stream)
        n = torch.full((v["R"],), v["B"], dtype=torch.int32, device="cuda")
        vf = ds.dspark_verify(dev(v["target"]), v["B"], dw[0], n, q, vseed=dev(v["vseed"]), step=step, stream=stream)
        d2 = ds.dspark_d2t_check(torch.zeros(100, dtype=torch.int64, device="cuda"), 100, stream=stream)
        stream.synchronize()
        for x in (cd, ct, cv, trans, gate) + tuple(ch[:3]) + tuple(lc[:3]) + tuple(smp[:2]) + tuple(dw[:2]) + \
                tuple(vf[:3]):
            out.append(x.cpu())
        for s in (st, ch[-1], lc[-1], smp[-1], dw[-1], vf[-1], d2):
            out.append(ds.read_status(s))
    return out


def test_two_host_threads_every_entry_point():
    import dspark_draft_selection_gb300 as ds
    w = di.lattice_workload(62, R=4, B=5, V_d=20000, K=64, rank=256, peak=8.0)
    v = di.config5(R=3, V=6000)
    ref = _all_entry_points(ds, w, v, torch.cuda.Stream())
    results, errors = [None, None], []

    def run(i):
        try:
            torch.cuda.set_device(0)
            res = None
            for _ in range(5):
                res = _all_entry_points(ds, w, v, torch.cuda.Stream())
            results[i] = res
        except Exception as e:  # surfaced below
            errors.append(repr(e))

    th = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    for res in results:
        assert len(res) == len(ref)
        for a, b in zip(ref, res):
            if isinstance(a, int):
                assert a == 0 and b == 0
            else:
                assert torch.equal(a, b)
