"""GPU parity of dspark_dense_walk against the oracle's dense Markov walk.

Every position is checked on its own: the oracle is teacher-forced with the GPU's previous
tokens. The biased row v = s + gamma * tau is float32 on both sides, but tau is a float32
tensor-core sum on the GPU and a float64 dot in the oracle, so v may differ by a few float32
ulps; a decision may then differ only where the oracle's margin is inside that rounding: the
top-2 gap for greedy positions, the distance of u * W_kept to a running-sum boundary (relative
to W_kept) for sampled ones.
"""
import numpy as np
import pytest
import torch

import dspark_inputs as di
from oracle import draft as od
from oracle import walk as ow
from oracle.sampling import draw_margin
from tests.gpu_util import as_f32, dev, host

pytestmark = pytest.mark.gpu

ULPS = 8


def run_gpu(w, T, top_p, gate=False, mult=1.0, record=True):
    import dspark_draft_selection_gb300 as ds
    R, B, V = w["R"], w["B"], w["V_d"]
    q = ds.dense_record(R * B, V) if record else None
    kw = {}
    if w["d2t"] is not None:
        kw["d2t"] = dev(w["d2t"])
    if gate:
        kw["hidden"], kw["g"] = dev(w["hidden"]), dev(w["g"])
    tgt, idx, st = ds.dspark_dense_walk(dev(w["logits"]), B, dev(w["prev"]), dev(w["E"]), dev(w["W"]),
                                        temperature=T, top_p=top_p, seed=dev(w["seed"]), step=dev(w["step"]),
                                        mult=mult, q=q, **kw)
    torch.cuda.synchronize()
    return host(tgt), host(idx), ds.read_status(st), (tuple(host(t) for t in q) if q is not None else None)


def check(w, T, top_p, gate=False, mult=1.0, reqs=None, record=True):
    tgt, idx, st, rec = run_gpu(w, T, top_p, gate, mult, record)
    assert st == 0
    R, B, V = w["R"], w["B"], w["V_d"]
    E, W = as_f32(w["E"]), as_f32(w["W"])
    m = od.d2t_map(np.arange(V), w["d2t"])
    Wm64 = W.astype(np.float64)[m]
    s = as_f32(w["logits"])
    amb = 0
    for r in (range(R) if reqs is None else reqs):
        gam = [od.gate(as_f32(w["hidden"])[r * B + j], as_f32(w["g"])) for j in range(B)] if gate else None
        res = ow.dense_walk_request(s[r * B:(r + 1) * B], int(w["prev"][r]), E, W, d2t=w["d2t"], gammas=gam,
                                    mult=mult, T=T, top_p=top_p, seed=int(w["seed"][r]), step=int(w["step"][r]),
                                    forced_prev=tgt[r], Wm64=Wm64)
        for j in range(B):
            assert tgt[r, j] == m[idx[r, j]]
            orec = res["records"][j]
            if record and T > 0:
                z = rec[0][r * B + j]
                tol = ULPS * np.spacing(np.abs(orec["z"]).astype(np.float32)) + 1e-6
                assert np.all(np.abs(z - orec["z"]) <= tol)
            if idx[r, j] == res["draft_idx"][j]:
                continue
            amb += 1
            if T > 0:
                assert draw_margin(orec["w"], orec["kept"], res["u"][j]) < 4e-7, (r, j)
            else:
                v = res["rows"][j].astype(np.float64)
                gap = v[res["draft_idx"][j]] - v[idx[r, j]]
                assert gap <= ULPS * np.spacing(np.float32(abs(v.max()))), (r, j, gap)
    return amb


@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.7, 0.9), (0.0, 1.0)])
def test_dense_walk_small(T, top_p):
    w = di.lattice_workload(70, R=3, B=5, V_d=20000, K=0, rank=64, with_seeds=True, head_sigma=0.3)
    assert check(w, T, top_p) <= 1


def test_dense_walk_gated_rank256_transform():
    w = di.lattice_workload(71, R=5, B=4, V_d=30011, K=0, rank=256, with_seeds=True, H=384, head_sigma=0.2)
    assert check(w, 0.9, 1.0, gate=True, mult=0.8) <= 1


def test_dense_walk_pruned_vocabulary():
    w = di.lattice_workload(72, R=3, B=4, V_d=6000, V_t=15000, K=0, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.3)
    assert check(w, 1.0, 1.0) <= 1
    assert check(w, 0.0, 1.0) <= 1


def test_dense_walk_without_record_and_many_requests():
    w = di.lattice_workload(73, R=130, B=2, V_d=3000, K=0, rank=64, with_seeds=True, head_sigma=0.3)
    assert check(w, 1.0, 1.0, record=False, reqs=[0, 64, 127, 128, 129]) <= 1


def test_dense_walk_full_size_config():
    # the benchmarked shape: 64 requests (MMA N = 64), 15 positions, V = 151,936; requests from the
    # first and the last 32-column epilogue chunks
    w = di.config5()
    assert check(w, w["temperature"], w["top_p"], reqs=[0, 17, 31, 32, 48, 63]) <= 1


def test_dense_walk_full_size_greedy():
    w = di.config5()
    assert check(w, 0.0, 1.0, reqs=[5, 40, 63], record=False) <= 1
