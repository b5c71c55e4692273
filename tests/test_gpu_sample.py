"""GPU parity of dspark_sample (full-row multinomial drafting and its proposal record).

The weights are the same float32 function on both sides, so draws must agree exactly; the only
admissible difference is a draw whose target u * W_kept lies within rounding (1e-12 of W_kept)
of a running-sum boundary in the oracle, where the double sums' association order decides.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import dspark_inputs as di
from oracle import draft as od
from oracle.philox import uniform
from oracle.sampling import draw_margin, sample_row
from tests.gpu_util import as_f32, dev, host

pytestmark = pytest.mark.gpu


def gpu_sample(logits, B, T, top_p, seed, step, record=None, cap=None, **kw):
    import dspark_draft_selection_gb300 as ds
    x = dev(logits)
    rows = x.shape[0]
    R = rows // B
    q = None
    if record == "dense":
        q = ds.dense_record(rows, x.shape[1])
    elif record == "sparse":
        q = (torch.full((rows, cap), -1, dtype=torch.int32, device="cuda"),
             torch.zeros((rows, cap), dtype=torch.float32, device="cuda"),
             torch.zeros((rows,), dtype=torch.int32, device="cuda"))
    tgt, idx, st = ds.dspark_sample(x, B, temperature=T, top_p=top_p, seed=dev(seed), step=dev(step), q=q, **kw)
    torch.cuda.synchronize()
    return host(tgt), host(idx), ds.read_status(st), (tuple(host(t) for t in q) if q is not None else None)


def seeds(R, cid=60):
    g = di.generator(cid, di.S_SEEDS)
    return (g.integers(0, 2**63, size=R, dtype=np.int64).astype(np.uint64),
            g.integers(0, 2**40, size=R, dtype=np.int64).astype(np.uint64))


def check_rows(s, B, T, top_p, seed, step, got_idx, d2t=None, rec=None, record=None, mult=1.0, softcap=0.0,
               min_p=0.0):
    amb = 0
    R = s.shape[0] // B
    for r in range(R):
        for j in range(B):
            row = od.row_transform(s[r * B + j], mult, softcap)
            u = float(uniform(seed[r], step[r], j, 0)) if T > 0 else 0.0
            tok, orec = sample_row(row, T, top_p, u, min_p)
            gi = int(got_idx[r, j])
            if gi != tok:
                assert T > 0 and draw_margin(orec["w"], orec["kept"], u) < 1e-12, (r, j, gi, tok)
                amb += 1
                continue
            i = r * B + j
            if record == "dense" and T > 0:
                z, zmax, wsum, wcut, icut = rec
                assert np.array_equal(z[i], orec["z"])
                assert zmax[i] == orec["zmax"]
                assert abs(wsum[i] - orec["wsum"]) <= 1e-12 * orec["wsum"]
                assert wcut[i] == orec["w_cut"] and icut[i] == orec["i_cut"]
            if record == "sparse" and T > 0:
                ids, qp, qn = rec
                n = len(orec["kept"])
                assert qn[i] == n
                assert np.array_equal(ids[i, :n], od.d2t_map(orec["kept"], d2t))
                np.testing.assert_allclose(qp[i, :n], orec["q"], rtol=2e-7, atol=0)
    return amb


@pytest.mark.parametrize("V,T,top_p", [(1000, 0.7, 1.0), (151936, 1.0, 1.0), (30011, 0.8, 0.9), (5000, 1.3, 0.5),
                                       (248320, 0.8, 0.95), (37, 1.0, 0.3)])
def test_draws_and_dense_record(V, T, top_p):
    R, B = 3, 4
    w = di.lattice_workload(61 + V % 97, R=R, B=B, V_d=V, K=1, rank=8)
    seed, step = seeds(R)
    tgt, idx, st, rec = gpu_sample(w["logits"], B, T, top_p, seed, step, record="dense")
    assert st == 0
    assert np.array_equal(tgt, idx)
    assert check_rows(as_f32(w["logits"]), B, T, top_p, seed, step, idx, rec=rec, record="dense") == 0


def test_sparse_record_with_pruned_vocabulary():
    R, B = 2, 5
    w = di.lattice_workload(62, R=R, B=B, V_d=4000, V_t=9000, K=1, rank=8, pruned=True)
    seed, step = seeds(R)
    tgt, idx, st, rec = gpu_sample(w["logits"], B, 0.6, 0.8, seed, step, record="sparse", cap=4000,
                                   d2t=dev(w["d2t"]), V_t=9000)
    assert st == 0
    assert np.array_equal(tgt, od.d2t_map(idx.ravel(), w["d2t"]).reshape(idx.shape))
    assert check_rows(as_f32(w["logits"]), B, 0.6, 0.8, seed, step, idx, d2t=w["d2t"], rec=rec, record="sparse") == 0


def test_large_flat_nucleus_takes_the_bisection_path():
    R, B = 1, 3
    w = di.lattice_workload(63, R=R, B=B, V_d=60000, K=1, rank=8, logit_sigma=0.05)
    seed, step = seeds(R)
    tgt, idx, st, rec = gpu_sample(w["logits"], B, 1.0, 0.9, seed, step, record="dense")
    assert st == 0
    assert check_rows(as_f32(w["logits"]), B, 1.0, 0.9, seed, step, idx, rec=rec, record="dense") == 0


def test_greedy_ties_unaligned_rows_and_transform():
    rng = np.random.default_rng(2)
    V, ld = 7001, 7003
    full = np.round(rng.standard_normal((6, ld)) * 2).astype(np.float32)
    full[1, :] = 3.0
    seed, step = seeds(2)
    import dspark_draft_selection_gb300 as ds
    x = dev(full)
    tgt, idx, st = ds.dspark_sample(x, 3, V_d=V, temperature=0.0, seed=dev(seed), step=dev(step))
    torch.cuda.synchronize()
    for i in range(6):
        assert host(idx).ravel()[i] == int(np.argmax(full[i, :V]))
    bits = di.f32_to_bf16_bits((rng.standard_normal((6, ld)) * 2).astype(np.float32))
    tgt, idx, st, rec = gpu_sample(bits, 3, 0.9, 0.95, seed, step, V_d=V, mult=0.5)
    assert st == 0
    assert check_rows(as_f32(bits)[:, :V], 3, 0.9, 0.95, seed, step, idx, mult=0.5) == 0


def test_non_finite_row_reports_status():
    s = np.full((2, 1000), -np.inf, dtype=np.float32)
    s[1, 5] = 0.0
    seed, step = seeds(1)
    tgt, idx, st, _ = gpu_sample(s, 2, 1.0, 1.0, seed, step)
    assert st == 5 and idx[0, 0] == -1 and idx[0, 1] == 5


def test_gpu_draws_follow_q_chi_square():
    V, R = 12, 20000
    rng = np.random.default_rng(3)
    row = (rng.standard_normal(V) * 1.5).astype(np.float32)
    logits = np.tile(row, (R, 1))
    seed = np.full(R, 77, dtype=np.uint64)
    step = np.arange(R, dtype=np.uint64)
    tgt, idx, st, _ = gpu_sample(logits, 1, 0.9, 1.0, seed, step)
    assert st == 0
    _, rec = sample_row(row, 0.9, 1.0, 0.5)
    q = np.zeros(V)
    q[rec["kept"]] = rec["w"][rec["kept"]] / rec["wsum"]
    counts = np.bincount(idx.ravel(), minlength=V)
    exp = q * R
    keep = exp > 5
    stat = np.sum((counts[keep] - exp[keep]) ** 2 / exp[keep])
    assert stat < stats.chi2.ppf(0.999, keep.sum() - 1)


def test_dense_walk_shaped_rows_full_size():
    w = di.config5(R=4)
    B = w["B"]
    tgt, idx, st, rec = gpu_sample(w["logits"], B, 1.0, 1.0, w["seed"], w["step"], record="dense")
    assert st == 0
    assert check_rows(as_f32(w["logits"]), B, 1.0, 1.0, w["seed"], w["step"], idx, rec=rec, record="dense") <= 1


@pytest.mark.parametrize("f32", [False, True])
def test_weight_scratch_and_recomputed_weights_agree(f32):
    """The nucleus passes read the weights from the workspace when it is large enough and recompute
    them otherwise: both give the same draws and records (unaligned rows, head and tail elements)."""
    import dspark_draft_selection_gb300 as ds
    R, B, V = 3, 4, 30011
    w = di.lattice_workload(64, R=R, B=B, V_d=V, K=1, rank=8)
    seed, step = seeds(R)
    x = dev(w["logits"])
    if f32:
        x = x.float()
    outs = []
    for ws in (None, torch.empty(1024, dtype=torch.uint8, device="cuda")):   # large enough / too small
        q = ds.dense_record(R * B, V)
        tgt, idx, st = ds.dspark_sample(x, B, temperature=0.8, top_p=0.9, seed=dev(seed), step=dev(step), q=q, ws=ws)
        torch.cuda.synchronize()
        assert ds.read_status(st) == 0
        outs.append((host(tgt), host(idx)) + tuple(host(t) for t in q))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    assert check_rows(host(x.float()), B, 0.8, 0.9, seed, step, outs[0][1], rec=outs[0][2:], record="dense") == 0
