"""GPU parity of dspark_topk against the oracle (bit-exact indices, ids and values)."""
import numpy as np
import pytest
import torch

import dspark_inputs as di
from oracle import draft as od
from tests.gpu_util import as_f32, dev, host

pytestmark = pytest.mark.gpu


def run_topk(rows_f32_or_bits, B, K, **kw):
    import dspark_draft_selection_gb300 as ds
    x = dev(rows_f32_or_bits)
    cd, ct, cv, st = ds.dspark_topk(x, B, K, **kw)
    torch.cuda.synchronize()
    return host(cd), host(ct), host(cv), ds.read_status(st)


def oracle_topk(s, K, d2t=None, mult=1.0, softcap=0.0, rows=None):
    rows = range(s.shape[0]) if rows is None else rows
    out = []
    for i in rows:
        idx, val = od.topk_row(od.row_transform(s[i], mult, softcap), K)
        out.append((idx, od.d2t_map(idx, d2t), val))
    return out


def assert_same(got, want, rows=None, B=None):
    cd, ct, cv, _ = got
    cd = cd.reshape(-1, cd.shape[-1])
    ct = ct.reshape(-1, ct.shape[-1])
    cv = cv.reshape(-1, cv.shape[-1])
    rows = range(len(want)) if rows is None else rows
    for k, (i, (idx, tgt, val)) in enumerate(zip(rows, want)):
        assert np.array_equal(cd[i], idx), f"row {i}"
        assert np.array_equal(ct[i], tgt), f"row {i}"
        assert np.array_equal(cv[i], val), f"row {i}"


def test_tiny_fp32_config():
    w = di.config1()
    got = run_topk(w["logits"], 7, 8)
    assert got[3] == 0
    assert_same(got, oracle_topk(w["logits"], 8))


@pytest.mark.parametrize("V,K", [(151936, 64), (10007, 64), (48, 64), (3000, 5), (70001, 33), (1, 64), (257, 64)])
def test_shapes_and_ragged_tails(V, K):
    w = di.lattice_workload(20, R=2, B=3, V_d=V, K=K, rank=8)
    got = run_topk(w["logits"], 3, K)
    assert got[3] == 0
    assert_same(got, oracle_topk(as_f32(w["logits"]), K))


def test_unaligned_rows_and_packed_row_start():
    rng = np.random.default_rng(3)
    V, ld, B, R = 30011, 30017, 4, 3
    full = di.normal(di.generator(21, 0), (40, ld), 2.0, "bf16")
    row_start = np.array([1, 11, 27], dtype=np.int64)        # blocks after context rows
    import dspark_draft_selection_gb300 as ds
    x = dev(full)
    cd, ct, cv, st = ds.dspark_topk(x, B, 64, R=R, V_d=V, row_start=dev(row_start))
    torch.cuda.synchronize()
    s = as_f32(full)
    rows = [int(row_start[r]) + j for r in range(R) for j in range(B)]
    want = oracle_topk(s[:, :V], 64, rows=rows)
    assert_same((host(cd), host(ct), host(cv), 0), want)


def test_ties_signed_zero_constant_and_infinite_rows():
    rng = np.random.default_rng(5)
    V = 9000
    s = np.round(rng.standard_normal((8, V)) * 2).astype(np.float32)   # heavy ties
    s[1] = 0.0                                                          # constant row: survivor flood
    s[2, rng.random(V) < 0.5] = -0.0
    s[2, rng.random(V) < 0.3] = 0.0
    s[3] = -np.inf
    s[4] = np.round(s[4] / 4)                                          # very few distinct values
    s[5, :] = 7.0
    s[5, 100:200] = 8.0                                                # 100 equal maxima
    bits = di.f32_to_bf16_bits(s)
    for data in (s, bits):
        got = run_topk(data, 4, 64)
        assert got[3] == 0
        assert_same(got, oracle_topk(as_f32(data), 64))


def test_output_multiplier_is_bit_exact():
    w = di.lattice_workload(22, R=2, B=3, V_d=40000, K=64, rank=8)
    got = run_topk(w["logits"], 3, 64, mult=0.37)
    assert_same(got, oracle_topk(as_f32(w["logits"]), 64, mult=0.37))


def test_soft_cap_within_tanh_rounding():
    w = di.lattice_workload(23, R=1, B=4, V_d=50000, K=64, rank=8)
    s = as_f32(w["logits"])
    cd, ct, cv, stt = run_topk(w["logits"], 4, 64, softcap=3.0)
    for i in range(4):
        x = od.row_transform(s[i], 1.0, 3.0)
        idx, val = od.topk_row(x, 64)
        np.testing.assert_allclose(cv[0, i], val, rtol=4e-7, atol=0)
        # the two tanh implementations may round one ulp apart: membership may only differ at the boundary
        kth = val[-1]
        diff = set(cd[0, i]) ^ set(idx)
        assert all(abs(x[j] - kth) <= 4e-7 * abs(kth) for j in diff)


def test_pruned_vocabulary_d2t_map_and_range_error():
    w = di.lattice_workload(24, R=2, B=3, V_d=5000, V_t=12000, K=64, rank=8, pruned=True)
    got = run_topk(w["logits"], 3, 64, d2t=dev(w["d2t"]), V_t=12000)
    assert got[3] == 0
    assert_same(got, oracle_topk(as_f32(w["logits"]), 64, d2t=w["d2t"]))
    bad = w["d2t"].copy()
    s = as_f32(w["logits"])
    top = int(np.argmax(s[0]))
    bad[top] = 12000 - top                                    # the top candidate maps out of range
    cd, ct, cv, st = run_topk(w["logits"], 3, 64, d2t=dev(bad), V_t=12000)
    assert st == 2 and ct[0, 0, 0] == -1


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_full_size_configs(cfg):
    w = di.CONFIGS[cfg]()
    kw = dict(d2t=dev(w["d2t"]), V_t=w["V_t"]) if w["d2t"] is not None else {}
    got = run_topk(w["logits"], w["B"], w["K"], **kw)
    assert got[3] == 0
    s = as_f32(w["logits"])
    nrows = s.shape[0]
    rows = range(nrows) if nrows <= 256 else np.random.default_rng(cfg).choice(nrows, 48, replace=False)
    assert_same(got, oracle_topk(s, w["K"], d2t=w["d2t"], rows=rows), rows=rows)


@pytest.mark.parametrize("dtype,V", [("bf16", 400000), ("f32", 200000)])
def test_long_rows(dtype, V):
    # long rows: 98 vectors per thread, the tracked maxima and the bound span the whole row
    w = di.lattice_workload(25, R=1, B=3, V_d=V, K=64, rank=8, dtype=dtype, peak=8.0)
    got = run_topk(w["logits"], 3, 64)
    assert got[3] == 0
    assert_same(got, oracle_topk(as_f32(w["logits"]), 64))


def test_long_rows_with_ties_and_constant_rows():
    rng = np.random.default_rng(6)
    V = 400000
    s = np.round(rng.standard_normal((4, V)) * 2).astype(np.float32)
    s[1] = 3.0
    s[2] = -np.inf
    bits = di.f32_to_bf16_bits(s)
    got = run_topk(bits, 4, 64)
    assert got[3] == 0
    assert_same(got, oracle_topk(as_f32(bits), 64))


def test_many_rows_per_block_with_flooded_rows():
    # a batch of the Qwen3-4B shape in which some rows flood the candidate list with ties at the
    # bound (constant, all -inf, few distinct values) and take the exact cut
    w = di.lattice_workload(26, R=32, B=7, V_d=151936, K=64, rank=8, peak=8.0)
    s = as_f32(w["logits"]).copy()
    rng = np.random.default_rng(7)
    s[5] = 1.5
    s[77] = -np.inf
    s[150] = np.round(s[150] / 8)
    s[223, rng.random(151936) < 0.5] = -0.0
    bits = di.f32_to_bf16_bits(s)
    got = run_topk(bits, 7, 64)
    assert got[3] == 0
    rows = [0, 5, 6, 77, 78, 113, 150, 151, 200, 223]
    assert_same(got, oracle_topk(as_f32(bits), 64, rows=rows), rows=rows)


def test_small_k_and_single_part_rows_in_bulk():
    w = di.lattice_workload(27, R=200, B=3, V_d=4099, K=3, rank=8)
    got = run_topk(w["logits"], 3, 3)
    assert got[3] == 0
    rows = list(range(0, 600, 37)) + [599]
    assert_same(got, oracle_topk(as_f32(w["logits"]), 3, rows=rows), rows=rows)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rising_falling_and_late_peak_rows(dtype):
    # a rising row (the bound comes from the last batch of every thread), a falling row (from the
    # first), the peak in the scalar tail, and a rising row with long runs of ties (the list
    # overflows and takes the exact cut)
    V = 100003
    s = np.zeros((4, V), dtype=np.float32)
    s[0] = np.arange(V, dtype=np.float32) / 64.0
    s[1] = -np.arange(V, dtype=np.float32) / 64.0
    s[2] = di.normal(di.generator(28, 0), (1, V), 2.0, "f32")[0]
    s[2, V - 1] = 50.0
    s[2, V - 2] = 49.0
    s[3] = np.round(s[0] / 512.0)                                      # rising with long runs of ties
    data = s if dtype == "f32" else di.f32_to_bf16_bits(s)
    got = run_topk(data, 4, 64)
    assert got[3] == 0
    assert_same(got, oracle_topk(as_f32(data), 64))


@pytest.mark.parametrize("mult,cap", [(1.0, 0.0), (0.37, 0.0), (1.0, 30.0), (0.5, 30.0)])
def test_no_head_argmax_fast_path(mult, cap):
    # no Markov head: the output multiplier and soft cap, then the argmax of full-vocabulary rows,
    # is the Top-K with K = 1 (one streaming pass; the bound is the row maximum)
    w = di.lattice_workload(29, R=8, B=7, V_d=151936, K=64, rank=8, peak=8.0)
    s = as_f32(w["logits"])
    cd, ct, cv, st = run_topk(w["logits"], 7, 1, mult=mult, softcap=cap)
    assert st == 0
    cd, cv = cd.reshape(-1), cv.reshape(-1)
    for i in range(s.shape[0]):
        x = od.row_transform(s[i], mult, cap)
        idx, val = od.topk_row(x, 1)
        if cap == 0.0:
            assert cd[i] == idx[0] and cv[i] == val[0], f"row {i}"
        else:                                              # CUDA's tanhf against tanh in double
            np.testing.assert_allclose(cv[i], val[0], rtol=4e-7, atol=0)
            assert cd[i] == idx[0] or abs(x[cd[i]] - val[0]) <= 4e-7 * abs(val[0]), f"row {i}"
