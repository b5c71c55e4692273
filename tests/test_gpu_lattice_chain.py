"""GPU parity of dspark_lattice_score and dspark_chain_select against the oracle.

Lattice values: float32 tensor-core (or FMA) accumulation against the oracle's float64 dot
products; the bound below is the float32 accumulation error of rank products plus the gate's
float32 partial dots, far inside the 1e-3 relative bar.
Chains: fed the same float32 inputs, the greedy and sampled walks must agree bit for bit (ids,
ranks, q). The max-sum chain is accumulated in float32 on the GPU and in float64 by the oracle:
chains must be equal unless the oracle's best and the GPU's chain score within the float32
rounding bound of each other, in which case the GPU chain must attain the maximum within it.
"""
import numpy as np
import pytest
import torch

import dspark_inputs as di
from oracle import draft as od
from oracle.fp32 import F32
from tests.gpu_util import as_f32, dev, host

pytestmark = pytest.mark.gpu


def gpu_draft(w, mode="maxsum", T=0.0, top_p=1.0, use_gate=True):
    import dspark_draft_selection_gb300 as ds
    kw = dict(d2t=dev(w["d2t"]), V_t=w["V_t"]) if w["d2t"] is not None else {}
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), w["B"], w["K"], **kw)
    hid = dev(w["hidden"]) if (use_gate and w["hidden"] is not None) else None
    g = dev(w["g"]) if hid is not None else None
    trans, gate, st2 = ds.dspark_lattice_score(ct, dev(w["prev"]), dev(w["E"]), dev(w["W"]), hidden=hid, g=g)
    out = ds.dspark_chain_select(cv, trans, ct, mode, temperature=T, top_p=top_p,
                                 seed=dev(w.get("seed")), step=dev(w.get("step")))
    torch.cuda.synchronize()
    for s in (st, st2, out[-1]):
        assert ds.read_status(s) == 0
    return dict(cand_draft=host(cd), cand_tgt=host(ct), cand_val=host(cv), trans=host(trans), gate=host(gate),
                chain=host(out[0]), chain_tgt=host(out[1]), score=host(out[2]),
                q=tuple(host(t) for t in out[3:6]) if len(out) > 4 else None)


def oracle_lattice(w, r, cand_tgt, use_gate=True):
    B = w["B"]
    E, W = as_f32(w["E"]), as_f32(w["W"])
    if use_gate and w["hidden"] is not None:
        h, g = as_f32(w["hidden"]), as_f32(w["g"])
        gam = [od.gate(h[r * B + j], g) for j in range(B)]
    else:
        gam = [1.0] * B
    return od.lattice_request(cand_tgt, int(w["prev"][r]), E, W, gam), np.array(gam)


def lattice_bound(w, r, cand_tgt):
    E, W = as_f32(w["E"]).astype(np.float64), as_f32(w["W"]).astype(np.float64)
    B = w["B"]
    rank = E.shape[1]
    absdot = np.zeros((B, cand_tgt.shape[1], cand_tgt.shape[1]))
    prev = int(w["prev"][r])
    absdot[0, 0] = np.abs(E[prev]) @ np.abs(W[cand_tgt[0]]).T
    for j in range(1, B):
        absdot[j] = np.abs(E[cand_tgt[j - 1]]) @ np.abs(W[cand_tgt[j]]).T
    return 1.01 * rank * 2.0 ** -24 * absdot + 1e-6 * np.abs(absdot)


def check_lattice(w, got, use_gate=True):
    for r in range(w["R"]):
        ref, gam = oracle_lattice(w, r, got["cand_tgt"][r], use_gate)
        np.testing.assert_allclose(got["gate"][r], gam, rtol=1e-6)
        err = np.abs(got["trans"][r] - ref)
        assert np.all(err <= lattice_bound(w, r, got["cand_tgt"][r])), r
        assert np.all(err <= 1e-3 * np.abs(ref) + 1e-5 * np.abs(ref).max())


@pytest.mark.parametrize("rank,K,H", [(256, 64, 0), (256, 48, 512), (64, 64, 0), (512, 17, 300), (128, 1, 0)])
def test_lattice_tensor_core_path(rank, K, H):
    w = di.lattice_workload(30 + rank + K, R=3, B=5, V_d=20000, K=K, rank=rank, H=H, head_sigma=0.3)
    check_lattice(w, gpu_draft(w))


def test_lattice_fma_path_tiny_config():
    w = di.config1()
    check_lattice(w, gpu_draft(w))


def test_lattice_pruned_table_zero_outside():
    w = di.lattice_workload(40, R=2, B=4, V_d=3000, V_t=9000, K=64, rank=64, pruned=True)
    got = gpu_draft(w)
    check_lattice(w, got)


def maxsum_tolerance(B, best, A):
    return 2.0 * B * (2.0 ** -23 * max(1.0, abs(best)) + 1e-6 * float(np.abs(A).max()))


def check_maxsum(got, r, u, A, B):
    chain, best = od.chain_maxsum(u, A)
    tol = maxsum_tolerance(B, best, A)
    if not np.array_equal(got["chain"][r], chain):
        # only a near-tie may differ, and the GPU's chain must then reach the maximum
        assert abs(od.chain_score(u, A, got["chain"][r]) - best) <= tol, r
        return 1
    assert abs(float(got["score"][r]) - best) <= 1e-3 * max(1.0, abs(best))
    return 0


def test_chain_maxsum_on_gpu_inputs_and_end_to_end():
    for cfg in (1, 2):
        w = di.CONFIGS[cfg]()
        got = gpu_draft(w)
        amb = 0
        for r in range(w["R"]):
            u = got["cand_val"][r]
            amb += check_maxsum(got, r, u, got["trans"][r].astype(np.float64), w["B"])
            # end to end from the raw inputs
            s = as_f32(w["logits"])[r * w["B"]:(r + 1) * w["B"]]
            res = od.select_request(s, w["K"], as_f32(w["E"]), as_f32(w["W"]), int(w["prev"][r]), "maxsum")
            assert np.array_equal(res["cand_draft"], got["cand_draft"][r])
            if not np.array_equal(res["chain"], got["chain"][r]):
                tol = maxsum_tolerance(w["B"], res["score"], res["A"])
                assert abs(od.chain_score(res["cand_val"], res["A"], got["chain"][r]) - res["score"]) <= tol
                amb += 1
        assert amb <= max(1, w["R"] // 16)


def test_chain_maxsum_strong_head_changes_chains():
    w = di.lattice_workload(41, R=8, B=7, V_d=4096, K=64, rank=64, head_sigma=0.35)
    got = gpu_draft(w)
    changed = 0
    for r in range(w["R"]):
        check_maxsum(got, r, got["cand_val"][r], got["trans"][r].astype(np.float64), w["B"])
        changed += int(np.any(got["chain"][r] != 0))
    assert changed >= 4


def test_chain_walk_bit_exact_on_gpu_inputs():
    w = di.lattice_workload(42, R=6, B=7, V_d=8192, K=64, rank=64, head_sigma=0.35)
    got = gpu_draft(w, mode="walk")
    for r in range(w["R"]):
        chain, score = od.chain_walk(got["cand_val"][r], got["trans"][r])
        assert np.array_equal(chain, got["chain"][r])
        assert abs(score - float(got["score"][r])) <= 1e-6 * max(1.0, abs(score))


@pytest.mark.parametrize("T,top_p", [(0.8, 0.95), (1.0, 1.0), (0.3, 0.5), (0.0, 1.0)])
def test_chain_sample_bit_exact_with_q_record(T, top_p):
    w = di.lattice_workload(43, R=5, B=15, V_d=3000, V_t=7000, K=64, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.3)
    got = gpu_draft(w, mode="sample", T=T, top_p=top_p)
    ids, qp, qn = got["q"]
    for r in range(w["R"]):
        u, A = got["cand_val"][r], got["trans"][r]
        chain, score, recs = od.chain_sample(u, A, got["cand_tgt"][r], T, top_p, int(w["seed"][r]), int(w["step"][r]))
        assert np.array_equal(chain, got["chain"][r]), r
        for j, rec in enumerate(recs):
            n = len(rec["kept"])
            assert qn[r, j] == n
            assert np.array_equal(ids[r, j, :n], rec["ids"])
            assert np.array_equal(qp[r, j, :n], rec["q"])


def test_chain_sample_pruned_config_full_size():
    w = di.config3()
    got = gpu_draft(w, mode="sample", T=w["temperature"], top_p=w["top_p"])
    ids, qp, qn = got["q"]
    for r in range(w["R"]):
        chain, score, recs = od.chain_sample(got["cand_val"][r], got["trans"][r], got["cand_tgt"][r],
                                             w["temperature"], w["top_p"], int(w["seed"][r]), int(w["step"][r]))
        assert np.array_equal(chain, got["chain"][r])
        assert np.array_equal(got["chain_tgt"][r], got["cand_tgt"][r][np.arange(w["B"]), chain])
        for j, rec in enumerate(recs):
            n = len(rec["kept"])
            assert qn[r, j] == n and np.array_equal(qp[r, j, :n], rec["q"])
        # every drafted token is in the draft vocabulary's image
        assert np.all(np.isin(got["chain_tgt"][r], w["subset"]))
    # the full-size pruned lattice against the oracle (rows gathered from the 248,100-row tables)
    for r in (0, 7, 15):
        check_lattice_rows(w, got, r)


def check_lattice_rows(w, got, r):
    """Lattice values of request r against the oracle, gathering only the table rows it uses."""
    B = w["B"]
    ct = got["cand_tgt"][r]
    ids = np.unique(np.concatenate([ct.ravel(), [int(w["prev"][r])]]))
    pos = {int(t): k for k, t in enumerate(ids)}
    E = as_f32(w["E"][ids]).astype(np.float64)
    W = as_f32(w["W"][ids]).astype(np.float64)
    loc = np.vectorize(lambda t: pos[int(t)])(ct)
    ref = od.lattice_request(loc, pos[int(w["prev"][r])], E, W, [1.0] * B)
    absdot = np.zeros_like(ref)
    absdot[0, 0] = np.abs(E[pos[int(w["prev"][r])]]) @ np.abs(W[loc[0]]).T
    for j in range(1, B):
        absdot[j] = np.abs(E[loc[j - 1]]) @ np.abs(W[loc[j]]).T
    bound = 1.01 * E.shape[1] * 2.0 ** -24 * absdot + 1e-6 * absdot
    err = np.abs(got["trans"][r] - ref)
    assert np.all(err <= bound), r
    assert np.all(err <= 1e-3 * np.abs(ref) + 1e-5 * np.abs(ref).max())


def test_gated_config_lattice_sampled_rows():
    w = di.config4()
    got = gpu_draft(w)
    rng = np.random.default_rng(4)
    for r in rng.choice(w["R"], 6, replace=False):
        ref, gam = oracle_lattice(w, r, got["cand_tgt"][r])
        np.testing.assert_allclose(got["gate"][r], gam, rtol=1e-6)
        err = np.abs(got["trans"][r] - ref)
        assert np.all(err <= 1e-3 * np.abs(ref) + 1e-5 * np.abs(ref).max())
        check_maxsum(got, r, got["cand_val"][r], got["trans"][r].astype(np.float64), w["B"])


def _two_call(ds, cv, ct, prev, E, W, mode, hidden=None, g=None):
    trans, gate, st = ds.dspark_lattice_score(ct, prev, E, W, hidden=hidden, g=g)
    rank_, tgt, score, st2 = ds.dspark_chain_select(cv, trans, ct, mode)
    torch.cuda.synchronize()
    assert ds.read_status(st) == 0 and ds.read_status(st2) == 0
    return trans, gate, rank_, tgt, score


@pytest.mark.parametrize("cfg,mode", [(2, "maxsum"), (2, "walk"), (4, "maxsum"), (1, "maxsum")])
def test_lattice_chain_fused_equals_two_calls(cfg, mode):
    # one cluster per request decides the chain on chip: same float32 operations as the two calls
    import dspark_draft_selection_gb300 as ds
    w = di.CONFIGS[cfg]()
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), w["B"], w["K"])
    hid = dev(w["hidden"]) if w["hidden"] is not None else None
    g = dev(w["g"]) if hid is not None else None
    prev, E, W = dev(w["prev"]), dev(w["E"]), dev(w["W"])
    trans, gate, rank_, tgt, score = _two_call(ds, cv, ct, prev, E, W, mode, hid, g)
    t2 = torch.full_like(trans, float("nan"))
    g2 = torch.full_like(gate, float("nan"))
    r2, tg2, sc2, st2 = ds.dspark_lattice_chain(cv, ct, prev, E, W, mode, hidden=hid, g=g, trans=t2, gate=g2)
    pairs = [(rank_, r2), (tgt, tg2), (score, sc2), (trans, t2), (gate, g2)]
    if w["table_dtype"] == "bf16":                      # one launch: the lattice need not be kept
        r3, tg3, sc3, st3 = ds.dspark_lattice_chain(cv, ct, prev, E, W, mode, hidden=hid, g=g)
        pairs += [(rank_, r3), (tgt, tg3), (score, sc3)]
    else:                                               # float32 tables: two launches need the lattice
        with pytest.raises(ds.DsparkError):
            ds.dspark_lattice_chain(cv, ct, prev, E, W, mode)
    torch.cuda.synchronize()
    assert ds.read_status(st2) == 0
    for a, b in pairs:
        assert torch.equal(a, b)


def test_lattice_chain_strong_head_and_long_block_fallback():
    import dspark_draft_selection_gb300 as ds
    for B in (8, 15):                                    # 8: the largest cluster; 15: two launches
        w = di.lattice_workload(44 + B, R=6, B=B, V_d=4096, K=64, rank=64, head_sigma=0.35)
        cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), B, 64)
        prev, E, W = dev(w["prev"]), dev(w["E"]), dev(w["W"])
        for mode in ("maxsum", "walk"):
            trans, gate, rank_, tgt, score = _two_call(ds, cv, ct, prev, E, W, mode)
            t2 = torch.empty_like(trans)
            r2, tg2, sc2, st2 = ds.dspark_lattice_chain(cv, ct, prev, E, W, mode, trans=t2)
            torch.cuda.synchronize()
            assert ds.read_status(st2) == 0
            assert torch.equal(rank_, r2) and torch.equal(tgt, tg2) and torch.equal(score, sc2)
            assert torch.equal(trans, t2)
    with pytest.raises(ds.DsparkError):                  # two launches need the lattice in memory
        ds.dspark_lattice_chain(cv, ct, prev, E, W, "maxsum")
