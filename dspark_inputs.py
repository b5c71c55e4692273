"""Seeded synthetic workloads for the block-draft selector and verifier.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. Both the CPU oracle (``oracle/``) and the CUDA path (through
the tests and ``bench.py``) take their inputs from here, so a parity test feeds
the two sides the very same arrays.

Shapes follow the workloads of the DFlash/DSpark pages: vocabulary sizes 151,936
(Qwen3-4B), 248,320 (DFlash v2 targets) and 114,688 drafted out of 248,100 target
tokens (MiniCPM-OCR-1.0-DSpark), block lengths 7 and 15, K = 64 candidates. The
pages' benchmark data (HumanEval, MT-Bench, OmniDocBench) is not used: logits,
hidden states and head tables are Gaussian with the scales below.

Random streams: numpy's PCG64 seeded by ``SeedSequence([BASE_SEED + 1000 * c,
stream])`` for config ``c`` and a fixed stream id per tensor. bf16 tensors are
drawn in float32 and rounded to the nearest bf16 (ties to even); they are held
as their uint16 bit patterns because numpy has no bf16 type.
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202

# stream ids, one per tensor kind
S_LOGITS, S_E, S_W, S_HIDDEN, S_G, S_PREV, S_SUBSET, S_SEEDS, S_PEAK, S_TARGET, S_VSEEDS = range(11)


def generator(config_id: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([BASE_SEED + 1000 * config_id, stream])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(gen: np.random.Generator, shape, sigma: float, dtype: str, chunk_rows: int = 64) -> np.ndarray:
    """N(0, sigma^2) samples as float32 or as bf16 bit patterns, drawn row-chunk by row-chunk."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16 if dtype == "bf16" else np.float32)
    rows = shape[0] if len(shape) > 1 else 1
    flat = out.reshape(rows, -1)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = gen.standard_normal((r1 - r0, flat.shape[1]), dtype=np.float32) * np.float32(sigma)
        flat[r0:r1] = f32_to_bf16_bits(x) if dtype == "bf16" else x
    return out


def lattice_workload(
    cid: int,
    R: int,
    B: int,
    V_d: int,
    K: int,
    rank: int,
    dtype: str = "bf16",
    table_dtype: str | None = None,
    logit_sigma: float = 2.0,
    head_sigma: float = 0.05,
    V_t: int | None = None,
    pruned: bool = False,
    H: int = 0,
    gate_sigma: float = 0.02,
    peak: float = 0.0,
    with_seeds: bool = False,
) -> dict:
    """Draft-side workload: logits [R*B, V_d], Markov head tables E, W [V_t, rank],
    optional hidden states [R*B, H] with gate vector g [H], previous tokens [R],
    optional pruned vocabulary (d2t) and per-request RNG seeds."""
    table_dtype = table_dtype or dtype
    V_t = V_d if V_t is None else V_t
    rows = R * B
    w = {"cid": cid, "R": R, "B": B, "V_d": V_d, "V_t": V_t, "K": K, "rank": rank, "dtype": dtype,
         "table_dtype": table_dtype, "H": H}
    w["logits"] = normal(generator(cid, S_LOGITS), (rows, V_d), logit_sigma, dtype)
    if peak:
        # one planted peak per row: +peak at a seeded index
        idx = generator(cid, S_PEAK).integers(0, V_d, size=rows)
        if dtype == "bf16":
            vals = bf16_bits_to_f32(w["logits"][np.arange(rows), idx]) + np.float32(peak)
            w["logits"][np.arange(rows), idx] = f32_to_bf16_bits(vals)
        else:
            w["logits"][np.arange(rows), idx] += np.float32(peak)
        w["peak_idx"] = idx
    w["E"] = normal(generator(cid, S_E), (V_t, rank), head_sigma, table_dtype)
    w["W"] = normal(generator(cid, S_W), (V_t, rank), head_sigma, table_dtype)
    if pruned:
        # a seeded random subset S of the target vocabulary, in shuffled order;
        # draft token i stands for target token S[i] = i + d2t[i]
        S = generator(cid, S_SUBSET).permutation(V_t)[:V_d].astype(np.int64)
        w["subset"] = S
        w["d2t"] = S - np.arange(V_d, dtype=np.int64)
        outside = np.ones(V_t, dtype=bool)
        outside[S] = False
        w["W"][outside] = 0  # the next-token table is zero outside the draft vocabulary
    else:
        w["d2t"] = None
    if H:
        w["hidden"] = normal(generator(cid, S_HIDDEN), (rows, H), 1.0, dtype)
        w["g"] = normal(generator(cid, S_G), (H,), gate_sigma, dtype)
    else:
        w["hidden"] = None
        w["g"] = None
    w["prev"] = generator(cid, S_PREV).integers(0, V_t, size=R).astype(np.int32)
    if with_seeds:
        g = generator(cid, S_SEEDS)
        w["seed"] = g.integers(0, 2**63, size=R, dtype=np.int64).astype(np.uint64)
        w["step"] = g.integers(0, 2**40, size=R, dtype=np.int64).astype(np.uint64)
    return w


def add_target(w: dict, corr: float = 0.8, sigma: float = 2.0) -> dict:
    """Target logits [R*(B+1), V] for verification: row j < B of request r is
    corr*draft + sqrt(1-corr^2)*z with z ~ N(0, sigma^2) independent; the bonus
    row B is a fresh N(0, sigma^2) row. Also draws separate verify seeds."""
    R, B, V = w["R"], w["B"], w["V_t"]
    assert w["d2t"] is None and w["V_d"] == V
    gen = generator(w["cid"], S_TARGET)
    dtype = w["dtype"]
    out = np.empty((R * (B + 1), V), dtype=np.uint16 if dtype == "bf16" else np.float32)
    c2 = np.float32(np.sqrt(1.0 - corr * corr))
    for r in range(R):
        d = w["logits"][r * B:(r + 1) * B]
        d = bf16_bits_to_f32(d) if dtype == "bf16" else d
        z = gen.standard_normal((B + 1, V), dtype=np.float32) * np.float32(sigma)
        t = np.empty((B + 1, V), dtype=np.float32)
        t[:B] = np.float32(corr) * d + c2 * z[:B]
        t[B] = z[B]
        out[r * (B + 1):(r + 1) * (B + 1)] = f32_to_bf16_bits(t) if dtype == "bf16" else t
    w["target"] = out
    g = generator(w["cid"], S_VSEEDS)
    w["vseed"] = g.integers(0, 2**63, size=R, dtype=np.int64).astype(np.uint64)
    return w


# ---- the five workloads ------------------------------------------------------------------

def config1() -> dict:
    """Tiny lattice: 1 request x block 7, V=1,024 fp32 logits ~N(0,3^2), K=8,
    head tables fp32 [1024 x 16] ~N(0,0.1^2), no gate; max-sum chain."""
    w = lattice_workload(1, R=1, B=7, V_d=1024, K=8, rank=16, dtype="f32", logit_sigma=3.0, head_sigma=0.1)
    w.update(name="tiny_lattice_R1_B7_V1024_K8", mode="maxsum")
    return w


def config2(R: int = 32, V: int = 151936) -> dict:
    """Qwen3-4B-shaped greedy draft: 32 x block 7, V=151,936 bf16 ~N(0,2^2) with
    one +8 peak per row, K=64, rank-256 bf16 head ~N(0,0.05^2), no gate."""
    w = lattice_workload(2, R=R, B=7, V_d=V, K=64, rank=256, peak=8.0)
    w.update(name=f"qwen3_4b_greedy_R{R}_B7_V{V}_K64_r256", mode="maxsum")
    return w


def config3(R: int = 16, V_d: int = 114688, V_t: int = 248100) -> dict:
    """Pruned-vocabulary DSpark (MiniCPM-OCR-shaped): 16 x block 15, draft V
    114,688 over target V 248,100, d2t from a seeded unsorted subset, table zero
    outside it, K = min(64, V_d), sampled T=0.8 top-p 0.95."""
    w = lattice_workload(3, R=R, B=15, V_d=V_d, V_t=V_t, K=64, rank=256, pruned=True, with_seeds=True)
    w.update(name=f"minicpm_ocr_pruned_sampled_R{R}_B15_Vd{V_d}_Vt{V_t}_K64", mode="sample",
             temperature=0.8, top_p=0.95)
    return w


def config4(R: int = 128, V: int = 248320) -> dict:
    """DFlash v2 gated head: 128 x block 7, V=248,320 bf16, hidden 5,120 bf16
    ~N(0,1), gate sigmoid(h.g) with g ~N(0,0.02^2), K=64, rank 256."""
    w = lattice_workload(4, R=R, B=7, V_d=V, K=64, rank=256, H=5120, gate_sigma=0.02)
    w.update(name=f"dflash2_gated_R{R}_B7_V{V}_K64_r256_H5120", mode="maxsum")
    return w


def config5(R: int = 64, V: int = 151936) -> dict:
    """Dense walk + verify: 64 x 15 candidates, V=151,936, full-V transition row
    per position, sampled at T=1.0, then rejection-sampling verification against
    target bf16 logits correlated 0.8 with the draft's."""
    w = lattice_workload(5, R=R, B=15, V_d=V, K=0, rank=256, with_seeds=True)
    add_target(w)
    w.update(name=f"dense_walk_verify_R{R}_B15_V{V}_r256", mode="dense", temperature=1.0, top_p=1.0)
    return w


def conv_workload(cid: int = 6, R: int = 128, B: int = 7, C: int = 5120, G: int = 32, L: int = 4,
                  ctx: int = 1, dtype: str = "bf16") -> dict:
    """Packed block rows for the DFlash-2 grouped dynamic convolution: R requests, each `ctx`
    context rows then B block rows (block ids 2r for the context rows, 2r + 1 for the block),
    x ~ N(0, 1) [N, C], dynamic taps k ~ N(0, 0.5^2) [N, G, L] float32 (synthetic weights)."""
    N = R * (ctx + B)
    block = np.repeat(np.arange(R, dtype=np.int32) * 2, ctx + B)
    block += np.tile(np.r_[np.zeros(ctx, np.int32), np.ones(B, np.int32)], R)
    x = normal(generator(cid, S_HIDDEN), (N, C), 1.0, dtype)
    k = normal(generator(cid, S_G), (N, G * L), 0.5, "f32").reshape(N, G, L)
    return dict(name=f"dflash2_grouped_conv_R{R}_B{B}_C{C}_G{G}_L{L}", x=x, x_dtype=dtype, k=k, block=block,
                R=R, B=B, C=C, G=G, L=L, N=N)


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}
