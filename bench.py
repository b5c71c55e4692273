"""Benchmark of the block-draft hot path on GB300: drafted blocks/s and logit HBM GB/s.

Default workload (the headline): the Qwen3-4B-shaped greedy draft (32 requests x block 7,
V = 151,936 bf16 logits with one +8 peak per row, K = 64, rank-256 bf16 Markov head, max-sum
chain). One step is one pass of the draft path over one batch: dspark_topk -> dspark_lattice_score
-> dspark_chain_select (the one-launch dspark_lattice_chain is timed beside it). Inputs are seeded synthetic tensors of the pages' shapes, resident in HBM;
the logits rotate over several independent sets whose total exceeds the 129 MB L2, so every step
reads cold logits. Steps are replayed as CUDA graphs (one graph runs every input set once), and
every timed region is repeated (`--repeats`): the reported time is the median region, with the
spread beside it.

The other workloads of the hot path are timed by the same run the same way (`secondary`): the
tiny lattice (latency), the pruned sampled DSpark draft, full-row top-p drafting on its rows, the
gated DFlash v2 head, the dense Markov walk with rejection-sampling verification, and the DFlash-2
grouped dynamic convolution over packed block rows.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--repeats M] [--impl ours|reference]
                    [--workloads c1,c2,c3,c3s,c4,c5,conv] [--no-cpu-baseline]

Multi-GPU (torchrun, one rank per GPU): every rank drafts its own batch (weak scaling, no
collective on the data path); timing is the max over ranks after a barrier.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import platform
import re
import subprocess
import sys
import time

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")  # one thread per oracle process; parallel legs use processes

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dspark_inputs as di  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20
METRIC = "drafted blocks/s and logit HBM GB/s (fraction of ~8 TB/s peak), 1×GB300"
UNIT = "blocks/s"
PROFILE_TOPK = os.path.join(ROOT, "profiles", "topk_row_kernel_qwen3_4b_R32_B7_V151936.md")
ALL_WORKLOADS = ("c2", "c1", "c3", "c3s", "c4", "c5", "conv")


def peaks():
    try:
        p = json.load(open(PEAKS_FILE))
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampler running while the timed regions run."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 9]
        busy = [r for r in rows if r[4].strip().isdigit() and int(r[4]) > 0] or rows
        sm = [float(r[1]) for r in busy if _isnum(r[1])]
        mx = [float(r[2]) for r in rows if _isnum(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in busy for n, v in zip(names, r[6:10]) if v.strip().lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(busy)}


def _isnum(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


def set_cid(rank: int, s: int, nsets: int) -> int:
    """Seed id of logit set `s` on `rank`: rank 0's first set is the named workload itself, and
    every other (rank, set) pair draws its own batch of requests of the same shape, so the ranks of
    a weak-scaling run draft disjoint requests."""
    return 2 + 100 * (rank * nsets + s)


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time: the job is done when its last rank is."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_blocks_per_s(world: int, requests_per_rank: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank drafts one block per request per step."""
    return world * requests_per_rank * steps / (ms / 1e3)


def median_spread(xs):
    xs = sorted(xs)
    return float(np.median(xs)), [round(xs[0], 6), round(xs[-1], 6)]


def algorithmic_logit_bytes(w):
    return w["R"] * w["B"] * w["V_d"] * (2 if w["dtype"] == "bf16" else 4)


def traffic_from_profile():
    """dram bytes per top-k launch from the committed ncu summary, if the kernel source is unchanged."""
    try:
        text = open(PROFILE_TOPK).read()
        sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text).group(1)
        dram = float(re.search(r"dram_bytes_per_launch:\s*([0-9.e+]+)", text).group(1))
    except Exception:
        return None
    src = open(os.path.join(ROOT, "dspark_draft_selection_gb300", "csrc", "topk.cu"), "rb").read()
    return dram if hashlib.sha256(src).hexdigest() == sha else None


# ------------------------------------------------------------------------------------------------
# graph timing
# ------------------------------------------------------------------------------------------------

class GraphTimer:
    """Captures sequences of library calls over rotating input sets into CUDA graphs and times
    their replays with CUDA events on the launching stream (max over ranks)."""

    def __init__(self, stream, device, world):
        self.stream, self.device, self.world = stream, device, world

    def capture(self, fns, nsets):
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for s in range(nsets):
                for fn in fns:
                    fn(s)
        return g

    def region_ms(self, graph, reps):
        """One timed region: `reps` replays between events, bracketed by barrier + sync."""
        import torch
        if self.world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            a.record(self.stream)
            for _ in range(reps):
                graph.replay()
            b.record(self.stream)
        torch.cuda.synchronize()
        if self.world > 1:
            torch.distributed.barrier()
        return max_over_ranks(a.elapsed_time(b), self.device)

    def per_call(self, fns, nsets, reps, repeats, warm=1):
        """Median ms per pass of `fns` over one input set, and the spread over the repeats."""
        g = self.capture(fns, nsets)
        for _ in range(warm):
            self.region_ms(g, 1)
        ms = [self.region_ms(g, reps) / (reps * nsets) for _ in range(repeats)]
        return median_spread(ms)


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------

def to_device(a, dev):
    import torch
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_ours(args):
    import torch

    import dspark_draft_selection_gb300 as ds

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    which = [x.strip() for x in args.workloads.split(",") if x.strip()]
    pool = None
    if rank == 0 and not args.no_cpu_baseline and "c2" in which:
        pool = OraclePool()            # spawned before any GPU work; workers build the workload
    stream = torch.cuda.Stream(device=dev)
    timer = GraphTimer(stream, dev, ws)
    hbm, hbm_kind = peaks()
    line = None
    clocks = Clocks(dev.index)
    if "c2" in which:
        line, clk = headline(args, ds, dev, stream, timer, hbm, hbm_kind, ws, rank, clocks)
    else:
        clocks.start()
    sec = {}
    if rank == 0:
        for name in which:
            if name != "c2":
                sec.update(SECONDARY[name](ds, dev, stream, timer, hbm, args))
    if "c2" not in which:
        clk = clocks.stop()
        line = {"metric": METRIC, "value": None, "unit": UNIT, "n_gpus": ws, "workloads": which, "clocks": clk}
    if sec:
        line["secondary"] = sec
    if pool is not None:
        w0 = di.config2()
        line["cpu_baseline"] = pool.baseline(w0)
        line["cpu_baseline_1core"] = cpu_baseline_1core(w0)
        pool.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def headline(args, ds, dev, stream, timer, hbm, hbm_kind, ws, rank, clocks):
    import torch
    w0 = di.config2()
    R, B, K = w0["R"], w0["B"], w0["K"]
    logit_bytes = algorithmic_logit_bytes(w0)
    nsets = max(2, int(np.ceil(2 * L2_BYTES / logit_bytes)))
    sets = []
    for s in range(nsets):
        cid = set_cid(rank, s, nsets)
        w = w0 if cid == w0["cid"] else di.lattice_workload(cid, R=R, B=B, V_d=w0["V_d"], K=K, rank=256, peak=8.0)
        sets.append(dict(logits=to_device(w["logits"], dev), prev=to_device(w["prev"], dev)))
    E, W = to_device(w0["E"], dev), to_device(w0["W"], dev)
    Kp = min(K, w0["V_d"])
    cand = (torch.empty((R, B, Kp), dtype=torch.int32, device=dev), torch.empty((R, B, Kp), dtype=torch.int32, device=dev),
            torch.empty((R, B, Kp), dtype=torch.float32, device=dev))
    trans = (torch.empty((R, B, Kp, Kp), dtype=torch.float32, device=dev),
             torch.empty((R, B), dtype=torch.float32, device=dev))
    chain = (torch.empty((R, B), dtype=torch.int32, device=dev), torch.empty((R, B), dtype=torch.int32, device=dev),
             torch.empty((R,), dtype=torch.float32, device=dev))
    status = ds.new_status(dev)

    def topk(s):
        ds.dspark_topk(sets[s]["logits"], B, K, out=cand, status=status, stream=stream)

    def lattice_chain(s):
        ds.dspark_lattice_chain(cand[2], cand[1], sets[s]["prev"], E, W, "maxsum", out=chain, status=status,
                                stream=stream)

    def lattice(s):
        ds.dspark_lattice_score(cand[1], sets[s]["prev"], E, W, out=trans, status=status, stream=stream)

    def chain_sel(s):
        ds.dspark_chain_select(cand[2], trans[0], cand[1], "maxsum", out=chain, status=status, stream=stream)

    def step(s):
        topk(s)
        lattice(s)
        chain_sel(s)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(nsets):       # first calls configure the kernels outside any capture
            step(s)
    torch.cuda.synchronize()
    assert ds.read_status(status) == 0

    # end to end through the same entry points with host buffers: H2D of the step's logits and
    # previous tokens, the draft path, D2H of the chosen chain and its score
    host_logits = [sets[s]["logits"].cpu().pin_memory() for s in range(nsets)]
    host_prev = [sets[s]["prev"].cpu().pin_memory() for s in range(nsets)]
    dev_logits = torch.empty_like(sets[0]["logits"])
    dev_prev = torch.empty_like(sets[0]["prev"])
    host_out = torch.empty((R, B), dtype=torch.int32).pin_memory()
    host_score = torch.empty((R,), dtype=torch.float32).pin_memory()

    def e2e(s):
        dev_logits.copy_(host_logits[s], non_blocking=True)
        dev_prev.copy_(host_prev[s], non_blocking=True)
        ds.dspark_topk(dev_logits, B, K, out=cand, status=status, stream=stream)
        ds.dspark_lattice_score(cand[1], dev_prev, E, W, out=trans, status=status, stream=stream)
        ds.dspark_chain_select(cand[2], trans[0], cand[1], "maxsum", out=chain, status=status, stream=stream)
        host_out.copy_(chain[1], non_blocking=True)
        host_score.copy_(chain[2], non_blocking=True)

    with torch.cuda.stream(stream):
        e2e(0)
    torch.cuda.synchronize()
    h2d_bytes = host_logits[0].numel() * host_logits[0].element_size() + host_prev[0].numel() * 4
    d2h_bytes = host_out.numel() * 4 + host_score.numel() * 4

    reps = max(1, -(-args.steps // nsets))
    steps = reps * nsets
    g_step = timer.capture([step], nsets)
    g_e2e = timer.capture([e2e], nsets)
    for _ in range(max(1, -(-args.warmup // nsets))):
        timer.region_ms(g_step, 1)
    clocks.start()
    time.sleep(0.2)
    regions = [timer.region_ms(g_step, reps) for _ in range(args.repeats)]
    ms_total, spread = median_spread(regions)
    k_topk, sp_topk = timer.per_call([topk], nsets, reps, args.repeats)
    k_lat, _ = timer.per_call([lattice], nsets, reps, args.repeats)
    k_chain, _ = timer.per_call([chain_sel], nsets, reps, args.repeats)
    k_lc, _ = timer.per_call([lattice_chain], nsets, reps, args.repeats)
    timer.region_ms(g_e2e, 1)
    e2e_regions = [timer.region_ms(g_e2e, reps) for _ in range(args.repeats)]
    ms_e2e, e2e_spread = median_spread(e2e_regions)
    clk = clocks.stop()
    torch.cuda.synchronize()
    assert ds.read_status(status) == 0, "device status set during the bench"
    ms_step = ms_total / steps
    value = job_blocks_per_s(ws, R, steps, ms_total)
    achieved = logit_bytes / (k_topk / 1e3) / 1e9
    traffic = traffic_from_profile()
    step_bytes = logit_bytes + R * ((B - 1) * Kp + 1) * 512 + R * B * Kp * 512   # logits + E and W gathers
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded Gaussian logits and head tables)",
        "config": {"workload": w0["name"], "requests": R, "block": B, "vocab": w0["V_d"], "k": K, "rank": 256,
                   "chain": "maxsum", "per_gpu_batch": R,
                   "parallelism": f"dp{ws}: {R} own requests per rank, no collective on the data path",
                   "l2": f"{nsets} rotating logit sets of {logit_bytes / 1e6:.1f} MB (> 129 MB L2)",
                   "graphs": "each step replayed as a CUDA graph",
                   "launches": "dspark_topk, dspark_lattice_score, dspark_chain_select"},
        "repeats": args.repeats,
        "ms_per_step_spread": [round(x / steps, 5) for x in spread],
        "logit_gbs": round(achieved, 1),
        "step_algorithmic_gbs": round(step_bytes / (ms_step / 1e3) / 1e9, 1),
        "kernels_ms": {"topk": round(k_topk, 5), "lattice": round(k_lat, 5), "chain": round(k_chain, 5),
                       "lattice_chain_fused_alternative": round(k_lc, 5)},
        "roofline": {"kernel": "topk_row_kernel (dspark_topk)", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": traffic, "algorithmic_bytes": logit_bytes,
                     "achieved_spread": [round(logit_bytes / (x / 1e3) / 1e9, 1) for x in sp_topk[::-1]]},
        "e2e": {"value": round(job_blocks_per_s(ws, R, steps, ms_e2e), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes),
                "ms_per_step_spread": [round(x / steps, 5) for x in e2e_spread]},
        "gpu_launches": 3 * steps,   # topk_row_kernel, lattice_tc_kernel, chain_kernel per step
        "clocks": clk,
    }
    return line, clk


# ------------------------------------------------------------------------------------------------
# the other workloads of the hot path (reported beside the headline, not part of its step)
# ------------------------------------------------------------------------------------------------

def _kernels(timer, parts, nsets, reps, repeats):
    out = {}
    for name, fns in parts:
        ms, _ = timer.per_call(fns, nsets, reps, repeats)
        out[name] = round(ms, 5)
    return out


def _check(ds, status, what):
    import torch
    torch.cuda.synchronize()
    st = ds.read_status(status)
    if st != 0:
        raise RuntimeError(f"device status {st} during {what}")


def bench_c1(ds, dev, stream, timer, hbm, args):
    """Tiny lattice (1 request x block 7, V = 1,024 fp32, K = 8, fp32 rank-16 tables): latency."""
    import torch
    w = di.config1()
    R, B, K = w["R"], w["B"], w["K"]
    logits, E, W, prev = (to_device(w[k], dev) for k in ("logits", "E", "W", "prev"))
    status = ds.new_status(dev)
    cand = ds.dspark_topk(logits, B, K, status=status, stream=stream)[:3]
    trans = ds.dspark_lattice_score(cand[1], prev, E, W, status=status, stream=stream)[:2]
    chain = ds.dspark_chain_select(cand[2], trans[0], cand[1], "maxsum", status=status, stream=stream)[:3]

    def step(s):
        ds.dspark_topk(logits, B, K, out=cand, status=status, stream=stream)
        ds.dspark_lattice_score(cand[1], prev, E, W, out=trans, status=status, stream=stream)
        ds.dspark_chain_select(cand[2], trans[0], cand[1], "maxsum", out=chain, status=status, stream=stream)

    n = 64                                   # steps per graph (one input set, L2-resident by design)
    ms, spread = timer.per_call([step], n, 4, args.repeats)
    _check(ds, status, "c1")
    return {w["name"]: {"us_per_block": round(ms * 1e3 / R, 3), "us_per_block_spread": [round(x * 1e3, 3) for x in spread],
                        "blocks_per_s": round(R / (ms / 1e3), 1), "graph": f"{n} steps per graph, 3 launches a step"}}


def bench_c3(ds, dev, stream, timer, hbm, args):
    """Pruned sampled DSpark draft: Top-K with d2t, lattice, sampled walk with a sparse q record."""
    import torch
    w = di.config3()
    R, B, K = w["R"], w["B"], w["K"]
    nsets = 3
    logits = [to_device(w["logits"], dev)] + [torch.roll(to_device(w["logits"], dev), s, 0) for s in (1, 2)]
    d2t, E, W, prev = (to_device(w[k], dev) for k in ("d2t", "E", "W", "prev"))
    seed, step_ = to_device(w["seed"], dev), to_device(w["step"], dev)
    status = ds.new_status(dev)
    cand = ds.dspark_topk(logits[0], B, K, d2t=d2t, V_t=w["V_t"], status=status, stream=stream)[:3]
    trans = ds.dspark_lattice_score(cand[1], prev, E, W, status=status, stream=stream)[:2]
    chain = ds.dspark_chain_select(cand[2], trans[0], cand[1], "sample", temperature=w["temperature"],
                                   top_p=w["top_p"], seed=seed, step=step_, status=status, stream=stream)
    chain_out, qrec = chain[:3], chain[3:6]

    def topk(s):
        ds.dspark_topk(logits[s], B, K, d2t=d2t, V_t=w["V_t"], out=cand, status=status, stream=stream)

    def lattice(s):
        ds.dspark_lattice_score(cand[1], prev, E, W, out=trans, status=status, stream=stream)

    def chain_sample(s):
        ds.dspark_chain_select(cand[2], trans[0], cand[1], "sample", temperature=w["temperature"], top_p=w["top_p"],
                               seed=seed, step=step_, q=qrec, out=chain_out, status=status, stream=stream)

    reps = 8
    ms, spread = timer.per_call([topk, lattice, chain_sample], nsets, reps, args.repeats)
    ker = _kernels(timer, [("topk", [topk]), ("lattice", [lattice]), ("chain_sample", [chain_sample])], nsets, reps,
                   args.repeats)
    _check(ds, status, "c3")
    lb = R * B * w["V_d"] * 2
    return {w["name"]: {"blocks_per_s": round(R / (ms / 1e3), 1), "ms_per_step": round(ms, 5), "ms_per_step_spread": spread,
                        "logit_gbs": round(lb / (ker["topk"] / 1e3) / 1e9, 1),
                        "logit_frac": round(lb / (ker["topk"] / 1e3) / 1e9 / hbm, 4), "kernels_ms": ker,
                        "l2": f"{nsets} rotating logit sets of {lb / 1e6:.1f} MB"}}


def bench_c3s(ds, dev, stream, timer, hbm, args):
    """Full-row multinomial drafting without a head on the pruned draft's rows (240 x 114,688 bf16,
    d2t to target ids, T = 0.8, top-p 0.95): the nucleus path of dspark_sample."""
    import torch
    w = di.config3()
    R, B = w["R"], w["B"]
    nsets = 3
    logits = [to_device(w["logits"], dev)] + [torch.roll(to_device(w["logits"], dev), s, 0) for s in (1, 2)]
    d2t = to_device(w["d2t"], dev)
    seed, step_ = to_device(w["seed"], dev), to_device(w["step"], dev)
    status = ds.new_status(dev)
    out = ds.dspark_sample(logits[0], B, d2t=d2t, V_t=w["V_t"], temperature=w["temperature"], top_p=w["top_p"],
                           seed=seed, step=step_, status=status, stream=stream)[:2]

    def sample(s):
        ds.dspark_sample(logits[s], B, d2t=d2t, V_t=w["V_t"], temperature=w["temperature"], top_p=w["top_p"],
                         seed=seed, step=step_, out=out, status=status, stream=stream)

    ms, spread = timer.per_call([sample], nsets, 4, args.repeats)
    _check(ds, status, "c3s")
    lb = R * B * w["V_d"] * 2
    return {f"full_row_top_p_R{R}_B{B}_Vd{w['V_d']}_T0.8_p0.95": {
        "blocks_per_s": round(R / (ms / 1e3), 1), "ms_per_step": round(ms, 5), "ms_per_step_spread": spread,
        "rows_per_s": round(R * B / (ms / 1e3), 1), "logit_gbs": round(lb / (ms / 1e3) / 1e9, 1),
        "logit_frac": round(lb / (ms / 1e3) / 1e9 / hbm, 4), "kernels_ms": {"sample": round(ms, 5)}}}


def bench_c4(ds, dev, stream, timer, hbm, args):
    """DFlash v2 gated head: 896 rows of 248,320 logits (445 MB, larger than L2)."""
    w = di.config4()
    R, B, K = w["R"], w["B"], w["K"]
    logits, E, W, prev, hidden, g = (to_device(w[k], dev) for k in ("logits", "E", "W", "prev", "hidden", "g"))
    status = ds.new_status(dev)
    cand = ds.dspark_topk(logits, B, K, status=status, stream=stream)[:3]
    trans = ds.dspark_lattice_score(cand[1], prev, E, W, hidden=hidden, g=g, status=status, stream=stream)[:2]
    chain = ds.dspark_chain_select(cand[2], trans[0], cand[1], "maxsum", status=status, stream=stream)[:3]

    def topk(s):
        ds.dspark_topk(logits, B, K, out=cand, status=status, stream=stream)

    def lattice(s):
        ds.dspark_lattice_score(cand[1], prev, E, W, hidden=hidden, g=g, out=trans, status=status, stream=stream)

    def chain_sel(s):
        ds.dspark_chain_select(cand[2], trans[0], cand[1], "maxsum", out=chain, status=status, stream=stream)

    def lattice_chain(s):
        ds.dspark_lattice_chain(cand[2], cand[1], prev, E, W, "maxsum", hidden=hidden, g=g, out=chain,
                                status=status, stream=stream)

    reps = 6
    ms, spread = timer.per_call([topk, lattice, chain_sel], 1, reps, args.repeats)
    ker = _kernels(timer, [("topk", [topk]), ("lattice_gated", [lattice]), ("chain", [chain_sel]),
                           ("lattice_chain_fused_alternative", [lattice_chain])], 1, reps, args.repeats)
    _check(ds, status, "c4")
    lb = R * B * w["V_d"] * 2
    return {w["name"]: {"blocks_per_s": round(R / (ms / 1e3), 1), "ms_per_step": round(ms, 5), "ms_per_step_spread": spread,
                        "logit_gbs": round(lb / (ker["topk"] / 1e3) / 1e9, 1),
                        "logit_frac": round(lb / (ker["topk"] / 1e3) / 1e9 / hbm, 4), "kernels_ms": ker}}


def bench_c5(ds, dev, stream, timer, hbm, args):
    """Dense Markov walk sampled at T = 1 with a dense q record, then rejection-sampling verification
    (64 x 15 draft rows and 64 x 16 target rows of 151,936 bf16 logits)."""
    import torch
    w = di.config5()
    R, B, V, rank = w["R"], w["B"], w["V_d"], w["rank"]
    logits, E, W, prev = (to_device(w[k], dev) for k in ("logits", "E", "W", "prev"))
    target, seed, step_, vseed = (to_device(w[k], dev) for k in ("target", "seed", "step", "vseed"))
    status = ds.new_status(dev)
    q = ds.dense_record(R * B, V, dev)
    ws_walk = ds.workspace(ds.OP_DENSE_WALK, R, B, V, 0, dev)
    ws_ver = ds.workspace(ds.OP_VERIFY, R, B, V, 0, dev)
    walk_out = ds.dspark_dense_walk(logits, B, prev, E, W, temperature=1.0, top_p=1.0, seed=seed, step=step_, q=q,
                                    ws=ws_walk, status=status, stream=stream)[:2]
    n = torch.full((R,), B, dtype=torch.int32, device=dev)
    ver_out = ds.dspark_verify(target, B, walk_out[0], n, q, temperature=1.0, top_p=1.0, vseed=vseed, step=step_,
                               ws=ws_ver, status=status, stream=stream)[:3]

    def walk(s):
        ds.dspark_dense_walk(logits, B, prev, E, W, temperature=1.0, top_p=1.0, seed=seed, step=step_, q=q,
                             out=walk_out, ws=ws_walk, status=status, stream=stream)

    def verify(s):
        ds.dspark_verify(target, B, walk_out[0], n, q, temperature=1.0, top_p=1.0, vseed=vseed, step=step_,
                         out=ver_out, ws=ws_ver, status=status, stream=stream)

    reps = 3
    ms, spread = timer.per_call([walk, verify], 1, reps, args.repeats)
    ker = _kernels(timer, [("dense_walk", [walk]), ("verify", [verify])], 1, reps, args.repeats)
    _check(ds, status, "c5")
    draft_b, target_b = R * B * V * 2, R * (B + 1) * V * 2
    # algorithmic bytes of the walk: W read once per position, the draft logits once, the dense
    # record's z rows written once (float32)
    walk_bytes = B * V * rank * 2 + draft_b + R * B * V * 4
    return {w["name"]: {"blocks_per_s": round(R / (ms / 1e3), 1), "ms_per_step": round(ms, 5), "ms_per_step_spread": spread,
                        "logit_gbs": round((draft_b + target_b) / (ms / 1e3) / 1e9, 1),
                        "dense_walk_gbs": round(walk_bytes / (ker["dense_walk"] / 1e3) / 1e9, 1),
                        "dense_walk_frac": round(walk_bytes / (ker["dense_walk"] / 1e3) / 1e9 / hbm, 4),
                        "dense_walk_bytes": walk_bytes,
                        "verify_logit_gbs": round(target_b / (ker["verify"] / 1e3) / 1e9, 1),
                        "verify_frac": round(target_b / (ker["verify"] / 1e3) / 1e9 / hbm, 4),
                        "kernels_ms": ker}}


def bench_conv(ds, dev, stream, timer, hbm, args):
    """DFlash-2 grouped dynamic convolution on C4-shaped packed rows: 128 requests x (1 context +
    7 block rows) x 5,120 channels, 32 groups, 4 taps; six input/output sets (189 MB, larger
    than L2) rotate between calls."""
    import torch
    w = di.conv_workload()
    nsets = 6
    x0 = to_device(w["x"], dev)
    xs = [x0] + [torch.roll(x0, s, 1) for s in range(1, nsets)]
    k, block = to_device(w["k"], dev), to_device(w["block"], dev)
    ys = [torch.empty((w["N"], w["C"]), dtype=torch.float32, device=dev) for _ in range(nsets)]

    def conv(s):
        ds.dspark_grouped_conv(xs[s], k, block, out=ys[s], stream=stream)

    ms, spread = timer.per_call([conv], nsets, 4, args.repeats)
    nb = w["N"] * w["C"] * (2 + 4) + k.numel() * 4 + block.numel() * 4
    return {w["name"]: {"ms_per_call": round(ms, 5), "ms_per_call_spread": spread,
                        "gbs": round(nb / (ms / 1e3) / 1e9, 1), "frac": round(nb / (ms / 1e3) / 1e9 / hbm, 4),
                        "bytes": nb, "kernels_ms": {"grouped_conv": round(ms, 5)}}}


SECONDARY = {"c1": bench_c1, "c3": bench_c3, "c3s": bench_c3s, "c4": bench_c4, "c5": bench_c5, "conv": bench_conv}


# ------------------------------------------------------------------------------------------------
# CPU oracle legs
# ------------------------------------------------------------------------------------------------

_W = {}


def _oracle_init():
    w = di.config2()
    _W["s"] = di.bf16_bits_to_f32(w.pop("logits"))
    _W["E"] = di.bf16_bits_to_f32(w.pop("E"))
    _W["W"] = di.bf16_bits_to_f32(w.pop("W"))
    _W["w"] = w


def _oracle_request(r):
    """The oracle's whole draft path for one request of the headline workload (in a worker)."""
    from oracle import draft as od
    w, s, B = _W["w"], _W["s"], _W["w"]["B"]
    od.select_request(s[r * B:(r + 1) * B], w["K"], _W["E"], _W["W"], int(w["prev"][r]), w["mode"])
    return 1


def _noop(_):
    return os.getpid()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1"}


def cpu_model():
    try:
        info = {}
        for ln in open("/proc/cpuinfo"):
            if ":" in ln:
                k, v = ln.split(":", 1)
                info.setdefault(k.strip().lower(), v.strip())
        if "model name" in info:
            return info["model name"]
        if "cpu part" in info:
            return ARM_PARTS.get(info["cpu part"], f"Arm part {info['cpu part']}")
    except Exception:
        pass
    return platform.processor() or platform.machine()


class OraclePool:
    """The oracle on every host core: one single-threaded process per core (spawned, so no CUDA
    state is inherited), requests distributed over them."""

    def __init__(self, procs=None):
        self.n = max(1, min(procs or host_cores(), 32))
        self.pool = mp.get_context("spawn").Pool(self.n, initializer=_oracle_init)
        self.pool.map(_noop, range(4 * self.n))                 # every worker is up

    def rate(self, reqs):
        t0 = time.perf_counter()
        done = sum(self.pool.map(_oracle_request, reqs, chunksize=1))
        return done / (time.perf_counter() - t0)

    def baseline(self, w):
        reqs = list(range(w["R"])) * max(1, -(-2 * self.n // w["R"]))
        reqs = reqs[:max(w["R"], 2 * self.n)]
        v = self.rate(reqs)
        return {"value": round(v, 3), "unit": UNIT, "cores": self.n, "kind": "oracle",
                "sample": f"{len(reqs)} requests of {w['name']} over {self.n} single-threaded processes "
                          f"(numpy oracle; {cpu_model()})"}

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline_1core(w, nreq=6):
    from oracle import draft as od
    s = di.bf16_bits_to_f32(w["logits"])
    E, W = di.bf16_bits_to_f32(w["E"]), di.bf16_bits_to_f32(w["W"])
    B = w["B"]
    t0 = time.perf_counter()
    for r in range(nreq):
        od.select_request(s[r * B:(r + 1) * B], w["K"], E, W, int(w["prev"][r]), w["mode"])
    v = nreq / (time.perf_counter() - t0)
    return {"value": round(v, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{nreq} of {w['R']} requests of {w['name']} (numpy oracle, one thread; {cpu_model()})"}


def run_reference(args):
    """The oracle, as it stands, on the host cores: every step drafts a batch of whole requests of
    the headline workload, one request per core, sized so the whole run ends within minutes."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    w = di.config2()
    pool = OraclePool()
    t0 = time.perf_counter()
    pool.rate(list(range(pool.n)))
    t_batch = time.perf_counter() - t0                       # one request per core
    budget = 150.0
    per_step = pool.n * max(1, int(budget / max(1e-3, t_batch * (args.steps + args.warmup))))
    per_step = min(per_step, 4 * pool.n)
    nxt = {"r": 0}

    def one_step():
        reqs = [(nxt["r"] + k) % w["R"] for k in range(per_step)]
        nxt["r"] += per_step
        return sum(pool.pool.map(_oracle_request, reqs, chunksize=1))

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    done = 0
    for _ in range(args.steps):
        done += one_step()
    dt = time.perf_counter() - t0
    pool.close()
    value = done / dt
    sample = (f"{per_step} whole requests of {w['name']} per step over {pool.n} single-threaded processes "
              f"(numpy oracle; {cpu_model()})")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Gaussian logits and head tables)",
        "config": {"workload": w["name"], "requests": w["R"], "block": w["B"], "vocab": w["V_d"], "k": w["K"],
                   "rank": 256, "chain": "maxsum"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": pool.n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--repeats", type=int, default=5, help="timed regions per measurement (median reported)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workloads", default=",".join(ALL_WORKLOADS),
                    help="comma list of c2 (headline), c1, c3, c3s, c4, c5")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.repeats = max(1, args.repeats)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
