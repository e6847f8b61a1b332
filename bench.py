#!/usr/bin/env python
"""Benchmark of the speculative-decoding verify-and-commit step on GB300.

Workload (one step = one spec_verify call over one batch): sampling verify,
B=256 requests, K=7 draft tokens each, V=151936, bf16 logits, T=0.7, peaked
rank-score rows (the configuration the throughput target is quoted on):
R_t = 2048 target rows + 1792 draft rows = 1,166,868,480 bytes of logits per
step, more than 9x the 129 MB L2, so every step streams from HBM (no flush).

Prints one JSON line (rank 0):
  value      spec_verify target rows/s, whole job (all ranks), device-timed
  e2e        the same metric through the C ABI with host buffers: pinned
             host->device copy of the step's inputs, the call, and the
             device->host read of out_tokens/out_len inside the timed region
  roofline   HBM: algorithmic bytes per launch / mean launch time (CUDA events
             on the launching stream) against the measured copy bandwidth
  cpu_baseline  the float64 oracle on the host cores, on a bounded sample

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--strong]
Under torchrun each rank runs its own batch on its own GPU (weak scaling; the
requests are independent, so there is no data-path collective). With
--strong the ranks split one global batch by requests (sharding.py, balanced
by the logit rows each request reads) and, after the timed region, gather
their outputs; rank 0 checks them against one verify of the whole batch.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

METRIC = "spec_verify rows/s, committed tokens/s and HBM GB/s (% of GB300 peak), 1 GPU"
WORKLOAD = ("sampling verify B=256 K=7 V=151936 bf16 T=0.7, peaked rank-score rows "
            "(z_t = -4.4 ln rank + N(0,1) over a random permutation, z_d = z_t + N(0,1), x̂ ~ q)")
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes (read + write) per verify launch on this workload from one ncu
# capture, valid only for the kernel sources whose hash is recorded with it.
TRAFFIC = {"sources_sha256": "07cd1b2605df1b3f5e0fb7aecfd57cf87d31deba716596232bf994a0c9b2cb35",
           "bytes_per_launch": 1235357440 + 4756224,
           "profile": "profiles/verify_kernel_sampling_B256_K7_V151936_bf16.md"}


VERIFY_SOURCES = ("spec_verify.cu", "sv_device.cuh", "sv_filter.cuh")


def kernel_sources_hash(names=VERIFY_SOURCES) -> str:
    """sha256 over the named kernel sources (the verify kernel's by default)."""
    d = os.path.join(ROOT, "speculative_decoding_verification_27_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(names):
        h.update(f.encode())
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks (the slowest rank's time); x itself
    when no process group is running."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(seed: int, rank: int) -> int:
    """Each rank verifies its own batch of the same shape (weak scaling)."""
    return seed + rank


def make_batch(seed: int, B: int = 256):
    from speculative_decoding_verification_27_gb300 import workloads as W
    return W.config3(seed=seed, B=B)


def oracle_sample(batch, requests: int):
    """The first `requests` requests of a batch, as their own packed batch."""
    import numpy as np
    from speculative_decoding_verification_27_gb300 import workloads as W
    cu = batch.cu_draft[:requests + 1].astype(np.int32)
    rt, rd = int(cu[-1]) + requests, int(cu[-1])
    return W.VerifyBatch(batch.name + "-sample", batch.target[:rt], None if batch.draft is None else batch.draft[:rd],
                         batch.draft_tokens[:rd], cu, batch.uniforms[:rt], batch.temperature,
                         None if batch.mode is None else batch.mode[:requests])


def time_oracle(batch, diagnostics: bool = False):
    """Wall time of one float64 oracle call over `batch` on all host cores."""
    import oracle
    threads = min(oracle.default_threads(), batch.B)
    t = time.perf_counter()
    res = oracle.spec_verify(batch.target, batch.draft, batch.draft_tokens, batch.cu_draft,
                             batch.uniforms, batch.temperature, batch.mode, threads, diagnostics)
    return time.perf_counter() - t, threads, res


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.gpu_id],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]) if f[3] not in ("[N/A]", "N/A") else None, f[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        import statistics
        maxclk = max(r[1] for r in rows)
        loaded = [r for r in rows if r[2] is None or r[2] > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": maxclk,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((r[2] for r in rows if r[2] is not None), default=None)}


def gpu_id_for_smi(torch, dev: int) -> str:
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev] if vis else str(dev)


def run_reference(args):
    """The oracle, as it stands, on the host cores: the reference arm."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    full = make_batch(args.seed)
    # Size each step's sample so that warm-up plus timed steps take about
    # ref_budget_s: whole rounds of one request per host thread.
    cores = oracle.default_threads()
    t1, _, _ = time_oracle(oracle_sample(full, cores))
    rounds = max(1, int(args.ref_budget_s / max(args.steps + args.warmup, 1) / max(t1, 1e-6)))
    args.ref_requests = min(full.B, cores * rounds)
    sample = oracle_sample(full, args.ref_requests)
    for _ in range(args.warmup):
        time_oracle(sample)
    times = []
    threads = None
    for _ in range(args.steps):
        dt, threads, res = time_oracle(sample)
        times.append(dt)
    t = float(np.mean(times))
    rows = sample.R_t
    value = rows / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": 256, "K": 7, "V": 151936, "temperature": 0.7,
                   "step": f"the first {args.ref_requests} requests of the batch ({rows} target rows)"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads, "kind": "oracle",
                         "sample": f"first {args.ref_requests} of 256 requests per step"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "committed_tokens_per_s": float(res.out_len.sum()) / t,
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import parity
    from speculative_decoding_verification_27_gb300 import api, build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.cuda.current_device()
    build.build_library()
    api.load()

    full = None
    if args.strong:
        # One global batch, the same on every rank; each verifies its share.
        from speculative_decoding_verification_27_gb300 import sharding
        full = make_batch(args.seed, args.batch)
        bounds = sharding.partition_requests(full.cu_draft, world, full.greedy_mask(), full.draft is not None)
        shard = sharding.shard_of(full.cu_draft, int(bounds[rank]), int(bounds[rank + 1]))
        batch = sharding.local_batch(full, shard)
    else:
        batch = make_batch(rank_seed(args.seed, rank), args.batch)
    db = parity.to_device(batch)
    B, R_t = batch.B, batch.R_t
    ws = api.new_workspace(B, R_t, batch.V)
    out_tokens = torch.full((R_t,), -1, dtype=torch.int32, device="cuda")
    out_len = torch.zeros(B, dtype=torch.int32, device="cuda")
    out_probs = torch.empty((R_t, 2), dtype=torch.float32, device="cuda")

    def step():
        api.spec_verify(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms, db.temperature,
                        db.mode, out_tokens=out_tokens, out_len=out_len, out_probs=out_probs,
                        workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if api.sv_check_status(ws) != 0:
        raise RuntimeError("device status bits set on the benchmark batch")

    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(gpu_id_for_smi(torch, dev)) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for k in range(args.steps):
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t_wall = time.perf_counter() - t_wall
    clocks = clk.summary()
    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    region_ms = max_over_ranks(starts[0].elapsed_time(ends[-1]), "cuda")
    ms_per_step = region_ms / args.steps
    mean_launch_ms = float(np.mean(per_launch_ms))

    lens = out_len.cpu().numpy()
    committed = int(lens.sum()) * world   # all ranks' batches have the same shape
    mean_len = float(lens.sum()) / B
    K = np.diff(batch.cu_draft)
    accepted = int((lens - 1).sum())
    alg_bytes = batch.algorithmic_bytes()
    value = R_t * world / (ms_per_step * 1e-3)
    strong = None
    if args.strong:
        # Strong scaling: the global batch's rows over the slowest rank's time;
        # the shards' outputs gathered in rank order must equal one verify of
        # the whole batch (rank 0 checks, on its own GPU, after the timing).
        from speculative_decoding_verification_27_gb300 import sharding
        g_tok, g_len, g_pr = out_tokens.cpu().numpy(), lens, out_probs.cpu().numpy()
        if world > 1:
            g_tok, g_len, g_pr = sharding.gather_outputs(g_tok, g_len, g_pr)
        value = full.R_t / (ms_per_step * 1e-3)
        committed = int(g_len.sum())
        mean_len = committed / full.B
        accepted = int((g_len - 1).sum())
        K = np.diff(full.cu_draft)
        if rank == 0:
            dfull = parity.to_device(full)
            w_tok, w_len, w_pr = api.spec_verify(dfull.target, dfull.draft, dfull.draft_tokens, dfull.cu_draft,
                                                 dfull.uniforms, dfull.temperature, dfull.mode)
            torch.cuda.synchronize()
            w_tok, w_len, w_pr = w_tok.cpu().numpy(), w_len.cpu().numpy(), w_pr.cpu().numpy()
            t0 = full.cu_draft[:-1].astype(np.int64) + np.arange(full.B)
            same = np.array_equal(w_len, g_len) and all(
                np.array_equal(w_tok[t0[i]:t0[i] + w_len[i]], g_tok[t0[i]:t0[i] + g_len[i]]) for i in range(full.B))
            strong = {"ranks": world, "global_requests": full.B, "global_rows": full.R_t,
                      "equal_to_one_verify_of_the_batch": bool(same),
                      "max_prob_diff": float(np.max(np.abs(w_pr - g_pr)))}
            del dfull

    peaks = measured_peaks()
    if peaks and "hbm_gbs" in peaks:
        peak, peak_src = float(peaks["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    else:
        peak, peak_src = FALLBACK_HBM_GBS, "fallback"
    achieved = alg_bytes / (mean_launch_ms * 1e-3) / 1e9
    traffic = TRAFFIC["bytes_per_launch"] if TRAFFIC["sources_sha256"] == kernel_sources_hash() else None

    # End to end through the C ABI with host buffers.
    e2e = None
    if not args.no_e2e:
        host = {k: getattr(db, k).cpu().pin_memory() for k in ("target", "draft", "draft_tokens", "cu_draft", "uniforms")}
        h_tok = torch.empty_like(out_tokens, device="cpu").pin_memory()
        h_len = torch.empty_like(out_len, device="cpu").pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = h_tok.numel() * 4 + h_len.numel() * 4

        def e2e_step():
            for k, t in host.items():
                getattr(db, k).copy_(t, non_blocking=True)
            step()
            h_tok.copy_(out_tokens, non_blocking=True)
            h_len.copy_(out_len, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, args.e2e_steps))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, "cuda")
        e2e = {"value": R_t * world / (e_ms * 1e-3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms, "steps": n_e2e}

    # CPU baseline (rank 0, N=1): the oracle's own work on the step's batch,
    # outputs only, timed over a few calls on all host threads. Then, untimed,
    # a parity spot check: the oracle with its per-row probabilities against
    # the GPU's outputs of the last timed step.
    cpu = None
    spot = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = batch if args.cpu_requests >= B else oracle_sample(batch, args.cpu_requests)
        times = []
        for _ in range(args.cpu_reps):
            dt, threads, _ = time_oracle(sample, diagnostics=False)
            times.append(dt)
        dt = float(np.mean(times))
        cpu = {"value": sample.R_t / dt, "unit": "rows/s", "cores": threads, "kind": "oracle",
               "sample": (f"{'the whole batch' if sample.B == B else f'first {sample.B} of {B} requests'} "
                          f"({sample.R_t} target rows, {sample.R_d} draft rows), {args.cpu_reps} calls, "
                          "all host threads, the step's outputs only")}
        _, _, res = time_oracle(sample, diagnostics=True)
        rt = sample.R_t
        g_tok, g_len, g_pr = out_tokens.cpu().numpy(), lens, out_probs.cpu().numpy()
        rep = parity.compare(sample, (g_tok[:rt], g_len[:sample.B], g_pr[:rt]), res,
                             flag_budget=parity.FLAG_BUDGET)
        spot = rep.as_dict()

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "strong" if args.strong else "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD if args.batch == 256 else WORKLOAD.replace("B=256", f"B={args.batch}"),
                   "B": args.batch, "K": 7, "V": batch.V, "temperature": batch.temperature,
                   "logits": "bf16", "rows_per_step": R_t, "draft_rows_per_step": batch.R_d,
                   "algorithmic_bytes_per_step": alg_bytes,
                   "l2": "inputs 1.17 GB > 129 MB L2 per step: no flush needed",
                   "parallelism": (f"one batch split by requests over {world} rank(s); outputs gathered after "
                                   "the timed region" if args.strong else
                                   f"requests sharded, {world} rank(s), no collective")},
        "committed_tokens_per_s": committed / (ms_per_step * 1e-3),
        "hbm_gbs": achieved,
        "acceptance": {"draft_acceptance_rate": accepted / int(K.sum()),
                       "mean_acceptance_length": mean_len},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                     "traffic_source": TRAFFIC["profile"] if traffic else None,
                     "kernel": "verify_kernel", "mean_launch_ms": mean_launch_ms,
                     "algorithmic_bytes_per_launch": alg_bytes},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "parity_spot_check": spot,
        "wall_s_timed_region": t_wall,
    }
    if strong is not None:
        line["strong_check"] = strong
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# The other configurations (one JSON line each with --workload NAME). Their
# working sets are small enough to sit in L2, so each timed launch follows a
# write of a 256 MB buffer and a read of another (each larger than the 129 MB
# L2), outside its events.
# ---------------------------------------------------------------------------
EXTRA_WORKLOADS = {
    "verify_b1": "sampling verify B=1 K=4 V=32000 fp32 T=1.0, z_t ~ N(0,2^2), z_d = z_t + N(0,0.5^2), "
                 "x̂ ~ q; 64 rounds of fresh inputs cycled",
    "greedy_b64": "strict verify B=64 K=5 V=128256 bf16, z ~ N(0,3^2) with a planted argmax margin, "
                  "x̂ = argmax w.p. 0.7",
    "ngram_b128": "ngram_propose over 128 histories x 8192 int32 tokens (V=32000) with planted copies "
                  "covering 30%, n=3, up to 5 tokens",
    "suffix_b128": "suffix_propose (frequency-ranked, min_share 0.5, up to 256 voters) over the same 128 "
                   "histories x 8192 int32 tokens, n=3, up to 5 tokens",
    "onehot_b128": "verify of the n-gram proposals (one-hot q), fp32 z ~ N(0,2^2), V=32000, T=1.0",
    "ragged_b512": "ragged mixed verify B=512 K_b~U{1..8} V=256000 bf16 T=1.0, half greedy requests",
    "metrics_b512": "acceptance statistics of 512 verify rounds (K_b~U{1..8}) added to a device "
                    "counter block",
    "topkp_b256": "top-k 50 / top-p 0.9 filtered sampling verify on the benchmark batch (B=256 K=7 "
                  "V=151936 bf16 T=0.7, peaked rank-score rows)",
    "vshard_b256x2": "vocabulary-sharded verify of the benchmark batch (B=256 K=7 V=151936 bf16 T=0.7, peaked "
                     "rows) split over 2 vocabulary shards held by one process on one GPU (shard kernels and "
                     "the local exchanges; no interconnect)",
    "candidates_b64x4": "64 requests x 4 draft candidates of 5 tokens (V=32000 bf16, T=1.0), verified as "
                        "256 requests, then one kept per request by its selection uniform (lossless rule)",
}
FILTER_K, FILTER_P = 50, 0.9
SUFFIX_SHARE, SUFFIX_OCC = 0.5, 256


def _extra_setup(name, seed):
    """(description dict, host inputs, device step(), units, unit, bytes, flush, oracle_fn, check_fn)."""
    import numpy as np
    import torch

    import parity
    from speculative_decoding_verification_27_gb300 import api
    from speculative_decoding_verification_27_gb300 import workloads as W

    if name in ("ngram_b128", "suffix_b128"):
        import oracle
        suffix = name == "suffix_b128"
        nb = W.config4_histories(seed=seed)
        h = torch.from_numpy(nb.histories).cuda()
        hl = torch.from_numpy(nb.hist_len).cuda()
        out = torch.empty((h.shape[0], nb.max_tokens), dtype=torch.int32, device="cuda")
        cnt = torch.empty(h.shape[0], dtype=torch.int32, device="cuda")
        nn = torch.empty(h.shape[0], dtype=torch.int32, device="cuda")
        host = {"h": (h, torch.from_numpy(nb.histories).pin_memory()),
                "hl": (hl, torch.from_numpy(nb.hist_len).pin_memory())}
        outs = [out, cnt, nn]

        def step():
            if suffix:
                api.suffix_propose(h, hl, nb.min_n, nb.max_n, nb.max_tokens, SUFFIX_SHARE, SUFFIX_OCC,
                                   out_tokens=out, out_count=cnt, out_n=nn)
            else:
                api.ngram_propose(h, hl, nb.min_n, nb.max_n, nb.max_tokens, out_tokens=out, out_count=cnt,
                                  out_n=nn)

        def oracle_fn():
            t = time.perf_counter()
            if suffix:
                o = oracle.suffix_propose(nb.histories, nb.hist_len, nb.min_n, nb.max_n, nb.max_tokens,
                                          min_share=SUFFIX_SHARE, max_occ=SUFFIX_OCC)
            else:
                o = oracle.ngram_propose(nb.histories, nb.hist_len, nb.min_n, nb.max_n, nb.max_tokens)
            return time.perf_counter() - t, 1, o  # the oracle's proposers are single-threaded

        def check(o):
            return {"histories": int(h.shape[0]),
                    "bit_exact": bool(np.array_equal(cnt.cpu().numpy(), o[1])
                                      and np.array_equal(nn.cpu().numpy(), o[2])
                                      and np.array_equal(out.cpu().numpy(), np.where(
                                          np.arange(nb.max_tokens)[None] < o[1][:, None], o[0], -1)))}
        desc = {"B": int(h.shape[0]), "L": int(nb.histories.shape[1]), "n": nb.max_n,
                "max_tokens": nb.max_tokens}
        if suffix:
            desc.update(min_share=SUFFIX_SHARE, max_occ=SUFFIX_OCC)
        return (desc, host, outs, step, int(h.shape[0]), "histories/s", int(nb.histories.nbytes),
                True, oracle_fn, check)

    if name == "metrics_b512":
        import oracle
        rng = np.random.default_rng(seed)
        B = 512
        K = rng.integers(1, 9, size=B)
        cu = np.concatenate([[0], np.cumsum(K)]).astype(np.int32)
        lens = rng.integers(1, K + 2).astype(np.int32)
        d_cu, d_len = torch.from_numpy(cu).cuda(), torch.from_numpy(lens).cuda()
        m = api.new_metrics()
        host = {"cu": (d_cu, torch.from_numpy(cu).pin_memory()),
                "len": (d_len, torch.from_numpy(lens).pin_memory())}

        def step():
            api.sv_accumulate_metrics(d_cu, d_len, m)

        def oracle_fn():
            t = time.perf_counter()
            o = oracle.acceptance_metrics(cu, lens)
            return time.perf_counter() - t, 1, o

        def check(o):
            m1 = api.new_metrics()
            api.sv_accumulate_metrics(d_cu, d_len, m1)
            g = api.metrics_dict(m1)
            return {"rounds": B, "bit_exact": all(g[k] == o[k] for k in o)}
        return ({"B": B, "K": "U{1..8}"}, host, [m], step, B, "rounds/s", int(cu.nbytes + lens.nbytes),
                True, oracle_fn, check)

    if name == "verify_b1":
        batches = [W.config1(seed=seed, round_index=r) for r in range(64)]
    elif name == "greedy_b64":
        batches = [W.config2(seed=seed)]
    elif name == "onehot_b128":
        import oracle
        nb = W.config4_histories(seed=seed)
        o = oracle.ngram_propose(nb.histories, nb.hist_len, nb.min_n, nb.max_n, nb.max_tokens)
        batches = [W.config4_verify(seed=seed, proposals=o[0], counts=o[1])]
    elif name == "ragged_b512":
        batches = [W.config5(seed=seed)]
    elif name in ("topkp_b256", "vshard_b256x2"):
        batches = [W.config3(seed=seed)]
    elif name == "candidates_b64x4":
        batches = [W.gaussian_sampling(seed=seed, B=256, K=5, V=32000, sigma=2.0, draft_sigma=0.5, T=1.0,
                                       dtype="bf16")]
    else:
        raise SystemExit(f"unknown workload {name}")
    dbs = [parity.to_device(b) for b in batches]
    b0 = batches[0]
    ws = api.new_workspace(max(b.B for b in batches), max(b.R_t for b in batches), b0.V)
    R_t = max(b.R_t for b in batches)
    ot = torch.full((R_t,), -1, dtype=torch.int32, device="cuda")
    ol = torch.zeros(max(b.B for b in batches), dtype=torch.int32, device="cuda")
    op = torch.empty((R_t, 2), dtype=torch.float32, device="cuda")
    k = [0]
    greedy_only = name == "greedy_b64"
    filtered = name == "topkp_b256"
    sharded = name == "vshard_b256x2"
    if sharded:
        from speculative_decoding_verification_27_gb300 import vshard
        bounds = vshard.split_vocab(b0.V, 2)
        d0_ = dbs[0]
        shards = [vshard.Shard(d0_.target[:, a:c].contiguous(), d0_.draft[:, a:c].contiguous(), a)
                  for a, c in zip(bounds[:-1], bounds[1:])]
    cands = name == "candidates_b64x4"
    if cands:
        cu_cand = torch.arange(0, 257, 4, dtype=torch.int32, device="cuda")
        u_sel = torch.from_numpy(W.selection_uniforms(64, seed=seed)).cuda()
        best = torch.empty(64, dtype=torch.int32, device="cuda")
        best_len = torch.empty(64, dtype=torch.int32, device="cuda")
    if filtered:
        ws = torch.zeros(api.spec_verify_filtered_workspace_size(b0.B, b0.R_t, b0.V), dtype=torch.uint8,
                         device="cuda")

    def step():
        db = dbs[k[0] % len(dbs)]
        k[0] += 1
        if filtered:
            api.spec_verify_filtered(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                                     db.temperature, FILTER_K, FILTER_P, db.mode, out_tokens=ot, out_len=ol,
                                     out_probs=op, workspace=ws)
        elif sharded:
            vshard.spec_verify_vsharded(shards, b0.V, db.draft_tokens, db.cu_draft, db.uniforms, db.temperature,
                                        db.mode, out_tokens=ot, out_len=ol, out_probs=op)
        elif greedy_only:
            api.spec_verify_greedy(db.target, db.draft_tokens, db.cu_draft, out_tokens=ot, out_len=ol,
                                   workspace=ws)
        else:
            api.spec_verify(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                            db.temperature, db.mode, out_tokens=ot, out_len=ol, out_probs=op,
                            workspace=ws)
            if cands:
                api.sv_select_candidates(cu_cand, ol, api.SV_SELECT_UNIFORM, u_sel, best=best, best_len=best_len)

    if sharded:
        # The sharded step is a dozen small launches and tensor ops with no
        # host synchronisation: it is captured once in a CUDA graph and the
        # graph replayed, as a serving loop would run it; the timed region
        # then holds the device's work, not the launch overhead between ops.
        raw_step = step
        for _ in range(3):
            raw_step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            raw_step()
        torch.cuda.synchronize()

        def step():
            graph.replay()

    d0 = dbs[0]
    host = {f: (getattr(d0, f), getattr(d0, f).cpu().pin_memory())
            for f in ("target", "draft", "draft_tokens", "cu_draft", "uniforms") if getattr(d0, f) is not None}
    if sharded:  # the step reads the shards' slices, not the whole matrices
        for f in ("target", "draft"):
            del host[f]
        for j, sh in enumerate(shards):
            host[f"target{j}"] = (sh.target, sh.target.cpu().pin_memory())
            host[f"draft{j}"] = (sh.draft, sh.draft.cpu().pin_memory())
    sample = b0 if b0.B <= 64 else oracle_sample(b0, 64)

    def oracle_run(diagnostics):
        if filtered:
            import oracle
            threads = min(oracle.default_threads(), sample.B)
            res = oracle.spec_verify(sample.target, sample.draft, sample.draft_tokens, sample.cu_draft,
                                     sample.uniforms, sample.temperature, sample.mode, threads,
                                     diagnostics=diagnostics, top_k=FILTER_K, top_p=FILTER_P)
            return threads, res
        _, threads, res = time_oracle(sample, diagnostics=diagnostics)
        return threads, res

    def oracle_fn():
        # Timed: the step's outputs only. Untimed: the run with per-row
        # probabilities that the spot check compares.
        reps = 200 if name == "verify_b1" else 3
        t = time.perf_counter()
        for _ in range(reps):
            threads, _ = oracle_run(False)
        dt = (time.perf_counter() - t) / reps
        return dt, threads, oracle_run(True)[1]

    def check(res):
        k[0] = 0
        step()
        torch.cuda.synchronize()
        g = (ot.cpu().numpy()[:sample.R_t], ol.cpu().numpy()[:sample.B],
             op.cpu().numpy()[:sample.R_t] if not greedy_only else np.full((sample.R_t, 2), -1.0, np.float32))
        return parity.compare(sample, g, res).as_dict()

    units = sum(b.R_t for b in batches) / len(batches)
    nbytes = sum(b.algorithmic_bytes() for b in batches) / len(batches)
    desc = {"B": b0.B, "V": b0.V, "R_t": b0.R_t, "R_d": b0.R_d, "logits": "bf16" if b0.elem_bytes == 2 else "fp32",
            "temperature": b0.temperature, "input_sets": len(batches)}
    if filtered:
        desc.update({"top_k": FILTER_K, "top_p": FILTER_P})
    # Kernels of this library per step: the filtered step runs the one-warp
    # and CTA threshold kernels, the filtered commit and the verify kernel;
    # the sharded step two statistics kernels per shard, the decisions, a
    # mass and a draw kernel per shard and the finish.
    desc["launches_per_step"] = {"topkp_b256": 4, "vshard_b256x2": 10, "candidates_b64x4": 2}.get(name, 1)
    outs = [ot, ol] if not cands else [ot, ol, best, best_len]
    if sharded:
        desc.update({"shards": 2, "shard_bounds": bounds, "launch": "the step captured once in a CUDA graph, replayed"})
    return desc, host, outs, step, units, "rows/s", nbytes, name not in ("ragged_b512", "topkp_b256", "vshard_b256x2"), \
        oracle_fn, check


def run_extra(args):
    import numpy as np
    import torch

    from speculative_decoding_verification_27_gb300 import api, build
    torch.cuda.set_device(0)
    build.build_library()
    api.load()
    (desc, host, outs, step, units, unit, nbytes, flush, oracle_fn,
     check) = _extra_setup(args.workload, args.seed)
    # Flush: write one 256 MB buffer, then read another, so that L2 holds
    # clean lines only and the timed launch pays no write-back of the flush.
    l2w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if flush else None
    l2r = torch.ones(64 << 20, dtype=torch.float32, device="cuda") if flush else None
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    n = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    with ClockSampler(gpu_id_for_smi(torch, 0)) as clk:
        torch.cuda.synchronize()
        for i in range(n):
            if flush:
                l2w.zero_()
                l2r.sum()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    clocks = clk.summary()
    ms = float(np.mean([a.elapsed_time(b) for a, b in zip(starts, ends)]))
    peaks = measured_peaks()
    peak = float(peaks["hbm_gbs"]) if peaks and "hbm_gbs" in peaks else FALLBACK_HBM_GBS
    achieved = nbytes / (ms * 1e-3) / 1e9

    # End to end: the step's inputs from pinned host memory, the call, the
    # outputs back to the host.
    h_outs = [o.cpu().pin_memory() for o in outs]
    h2d = sum(hv.numel() * hv.element_size() for _, hv in host.values())
    d2h = sum(o.numel() * o.element_size() for o in outs)

    def e2e_step():
        for dv, hv in host.values():
            dv.copy_(hv, non_blocking=True)
        step()
        for o, hcopy in zip(outs, h_outs):
            hcopy.copy_(o, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    n_e2e = max(3, min(n, args.e2e_steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1) / n_e2e

    dt, threads, res = oracle_fn()
    spot = check(res)
    line = {
        "metric": METRIC, "value": units / (ms * 1e-3), "unit": unit, "n_gpus": 1, "steps": n,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "i32" if args.workload in ("ngram_b128", "suffix_b128", "metrics_b512") else "f32",
        "data": "synthetic",
        "config": dict({"workload": EXTRA_WORKLOADS[args.workload],
                        "l2": "before each timed launch a 256 MB buffer is written and another "
                              "256 MB read (flush, clean lines)" if flush
                        else "inputs larger than L2: no flush"}, **desc),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "note": {"ngram_b128": "latency-bound: one CTA per history",
                              "suffix_b128": "latency-bound: one CTA per history",
                              "metrics_b512": "latency-bound: 4 KB of inputs"}.get(args.workload)},
        "e2e": {"value": units / (e_ms * 1e-3), "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e_ms},
        "gpu_launches": n * desc.get("launches_per_step", 1),
        "clocks": clocks,
        "cpu_baseline": {"value": (units if args.workload in ("ngram_b128", "suffix_b128", "verify_b1", "greedy_b64",
                                                            "onehot_b128", "metrics_b512")
                                   else spot["rows"]) / dt,
                         "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": {"ragged_b512": "64 of 512 requests", "topkp_b256": "64 of 256 requests",
                                    "vshard_b256x2": "64 of 256 requests (whole vocabulary)",
                                    "candidates_b64x4": "64 of 256 candidates (verify only)"}.get(
                                        args.workload, "the whole step")},
        "parity_spot_check": spot,
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=3)
    ap.add_argument("--batch", type=int, default=256,
                    help="requests per step (256 is the benchmark workload; smaller only for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-requests", type=int, default=256,
                    help="requests of the batch the CPU baseline times (default: all)")
    ap.add_argument("--cpu-reps", type=int, default=3)
    ap.add_argument("--ref-budget-s", type=float, default=100.0)
    ap.add_argument("--strong", action="store_true",
                    help="split one global batch over the ranks (strong scaling) instead of one batch per rank")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="verify_b256", choices=["verify_b256", *EXTRA_WORKLOADS],
                    help="verify_b256 is the benchmark workload; the others print their own line")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "verify_b256":
        return run_extra(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
