#!/usr/bin/env python3
"""Benchmark of the speculative-sampling verification step.

Workload (the headline chain configuration): B=64 requests, K=6 drafts,
V=128256, bf16 logits; target ~ N(0, 3^2) with a Zipf(1.1) boost on token ids,
draft = target + N(0, 1.5^2); even requests greedy (t = 0), odd ones t = 1;
seeded synthetic data (speculative_decoding_verification_63_gb300.workloads).

One step = one call of sv_verify_chain on one batch: the whole verification
(row reductions, accept tests, prefix scan, residual / bonus draws).  Inputs
are 213 MB per batch (larger than the 129 MB L2) and two batches rotate, so
every step reads its logits from HBM.

Metric: verify rounds per second, one round = one request's verification of
its K drafts (B rounds per step).  The JSON line also carries tokens
verified per second, logit GB/s and the roofline of the kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--kernel-only]     (eager launches only, for ncu runs)

Under torchrun (WORLD_SIZE > 1) every rank runs an independent replica on
its own GPU (the step does not shard); value = rounds of all ranks / the
slowest rank's time.  --impl reference times the fp64 CPU oracle on the
host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

WORKLOAD = 3          # headline chain workload in workloads.CHAIN_SHAPES
N_SETS = 2            # rotating input batches (each larger than L2)
GRAPH_LEN = 100       # launches per captured CUDA graph
METRIC = "verify rounds/s & logit GB/s vs HBM peak (B=64, K=6, V=128256 bf16)"
UNIT = "verify rounds/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 20000 launches; reference arm: 256 rounds)")
    ap.add_argument("--warmup", type=int, default=None,
                    help="untimed steps (default: 50; reference arm: 3)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--kernel-only", action="store_true",
                    help="profiling runs: eager launches only (no graphs, no end-to-end leg, "
                         "no CPU baseline, no clock sampling)")
    return ap.parse_args()


# ------------------------------------------------------------ distribution

class Dist:
    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, device_ok: bool):
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("nccl" if device_ok else "gloo")
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# -------------------------------------------------------------- helpers

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# the sources the chain verification kernel is compiled from
CHAIN_KERNEL_SOURCES = ("sv_device.cuh", "sv_rowpass.cuh", "sv_kernel.cuh", "sv_chain.cuh",
                        "sv_topk.cuh")


def source_hash() -> str:
    """Hash of the chain kernel's CUDA sources, to tell whether a stored ncu
    figure is current.  Comments and blank lines are left out, so editing a
    comment keeps the figure; any change to the code drops it."""
    import re
    d = os.path.join(ROOT, "speculative_decoding_verification_63_gb300", "csrc")
    h = hashlib.sha256()
    for name in CHAIN_KERNEL_SOURCES:
        with open(os.path.join(d, name)) as f:
            code = [re.sub(r"//.*", "", line).rstrip() for line in f]
        h.update(name.encode() + b"\0" + "\n".join(l for l in code if l).encode())
    return h.hexdigest()[:16]


def stored_traffic():
    """DRAM bytes per launch of the verification kernel from the committed ncu
    summary, if it was taken on the current sources; else None."""
    path = os.path.join(ROOT, "profiles", "verify_chain_b64_k6_v128256.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_hash") != source_hash():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(torch):
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:  # noqa: BLE001 -- older torch: sample every GPU, take the lines we get
        return None


def config_dict(inp):
    return {"workload": "chain verify B=64 K=6 V=128256 bf16, half greedy (t=0) / half t=1",
            "B": inp["B"], "K": inp["K"], "V": inp["V"], "logits": "bf16",
            "parallelism": "replicas", "l2": f"{N_SETS} rotating input batches of "
            f"{(inp['target'].nbytes + inp['draft'].nbytes) / 1e6:.0f} MB each (> 129 MB L2)"}


def _make_set(s: int):
    from speculative_decoding_verification_63_gb300 import workloads as wl
    return wl.make_chain(WORKLOAD, seed=wl.SEED_BASE + WORKLOAD + 100 * s)


def make_inputs():
    """The rotating batches, generated in parallel worker processes (spawned,
    before this process touches the GPU)."""
    import multiprocessing as mp
    with mp.get_context("spawn").Pool(N_SETS) as pool:
        return pool.map(_make_set, range(N_SETS))


# ---------------------------------------------------------- CPU oracle arm

def time_oracle(inp, budget_s: float, max_steps: int | None = None):
    """Full verification steps of the oracle on batch `inp`, repeated until
    budget_s of wall time or max_steps steps (at least one).  Returns
    (steps, seconds)."""
    import oracle
    lib = oracle.load()
    oracle.verify_chain_inputs(inp, requests=[0, 1], lib=lib)  # warm (page in, build)
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle.verify_chain_inputs(inp, lib=lib)
        steps += 1
        el = time.perf_counter() - t0
        if (max_steps is not None and steps >= max_steps) or (max_steps is None and el >= budget_s):
            return steps, el


def run_reference(args, dist):
    """The reference arm: the fp64 CPU oracle, as it stands, on one host
    core.  One step is one request round of the headline batch (requests
    taken in order, so greedy and sampled rounds alternate as in the batch);
    W untimed steps, then exactly K timed ones.  Without --steps/--warmup
    the arm runs 256 timed rounds after 3 warm-up rounds (a few seconds)."""
    if dist.rank != 0:
        return 0
    import oracle
    lib = oracle.load()
    inp = _make_set(0)
    B = inp["B"]
    keys = ("target", "draft", "tokens", "temperature", "uniforms", "num_drafts", "top_k")
    rounds = [{k: inp[k][b:b + 1] for k in keys} for b in range(B)]  # views, no copies

    def step(i):
        r = rounds[i % B]
        oracle.verify_chain(r["target"], r["draft"], r["tokens"], r["temperature"],
                            r["uniforms"], num_drafts=r["num_drafts"], top_k=r["top_k"], lib=lib)

    K = args.steps if args.steps is not None else 256
    W = max(args.warmup if args.warmup is not None else 3, 3)
    for i in range(W):
        step(i)
    t0 = time.perf_counter()
    for i in range(K):
        step(W + i)
    el = time.perf_counter() - t0
    value = K / el
    sample = (f"{K} request rounds of the headline batch, one per step, requests in batch "
              "order (half greedy, half sampled), fp64 C, one host thread")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": K,
            "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(inp), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- GPU arm

def run_ours(args, dist):
    import torch
    import speculative_decoding_verification_63_gb300 as sv
    from speculative_decoding_verification_63_gb300 import _binding, workloads as wl

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the verification runs only on the GPU)")
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    sv.lib()  # fail loudly when the extension is missing

    sets = make_inputs()
    inp0 = sets[0]
    B, K, V = inp0["B"], inp0["K"], inp0["V"]
    alg_bytes = wl.chain_algorithmic_bytes(inp0)
    assert all(wl.chain_algorithmic_bytes(s) == alg_bytes for s in sets)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
                torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    keys = ("target", "draft", "tokens", "temperature", "uniforms", "num_drafts")
    dsets = [{k: to_dev(s[k]) for k in keys} for s in sets]
    outs = [dict(out_tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                 out_len=torch.empty(B, dtype=torch.int32, device=dev),
                 accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                 p_at=torch.empty((B, K), dtype=torch.float32, device=dev),
                 q_at=torch.empty((B, K), dtype=torch.float32, device=dev))
            for _ in range(N_SETS)]
    need = sv.sv_chain_workspace_bytes(B, K, V, sv.dtype_code(dsets[0]["target"]), 0)
    ws = sv.workspace(need, dev, "bench")

    def step(i):
        d, o = dsets[i % N_SETS], outs[i % N_SETS]
        _binding.sv_verify_chain(d["target"], d["draft"], d["tokens"], d["temperature"],
                                 d["uniforms"], o["out_tokens"], o["out_len"],
                                 o["accept_len"], ws, num_drafts=d["num_drafts"],
                                 p_at_draft=o["p_at"], q_at_draft=o["q_at"])

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize(dev)
    sv.check_device_errors(ws)

    if args.kernel_only:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(args.steps):
                step(i)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        sv.check_device_errors(ws)
        ms = e0.elapsed_time(e1)
        if dist.rank == 0:
            print(json.dumps({"kernel_only": True, "steps": args.steps,
                              "ms_per_step": ms / max(args.steps, 1),
                              "logit_gbs": alg_bytes * args.steps / (ms / 1e3) / 1e9}),
                  flush=True)
        return 0

    # parity spot check of the timed configuration: every batch against the oracle
    # on a sample of requests (full batch for set 0 would take seconds of CPU)
    if dist.rank == 0:
        import oracle
        for si in range(N_SETS):
            with torch.cuda.stream(stream):
                step(si)
            torch.cuda.synchronize(dev)
            req = np.arange(0, B, 16) + si
            ref = oracle.verify_chain_inputs(sets[si], requests=req)
            got = outs[si]["out_tokens"].cpu().numpy()[req]
            ok = ref["margin"] >= 1e-6
            if not np.array_equal(got[ok], ref["out_tokens"][ok]):
                raise SystemExit("bench.py: parity check against the oracle failed")

    # CUDA graphs of GRAPH_LEN launches (rotating the batches), exactly K launches timed
    K_steps = args.steps
    L = max(1, min(GRAPH_LEN, K_steps))
    graphs = []
    for length in (L, K_steps % L):
        if length == 0:
            graphs.append(None)
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(length):
                    step(i)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for g in graphs:
            if g is not None:
                g.replay()
    torch.cuda.synchronize(dev)
    sv.check_device_errors(ws)

    sampler = ClockSampler(gpu_uuid(torch))
    dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)  # let the sampler come up before the timed region
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K_steps // L):
            graphs[0].replay()
        if graphs[1] is not None:
            graphs[1].replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms_local = e0.elapsed_time(e1)
    dist.barrier()
    ms = dist.max(ms_local)
    sv.check_device_errors(ws)

    launch_s = ms_local / 1e3 / K_steps
    rounds_per_s = dist.world * B * K_steps / (ms / 1e3)
    tokens_verified = int(inp0["num_drafts"].sum())
    peak, peak_kind = hbm_peak()
    achieved = alg_bytes / launch_s / 1e9
    traffic = stored_traffic()

    # end to end through the public API: pinned host inputs -> device, the
    # call, results -> pinned host, every step
    e2e_steps = max(10, min(K_steps, 300))
    host = []
    for s in sets:
        h = {}
        for k in keys:
            a = np.ascontiguousarray(s[k])
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
            h[k] = t.pin_memory()
        host.append(h)
    h2d = sum(int(host[0][k].numel() * host[0][k].element_size()) for k in keys)
    res_host = [torch.empty((B, K + 1), dtype=torch.int32).pin_memory(),
                torch.empty(B, dtype=torch.int32).pin_memory(),
                torch.empty(B, dtype=torch.int32).pin_memory()]
    d2h = sum(int(t.numel() * t.element_size()) for t in res_host)

    def e2e_step(i):
        h = host[i % N_SETS]
        d = {k: h[k].to(dev, non_blocking=True) for k in keys}
        d["target"] = d["target"].view(torch.bfloat16)
        d["draft"] = d["draft"].view(torch.bfloat16)
        out = sv.verify_chain(d["target"], d["draft"], d["tokens"], d["temperature"],
                              d["uniforms"], num_drafts=d["num_drafts"], ws=ws)
        res_host[0].copy_(out["out_tokens"], non_blocking=True)
        res_host[1].copy_(out["out_len"], non_blocking=True)
        res_host[2].copy_(out["accept_len"], non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
    torch.cuda.synchronize(dev)
    dist.barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_s = dist.max(time.perf_counter() - t0)
    sv.check_device_errors(ws)
    e2e_value = dist.world * B * e2e_steps / e2e_s

    cpu = None
    if dist.rank == 0 and dist.world == 1:
        n, el = time_oracle(sets[0], 10.0)
        cpu = {"value": B * n / el, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n} full steps of one headline batch ({n * B} request rounds), "
                         "fp64 C, one host thread, about 10 s"}

    if dist.rank == 0:
        line = {"metric": METRIC, "value": rounds_per_s, "unit": UNIT, "n_gpus": dist.world,
                "steps": K_steps, "warmup": max(args.warmup, 3), "ms_per_step": ms / K_steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic", "config": config_dict(inp0),
                "tokens_verified_per_s": dist.world * tokens_verified * K_steps / (ms / 1e3),
                "logit_gbs": dist.world * alg_bytes * K_steps / (ms / 1e3) / 1e9,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                             "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                             "traffic": traffic, "algorithmic_bytes": alg_bytes},
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "steps": e2e_steps},
                "gpu_launches": K_steps,
                "clocks": clocks}
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    dist = Dist()
    if args.impl == "reference":
        dist.init(device_ok=False)
        rc = run_reference(args, dist)
    else:
        args.steps = 20000 if args.steps is None else args.steps
        args.warmup = 50 if args.warmup is None else args.warmup
        dist.init(device_ok=True)
        rc = run_ours(args, dist)
    dist.close()
    return rc


if __name__ == "__main__":
    sys.exit(main())
