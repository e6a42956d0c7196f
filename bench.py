#!/usr/bin/env python3
"""Benchmark of the speculative-sampling verification step.

Workloads (seeded synthetic data, speculative_decoding_verification_63_gb300
.workloads; seed 63000 + workload + 100 s for input set s):

  3 (default, the headline)  chain B=64, K=6, V=128256 bf16; target ~ N(0,
      3^2) with a Zipf(1.1) boost on token ids, draft = target + N(0, 1.5^2);
      even requests greedy (t = 0), odd ones t = 1.
  2  chain B=1, K=4, V=32000 bf16, peaked target, t = 0.8 (latency).
  4  token tree, B=16 trees of 32 nodes, depth <= 5, branching <= 3,
     V=32000 bf16, multi-step speculative sampling, t = 0.8.
  5  chain B=256, K=8, V=152064 bf16, t = 0.7, top-k 50 on p and q.

One step = one call of the library on one batch: the whole verification
(row reductions, accept tests, prefix scan, residual / bonus draws).  The
device holds a pool of batches larger than the 129 MB L2 and the steps
rotate over it, so every step reads its logits from HBM.

Metric: verify rounds per second, one round = one request's verification
(B rounds per step); the line also carries steps/s, us/step, tokens
verified/s, logit GB/s, the roofline of the kernel, the near-boundary counts
of the timed batches against the oracle, the oracle timed on the host
cores (one thread and all cores) and an end-to-end figure through the
public API with host buffers.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload 2|3|4|5] [--kernel-only]

Under torchrun (WORLD_SIZE > 1) every rank runs an independent replica on
its own GPU (the step does not shard); value = rounds of all ranks / the
slowest rank's time.  --impl reference times the fp64 CPU oracle on the
host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

GRAPH_LEN = 100       # launches per captured CUDA graph
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 << 20
NEAR = 1e-6           # relative distance from a decision boundary counted as near

HEADLINE_METRIC = "verify rounds/s & logit GB/s vs HBM peak (B=64, K=6, V=128256 bf16)"
UNIT = "verify rounds/s"


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 20000 launches; reference arm: 256 rounds)")
    ap.add_argument("--warmup", type=int, default=None,
                    help="untimed steps (default: 50; reference arm: 3)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", type=int, choices=(2, 3, 4, 5), default=3)
    ap.add_argument("--kernel-only", action="store_true",
                    help="profiling runs: eager launches only (no graphs, no end-to-end leg, "
                         "no CPU baseline, no clock sampling, no variants)")
    return ap.parse_args(argv)


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


# the sources each workload's dominant kernel is compiled from (the stored
# ncu figures are keyed to them): the persistent chain kernel, the top-k
# pass, the tree walk
KERNEL_SOURCES = {
    "chain": ("sv_device.cuh", "sv_rowpass.cuh", "sv_kernel.cuh", "sv_chain.cuh"),
    "topk": ("sv_device.cuh", "sv_rowpass.cuh", "sv_topk.cuh"),
    "tree": ("sv_device.cuh", "sv_rowpass.cuh", "sv_cluster.cuh", "sv_treewalk.cuh"),
}


def strip_comments(text: str) -> str:
    """C/C++ source without comments and blank lines (string literals in the
    kernels hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    lines = [re.sub(r"//.*", "", line).rstrip() for line in text.splitlines()]
    return "\n".join(line for line in lines if line)


def source_hash(kind: str = "chain") -> str:
    """Hash of a kernel's CUDA sources, to tell whether a stored ncu figure
    is current.  Comments and blank lines are left out, so editing a comment
    keeps the figure; any change to the code drops it."""
    d = os.path.join(ROOT, "speculative_decoding_verification_63_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(d, name)) as f:
            code = strip_comments(f.read())
        h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def stored_traffic(profile: str, kind: str = "chain"):
    """DRAM bytes per launch of a kernel from a committed ncu summary
    (profiles/<profile>.md), if it was taken on the current sources; else
    None."""
    path = os.path.join(ROOT, "profiles", profile + ".md")
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
    if vals.get("source_hash") != source_hash(kind):
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


# ------------------------------------------------------------ workloads
#
# A workload is a pool of requests held on the device ("pool", Btot of
# them), verified B at a time: step i takes window i % (Btot / B).  Every
# window's outputs go to that window's rows of pool-sized output arrays, so
# after one pass over the windows the outputs of every request are there to
# compare with the oracle.

def _gen_chain(args):
    from speculative_decoding_verification_63_gb300 import workloads as wl
    cfg, seed, B, greedy = args
    return wl.make_chain(cfg, seed=seed, B=B, greedy=greedy)


def _gen_tree(args):
    from speculative_decoding_verification_63_gb300 import workloads as wl
    seed, B = args
    return wl.make_tree(seed=seed, B=B)


def _concat(parts: list[dict]) -> dict:
    out = dict(parts[0])
    for k, v in parts[0].items():
        if isinstance(v, np.ndarray):
            out[k] = np.concatenate([p[k] for p in parts], axis=0)
    out["B"] = sum(p["B"] for p in parts)
    return out


def _slice(inp: dict, lo: int, hi: int) -> dict:
    out = dict(inp)
    for k, v in inp.items():
        if isinstance(v, np.ndarray):
            out[k] = v[lo:hi]
    out["B"] = hi - lo
    return out


class Workload:
    """Sizes, pool and bookkeeping of one benchmark workload."""

    def __init__(self, key: int):
        from speculative_decoding_verification_63_gb300 import workloads as wl
        self.key = key
        self.kind = "tree" if key == 4 else "chain"
        self.kernel = {4: "tree", 5: "topk"}.get(key, "chain")  # the dominant kernel
        S = wl.SEED_BASE + key
        if key == 3:
            self.B = 64
            self.jobs = [("chain", (3, S + 100 * s, None, None)) for s in range(2)]
            self.name = ("chain verify B=64 K=6 V=128256 bf16, half greedy (t=0) / half t=1")
            self.metric = HEADLINE_METRIC
            self.profile = "verify_chain_b64_k6_v128256"
        elif key == 2:
            self.B = 1
            self.jobs = [("chain", (2, S, 512, None))]
            self.name = "chain verify B=1 K=4 V=32000 bf16, t=0.8 (latency)"
            self.metric = ("verify rounds/s & latency (chain B=1, K=4, V=32000 bf16)")
            self.profile = "verify_chain_b1_k4_v32000"
        elif key == 5:
            self.B = 256
            # eight slices of 32 requests, generated in parallel
            self.jobs = [("chain", (5, S + 1000 * j, 32, None)) for j in range(8)]
            self.name = "chain verify B=256 K=8 V=152064 bf16, t=0.7, top-k 50 on p and q"
            self.metric = ("verify rounds/s & logit GB/s vs HBM peak "
                           "(B=256, K=8, V=152064 bf16, top-k 50)")
            self.profile = "verify_chain_b256_k8_v152064_topk50"
        elif key == 4:
            self.B = 16
            self.jobs = [("tree", (S + 100 * s, 16)) for s in range(8)]
            self.name = ("tree verify (MSS) B=16 N=32 depth<=5 branching<=3 V=32000 bf16, t=0.8")
            self.metric = ("verify rounds/s & logit GB/s vs HBM peak "
                           "(tree MSS B=16, N=32, V=32000 bf16)")
            self.profile = "verify_tree_b16_n32_v32000"
        self.extra_jobs = []
        if key == 3:
            # the all-sampled variant of the headline batch
            self.extra_jobs = [("chain", (3, S + 700, None, "none"))]

    def generate(self):
        """The pool (and extra batches), generated in spawned workers (before
        this process touches the GPU)."""
        import multiprocessing as mp
        jobs = self.jobs + self.extra_jobs
        with mp.get_context("spawn").Pool(min(len(jobs), os.cpu_count() or 1)) as pool:
            res = [pool.apply_async(_gen_tree if k == "tree" else _gen_chain, (a,))
                   for k, a in jobs]
            parts = [r.get() for r in res]
        self.pool = _concat(parts[:len(self.jobs)])
        self.extras = parts[len(self.jobs):]
        self.Btot = self.pool["B"]
        self.windows = self.Btot // self.B
        self.V = self.pool["V"]

    def window(self, w: int) -> dict:
        return _slice(self.pool, w * self.B, (w + 1) * self.B)

    def alg_bytes(self, inp: dict) -> int:
        from speculative_decoding_verification_63_gb300 import workloads as wl
        if self.kind == "tree":
            return wl.tree_algorithmic_bytes(inp)
        return wl.chain_algorithmic_bytes(inp)

    def tokens_verified(self, inp: dict) -> int:
        if self.kind == "tree":
            return int(np.sum(inp["num_nodes"] - 1))
        return int(np.sum(inp["num_drafts"]))

    def launches_per_step(self) -> int:
        return 2 if self.key == 5 else 1


def to_dev(a, dev):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


CHAIN_KEYS = ("target", "draft", "tokens", "temperature", "uniforms", "num_drafts", "top_k")
TREE_KEYS = ("target", "draft", "node_tokens", "parent", "q_row", "temperature", "u_accept",
             "u_sample", "num_nodes")


class DevicePool:
    """A workload's pool on the device, pool-sized outputs and a stepper."""

    def __init__(self, wk: Workload, inp: dict, B: int, dev):
        import torch
        import speculative_decoding_verification_63_gb300 as sv
        self.wk, self.inp, self.B, self.dev = wk, inp, B, dev
        self.Btot = inp["B"]
        self.windows = self.Btot // B
        keys = TREE_KEYS if wk.kind == "tree" else CHAIN_KEYS
        self.d = {k: to_dev(inp[k], dev) for k in keys}
        i32 = dict(dtype=torch.int32, device=dev)
        if wk.kind == "chain":
            K = inp["K"]
            self.max_top_k = int(inp["top_k"].max())
            self.out = dict(out_tokens=torch.empty((self.Btot, K + 1), **i32),
                            out_len=torch.empty(self.Btot, **i32),
                            accept_len=torch.empty(self.Btot, **i32))
            need = sv.sv_chain_workspace_bytes(B, K, inp["V"], sv.dtype_code(self.d["target"]),
                                               self.max_top_k)
        else:
            D = int(inp["max_depth"])
            self.out = dict(out_tokens=torch.empty((self.Btot, D + 1), **i32),
                            out_len=torch.empty(self.Btot, **i32),
                            accept_len=torch.empty(self.Btot, **i32),
                            accepted_nodes=torch.empty((self.Btot, max(D, 1)), **i32))
            need = sv.sv_tree_workspace_bytes(B, inp["N"], inp["M"], inp["V"],
                                              sv.dtype_code(self.d["target"]), 0)
        self.ws = sv.workspace(need, dev, ("bench", wk.key, B))

    def step(self, i: int):
        from speculative_decoding_verification_63_gb300 import _binding
        w = i % self.windows
        s = slice(w * self.B, (w + 1) * self.B)
        d, o = self.d, self.out
        if self.wk.kind == "chain":
            tk = d["top_k"][s] if self.max_top_k > 0 else None
            _binding.sv_verify_chain(d["target"][s], d["draft"][s], d["tokens"][s],
                                     d["temperature"][s], d["uniforms"][s],
                                     o["out_tokens"][s], o["out_len"][s], o["accept_len"][s],
                                     self.ws, num_drafts=d["num_drafts"][s], top_k=tk,
                                     max_top_k=self.max_top_k)
        else:
            _binding.sv_verify_tree(d["target"][s], d["draft"][s], d["node_tokens"][s],
                                    d["parent"][s], d["q_row"][s], d["temperature"][s],
                                    d["u_accept"][s], d["u_sample"][s], o["out_tokens"][s],
                                    o["out_len"][s], o["accept_len"][s],
                                    o["accepted_nodes"][s], self.ws,
                                    max_depth=int(self.inp["max_depth"]),
                                    num_nodes=d["num_nodes"][s])

    def outputs(self) -> dict:
        return {k: v.cpu().numpy() for k, v in self.out.items()}


def time_graphs(torch, stepper, steps: int, stream, dev, sampler=None, windows=1):
    """steps launches of stepper(i), captured in CUDA graphs of about
    GRAPH_LEN launches (a multiple of the pool's windows, so that every
    replay walks the whole pool), timed with CUDA events on `stream`.
    Returns milliseconds."""
    L = -(-GRAPH_LEN // windows) * windows if windows <= GRAPH_LEN else windows
    L = max(1, min(L, steps))
    graphs = []
    for length in (L, steps % L):
        if length == 0:
            graphs.append(None)
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(length):
                    stepper(i)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for g in graphs:
            if g is not None:
                g.replay()
    torch.cuda.synchronize(dev)
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)  # let the sampler come up before the timed region
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps // L):
            graphs[0].replay()
        if graphs[1] is not None:
            graphs[1].replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1)


# ----------------------------------------------------- parity of the batches

def parity_counts(got: dict, ref: dict) -> dict:
    """Near-boundary counts of GPU outputs against the oracle's (the rule of
    tests/gpu_util.compare): the path (lengths, accepted tokens / nodes) must
    be bit-exact unless an accept test (or a naive walk's draw) is within
    NEAR of its boundary; the emitted token must be the oracle's, or, for a
    near final draw, inside the oracle's window.  `firm_mismatch` counts
    breaches of that rule (must be 0)."""
    B = len(ref["status"])
    ok = ref["status"] == 0
    walk = ref.get("margin_walk", np.full(B, np.inf))
    near_path = ok & ((ref["margin_accept"] < NEAR) | (walk < NEAR))
    near_draw = ok & ~near_path & (ref["margin_draw"] < NEAR)
    firm = ok & ~near_path
    bad = np.zeros(B, dtype=bool)
    for k in ("out_len", "accept_len", "accepted_nodes"):
        if k in ref and k in got:
            bad |= np.any((got[k] != ref[k]).reshape(B, -1), axis=1)
    rows = np.arange(B)
    last = np.clip(ref["out_len"] - 1, 0, got["out_tokens"].shape[1] - 1)
    mask = np.ones_like(got["out_tokens"], dtype=bool)
    mask[rows, last] = False
    bad |= np.any((got["out_tokens"] != ref["out_tokens"]) & mask, axis=1)
    tok = got["out_tokens"][rows, last]
    bad |= ~((tok >= ref["draw_lo"]) & (tok <= ref["draw_hi"]))
    draw_mism = near_draw & ~bad & (tok != ref["out_tokens"][rows, last])
    path_mism = near_path & np.any(got["out_tokens"] != ref["out_tokens"], axis=1)
    return {"requests": int(ok.sum()), "draws": int(ok.sum()),
            "near_accept": int(near_path.sum()), "near_draw": int(near_draw.sum()),
            "near_draw_mismatch": int(draw_mism.sum()),
            "near_accept_mismatch": int(path_mism.sum()),
            "firm_mismatch": int((bad & firm).sum()),
            "failed": int((~ok).sum())}


def _oracle_requests(inp: dict, kind: str, reqs, lib=None) -> dict:
    import oracle
    if kind == "tree":
        return oracle.verify_tree_inputs(inp, requests=reqs, lib=lib)
    return oracle.verify_chain_inputs(inp, requests=reqs, lib=lib)


# ------------------------------------------------------ CPU oracle (baseline)

def _worker_init(path: str, kind: str):
    global _W_INP, _W_KIND
    import oracle
    oracle.load()
    with open(os.path.join(path, "meta.json")) as f:
        meta = json.load(f)
    _W_INP = {k: np.load(os.path.join(path, k + ".npy"), mmap_mode="r")
              for k in meta.pop("_arrays")}
    _W_INP.update(meta)
    _W_KIND = kind


def _worker_run(args):
    """Oracle passes over requests `reqs` of the shared pool until `seconds`
    of wall time (at least one).  Returns the rounds done."""
    reqs, seconds = args
    t0 = time.perf_counter()
    n = 0
    while n == 0 or time.perf_counter() - t0 < seconds:
        _oracle_requests(_W_INP, _W_KIND, reqs)
        n += len(reqs)
    return n


def _save_pool(inp: dict, kind: str, reqs) -> str:
    """The requests `reqs` of the pool as .npy files in a temporary folder,
    which the workers map read-only (each reads only its own requests)."""
    d = tempfile.mkdtemp(prefix="svbench")
    keys = TREE_KEYS + ("top_k",) if kind == "tree" else CHAIN_KEYS
    for k in keys:
        np.save(os.path.join(d, k + ".npy"), np.ascontiguousarray(inp[k][reqs]))
    meta = {k: (int(v) if isinstance(v, (np.integer,)) else v)
            for k, v in inp.items() if not isinstance(v, np.ndarray)}
    meta["B"] = len(reqs)
    meta["_arrays"] = list(keys)
    with open(os.path.join(d, "meta.json"), "w") as f:
        json.dump(meta, f)
    return d


def cpu_oracle(wk: Workload, one_thread_s: float, all_cores_s: float, sample_reqs):
    """The oracle, as it stands, on the host cores: one thread on
    `sample_reqs` for about one_thread_s, then every core
    (os.cpu_count() spawned worker processes, requests split round robin)
    for about all_cores_s.  Returns (baseline dict, oracle outputs of the
    sample's requests, in sample order)."""
    import multiprocessing as mp
    import oracle
    lib = oracle.load()
    inp = wk.pool
    reqs = np.asarray(sample_reqs)
    _oracle_requests(inp, wk.kind, reqs[:2], lib=lib)  # warm
    t0 = time.perf_counter()
    ref = _oracle_requests(inp, wk.kind, reqs, lib=lib)
    n1 = len(reqs)
    while time.perf_counter() - t0 < one_thread_s:
        _oracle_requests(inp, wk.kind, reqs, lib=lib)
        n1 += len(reqs)
    el1 = time.perf_counter() - t0

    cores = os.cpu_count() or 1
    path = _save_pool(inp, wk.kind, reqs)
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(cores, initializer=_worker_init, initargs=(path, wk.kind)) as pool:
            # every worker loaded: one tiny task each
            pool.map(_worker_run, [([0], 0.0)] * cores)
            shares = [list(range(w, len(reqs), cores)) for w in range(cores)]
            shares = [s for s in shares if s]
            t0 = time.perf_counter()
            res = pool.map(_worker_run, [(s, all_cores_s) for s in shares])
            el_all = time.perf_counter() - t0
    finally:
        shutil.rmtree(path, ignore_errors=True)
    n_all = sum(res)
    base = {"value": n1 / el1, "unit": UNIT, "cores": 1, "kind": "oracle",
            "value_all_cores": n_all / el_all, "cores_all": cores,
            "host_cpu_count": cores,
            "sample": (f"{len(reqs)} requests of the timed pool, repeated: one thread "
                       f"{n1} rounds in {el1:.1f} s; {len(shares)} worker processes "
                       f"{n_all} rounds in {el_all:.1f} s; fp64 C oracle as it stands")}
    return base, ref


# ------------------------------------------------------------- reference arm

def run_reference(args, dist):
    """The reference arm: the fp64 CPU oracle, as it stands, on one host
    core.  One step is one request round of the workload's pool (requests in
    pool order, so greedy and sampled rounds alternate as in the headline
    batch); W untimed steps, then exactly K timed ones.  Without
    --steps/--warmup the arm runs 256 timed rounds after 3 warm-up rounds."""
    if dist.rank != 0:
        return 0
    import oracle
    lib = oracle.load()
    wk = Workload(args.workload)
    wk.jobs = wk.jobs[:1]  # one batch is enough for per-request rounds
    wk.extra_jobs = []
    wk.generate()
    inp = wk.pool

    def step(i):
        b = i % wk.Btot
        _oracle_requests(inp, wk.kind, [b], lib=lib)

    K = args.steps if args.steps is not None else 256
    W = max(args.warmup if args.warmup is not None else 3, 3)
    for i in range(W):
        step(i)
    t0 = time.perf_counter()
    for i in range(K):
        step(W + i)
    el = time.perf_counter() - t0
    value = K / el
    sample = (f"{K} request rounds of the {wk.name} pool, one per step, requests in pool "
              "order, fp64 C, one host thread")
    line = {"metric": wk.metric, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": K,
            "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wk.name, "parallelism": "replicas"}, "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- GPU arm

def e2e_leg(torch, sv, wk: Workload, dp: DevicePool, stream, dev, steps: int, dist):
    """The same steps through the public API from pinned host buffers: every
    step copies its batch's inputs host -> device (the rows the kernel
    reads: greedy requests' draft rows are not copied; a tree's draft rows
    go as one block), calls the library and reads its results back."""
    inp = dp.inp
    B = dp.B
    keys = TREE_KEYS if wk.kind == "tree" else CHAIN_KEYS
    host = {}
    for k in keys:
        a = np.ascontiguousarray(inp[k])
        host[k] = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
    windows = dp.windows

    def window_bytes(w):
        s = slice(w * B, (w + 1) * B)
        n = 0
        for k in keys:
            t = host[k][s]
            if k == "draft" and wk.kind == "chain":
                n += int(t[0].numel() * t.element_size()) * int(
                    np.sum(inp["temperature"][s] > 0))
            else:
                n += int(t.numel() * t.element_size())
        return n

    if wk.kind == "chain":
        K = inp["K"]
        res = [torch.empty((B, K + 1), dtype=torch.int32).pin_memory(),
               torch.empty(B, dtype=torch.int32).pin_memory(),
               torch.empty(B, dtype=torch.int32).pin_memory()]
    else:
        D = int(inp["max_depth"])
        res = [torch.empty((B, D + 1), dtype=torch.int32).pin_memory(),
               torch.empty(B, dtype=torch.int32).pin_memory(),
               torch.empty(B, dtype=torch.int32).pin_memory(),
               torch.empty((B, max(D, 1)), dtype=torch.int32).pin_memory()]
    d2h = sum(int(t.numel() * t.element_size()) for t in res)
    sampled = [np.nonzero(inp["temperature"][w * B:(w + 1) * B] > 0)[0] for w in range(windows)]
    ws = dp.ws

    def e2e_step(i):
        w = i % windows
        s = slice(w * B, (w + 1) * B)
        d = {}
        for k in keys:
            if k == "draft" and wk.kind == "chain" and len(sampled[w]) < B:
                t = torch.empty(host[k][s].shape, dtype=host[k].dtype, device=dev)
                for b in sampled[w]:  # greedy requests' draft rows are never read
                    t[b].copy_(host[k][s][b], non_blocking=True)
                d[k] = t
            else:
                d[k] = host[k][s].to(dev, non_blocking=True)
        for k in ("target", "draft"):
            d[k] = d[k].view(torch.bfloat16) if inp["dtype"] == "bf16" else d[k]
        if wk.kind == "chain":
            mt = int(inp["top_k"].max())
            out = sv.verify_chain(d["target"], d["draft"], d["tokens"], d["temperature"],
                                  d["uniforms"], num_drafts=d["num_drafts"],
                                  top_k=d["top_k"] if mt > 0 else None,
                                  max_top_k=mt, ws=ws)
            names = ("out_tokens", "out_len", "accept_len")
        else:
            out = sv.verify_tree(d["target"], d["draft"], d["node_tokens"], d["parent"],
                                 d["q_row"], d["temperature"], d["u_accept"], d["u_sample"],
                                 max_depth=int(inp["max_depth"]), num_nodes=d["num_nodes"],
                                 ws=ws)
            names = ("out_tokens", "out_len", "accept_len", "accepted_nodes")
        for r, n in zip(res, names):
            r.copy_(out[n], non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
    torch.cuda.synchronize(dev)
    dist.barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(steps):
            e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_s = dist.max(time.perf_counter() - t0)
    sv.check_device_errors(ws)
    h2d = sum(window_bytes(i % windows) for i in range(steps)) // steps
    return {"value": dist.world * B * steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps}


def single_call_latency(torch, dp: DevicePool, stream, dev, n: int = 200) -> float:
    """Median device time of one call, each timed alone (synchronised), in
    microseconds."""
    ts = []
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for i in range(n):
        with torch.cuda.stream(stream):
            e0.record(stream)
            dp.step(i)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts)


def run_ours(args, dist):
    import torch
    import speculative_decoding_verification_63_gb300 as sv

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the verification runs only on the GPU)")
    wk = Workload(args.workload)
    if args.kernel_only:
        wk.extra_jobs = []
    wk.generate()  # spawned workers, before this process touches the GPU
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    sv.lib()  # fail loudly when the extension is missing

    dp = DevicePool(wk, wk.pool, wk.B, dev)
    win0 = wk.window(0)
    alg_bytes = wk.alg_bytes(win0)
    per_win = [wk.alg_bytes(wk.window(w)) for w in range(wk.windows)]
    alg_mean = sum(per_win) / len(per_win)
    pool_bytes = sum(int(dp.d[k].numel() * dp.d[k].element_size()) for k in ("target", "draft"))

    stream = torch.cuda.Stream(device=dev)
    warm = max(args.warmup, 3)
    with torch.cuda.stream(stream):
        for i in range(max(warm, wk.windows)):
            dp.step(i)
    torch.cuda.synchronize(dev)
    sv.check_device_errors(dp.ws)

    if args.kernel_only:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(args.steps):
                dp.step(i)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        sv.check_device_errors(dp.ws)
        ms = e0.elapsed_time(e1)
        if dist.rank == 0:
            print(json.dumps({"kernel_only": True, "workload": wk.key, "steps": args.steps,
                              "ms_per_step": ms / max(args.steps, 1),
                              "logit_gbs": alg_mean * args.steps / (ms / 1e3) / 1e9}),
                  flush=True)
        return 0

    # outputs of one pass over the pool (the timed steps compute the same)
    gpu_out = dp.outputs()

    K_steps = args.steps
    sampler = ClockSampler(gpu_uuid(torch))
    dist.barrier()
    torch.cuda.synchronize(dev)
    ms_local = time_graphs(torch, dp.step, K_steps, stream, dev, sampler, dp.windows)
    clocks = sampler.stop()
    dist.barrier()
    ms = dist.max(ms_local)
    sv.check_device_errors(dp.ws)

    launch_s = ms_local / 1e3 / K_steps
    steps_per_s = K_steps / (ms / 1e3)
    rounds_per_s = dist.world * wk.B * steps_per_s
    peak, peak_kind = hbm_peak()
    achieved = alg_mean / launch_s / 1e9
    traffic = stored_traffic(wk.profile, wk.kernel)

    extra = {}
    if wk.key == 2 and dist.rank == 0:
        extra["latency_us_single_call"] = single_call_latency(torch, dp, stream, dev)
    variants = {}
    if wk.key == 3 and dist.rank == 0:
        # the fixed cost per step shows most on smaller or draw-heavy batches
        for name, vinp, vB in (("all_sampled_b64", wk.extras[0], 64),
                               ("half_greedy_b32", wk.pool, 32),
                               ("half_greedy_b128", wk.pool, 128)):
            vdp = DevicePool(wk, vinp, vB, dev)
            with torch.cuda.stream(stream):
                for i in range(max(3, vdp.windows)):
                    vdp.step(i)
            vsteps = 2000
            vms = time_graphs(torch, vdp.step, vsteps, stream, dev, windows=vdp.windows)
            sv.check_device_errors(vdp.ws)
            vb = sum(wk.alg_bytes(_slice(vinp, w * vB, (w + 1) * vB))
                     for w in range(vdp.windows)) / vdp.windows
            us = vms / vsteps * 1e3
            variants[name] = {"us_per_step": us, "algorithmic_bytes": vb,
                              "gbs": vb / (us * 1e-6) / 1e9,
                              "frac": vb / (us * 1e-6) / 1e9 / peak}
            del vdp
    e2e = e2e_leg(torch, sv, wk, dp, stream, dev, max(10, min(K_steps, 300)), dist)

    cpu, parity = None, None
    if dist.rank == 0 and dist.world == 1:
        if wk.key == 5:
            sample = np.arange(0, wk.Btot, 8)            # 32 requests
        elif wk.key == 2:
            sample = np.arange(0, wk.Btot, 4)            # 128 requests
        else:
            sample = np.arange(wk.Btot)
        cpu, ref = cpu_oracle(wk, 10.0, 10.0, sample)
        got = {k: v[sample] for k, v in gpu_out.items()}
        parity = parity_counts(got, ref)
        parity["sample"] = f"{len(sample)} requests of the timed pool (every window)"
        if parity["firm_mismatch"]:
            raise SystemExit(f"bench.py: parity check against the oracle failed: {parity}")

    if dist.rank == 0:
        config = {"workload": wk.name, "B": wk.B, "V": wk.V, "logits": "bf16",
                  "parallelism": "replicas",
                  "l2": f"{wk.windows} rotating batches, {pool_bytes / 1e6:.0f} MB of logits "
                        f"in all ({'>' if pool_bytes > L2_BYTES else '<='} 129 MB L2)"}
        if wk.kind == "chain":
            config["K"] = int(wk.pool["K"])
        else:
            config["N"] = int(wk.pool["N"])
        line = {"metric": wk.metric, "value": rounds_per_s, "unit": UNIT, "n_gpus": dist.world,
                "steps": K_steps, "warmup": warm, "ms_per_step": ms / K_steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic", "config": config,
                "steps_per_s": steps_per_s, "us_per_step": ms / K_steps * 1e3,
                "tokens_verified_per_s":
                    dist.world * wk.tokens_verified(win0) * steps_per_s,
                "logit_gbs": dist.world * alg_mean * steps_per_s / 1e9,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                             "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                             "traffic": traffic, "algorithmic_bytes": alg_mean,
                             "frac_of_8tbs": achieved / 8000.0},
                "parity": parity,
                "cpu_baseline": cpu,
                "e2e": e2e,
                "gpu_launches": K_steps * wk.launches_per_step(),
                "clocks": clocks}
        if variants:
            line["variants"] = variants
        line.update(extra)
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
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
