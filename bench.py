"""Benchmark of the speculative-decoding verification step on GB300.

python bench.py [--gpus N --steps K --warmup W] [--workload mixed] [--impl ours|reference]

One step = one spec_verify call over one batch of the workload (all rows of
the verification: row statistics, acceptance scan, residual or extra-token
draw, outputs). The default workload is the mixed batch (B=256, gamma=8,
V=128256, bf16, T in {0, 0.3, 0.7, 1}): every part of the path runs in it at
full form. Inputs (1.57 GB of logits) are larger than the 129 MB L2, so
consecutive steps re-read them from HBM.

value: verified rows/s = steps * B * (gamma+1) / time, the whole job (all
ranks; each rank verifies its own batch: weak scaling), timed on the device
with CUDA events, max over ranks. e2e: the same metric through
spec_verify_host (host buffers; copies inside the timed region).
roofline: algorithmic bytes per call / average call duration, against the
measured HBM copy bandwidth. cpu_baseline / --impl reference: the CPU oracle
(test infrastructure) timed on this host's cores on a bounded sample.
near_ties (N = 1): the headline batch's outputs judged by the oracle under the
parity rules, with the near-tie counts and their exact expectation.
per_workload (N = 1): each of the five workloads timed alone in the same run
(per-call figures, rows/s, achieved GB/s and roofline fraction, clocks; for
calls under 40 us also the device time per call from CUDA-graph replay, since
eager calls that short run at the host's enqueue rate).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "spec-verify rows/s and achieved HBM GB/s vs ~8 TB/s peak, B×(γ+1)×V"
UNIT = "rows/s"
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
# The files each captured kernel is compiled from (its own source plus the
# shared headers): a captured DRAM traffic applies while they are unchanged.
_CSRC = "speculative_decoding_verification_06_gb300/csrc/"
KERNEL_COMMON = [_CSRC + "sv_common.cuh", _CSRC + "sv_internal.h", "include/specverify.h"]
KERNEL_FILES = {"stream_kernel": _CSRC + "sv_stream.cu", "early_kernel": _CSRC + "sv_stream.cu",
                "rowwise_kernel": _CSRC + "sv_rowwise.cu", "cluster_kernel": _CSRC + "sv_cluster.cu"}
KERNEL_SOURCES = sorted(set(KERNEL_FILES.values())) + KERNEL_COMMON


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed",
                    help="tiny | greedy | sampling | mixed | large (default: mixed)")
    ap.add_argument("--path", choices=["auto", "rowwise", "streaming"], default="auto")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the per-workload block (all five workloads, timed in the same run at N = 1)")
    ap.add_argument("--no-near-ties", action="store_true",
                    help="skip the near-tie counts (the oracle over the headline batch, threaded)")
    ap.add_argument("--early-exit", action="store_true",
                    help="early-exit verification: nothing after a request's first rejection is read")
    ap.add_argument("--op", choices=["verify", "onehot", "ngram", "commit", "loop", "tree"], default="verify",
                    help="verify (default, the headline); onehot: spec_verify_onehot on the workload's "
                         "target rows; ngram: spec_ngram_propose; commit: spec_commit; loop: ngram -> "
                         "onehot verify -> commit, the model-free decoding step with no host sync; tree: "
                         "spec_verify_tree over the workload's target rows")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed_k(rank: int) -> int:
    """Weak scaling: rank r verifies its own batch, seeded 1000 * config + r."""
    return rank


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's time (all ranks get it); x itself without a group."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peak_hbm():
    try:
        with open(PEAKS) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash(kernel: str = "stream_kernel") -> str:
    """Hash of the sources `kernel` (a name as in the launch list, template
    arguments dropped) is compiled from."""
    h = hashlib.sha256()
    for rel in [KERNEL_FILES[kernel.split("<")[0]]] + KERNEL_COMMON:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(os.path.basename(rel).encode() + f.read())
    return h.hexdigest()[:16]


def algorithmic_bytes_early(batch, num_accepted) -> int:
    """Early exit: the rows the method needs. Per request with n accepted:
    target rows 0..n (n + 1 rows), the draft rows of the positions evaluated
    (T > 0: min(n + 1, g)), and the draw's re-read (2 rows for a residual, 1
    for the extra token); plus the small inputs and outputs."""
    w = batch.workload
    s, V, G, B = w.elem_bytes, w.V, w.gamma, batch.B
    rows = 0
    for b in range(B):
        n = int(num_accepted[b])
        if n < 0:
            rows += 1
            continue
        rows += n + 1
        if 0 < batch.temperature[b] < np.inf:
            rows += min(n + 1, G) + (2 if n < G else 1)
    return int(s * V * rows + B * G * 8 + B * 12 + B * (G + 1) * 4)


def algorithmic_bytes(batch, num_accepted) -> int:
    """Logit bytes the method must read once, plus the re-read of the rows the
    draw needs, plus the small inputs and outputs: s*V*[B(g+1) + g*B_samp +
    sum over valid sampled requests (2 if n < g else 1)] + B*g*8 + B*12 +
    B*(g+1)*4, B_samp the requests with 0 < T < inf (their draft rows are read
    whether or not the request turns out valid)."""
    w = batch.workload
    s, V, G, B = w.elem_bytes, w.V, w.gamma, batch.B
    T = batch.temperature
    samp = (T > 0) & np.isfinite(T)
    drawn = samp & (num_accepted >= 0)
    reread = np.where(num_accepted[drawn] < G, 2, 1).sum()
    rows = B * (G + 1) + G * int(samp.sum()) + int(reread)
    return int(s * V * rows + B * G * 8 + B * 12 + B * (G + 1) * 4)


def captured_traffic(workload: str, early: bool, path: str | None = None):
    """DRAM bytes per launch of this workload's kernel from the committed ncu
    capture (`profiles/traffic.json`, keyed by workload, `-early` for early
    exit), or None: no capture, or the kernel sources changed since."""
    try:
        with open(path or PROFILE_TRAFFIC) as f:
            prof = json.load(f)
        entry = prof.get(workload + ("-early" if early else ""))
        if entry and entry.get("kernel_hash") == kernel_hash(entry.get("kernel", "stream_kernel")):
            return entry.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(batch, seconds: float, rows_per_request: int):
    """The oracle as it stands, one host thread, over whole passes of the
    batch (or a prefix of it) until about ``seconds`` of CPU time."""
    import oracle
    lib = oracle.load()
    t0 = time.perf_counter()
    oracle.verify(*batch.slice(0, 1).arrays(), lib=lib)
    one = max(time.perf_counter() - t0, 1e-6)
    n_req = int(min(batch.B, max(1, seconds / one)))
    sample = batch.slice(0, n_req)
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.verify(*sample.arrays(), lib=lib)
        done += n_req
        el = time.perf_counter() - t0
        if el >= seconds or done >= 3 * batch.B:
            break
    return {"value": done * rows_per_request / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"requests 0..{n_req - 1} of the same batch, {done // n_req} pass(es), "
                      f"{el:.1f} s single-threaded fp64 C"}


def run_reference(args, w, rank, world):
    """--impl reference: the CPU oracle on the host cores, bounded sample per step."""
    from workloads import synthetic
    if rank != 0:
        return
    batch = synthetic.generate(w, k=0)
    rows = w.gamma + 1
    import oracle
    lib = oracle.load()
    t0 = time.perf_counter()
    oracle.verify(*batch.slice(0, 1).arrays(), lib=lib)
    one = max(time.perf_counter() - t0, 1e-6)
    per_step_s = max(0.2, min(2.0, 60.0 / max(1, args.steps + args.warmup)))
    n_req = int(min(batch.B, max(1, per_step_s / one)))
    sample = batch.slice(0, n_req)
    for _ in range(args.warmup):
        oracle.verify(*sample.arrays(), lib=lib)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify(*sample.arrays(), lib=lib)
    el = time.perf_counter() - t0
    value = args.steps * n_req * rows / el
    desc = f"requests 0..{n_req - 1} of the {w.name} batch per step, single-threaded fp64 C oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.description, "B": w.B, "gamma": w.gamma, "V": w.V,
                   "logits": w.dtype, "sample_requests": n_req},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_calls(call, K, W, stream):
    """W warm-up calls, then K calls each bracketed by CUDA events on `stream`.
    Returns (total ms, per-call ms array)."""
    import torch
    for _ in range(max(3, W)):
        call()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), np.array([a.elapsed_time(b) for a, b in zip(starts, ends)])


def replay_us_per_call(call, GN=50, R=20):
    """Device time per call: GN calls captured in one CUDA graph, 3 warm-up
    replays, then R replays between CUDA events."""
    import torch
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(GN):
            call()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(R):
        graph.replay()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) * 1e3 / (R * GN)


def graph_us_per_call(op, sv, B, G, out_t, out_n, buf0, lens0, props, nprop, GN=50, R=20):
    """Device time per call of a latency-bound op (eager calls there measure the
    host's enqueue rate): GN calls captured in one CUDA graph, 3 warm-up
    replays, then R replays between CUDA events. The commit appends into a
    buffer of its own with room for every replayed call."""
    import torch
    if op == "commit":
        gbuf = torch.zeros((B, (G + 1) * GN * (R + 4)), dtype=torch.int32, device="cuda")
        glens = torch.zeros((B,), dtype=torch.int32, device="cuda")

        def call():
            sv.spec_commit(out_t, out_n, gbuf, glens)
    else:
        def call():
            sv.spec_ngram_propose(buf0, lens0, G, 2, 5, props, nprop)
    return replay_us_per_call(call, GN, R)  # the binding enqueues on the current (capturing) stream


def run_aux(args, w, local):
    """--op onehot | ngram | commit | loop | tree on one GPU: one JSON line each, with
    the same timing rules as the headline (warm-up, CUDA events on the
    launching stream, per-call roofline)."""
    import torch
    import speculative_decoding_verification_06_gb300 as sv
    from workloads import synthetic
    torch.cuda.set_device(local)
    sv.build.build()
    sv.load()
    stream = torch.cuda.current_stream()
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    batch = synthetic.generate(w, k=0)
    B, G, V, es = batch.B, w.gamma, w.V, w.elem_bytes
    dt = sv.SV_F32 if w.dtype == "f32" else sv.SV_BF16
    peak, peak_src = peak_hbm()
    M = 4096
    hist = synthetic.histories(B, M, (256, M), vocab=V, copy_prob=0.5, seed=1)
    out_t = torch.empty((B, G + 1), dtype=torch.int32, device="cuda")
    out_n = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = torch.empty(max(16, sv.workspace_size(B, G, V, dt)), dtype=torch.uint8, device="cuda")
    tgt, ua, us, T = d(batch.target), d(batch.u_accept), d(batch.u_sample), d(batch.temperature)
    tok = d(batch.tokens)
    full = torch.full((B,), G, dtype=torch.int32, device="cuda")
    buf0, lens0 = d(hist.token_buf), d(hist.seq_lens)
    buf, lens = buf0.clone(), lens0.clone()
    props = torch.empty((B, G), dtype=torch.int32, device="cuda")
    nprop = torch.empty((B,), dtype=torch.int32, device="cuda")
    extra = {}
    if args.op == "onehot":
        def call():
            sv.spec_verify_onehot(tgt, tok, full, ua, us, T, out_t, out_n, ws, stream)
        unit, per_step = "rows/s", B * (G + 1)
        metric = "spec-verify-onehot rows/s (deterministic proposals, target rows only), B×(γ+1)×V"
    elif args.op == "ngram":
        def call():
            sv.spec_ngram_propose(buf0, lens0, G, 2, 5, props, nprop, stream=stream)
        unit, per_step = "requests/s", B
        metric = "n-gram proposals requests/s (prompt_lookup_min 2, max 5)"
    elif args.op == "commit":
        def call():
            sv.spec_commit(out_t, out_n, buf, lens, stream=stream)
        unit, per_step = "requests/s", B
        metric = "post-verify commit requests/s"
    elif args.op == "tree":
        # a candidate tree per request over the workload's target rows: gamma
        # nodes, half chain, half branches (synthetic.tree_parents)
        tree_par = d(synthetic.tree_parents(B, G, seed=5))
        tree_m = torch.full((B,), G, dtype=torch.int32, device="cuda")
        tree_nodes = torch.empty((B, G), dtype=torch.int32, device="cuda")

        def call():
            sv.spec_verify_tree(tgt, tok, tree_par, tree_m, ua, us, T, out_t, out_n, tree_nodes, workspace=ws,
                                stream=stream)
        unit, per_step = "rows/s", B * (G + 1)
        metric = "tree verification rows/s (gamma nodes per request, one row each), B×(γ+1)×V"
    else:
        def call():
            sv.spec_ngram_propose(buf, lens, G, 2, 5, props, nprop, stream=stream)
            sv.spec_verify_onehot(tgt, props, nprop, ua, us, T, out_t, out_n, ws, stream)
            sv.spec_commit(out_t, out_n, buf, lens, stream=stream)
        unit, per_step = "rows/s", B * (G + 1)
        metric = "model-free decoding step (ngram -> onehot verify -> commit) rows/s, B×(γ+1)×V"
    if args.op == "commit":  # a verification result to commit, and room for every step
        sv.spec_verify_onehot(tgt, tok, full, ua, us, T, out_t, out_n, ws, stream)
        buf = torch.zeros((B, M + 70 * (args.steps + args.warmup + 8)), dtype=torch.int32, device="cuda")
        lens = torch.zeros((B,), dtype=torch.int32, device="cuda")
    if args.op == "loop":  # histories with room for every step
        buf = torch.zeros((B, M + (G + 1) * (args.steps + args.warmup + 8)), dtype=torch.int32, device="cuda")
        buf[:, :M] = buf0
        lens = lens0.clone()
    K = args.steps
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    total_ms, per_call = time_calls(call, K, args.warmup, stream)
    clk = clocks.stop()
    n_acc = out_n.cpu().numpy()
    if args.op == "tree":
        samp = int(((batch.temperature > 0) & (n_acc >= 0)).sum())
        abytes = es * V * (B * (G + 1) + samp) + B * G * 12 + B * 12 + B * (G + 1) * 4 + B * G * 4
        extra["mean_accepted"] = float(n_acc[n_acc >= 0].mean())
    elif args.op in ("onehot", "loop"):
        samp = int(((batch.temperature > 0) & (n_acc >= 0)).sum())
        abytes = es * V * (B * (G + 1) + samp) + B * G * 8 + B * 12 + B * (G + 1) * 4
        extra["mean_accepted"] = float(n_acc[n_acc >= 0].mean())
        if args.op == "loop":
            abytes += 4 * int(hist.seq_lens.sum()) + B * (G + 1) * 4
            extra["mean_proposed"] = float(nprop.float().mean().item())
    elif args.op == "ngram":
        abytes = 4 * int(hist.seq_lens.sum()) + B * G * 4 + B * 8
        extra["mean_proposed"] = float(nprop.float().mean().item())
    else:
        abytes = B * (G + 1) * 4 + B * 4 * 3 + int((np.maximum(n_acc, -1) + 1).sum()) * 4
    if args.op in ("ngram", "commit"):
        extra["graph_us_per_call"] = graph_us_per_call(args.op, sv, B, G, out_t, out_n, buf0, lens0, props, nprop)
    avg = float(per_call.mean()) * 1e-3
    achieved = abytes / avg / 1e9
    line = {
        "metric": metric, "value": K * per_step / (total_ms * 1e-3), "unit": unit, "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype if args.op in ("onehot", "loop", "tree") else "int32",
        "data": "synthetic",
        "op": args.op,
        "config": {"workload": w.description, "B": B, "gamma": G, "V": V,
                   "histories": f"lengths U(256, {M}), copy probability 0.5, vocab {V}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_call": int(abytes), "avg_call_us": avg * 1e6},
        "clocks": clk,
    }
    line.update(extra)
    print(json.dumps(line), flush=True)


def measure_workload(sv, w, path, early, stream, seconds=0.5, steps=None, warmup=10):
    """One workload timed alone: its batch resident on the device, calls
    bracketed by CUDA events on `stream` after warm-up, a clock sampler
    running. The number of calls fills about `seconds` (at least 200) unless
    `steps` is given. Returns the per-call figures and the roofline."""
    import torch
    from workloads import synthetic
    batch = synthetic.generate(w, k=0)
    dev = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in batch.arrays()]
    B, G, V = batch.B, w.gamma, w.V
    dt = sv.SV_F32 if w.dtype == "f32" else sv.SV_BF16
    out_t = torch.empty((B, G + 1), dtype=torch.int32, device="cuda")
    out_n = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = torch.empty(max(16, sv.workspace_size(B, G, V, dt)), dtype=torch.uint8, device="cuda")

    def call():
        sv.spec_verify(*dev, out_tokens=out_t, out_num_accepted=out_n, workspace=ws, stream=stream, path=path,
                       early_exit=early)

    _, probe = time_calls(call, 20, warmup, stream)
    K = steps or int(min(20000, max(200, seconds / max(float(np.median(probe)) * 1e-3, 1e-6))))
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    total_ms, per_call = time_calls(call, K, 3, stream)
    clk = clocks.stop()
    num_acc = out_n.cpu().numpy()
    abytes = (algorithmic_bytes_early if early else algorithmic_bytes)(batch, num_acc)
    peak, _ = peak_hbm()
    avg = float(per_call.mean()) * 1e-3
    achieved = abytes / avg / 1e9
    graph_us = None
    if avg < 40e-6:
        # a call this short: eager calls measure the host's enqueue rate, so
        # the device time per call is also taken from CUDA-graph replay
        def call_current():  # the binding enqueues on the current (capturing) stream
            sv.spec_verify(*dev, out_tokens=out_t, out_num_accepted=out_n, workspace=ws, path=path,
                           early_exit=early)

        graph_us = replay_us_per_call(call_current)
    del dev, ws
    torch.cuda.empty_cache()
    return {"workload": w.description, "calls": K, "avg_call_us": avg * 1e6,
            "graph_us_per_call": graph_us,
            "p10_p50_p90_call_us": [float(np.percentile(per_call, q)) * 1e3 for q in (10, 50, 90)],
            "rows_per_s": K * B * (G + 1) / (total_ms * 1e-3), "algorithmic_bytes_per_call": int(abytes),
            "achieved_gbs": achieved, "frac": achieved / peak, "clocks": clk,
            "launches_per_call": sv.last_launch_count()}


def near_tie_counts(batch, out_tokens, num_acc):
    """The headline batch's outputs judged by the oracle under the parity
    rules (test infrastructure, run here on the host cores): near-tie counts
    and their expectation. Returns a dict, with "parity": "ok" or the first
    mismatch."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import parity
    t0 = time.perf_counter()
    ora, det = parity.run_oracle(batch)
    gpu = {"out_tokens": out_tokens, "out_num_accepted": num_acc}
    res = {"requests": int(batch.B)}
    try:
        rep = parity.compare(batch, gpu, ora, det)
        res["parity"] = "ok"
    except AssertionError as e:
        return {"requests": int(batch.B), "parity": f"mismatch: {str(e)[:200]}"}
    res.update({"accept_decisions": rep.accept_decisions, "accept_near_ties": rep.accept_near_ties,
                "accept_near_ties_expected": rep.accept_ties_expected, "accept_cap": rep.accept_tie_cap(),
                "draws": rep.draws, "draw_near_ties": rep.sample_near_ties,
                "draw_near_ties_at_margin": rep.draw_ties_at_margin,
                "draw_near_ties_expected": rep.draw_ties_expected,
                "draw_near_ties_sigma": rep.draw_ties_var ** 0.5,
                "draw_ties_within_5_sigma": bool(rep.draw_ties_consistent()),
                "oracle_s": time.perf_counter() - t0})
    return res


def main():
    args = parse()
    rank, world, local = dist_env()
    from workloads import synthetic
    w = synthetic.BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if args.op != "verify":
        if rank == 0:
            run_aux(args, w, local)
        return

    import torch
    import speculative_decoding_verification_06_gb300 as sv
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sv.build.build()
    sv.load()

    batch = synthetic.generate(w, k=rank_seed_k(rank))
    dev = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in batch.arrays()]
    B, G, V = batch.B, w.gamma, w.V
    dt = sv.SV_F32 if w.dtype == "f32" else sv.SV_BF16
    path = {"auto": sv.SV_PATH_AUTO, "rowwise": sv.SV_PATH_ROWWISE,
            "streaming": sv.SV_PATH_STREAMING}[args.path]
    out_tokens = torch.empty((B, G + 1), dtype=torch.int32, device="cuda")
    out_n = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = torch.empty(max(16, sv.workspace_size(B, G, V, dt)), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        sv.spec_verify(*dev, out_tokens=out_tokens, out_num_accepted=out_n, workspace=ws,
                       stream=stream, path=path, early_exit=args.early_exit)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    launches_per_call = sv.last_launch_count()
    num_acc = out_n.cpu().numpy()

    # ---- timed region (device events on the launching stream)
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for i in range(K):
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t_begin.elapsed_time(t_end)
    per_call_ms = np.array([s.elapsed_time(e) for s, e in zip(starts, ends)])
    if dist:
        total_ms = max_over_ranks(total_ms, dist, "cuda")
    rows_per_step = B * (G + 1)
    value = world * K * rows_per_step / (total_ms * 1e-3)

    abytes = (algorithmic_bytes_early if args.early_exit else algorithmic_bytes)(batch, num_acc)
    peak, peak_src = peak_hbm()
    avg_call_s = float(per_call_ms.mean()) * 1e-3
    achieved = abytes / avg_call_s / 1e9
    traffic = captured_traffic(args.workload, args.early_exit)

    # ---- end to end through host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        host = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in batch.arrays()]
        h_out = torch.empty((B, G + 1), dtype=torch.int32).pin_memory()
        h_n = torch.empty((B,), dtype=torch.int32).pin_memory()
        staging = torch.empty(sv.host_staging_size(B, G, V, dt), dtype=torch.uint8, device="cuda")
        for _ in range(2):
            sv.spec_verify_host(*host, h_out, h_n, staging, stream=stream)
        torch.cuda.synchronize()
        KE = max(1, args.e2e_steps)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        e0.record(stream)
        for _ in range(KE):
            sv.spec_verify_host(*host, h_out, h_n, staging, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
        if dist:
            e2e_ms = max_over_ranks(e2e_ms, dist, "cuda")
        es = w.elem_bytes
        samp = int((batch.temperature > 0).sum())
        h2d = B * (G + 1) * V * es + samp * G * V * es + B * G * 8 + B * 8
        d2h = B * (G + 1) * 4 + B * 4
        assert np.array_equal(h_n.numpy(), num_acc), "host entry disagrees with device entry"
        e2e = {"value": world * KE * rows_per_step / (e2e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": KE}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(batch, args.cpu_seconds, G + 1)

    ties = None
    if rank == 0 and world == 1 and not args.no_near_ties:
        ties = near_tie_counts(batch, out_tokens.cpu().numpy(), num_acc)

    per_workload = None
    if rank == 0 and world == 1 and not args.no_per_workload:
        headline = {"workload": w.description, "calls": K, "avg_call_us": avg_call_s * 1e6,
                    "p10_p50_p90_call_us": [float(np.percentile(per_call_ms, q)) * 1e3 for q in (10, 50, 90)],
                    "rows_per_s": value / world, "algorithmic_bytes_per_call": int(abytes),
                    "achieved_gbs": achieved, "frac": achieved / peak, "clocks": clk,
                    "launches_per_call": launches_per_call}
        per_workload = {}
        del dev, ws
        torch.cuda.empty_cache()
        for name in ("tiny", "greedy", "sampling", "mixed", "large"):
            if name == args.workload:
                per_workload[name] = headline
            else:
                per_workload[name] = measure_workload(sv, synthetic.BY_NAME[name], path, args.early_exit, stream)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    samp_mask = (batch.temperature > 0) & (num_acc >= 0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.description, "B": B, "gamma": G, "V": V, "logits": w.dtype,
                   "seeds": f"1000*{w.config}+rank", "path": args.path,
                   "early_exit": bool(args.early_exit),
                   "l2": f"inputs {(batch.target.nbytes + batch.draft.nbytes) / 1e9:.2f} GB > 129 MB L2; "
                         "no flush between steps",
                   "parallelism": f"replicas: {world} independent batches"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_call": abytes,
                     "avg_call_us": avg_call_s * 1e6,
                     "p10_p50_p90_call_us": [float(np.percentile(per_call_ms, q)) * 1e3 for q in (10, 50, 90)]},
        "gpu_launches": int(K * launches_per_call),
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "requests_per_s": world * K * B / (total_ms * 1e-3),
        "mean_accepted": float(num_acc[num_acc >= 0].mean()),
        "acceptance_rate_sampled": float(num_acc[samp_mask].mean() / G) if samp_mask.any() else None,
        "near_ties": ties,
        "per_workload": per_workload,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
