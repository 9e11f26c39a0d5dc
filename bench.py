"""Benchmark of the GB300 gated delta rule forward library.

One step = one chunked-prefill call (gdr_chunk_fwd: chunk metadata, intra-chunk
cumsum / A / solve / WY, inter-chunk state recurrence, output) over the long
KDA-style workload: one sequence of 32768 tokens, Hk = 16, Hv = 32 (two value
heads per key head), K = V = 128, bf16, per-key-channel decays gk ~ U[-0.1, 0]
of shape [T, 32, 128]; the largest prefill configuration that fits one GPU.
`value` is prefill tokens/s with inputs resident in HBM; the step's inputs
(1.1 GB) are larger than L2 (129 MB), and L2 is flushed before every timed step
as well by writing a 256 MB buffer outside the step's events.  The same line
carries the varlen prefill (4 sequences {65, 1000, 2048, 3000}, 16 heads,
g ~ U[-2, 0], fp32 initial state), the recurrent decode (256 sequences, fp32
pool, commit), the multi-step verify (64 sequences, 1..12 tokens, bf16 pool +
per-token states), the same verify with the gates formed in the kernel from
raw projections, the decode with per-key-channel gates, the decode with the
gated RMSNorm output epilogue and the long few-head prefill with the
chunk-parallel scan as extra objects, each with its own roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs the same workload on its own GPU (replicas, no
collective on the data path) and rank 0 prints one JSON line with the
whole-job throughput over the slowest rank.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gated_delta_rule_37_gb300 as gdr  # noqa: E402
from gated_delta_rule_37_gb300 import workloads  # noqa: E402

METRIC = "prefill tokens/s (% bf16 TC peak); decode tokens/s (% HBM GB/s) on 1 GB300"
L2_FLUSH_BYTES = 256 << 20

# Algorithmic work per token and value-head (K = V = D, chunk C = 64), split by
# the kernel that performs it.  Tensor-core path (bf16, D = 128):
#   chunk_prep  : K K^T, Q K^T, Tm K (each C*K, triangular) + Tm V (C*V)
#   chunk_chain : W S^T, state update, Q S^T (2*K*V each) + P N (C*V)
# fp32 / D = 64 path: chunk_intra as chunk_prep; chunk_state 4KV; chunk_out 2KV + CV.
# Chunk-parallel scan (GDR_CHUNK_SCAN): chunk_chain_summary forms each
# segment's transition (K columns) and offset (V columns), W S^T and the state
# update for each: 4K(K + V); chunk_seg_scan is fp32 CUDA-core work (not counted).
# Each split sums to 6KV + 3CK + 2CV = 139,264 flop at K = V = 128.


def kernel_flops_per_token_head(name, K, V, C=64):
    return {"chunk_prep": 3 * C * K + C * V, "chunk_chain": 6 * K * V + C * V,
            "chunk_chain_summary": 4 * K * (K + V), "chunk_seg_scan": 0,
            "chunk_intra": 3 * C * K + C * V, "chunk_state": 4 * K * V, "chunk_out": 2 * K * V + C * V}.get(name)


def prefill_flops(T, Hv, K, V, C=64):
    return T * Hv * (6 * K * V + 3 * C * K + 2 * C * V)


def prefill_bytes(case):
    """Algorithmic HBM bytes of one prefill call: inputs read once, outputs
    written once (q, k, v, gate, beta, o, initial and final state)."""
    n = sum(t.numel() * t.element_size() for t in (case.q, case.k, case.v, case.beta))
    n += (case.g if case.g is not None else case.gk).numel() * 4
    n += case.v.numel() * case.v.element_size()  # o
    if case.initial_state is not None:
        n += case.initial_state.numel() * 4
    n += case.N * case.v.shape[1] * case.v.shape[2] * case.q.shape[2] * 4  # final state
    return n


def pool_bytes(case):
    """Algorithmic HBM bytes of one decode / verify call over valid rows:
    slab read, slab write back (commit) or per-token states (verify), and the
    per-token q, k, v, g, beta, o."""
    Hv, V, K = case.pool.shape[1:]
    esz = case.pool.element_size()
    slab = Hv * V * K * esz
    cu = case.cu_seqlens.tolist()
    valid = [b for b in range(case.N) if int(case.state_indices[b]) >= 0]
    toks = sum(cu[b + 1] - cu[b] for b in valid)
    n = len(valid) * slab
    if case.commit:
        n += len(valid) * slab
    if case.steps:
        n += toks * slab
    if case.raw is not None:  # raw projections a, b [Hv] per token (A_log, dt_bias are per head)
        gate_per_tok = 2 * Hv * case.raw["a"].element_size()
    else:  # g [Hv] or, per key channel, [Hv, K] fp32, and beta [Hv]
        gate_per_tok = case.g[0].numel() * 4 + Hv * case.beta.element_size()
    per_tok = 2 * case.q.shape[1] * K * case.q.element_size() + 2 * Hv * V * case.v.element_size() + gate_per_tok
    if case.norm is not None:  # the epilogue's gate [Hv, V] per token
        per_tok += Hv * V * case.norm["gate"].element_size()
    return n + toks * per_tok, toks


class Dist:
    """Process-group plumbing for N > 1 (one process per GPU, replicas): a
    barrier and a max over ranks.  Works with NCCL (GPU tensors) and gloo (CPU
    tensors, used by the tests)."""

    def __init__(self, world: int, device):
        self.world = world
        self.device = device

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return float(x)
        import torch.distributed as dist
        t = torch.tensor([float(x)], dtype=torch.float64, device=self.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())


def whole_job_throughput(units_per_rank: float, ms_per_step_max: float, world: int) -> float:
    """Units all ranks processed in one step / the slowest rank's step time."""
    return world * units_per_rank / (ms_per_step_max / 1e3)


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    record (one record or a list of records per kernel), or None when there is
    no record for this workload or the kernel's source changed since the
    counters were taken."""
    import hashlib
    try:
        recs = json.load(open(TRAFFIC_FILE))[kernel]
    except (OSError, KeyError, ValueError):
        return None
    for rec in recs if isinstance(recs, list) else [recs]:
        if rec.get("workload") != workload:
            continue
        try:
            sha = hashlib.sha256(open(os.path.join(ROOT, rec["source"]), "rb").read()).hexdigest()
        except OSError:
            return None
        return rec["dram_bytes_per_launch"] if sha == rec.get("source_sha256") else None
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sustained=d.get("bf16_tflops_sustained"),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="gdr_clocks_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            rows = f.read().splitlines()
        os.unlink(self.path)
        for line in rows:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def timed_steps(step, K, flush, stream, profile=True):
    """Run K steps, each bracketed by CUDA events on `stream`, with the L2
    flushed (outside the events) before each.  Returns per-step ms and the
    per-kernel profile of an identical pass of K steps run right after: the
    library's per-launch profiling events sit between its launches and would
    keep the kernels of one call from overlapping, so the timed pass runs
    without them."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K):
            flush()
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
    torch.cuda.synchronize()
    prof = {}
    if profile:
        gdr.profile_read()
        gdr.profile_enable(True)
        with torch.cuda.stream(stream):
            for i in range(K):
                flush()
                step()
        torch.cuda.synchronize()
        gdr.profile_enable(False)
        prof = gdr.profile_read()
    return [a.elapsed_time(b) for a, b in evs], prof


def roofline(prof, steps, work_per_kernel, peaks, bound_of, workload=""):
    """Dominant kernel (largest device time) -> roofline object."""
    name = max(prof, key=lambda k: prof[k][0])
    total_ms, launches = prof[name]
    avg_s = total_ms / launches / 1e3
    work = work_per_kernel(name)
    bound = bound_of(name)
    if bound == "hbm":
        ach = work / avg_s / 1e9
        peak, unit = peaks["hbm"], "GB/s"
    else:
        ach = work / avg_s / 1e12
        peak, unit = peaks["bf16"], "TFLOP/s"
    share = {k: round(v[0] / sum(x[0] for x in prof.values()), 4) for k, v in prof.items()}
    return {"kernel": name, "bound": bound, "achieved": round(ach, 3), "peak": peak, "unit": unit,
            "frac": round(ach / peak, 5), "peak_source": peaks["source"], "traffic": ncu_traffic(name, workload),
            "avg_launch_us": round(avg_s * 1e6, 3), "launches": launches, "time_share": share}


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------
class Prefill:
    def __init__(self, case, dev, flags=0):
        self.case = case
        self.flags = flags
        c = case
        self.dev = dev
        self.q, self.k, self.v, self.beta = (t.to(dev) for t in (c.q, c.k, c.v, c.beta))
        self.g = c.g.to(dev) if c.g is not None else None
        self.gk = c.gk.to(dev) if c.gk is not None else None
        self.h0 = c.initial_state.to(dev) if c.initial_state is not None else None
        self.cu = c.cu_seqlens.to(dev)
        d = c.dims
        self.o = torch.empty(c.T, d["Hv"], d["V"], dtype=c.q.dtype, device=dev)
        self.hT = torch.empty(c.N, d["Hv"], d["V"], d["K"], dtype=torch.float32, device=dev)
        gk_kind = gdr.GDR_GATE_SCALAR if c.g is not None else gdr.GDR_GATE_CHANNEL
        dt = gdr.GDR_BF16 if c.q.dtype == torch.bfloat16 else gdr.GDR_F32
        self.ws = torch.empty(gdr.chunk_workspace_size(c.N, c.T, d["Hk"], d["Hv"], d["K"], d["V"],
                                                       gate_kind=gk_kind, dtype=dt, flags=flags),
                              dtype=torch.uint8, device=dev)

    def step(self, stream=None):
        gdr.chunk_fwd(self.q, self.k, self.v, self.beta, self.cu, g=self.g, gk=self.gk, initial_state=self.h0,
                      scale=self.case.scale, flags=self.flags, o=self.o, final_state=self.hT, workspace=self.ws,
                      stream=stream)

    def e2e(self, K, stream):
        """The same call through the public API from pinned host buffers: every
        step copies its inputs host -> device, runs the call and copies o and
        the final state back, all inside the timed region.  Steps are
        pipelined the way a serving loop would run them: inputs and outputs
        are double-buffered on the device, the copies run on their own streams
        and overlap the neighbouring steps' compute."""
        c = self.case
        host_in = [t.pin_memory() for t in (c.q, c.k, c.v, c.beta, c.cu_seqlens)]
        host_in.append((c.g if c.g is not None else c.gk).pin_memory())
        if c.initial_state is not None:
            host_in.append(c.initial_state.pin_memory())
        dev_in = [[torch.empty_like(h, device=self.dev) for h in host_in] for _ in range(2)]
        dev_out = [(torch.empty_like(self.o), torch.empty_like(self.hT)) for _ in range(2)]
        o_host = torch.empty(self.o.shape, dtype=self.o.dtype).pin_memory()
        hT_host = torch.empty(self.hT.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = o_host.numel() * o_host.element_size() + hT_host.numel() * 4
        s_in, s_out = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_ready = [ev() for _ in range(2)]
        in_free = [ev() for _ in range(2)]
        out_ready = [ev() for _ in range(2)]
        out_free = [ev() for _ in range(2)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(K):
            b = i & 1
            if i >= 2:
                s_in.wait_event(in_free[b])
            with torch.cuda.stream(s_in):
                for d, h in zip(dev_in[b], host_in):
                    d.copy_(h, non_blocking=True)
                in_ready[b].record(s_in)
            stream.wait_event(in_ready[b])
            if i >= 2:
                stream.wait_event(out_free[b])
            q, k, v, beta, cu, gate = dev_in[b][:6]
            h0 = dev_in[b][6] if c.initial_state is not None else None
            o, hT = dev_out[b]
            gdr.chunk_fwd(q, k, v, beta, cu, g=gate if c.g is not None else None,
                          gk=gate if c.gk is not None else None, initial_state=h0, scale=c.scale,
                          o=o, final_state=hT, workspace=self.ws, stream=stream)
            in_free[b].record(stream)
            out_ready[b].record(stream)
            s_out.wait_event(out_ready[b])
            with torch.cuda.stream(s_out):
                o_host.copy_(o, non_blocking=True)
                hT_host.copy_(hT, non_blocking=True)
                out_free[b].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        end.record(stream)
        torch.cuda.synchronize()
        ms = start.elapsed_time(end) / K
        return ms, h2d, d2h


def prefill_work_fn(case):
    d = case.dims
    tok_heads = case.T * d["Hv"]

    def work(name):
        f = kernel_flops_per_token_head(name, d["K"], d["V"])
        return 0.0 if f is None else f * tok_heads
    return work


# ---------------------------------------------------------------------------
# decode / verify
# ---------------------------------------------------------------------------
class PoolRun:
    def __init__(self, case, dev):
        self.case = case
        c = case
        self.q, self.k, self.v, self.g, self.beta = (t.to(dev) for t in (c.q, c.k, c.v, c.g, c.beta))
        self.pool = c.pool.to(dev)
        self.idx, self.cu = c.state_indices.to(dev), c.cu_seqlens.to(dev)
        self.o = torch.empty(c.T, c.v.shape[1], c.v.shape[2], dtype=c.q.dtype, device=dev)
        self.ib = None
        if c.steps:
            self.ib = torch.empty((c.ibuf_rows, c.steps) + tuple(c.pool.shape[1:]), dtype=c.pool.dtype, device=dev)
        self.flags = gdr.GDR_COMMIT if c.commit else 0
        self.raw = None if c.raw is None else {n: t.to(dev) for n, t in c.raw.items()}
        self.norm = None if c.norm is None else {n: (t.to(dev) if torch.is_tensor(t) else t) for n, t in c.norm.items()}

    def step(self, stream=None):
        if self.norm is not None:
            gdr.recurrent_fwd_norm(self.q, self.k, self.v, self.g, self.beta, self.pool, self.idx, self.cu,
                                   self.norm["weight"], self.norm["gate"], eps=self.norm["eps"], scale=self.case.scale,
                                   flags=self.flags, o=self.o, intermediate_states=self.ib, stream=stream)
            return
        if self.raw is not None:
            r = self.raw
            gdr.recurrent_fwd_gated(self.q, self.k, self.v, r["a"], r["b"], r["A_log"], r["dt_bias"], self.pool,
                                    self.idx, self.cu, scale=self.case.scale, flags=self.flags, o=self.o,
                                    intermediate_states=self.ib, stream=stream)
            return
        gdr.recurrent_fwd(self.q, self.k, self.v, self.g, self.beta, self.pool, self.idx, self.cu,
                          scale=self.case.scale, flags=self.flags, o=self.o, intermediate_states=self.ib,
                          stream=stream)


def measure(runner, K, W, flush, stream, work_fn, bound_of, peaks, units_per_step):
    for _ in range(W):
        runner.step(stream)
    torch.cuda.synchronize()
    times, prof = timed_steps(lambda: runner.step(stream), K, flush, stream)
    ms = float(np.mean(times))
    return ms, prof, roofline(prof, K, work_fn, peaks, bound_of, runner.case.name), units_per_step / (ms / 1e3)


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine() or "unknown"


ORACLE_SAMPLE_TOKENS = 1024


def oracle_sample(case):
    """A bounded sample of a prefill workload for the oracle: the first
    ORACLE_SAMPLE_TOKENS tokens of its longest sequence (with that sequence's
    initial state), all heads.  Returns (keyword arguments of oracle.tokenwise,
    tokens, description)."""
    cu = case.cu_seqlens.tolist()
    b = max(range(case.N), key=lambda i: cu[i + 1] - cu[i])
    ntok = min(ORACLE_SAMPLE_TOKENS, cu[b + 1] - cu[b])
    sl = slice(cu[b], cu[b] + ntok)
    h0 = case.initial_state[b:b + 1] if case.initial_state is not None else None
    kw = dict(q=case.q[sl], k=case.k[sl], v=case.v[sl], beta=case.beta[sl],
              g=case.g[sl] if case.g is not None else None, gk=case.gk[sl] if case.gk is not None else None,
              initial_state=h0, cu_seqlens=[0, ntok], scale=case.scale)
    Hv = case.v.shape[1]
    return kw, ntok, f"the first {ntok} tokens of the longest sequence x all {Hv} heads of {case.name}"


def cpu_baseline_prefill(case, budget_s=12.0):
    """The oracle as it stands (fp64 tokenwise, OpenMP over sequence x head) on a
    bounded sample of the workload (oracle_sample), repeated until about
    `budget_s` seconds of wall time have passed."""
    import oracle
    args, ntok, what = oracle_sample(case)
    cores = len(os.sched_getaffinity(0))
    oracle.tokenwise(**args, nthreads=cores)      # load + warm
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.tokenwise(**args, nthreads=cores)
        reps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = (time.perf_counter() - t0) / reps
    used = min(cores, oracle.num_threads())  # threads of the run above (the one-core run below changes it)
    # one core: 2 of the heads, scaled to all heads (the oracle's work is
    # independent per (sequence, head))
    Hv, Hk = case.v.shape[1], case.q.shape[1]
    hs = [0, 1]
    kh = sorted({h // (Hv // Hk) for h in hs})
    one = dict(args, q=args["q"][:, kh], k=args["k"][:, kh], v=args["v"][:, hs], beta=args["beta"][:, hs],
               g=args["g"][:, hs] if args["g"] is not None else None,
               gk=args["gk"][:, hs] if args["gk"] is not None else None,
               initial_state=args["initial_state"][:, hs] if args["initial_state"] is not None else None)
    t1 = time.perf_counter()
    oracle.tokenwise(**one, nthreads=1)
    d1 = (time.perf_counter() - t1) * Hv / len(hs)
    return {"value": round(ntok / dt, 2), "unit": "tokens/s", "cores": used, "cpu_model": cpu_model(),
            "kind": "oracle", "sample": f"{what}, {reps} repetitions ({dt * reps:.1f} s)",
            "value_1core": round(ntok / d1, 2),
            "sample_1core": f"the same tokens, {len(hs)} of the {Hv} heads on 1 thread, scaled to all heads"}


def config_of(case):
    d = case.dims
    return {"workload": case.name, "global_batch": case.N, "seq_len": case.T, "heads_k": d["Hk"],
            "heads_v": d["Hv"], "head_dim": d["K"], "chunk": 64,
            "gate": "per-key-channel gk [T, Hv, K]" if case.gk is not None else "scalar g [T, Hv]",
            "parallelism": "replicas", "l2": "flushed (256 MB write) before every timed step"}


def reference_arm(args):
    """--impl reference: the oracle, as it stands, timed on the host cores on a
    bounded sample of the same workload (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    case = workloads.kda_long_prefill(args.kda_T)
    kw, ntok, what = oracle_sample(case)
    cores = len(os.sched_getaffinity(0))
    for _ in range(args.warmup):
        oracle.tokenwise(**kw, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.tokenwise(**kw, nthreads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    val = ntok / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 2), "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(case),
            "cpu_baseline": {"value": round(val, 2), "unit": "tokens/s", "cores": min(cores, oracle.num_threads()),
                             "cpu_model": cpu_model(), "kind": "oracle", "sample": f"{what} per step"},
            "e2e": {"value": round(val, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PREFILL_TARGET_FRAC_BF16 = 0.5  # the chunked prefill's target share of the bf16 tensor peak


def prefill_whole_call(case, ms, peaks):
    """The whole prefill call against both peaks (algorithmic flop and bytes)."""
    d = case.dims
    fl = prefill_flops(case.T, d["Hv"], d["K"], d["V"])
    by = prefill_bytes(case)
    return {"tflops": round(fl / (ms / 1e3) / 1e12, 3), "frac_bf16": round(fl / (ms / 1e3) / 1e12 / peaks["bf16"], 5),
            "gbs": round(by / (ms / 1e3) / 1e9, 2), "frac_hbm": round(by / (ms / 1e3) / 1e9 / peaks["hbm"], 5),
            "algorithmic_flop_per_step": fl, "algorithmic_bytes_per_step": by}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="", help="comma list of extra sections: varlen,decode,verify,kda_decode,"
                                               "verify_gated,decode_norm,long_scan (the headline always runs)")
    ap.add_argument("--kda-T", type=int, default=32768,
                    help="tokens of the long KDA prefill (32768 is the workload; smaller for profiling)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end run (profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        reference_arm(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    gdr.load()
    peaks = load_peaks()
    stream = torch.cuda.Stream()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush = lambda: flush_buf.fill_(1)
    only = set(filter(None, args.only.split(","))) or {"varlen", "decode", "verify", "kda_decode",
                                                        "verify_gated", "decode_norm", "long_scan"}

    dist_ = Dist(world, dev)

    def barrier():
        dist_.barrier()
        torch.cuda.synchronize()

    max_over_ranks = dist_.max

    head_case = workloads.kda_long_prefill(args.kda_T)
    head = Prefill(head_case, dev)
    extra = {}
    var = dec = ver = kdec = vg = dn = None
    if "varlen" in only:
        var = Prefill(workloads.varlen_bf16_prefill(), dev)
    if "decode" in only:
        dec = PoolRun(workloads.decode_fp32_pool(), dev)
    if "kda_decode" in only:
        kdec = PoolRun(workloads.decode_kda_fp32_pool(), dev)
    if "verify_gated" in only:
        vg = PoolRun(workloads.verify_bf16_pool_raw_gates(), dev)
    if "decode_norm" in only:
        dn = PoolRun(workloads.decode_fp32_pool_norm(), dev)
    if "verify" in only:
        ver = PoolRun(workloads.verify_bf16_pool(), dev)
    lsc = lpl = None
    if "long_scan" in only:
        long_case = workloads.long_few_heads_prefill()
        lsc = Prefill(long_case, dev, flags=gdr.GDR_CHUNK_SCAN)
        lpl = Prefill(long_case, dev)
    for _ in range(args.warmup):
        head.step(stream)
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    times, prof = timed_steps(lambda: head.step(stream), args.steps, flush, stream)
    barrier()
    ms = max_over_ranks(float(np.mean(times)))
    launches = sum(v[1] for v in prof.values())
    roof = roofline(prof, args.steps, prefill_work_fn(head_case), peaks, lambda n: "tensor", head_case.name)
    value = whole_job_throughput(head_case.T, ms, world)
    whole = prefill_whole_call(head_case, ms, peaks)
    target = {"prefill_frac_bf16_target": PREFILL_TARGET_FRAC_BF16,
              "dominant_kernel_frac_bf16": roof["frac"], "whole_call_frac_bf16": whole["frac_bf16"],
              "met": roof["frac"] >= PREFILL_TARGET_FRAC_BF16,
              "gap_x": round(PREFILL_TARGET_FRAC_BF16 / max(roof["frac"], 1e-9), 1)}

    if var is not None:
        v_ms, v_prof, v_roof, _ = measure(var, args.steps, args.warmup, flush, stream, prefill_work_fn(var.case),
                                          lambda n: "tensor", peaks, var.case.T)
        launches += sum(v[1] for v in v_prof.values())
        v_ms = max_over_ranks(v_ms)
        extra["varlen_prefill"] = {"workload": var.case.name,
                                   "tokens_per_s": round(world * var.case.T / (v_ms / 1e3), 1),
                                   "ms_per_step": round(v_ms, 5), "roofline": v_roof,
                                   "whole_call": prefill_whole_call(var.case, v_ms, peaks)}
    for key, run in (("decode", dec), ("verify", ver), ("kda_decode", kdec), ("verify_gated", vg),
                     ("decode_norm", dn)):
        if run is None:
            continue
        nbytes, toks = pool_bytes(run.case)
        p_ms, p_prof, p_roof, _ = measure(run, max(args.steps, 20), args.warmup, flush, stream,
                                          lambda n, nb=nbytes: nb, lambda n: "hbm", peaks, toks)
        launches += sum(v[1] for v in p_prof.values())
        p_ms = max_over_ranks(p_ms)
        extra[key] = {"workload": run.case.name, "tokens_per_s": round(world * toks / (p_ms / 1e3), 1),
                      "ms_per_step": round(p_ms, 4), "valid_tokens": toks, "roofline": p_roof}
    if lsc is not None:
        # the long few-head sequence with the chunk-parallel scan, and the
        # one-pass chain on the same inputs for comparison
        nst = max(5, args.steps // 5)
        ls_ms, ls_prof, ls_roof, _ = measure(lsc, nst, args.warmup, flush, stream, prefill_work_fn(lsc.case),
                                             lambda n: "tensor", peaks, lsc.case.T)
        lp_ms, lp_prof, _, _ = measure(lpl, nst, args.warmup, flush, stream, prefill_work_fn(lpl.case),
                                       lambda n: "tensor", peaks, lpl.case.T)
        launches += sum(v[1] for v in ls_prof.values()) + sum(v[1] for v in lp_prof.values())
        ls_ms, lp_ms = max_over_ranks(ls_ms), max_over_ranks(lp_ms)
        extra["long_scan"] = {
            "workload": lsc.case.name, "flags": "GDR_CHUNK_SCAN",
            "tokens_per_s": round(world * lsc.case.T / (ls_ms / 1e3), 1), "ms_per_step": round(ls_ms, 4),
            "one_pass_chain": {"tokens_per_s": round(world * lpl.case.T / (lp_ms / 1e3), 1),
                               "ms_per_step": round(lp_ms, 4),
                               "time_share": {k: round(v[0] / sum(x[0] for x in lp_prof.values()), 4)
                                              for k, v in lp_prof.items()}},
            "speedup_vs_one_pass": round(lp_ms / ls_ms, 3),
            "kernel_ms": {k: round(v[0] / v[1], 4) for k, v in ls_prof.items()},
            "whole_call": prefill_whole_call(lsc.case, ls_ms, peaks),
            "roofline": ls_roof}
    clocks = sampler.stop()

    # end to end through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = head.e2e(max(5, args.steps // 4), stream)
        e2e_ms = max_over_ranks(e2e_ms)
        e2e = {"value": round(world * head_case.T / (e2e_ms / 1e3), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_prefill(head_case)
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": config_of(head_case),
                "roofline": roof, "whole_call": whole, "target": target, "e2e": e2e,
                "gpu_launches": launches, "clocks": clocks, "cpu_baseline": cpu, **extra}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
