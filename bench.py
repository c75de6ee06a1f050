"""Benchmark of the GSI gated linear map on GB300.

Workload (one "step"): the GPT-J-6B-shaped decoder layer at decode, T = 1:
512 sequential tokens, each through three gated linears -- the stacked
q/k/v/fc_in linear (4096 -> 28672), out_proj (4096 -> 4096) and fc_out
(16384 -> 4096) -- with k = 256, eps = 0.10 and exactly one slow token (in
all three linears), i.e. 1536 gsi_forward calls per step, captured in one
CUDA graph.  Inputs are seeded synthetic draws (no trained weights exist
here).  The per-token working set (32 MB) would fit in L2, so the layer is
replicated R times (V_k, M and the handle per replica; W shared, as it is
read only by the slow token) and token t uses replica t mod R: each step
streams ~17 GB and no replica is reused within R x 32 MB >= 4 x L2.

Reported (one JSON line on rank 0): us per gated linear (the metric), the
effective HBM GB/s and its fraction of the measured copy peak (and of
8 TB/s), a roofline object for the decode kernel, an end-to-end number
through the C ABI's host-buffer entry point, the oracle timed on the host
cores, the SM clocks sampled during the timed region, and under "configs"
the other configurations (GPT-2 QKV call, 28-layer GPT-J stack, OPT MLP
slow-fraction sweep, batched T = 512 call), each with its own metric,
roofline fraction and oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gsi|reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs per gated linear & effective HBM GB/s (GPT-J 4096 shapes, B=1) vs roofline"
UNIT = "us per gated linear"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DECODE_KERNEL = "gsi_decode_cr_group_kernel<256> (qkv_fc_in as a group of one; out_proj + fc_out)"
DECODE_SRC = os.path.join(ROOT, "gated_rank_subspace_gsi_gb300", "csrc", "gsi_decode_cr.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gsi_decode_cr__gptj_layer_traffic.txt")


# --------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# --------------------------------------------------------------------------

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """The slowest rank's time (weak scaling: every rank does the same work)."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# peaks, clocks, traffic
# --------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(smax) if smax else None,
                    samples=len(sm), reasons=sorted(reasons))


def kernel_traffic():
    """DRAM bytes per gated linear of the decode kernels from the committed ncu
    summary, if it was taken on the decode kernel source as it is now."""
    try:
        with open(DECODE_SRC, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        vals = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    vals[k.strip()] = v.strip()
        if vals.get("decode_source_sha256_16") != sha:
            return None
        return float(vals["dram_bytes_per_gated_linear"])
    except Exception:
        return None


# --------------------------------------------------------------------------
# workload names (one string per workload, shared by both arms of the bench)
# --------------------------------------------------------------------------

DECODE_WORKLOAD = ("gptj_layer_decode: 512 sequential T=1 tokens x 3 gated linears "
                   "(4096->28672 stacked qkv+fc_in, 4096->4096 out_proj, 16384->4096 fc_out), "
                   "k=256, eps=0.10, 1 slow token (0.2%)")


def cal_workload(n, d, k, iters):
    return (f"calibrate_gptj: n={n} calibration tokens (seeded planted-spectrum activations), "
            f"d={d}, k={k}, {iters} iterations, Q0 seeded Gaussian")


def casc_workload(L, n, d, k, it_first, it_next):
    return (f"cascade_gptj: {L} layers of depth-coherent planted-spectrum calibration tokens "
            f"(adjacent planted subspaces: mean principal cosine ~0.96), n={n}, d={d}, k={k}, "
            f"iterations {it_first} then {it_next}")


BATCHED_METRIC = "µs per gated linear call, batched T=512 prefill (4096 -> 16384, k=256, 30% slow)"
BATCHED_UNIT = "us per gated linear call"
BATCHED_WORKLOAD = ("batched_T512: T=512 tokens per call, W 16384x4096, k=256, eps=0.10, "
                    "154 slow / 358 fast tokens")
GPT2_METRIC = "µs per gated linear call, GPT-2 QKV T=64"
GPT2_UNIT = "us per call"
GPT2_WORKLOAD = "gpt2_qkv_T64: 768 -> 2304, k=256, eps=0.10, T=64 tokens per call, 6 slow"
STACK_METRIC = "µs per decode step through a 28-layer GPT-J stack (3 gated linears per layer)"
STACK_UNIT = "us per decode step"
OPT_METRIC = "µs per OPT-6.7B MLP layer (fc1 + fc2) at decode, slow-fraction sweep"
OPT_UNIT = "us per layer (f = 0 point)"


def stack_workload(S, n_slow):
    return ("gptj_stack: 28 layers x (4096->28672 qkv+fc_in, then 4096->4096 out_proj || "
            f"16384->4096 fc_out grouped), k=256, eps=0.10, {S} decode steps, {n_slow} slow draws")


def opt_workload(S):
    return (f"opt_mlp: 32 layers x (4096->16384 fc1, 16384->4096 fc2), k=256, eps=0.05, "
            f"{S} decode steps per point")


def sweep_workload(T):
    return (f"sweep_gptj: W 28672x4096, k in {list(SWEEP_KS)}, eps in "
            f"[0.02, 0.05, 0.10, 0.20, inf], {T} sequential decode tokens per point (gapless "
            f"power-law spectrum, r=1024), V_k = population top-k basis")


# --------------------------------------------------------------------------
# the workload
# --------------------------------------------------------------------------

def build_layer(n_tokens: int, replicas: int):
    """Device tensors, handles and groups of the GPT-J decode layer workload:
    per replica r the three handles and one group of out_proj and fc_out
    (their inputs, the attention output and the GELU of fc_in, do not depend
    on each other: GPT-J's parallel residual).  Prefetch links are set by
    link_schedule()."""
    import torch

    import gsi_inputs as gi
    from gated_rank_subspace_gsi_gb300 import lib

    wl = gi.gptj_layer(n_tokens)
    slow = gi.slow_positions(n_tokens, wl.extra["n_slow"], wl.seed)
    layer = []
    for li, spec in enumerate(wl.linears):
        W = gi.gaussian_weights(spec.d_out, spec.d, wl.seed, li, device="cuda")
        basis = gi.random_basis(spec.d, spec.k, wl.seed, li)
        rs = gi.rho_targets(n_tokens, spec.rho_fast, spec.rho_slow, slow, wl.seed, li)
        X = gi.tokens(basis, rs, wl.seed, li)
        V = torch.from_numpy(basis.V_bits.view(np.int16)).view(torch.bfloat16).cuda()
        M = torch.empty((spec.d_out, spec.k), dtype=torch.bfloat16, device="cuda")
        lib.gsi_precompute_M(W, V, M)
        reps = []
        for r in range(replicas):
            Vr = V if r == 0 else V.clone()
            Mr = M if r == 0 else M.clone()
            torch.cuda.synchronize()
            h = lib.gsi_create(W, Vr, Mr, spec.eps)
            reps.append((Vr, Mr, h))
        x = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
        layer.append(dict(spec=spec, W=W, reps=reps, x=x, X_bits=X, basis=basis,
                          y=torch.zeros((n_tokens, spec.d_out), dtype=torch.float32, device="cuda"),
                          gate=torch.zeros((n_tokens,), dtype=torch.uint8, device="cuda"),
                          rho=torch.zeros((n_tokens,), dtype=torch.float32, device="cuda")))
    groups = [lib.gsi_group_create([layer[1]["reps"][r][2], layer[2]["reps"][r][2]])
              for r in range(replicas)]
    torch.cuda.synchronize()
    return wl, slow, layer, groups


def link_schedule(layer, groups, replicas, schedule: str, prefetch: int):
    """Prefetch links in the order the schedule issues its launches: each
    launch streams the operands of the launch `prefetch` places later into
    L2 (0: no links).  sequential: linear 0, 1, 2 of replica r, then replica
    r + 1; grouped: linear 0 of replica r, then the group of replica r."""
    from gated_rank_subspace_gsi_gb300 import lib
    for L in layer:
        for (_, _, h) in L["reps"]:
            lib.gsi_set_prefetch(h, None)
    for g in groups:
        lib.gsi_group_set_prefetch(g, None)
    if prefetch <= 0:
        return
    if schedule == "sequential":
        order = [layer[li]["reps"][r][2] for r in range(replicas) for li in range(len(layer))]
        for i, h in enumerate(order):
            lib.gsi_set_prefetch(h, order[(i + prefetch) % len(order)])
        return
    for r in range(replicas):
        lib.gsi_set_prefetch_group(layer[0]["reps"][r][2], groups[r])
        lib.gsi_group_set_prefetch(groups[r], layer[0]["reps"][(r + 1) % replicas][2])


def correction_bytes(k: int) -> int:
    """The bf16 upper 16 x 16 tiles of E = V_k^T V_k - I that every one-token
    call reads to form ||r||: (k/16)(k/16 + 1)/2 tiles of 512 bytes."""
    t = k // 16
    return t * (t + 1) // 2 * 512


def linear_bytes(s, n_tokens: int, n_slow: int) -> float:
    """Algorithmic bytes of n_tokens one-token calls of one gated linear:
    V_k + correction triangle + x + y (fp32) + gate + rho per call, plus M
    per fast call or W per slow call."""
    per_call = s.d * s.k * 2 + correction_bytes(s.k) + s.d * 2 + s.d_out * 4 + 5
    return (per_call * n_tokens + s.d_out * s.k * 2 * (n_tokens - n_slow)
            + s.d_out * s.d * 2 * n_slow)


def step_bytes(layer, slow) -> float:
    """Algorithmic bytes of one step (all gated linears, all tokens)."""
    n_slow = int(slow.sum())
    return float(sum(linear_bytes(L["spec"], len(slow), n_slow) for L in layer))


def capture_step(layer, n_tokens, replicas, stream, handles_subset=None, host=None,
                 groups=None):
    """One step in a CUDA graph.  With `groups` (the grouped schedule) each
    token is a call on linear 0 and one launch of its replica's group;
    otherwise one call per linear in `handles_subset` (all by default), in
    order, on device buffers or (host) through gsi_forward_host."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            record_step(layer, n_tokens, replicas, stream, handles_subset, host, groups)
    return g


def record_step(layer, n_tokens, replicas, stream, handles_subset=None, host=None, groups=None):
    """Issue one step's calls on `stream` (inside a graph capture)."""
    from gated_rank_subspace_gsi_gb300 import lib
    idx = range(len(layer)) if handles_subset is None else handles_subset
    for t in range(n_tokens):
        r = t % replicas
        if groups is not None:
            sl = slice(t, t + 1)
            if host is not None:  # host buffers: the C ABI's host-buffer entries
                if 0 in idx:
                    H = host[0]
                    lib.gsi_forward_host(layer[0]["reps"][r][2], H["x"][sl], H["yp"][t],
                                         H["gp"][t], H["rp"][t], stream)
                if 1 in idx or 2 in idx:
                    Hs = host[1:]
                    lib.gsi_group_forward_host(groups[r], [H["x"][sl] for H in Hs],
                                               [H["yp"][t] for H in Hs], [H["gp"][t] for H in Hs],
                                               [H["rp"][t] for H in Hs], stream)
                continue
            if 0 in idx:
                L0 = layer[0]
                lib.gsi_forward(L0["reps"][r][2], L0["x"][sl], L0["y"][sl], L0["gate"][sl],
                                L0["rho"][sl], stream)
            if 1 in idx or 2 in idx:
                m = layer[1:]
                lib.gsi_group_forward(groups[r], [L["x"][sl] for L in m],
                                      [L["y"][sl] for L in m], [L["gate"][sl] for L in m],
                                      [L["rho"][sl] for L in m], stream)
            continue
        for li in idx:
            L = layer[li]
            h = L["reps"][r][2]
            if host is None:
                lib.gsi_forward(h, L["x"][t:t + 1], L["y"][t:t + 1], L["gate"][t:t + 1],
                                L["rho"][t:t + 1], stream)
            else:
                H = host[li]
                lib.gsi_forward_host(h, H["x"][t:t + 1], H["yp"][t], H["gp"][t], H["rp"][t],
                                     stream)


def _release():
    """Return freed device memory to the driver between workloads."""
    import gc

    import torch
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def replay(graph, stream, n: int):
    """Replay on `stream` (a graph launches on torch's current stream)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(n):
            graph.replay()


def time_graph(graph, stream, reps: int, warmup: int):
    import torch
    replay(graph, stream, warmup)
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    replay(graph, stream, reps)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps  # ms per replay


def cpu_baseline(layer, slow, budget_s: float = 12.0):
    """The fp64 oracle as it stands, on this host's cores, on a bounded
    sample of the step: the slow token plus fast tokens until the budget."""
    import oracle
    orc = oracle.default()
    prep = []
    for L in layer:
        s = L["spec"]
        W_bits = L["W"].view(__import__("torch").int16).cpu().numpy().view(np.uint16)
        M_ref = orc.precompute_M_bf16(W_bits, L["basis"].V_bits)
        prep.append((orc.bf16_decode(W_bits), orc.bf16_decode(L["basis"].V_bits),
                     orc.bf16_decode(M_ref), float(np.float32(s.eps)), L["X_bits"]))
    order = list(np.nonzero(slow)[0]) + [t for t in range(len(slow)) if not slow[t]]
    n_lin = 0
    t0 = time.perf_counter()
    for t in order:
        for (W, V, M, eps, X) in prep:
            orc.forward(W, V, M, eps, orc.bf16_decode(X[t:t + 1]))
            n_lin += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    n_tok = n_lin // len(prep)
    return dict(value=dt / n_lin * 1e6, unit=UNIT, cores=orc.num_threads(), kind="oracle",
                sample=f"{n_tok} decode tokens x 3 gated linears of the step (the slow "
                       f"token first, then fast tokens), fp64 C oracle, {dt:.1f} s")


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def run_gsi(args, world, rank, local):
    import torch

    from gated_rank_subspace_gsi_gb300 import lib
    torch.cuda.set_device(local)
    lib.library()
    n_tokens = 512
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    per_token = 32.44e6
    replicas = max(16, int(math.ceil(4 * l2 / per_token)))
    wl, slow, layer, groups = build_layer(n_tokens, replicas)
    nbytes = step_bytes(layer, slow)
    n_lin = n_tokens * len(layer)
    stream = torch.cuda.Stream()
    grouped = args.schedule == "grouped"
    other = "sequential" if grouped else "grouped"

    # the other schedule's graph first (links are captured with the graph)
    link_schedule(layer, groups, replicas, other, args.prefetch)
    graph_other = None if args.no_extras else capture_step(
        layer, n_tokens, replicas, stream, groups=groups if not grouped else None)
    link_schedule(layer, groups, replicas, args.schedule, args.prefetch)
    graph = capture_step(layer, n_tokens, replicas, stream, groups=groups if grouped else None)
    for L in layer:
        L["gate"].fill_(7)
    torch.cuda.synchronize()
    replay(graph, stream, max(args.warmup, 3))
    stream.synchronize()
    for L in layer:
        st = lib.gsi_device_status(L["reps"][0][2], stream)
        if st != 0:
            raise RuntimeError(f"device status: {lib.gsi_status_string(st)}")
        if not np.array_equal(L["gate"].cpu().numpy().astype(bool), slow):
            raise RuntimeError("gates differ from the generated slow/fast mix")

    # ---- timed region: K steps, barrier + synchronize on both sides -------
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    replay(graph, stream, args.steps)
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ms_local = e0.elapsed_time(e1) / args.steps
    clk = clocks.stop()
    ms = max_over_ranks(ms_local, world)

    us_per_lin = ms * 1e3 / n_lin
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    schedules = {args.schedule: round(us_per_lin, 4)}
    if graph_other is not None:
        ms_o = max_over_ranks(time_graph(graph_other, stream, reps=max(3, args.steps // 10),
                                         warmup=2), world)
        schedules[other] = round(ms_o * 1e3 / n_lin, 4)
        del graph_other

    # ---- per-launch breakdown: each linear (or the group) alone ----------
    per = {}
    parts = [([0], "qkv_fc_in"), ([1, 2], "out_proj+fc_out (one grouped launch)")] if grouped \
        else [([li], L["spec"].name) for li, L in enumerate(layer)]
    for subset, name in (parts if not args.no_extras else []):
        g1 = capture_step(layer, n_tokens, replicas, stream, handles_subset=subset,
                          groups=groups if grouped else None)
        ms1 = time_graph(g1, stream, reps=5, warmup=2)
        b1 = sum(linear_bytes(layer[li]["spec"], n_tokens, int(slow.sum())) for li in subset)
        per[name] = dict(us_per_launch=round(ms1 * 1e3 / n_tokens, 3),
                         gbs=round(b1 / (ms1 * 1e-3) / 1e9, 1))
        del g1

    # ---- end to end through the C ABI's host-buffer call: every call's x and
    # its y, rho and gate in page-locked host memory (y, rho and gate
    # consecutive), sequential schedule (the grouped launch has no host-buffer
    # form) ---------------------------------------------------------------
    host = []
    h2d = d2h = 0
    ms_call = ms_bulk = float("nan")
    for L in (layer if not args.no_extras else []):
        s_ = L["spec"]
        stride = (s_.d_out * 4 + 5 + 15) // 16 * 16
        buf = torch.empty((n_tokens, stride), dtype=torch.uint8).pin_memory()
        H = dict(x=L["x"].cpu().pin_memory(), buf=buf,
                 yp=[buf[t, :4 * s_.d_out].view(torch.float32).view(1, s_.d_out)
                     for t in range(n_tokens)],
                 rp=[buf[t, 4 * s_.d_out:4 * s_.d_out + 4].view(torch.float32)
                     for t in range(n_tokens)],
                 gp=[buf[t, 4 * s_.d_out + 4:4 * s_.d_out + 5] for t in range(n_tokens)])
        host.append(H)
        h2d += n_tokens * s_.d * 2
        d2h += n_tokens * (s_.d_out * 4 + 5)
    if host:
        link_schedule(layer, groups, replicas, args.schedule, args.prefetch)
        gc_ = capture_step(layer, n_tokens, replicas, stream, host=host,
                           groups=groups if args.schedule == "grouped" else None)
        for H in host:
            H["buf"].fill_(0xEE)
        ms_call = max_over_ranks(time_graph(gc_, stream, reps=max(3, args.steps // 10), warmup=2),
                                 world)
        gates_h = np.array([int(g[0]) for g in host[0]["gp"]], dtype=bool)
        if not np.array_equal(gates_h, slow):
            raise RuntimeError("host-buffer gates differ from the generated mix")
        del gc_
        link_schedule(layer, groups, replicas, args.schedule, args.prefetch)
        # the same step with one bulk copy of all its inputs and outputs
        # around the device calls (torch copies), for comparison
        ge = torch.cuda.CUDAGraph()
        bulk = [dict(x=H["x"], y=torch.empty((n_tokens, L["spec"].d_out),
                                                 dtype=torch.float32).pin_memory())
                for L, H in zip(layer, host)]
        with torch.cuda.stream(stream):
            with torch.cuda.graph(ge, stream=stream):
                for L, B in zip(layer, bulk):
                    L["x"].copy_(B["x"], non_blocking=True)
                record_step(layer, n_tokens, replicas, stream, groups=groups if grouped else None)
                for L, B in zip(layer, bulk):
                    B["y"].copy_(L["y"], non_blocking=True)
        ms_bulk = max_over_ranks(time_graph(ge, stream, reps=max(3, args.steps // 10), warmup=2),
                                 world)
        del ge

    launches = args.steps * n_tokens * (2 if grouped else len(layer))
    out = {
        "metric": METRIC,
        "value": round(us_per_lin, 4),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded Gaussian weights, QR bases, activations with set residual ratios)",
        "impl": "gsi",
        "config": {
            "workload": DECODE_WORKLOAD,
            "schedule": ("grouped: per token the qkv+fc_in call, then out_proj and fc_out in "
                         "one launch (independent inputs: parallel residual)") if grouped
                        else "sequential: three launches per token",
            "gated_linears_per_step": n_lin,
            "replicas": replicas,
            "l2": f"inputs larger than L2: {replicas} replicas x 32.4 MB per token, "
                  f"{nbytes / 1e9:.2f} GB streamed per step, L2 {l2 / 2**20:.0f} MiB",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "l2_prefetch_distance": args.prefetch,
        },
        "effective_hbm_gbs": round(gbs * world, 1),
        "frac_of_measured_hbm": round(gbs / peak, 4),
        "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
        "us_per_layer": round(ms * 1e3 / n_tokens, 3),
        "per_launch": per,
        "schedules_us_per_linear": schedules,
        "algorithmic_bytes_per_step": int(nbytes),
        "roofline": {
            "bound": "hbm",
            "achieved": round(gbs, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(gbs / peak, 4),
            "traffic": kernel_traffic(),
            "kernel": DECODE_KERNEL,
            "peak_kind": f"{peak_kind} HBM copy",
            "per": "gated linear (achieved = algorithmic bytes per gated linear / us per gated linear)",
            "bytes_per_gated_linear": round(nbytes / n_lin, 1),
            "us_per_gated_linear": round(us_per_lin, 4),
        },
        "e2e": {
            "value": None if math.isnan(ms_call) else round(ms_call * 1e3 / n_lin, 4),
            "unit": UNIT,
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "how": "every call through the C ABI's host-buffer entries (gsi_forward_host, "
                   "gsi_group_forward_host) on page-locked host buffers, in the same schedule "
                   "as the device step: a one-CTA-per-call kernel brings x over the host link "
                   "into device staging and the one-token kernel writes y, rho and gate in place "
                   "(no copy nodes), graph-captured",
            "copies_per_call": 0,
            "bulk_copies_us_per_linear": None if math.isnan(ms_bulk)
            else round(ms_bulk * 1e3 / n_lin, 4),
            "bulk_copies_how": "one torch copy of all the step's x in and of all its y out around "
                               "the device calls (grouped schedule)",
        },
        "gpu_launches": launches,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(layer, slow, budget_s=args.cpu_budget)
    if not args.no_extras and not args.no_configs:
        # the other configurations, each measured on its own after the decode
        # layer's memory is returned
        del graph
        for g in groups:
            lib.gsi_group_destroy(g)
        for L in layer:
            for (_, _, h) in L["reps"]:
                lib.gsi_destroy(h)
        del layer, groups
        _release()
        out["configs"] = measure_configs(args, world, rank, local)
        out["gpu_launches"] = launches + sum(c["gpu_launches"] for c in out["configs"].values())
    if rank == 0:
        print(json.dumps(out), flush=True)


def measure_configs(args, world, rank, local):
    """The GPT-2 QKV call, the 28-layer GPT-J stack, the OPT MLP slow-fraction
    sweep and the batched T = 512 call, each with its own metric, roofline
    fraction and oracle baseline on a bounded sample (the same fields as the
    headline line)."""
    res = {}
    for key, wname, fn in (("gpt2_qkv_T64", "gpt2_qkv_T64", measure_gpt2),
                           ("gptj_stack", "gptj_stack", measure_stack),
                           ("opt_mlp", "opt_mlp", measure_opt),
                           ("batched_T512", "batched_T512", measure_batched)):
        d = fn(args, world, rank, local)
        e = {k: d[k] for k in ("metric", "value", "unit", "steps", "ms_per_step") if k in d}
        e["workload"] = d["config"]["workload"]
        e["roofline"] = {k: d["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                       "peak_kind") if k in d["roofline"]}
        for k in ("tensor", "curve", "us_per_gated_linear", "e2e", "clocks", "gpu_launches"):
            if k in d:
                e[k] = d[k]
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            e["cpu_baseline"] = ref_linear(wname, 1)[4]
        res[key] = e
    return res


def run_gsi_rowshard(args, world, rank, local):
    """The decode layer split by rows over the ranks (one GPU each): rank r
    holds rows row_ranges(d_out, N)[r] of every linear's W and M and the full
    V_k, computes g, rho and the gate itself, and the y parts of each call are
    gathered (NCCL all_gather) before the next call.  Strong scaling: the N
    ranks share one layer.  Calls are issued one by one (no CUDA graph)."""
    import torch

    import gsi_inputs as gi
    from gated_rank_subspace_gsi_gb300 import lib, shard
    torch.cuda.set_device(local)
    lib.library()
    n_tokens = 512
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    replicas = max(16, int(math.ceil(4 * l2 * world / 32.44e6)))
    wl = gi.gptj_layer(n_tokens)
    slow = gi.slow_positions(n_tokens, wl.extra["n_slow"], wl.seed)
    layer = []
    for li, spec in enumerate(wl.linears):
        W = gi.gaussian_weights(spec.d_out, spec.d, wl.seed, li, device="cuda")
        basis = gi.random_basis(spec.d, spec.k, wl.seed, li)
        rs = gi.rho_targets(n_tokens, spec.rho_fast, spec.rho_slow, slow, wl.seed, li)
        X = gi.tokens(basis, rs, wl.seed, li)
        V = torch.from_numpy(basis.V_bits.view(np.int16)).view(torch.bfloat16).cuda()
        M = torch.empty((spec.d_out, spec.k), dtype=torch.bfloat16, device="cuda")
        lib.gsi_precompute_M(W, V, M)
        torch.cuda.synchronize()
        parts = []
        for r in range(replicas):
            Vr = V if r == 0 else V.clone()
            Mr = M if r == 0 else M.clone()
            parts.append((Vr, Mr, shard.RowShard(W, Vr, Mr, spec.eps, rank, world)))
        x = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
        layer.append(dict(spec=spec, W=W, parts=parts, x=x,
                          y=torch.zeros((n_tokens, spec.d_out), dtype=torch.float32, device="cuda"),
                          gate=torch.zeros((n_tokens,), dtype=torch.uint8, device="cuda")))
    stream = torch.cuda.current_stream()

    def step():
        for t in range(n_tokens):
            r = t % replicas
            for L in layer:
                p = L["parts"][r][2]
                y, g, _ = p.forward(L["x"][t:t + 1], stream=stream)
                L["y"][t:t + 1].copy_(y)
                L["gate"][t:t + 1].copy_(g)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    for L in layer:
        if not np.array_equal(L["gate"].cpu().numpy().astype(bool), slow):
            raise RuntimeError("gates differ from the generated slow/fast mix")
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    e1.synchronize()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    clk = clocks.stop()
    n_lin = n_tokens * len(layer)
    nbytes = step_bytes([dict(spec=L["spec"]) for L in layer], slow)
    peak, peak_kind = hbm_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(ms * 1e3 / n_lin, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": False, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian weights, QR bases, activations with set residual ratios)",
        "impl": "gsi",
        "config": {"workload": DECODE_WORKLOAD,
                   "parallelism": f"rows x{world}: W and M split by output rows, V_k and the gate "
                                  f"replicated, y parts all-gathered after every call",
                   "schedule": "sequential, calls issued one by one (no CUDA graph)",
                   "replicas": replicas},
        "effective_hbm_gbs": round(gbs, 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs / world, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / world / peak, 4), "traffic": None,
                     "kernel": DECODE_KERNEL + " (per GPU)", "peak_kind": f"{peak_kind} HBM copy"},
        "gpu_launches": args.steps * n_tokens * len(layer),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def measure_batched(args, world, rank, local):
    """The batched prefill-style gated linear: T = 512 tokens per call through
    one 4096 -> 16384 linear (k = 256, eps = 0.10, 154 slow tokens at seeded
    positions): projection, gate, compaction, gather and the two tcgen05
    GEMMs.  R replicas of (W, V_k, M) cycle so that the calls stream more than
    L2 holds."""
    import torch

    import gsi_inputs as gi
    from gated_rank_subspace_gsi_gb300 import lib
    torch.cuda.set_device(local)
    lib.library()
    wl = gi.batched_prefill()
    spec = wl.linears[0]
    T, n_slow = wl.T, wl.extra["n_slow"]
    inp = gi.make_linear_inputs(spec, T, n_slow, wl.seed, w_device="cuda")
    V = torch.from_numpy(inp.basis.V_bits.view(np.int16)).view(torch.bfloat16).cuda()
    M = torch.empty((spec.d_out, spec.k), dtype=torch.bfloat16, device="cuda")
    lib.gsi_precompute_M(inp.W, V, M)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    w_bytes = spec.d_out * spec.d * 2
    replicas = max(2, int(math.ceil(4 * l2 / w_bytes)))
    reps = []
    for r in range(replicas):
        Wr = inp.W if r == 0 else inp.W.clone()
        Vr = V if r == 0 else V.clone()
        Mr = M if r == 0 else M.clone()
        torch.cuda.synchronize()
        reps.append((Wr, Vr, Mr, lib.gsi_create(Wr, Vr, Mr, spec.eps)))
    x = torch.from_numpy(inp.X_bits.view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.zeros((T, spec.d_out), dtype=torch.float32, device="cuda")
    gate = torch.zeros((T,), dtype=torch.uint8, device="cuda")
    rho = torch.zeros((T,), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    calls = 2 * replicas
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for c in range(calls):
                lib.gsi_forward(reps[c % replicas][3], x, y, gate, rho, stream)
    replay(graph, stream, max(args.warmup, 3))
    stream.synchronize()
    st = lib.gsi_device_status(reps[0][3], stream)
    if st != 0:
        raise RuntimeError(f"device status: {lib.gsi_status_string(st)}")
    if not np.array_equal(gate.cpu().numpy().astype(bool), inp.slow_mask):
        raise RuntimeError("gates differ from the generated slow/fast mix")
    steps = max(1, args.steps // 10)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    replay(graph, stream, steps)
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ms_local = e0.elapsed_time(e1) / steps
    clk = clocks.stop()
    ms = max_over_ranks(ms_local, world)
    us_call = ms * 1e3 / calls
    n_fast = T - n_slow
    nbytes = (T * spec.d * 2 + spec.d * spec.k * 2 + spec.k * spec.k * 4 + spec.d_out * spec.k * 2
              + w_bytes + T * spec.d_out * 4 + T * 5)
    flops = 2.0 * (T * spec.d * spec.k + n_fast * spec.k * spec.d_out * 2
                   + n_slow * spec.d * spec.d_out)
    peak, peak_kind = hbm_peak()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpk = float(json.load(f)["bf16_tflops"])
        tpk_kind = "measured bf16 burst"
    except Exception:
        tpk, tpk_kind = 1900.0, "fallback bf16 burst"
    gbs = nbytes / (us_call * 1e-6) / 1e9
    tfs = flops / (us_call * 1e-6) / 1e12
    # end to end: pinned host x in, y / gate / rho out, per call
    Hx = x.cpu().pin_memory()
    Hbuf = torch.empty((T * (spec.d_out * 4 + 5),), dtype=torch.uint8).pin_memory()
    Hy = Hbuf[:T * spec.d_out * 4].view(torch.float32).view(T, spec.d_out)
    Hr = Hbuf[T * spec.d_out * 4:T * spec.d_out * 4 + 4 * T].view(torch.float32)
    Hg = Hbuf[T * spec.d_out * 4 + 4 * T:]
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(ge, stream=stream):
            for c in range(calls):
                lib.gsi_forward_host(reps[c % replicas][3], Hx, Hy, Hg, Hr, stream)
    ms_e2e = max_over_ranks(time_graph(ge, stream, reps=max(3, steps), warmup=2), world)
    launches_per_call = lib.gsi_forward_launch_count(reps[0][3], T)
    out = {
        "metric": BATCHED_METRIC,
        "value": round(us_call, 3), "unit": BATCHED_UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian weights, QR basis, activations with set residual ratios)",
        "impl": "gsi",
        "config": {"workload": BATCHED_WORKLOAD,
                   "calls_per_step": calls, "replicas": replicas,
                   "l2": f"inputs larger than L2: {replicas} replicas of W/V_k/M "
                         f"({w_bytes / 2**20:.0f} MiB W each), L2 {l2 / 2**20:.0f} MiB",
                   "parallelism": "1 GPU" if world == 1 else f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None, "kernel": "whole call",
                     "peak_kind": f"{peak_kind} HBM copy", "bytes_per_call": int(nbytes)},
        "tensor": {"achieved": round(tfs, 1), "peak": tpk, "unit": "TFLOP/s",
                   "frac": round(tfs / tpk, 4), "peak_kind": tpk_kind,
                   "flops_per_call": flops},
        "e2e": {"value": round(ms_e2e * 1e3 / calls, 3), "unit": "us per gated linear call",
                "h2d_bytes_per_step": calls * T * spec.d * 2,
                "d2h_bytes_per_step": calls * T * (spec.d_out * 4 + 5),
                "how": "gsi_forward_host per call on pinned host buffers: x copied in, the "
                       "kernels write y, rho and gate in place over the host link while "
                       "they run, graph-captured",
                "copies_per_call": 1},
        "gpu_launches": steps * calls * launches_per_call,
        "clocks": clk,
    }
    del graph, ge
    for rep in reps:
        lib.gsi_destroy(rep[3])
    del reps
    _release()
    return out


def run_batched(args, world, rank, local):
    out = measure_batched(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)


CAL_METRIC = ("ms per calibration of V_k, GPT-J-shaped linear input (n=2048 calibration tokens, "
              "d=4096, k=256, 8 block power iterations)")
CAL_UNIT = "ms per calibration"


def _cal_inputs():
    import gsi_inputs as gi
    c = gi.calibration_gptj()
    cs = gi.calibration_activations(c["n"], c["d"], c["k"], seed=c["seed"])
    Q0 = gi.calibration_start(c["d"], c["k"], seed=c["seed"])
    return c, cs, Q0


def cal_cpu_baseline(c, cs, Q0, budget_s: float = 12.0):
    """The oracle's subspace iteration (numpy fp64, the host BLAS threads) on
    the same inputs: whole calibrations until the budget is spent."""
    import gsi_inputs as gi
    from oracle import calibration as cal
    X = gi.bf16_bits_to_f64(cs.X_bits)
    Q = gi.bf16_bits_to_f64(Q0)
    n_done = 0
    t0 = time.perf_counter()
    while True:
        cal.subspace_iteration(X, Q, c["iters"])
        n_done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return dict(value=round(dt / n_done * 1e3, 3), unit=CAL_UNIT, cores=os.cpu_count(),
                kind="oracle",
                sample=f"{n_done} whole calibrations (fp64 numpy subspace iteration, "
                       f"Householder QR per iteration), {dt:.1f} s")


def run_calibrate(args, world, rank, local):
    """Calibration of one GPT-J-shaped linear's basis: n = 2048 tokens (one
    GPT-J context), d = 4096, k = 256, 8 iterations of block power iteration
    with CholeskyQR2, through gsi_calibrate.  R replicas of the calibration
    tokens cycle so that the inputs stream from HBM (more than L2 holds)."""
    import torch

    from gated_rank_subspace_gsi_gb300 import lib
    torch.cuda.set_device(local)
    lib.library()
    c, cs, Q0b = _cal_inputs()
    n, d, k, iters = c["n"], c["d"], c["k"], c["iters"]
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    x_bytes = n * d * 2
    replicas = max(2, int(math.ceil(1.5 * l2 / x_bytes)))
    X0 = torch.from_numpy(cs.X_bits.view(np.int16)).view(torch.bfloat16).cuda()
    Xs = [X0] + [X0.clone() for _ in range(replicas - 1)]
    Q0 = torch.from_numpy(Q0b.view(np.int16)).view(torch.bfloat16).cuda()
    V = torch.empty((d, k), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(lib.gsi_calibrate_workspace_size(n, d, k), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    calls = replicas
    with torch.cuda.stream(stream):
        lib.gsi_calibrate(Xs[0], Q0, iters, V, ws, stream)   # attributes, first-use setup
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for r in range(calls):
                lib.gsi_calibrate(Xs[r], Q0, iters, V, ws, stream)
    replay(graph, stream, max(args.warmup, 3))
    st = lib.gsi_calibrate_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"calibration status: {lib.gsi_status_string(st)}")
    steps = max(1, args.steps // 30)
    ms, clk = _timed(graph, stream, steps, args.warmup, world, local)
    ms_cal = ms / calls
    # end to end: pinned host X and Q0 in, V out, per calibration
    Hx = torch.from_numpy(cs.X_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    Hq = torch.from_numpy(Q0b.view(np.int16)).view(torch.bfloat16).pin_memory()
    Hv = torch.empty((d, k), dtype=torch.bfloat16).pin_memory()
    Xd = torch.empty_like(X0)
    Qd = torch.empty_like(Q0)
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(ge, stream=stream):
            for r in range(calls):
                Xd.copy_(Hx, non_blocking=True)
                Qd.copy_(Hq, non_blocking=True)
                lib.gsi_calibrate(Xd, Qd, iters, V, ws, stream)
                Hv.copy_(V, non_blocking=True)
    ms_e2e = max_over_ranks(time_graph(ge, stream, reps=max(3, steps), warmup=2), world)
    launches = lib.gsi_calibrate_launch_count(n, d, k, iters)
    flops_gemm = 2 * 2.0 * n * d * k * iters          # Z = X Q and Y = X^T Z per iteration
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cal_cpu_baseline(c, cs, Q0b, budget_s=args.cpu_budget)
    rl = cal_roofline(lib, Xs[0], Q0, iters, V, ws, stream, k)
    out = _line(CAL_METRIC, round(ms_cal, 4), CAL_UNIT, world, steps, args.warmup, ms,
                {"workload": cal_workload(n, d, k, iters),
                 "calls_per_step": calls, "replicas": replicas,
                 "l2": f"inputs larger than L2: {replicas} replicas of X "
                       f"({x_bytes / 2**20:.0f} MiB each), L2 {l2 / 2**20:.0f} MiB",
                 "parallelism": "1 GPU" if world == 1 else f"replicas x{world}"},
                roofline=rl,
                tensor_gemm_tflops=round(flops_gemm / (ms_cal * 1e-3) / 1e12, 2),
                e2e={"value": round(ms_e2e / calls, 4), "unit": CAL_UNIT,
                     "h2d_bytes_per_step": calls * (n * d * 2 + d * k * 2),
                     "d2h_bytes_per_step": calls * d * k * 2,
                     "how": "pinned X, Q0 copied in and V_k copied out around each "
                            "gsi_calibrate, graph-captured"},
                gpu_launches=steps * calls * launches, clocks=clk)
    out["data"] = ("synthetic (seeded planted-spectrum calibration activations, seeded "
                   "Gaussian start block)")
    out["dtype"] = "bf16 GEMMs, fp32 orthonormalisation"
    if cpu is not None:
        out["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(out), flush=True)


CAL_SRC = os.path.join(ROOT, "gated_rank_subspace_gsi_gb300", "csrc", "gsi_calib.cu")
CAL_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "cal_chol_kernel__calibrate_gptj.md")


def cal_chol_traffic():
    """DRAM bytes per launch of the Cholesky kernel from the committed ncu
    summary, if it was taken on the calibration source as it is now."""
    try:
        with open(CAL_SRC, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        vals = {}
        with open(CAL_TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line:
                    key, v = line.split(":", 1)
                    vals[key.strip().lstrip("- ")] = v.strip()
        if vals.get("calib_source_sha256_16") != sha:
            return None
        return float(vals["dram_bytes_per_active_launch"])
    except Exception:
        return None


def cal_roofline(lib, X, Q0, iters, V, ws, stream, k, reps=3):
    """Per-launch durations from gsi_calibrate_timed (CUDA events on the
    launching stream, around each launch) over a few calibrations; the
    dominant kind by total time gets the roofline.  For the Cholesky the
    algorithmic work is k^3/3 flops per launch that factors (the second-pass
    launches that find their pass not needed return at once and count as no
    work), against the fp32 FMA rate of the GPU (152 SMs x 128 FMA/clk x
    2 flops at the 2.07 GHz maximum SM clock) and of the one SM it runs on."""
    totals, counts, chol = {}, {}, []
    for _ in range(reps):
        for kind, ms in lib.gsi_calibrate_timed(X, Q0, iters, V, ws, stream):
            totals[kind] = totals.get(kind, 0.0) + ms
            counts[kind] = counts.get(kind, 0) + 1
            if kind == "Cholesky":
                chol.append(ms)
    dom = max(totals, key=totals.get)
    share = {kd: round(t / sum(totals.values()), 4) for kd, t in totals.items()}
    info = {"kernel": {"Cholesky": "cal_chol_kernel"}.get(dom, dom), "shares": share,
            "avg_ms_by_kind": {kd: round(totals[kd] / counts[kd], 5) for kd in totals},
            "source": "gsi_calibrate_timed: CUDA events around each launch on its stream"}
    if dom == "Cholesky":
        top = max(chol)
        active = [t for t in chol if t > 0.2 * top]
        flops = k ** 3 / 3.0
        peak_gpu = 152 * 128 * 2 * 2.07e9 / 1e12
        ach = flops * len(active) / (sum(chol) * 1e-3) / 1e12
        traffic = cal_chol_traffic()
        info.update(bound="alu", unit="TFLOP/s", achieved=round(ach, 4), peak=round(peak_gpu, 1),
                    frac=round(ach / peak_gpu, 6), frac_of_one_sm=round(ach / (peak_gpu / 152), 4),
                    traffic=traffic, traffic_per="active launch (ncu)",
                    active_launch_avg_ms=round(sum(active) / len(active), 5),
                    flops_per_active_launch=flops,
                    peak_kind="derived fp32 FMA rate: 152 SMs x 128 FMA/clk x 2 x 2.07 GHz; "
                              "the kernel is one CTA on one SM")
    else:
        info.update(bound=None, achieved=None, peak=None, frac=None, traffic=None)
    return info


def _linear_setup(spec, basis, seed, tag, eps=None):
    """W (device draw), V_k, M (gsi_precompute_M) and a handle of one linear."""
    import torch

    import gsi_inputs as gi
    from gated_rank_subspace_gsi_gb300 import lib
    W = gi.gaussian_weights(spec.d_out, spec.d, seed, tag, device="cuda")
    V = torch.from_numpy(basis.V_bits.view(np.int16)).view(torch.bfloat16).cuda()
    M = torch.empty((spec.d_out, spec.k), dtype=torch.bfloat16, device="cuda")
    lib.gsi_precompute_M(W, V, M)
    torch.cuda.synchronize()
    h = lib.gsi_create(W, V, M, spec.eps if eps is None else eps)
    return dict(W=W, V=V, M=M, h=h, spec=spec)


def _fast_bytes(spec) -> int:
    return (spec.d * spec.k * 2 + correction_bytes(spec.k) + spec.d_out * spec.k * 2
            + spec.d * 2 + spec.d_out * 4 + 5)


def _timed(graph, stream, steps, warmup, world, local):
    import torch
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    replay(graph, stream, max(warmup, 3))
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    replay(graph, stream, steps)
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    return ms, clocks.stop()


def _line(metric, value, unit, world, steps, warmup, ms, config, **extra):
    out = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": steps,
           "warmup": warmup, "ms_per_step": round(ms, 4), "higher_is_better": False,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded Gaussian weights, QR bases, activations with set residual "
                   "ratios)", "impl": "gsi", "config": config}
    out.update(extra)
    return out


def measure_gpt2(args, world, rank, local):
    """GPT-2-small-shaped QKV linear (768 -> 2304, k = 256, eps = 0.10), T = 64
    tokens per call with 6 slow: L2-resident and latency-bound (a parity
    configuration), timed as calls in a CUDA graph."""
    import torch

    import gsi_inputs as gi
    from gated_rank_subspace_gsi_gb300 import lib
    torch.cuda.set_device(local)
    wl = gi.gpt2_qkv()
    spec = wl.linears[0]
    inp = gi.make_linear_inputs(spec, wl.T, wl.extra["n_slow"], wl.seed)
    L = _linear_setup(spec, inp.basis, wl.seed, 0)
    x = torch.from_numpy(inp.X_bits.view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.zeros((wl.T, spec.d_out), dtype=torch.float32, device="cuda")
    gate = torch.zeros((wl.T,), dtype=torch.uint8, device="cuda")
    rho = torch.zeros((wl.T,), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    calls = 100
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(calls):
                lib.gsi_forward(L["h"], x, y, gate, rho, stream)
    steps = max(3, args.steps // 10)
    ms, clk = _timed(graph, stream, steps, args.warmup, world, local)
    if not np.array_equal(gate.cpu().numpy().astype(bool), inp.slow_mask):
        raise RuntimeError("gates differ from the generated mix")
    us = ms * 1e3 / calls
    per_call = (spec.d * spec.k * 2 + 2 * spec.d * wl.T + spec.k * spec.k * 4
                + spec.d_out * spec.k * 2 + spec.d_out * spec.d * 2 + wl.T * spec.d_out * 4)
    peak, kind = hbm_peak()
    out = _line(GPT2_METRIC, round(us, 3), GPT2_UNIT, world,
                steps, args.warmup, ms,
                {"workload": GPT2_WORKLOAD, "calls_per_step": calls,
                 "l2": "L2-resident (5 MB working set, as the configuration describes)"},
                roofline={"bound": "latency", "achieved": round(per_call / (us * 1e-6) / 1e9, 1),
                          "peak": peak, "unit": "GB/s",
                          "frac": round(per_call / (us * 1e-6) / 1e9 / peak, 4),
                          "traffic": None, "bytes_per_call": per_call,
                          "peak_kind": f"{kind} HBM copy (L2-resident: not the bound)"},
                gpu_launches=steps * calls * lib.gsi_forward_launch_count(L["h"], wl.T),
                clocks=clk)
    lib.gsi_destroy(L["h"])
    del graph, L
    _release()
    return out


def run_gpt2(args, world, rank, local):
    out = measure_gpt2(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)


def measure_stack(args, world, rank, local):
    """GPT-J-shaped 28-layer stack at decode: per layer the stacked qkv+fc_in
    call, then out_proj and fc_out as one grouped launch; depth-coherent bases
    per input chain; 256 distinct decode steps of synthetic tokens (43 slow
    draws over step x layer x linear), weights (11 GB) beyond L2 by size."""
    import torch

    import gsi_inputs as gi
    from gated_rank_subspace_gsi_gb300 import lib
    torch.cuda.set_device(local)
    wl = gi.gptj_stack()
    nL, S, specs = wl.extra["n_layers"], wl.extra["n_steps"], wl.linears
    slow = gi.slow_positions(S * nL * 3, wl.extra["n_slow"], wl.seed).reshape(S, nL, 3)
    layers = []
    chain = [None, None, None]
    for l in range(nL):
        lay = []
        for i, sp in enumerate(specs):
            chain[i] = (gi.random_basis(sp.d, sp.k, wl.seed, tag=i) if l == 0 else
                        gi.coherent_next_basis(chain[i], wl.seed, tag=1000 * i + l))
            L = _linear_setup(sp, chain[i], wl.seed, 100 * l + i)
            rs = gi.rho_targets(S, sp.rho_fast, sp.rho_slow, slow[:, l, i], wl.seed, 100 * l + i)
            X = gi.tokens(chain[i], rs, wl.seed, 100 * l + i)
            L["x"] = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
            L["y"] = torch.zeros((S, sp.d_out), dtype=torch.float32, device="cuda")
            L["gate"] = torch.zeros((S,), dtype=torch.uint8, device="cuda")
            L["rho"] = torch.zeros((S,), dtype=torch.float32, device="cuda")
            lay.append(L)
        g = lib.gsi_group_create([lay[1]["h"], lay[2]["h"]])
        layers.append((lay, g))
    if args.prefetch > 0:
        for l, (lay, g) in enumerate(layers):
            lib.gsi_set_prefetch_group(lay[0]["h"], g)
            lib.gsi_group_set_prefetch(g, layers[(l + 1) % nL][0][0]["h"])
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for t in range(S):
                sl = slice(t, t + 1)
                for lay, g in layers:
                    A = lay[0]
                    lib.gsi_forward(A["h"], A["x"][sl], A["y"][sl], A["gate"][sl], A["rho"][sl],
                                    stream)
                    m = lay[1:]
                    lib.gsi_group_forward(g, [L["x"][sl] for L in m], [L["y"][sl] for L in m],
                                          [L["gate"][sl] for L in m], [L["rho"][sl] for L in m],
                                          stream)
    steps = max(1, args.steps // 100)
    ms, clk = _timed(graph, stream, steps, args.warmup, world, local)
    for l, (lay, _) in enumerate(layers):
        for i, L in enumerate(lay):
            if not np.array_equal(L["gate"].cpu().numpy().astype(bool), slow[:, l, i]):
                raise RuntimeError(f"gates differ from the generated mix (layer {l}, linear {i})")
    per_fast = sum(_fast_bytes(sp) for sp in specs) * nL
    n_slow = int(slow.sum())
    slow_extra = sum(int(slow[:, :, i].sum()) * (specs[i].d_out * specs[i].d * 2
                                                  - specs[i].d_out * specs[i].k * 2)
                     for i in range(3))
    total = per_fast * S + slow_extra
    us_token = ms * 1e3 / S
    gbs = total / (ms * 1e-3) / 1e9
    peak, kind = hbm_peak()
    out = _line(STACK_METRIC, round(us_token, 2), STACK_UNIT, world, steps, args.warmup, ms,
                {"workload": stack_workload(S, n_slow),
                 "l2": f"weights {sum(sp.d_out * sp.d * 2 for sp in specs) * nL / 1e9:.1f} GB, "
                       f"V_k + M {sum((sp.d + sp.d_out) * sp.k * 2 for sp in specs) * nL / 1e9:.2f}"
                       " GB: beyond L2 by size"},
                us_per_gated_linear=round(us_token / (3 * nL), 4),
                roofline={"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                          "frac": round(gbs / peak, 4), "traffic": None,
                          "bytes_per_fast_step": per_fast, "peak_kind": f"{kind} HBM copy"},
                gpu_launches=steps * S * nL * 2, clocks=clk)
    del graph
    for lay, g in layers:
        lib.gsi_group_destroy(g)
        for L in lay:
            lib.gsi_destroy(L["h"])
    del layers
    _release()
    return out


def run_stack(args, world, rank, local):
    out = measure_stack(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)


def measure_opt(args, world, rank, local):
    """OPT-6.7B-shaped MLP (fc1 4096 -> 16384, fc2 16384 -> 4096) x 32 layers at
    decode, eps = 0.05, over slow fractions 0, 2, 10, 50 and 100% (exact counts
    over step x layer x linear), with the dense bf16 W x (torch.matmul) on the
    same weights and inputs beside each point."""
    import torch

    import gsi_inputs as gi
    from gated_rank_subspace_gsi_gb300 import lib
    torch.cuda.set_device(local)
    S = 32
    fracs = [0.0, 0.02, 0.10, 0.50, 1.00]
    wl0 = gi.opt_mlp(n_steps=S, slow_fraction=0.0)
    nL, specs = wl0.extra["n_layers"], wl0.linears
    layers = []
    for l in range(nL):
        lay = []
        for i, sp in enumerate(specs):
            basis = gi.random_basis(sp.d, sp.k, wl0.seed, tag=100 * l + i)
            L = _linear_setup(sp, basis, wl0.seed, 100 * l + i)
            L["basis"] = basis
            L["y"] = torch.zeros((S, sp.d_out), dtype=torch.float32, device="cuda")
            L["gate"] = torch.zeros((S,), dtype=torch.uint8, device="cuda")
            L["rho"] = torch.zeros((S,), dtype=torch.float32, device="cuda")
            L["yd"] = torch.zeros((S, sp.d_out), dtype=torch.bfloat16, device="cuda")
            lay.append(L)
        layers.append(lay)
    order = [L["h"] for lay in layers for L in lay]
    for i, h in enumerate(order):
        lib.gsi_set_prefetch(h, order[(i + args.prefetch) % len(order)] if args.prefetch > 0
                             else None)
    stream = torch.cuda.Stream()
    peak, kind = hbm_peak()
    steps = max(1, args.steps // 30)
    curve = []
    clk = None
    for f in fracs:
        wl = gi.opt_mlp(n_steps=S, slow_fraction=f)
        slow = gi.slow_positions(S * nL * 2, wl.extra["n_slow"], wl.seed).reshape(S, nL, 2)
        for l, lay in enumerate(layers):
            for i, L in enumerate(lay):
                sp = L["spec"]
                rs = gi.rho_targets(S, sp.rho_fast, sp.rho_slow, slow[:, l, i], wl.seed,
                                    100 * l + i)
                X = gi.tokens(L["basis"], rs, wl.seed, 100 * l + i)
                L["x"] = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).cuda()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for t in range(S):
                    sl = slice(t, t + 1)
                    for lay in layers:
                        for L in lay:
                            lib.gsi_forward(L["h"], L["x"][sl], L["y"][sl], L["gate"][sl],
                                            L["rho"][sl], stream)
        ms, clk = _timed(graph, stream, steps, args.warmup, world, local)
        for l, lay in enumerate(layers):
            for i, L in enumerate(lay):
                if not np.array_equal(L["gate"].cpu().numpy().astype(bool), slow[:, l, i]):
                    raise RuntimeError(f"gates differ (f={f}, layer {l}, linear {i})")
        dense = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            L0 = layers[0][0]  # cuBLAS sets itself up outside the capture
            torch.matmul(L0["x"][0:1], L0["W"].t(), out=L0["yd"][0:1])
            stream.synchronize()
            with torch.cuda.graph(dense, stream=stream):
                for t in range(S):
                    for lay in layers:
                        for L in lay:
                            torch.matmul(L["x"][t:t + 1], L["W"].t(), out=L["yd"][t:t + 1])
        ms_d, _ = _timed(dense, stream, steps, args.warmup, world, local)
        n_slow = int(slow.sum())
        total = sum(_fast_bytes(L["spec"]) for lay in layers for L in lay) * S + sum(
            int(slow[:, :, i].sum()) * (specs[i].d_out * specs[i].d * 2
                                        - specs[i].d_out * specs[i].k * 2) for i in range(2))
        curve.append({"slow_fraction": f, "n_slow": n_slow,
                      "us_per_layer": round(ms * 1e3 / (S * nL), 3),
                      "gbs": round(total / (ms * 1e-3) / 1e9, 1),
                      "frac_of_measured_hbm": round(total / (ms * 1e-3) / 1e9 / peak, 4),
                      "dense_us_per_layer": round(ms_d * 1e3 / (S * nL), 3),
                      "speedup_vs_dense": round(ms_d / ms, 3)})
        del graph, dense
    c0 = curve[0]
    out = _line(OPT_METRIC, c0["us_per_layer"], OPT_UNIT, world, steps, args.warmup,
                c0["us_per_layer"] * nL * S / 1e3,
                {"workload": opt_workload(S),
                 "l2": "weights 8.6 GB: beyond L2 by size"},
                curve=curve, roofline={"bound": "hbm", "achieved": c0["gbs"], "peak": peak,
                                       "unit": "GB/s", "frac": c0["frac_of_measured_hbm"],
                                       "traffic": None, "peak_kind": f"{kind} HBM copy"},
                gpu_launches=steps * S * nL * 2 * len(fracs), clocks=clk)
    for lay in layers:
        for L in lay:
            lib.gsi_destroy(L["h"])
    del layers
    _release()
    return out


def run_opt(args, world, rank, local):
    out = measure_opt(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference(args, world, rank):
    """The oracle (fp64 C) on the host cores, each step a bounded sample of the
    decode layer workload: 8 tokens x 3 gated linears, slow token included in
    the first step."""
    if rank != 0:
        return
    import oracle

    import gsi_inputs as gi
    orc = oracle.default()
    wl = gi.gptj_layer()
    n = wl.extra["n_tokens"]
    slow = gi.slow_positions(n, wl.extra["n_slow"], wl.seed)
    prep = []
    for li, spec in enumerate(wl.linears):
        inp = gi.make_linear_inputs(spec, n, 0, wl.seed, tag=li, slow_mask=slow)
        Wd = orc.bf16_decode(inp.W)
        Vd = orc.bf16_decode(inp.V_bits)
        Md = orc.bf16_decode(orc.bf16_encode(orc.precompute_M(Wd, Vd)))
        prep.append((Wd, Vd, Md, float(np.float32(spec.eps)), inp.X_bits))
    order = list(np.nonzero(slow)[0]) + [t for t in range(n) if not slow[t]]
    per_step = 8

    def one_step(s):
        toks = [order[(s * per_step + i) % n] for i in range(per_step)]
        for t in toks:
            for (W, V, M, eps, X) in prep:
                orc.forward(W, V, M, eps, orc.bf16_decode(X[t:t + 1]))

    for s in range(args.warmup):
        one_step(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        one_step(args.warmup + s)
    dt = time.perf_counter() - t0
    n_lin = args.steps * per_step * len(prep)
    v = dt / n_lin * 1e6
    out = {
        "metric": METRIC, "value": round(v, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": DECODE_WORKLOAD},
        "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": orc.num_threads(),
                         "kind": "oracle",
                         "sample": f"{per_step} decode tokens x 3 gated linears per step, "
                                   f"{args.steps} steps"},
        "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)



def _ref_token_seconds(orc, spec, seed, tag, steps, n_fast=2, n_slow=1, batch=False):
    """Seconds per token of the oracle's gated linear on one shape, fast and
    slow tokens apart: `steps` x (n_fast fast + n_slow slow) tokens of the
    workload's token mix, one forward call per token (decode) or one call
    for all fast and one for all slow tokens (batch: the call carries T
    tokens in the workload too)."""
    import gsi_inputs as gi
    T = (n_fast + n_slow) * steps
    inp = gi.make_linear_inputs(spec, T, n_slow * steps, seed, tag=tag)
    W = orc.bf16_decode(inp.W)
    V = orc.bf16_decode(inp.V_bits)
    M = orc.bf16_decode(orc.bf16_encode(orc.precompute_M(W, V)))
    eps = float(np.float32(spec.eps))
    fast = [t for t in range(T) if not inp.slow_mask[t]]
    slow = [t for t in range(T) if inp.slow_mask[t]]

    def per_token(toks):
        t0 = time.perf_counter()
        if batch:
            orc.forward(W, V, M, eps, orc.bf16_decode(inp.X_bits[toks]))
        else:
            for t in toks:
                orc.forward(W, V, M, eps, orc.bf16_decode(inp.X_bits[t:t + 1]))
        return (time.perf_counter() - t0) / len(toks)

    per_token(fast[:1])  # warm-up
    return per_token(fast), per_token(slow)


def ref_linear(wname: str, steps: int):
    """The oracle (fp64 C) on the host cores for a workload made of gated
    linears of fixed shapes (batched_T512, gpt2_qkv_T64, gptj_stack, opt_mlp):
    per shape, fast and slow tokens are timed one by one on a bounded sample,
    and the metric's unit is composed from the workload's exact fast and slow
    counts.  Returns (value, metric, unit, workload, cpu_baseline dict)."""
    import oracle

    import gsi_inputs as gi
    orc = oracle.default()
    batched = wname in ("batched_T512", "gpt2_qkv_T64")
    if wname == "batched_T512":
        wl = gi.batched_prefill()
        sp, n_slow = wl.linears[0], wl.extra["n_slow"]
        tf, ts = _ref_token_seconds(orc, sp, wl.seed, 0, steps, n_fast=4, n_slow=2, batch=True)
        v = ((wl.T - n_slow) * tf + n_slow * ts) * 1e6
        metric, unit, workload = BATCHED_METRIC, BATCHED_UNIT, BATCHED_WORKLOAD
        how = f"{wl.T - n_slow} fast x t_fast + {n_slow} slow x t_slow per call"
    elif wname == "gpt2_qkv_T64":
        wl = gi.gpt2_qkv()
        sp, n_slow = wl.linears[0], wl.extra["n_slow"]
        tf, ts = _ref_token_seconds(orc, sp, wl.seed, 0, steps, n_fast=16, n_slow=4, batch=True)
        v = ((wl.T - n_slow) * tf + n_slow * ts) * 1e6
        metric, unit, workload = GPT2_METRIC, GPT2_UNIT, GPT2_WORKLOAD
        how = f"{wl.T - n_slow} fast x t_fast + {n_slow} slow x t_slow per call"
    elif wname == "gptj_stack":
        wl = gi.gptj_stack()
        nL, S, n_slow = wl.extra["n_layers"], wl.extra["n_steps"], wl.extra["n_slow"]
        per_lin = n_slow / (S * 3)  # expected slow draws per linear per decode step
        v = 0.0
        for i, sp in enumerate(wl.linears):
            tf, ts = _ref_token_seconds(orc, sp, wl.seed, i, steps)
            v += ((nL - per_lin) * tf + per_lin * ts) * 1e6
        metric, unit, workload = STACK_METRIC, STACK_UNIT, stack_workload(S, n_slow)
        how = (f"per linear shape: {nL} layers x t_fast, with {n_slow} slow draws over {S} steps "
               f"x {nL} layers x 3 linears taken at their mean rate")
    elif wname == "opt_mlp":
        wl = gi.opt_mlp(n_steps=32, slow_fraction=0.0)
        v = 0.0
        for i, sp in enumerate(wl.linears):
            tf, _ = _ref_token_seconds(orc, sp, wl.seed, i, steps, n_fast=3, n_slow=1)
            v += tf * 1e6
        metric, unit, workload = OPT_METRIC, OPT_UNIT, opt_workload(32)
        how = "t_fast(fc1) + t_fast(fc2): the f = 0 point"
    else:
        raise ValueError(wname)
    batched = wname in ("batched_T512", "gpt2_qkv_T64")
    cpu = {"value": round(v, 3), "unit": unit, "cores": orc.num_threads(), "kind": "oracle",
           "sample": f"per linear shape, fast and slow tokens of {steps} steps timed apart "
                     f"({'in one call each' if batched else 'one call per token'}); {how}"}
    return v, metric, unit, workload, cpu


def run_reference_linear(args, world, rank):
    """The oracle on the host cores for the workloads made of gated linears
    of fixed shapes (ref_linear)."""
    if rank != 0:
        return
    steps = max(1, min(args.steps, 4))
    v, metric, unit, workload, cpu = ref_linear(args.workload, steps)
    out = {"metric": metric, "value": round(v, 3), "unit": unit, "n_gpus": world,
           "steps": steps, "warmup": 1, "ms_per_step": round(v / 1e3, 3),
           "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": {"workload": workload},
           "cpu_baseline": cpu,
           "e2e": {"value": round(v, 3), "unit": unit, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_reference_calibrate(args, world, rank):
    """The oracle's subspace iteration (numpy fp64) on the host cores: each
    step one whole GPT-J-shaped calibration on the same inputs."""
    if rank != 0:
        return
    c, cs, Q0b = _cal_inputs()
    import gsi_inputs as gi
    from oracle import calibration as cal
    X = gi.bf16_bits_to_f64(cs.X_bits)
    Q = gi.bf16_bits_to_f64(Q0b)
    steps = max(1, min(args.steps, 8))
    warm = min(args.warmup, 1)
    for _ in range(warm):
        cal.subspace_iteration(X, Q, c["iters"])
    t0 = time.perf_counter()
    for _ in range(steps):
        cal.subspace_iteration(X, Q, c["iters"])
    dt = time.perf_counter() - t0
    v = dt / steps * 1e3
    out = {
        "metric": CAL_METRIC, "value": round(v, 3), "unit": CAL_UNIT, "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": round(v, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": cal_workload(c["n"], c["d"], c["k"], c["iters"])},
        "cpu_baseline": {"value": round(v, 3), "unit": CAL_UNIT, "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{steps} whole calibrations (numpy fp64 subspace iteration)"},
        "e2e": {"value": round(v, 3), "unit": CAL_UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


CASC_METRIC = ("ms per layer, depth cascade of 28 GPT-J-shaped layers (n=2048 calibration tokens, "
               "d=4096, k=256; 8 iterations for layer 0, 2 from the previous layer's basis after)")


def _casc_inputs(layers):
    import gsi_inputs as gi
    c = gi.calibration_gptj()
    sets = gi.calibration_cascade(layers, c["n"], c["d"], c["k"], seed=c["seed"] + 100)
    Q0 = gi.calibration_start(c["d"], c["k"], seed=c["seed"] + 100)
    return c, sets, Q0


def run_cascade(args, world, rank, local):
    """Depth cascade (section 2.3) over 28 GPT-J-shaped layers through
    gsi_calibrate_cascade, against per-layer calibration from a random start
    (8 iterations each) on the same tokens: time per layer, the cost cut, and
    the energy each basis captures (measured on the device)."""
    import torch

    from gated_rank_subspace_gsi_gb300 import lib
    torch.cuda.set_device(local)
    lib.library()
    L, it_first, it_next = 28, 8, 2
    c, sets, Q0b = _casc_inputs(L)
    n, d, k = c["n"], c["d"], c["k"]
    Xs = [torch.from_numpy(s.X_bits.view(np.int16)).view(torch.bfloat16).cuda() for s in sets]
    Q0 = torch.from_numpy(Q0b.view(np.int16)).view(torch.bfloat16).cuda()
    Vc = [torch.empty((d, k), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    Vp = [torch.empty((d, k), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    ws = torch.empty(lib.gsi_calibrate_workspace_size(n, d, k), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        lib.gsi_calibrate(Xs[0], Q0, 1, Vp[0], ws, stream)
    stream.synchronize()
    g_casc = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_casc, stream=stream):
            lib.gsi_calibrate_cascade(Xs, Q0, it_first, it_next, Vc, ws, stream)
    g_cold = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_cold, stream=stream):
            for layer in range(L):
                lib.gsi_calibrate(Xs[layer], Q0, it_first, Vp[layer], ws, stream)
    replay(g_casc, stream, 1)
    replay(g_cold, stream, 1)
    st = lib.gsi_calibrate_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"calibration status: {lib.gsi_status_string(st)}")
    steps = max(1, args.steps // 100)
    ms, clk = _timed(g_casc, stream, steps, args.warmup, world, local)
    ms_cold = max_over_ranks(time_graph(g_cold, stream, reps=steps, warmup=1), world)
    # captured energy ||X V||_F^2 / ||X||_F^2 of each basis (device matmuls:
    # measurement, not part of the calibration)
    e_c, e_p = [], []
    for layer in range(L):
        X = Xs[layer].float()
        tot = float((X * X).sum())
        e_c.append(float((X @ Vc[layer].float()).pow(2).sum()) / tot)
        e_p.append(float((X @ Vp[layer].float()).pow(2).sum()) / tot)
    rl = cal_roofline(lib, Xs[1], Vc[0], it_next, Vp[1], ws, stream, k)
    launches = (lib.gsi_calibrate_launch_count(n, d, k, it_first)
                + (L - 1) * lib.gsi_calibrate_launch_count(n, d, k, it_next))
    rank1 = cascade_rank1_curve(lib, Xs, Q0, it_first, stream=stream, world=world,
                                e_cold=e_p, ms_cold=ms_cold, steps=steps,
                                counts=[int(c) for c in args.rank1.split(",") if c.strip()])
    out = _line(CASC_METRIC, round(ms / L, 4), "ms per layer", world, steps, args.warmup, ms,
                {"workload": casc_workload(L, n, d, k, it_first, it_next),
                 "l2": f"inputs larger than L2: {L} layers x {n * d * 2 / 2**20:.0f} MiB of tokens",
                 "parallelism": "1 GPU" if world == 1 else f"replicas x{world}"},
                roofline=rl,
                per_layer_cold_ms=round(ms_cold / L, 4),
                cost_cut_vs_per_layer=round(1.0 - ms / ms_cold, 4),
                captured_energy={"cascade_mean": round(float(np.mean(e_c)), 6),
                                 "per_layer_cold_mean": round(float(np.mean(e_p)), 6),
                                 "max_shortfall": round(float(np.max(np.array(e_p) - np.array(e_c))), 6)},
                gpu_launches=steps * launches, clocks=clk, rank1=rank1)
    out["data"] = ("synthetic (seeded depth-coherent planted-spectrum calibration activations, "
                   "seeded Gaussian start block)")
    out["dtype"] = "bf16 GEMMs, fp32 orthonormalisation"
    # end to end: the layers' tokens from pinned host memory, the bases back
    Hx = [x.cpu().pin_memory() for x in Xs]
    Hv = [torch.empty((d, k), dtype=torch.bfloat16).pin_memory() for _ in range(L)]
    Hq = Q0.cpu().pin_memory()
    Xd = [torch.empty_like(x) for x in Xs]
    Qd = torch.empty_like(Q0)
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(ge, stream=stream):
            for layer in range(L):
                Xd[layer].copy_(Hx[layer], non_blocking=True)
            Qd.copy_(Hq, non_blocking=True)
            lib.gsi_calibrate_cascade(Xd, Qd, it_first, it_next, Vc, ws, stream)
            for layer in range(L):
                Hv[layer].copy_(Vc[layer], non_blocking=True)
    ms_e2e = max_over_ranks(time_graph(ge, stream, reps=steps, warmup=1), world)
    out["e2e"] = {"value": round(ms_e2e / L, 4), "unit": "ms per layer",
                  "h2d_bytes_per_step": L * n * d * 2 + d * k * 2,
                  "d2h_bytes_per_step": L * d * k * 2,
                  "how": "pinned tokens of every layer and Q0 copied in, every basis copied out, "
                         "around one gsi_calibrate_cascade, graph-captured"}
    if rank == 0 and not args.no_cpu_baseline:
        import gsi_inputs as gi
        from oracle import calibration as cal
        t0 = time.perf_counter()
        done = 0
        V = cal.subspace_iteration(gi.bf16_bits_to_f64(sets[0].X_bits), gi.bf16_bits_to_f64(Q0b),
                                   it_first)
        done = 1
        while done < L and time.perf_counter() - t0 < args.cpu_budget:
            V = cal.subspace_iteration(gi.bf16_bits_to_f64(sets[done].X_bits), V, it_next)
            done += 1
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": round(dt / done * 1e3, 3), "unit": "ms per layer",
                               "cores": os.cpu_count(), "kind": "oracle",
                               "sample": f"the oracle's cascade over the first {done} layers "
                                         f"(fp64 numpy), {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(out), flush=True)


RANK1_CORRECTIONS = (16, 64, 256)


def cascade_rank1_curve(lib, Xs, Q0, it_first, stream, world, e_cold, ms_cold,
                        steps, counts=RANK1_CORRECTIONS):
    """The cascade in the page's rank-1 form (gsi_calibrate_cascade_rank1) on
    the same layers, for a few correction counts: ms per layer (graph
    replays), the cost cut against per-layer calibration from a random start,
    and the energy each layer's basis captures against those per-layer
    calibrations."""
    import torch
    L = len(Xs)
    n, d = Xs[0].shape
    k = Q0.shape[1]
    ws = torch.empty(lib.gsi_refine_rank1_workspace_size(n, d, k), dtype=torch.uint8,
                     device="cuda")
    out = {"how": "layer 0 by 8 block iterations, then per layer c rank-1 corrections "
                  "re-orthogonalised by DGKS from the previous layer's basis", "curve": []}
    prev = None
    for c in counts:
        Vr = [torch.empty((d, k), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                lib.gsi_calibrate_cascade_rank1(Xs, Q0, it_first, c, Vr, ws, stream=stream)
        replay(g, stream, 1)
        st = lib.gsi_calibrate_status(ws, stream)
        if st != 0:
            raise RuntimeError(f"rank-1 cascade status: {lib.gsi_status_string(st)}")
        ms = max_over_ranks(time_graph(g, stream, reps=steps, warmup=1), world)
        e = []
        for layer in range(L):
            X = Xs[layer].float()
            e.append(float((X @ Vr[layer].float()).pow(2).sum()) / float((X * X).sum()))
        short = np.array(e_cold) - np.array(e)
        pt = {"corrections": c, "ms_per_layer": round(ms / L, 4),
              "cost_cut_vs_per_layer": round(1.0 - ms / ms_cold, 4),
              "energy_mean": round(float(np.mean(e)), 6),
              "max_shortfall_vs_per_layer": round(float(np.max(short[1:])), 6),
              "launches_per_layer": lib.gsi_refine_rank1_launch_count(n, d, k, c)}
        if prev is not None:
            pt["us_per_correction"] = round((ms - prev[1]) / ((L - 1) * (c - prev[0])) * 1e3, 2)
        prev = (c, ms)
        out["curve"].append(pt)
        del g
    return out


def run_reference_cascade(args, world, rank):
    """The oracle's cascade (numpy fp64) over the 28 layers, one whole cascade
    per step."""
    if rank != 0:
        return
    import gsi_inputs as gi
    from oracle import calibration as cal
    L = 28
    c, sets, Q0b = _casc_inputs(L)
    Xs = [gi.bf16_bits_to_f64(s.X_bits) for s in sets]
    Q = gi.bf16_bits_to_f64(Q0b)
    steps = max(1, min(args.steps, 3))
    t0 = time.perf_counter()
    for _ in range(steps):
        cal.cascade(Xs, Q, 8, 2)
    dt = time.perf_counter() - t0
    v = dt / steps / L * 1e3
    out = {"metric": CASC_METRIC, "value": round(v, 3), "unit": "ms per layer", "n_gpus": world,
           "steps": steps, "warmup": 0, "ms_per_step": round(dt / steps * 1e3, 3),
           "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": {"workload": casc_workload(L, c["n"], c["d"], c["k"], 8, 2)},
           "cpu_baseline": {"value": round(v, 3), "unit": "ms per layer", "cores": os.cpu_count(),
                            "kind": "oracle",
                            "sample": f"{steps} whole cascades of {L} layers (numpy fp64)"},
           "e2e": {"value": round(v, 3), "unit": "ms per layer", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


SWEEP_KS = (128, 256, 512)
SWEEP_EPS = (0.02, 0.05, 0.10, 0.20, math.inf)


def run_sweep(args, world, rank, local):
    """Operating points of the GPT-J-shaped stacked qkv+fc_in linear (4096 ->
    28672) at decode: k in {128, 256, 512} x eps in {0.02, 0.05, 0.10, 0.20,
    inf}; eps = inf is the static projection (no residual path), the page's
    negative control.  512 sequential one-token calls per point on tokens with
    a gapless power-law spectrum; V_k = the population top-k basis.  Per point:
    the fast fraction, the algorithmic bytes per call, the relative output
    error against W x (the same kernel at eps = 0), the largest ratio of a
    fast token's error to Theorem 4's bound ||W||_2 eps ||x||, and the time
    per call.  Replicas of (V_k, M) per k cycle so that the fast path streams
    from HBM."""
    import torch

    import gsi_inputs as gi
    from gated_rank_subspace_gsi_gb300 import lib
    torch.cuda.set_device(local)
    lib.library()
    seed = gi.CONFIG_SEED_BASE + 7
    d_out, d, T = 28672, 4096, 512
    cs = gi.sweep_activations(T, d, seed)
    W = gi.gaussian_weights(d_out, d, seed, device="cuda")
    x = torch.from_numpy(cs.X_bits.view(np.int16)).view(torch.bfloat16).cuda()
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    stream = torch.cuda.Stream()
    steps = max(1, args.steps // 60)
    peak, pkind = hbm_peak()
    # ||W||_2 by power iteration (fp32 on the device; measurement only)
    v = torch.randn(d, device="cuda", generator=torch.Generator(device="cuda").manual_seed(seed))
    Wf = W.float()
    for _ in range(60):
        v = Wf.t() @ (Wf @ v)
        v = v / v.norm()
    w_norm = float((Wf @ v).norm())
    del Wf
    xnorm = x.float().norm(dim=1)

    def run_point(handles, eps_is_inf):
        y = torch.zeros((T, d_out), dtype=torch.float32, device="cuda")
        gate = torch.zeros((T,), dtype=torch.uint8, device="cuda")
        rho = torch.zeros((T,), dtype=torch.float32, device="cuda")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for t in range(T):
                    sl = slice(t, t + 1)
                    lib.gsi_forward(handles[t % len(handles)], x[sl], y[sl], gate[sl], rho[sl],
                                    stream)
        ms, clk = _timed(graph, stream, steps, args.warmup, world, local)
        st = lib.gsi_device_status(handles[0], stream)
        if st != 0:
            raise RuntimeError(f"device status: {lib.gsi_status_string(st)}")
        del graph
        return y, gate, rho, ms, clk

    # exact W x: the slow path everywhere (eps = 0), any basis
    V0 = torch.from_numpy(gi.to_bf16_bits(cs.U[:, :128]).view(np.int16)).view(torch.bfloat16).cuda()
    M0 = torch.empty((d_out, 128), dtype=torch.bfloat16, device="cuda")
    lib.gsi_precompute_M(W, V0, M0)
    torch.cuda.synchronize()
    h0 = lib.gsi_create(W, V0, M0, 0.0)
    y_exact, g0, _, ms_dense, clk = run_point([h0], False)
    lib.gsi_destroy(h0)
    ynorm = y_exact.norm(dim=1)
    points = []
    for k in SWEEP_KS:
        V = torch.from_numpy(gi.to_bf16_bits(cs.U[:, :k]).view(np.int16)).view(torch.bfloat16).cuda()
        M = torch.empty((d_out, k), dtype=torch.bfloat16, device="cuda")
        lib.gsi_precompute_M(W, V, M)
        torch.cuda.synchronize()
        op_bytes = d * k * 2 + d_out * k * 2
        R = max(2, int(math.ceil(1.5 * l2 / op_bytes)))
        Vs = [V] + [V.clone() for _ in range(R - 1)]
        Ms = [M] + [M.clone() for _ in range(R - 1)]
        torch.cuda.synchronize()
        for eps in SWEEP_EPS:
            hs = [lib.gsi_create(W, Vs[r], Ms[r], eps) for r in range(R)]
            for r in range(R):
                lib.gsi_set_prefetch(hs[r], hs[(r + 1) % R])
            y, gate, rho, ms, clk = run_point(hs, math.isinf(eps))
            fast = gate == 0
            err = (y - y_exact).norm(dim=1)
            rel = err / ynorm
            n_fast = int(fast.sum())
            fast_b = _fast_bytes(gi.LinearSpec("qkv_fc_in", d_out, d, k, eps, 0, 0))
            if k > 256:  # the k = 512 kernel forms the residual explicitly: no correction tiles
                fast_b -= correction_bytes(k)
            bytes_call = fast_b + (T - n_fast) / T * (d_out * d * 2)
            us = ms * 1e3 / T
            pt = {"k": k, "eps": "inf" if math.isinf(eps) else eps, "fast_fraction": n_fast / T,
                  "us_per_call": round(us, 3), "bytes_per_call": int(bytes_call),
                  "gbs": round(bytes_call / (us * 1e-6) / 1e9, 1),
                  "rel_err_mean": float(rel.mean()), "rel_err_max": float(rel.max()),
                  "weight_read_speedup": round(d_out * d * 2 / bytes_call, 2),
                  "time_speedup_vs_eps0": round(ms_dense / ms, 3), "replicas": R}
            if n_fast and not math.isinf(eps):
                bound = w_norm * eps * xnorm
                pt["theorem4_max_ratio"] = float((err[fast] / bound[fast]).max())
            points.append(pt)
            for h in hs:
                lib.gsi_destroy(h)
        del Vs, Ms
    main_pt = next(p for p in points if p["k"] == 256 and p["eps"] == 0.10)
    out = _line("µs per gated linear at k=256, eps=0.10 (GPT-J qkv+fc_in 4096 -> 28672, decode), "
                "operating-point sweep", main_pt["us_per_call"], "us per gated linear", world,
                steps, args.warmup, main_pt["us_per_call"] * T / 1e3,
                {"workload": sweep_workload(T),
                 "l2": "replicas of (V_k, M) per k exceed L2 (1.5x); W 235 MB beyond L2 by size"},
                sweep=points, w_spectral_norm=round(w_norm, 4),
                eps0_us_per_call=round(ms_dense * 1e3 / T, 3),
                roofline={"bound": "hbm", "achieved": main_pt["gbs"], "peak": peak, "unit": "GB/s",
                          "frac": round(main_pt["gbs"] / peak, 4), "traffic": None,
                          "kernel": "gsi_decode_cr_group_kernel<256> (whole call)",
                          "peak_kind": f"{pkind} HBM copy"},
                gpu_launches=steps * T * (1 + len(points)), clocks=clk)
    out["data"] = ("synthetic (seeded Gaussian W, power-law activations, planted population "
                   "basis)")
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference_sweep(args, world, rank):
    """The oracle (fp64 C) at the sweep's main operating point (k = 256,
    eps = 0.10) on the host cores: each step 4 of the sweep's tokens through
    the 4096 -> 28672 linear."""
    if rank != 0:
        return
    import oracle

    import gsi_inputs as gi
    orc = oracle.default()
    seed = gi.CONFIG_SEED_BASE + 7
    d_out, d, T, k = 28672, 4096, 512, 256
    cs = gi.sweep_activations(T, d, seed)
    Wd = orc.bf16_decode(gi.gaussian_weights(d_out, d, seed))
    Vb = gi.to_bf16_bits(cs.U[:, :k])
    Vd = orc.bf16_decode(Vb)
    Md = orc.bf16_decode(orc.bf16_encode(orc.precompute_M(Wd, Vd)))
    per_step = 4
    steps = max(1, min(args.steps, 10))
    t0 = time.perf_counter()
    for st in range(steps):
        toks = [(st * per_step + i) % T for i in range(per_step)]
        orc.forward(Wd, Vd, Md, 0.10, orc.bf16_decode(cs.X_bits[toks]))
    dt = time.perf_counter() - t0
    v = dt / (steps * per_step) * 1e6
    out = {"metric": "µs per gated linear at k=256, eps=0.10 (GPT-J qkv+fc_in 4096 -> 28672, "
                     "decode), operating-point sweep", "value": round(v, 3),
           "unit": "us per gated linear", "n_gpus": world, "steps": steps, "warmup": 0,
           "ms_per_step": round(dt / steps * 1e3, 3), "higher_is_better": False,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference",
           "config": {"workload": sweep_workload(T)},
           "cpu_baseline": {"value": round(v, 3), "unit": "us per gated linear",
                            "cores": orc.num_threads(), "kind": "oracle",
                            "sample": f"{steps * per_step} tokens at k=256, eps=0.10"},
           "e2e": {"value": round(v, 3), "unit": "us per gated linear", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gsi", "reference"], default="gsi")
    ap.add_argument("--workload", choices=["gptj_layer_decode", "batched_T512", "gpt2_qkv_T64",
                                           "gptj_stack", "opt_mlp", "calibrate_gptj",
                                           "cascade_gptj", "sweep_gptj"],
                    default="gptj_layer_decode")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--schedule", choices=["grouped", "sequential"], default="grouped",
                    help="grouped: out_proj and fc_out of a token in one launch")
    ap.add_argument("--prefetch", type=int, default=0,
                    help="each call prefetches into L2 the operands of the call this many "
                         "places later (0: none; the one-token kernel's next call already "
                         "stages its operands while the current call runs)")
    ap.add_argument("--shard", choices=["none", "rows"], default="none",
                    help="rows: split the decode layer's linears by output rows over the GPUs "
                         "(NCCL all_gather of y after every call) instead of running replicas")
    ap.add_argument("--no-configs", action="store_true",
                    help="report the decode layer only (without the other configurations)")
    ap.add_argument("--rank1", default=",".join(str(c) for c in RANK1_CORRECTIONS),
                    help="cascade_gptj: rank-1 corrections per layer to measure (comma list)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-linear breakdown and the end-to-end leg (profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference" and args.workload == "calibrate_gptj":
            run_reference_calibrate(args, world, rank)
        elif args.impl == "reference" and args.workload == "cascade_gptj":
            run_reference_cascade(args, world, rank)
        elif args.impl == "reference" and args.workload == "sweep_gptj":
            run_reference_sweep(args, world, rank)
        elif args.impl == "reference" and args.workload in ("batched_T512", "gpt2_qkv_T64",
                                                             "gptj_stack", "opt_mlp"):
            run_reference_linear(args, world, rank)
        elif args.workload == "cascade_gptj":
            run_cascade(args, world, rank, local)
        elif args.workload == "sweep_gptj":
            run_sweep(args, world, rank, local)
        elif args.impl == "reference":
            run_reference(args, world, rank)
        elif args.workload == "calibrate_gptj":
            run_calibrate(args, world, rank, local)
        elif args.workload == "batched_T512":
            run_batched(args, world, rank, local)
        elif args.workload == "gpt2_qkv_T64":
            run_gpt2(args, world, rank, local)
        elif args.workload == "gptj_stack":
            run_stack(args, world, rank, local)
        elif args.workload == "opt_mlp":
            run_opt(args, world, rank, local)
        elif args.shard == "rows":
            run_gsi_rowshard(args, world, rank, local)
        else:
            run_gsi(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
