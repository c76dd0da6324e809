"""Benchmark of the MoE dispatch + combine hot path on GB300.

One step = ep_dispatch_layout + ep_dispatch_nvfp4 (with the fused shared-expert copy) +
ep_combine over one batch of the DeepSeek-V3-shaped layer: T=4096 tokens, hidden 7168,
256 routed experts in 8 logical partitions (capacity 4096 tokens each), top-8, one shared
expert.  Inputs are seeded synthetic (workloads.CONFIGS["dsv3"]), resident in HBM before the
timed region; L2 is flushed between steps (outside the step's events).

Prints one JSON line.  `value` is tokens/s over all ranks (independent replicas, one per GPU:
the path does not shard), `e2e` the same metric through the C ABI with pinned host buffers
(host->device inputs and device->host results inside the timed region), `roofline` the
dominant kernel (combine) against the measured HBM copy bandwidth, `cpu_baseline` the CPU
oracle on a bounded sample.  `configs_sweep` runs the step on every workload recipe, with
the other calls each workload names, its end-to-end figure from pinned host buffers and the
oracle timed per op.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "dispatch+combine tokens/s; achieved HBM GB/s vs peak (DSv3-shape MoE layer)"
UNIT = "tokens/s"
WORKLOAD = "dsv3"
FLUSH_BYTES = 256 << 20
L2_NOTE = ("flushed between steps: a 256 MiB write, then a 256 MiB read of another buffer so the "
           "flush's own dirty lines are written back before the step; both outside the step events")


def workload_config(cfg: W.Config) -> dict:
    return {"workload": f"{cfg.name}: DeepSeek-V3-like MoE layer, T={cfg.T} tokens, hidden={cfg.H}, "
                        f"{cfg.E} routed experts in {cfg.P} logical partitions (capacity {cfg.capacity} "
                        f"tokens), top-{cfg.K}, {'1 fused shared expert' if cfg.S else 'no shared expert'}",
            "step": "layout + NVFP4 dispatch (2688/rowmax global scale, E2M1 / E4M3 blocks of 16) + combine",
            "tokens_per_step": cfg.T, "hidden": cfg.H, "n_experts": cfg.E, "top_k": cfg.K,
            "fused_shared": cfg.S, "n_parts": cfg.P, "capacity": cfg.capacity,
            "l2": L2_NOTE}


def algorithmic_bytes(cfg: W.Config, R: int) -> dict:
    """Minimum bytes each kernel must move: x read once, every copy written once, every expert
    row read once, the metadata once.  R = rows in use; R - S*T of them are routed rows."""
    T, H, K, S = cfg.T, cfg.H, cfg.K, cfg.S
    routed = R - S * T
    return {
        "layout": 4 * T * K + 12 * R + 4 * T * K,
        "dispatch_nvfp4": 2 * T * H + R * (H // 2 + H // 16 + 2),
        "combine": 2 * R * H + 8 * T * K + 2 * T * H,
        # the rows the benchmark step does not run, timed on the same workload
        "dispatch_bf16": 2 * T * H + 2 * R * H + 4 * T * K,
        "combine_bwd": 2 * T * H + 2 * routed * H + 2 * R * H + 12 * T * K,
        "dispatch_bwd": 2 * R * H + 4 * T * K + 2 * T * H,
        "dispatch_fp8": 2 * T * H + R * (H + 4 * (H // 128)),
        # dense routing map in (T*E bytes + T*E fp32 probabilities), compact ids / probs out,
        # then the layout of those ids
        "routing_map_layout": 5 * T * cfg.E + 8 * T * K + (4 * T * K + 12 * R + 4 * T * K),
        "indices_to_multihot": 8 * T * K + 5 * T * cfg.E,
    }


def padded_bytes(cfg: W.Config, R_pad: int) -> dict:
    """Layout and NVFP4 dispatch of a padded layout: every row below R_pad (padding rows
    included) is written once."""
    T, H, K = cfg.T, cfg.H, cfg.K
    return {"layout": 4 * T * K + 12 * R_pad + 4 * T * K,
            "dispatch_nvfp4": 2 * T * H + R_pad * (H // 2 + H // 16 + 2)}


def load_peaks() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


COMBINE_SOURCES = ("ep_common.cuh", "ep_padding.cuh", "ep_combine.cu")   # device code of combine's unit


def kernel_source_hash(files=COMBINE_SOURCES) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "combine_topk_ids_histogram_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name: str) -> float | None:
    """DRAM bytes (read + written) per launch from the ncu capture recorded in
    profiles/<name>.json, if that capture was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{name}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    files = tuple(rec.get("source_files", COMBINE_SOURCES))
    if rec.get("source_sha256_16") != kernel_source_hash(files):
        return None
    return float(rec["traffic_bytes_per_launch"])


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self) -> None:
        """End sampling; summary() then reads the samples of any time window."""
        self.out = ""
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.out, _ = self.proc.communicate()

    def summary(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows, reasons = [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and self.uuid not in parts[1]:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smax = float(parts[2].split()[0]), float(parts[3].split()[0])
            except (ValueError, IndexError):
                continue
            if t0 - 0.05 <= ts <= t1 + 0.05:
                rows.append((sm, smax))
                for n, v in zip(names, parts[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = sorted(r[0] for r in rows)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------------------------------
# distributed helpers (independent replicas; only the timing is reduced)
# ------------------------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(v: float, ws: int, device) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------------------
# CPU oracle (reported baseline and the reference arm)
# ------------------------------------------------------------------------------------------
def oracle_step(oracle, cfg: W.Config, inp: dict, y: np.ndarray, T_s: int) -> None:
    """The same step on the CPU oracle for the first T_s tokens of the workload."""
    ids = inp["topk_ids"][:T_s]
    L = oracle.layout(ids, cfg.E, P=cfg.P, C=cfg.capacity, S=cfg.S)
    oracle.dispatch_nvfp4(inp["x"][:T_s], L)
    oracle.combine(y[:L.R_max], inp["probs"][:T_s], L)


def host_cpu() -> dict:
    """The host the oracle runs on: its logical CPU count and model name (from lscpu when it is
    there, else the platform string)."""
    import platform
    import subprocess
    model = platform.processor() or platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"host_cpus": os.cpu_count(), "host_cpu_model": model}


def time_oracle(cfg: W.Config, inp: dict, y: np.ndarray, budget_s: float, T_s: int | None = None):
    import oracle
    oracle.build()
    if T_s is None:
        # size the sample from a short probe so it takes about budget_s
        probe = max(16, cfg.T // 64)
        t0 = time.perf_counter()
        oracle_step(oracle, cfg, inp, y, probe)
        per_tok = (time.perf_counter() - t0) / probe
        T_s = int(min(cfg.T, max(probe, budget_s / max(per_tok, 1e-9))))
    reps, t_tot = 0, 0.0
    while True:
        t0 = time.perf_counter()
        oracle_step(oracle, cfg, inp, y, T_s)
        t_tot += time.perf_counter() - t0
        reps += 1
        if t_tot >= budget_s or reps >= 8:
            break
    return T_s * reps / t_tot, T_s, reps, t_tot


def oracle_ops(cfg: W.Config, elems: int = 1 << 21, reps: int = 3) -> dict:
    """The oracle as it stands, timed per op on a bounded sample of one workload: T_s tokens
    drawn by the workload's own recipe (its routing distribution, outliers and zero rows), about
    `elems` hidden elements in all.  Each op's wall time is the best of `reps`, on one thread.
    The ops are those the sweep times on the GPU (layout, NVFP4 dispatch, combine), plus the BF16
    dispatch where the workload names it and, on the Qwen3-like layer, both backward passes.
    The layout, which touches no hidden elements, runs on the workload's full routing."""
    import oracle
    oracle.build()
    T_s = min(cfg.T, max(64, elems // cfg.H))
    C = cfg.rerun_C if cfg.rerun_C else cfg.capacity
    sc = W.scaled(cfg, T=T_s, C=C, rerun_C=None, num_permuted_tokens=None)
    inp = W.make_inputs(sc)
    y = W.make_expert_out(sc)
    x, ids, probs = inp["x"], inp["topk_ids"], inp["probs"]
    L = oracle.layout(ids, sc.E, P=sc.P, C=sc.capacity, S=sc.S)
    ids_full = W.make_routing(cfg)[0]
    ops = {
        "layout": lambda: oracle.layout(ids_full, cfg.E, P=cfg.P, C=C, S=cfg.S),
        "dispatch_nvfp4": lambda: oracle.dispatch_nvfp4(x, L),
        "combine": lambda: oracle.combine(y, probs, L),
    }
    if cfg.name in ("tiny", "mixtral"):
        ops["dispatch_bf16"] = lambda: oracle.dispatch_bf16(x, L)
    if cfg.name == "qwen3":
        g = W.make_grad_out(sc)
        gr = W.make_grad_rows(sc)
        ops["combine_bwd"] = lambda: oracle.combine_bwd(g, y, probs, L)
        ops["dispatch_bwd"] = lambda: oracle.dispatch_bwd(gr, L)
    secs = {}
    for name, fn in ops.items():
        best = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            best = min(best, time.perf_counter() - t0)
        secs[name] = best
    tokens = {k: (cfg.T if k == "layout" else T_s) for k in secs}
    return {"kind": "oracle", "cores": 1, "tokens_sampled": T_s, "reps": reps,
            "sample": f"layout over all {cfg.T} tokens; the other ops on {T_s} tokens drawn by the "
                      f"workload's recipe (capacity {C}); best of {reps} per op, single-threaded C oracle",
            "s": secs, "tokens/s": {k: tokens[k] / v for k, v in secs.items()}}


def run_reference(args, cfg):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = W.make_inputs(cfg)
    y = W.make_expert_out(cfg)
    steps, warm = args.steps, args.warmup
    budget_total = 150.0
    per_step = max(0.05, min(3.0, budget_total / max(1, steps + warm)))
    import oracle
    oracle.build()
    probe = max(16, cfg.T // 64)
    t0 = time.perf_counter()
    oracle_step(oracle, cfg, inp, y, probe)
    per_tok = (time.perf_counter() - t0) / probe
    T_s = int(min(cfg.T, max(16, per_step / max(per_tok, 1e-9))))
    for _ in range(warm):
        oracle_step(oracle, cfg, inp, y, T_s)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(oracle, cfg, inp, y, T_s)
    dt = time.perf_counter() - t0
    value = T_s * steps / dt
    sample = (f"first {T_s} of {cfg.T} tokens of the {cfg.name} workload per step (layout over those "
              f"tokens, NVFP4 dispatch, combine), single-threaded C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": steps, "warmup": warm, "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64", "data": "synthetic",
            "config": workload_config(cfg),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                             **host_cpu()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------
def run_ours(args, cfg):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    import combine_topk_ids_histogram_gb300 as ep

    inp = W.make_inputs(cfg)
    y_host = W.make_expert_out(cfg)
    T, H, E, K, S, P, C = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P, cfg.capacity
    R_max = W.r_max(cfg)

    def to_dev_bf16(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    x = to_dev_bf16(inp["x"])
    ids = torch.from_numpy(inp["topk_ids"]).to(dev)
    probs = torch.from_numpy(inp["probs"]).to(dev)
    y = to_dev_bf16(y_host)
    L = ep.Layout(T, K, E, P, bool(S), device=dev)
    fp4 = torch.empty(R_max, H // 2, dtype=torch.uint8, device=dev)
    sc = torch.empty(R_max, H // 16, dtype=torch.uint8, device=dev)
    inv = torch.empty(R_max, dtype=torch.bfloat16, device=dev)
    so = torch.empty(E + S + 1, dtype=torch.int32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_sink = torch.empty((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2():
        flush.fill_(1)
        torch.amax(flush_rd, dim=0, out=flush_sink)

    def step(evs=(None, None, None, None), per_kernel=False):
        """One step: ep_dispatch_layout_nvfp4 (layout and NVFP4 dispatch in one call, the
        quantisation overlapping the layout) then ep_combine.  evs holds the events to record:
        at the start, after the layout (per-kernel loop only), between dispatch and combine, and
        at the end (None: not recorded).  The timed steps record only the first and the last:
        an event recorded between two kernels holds the GPU idle for a few microseconds before
        the next one starts.  A second pass with an event between dispatch and combine times
        combine, the dominant kernel, on its own stream.  The per-kernel breakdown loop instead
        calls ep_dispatch_layout and ep_dispatch_nvfp4 separately, with events between them."""
        def rec(i):
            if evs[i] is not None:
                evs[i].record(stream)
        rec(0)
        if per_kernel:
            ep.dispatch_layout(ids, E, P, C, bool(S), out=L, stream=stream)
            rec(1)
            ep.dispatch_nvfp4(x, L, out=(fp4, sc, inv, so), stream=stream)
        else:
            ep.dispatch_layout_nvfp4(ids, x, E, P, C, bool(S), out_layout=L, out=(fp4, sc, inv, so),
                                     stream=stream)
        rec(2)
        ep.combine(y, probs, L, out=out, stream=stream)
        rec(3)

    # correctness of the run itself: no overflow, every row in use
    step()
    torch.cuda.synchronize(dev)
    status = ep.read_status(L)
    R = int(L.row_offsets[L.G].item())
    if status != 0:
        raise RuntimeError(f"layout status {status} on the benchmark workload")

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize(dev)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    def ev():
        return torch.cuda.Event(enable_timing=True)
    evs = [(ev(), None, None, ev()) for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    for i in range(args.steps):
        flush_l2()
        step(evs[i])
    torch.cuda.synchronize(dev)
    barrier(ws)
    t_host1 = time.time()
    per_step = np.array([e[0].elapsed_time(e[3]) for e in evs]) * 1e-3   # s
    total = float(per_step.sum())
    total_max = reduce_max(total, ws, dev)
    value = ws * T * args.steps / total_max

    # the same steps again with an event between the two calls: combine (the dominant kernel)
    # and the fused call timed live on their stream
    evm = [(ev(), None, ev(), ev()) for _ in range(args.steps)]
    for i in range(args.steps):
        flush_l2()
        step(evm[i])
    torch.cuda.synchronize(dev)
    per = np.array([[e[2].elapsed_time(e[3]), e[0].elapsed_time(e[3]), e[0].elapsed_time(e[2])]
                    for e in evm]) * 1e-3  # s: combine, step with the middle event, fused call
    comb_s = float(per[:, 0].mean())

    # per-kernel breakdown (diagnostic, after the timed region): an event between every kernel
    nb = min(args.steps, 200)
    evb = [(ev(), ev(), ev(), ev()) for _ in range(nb)]
    for i in range(nb):
        flush_l2()
        step(evb[i], per_kernel=True)
    torch.cuda.synchronize(dev)
    brk = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3])]
                    for e in evb]).mean(axis=0) * 1e-3

    # the other kernels of the path (BF16 dispatch and both backward passes), timed the same way
    # on the same layout: events around each launch, L2 flushed before each
    rows_bf16 = torch.empty(R_max, H, dtype=torch.bfloat16, device=dev)
    g_out = torch.from_numpy(W.make_grad_out(cfg).view(np.int16)).to(dev).view(torch.bfloat16)
    g_rows = torch.empty(R_max, H, dtype=torch.bfloat16, device=dev)
    g_probs = torch.empty(T, K, dtype=torch.float32, device=dev)
    g_x = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    fp8_codes = torch.empty(R_max, H, dtype=torch.uint8, device=dev)
    fp8_scales = torch.empty(R_max, H // 128, dtype=torch.float32, device=dev)
    # the same routing as a dense map [T, E] with dense probabilities
    rmap, dprobs = ep.indices_to_multihot(ids, probs, E)
    Lm = ep.Layout(T, K, E, P, bool(S), device=dev)
    map_ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    map_probs = torch.empty(T, K, dtype=torch.float32, device=dev)
    mh_map = torch.empty(T, E, dtype=torch.uint8, device=dev)
    mh_dense = torch.empty(T, E, dtype=torch.float32, device=dev)
    # groups padded to 128 rows (a grouped-GEMM tile), buffers sized for the padded rows
    PAD = 128
    Lp = ep.Layout(T, K, E, P, bool(S), device=dev, pad_multiple=PAD)
    p_fp4 = torch.empty(Lp.R_max, H // 2, dtype=torch.uint8, device=dev)
    p_sc = torch.empty(Lp.R_max, H // 16, dtype=torch.uint8, device=dev)
    p_inv = torch.empty(Lp.R_max, dtype=torch.bfloat16, device=dev)
    p_so = torch.empty(E + S + 1, dtype=torch.int32, device=dev)
    ep.dispatch_layout_routed(E, topk_ids=ids, n_parts=P, capacity=C, fused_shared=bool(S),
                              pad_multiple=PAD, out=Lp, stream=stream)
    extra_fns = {
        "dispatch_bf16": lambda: ep.dispatch_bf16(x, L, out=rows_bf16, stream=stream),
        "combine_bwd": lambda: ep.combine_bwd(g_out, y, probs, L, out=(g_rows, g_probs), stream=stream),
        "dispatch_bwd": lambda: ep.dispatch_bwd(y, L, out=g_x, stream=stream),
        "dispatch_fp8": lambda: ep.dispatch_fp8(x, L, out=(fp8_codes, fp8_scales), stream=stream),
        "routing_map_layout": lambda: ep.dispatch_layout_routed(
            E, routing_map=rmap, dense_probs=dprobs, K=K, n_parts=P, capacity=C, fused_shared=bool(S),
            out=Lm, map_out=(map_ids, map_probs), stream=stream),
        "indices_to_multihot": lambda: ep.indices_to_multihot(ids, probs, E, out=(mh_map, mh_dense),
                                                              stream=stream),
        f"layout (pad {PAD})": lambda: ep.dispatch_layout_routed(
            E, topk_ids=ids, n_parts=P, capacity=C, fused_shared=bool(S), pad_multiple=PAD, out=Lp,
            stream=stream),
        f"dispatch_nvfp4 (pad {PAD})": lambda: ep.dispatch_nvfp4(x, Lp, out=(p_fp4, p_sc, p_inv, p_so),
                                                                 stream=stream),
        f"layout+dispatch_nvfp4 (pad {PAD}, fused call)": lambda: ep.dispatch_layout_padded_nvfp4(
            ids, x, E, P, C, bool(S), PAD, None, out_layout=Lp, out=(p_fp4, p_sc, p_inv, p_so),
            stream=stream),
    }
    extra = {}
    for name, fn in extra_fns.items():
        for _ in range(3):
            flush_l2()
            fn()
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(nb // 2)]
        for a, b in pairs:
            flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        extra[name] = float(np.mean([a.elapsed_time(b) for a, b in pairs])) * 1e-3

    torch.cuda.synchronize(dev)
    if ep.read_status(Lp) != 0 or ep.read_status(Lm) != 0:
        raise RuntimeError("padded or routing-map layout reported an error on the benchmark workload")
    R_pad = int(Lp.row_offsets[Lp.G].item())
    static = static_routing_step(ep, dev, stream, flush_l2, nb)
    graphs = graph_replay(ep, dev, stream, flush_l2, nb)
    # the per-workload sweep (with its pinned-host e2e legs) runs on one GPU only: a run over
    # several GPUs measures the headline step, whose replicas are what scale
    sweep = (config_sweep(ep, dev, stream, flush_l2, min(nb, 100))
             if not args.no_sweep and ws == 1 else None)
    torch.cuda.synchronize(dev)
    t_host2 = time.time()
    clocks = clocks_run = None
    if sampler:   # the timed steps alone, and every GPU phase of the run from them to the sweep
        sampler.stop()
        clocks = sampler.summary(t_host0, t_host1)
        clocks_run = sampler.summary(t_host0, t_host2)
        clocks_run["window"] = "the timed steps through the configs sweep (every GPU phase but e2e)"

    # ---- e2e through the public API with pinned host buffers ----
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    hx = torch.from_numpy(inp["x"].view(np.int16)).pin_memory()
    hids = torch.from_numpy(inp["topk_ids"]).pin_memory()
    hprobs = torch.from_numpy(inp["probs"]).pin_memory()
    hy = torch.from_numpy(y_host.view(np.int16)).pin_memory()
    ho = {n: torch.empty(t.shape, dtype=t.dtype if t.dtype != torch.bfloat16 else torch.int16).pin_memory()
          for n, t in (("fp4", fp4), ("sc", sc), ("inv", inv), ("so", so), ("out", out),
                       ("row_offsets", L.row_offsets), ("expert_ids", L.expert_ids),
                       ("src_info", L.src_info), ("status", L.status))}
    xd16 = x.view(torch.int16)
    yd16 = y.view(torch.int16)

    def e2e_step():
        xd16.copy_(hx, non_blocking=True)
        ids.copy_(hids, non_blocking=True)
        probs.copy_(hprobs, non_blocking=True)
        yd16.copy_(hy, non_blocking=True)
        step()
        for n, t in (("fp4", fp4), ("sc", sc), ("inv", inv.view(torch.int16)), ("so", so),
                     ("out", out.view(torch.int16)), ("row_offsets", L.row_offsets),
                     ("expert_ids", L.expert_ids), ("src_info", L.src_info), ("status", L.status)):
            ho[n].copy_(t, non_blocking=True)

    h2d = sum(t.numel() * t.element_size() for t in (hx, hids, hprobs, hy))
    d2h = sum(t.numel() * t.element_size() for t in ho.values())
    # serial: every step's copies and kernels one after another on one stream
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_serial_t = reduce_max(e0.elapsed_time(e1) * 1e-3, ws, dev)
    barrier(ws)
    # the e2e results are the same bytes as the device-resident run
    if not torch.equal(ho["out"].to(dev), out.view(torch.int16)):
        raise RuntimeError("e2e output differs from the device-resident step")
    del xd16, yd16
    # pipelined: the same copies and calls for every step, with step i's input copies, step
    # i-1's kernels and step i-2's output copies in flight together (three streams, two sets of
    # device buffers)
    e2e_t = pipelined_e2e(ep, cfg, dev, hx, hids, hprobs, hy, e2e_steps, out)
    e2e_t = reduce_max(e2e_t, ws, dev)
    barrier(ws)

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    ab = algorithmic_bytes(cfg, R)
    pb = padded_bytes(cfg, R_pad)
    ab[f"layout (pad {PAD})"] = pb["layout"]
    ab[f"dispatch_nvfp4 (pad {PAD})"] = pb["dispatch_nvfp4"]
    ab[f"layout+dispatch_nvfp4 (pad {PAD}, fused call)"] = pb["layout"] + pb["dispatch_nvfp4"]
    peak, peak_kind = load_peaks()
    achieved = ab["combine"] / comb_s / 1e9
    traffic = recorded_traffic("combine_dsv3")
    kernels = {}
    times = dict(zip(("layout", "dispatch_nvfp4", "combine"), brk))
    times.update(extra)
    ab["layout+dispatch_nvfp4 (fused call)"] = ab["layout"] + ab["dispatch_nvfp4"]
    times["layout+dispatch_nvfp4 (fused call)"] = float(per[:, 2].mean())
    step_timing = {
        "us_per_step": total / args.steps * 1e6,
        "us_per_step_with_middle_event": float(per[:, 1].mean()) * 1e6,
        "note": ("the timed steps record an event at each step's start and end only; the second "
                 "pass records one more between the fused call and combine, which times both but "
                 "holds the GPU idle for a few microseconds before combine starts"),
    }
    for name, sec in times.items():
        gbs = ab[name] / sec / 1e9
        kernels[name] = {"us": sec * 1e6, "algorithmic_bytes": ab[name], "GB/s": gbs,
                         "frac_of_measured_peak": gbs / peak}
    step_bytes = ab["layout"] + ab["dispatch_nvfp4"] + ab["combine"]
    step_s = total / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "dtypes": {"arithmetic": "f32 (quantisation scales, E2M1/E4M3 encoding, combine accumulation)",
                   "activations": "bf16 (x, expert outputs, combined output)",
                   "dispatch_out": "nvfp4: e2m1 codes + e4m3 block scales (16 elements) + bf16 inverse "
                                   "global scale per row",
                   "probs": "f32"},
        "data": "synthetic (seeded: workloads.CONFIGS['dsv3'])",
        "config": workload_config(cfg),
        "roofline": {"kernel": "ep_combine_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": ab["combine"]},
        "step_roofline": {"algorithmic_bytes": step_bytes, "achieved_GB/s": step_bytes / step_s / 1e9,
                          "frac_of_measured_peak": step_bytes / step_s / 1e9 / peak,
                          "frac_of_8TB/s": step_bytes / step_s / 8e12},
        "step_timing": step_timing,
        "kernels": kernels,
        "kernels_note": (f"layout, dispatch_nvfp4 and combine: mean of {nb} diagnostic steps after the "
                         "timed region that call ep_dispatch_layout and ep_dispatch_nvfp4 separately, "
                         "events between kernels; the fused call from the second pass of the step "
                         "(an event between the fused call and combine); the other "
                         "entries (not in the step) timed alone on the same routing, L2 flushed before "
                         f"each call: dispatch_bf16, combine_bwd, dispatch_bwd, dispatch_fp8, the layout "
                         f"from the routing as a dense map (map -> ids, then the layout), "
                         f"indices_to_multihot, and the layout and NVFP4 dispatch with groups padded to "
                         f"{PAD} rows ({R_pad} rows, {R_pad - R} of them padding, written as an "
                         f"all-zero token), as two calls and as one ep_dispatch_layout_padded_nvfp4 "
                         f"call"),
        "static_routing_step": static,
        "graph_replay": graphs,
        "configs_sweep": sweep,
        "e2e": {"value": ws * T * e2e_steps / e2e_t, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "serial_value": ws * T * e2e_steps / e2e_serial_t,
                "schedule": "pipelined: each step copies its inputs host->device, runs the fused "
                            "layout + NVFP4 dispatch call and combine, and copies its results "
                            "device->host; the three overlap across consecutive steps on three "
                            "streams with two sets of device buffers. serial_value runs the same "
                            "steps one after another on one stream",
                "path": "pinned host x/ids/probs/expert outputs -> device, layout + NVFP4 dispatch + "
                        "combine through the C ABI, dispatched rows + metadata + combined output -> host"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "clocks_run": clocks_run,
        "rows": R,
    }
    if ws == 1 and not args.no_cpu_baseline and sweep:
        for entry in sweep:   # the oracle per op on every workload of the sweep
            entry["cpu_oracle"] = oracle_ops(W.CONFIGS[entry["workload"]])
    if ws == 1 and not args.no_cpu_baseline:
        v, T_s, reps, secs = time_oracle(cfg, inp, y_host, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"first {T_s} of {T} tokens per step (layout over them, NVFP4 "
                                          f"dispatch, combine), {reps} step(s), {secs:.1f} s, single thread",
                                **host_cpu()}
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def pipelined_e2e(ep, cfg: W.Config, dev, hx, hids, hprobs, hy, n_steps: int, ref_out,
                  n_in: int = 1, n_out: int = 1) -> float:
    """Seconds for n_steps end-to-end steps through the C ABI, pipelined: host->device copies
    of step i's inputs, step i's fused layout + NVFP4 dispatch and combine, and device->host
    copies of its dispatched rows, metadata and combined output.  Two sets of device buffers
    alternate, so step i's copies overlap the kernels of step i-1 and the result copies of step
    i-2.  The input / result copies can be split by rows over n_in / n_out streams (one
    cudaMemcpyAsync per slice); on GB300 four input and two result streams measured no faster
    than one each, the host link being the limit, so one each is the default.  Checks that the
    last step's host output equals ref_out."""
    import torch
    T, H, E, K, S, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P
    C = cfg.rerun_C if cfg.rerun_C else cfg.capacity
    R_max = W.r_max(cfg)

    def slices(n_rows, n):
        step = (n_rows + n - 1) // n
        return [(j * step, min(n_rows, (j + 1) * step)) for j in range(n) if j * step < n_rows]

    sets = []
    for _ in range(2):
        L = ep.Layout(T, K, E, P, bool(S), device=dev)
        d = {"x": torch.empty(T, H, dtype=torch.int16, device=dev),
             "ids": torch.empty(T, K, dtype=torch.int32, device=dev),
             "probs": torch.empty(T, K, dtype=torch.float32, device=dev),
             "y": torch.empty(R_max, H, dtype=torch.int16, device=dev),
             "fp4": torch.empty(R_max, H // 2, dtype=torch.uint8, device=dev),
             "sc": torch.empty(R_max, H // 16, dtype=torch.uint8, device=dev),
             "inv": torch.empty(R_max, dtype=torch.int16, device=dev),
             "so": torch.empty(E + S + 1, dtype=torch.int32, device=dev),
             "out": torch.empty(T, H, dtype=torch.int16, device=dev), "L": L}
        d_out = [("fp4", d["fp4"]), ("sc", d["sc"]), ("inv", d["inv"]), ("so", d["so"]), ("out", d["out"]),
                 ("row_offsets", L.row_offsets), ("expert_ids", L.expert_ids), ("src_info", L.src_info),
                 ("status", L.status)]
        host = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in d_out}
        ev = {"h2d": [torch.cuda.Event() for _ in range(n_in)], "comp": torch.cuda.Event(),
              "d2h": [torch.cuda.Event() for _ in range(n_out)]}
        sets.append((d, d_out, host, ev))
    s_in = [torch.cuda.Stream(dev) for _ in range(n_in)]
    s_out = [torch.cuda.Stream(dev) for _ in range(n_out)]
    s_comp = torch.cuda.Stream(dev)
    big_in = [("x", hx), ("y", hy)]
    small_in = [("ids", hids), ("probs", hprobs)]

    def one(i):
        d, d_out, host, ev = sets[i % 2]
        L = d["L"]
        for j, s in enumerate(s_in):
            s.wait_event(ev["comp"])          # step i-2's kernels are done with this set's inputs
            with torch.cuda.stream(s):
                for n, h in big_in:
                    a, b = slices(h.shape[0], n_in)[j]
                    d[n][a:b].copy_(h[a:b], non_blocking=True)
                if j == 0:
                    for n, h in small_in:
                        d[n].copy_(h, non_blocking=True)
            ev["h2d"][j].record(s)
        for e in ev["h2d"]:
            s_comp.wait_event(e)
        for e in ev["d2h"]:
            s_comp.wait_event(e)              # step i-2's results have left this set's outputs
        ep.dispatch_layout_nvfp4(d["ids"], d["x"].view(torch.bfloat16), E, P, C, bool(S), out_layout=L,
                                 out=(d["fp4"], d["sc"], d["inv"].view(torch.bfloat16), d["so"]),
                                 stream=s_comp)
        ep.combine(d["y"].view(torch.bfloat16), d["probs"], L, out=d["out"].view(torch.bfloat16),
                   stream=s_comp)
        ev["comp"].record(s_comp)
        for j, s in enumerate(s_out):
            s.wait_event(ev["comp"])
            with torch.cuda.stream(s):
                for n, t in d_out:
                    sl = slices(t.shape[0], n_out)
                    if j < len(sl):
                        a, b = sl[j]
                        host[n][a:b].copy_(t[a:b], non_blocking=True)
            ev["d2h"][j].record(s)

    for i in range(2):
        one(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in[0])
    for s in s_in[1:]:
        s.wait_event(e0)
    for i in range(n_steps):
        one(i)
    for s in s_in + [s_comp] + s_out[1:]:
        s_out[0].wait_stream(s)
    e1.record(s_out[0])
    torch.cuda.synchronize(dev)
    last = sets[(n_steps - 1) % 2][2]["out"]
    if not torch.equal(last.to(dev), ref_out.view(torch.int16)):
        raise RuntimeError("pipelined e2e output differs from the device-resident step")
    return e0.elapsed_time(e1) * 1e-3


def config_sweep(ep, dev, stream, flush_l2, n_steps: int) -> list:
    """The benchmark step (fused layout + NVFP4 dispatch call, then combine) on every workload
    recipe, timed like the headline step: L2 flushed before each step; the step timed with an
    event at its start and end, then the two calls timed in a second pass with an event between.
    Routing comes from the seeded recipes; x and the expert outputs are seeded device draws
    (N(0,1) bf16): the kernels' work does not depend on their values.  The large microbatch runs
    at its rerun capacity, where nothing overflows.

    Each entry also carries:
      ops  -- the other calls the workload names, each timed alone on the same layout (L2
              flushed before each call, events around it): the BF16 dispatch (tiny, Mixtral-like),
              both backward passes (Qwen3-like), and for the large microbatch the fused call at
              its first capacity, which must raise the overflow flag;
      e2e  -- the step through the C ABI from pinned host buffers, pipelined as the headline
              e2e figure is (pipelined_e2e): host->device copies of x, ids, probs and the
              expert outputs, the two calls, device->host copies of every result."""
    import torch
    peak, _ = load_peaks()
    res = []
    for name, cfg in W.CONFIGS.items():
        C = cfg.rerun_C if cfg.rerun_C else cfg.capacity
        T, H, E, K, S, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P
        ids_h, probs_h = W.make_routing(cfg)
        ids = torch.from_numpy(ids_h).to(dev)
        probs = torch.from_numpy(probs_h).to(dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(9000 + cfg.index)
        x = torch.randn(T, H, device=dev, generator=gen).to(torch.bfloat16)
        R_max = W.r_max(cfg)
        y = torch.randn(R_max, H, device=dev, generator=gen).to(torch.bfloat16)
        L = ep.Layout(T, K, E, P, bool(S), device=dev)
        rows = (torch.empty(R_max, H // 2, dtype=torch.uint8, device=dev),
                torch.empty(R_max, H // 16, dtype=torch.uint8, device=dev),
                torch.empty(R_max, dtype=torch.bfloat16, device=dev),
                torch.empty(E + S + 1, dtype=torch.int32, device=dev))
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)

        def step(evs=(None, None, None)):
            if evs[0] is not None:
                evs[0].record(stream)
            ep.dispatch_layout_nvfp4(ids, x, E, P, C, bool(S), out_layout=L, out=rows, stream=stream)
            if evs[1] is not None:
                evs[1].record(stream)
            ep.combine(y, probs, L, out=out, stream=stream)
            if evs[2] is not None:
                evs[2].record(stream)

        step()
        torch.cuda.synchronize(dev)
        if ep.read_status(L) != 0:
            raise RuntimeError(f"layout status on workload {name}")
        R = int(L.row_offsets[L.G].item())
        for _ in range(3):
            flush_l2()
            step()
        def ev():
            return torch.cuda.Event(enable_timing=True)
        evs = [(ev(), None, ev()) for _ in range(n_steps)]
        for e in evs:
            flush_l2()
            step(e)
        evm = [(ev(), ev(), ev()) for _ in range(n_steps)]
        for e in evm:
            flush_l2()
            step(e)
        torch.cuda.synchronize(dev)
        t = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])] for e in evm]).mean(axis=0) * 1e-3
        t = np.append(t, np.mean([e[0].elapsed_time(e[2]) for e in evs]) * 1e-3)
        ab = algorithmic_bytes(cfg, R)
        disp_b, comb_b = ab["layout"] + ab["dispatch_nvfp4"], ab["combine"]
        res.append({
            "workload": name, "T": T, "hidden": H, "n_experts": E, "top_k": K, "fused_shared": S,
            "n_parts": P, "capacity": C, "rows": R, "steps": n_steps,
            "us": {"dispatch": t[0] * 1e6, "combine": t[1] * 1e6, "step": t[2] * 1e6},
            "tokens/s": {"dispatch": T / t[0], "combine": T / t[1], "step": T / t[2]},
            "algorithmic_bytes": {"dispatch": disp_b, "combine": comb_b, "step": disp_b + comb_b},
            "frac_of_measured_peak": {"dispatch": disp_b / t[0] / 1e9 / peak,
                                      "combine": comb_b / t[1] / 1e9 / peak,
                                      "step": (disp_b + comb_b) / t[2] / 1e9 / peak},
            "frac_of_8TB/s": {"step": (disp_b + comb_b) / t[2] / 8e12},
            "ops": sweep_ops(ep, cfg, dev, stream, flush_l2, max(3, n_steps // 2), ids, probs, x, y, L,
                             R, ab, peak),
            "e2e": sweep_e2e(ep, cfg, dev, ids_h, probs_h, x, y, out),
        })
        del x, y, rows, out, L
        torch.cuda.empty_cache()
    return res


def sweep_ops(ep, cfg: W.Config, dev, stream, flush_l2, n: int, ids, probs, x, y, L, R: int, ab: dict,
              peak: float) -> dict:
    """The calls a workload names besides the benchmark step, each timed alone on the step's
    layout and inputs: mean of n launches, L2 flushed before each, events around each.  Combine
    is also timed alone: in the step it carries the write-back of the dispatch's rows that are
    still dirty in L2 when it starts, alone it does not."""
    import torch
    T, H, E, K, S, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P
    R_max = W.r_max(cfg)
    fns, status_of = {}, {}
    out_alone = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    fns["combine"] = lambda: ep.combine(y, probs, L, out=out_alone, stream=stream)
    if cfg.name in ("tiny", "mixtral"):
        rows_bf16 = torch.empty(R_max, H, dtype=torch.bfloat16, device=dev)
        fns["dispatch_bf16"] = lambda: ep.dispatch_bf16(x, L, out=rows_bf16, stream=stream)
    if cfg.name == "qwen3":
        gen = torch.Generator(device=dev)
        gen.manual_seed(9100 + cfg.index)
        g_out = torch.randn(T, H, device=dev, generator=gen).to(torch.bfloat16)
        g_rows = torch.empty(R_max, H, dtype=torch.bfloat16, device=dev)
        g_probs = torch.empty(T, K, dtype=torch.float32, device=dev)
        g_x = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        fns["combine_bwd"] = lambda: ep.combine_bwd(g_out, y, probs, L, out=(g_rows, g_probs), stream=stream)
        fns["dispatch_bwd"] = lambda: ep.dispatch_bwd(y, L, out=g_x, stream=stream)
    if cfg.rerun_C:
        # the first capacity: the layout flags the overflow and the dispatch writes no row
        Lo = ep.Layout(T, K, E, P, bool(S), device=dev)
        o_rows = (torch.empty(R_max, H // 2, dtype=torch.uint8, device=dev),
                  torch.empty(R_max, H // 16, dtype=torch.uint8, device=dev),
                  torch.empty(R_max, dtype=torch.bfloat16, device=dev),
                  torch.empty(E + S + 1, dtype=torch.int32, device=dev))
        name = f"dispatch_layout_nvfp4 (capacity {cfg.capacity}, overflow)"
        fns[name] = lambda: ep.dispatch_layout_nvfp4(ids, x, E, P, cfg.capacity, bool(S), out_layout=Lo,
                                                     out=o_rows, stream=stream)
        status_of[name] = Lo
    res = {}
    for name, fn in fns.items():
        for _ in range(3):
            flush_l2()
            fn()
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(n)]
        for a, b in pairs:
            flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        sec = float(np.mean([a.elapsed_time(b) for a, b in pairs])) * 1e-3
        entry = {"us": sec * 1e6, "tokens/s": T / sec, "launches": n}
        if name in status_of:
            st = ep.read_status(status_of[name])
            if not st & ep.STATUS_OVERFLOW:
                raise RuntimeError(f"{cfg.name}: no overflow flag at capacity {cfg.capacity}")
            entry["status"] = st
        else:
            entry["algorithmic_bytes"] = ab[name]
            entry["frac_of_measured_peak"] = ab[name] / sec / 1e9 / peak
        res[name] = entry
    return res


def sweep_e2e(ep, cfg: W.Config, dev, ids_h, probs_h, x, y, ref_out) -> dict:
    """The step end to end through the C ABI from pinned host buffers (pipelined_e2e), on the
    workload's own inputs; about 1 s of host-link time, 5 to 50 steps."""
    import torch
    hx = x.view(torch.int16).cpu().pin_memory()
    hy = y.view(torch.int16).cpu().pin_memory()
    hids = torch.from_numpy(ids_h).pin_memory()
    hprobs = torch.from_numpy(probs_h).pin_memory()
    T, H, E, K, S, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P
    R_max = W.r_max(cfg)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hids, hprobs, hy))
    # the copies pipelined_e2e makes back: dispatched rows (codes, scales, inverse scales),
    # scales offsets, combined output and the layout's row_offsets, expert_ids, src_info, status
    Ls = ep.Layout(T, K, E, P, bool(S), device=dev)
    d2h = (R_max * (H // 2 + H // 16 + 2) + 4 * (E + S + 1) + 2 * T * H
           + sum(t.numel() * t.element_size() for t in (Ls.row_offsets, Ls.expert_ids, Ls.src_info, Ls.status)))
    del Ls
    n = int(max(5, min(50, 1.0 / max(h2d / 2e11, 1e-6))))
    sec = pipelined_e2e(ep, cfg, dev, hx, hids, hprobs, hy, n, ref_out)
    return {"tokens/s": T * n / sec, "us_per_step": sec / n * 1e6, "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "host_link_GB/s": (h2d + d2h) * n / sec / 1e9}


def graph_replay(ep, dev, stream, flush_l2, n_steps: int) -> list:
    """The benchmark step (fused layout + NVFP4 call, then combine) captured once in a CUDA
    graph and replayed, against the same step launched call by call, on the tiny workload
    (launch-bound) and the DSv3 one.  L2 is flushed before each step; events at each step's
    start and end.  Replays read the buffers captured in the graph."""
    import torch
    res = []
    for name in ("tiny", "dsv3"):
        cfg = W.CONFIGS[name]
        C = cfg.rerun_C if cfg.rerun_C else cfg.capacity
        T, H, E, K, S, P = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P
        ids_h, probs_h = W.make_routing(cfg)
        ids = torch.from_numpy(ids_h).to(dev)
        probs = torch.from_numpy(probs_h).to(dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(9500 + cfg.index)
        x = torch.randn(T, H, device=dev, generator=gen).to(torch.bfloat16)
        R_max = W.r_max(cfg)
        y = torch.randn(R_max, H, device=dev, generator=gen).to(torch.bfloat16)
        L = ep.Layout(T, K, E, P, bool(S), device=dev)
        rows = (torch.empty(R_max, H // 2, dtype=torch.uint8, device=dev),
                torch.empty(R_max, H // 16, dtype=torch.uint8, device=dev),
                torch.empty(R_max, dtype=torch.bfloat16, device=dev),
                torch.empty(E + S + 1, dtype=torch.int32, device=dev))
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)

        def step(st):
            ep.dispatch_layout_nvfp4(ids, x, E, P, C, bool(S), out_layout=L, out=rows, stream=st)
            ep.combine(y, probs, L, out=out, stream=st)

        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            step(cap)                      # the first call sets up the launch configuration
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(cap)
        torch.cuda.synchronize(dev)

        def timed(run):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_steps)]
            for _ in range(3):
                flush_l2()
                run()
            for a, b in evs:
                flush_l2()
                a.record(stream)
                run()
                b.record(stream)
            torch.cuda.synchronize(dev)
            return float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e-3

        eager_s = timed(lambda: step(stream))
        graph_s = timed(g.replay)
        if ep.read_status(L) != 0:
            raise RuntimeError(f"layout status on workload {name}")
        res.append({"workload": name, "T": T, "hidden": H, "steps": n_steps,
                    "us_per_step": {"launched": eager_s * 1e6, "graph": graph_s * 1e6},
                    "tokens/s": {"launched": T / eager_s, "graph": T / graph_s}})
        del g, x, y, rows, out, L
        torch.cuda.empty_cache()
    return res


def static_routing_step(ep, dev, stream, flush_l2, n_steps: int) -> dict:
    """Layout + NVFP4 dispatch + combine on the forced-balanced static routing workload, with its
    persisted row count passed as the static row capacity and groups padded to 128 rows: the
    padded layout + NVFP4 call then combine, and for comparison the layout and the dispatch as
    two calls.  L2 flushed before each step, events around it."""
    import torch
    cfg = W.CONFIGS["dsv3_static"]
    T, H, E, K, S, P, C = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P, cfg.capacity
    inp = W.make_inputs(cfg)
    x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    ids = torch.from_numpy(inp["topk_ids"]).to(dev)
    probs = torch.from_numpy(inp["probs"]).to(dev)
    Ls = ep.Layout(T, K, E, P, bool(S), device=dev, pad_multiple=cfg.pad_multiple,
                   num_permuted_tokens=cfg.num_permuted_tokens)
    Rm = Ls.R_max
    y = torch.from_numpy(np.resize(W.make_expert_out(cfg), (Rm, H)).view(np.int16)).to(dev).view(torch.bfloat16)
    fp4 = torch.empty(Rm, H // 2, dtype=torch.uint8, device=dev)
    sc = torch.empty(Rm, H // 16, dtype=torch.uint8, device=dev)
    inv = torch.empty(Rm, dtype=torch.bfloat16, device=dev)
    so = torch.empty(E + S + 1, dtype=torch.int32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)

    def step():   # the padded layout and the NVFP4 dispatch in one call, then combine
        ep.dispatch_layout_padded_nvfp4(ids, x, E, P, C, bool(S), cfg.pad_multiple, cfg.num_permuted_tokens,
                                        out_layout=Ls, out=(fp4, sc, inv, so), stream=stream)
        ep.combine(y, probs, Ls, out=out, stream=stream)

    def step_two_calls():
        ep.dispatch_layout_routed(E, topk_ids=ids, n_parts=P, capacity=C, fused_shared=bool(S),
                                  pad_multiple=cfg.pad_multiple,
                                  num_permuted_tokens=cfg.num_permuted_tokens, out=Ls, stream=stream)
        ep.dispatch_nvfp4(x, Ls, out=(fp4, sc, inv, so), stream=stream)
        ep.combine(y, probs, Ls, out=out, stream=stream)

    step()
    torch.cuda.synchronize(dev)
    if ep.read_status(Ls) != 0:
        raise RuntimeError("static routing layout reported an error")
    R = int(Ls.row_offsets[Ls.G].item())

    def timed(fn):
        for _ in range(3):
            flush_l2()
            fn()
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(n_steps)]
        for a, b in pairs:
            flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return float(np.mean([a.elapsed_time(b) for a, b in pairs])) * 1e-3

    sec = timed(step)
    sec_two = timed(step_two_calls)
    ab = algorithmic_bytes(cfg, R)
    nbytes = ab["layout"] + ab["dispatch_nvfp4"] + ab["combine"]
    return {"workload": f"{cfg.name}: T={T}, hidden={H}, {E} experts, top-{K}, shared expert, "
                        f"balanced routing ({T * K // E} rows per expert), pad {cfg.pad_multiple}, "
                        f"static row capacity {cfg.num_permuted_tokens}",
            "us_per_step": sec * 1e6, "tokens/s": T / sec, "rows": R, "algorithmic_bytes": nbytes,
            "GB/s": nbytes / sec / 1e9, "steps": n_steps,
            "calls": "ep_dispatch_layout_padded_nvfp4 (+ padding fill) + ep_combine",
            "us_per_step_two_calls": sec_two * 1e6,
            "two_calls": "ep_dispatch_layout_routed + ep_dispatch_nvfp4 (+ padding fill) + ep_combine"}


ONLY_OPS = ("layout", "layout_noalloc", "dispatch_layout_nvfp4", "dispatch_nvfp4", "dispatch_bf16",
            "dispatch_fp8", "combine", "combine_bwd", "dispatch_bwd", "indices_to_multihot",
            "routing_map_layout", "dispatch_nvfp4_padded", "dispatch_layout_padded_nvfp4")


def run_only(args, cfg):
    """One library call alone on one workload, for profiling: only that call's buffers are
    allocated; the routing comes from the workload's recipe and x / expert outputs / gradients
    are seeded device draws.  W + K launches, the L2 flushed before each, CUDA events around the
    K timed ones; prints one JSON line with the mean time and the algorithmic bytes."""
    import torch
    import combine_topk_ids_histogram_gb300 as ep
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    T, H, E, K, S, P, C = cfg.T, cfg.H, cfg.E, cfg.K, cfg.S, cfg.P, cfg.capacity
    R_max = W.r_max(cfg)
    ids_h, probs_h = W.make_routing(cfg)
    ids = torch.from_numpy(ids_h).to(dev)
    probs = torch.from_numpy(probs_h).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(9700 + cfg.index)

    def randn(*shape):
        return torch.randn(*shape, device=dev, generator=gen).to(torch.bfloat16)

    op = args.only
    padded = op in ("dispatch_nvfp4_padded", "dispatch_layout_padded_nvfp4")
    pad = args.pad if padded else 1
    L = ep.Layout(T, K, E, P, bool(S), device=dev, pad_multiple=pad)
    if padded:
        ep.dispatch_layout_routed(E, topk_ids=ids, n_parts=P, capacity=C, fused_shared=bool(S),
                                  pad_multiple=pad, out=L, stream=stream)
        R_max = L.R_max
    else:
        ep.dispatch_layout(ids, E, P, C, bool(S), out=L, stream=stream)
    if op == "layout":
        fn = lambda: ep.dispatch_layout(ids, E, P, C, bool(S), out=L, stream=stream)
    elif op == "layout_noalloc":
        fn = lambda: ep.dispatch_layout_noalloc(ids, E, P, C, bool(S), out=L, stream=stream)
    elif op in ("dispatch_layout_nvfp4", "dispatch_nvfp4", "dispatch_nvfp4_padded",
                "dispatch_layout_padded_nvfp4"):
        x = randn(T, H)
        rows = (torch.empty(R_max, H // 2, dtype=torch.uint8, device=dev),
                torch.empty(R_max, H // 16, dtype=torch.uint8, device=dev),
                torch.empty(R_max, dtype=torch.bfloat16, device=dev),
                torch.empty(E + S + 1, dtype=torch.int32, device=dev))
        if op in ("dispatch_nvfp4", "dispatch_nvfp4_padded"):
            fn = lambda: ep.dispatch_nvfp4(x, L, out=rows, stream=stream)
        elif op == "dispatch_layout_padded_nvfp4":
            fn = lambda: ep.dispatch_layout_padded_nvfp4(ids, x, E, P, C, bool(S), pad, None, out_layout=L,
                                                         out=rows, stream=stream)
        else:
            fn = lambda: ep.dispatch_layout_nvfp4(ids, x, E, P, C, bool(S), out_layout=L, out=rows,
                                                  stream=stream)
    elif op == "dispatch_bf16":
        x, out = randn(T, H), torch.empty(R_max, H, dtype=torch.bfloat16, device=dev)
        fn = lambda: ep.dispatch_bf16(x, L, out=out, stream=stream)
    elif op == "dispatch_fp8":
        x = randn(T, H)
        out = (torch.empty(R_max, H, dtype=torch.uint8, device=dev),
               torch.empty(R_max, H // 128, dtype=torch.float32, device=dev))
        fn = lambda: ep.dispatch_fp8(x, L, out=out, stream=stream)
    elif op in ("combine", "dispatch_bwd"):
        y, out = randn(R_max, H), torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        if op == "combine":
            fn = lambda: ep.combine(y, probs, L, out=out, stream=stream)
        else:
            fn = lambda: ep.dispatch_bwd(y, L, out=out, stream=stream)
    elif op == "combine_bwd":
        y, g = randn(R_max, H), randn(T, H)
        out = (torch.empty(R_max, H, dtype=torch.bfloat16, device=dev),
               torch.empty(T, K, dtype=torch.float32, device=dev))
        fn = lambda: ep.combine_bwd(g, y, probs, L, out=out, stream=stream)
    elif op == "indices_to_multihot":
        out = (torch.empty(T, E, dtype=torch.uint8, device=dev), torch.empty(T, E, dtype=torch.float32, device=dev))
        fn = lambda: ep.indices_to_multihot(ids, probs, E, out=out, stream=stream)
    else:   # routing_map_layout
        rmap, dprobs = ep.indices_to_multihot(ids, probs, E)
        Lm = ep.Layout(T, K, E, P, bool(S), device=dev)
        mo = (torch.empty(T, K, dtype=torch.int32, device=dev), torch.empty(T, K, dtype=torch.float32, device=dev))
        fn = lambda: ep.dispatch_layout_routed(E, routing_map=rmap, dense_probs=dprobs, K=K, n_parts=P,
                                               capacity=C, fused_shared=bool(S), out=Lm, map_out=mo,
                                               stream=stream)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        flush.fill_(1)
        torch.amax(flush_rd, dim=0, out=sink)
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        flush.fill_(1)
        torch.amax(flush_rd, dim=0, out=sink)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize(dev)
    sec = float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e-3
    R = int(L.row_offsets[L.G].item())
    ab = padded_bytes(cfg, R) if padded else algorithmic_bytes(cfg, R)
    key = {"layout_noalloc": "layout", "dispatch_nvfp4_padded": "dispatch_nvfp4"}.get(op, op)
    if op in ("dispatch_layout_nvfp4", "dispatch_layout_padded_nvfp4"):
        nbytes = ab["layout"] + ab["dispatch_nvfp4"]
    else:
        nbytes = ab.get(key)
    line = {"only": op, "workload": cfg.name, "T": T, "hidden": H, "pad_multiple": pad, "rows": R,
            "steps": args.steps,
            "warmup": args.warmup, "us": sec * 1e6, "algorithmic_bytes": nbytes,
            "GB/s": nbytes / sec / 1e9 if nbytes else None}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=WORKLOAD, choices=sorted(W.CONFIGS))
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the per-workload sweep (fused layout + NVFP4 dispatch, combine, step)")
    ap.add_argument("--only", choices=ONLY_OPS,
                    help="run one library call alone on --config (for profiling) and print its time")
    ap.add_argument("--tokens", type=int, default=None,
                    help="with --only: the workload's recipe at this many tokens")
    ap.add_argument("--pad", type=int, default=128,
                    help="with --only dispatch_nvfp4_padded / dispatch_layout_padded_nvfp4: rows per "
                         "group multiple")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = W.CONFIGS[args.config]
    if cfg.rerun_C is not None:
        cfg = W.scaled(cfg, C=cfg.rerun_C)
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.only:
        if args.tokens:
            cfg = W.scaled(cfg, T=args.tokens, C=max(cfg.capacity, args.tokens) if cfg.C else None)
        return run_only(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
