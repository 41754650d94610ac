#!/usr/bin/env python3
"""Benchmark of branch attention forward + backward on one GB300.

One step = ba_forward + ba_backward over the whole 256K-token EAGLE-3 TTT
workload (1 sequence of 262144 main tokens, depth 7, 32 q / 8 kv heads,
head_dim 128, virtual CP degree 8), inputs resident in HBM.  Prints ONE JSON
line (rank 0).  Under torchrun each rank runs an independent replica (the
path has no data exchange on one GPU per process: replicas only) and the
timing is the max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle instead (host cores, bounded
sample of the same workload).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "branch-attn fwd+bwd useful TFLOP/s at 256K tokens; % of bf16 tensor peak"
UNIT = "TFLOP/s"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# --------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        top = max(smax)
        loaded = [x for x in sm if x >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": top, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- distributed


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over the ranks (timings: the job is as slow as its slowest
    replica).  Uses a CUDA tensor under NCCL and a CPU tensor under gloo."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(ms_local: float, flops_per_replica: float, world: int):
    """Whole-job throughput of ``world`` independent replicas (weak scaling):
    every rank runs the full workload, the step time is the max over ranks.
    Returns (TFLOP/s over all ranks, ms per step)."""
    ms = max_over_ranks(ms_local, world)
    return world * flops_per_replica / (ms / 1e3) / 1e12, ms


# --------------------------------------------------------------------------- oracle sample (CPU)


class _HostSource:
    """Oracle input source prefetched to host memory (rows of the sampled
    units and the main K/V columns), so that only the oracle is timed."""

    def __init__(self, wl, tensors, units):
        import oracle
        self.wl = wl
        qids = np.concatenate([oracle.keysets.queries_of_unit(wl, u) for u in units])
        self.qpos = {int(q): i for i, q in enumerate(qids)}
        self.bpos = self.qpos
        fetch = lambda name, heads: tensors[name].reshape(-1, heads, wl.head_dim).index_select(
            0, _idx(qids, tensors[name].device)).float().cpu().double().numpy()
        self.q = fetch("q_b", wl.heads_q)
        self.do = fetch("d_o", wl.heads_q)
        self.kb = fetch("k_b", wl.heads_kv)
        self.vb = fetch("v_b", wl.heads_kv)
        self.km = tensors["k_m"].float().cpu().double().numpy()
        self.vm = tensors["v_m"].float().cpu().double().numpy()
        self._main = {}

    def rows(self, name, ids):
        src = {"q_b": self.q, "d_o": self.do, "k_b": self.kb, "v_b": self.vb}[name]
        return src[[self.qpos[int(i)] for i in ids]]

    def main(self, name, kh):
        key = (name, kh)
        if key not in self._main:
            self._main[key] = np.ascontiguousarray((self.km if name == "k_m" else self.vm)[:, kh])
        return self._main[key]


def _idx(ids, device):
    import torch
    return torch.as_tensor(np.asarray(ids, dtype=np.int64), device=device)


def _unit_flops(wl, unit):
    """Useful fwd + bwd flops of every query-head row of one anchor unit."""
    import oracle
    qids = oracle.keysets.queries_of_unit(wl, unit)
    pairs = int(oracle.keysets.key_count(wl, qids).sum()) * wl.heads_q
    return 4.0 * wl.head_dim * pairs * 3.5


def oracle_sample(wl, tensors, budget_s: float, seed: int = 7, max_units: int = 256):
    """Times the CPU oracle on seeded anchor units until ~budget_s of work.
    Returns (useful TFLOP/s, units, seconds, threads)."""
    import oracle
    rng = np.random.default_rng(seed)
    nu = oracle.keysets.num_units(wl)
    units = [int(u) for u in rng.choice(nu, size=min(nu, max_units), replace=False)]
    src = _HostSource(wl, tensors, units)
    done, flops, t0 = 0, 0.0, time.perf_counter()
    for u in units:
        oracle.attention.unit_eval(wl, src, [u], grads=True)
        done += 1
        flops += _unit_flops(wl, u)
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, done, dt


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------- our arm


# GEMMs per (row, key) pair each main-attention kernel runs: forward S and PV;
# backward: key-stationary S, dP, dV, dK and query-stationary S, dP, dQ.
MAIN_KERNEL_GEMMS = {"main_fwd": 2, "main_bwd_kv": 4, "main_bwd_dq": 3}


def kernel_bytes(wl, info, name):
    """Algorithmic HBM bytes per step of a memory-bound kernel."""
    R = info["query_rows"]
    d = wl.head_dim
    T = wl.tokens
    nbk = (wl.depth * T if wl.family == "ttt" else wl.num_anchors * wl.block) * wl.heads_kv
    if name == "zigzag_pack":  # one pass packing q, k_m, v_m, k_b, v_b: read + write
        return 2 * 2 * (R * d + 2 * T * wl.heads_kv * d + 2 * nbk * d)
    if name == "lse_merge":
        return R * (2 * d * 4 + 2 * 4) + R * (d * 2 + 4)
    if name == "bwd_prep":  # read o, dO, lse; write the row record
        return R * (2 * d * 2 + 4) + R * 16
    if name == "branch_bwd":  # read q, dO, dq (main part), the row records, k_b, v_b; write dq, dk_b, dv_b
        return R * (3 * d * 2 + 16) + 2 * nbk * d * 2 + R * d * 2 + 2 * nbk * d * 2
    return None


def run_ours(args, rank, world, local):
    import torch
    from branch_attention_speculative_gb300 import api, workloads as W

    peaks = load_peaks()
    wl = W.config(args.config)
    if args.tokens:
        wl = resize_workload(wl, args.tokens)
    plan = api.Plan.from_workload(wl)
    info = plan.info()
    t = W.make_tensors(wl, device="cuda")
    ws = plan.workspace()
    o = torch.empty_like(t["q_b"])
    lse = torch.empty(t["q_b"].shape[:-1], dtype=torch.float32, device="cuda")
    grads = {"dq_b": torch.empty_like(t["q_b"]), "dk_m": torch.empty_like(t["k_m"]),
             "dv_m": torch.empty_like(t["v_m"]), "dk_b": torch.empty_like(t["k_b"]),
             "dv_b": torch.empty_like(t["v_b"])}

    def step():
        plan.forward(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"], o=o, lse=lse, workspace=ws)
        plan.backward(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"], o, lse, t["d_o"], grads=grads,
                      workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = plan.check_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    plan.profile(True)
    plan.profile_read()
    sampler = ClockSampler(local)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    barrier(world)
    clocks = sampler.stop()
    kt = plan.profile_read()
    plan.profile(False)
    ms_local = e0.elapsed_time(e1) / args.steps
    status = plan.check_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after timed steps")

    flops = info["fwd_flops"] + info["bwd_flops"]
    value, ms = aggregate_throughput(ms_local, flops, world)
    peak_t = peaks["bf16_tflops_sustained"]

    kernels = {}
    for name, (n, tot) in kt.items():
        per = tot / max(n, 1)
        ent = {"launches": n, "ms_total_per_step": tot / args.steps, "ms_per_launch": per}
        gemms = MAIN_KERNEL_GEMMS.get(name)
        if gemms is not None:
            # algorithmic flops of the GEMMs the kernel must run: 2 d flops per
            # (row, key) pair per GEMM (S, P V, dP, dV, dK, dQ, ...)
            f = 2.0 * wl.head_dim * info["main_pairs"] * gemms
            ent["gemms_per_pair"] = gemms
            ent["achieved"] = f / (tot / args.steps / 1e3) / 1e12
            ent["unit"] = "TFLOP/s"
        else:
            b = kernel_bytes(wl, info, name)
            if b is not None:
                ent["achieved"] = b / (tot / args.steps / 1e3) / 1e9
                ent["unit"] = "GB/s"
        kernels[name] = ent
    dom = max(kt.items(), key=lambda kv: kv[1][1])[0] if kt else None
    roofline = None
    if dom is not None and "achieved" in kernels[dom]:
        e = kernels[dom]
        if e.get("unit") == "TFLOP/s":
            roofline = {"kernel": dom, "bound": "tensor", "achieved": e["achieved"], "peak": peak_t,
                        "unit": "TFLOP/s", "frac": e["achieved"] / peak_t,
                        "traffic": measured_traffic(dom, wl.name),
                        "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                        "peak_source": f"bf16_tflops_sustained ({peaks['source']})"}
            if clocks.get("sm_mhz"):
                # The measured peak ran at its own clock; this is the dense bf16
                # rate of the tensor pipes at this run's median SM clock: 8192
                # FLOP per clock per SM (one M=128, N=128, K=16 MMA every 64
                # cycles, measured) times the SMs.
                sms = torch.cuda.get_device_properties(local).multi_processor_count
                at_clock = 8192.0 * sms * clocks["sm_mhz"] * 1e6 / 1e12
                roofline["peak_at_clock"] = at_clock
                roofline["frac_at_clock"] = e["achieved"] / at_clock
        else:
            roofline = {"kernel": dom, "bound": "hbm", "achieved": e["achieved"], "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": e["achieved"] / peaks["hbm_gbs"], "traffic": None,
                        "peak_source": f"hbm_gbs ({peaks['source']})"}
    launches = sum(n for n, _ in kt.values())

    extra = {}
    if args.extras:
        extra = run_extras(args, plan, wl, t, info, peaks, ws, o, lse, grads)

    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, plan, wl, t, info, world, ws, o, lse, grads)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, units, secs = oracle_sample(wl, t, args.cpu_budget)
        cpu = {"value": tf, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"{units} seeded anchor units (all {wl.steps} steps x {wl.heads_q} heads each, fwd+bwd, "
                         f"fp64 numpy) of the same workload, {secs:.1f} s"}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 inputs)",
        "config": {"workload": wl.name, "family": wl.family, "tokens": wl.tokens, "ttt_depth": wl.depth,
                   "heads_q": wl.heads_q, "heads_kv": wl.heads_kv, "head_dim": wl.head_dim, "cp_virtual": wl.cp,
                   "fwd_flops": info["fwd_flops"], "bwd_flops": info["bwd_flops"],
                   "l2": "inputs larger than L2 (tens of GB per step)", "parallelism": f"replicas x{world}"},
        "pct_of_bf16_peak": value / world / peak_t,
        "wall_s_timed": wall1 - wall0,
        "roofline": roofline,
        "kernels": kernels,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    line.update(extra)
    return line


def _time_launches(fn, n, warm=1):
    """Mean device time (ms) of ``fn`` over ``n`` calls on the current stream,
    after ``warm`` untimed calls; CUDA events on that stream."""
    import torch
    for _ in range(warm):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def run_extras(args, plan, wl, t, info, peaks, ws, o, lse, grads):
    """Measurements outside the timed fwd+bwd steps, on the same workload:
    the 8-bit forward (its TFLOP/s against an fp8 peak of twice the measured
    bf16 one: the nominal dense rates are 4.5 and 2.25 PFLOP/s) and the
    memory-bound kernels that the step does not launch (the zigzag pack, folded
    into the kernels' load coordinates, and the stand-alone Eq. 2 merge)."""
    import torch
    from branch_attention_speculative_gb300 import api
    out = {}
    # ---- 8-bit forward
    f8 = None
    try:
        ws8 = torch.empty(plan.workspace_bytes_fp8, dtype=torch.uint8, device="cuda")
    except RuntimeError as e:  # out of memory
        ws8 = None
        f8 = {"skipped": str(e).splitlines()[0]}
    if ws8 is not None:
        run = lambda: plan.forward_fp8(t["q_b"], t["k_m"], t["v_m"], t["k_b"], t["v_b"], o=o, lse=lse, workspace=ws8)
        run()
        torch.cuda.synchronize()
        if plan.check_device_status(ws8) != 0:
            raise RuntimeError("device status after the 8-bit forward")
        plan.profile(True)
        plan.profile_read()
        ms = _time_launches(run, args.steps, warm=0)
        kt = plan.profile_read()
        plan.profile(False)
        peak8 = 2.0 * peaks["bf16_tflops_sustained"]
        main_f = 4.0 * wl.head_dim * info["main_pairs"]
        km = kt.get("main_fwd_fp8", (1, float("nan")))
        kmain = km[1] / max(km[0], 1)
        f8 = {"value": info["fwd_flops"] / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_forward": ms,
              "dtype": "e4m3 QK^T and PV, fp32 softmax / lse, bf16 in and out",
              "main_kernel": {"name": "main_fwd_fp8", "ms_per_launch": kmain,
                              "achieved": main_f / (kmain / 1e3) / 1e12, "unit": "TFLOP/s", "peak": peak8,
                              "frac": main_f / (kmain / 1e3) / 1e12 / peak8,
                              "peak_source": f"2 x bf16_tflops_sustained ({peaks['source']}); nominal fp8 / bf16 "
                                             "dense ratio 4.5 / 2.25"},
              "kernels": {k: {"launches": n, "ms_per_launch": v / max(n, 1)} for k, (n, v) in kt.items()}}
    out["fp8_forward"] = f8
    # ---- memory-bound kernels outside the step
    mb = {}
    hbm = peaks["hbm_gbs"]
    ms = _time_launches(lambda: plan.zigzag_pack("query", t["q_b"], dst=grads["dq_b"], workspace=ws), 5)
    by = 2 * t["q_b"].numel() * 2
    mb["zigzag_pack"] = {"bytes_per_launch": by, "ms_per_launch": ms, "achieved": by / (ms / 1e3) / 1e9,
                         "unit": "GB/s", "peak": hbm, "frac": by / (ms / 1e3) / 1e9 / hbm,
                         "what": f"q_b {tuple(t['q_b'].shape)} bf16 into zigzag order (read + write)"}
    del ws8
    torch.cuda.empty_cache()
    rows, d = 1 << 24, wl.head_dim
    try:
        buf = torch.empty(2 * rows * d + 2 * rows, dtype=torch.float32, device="cuda")
    except RuntimeError as e:  # out of memory
        buf = None
        mb["lse_merge"] = {"skipped": str(e).splitlines()[0]}
    if buf is not None:
        om, ob = buf[: rows * d].view(rows, d), buf[rows * d: 2 * rows * d].view(rows, d)
        lm, lb = buf[2 * rows * d: 2 * rows * d + rows], buf[2 * rows * d + rows:]
        g = torch.Generator(device="cuda").manual_seed(5)
        for x in (om, ob, lm, lb):
            x.normal_(generator=g)
        res = {}

        def merge():
            res["o"] = api.lse_merge(om, lm, ob, lb)

        ms = _time_launches(merge, 5)
        by = rows * (2 * d * 4 + 2 * 4) + rows * (d * 2 + 4)
        mb["lse_merge"] = {"bytes_per_launch": by, "ms_per_launch": ms, "achieved": by / (ms / 1e3) / 1e9,
                           "unit": "GB/s", "peak": hbm, "frac": by / (ms / 1e3) / 1e9 / hbm,
                           "what": f"Eq. 2 over {rows} rows x {d}: fp32 partials in, bf16 o and fp32 lse out "
                                   "(includes the output allocation of the binding)"}
        del res, buf
    out["memory_bound"] = mb
    torch.cuda.empty_cache()
    return out


def resize_workload(wl, tokens: int):
    """The same shape with one main sequence of ``tokens`` tokens (a multiple
    of 2C); block families keep their anchor density.  Used for profiling
    captures that must stay small."""
    from branch_attention_speculative_gb300 import workloads as W
    if tokens % (2 * wl.cp) != 0:
        raise SystemExit(f"--tokens must be a multiple of 2C = {2 * wl.cp}")
    cu = W.cu_from_lens([tokens])
    anchors = None
    if wl.family == "block":
        per = max(1, int(round(wl.anchors_per_seq * tokens / (wl.tokens / wl.num_seqs))))
        anchors = W.sample_anchors(np.random.default_rng(wl.seed), cu, per)
    return W.Workload(f"{wl.name}_T{tokens}", wl.family, cu, wl.heads_q, wl.heads_kv, wl.head_dim, wl.cp,
                      wl.depth, wl.block, anchors, wl.seed)


KERNEL_SOURCES = {
    "main_fwd": "main_fwd_tc.cu", "main_bwd_kv": "main_bwd_tc.cu", "main_bwd_dq": "main_bwd_q_tc.cu",
}


def source_sha256(kernel: str):
    import hashlib
    f = KERNEL_SOURCES.get(kernel)
    if f is None:
        return None
    path = os.path.join(ROOT, "branch_attention_speculative_gb300", "csrc", f)
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) of ``kernel`` on ``workload`` from
    the committed ncu summary profiles/dram_traffic.md, or None when there is
    no capture or the kernel's source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    if not os.path.exists(path):
        return None
    want = source_sha256(kernel)
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 6 and cells[0] == kernel and cells[1] == workload:
            try:
                sha, rd, wr = cells[2], float(cells[3]), float(cells[4])
            except ValueError:
                continue
            return rd + wr if sha == want else None
    return None


def _mem_available_bytes():
    try:
        for ln in open("/proc/meminfo"):
            if ln.startswith("MemAvailable:"):
                return int(ln.split()[1]) * 1024
    except OSError:
        pass
    return 0


def run_e2e(args, plan, wl, t, info, world, ws, o, lse, grads):
    """Same metric through the public API with host buffers: every step
    copies its inputs host->device from pinned memory and reads every result
    back device->host, inside the timed region.

    The copies run on their own streams and overlap the compute the way a
    training loop's input pipeline does: step k+1's forward inputs go up while
    step k runs its backward (into a second set of input buffers), step k's
    d_o goes up during its forward, o / lse come down during the backward and
    the gradients during the next step's forward.  Events order every buffer
    reuse.  The first step's forward inputs and the last step's gradients
    cannot overlap anything, so they are exposed inside the timed region."""
    import torch
    fwd_in = ["q_b", "k_m", "v_m", "k_b", "v_b"]
    ins = fwd_in + ["d_o"]
    fwd_out = {"o": o, "lse": lse}
    outs = {**fwd_out, **grads}
    in_bytes = sum(t[n].numel() * t[n].element_size() for n in ins)
    out_bytes = sum(v.numel() * v.element_size() for v in outs.values())
    extra = sum(t[n].numel() * t[n].element_size() for n in fwd_in)
    need = in_bytes + out_bytes
    if _mem_available_bytes() < 1.25 * need:
        return {"value": None, "unit": UNIT, "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
                "skipped": f"host memory available {_mem_available_bytes() / 1e9:.0f} GB < {1.25 * need / 1e9:.0f} GB"}
    free_dev, _ = torch.cuda.mem_get_info()
    pipelined = free_dev > extra + (4 << 30)
    h_in = {n: torch.empty(t[n].shape, dtype=t[n].dtype, pin_memory=True) for n in ins}
    for n in ins:
        h_in[n].copy_(t[n])
    h_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    # two sets of forward-input buffers (the second only when it fits)
    dev_in = [{n: t[n] for n in fwd_in}]
    if pipelined:
        dev_in.append({n: torch.empty_like(t[n]) for n in fwd_in})
    comp = torch.cuda.current_stream()
    up = torch.cuda.Stream()
    down = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()

    def run(nsteps):
        nb = len(dev_in)
        in_ready = [None] * nsteps
        bwd_done = [None] * nsteps
        olse_read, grads_read = None, None
        with torch.cuda.stream(up):
            for n in fwd_in:
                dev_in[0][n].copy_(h_in[n], non_blocking=True)
            in_ready[0] = ev()
            in_ready[0].record(up)
        for k in range(nsteps):
            buf = dev_in[k % nb]
            # d_o of step k (single buffer): after step k-1's backward read it
            with torch.cuda.stream(up):
                if k > 0:
                    up.wait_event(bwd_done[k - 1])
                t["d_o"].copy_(h_in["d_o"], non_blocking=True)
                do_ready = ev()
                do_ready.record(up)
            comp.wait_event(in_ready[k])
            if olse_read is not None:
                comp.wait_event(olse_read)  # o / lse of step k-1 are on the host
            plan.forward(buf["q_b"], buf["k_m"], buf["v_m"], buf["k_b"], buf["v_b"], o=o, lse=lse, workspace=ws)
            fwd_done = ev()
            fwd_done.record(comp)
            with torch.cuda.stream(down):
                down.wait_event(fwd_done)
                for kk, v in fwd_out.items():
                    h_out[kk].copy_(v, non_blocking=True)
                olse_read = ev()
                olse_read.record(down)
            # the next step's forward inputs, into the other buffer set, once
            # step k-1 (its last user) has finished its backward
            if k + 1 < nsteps and nb == 2:
                with torch.cuda.stream(up):
                    if k >= 1:
                        up.wait_event(bwd_done[k - 1])
                    for n in fwd_in:
                        dev_in[(k + 1) % nb][n].copy_(h_in[n], non_blocking=True)
                    in_ready[k + 1] = ev()
                    in_ready[k + 1].record(up)
            comp.wait_event(do_ready)
            if grads_read is not None:
                comp.wait_event(grads_read)  # step k-1's gradients are on the host
            plan.backward(buf["q_b"], buf["k_m"], buf["v_m"], buf["k_b"], buf["v_b"], o, lse, t["d_o"],
                          grads=grads, workspace=ws)
            bwd_done[k] = ev()
            bwd_done[k].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(bwd_done[k])
                for kk, v in grads.items():
                    if v is not None:
                        h_out[kk].copy_(v, non_blocking=True)
                grads_read = ev()
                grads_read.record(down)
            if k + 1 < nsteps and nb == 1:
                with torch.cuda.stream(up):
                    up.wait_event(bwd_done[k])
                    for n in fwd_in:
                        dev_in[0][n].copy_(h_in[n], non_blocking=True)
                    in_ready[k + 1] = ev()
                    in_ready[k + 1].record(up)
        torch.cuda.synchronize()

    run(1)
    steps = max(args.e2e_steps, 1)
    t0 = time.perf_counter()
    run(steps)
    dt = (time.perf_counter() - t0) / steps
    dt = max_over_ranks(dt, world)
    flops = info["fwd_flops"] + info["bwd_flops"]
    return {"value": world * flops / dt / 1e12, "unit": UNIT, "h2d_bytes_per_step": in_bytes,
            "d2h_bytes_per_step": out_bytes, "ms_per_step": dt * 1e3, "steps": steps,
            "copies": "overlapped with compute on two copy streams" + ("" if pipelined else
                                                                           " (one input buffer set)")}


# --------------------------------------------------------------------------- reference arm


def run_reference(args, rank, world):
    import torch
    from branch_attention_speculative_gb300 import workloads as W
    wl = W.config(args.config)
    t = W.make_tensors(wl, device="cuda")
    budget = args.ref_step_s
    vals, units_total, secs_total = [], 0, 0.0
    for i in range(args.warmup + args.steps):
        tf, units, secs = oracle_sample(wl, t, budget, seed=100 + i, max_units=64)
        if i >= args.warmup:
            vals.append((tf, units, secs))
            units_total += units
            secs_total += secs
    value = sum(v[0] * v[2] for v in vals) / max(secs_total, 1e-9)
    ms = secs_total / max(args.steps, 1) * 1e3
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs, upcast to fp64)",
        "config": {"workload": wl.name, "family": wl.family, "tokens": wl.tokens, "ttt_depth": wl.depth,
                   "heads_q": wl.heads_q, "heads_kv": wl.heads_kv, "head_dim": wl.head_dim, "cp_virtual": wl.cp},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": f"{units_total} seeded anchor units over {args.steps} steps "
                                   f"(~{budget:.0f} s of fp64 numpy each), fwd+bwd rows"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5, help="measured shape 1..5 (5 = 256K TTT, the headline)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-step-s", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="skip the 8-bit forward and memory-bound kernel measurements")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: shrink the main sequence to this many tokens")
    args = ap.parse_args()

    rank, world, local = dist_setup()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    from branch_attention_speculative_gb300 import build as B
    if rank == 0:
        B.build()
    barrier(world)
    if world > 1 and rank != 0:
        B.build()  # no-op once rank 0 has built; loads the same library
    line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
