"""Benchmark: per-token logprob + entropy + weighted backward at V = 151,936.

One step is one pass of the hot path over one batch of T = 8192 rows of bf16
logits N(0, 2^2), labels sampled from each row's softmax, weights N(0, 1) x a
0/1 mask with 20% zeros: logprob, entropy and bf16 dlogits.  The headline
step is pstat_forward_backward (statistics and gradient in one pass over the
logits); the same workload through pstat_forward + pstat_backward is timed in
the same run under `two_call`, with each kernel's bandwidth.

Prints ONE JSON line (rank 0).  `value` is whole-job tokens/s with inputs
resident in HBM, over R back-to-back blocks of `--steps` steps (R sized so
the timed region lasts at least a second); `e2e` is the same metric through
the Python/C-ABI calls with the inputs copied from pinned host memory and
logprob/entropy copied back inside the timed region (dlogits stays on the
device), `e2e_dlogits_to_host` the same with the dlogits copied back to
pinned host memory as well; `roofline` is the dominant kernel's algorithmic
bytes per launch over its CUDA-event duration against the measured HBM copy
bandwidth; `cpu_baseline` times the float64 oracle on the host cores over a
bounded sample of the same workload.

`--impl reference` times the oracle alone (the reference arm): each step is a
bounded sample of the same workload on the host cores.

Multi-GPU (torchrun): tokens are independent rows, so each rank processes its
own batch with no data-path collective (weak scaling); only the timing uses a
barrier and a MAX reduction.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s and HBM GB/s (% of roofline) for logprob+entropy+bwd at V=151936"
V = 151936
MIN_REGION_S = 1.0  # each timed region lasts at least this long


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--tokens", type=int, default=8192, help="rows per rank (profiling: smaller)")
    p.add_argument("--cpu-rows", type=int, default=256, help="oracle sample rows")
    p.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    p.add_argument("--no-lmhead", action="store_true", help="skip the fused lm_head variant")
    p.add_argument("--no-rows", action="store_true",
                   help="skip the per-row timings of the other configurations")
    p.add_argument("--lmhead-tokens", type=int, default=16384,
                   help="tokens of the lm_head variant (profiling: smaller)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own batch of the workload (independent rows)."""
    return base + 1000 * rank


def max_over_ranks(x: float, device=None) -> float:
    """The slowest rank's value (MAX all-reduce); identity on one process."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, steps: int, world: int, ms: float) -> float:
    """Units processed by all ranks per second, timed by the slowest rank."""
    return world * units_per_rank * steps / (ms / 1e3)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.idx = gpu_index
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        t0, t1 = self.window or (0, 1e30)
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        if not inside:  # timed region shorter than the sampling period: nearest samples
            mid = (t0 + t1) / 2
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in inside:
            f = [x.strip() for x in line.split(",")]
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside)}


def oracle_sample(rows: int, seed: int = 2):
    """A bounded sample of the workload drawn on the host (same law)."""
    import torch
    from vocab_wide_token_gb300 import inputs

    d = inputs.fwdbwd_workload(seed, "cpu", T=rows)
    z = d["logits"].contiguous().view(torch.int16).numpy().view("uint16")
    return z, d["labels"].numpy(), d["weights"].double().numpy()


def time_oracle(z, y, w):
    import oracle

    t0 = time.perf_counter()
    oracle.forward(z, y, -100)
    oracle.backward(z, y, w, -100)
    return time.perf_counter() - t0, oracle.threads()


def arm_config(T: int, world: int) -> dict:
    """The workload both arms report (the reference arm times bounded samples of it)."""
    gb = T * V * 2 / 1e9
    return {"workload": f"fwdbwd: T={T} rows per GPU x V={V} bf16 logits N(0,2^2), "
                        "sampled labels, weights N(0,1) x mask(20% zero), bf16 dlogits; "
                        "step = pstat_forward_backward (one pass over the logits)",
            "global_batch": T * world, "seq_len": None, "parallelism": f"dp{world}",
            "l2": f"inputs larger than L2 ({gb:.2f} GB logits per rank)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    rows = args.cpu_rows
    z, y, w = oracle_sample(rows)
    for _ in range(args.warmup):
        time_oracle(z, y, w)
    t = 0.0
    cores = oracle.threads()
    for _ in range(args.steps):
        dt, cores = time_oracle(z, y, w)
        t += dt
    tok_s = rows * args.steps / t
    sample = (f"{rows} rows of the fwdbwd workload (V={V}, bf16) per step, forward+backward, "
              f"float64 on the host cores; tokens/s of the sample stand for the {args.tokens}-row "
              "workload, whose rows are independent")
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": arm_config(args.tokens, world),
        "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def traffic_record(kernel: str):
    """DRAM bytes per launch that ncu recorded for `kernel` (profiles/
    ncu_traffic.json), scaled later to this run's rows; None once any source
    file the record lists has changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
        for src, sha in rec["sources"].items():
            with open(os.path.join(ROOT, src), "rb") as fh:
                if hashlib.sha256(fh.read()).hexdigest() != sha:
                    return None, None
        return float(rec["dram_bytes_per_launch"]), float(rec["rows"])
    except Exception:
        return None, None


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from vocab_wide_token_gb300 import inputs, pstat

    T = args.tokens
    d = inputs.fwdbwd_workload(rank_seed(2, rank), dev, T=T)
    z, y, w = d["logits"], d["labels"], d["weights"]
    err = pstat.new_error_flag(dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev)
    ent = torch.empty(T, dtype=torch.float32, device=dev)
    rs = torch.empty(T, 2, dtype=torch.float32, device=dev)
    g = torch.empty(T, V, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(pstat.workspace_size(T, V, torch.bfloat16), dtype=torch.uint8, device=dev)
    active_rows = int(((w != 0) & (y != -100)).sum().item())

    def two_call():
        pstat.forward(z, y, -100, None, out=(lp, ent, rs), workspace=ws, dev_error=err)
        pstat.backward(z, y, w, rs, -100, out=g, dev_error=err)

    def fused():
        pstat.forward_backward(z, y, w, -100, out=(lp, ent, rs), dlogits=g, dev_error=err)

    for _ in range(max(args.warmup, 3)):
        two_call()
        fused()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # ---- timed regions: device-resident inputs --------------------------------
    # Each timed region is R back-to-back blocks of K steps, R chosen by an
    # untimed pilot block so that a region lasts at least MIN_REGION_S (the
    # clock sampler then holds at least ~10 samples of it).  (a) the two
    # calls, with events around each; (b) the fused single pass.
    stream = torch.cuda.current_stream(dev)
    K = args.steps
    pa = torch.cuda.Event(enable_timing=True)
    pb = torch.cuda.Event(enable_timing=True)
    barrier()
    pa.record(stream)
    for _ in range(K):
        fused()
    pb.record(stream)
    barrier()
    R = max(1, math.ceil(MIN_REGION_S * 1e3 / max(pa.elapsed_time(pb), 1e-3)))
    R = int(max_over_ranks(R, dev))
    N = R * K
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(N)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    t_wall0 = time.time()
    start_a = torch.cuda.Event(enable_timing=True)
    end_a = torch.cuda.Event(enable_timing=True)
    start_a.record(stream)
    for k in range(N):
        ev[k][0].record(stream)
        pstat.forward(z, y, -100, None, out=(lp, ent, rs), workspace=ws, dev_error=err)
        ev[k][1].record(stream)
        pstat.backward(z, y, w, rs, -100, out=g, dev_error=err)
        ev[k][2].record(stream)
    end_a.record(stream)
    barrier()
    evb = [torch.cuda.Event(enable_timing=True) for _ in range(N + 1)]
    start_b = torch.cuda.Event(enable_timing=True)
    end_b = torch.cuda.Event(enable_timing=True)
    start_b.record(stream)
    for k in range(N):
        evb[k].record(stream)
        pstat.forward_backward(z, y, w, -100, out=(lp, ent, rs), dlogits=g, dev_error=err)
    evb[N].record(stream)
    end_b.record(stream)
    barrier()
    t_wall1 = time.time()
    clocks.window = (t_wall0, t_wall1)
    time.sleep(0.25)
    clocks.stop()
    ms_a = max_over_ranks(start_a.elapsed_time(end_a), dev)
    ms_b = max_over_ranks(start_b.elapsed_time(end_b), dev)
    fwd_ms = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(N)) / N
    bwd_ms = sum(ev[k][1].elapsed_time(ev[k][2]) for k in range(N)) / N
    fused_ms = sum(evb[k].elapsed_time(evb[k + 1]) for k in range(N)) / N
    assert err.item() == 0, f"device error bits {err.item()}"

    # Algorithmic bytes.  Two calls: the forward reads every row; the backward
    # reads the rows whose gradient is not identically zero (ignored rows and
    # zero weights are written as +0.0 without reading) and writes every row.
    # Fused: every row is read once from HBM and written once.
    fwd_bytes = T * (2 * V + 8 + 16)                    # logits, label, logprob/entropy/rowstats
    bwd_bytes = active_rows * 2 * V + T * (2 * V + 20)  # reads of active rows, writes, row data
    fused_bytes = T * (2 * V + 2 * V + 8 + 4 + 16)
    hbm, tflops, tflops_sus, peak_kind = measured_peaks()
    bwd_gbs = bwd_bytes / (bwd_ms / 1e3) / 1e9
    fwd_gbs = fwd_bytes / (fwd_ms / 1e3) / 1e9
    fused_gbs = fused_bytes / (fused_ms / 1e3) / 1e9
    traffic, traffic_rows = traffic_record("fwdbwd_kernel")
    if traffic is not None and traffic_rows:
        traffic = traffic * T / traffic_rows
    roof = {"bound": "hbm", "kernel": "fwdbwd_kernel", "achieved": fused_gbs, "peak": hbm,
            "unit": "GB/s", "frac": fused_gbs / hbm, "peak_kind": peak_kind, "traffic": traffic,
            "algorithmic_bytes_per_launch": fused_bytes}
    ms_step = ms_b / N
    tok_s = whole_job_rate(T, N, world, ms_b)

    line = {
        "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "timed_blocks": R, "timed_steps": N,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": arm_config(T, world),
        "gbs": fused_gbs,
        "roofline": roof,
        "gpu_launches": N,
        "two_call": {"step": "pstat_forward + pstat_backward",
                     "value": whole_job_rate(T, N, world, ms_a), "ms_per_step": ms_a / N,
                     "gbs": (fwd_bytes + bwd_bytes) / (ms_a / N / 1e3) / 1e9,
                     "forward_ms": fwd_ms, "forward_gbs": fwd_gbs, "forward_frac": fwd_gbs / hbm,
                     "backward_ms": bwd_ms, "backward_gbs": bwd_gbs,
                     "backward_frac": bwd_gbs / hbm, "active_rows": active_rows,
                     "gpu_launches": 2 * N},
        "clocks": clocks.summary(),
    }

    # ---- e2e: host buffers through the public API ---------------------------
    # Inputs come from pinned host memory every step.  `e2e`: logprob and
    # entropy are read back; dlogits stays in device memory, where the
    # trainer's next backward step consumes it.  `e2e_dlogits_to_host`: the
    # bf16 dlogits are copied back to pinned host memory as well, block by
    # block as the kernel finishes each.
    if not args.no_e2e:
        zh = z.cpu().pin_memory()
        yh = y.cpu().pin_memory()
        wh = w.cpu().pin_memory()
        outh = torch.empty(2, T, dtype=torch.float32).pin_memory()
        gh = torch.empty(T, V, dtype=torch.bfloat16).pin_memory()
        Ke = min(K, 20)
        h2d = zh.numel() * 2 + yh.numel() * 8 + wh.numel() * 4

        def e2e_step(dlogits_host=None):
            # host logits, labels, weights -> device results, the row blocks'
            # copies overlapping the kernel on the previous block
            pstat.forward_backward_from_host(zh, yh, wh, -100, device=dev, out=(lp, ent, rs),
                                             dlogits=g, dev_error=err,
                                             dlogits_host=dlogits_host)
            outh[0].copy_(lp, non_blocking=True)
            outh[1].copy_(ent, non_blocking=True)

        def timed_e2e(dlogits_host):
            for _ in range(2):
                e2e_step(dlogits_host)
            barrier()
            s2 = torch.cuda.Event(enable_timing=True)
            e2 = torch.cuda.Event(enable_timing=True)
            s2.record(stream)
            for _ in range(Ke):
                e2e_step(dlogits_host)
            e2.record(stream)
            barrier()
            return max_over_ranks(s2.elapsed_time(e2), dev)

        ms2 = timed_e2e(None)
        line["e2e"] = {"value": whole_job_rate(T, Ke, world, ms2), "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": outh.numel() * 4,
                       "steps": Ke, "dlogits": "stays in device memory"}
        ms3 = timed_e2e(gh)
        d2h = outh.numel() * 4 + gh.numel() * 2
        line["e2e_dlogits_to_host"] = {
            "value": whole_job_rate(T, Ke, world, ms3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": Ke, "dlogits": "copied to pinned host memory inside the timed region"}
        # The host link in this run: pinned copies of the same buffers in, out
        # and both ways at once; the e2e forms are bounded by the bytes each
        # step moves over it.
        link = host_link(zh, gh, z, g, dev)
        t_in = h2d / (link["h2d_gbs"] * 1e9)
        t_both = max(t_in, d2h / (link["d2h_gbs"] * 1e9),
                     (h2d + d2h) / (link["both_gbs"] * 1e9))
        line["e2e"]["link_bound_frac"] = t_in / (ms2 / Ke / 1e3)
        line["e2e_dlogits_to_host"]["link_bound_frac"] = t_both / (ms3 / Ke / 1e3)
        line["e2e"]["link"] = link
        del zh, gh

    # ---- fused lm_head variant (rank 0 reports) ------------------------------
    if not args.no_lmhead:
        line["lmhead"] = bench_lmhead(pstat, dev, tflops, tflops_sus, peak_kind,
                                      T=args.lmhead_tokens)

    # ---- the other rows and configurations, each timed alone ------------------
    if not args.no_rows:
        line["rows"] = bench_rows(pstat, dev, hbm, peak_kind, z, y, rs)

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1 only) ------
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        rows = args.cpu_rows
        zs, ys, ws_ = oracle_sample(rows)
        dt, cores = time_oracle(zs, ys, ws_)
        line["cpu_baseline"] = {"value": rows / dt, "unit": "tokens/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"{rows} rows of the same workload law (V={V}, bf16), "
                                          "float64 forward+backward, one pass"}
        line["cpu_baseline"]["parity"] = sample_parity(pstat, oracle, zs, ys, ws_, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def host_link(zh, gh, z, g, dev, reps=3):
    """GB/s of pinned host <-> device copies of these buffers: host to device,
    device to host, and both at once on two streams."""
    import torch

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    s1 = torch.cuda.Stream(dev)
    s2 = torch.cuda.Stream(dev)

    def both():
        with torch.cuda.stream(s1):
            z.copy_(zh, non_blocking=True)
        with torch.cuda.stream(s2):
            gh.copy_(g, non_blocking=True)

    nz, ng = zh.numel() * zh.element_size(), gh.numel() * gh.element_size()
    return {"h2d_gbs": nz / timed(lambda: z.copy_(zh, non_blocking=True)) / 1e9,
            "d2h_gbs": ng / timed(lambda: gh.copy_(g, non_blocking=True)) / 1e9,
            "both_gbs": (nz + ng) / timed(both) / 1e9}


def sample_parity(pstat, oracle, zs, ys, ws_, dev):
    """The headline step on the oracle's sample, against the oracle: the
    largest logprob and entropy errors, the largest dlogits error beyond the
    bf16 rule's allowance (<= 0 passes), and a bitwise batch-invariance check
    of a few rows computed alone against the same rows in the sample batch."""
    import numpy as np
    import torch

    z = torch.from_numpy(zs.view("int16")).view(torch.bfloat16).to(dev)
    y = torch.from_numpy(ys).to(dev)
    w = torch.from_numpy(ws_).float().to(dev)
    lp, ent, rs, g = pstat.forward_backward(z, y, w, -100)
    probes = [0, 1, z.shape[0] // 2, z.shape[0] - 1]
    alone = [pstat.forward_backward(z[r:r + 1], y[r:r + 1], w[r:r + 1], -100) for r in probes]
    torch.cuda.synchronize()
    ref = oracle.forward(zs, ys, -100)
    gref = oracle.backward(zs, ys, ws_, -100)
    a = g.double().cpu().numpy()
    br = torch.from_numpy(gref).to(torch.bfloat16).double().numpy()
    ax = np.abs(gref)
    e = np.floor(np.log2(np.maximum(ax, 2.0**-126)))
    allow = np.maximum(1e-3 * ax, np.maximum(2.0 ** (e - 7), 2.0**-133))
    bits = lambda t: t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)
    invariant = all(torch.equal(bits(o[0]), bits(lp[r:r + 1])) and
                    torch.equal(bits(o[1]), bits(ent[r:r + 1])) and
                    torch.equal(bits(o[3]), bits(g[r:r + 1]))
                    for r, o in zip(probes, alone))
    return {"rows": int(z.shape[0]),
            "max_abs_logprob_err": float(np.max(np.abs(lp.double().cpu().numpy() - ref["logprob"]))),
            "max_abs_entropy_err": float(np.max(np.abs(ent.double().cpu().numpy() - ref["entropy"]))),
            "dlogits_max_excess_over_bf16_rule": float(np.max(np.abs(a - br) - allow)),
            "batch_invariant_rows": len(probes), "batch_invariant": bool(invariant)}


def bench_rows(pstat, dev, hbm, peak_kind, z8, y8, rs8, steps=50):
    """The rows and configurations besides the headline step, each timed alone
    with CUDA events on the launching stream (device-resident inputs larger
    than L2, mean over `steps` launches after 3 warm-up launches).  Bytes are
    algorithmic; fractions are against the measured HBM copy bandwidth.
      forward_T4096   pstat_forward (one kernel) on the forward-only
                      configuration: T=4096, 10% of rows with one logit +15;
      uneven_{bf16,f32}  pstat_forward and pstat_forward_backward with the
                      3-shard plan (50000 / 50000 / 51936), 10% of the
                      vocabulary at -inf on 25% of rows, 5% ignored labels,
                      unit weights; dlogits in the logits' dtype;
      log_softmax     pstat_log_softmax on the headline workload from its
                      (M, ln S), bf16 out;
      policy          the loss-side epilogue on T=8192 tokens:
                      pstat_logprob_diff_metrics + pstat_clipped_surrogate."""
    import torch
    from vocab_wide_token_gb300 import inputs

    stream = torch.cuda.current_stream(dev)
    err = pstat.new_error_flag(dev)

    def timed(fn, n=steps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    def hbm_row(workload, T, ms, nbytes, launches):
        gbs = nbytes / (ms / 1e3) / 1e9
        return {"workload": workload, "ms": ms, "tokens_per_s": T / (ms / 1e3), "gbs": gbs,
                "frac": gbs / hbm, "peak_kind": peak_kind, "algorithmic_bytes": nbytes,
                "gpu_launches_per_call": launches}

    out = {}
    d = inputs.forward_workload(1, dev)
    z, y = d["logits"], d["labels"]
    T = z.shape[0]
    o = (torch.empty(T, device=dev), torch.empty(T, device=dev), torch.empty(T, 2, device=dev))
    ms = timed(lambda: pstat.forward(z, y, -100, out=o, dev_error=err))
    out["forward_T4096"] = hbm_row(f"forward only: T={T} x V={V} bf16, 10% peaked rows", T, ms,
                                   T * (2 * V + 8 + 16), 1)
    del d, z, y
    for dt, tag in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
        d = inputs.uneven_workload(3, dev, dtype=dt)
        z, y, b = d["logits"], d["labels"], d["shard_bounds"]
        T, es = z.shape[0], z.element_size()
        o = (torch.empty(T, device=dev), torch.empty(T, device=dev),
             torch.empty(T, 2, device=dev))
        g = torch.empty_like(z)
        ms_f = timed(lambda: pstat.forward(z, y, -100, b, out=o, dev_error=err))
        ms_fb = timed(lambda: pstat.forward_backward(z, y, None, -100, b, out=o, dlogits=g,
                                                     dev_error=err))
        wl = f"uneven shards {b}: T={T} x V={V} {tag}, masked vocabulary, 5% ignored"
        out[f"uneven_{tag}_forward"] = hbm_row(wl, T, ms_f, T * (es * V + 8 + 16), 1)
        out[f"uneven_{tag}_forward_backward"] = hbm_row(wl, T, ms_fb,
                                                        T * (2 * es * V + 8 + 4 + 16), 1)
        del d, z, y, g
    T = z8.shape[0]
    ls = torch.empty_like(z8)
    ms = timed(lambda: pstat.log_softmax(z8, rs8, out=ls, dev_error=err))
    out["log_softmax"] = hbm_row(f"T={T} x V={V} bf16 from (M, ln S), bf16 out", T, ms,
                                 T * (2 * V + 2 * V + 8), 1)
    del ls
    lp = torch.randn(T, device=dev)
    lp_old = lp + 1e-3 * torch.randn(T, device=dev)
    adv = torch.randn(T, device=dev)

    def policy():
        pstat.logprob_diff_metrics(lp, lp_old, y8)
        pstat.clipped_surrogate(lp, lp_old, adv, y8)

    ms = timed(policy)
    out["policy"] = {"workload": f"T={T} tokens: logprob_diff_metrics + clipped_surrogate",
                     "us": ms * 1e3, "gpu_launches_per_call": 2}
    torch.cuda.synchronize()
    assert err.item() == 0, f"device error bits {err.item()}"
    return out


def bench_lmhead(pstat, dev, tflops, tflops_sus, peak_kind, T=16384, steps=3, warmup=1):
    """Fused lm_head on hidden [T, 4096] x W [151936, 4096] bf16: the forward
    (tcgen05 GEMM with the statistics epilogue + combine; 2 T V d flops) and
    the backward (one fp16 conversion of W and w hidden, then per 32768-column
    chunk: recompute GEMM -> fp16 gradient tile, one launch of the dhidden and
    dW GEMMs; 6 T V d flops)."""
    import torch
    from vocab_wide_token_gb300 import inputs

    try:
        pstat.lmhead_workspace_size(16, V, 4096)
    except pstat.PstatError as e:
        return {"status": f"unavailable: {e}"}
    d = inputs.lmhead_workload(4, dev, T=T)
    h, W, y, w = d["hidden"], d["W"], d["labels"], d["weights"]
    T, dm = h.shape
    err = pstat.new_error_flag(dev)
    ws = torch.empty(pstat.lmhead_workspace_size(T, V, dm), dtype=torch.uint8, device=dev)
    dh = torch.zeros(T, dm, dtype=torch.float32, device=dev)
    dW = torch.zeros(V, dm, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    out = {}

    def fwd():
        out["fwd"] = pstat.lmhead_forward(h, W, y, -100, workspace=ws, dev_error=err)

    fwd_ms = timed(fwd)
    rs = out["fwd"][2]

    def bwd():
        pstat.lmhead_backward(h, W, y, w, rs, -100, dhidden=dh, dW=dW, workspace=ws,
                              dev_error=err)

    bwd_ms = timed(bwd)
    assert err.item() == 0, f"device error bits {err.item()}"
    flop_f = 2.0 * T * V * dm
    flop_b = 6.0 * T * V * dm
    af = flop_f / (fwd_ms / 1e3) / 1e12
    ab = flop_b / (bwd_ms / 1e3) / 1e12
    n_chunks = (V + 32767) // 32768  # vocabulary columns staged per backward chunk
    return {"status": "ok", "workload": f"hidden [{T}, {dm}] x W [{V}, {dm}] bf16, sampled labels",
            "forward_ms": fwd_ms, "forward_tokens_per_s": T / (fwd_ms / 1e3),
            "backward_ms": bwd_ms, "backward_tokens_per_s": T / (bwd_ms / 1e3),
            "roofline": {"bound": "tensor", "kernel": "tc_gemm_kernel<StatsEpi>",
                         "achieved": af, "peak": tflops, "unit": "TFLOP/s",
                         "frac": af / tflops, "peak_kind": f"{peak_kind} burst",
                         "traffic": None},
            "backward_roofline": {"bound": "tensor", "achieved": ab, "peak": tflops_sus,
                                  "unit": "TFLOP/s", "frac": ab / tflops_sus,
                                  "peak_kind": f"{peak_kind} sustained",
                                  "algorithmic_flop": flop_b},
            "gpu_launches_per_forward": 2, "gpu_launches_per_backward": 1 + 2 * n_chunks}


if __name__ == "__main__":
    main()
