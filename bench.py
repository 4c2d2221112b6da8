#!/usr/bin/env python
"""Throughput of exact ring attention on GB300; prints one JSON line.

Default workload: bf16, causal, B=1, H=32, S=32768, D=128, P=8 virtual ranks
in zig-zag order (the long-context headline shape). One step = one call of
``ring_attn_fwd_ex`` = all P ring steps of every virtual rank, fused in one
kernel launch. The metric is algorithmic TFLOP/s (2*B*H*S^2*D for causal).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the method needs no exchange on one device: "replicas only");
``value`` is the FLOP of all ranks over the slowest rank's time.
``--impl reference`` times the float64 CPU oracle on a bounded row sample of
the same workload (rank 0 only).
"""

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring-attn fwd TFLOP/s, bf16 S=32K causal, 1 GB300; % of dense BF16 peak"


def _fwd_metric(w):
    """The headline metric for the headline workload; the other forward
    workloads name themselves."""
    from sequence_exact_attention_gb300.workloads import HEADLINE
    if w.name == HEADLINE:
        return METRIC
    return f"ring-attn fwd TFLOP/s, {w.name}, 1 GB300"


UNIT = "TFLOP/s"
VARLEN_METRIC = "ring-attn fwd TFLOP/s, packed variable-length batch, 1 GB300"
ULYSSES_METRIC = "ring-attn fwd TFLOP/s, Ulysses sequence-parallel layout, 1 GB300"
MERGE_METRIC = "LSE merge GB/s (algorithmic bytes)"

# ncu DRAM bytes (read + write) of one launch of the timed kernel, per
# workload; an entry holds only while the kernel's sources have the digest
# stored with it (see _kernel_digest). The forward's bytes were captured at
# digest 419f638ff48490a0; the sources of the digest below differ from those
# only in the indentation of eight pragmas and compile to the same sm_103a
# cubin.
TRAFFIC = {
    "attn_tc": {"sha256_16": "474c78bee5b5ebb2", "bytes_per_launch": {
        "bf16_s32k_causal_zigzag": 846791168 + 255732992,
        "bf16_s16k_d64": 402796032 + 119514368,
        "bf16_s128k_gqa_causal": 2724986368 + 1058387712,
        "bf16_s4k_causal": 105313536 + 10988800,
        "bf16_s32760_uneven_causal_zigzag": 845622016 + 255803648,
        "bf16_varlen_32k_causal_zigzag": 828308736 + 255260672,
        "bf16_ulysses_s16k_b2_causal": 805500160 + 253177088,
    }},
    # the merge was captured on S = 8192 (1.15 GiB on the device) and scaled by
    # 65536 / 8192 = 8: a streaming kernel whose bytes grow with the rows
    "merge": {"sha256_16": "6fac89657b942f3c", "bytes_per_launch": {
        "merge_p8_s64k": 8 * (1082154240 + 112507904),
    }},
}
KERNEL_SOURCES = {
    "attn_tc": ("attn_tc.cu", "checks.cuh", "fastmath.cuh", "ring_iter.cuh", "sm100.cuh",
                "ra_internal.h", "tensor_map.cpp"),
    "merge": ("merge.cu", "ra_internal.h"),
}


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                "bf16_tflops_sustained": 1700.0}, "fallback"


def _kernel_digest(kernel="attn_tc"):
    """sha256 (first 16 hex) of a kernel's sources -- its .cu file and the
    headers it includes -- with // comments and blank lines removed: any code
    change invalidates the stored traffic, a comment edit does not."""
    import re
    code = []
    for name in KERNEL_SOURCES[kernel]:
        path = os.path.join(ROOT, "sequence_exact_attention_gb300", "csrc", name)
        with open(path, encoding="utf-8") as f:
            lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in f]
        code.append("\n".join(ln for ln in lines if ln.strip()))
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


def _traffic(kernel, workload):
    """Stored DRAM bytes per launch of `kernel` on `workload`, or None when
    none was captured or the kernel's sources changed since."""
    entry = TRAFFIC[kernel]
    if entry["sha256_16"] != _kernel_digest(kernel):
        return None
    return entry["bytes_per_launch"].get(workload)


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        # under load: samples with power above the midpoint of the range
        if power:
            thr = (min(power) + max(power)) / 2
            loaded = [num(r[1]) for r in rows if num(r[3]) is not None and num(r[3]) >= thr]
        else:
            loaded = sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


def _dist_setup(n_gpus, backend="nccl"):
    """(world, rank, local rank, torch.distributed or None) from the launcher's
    environment; one process per GPU, every rank an independent replica."""
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend)
        return world, rank, local, dist
    return 1, 0, local, None


def _max_over_ranks(x, dist, device):
    """The largest value of x over all ranks (x itself without a process group)."""
    if not dist:
        return float(x)
    import torch
    t = torch.tensor([float(x)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(world, units_per_step, steps, max_ms):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (weak scaling: every rank does the same work)."""
    return world * units_per_step * steps / (max_ms / 1e3)


def _oracle_sample_rate(w, q, k, v, n_rows, seed, want=None):
    """float64 oracle on n_rows sampled query rows (all heads); returns
    (TFLOP/s by the algorithmic count of those rows, seconds, rows). With a
    list `want`, the oracle's (out rows, lse rows) are appended to it."""
    import numpy as np
    import oracle
    rows = np.sort(np.random.default_rng(seed).choice(w.S, n_rows, replace=False))
    t0 = time.perf_counter()
    res = oracle.attention_rows(q, k, v, w.causal, w.scale, rows)
    dt = time.perf_counter() - t0
    if want is not None:
        want.append(res)
    pairs = float((rows + 1).sum()) if w.causal else float(n_rows * w.S)
    flop = 4.0 * w.D * pairs * w.B * w.H_q
    return flop / dt / 1e12, dt, rows


def _parity(w, out, lse, rows, want):
    """Errors of the timed call's own output on the oracle's sampled rows
    (the CPU baseline's sample), against the workload's tolerance."""
    import numpy as np
    try:
        want_o, want_l = want
        eo = np.abs(out[:, rows].float().cpu().numpy() - want_o)
        el = np.abs(lse[:, :, rows].float().cpu().numpy() - want_l)
        tol = {"max": 2e-2, "mean": 2e-3} if w.dtype == "bf16" else {"max": 1e-4, "mean": 1e-4}
        res = {"rows": int(len(rows)), "out_max_abs_err": float(eo.max()),
               "out_mean_abs_err": float(eo.mean()), "lse_max_abs_err": float(el.max()),
               "lse_mean_abs_err": float(el.mean()), "tolerance": tol}
        res["within_tolerance"] = bool(
            res["out_max_abs_err"] <= tol["max"] and res["out_mean_abs_err"] <= tol["mean"]
            and res["lse_max_abs_err"] <= tol["max"] and res["lse_mean_abs_err"] <= tol["mean"])
        return res
    except Exception as e:       # reporting only: never stop the bench
        return {"error": repr(e)}


def _device_info(dev):
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        return {"name": p.name, "sm_count": int(p.multi_processor_count)}
    except Exception as e:       # reporting only
        return {"error": repr(e)}


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def run_reference(args, w):
    world, rank, _, _ = _dist_setup(args.gpus)
    if rank != 0:
        return 0
    from sequence_exact_attention_gb300.workloads import make_qkv
    q, k, v = make_qkv(w)
    rows_per_step = min(args.ref_rows, w.S)
    for i in range(args.warmup):
        _oracle_sample_rate(w, q, k, v, rows_per_step, seed=100 + i)
    total_flop, total_t = 0.0, 0.0
    for i in range(args.steps):
        rate, dt, rows = _oracle_sample_rate(w, q, k, v, rows_per_step, seed=1000 + i)
        total_flop += rate * dt * 1e12
        total_t += dt
    value = total_flop / total_t / 1e12
    cores = _blas_threads()
    sample = (f"{rows_per_step} random query rows x all {w.H_q} heads per step "
              f"(float64 NumPy oracle, full key range per row)")
    line = {
        "impl": "reference", "metric": _fwd_metric(w), "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_MIB = 126
FLUSH_MIB = 256


def _inputs_mib(w):
    esz = 2 if w.dtype == "bf16" else 4
    return w.B * w.S * (w.H_q + 2 * w.H_kv) * w.D * esz / 2**20


def _l2_flusher(w, dev, stream):
    """None when the workload's inputs are larger than L2; else a call that
    writes a buffer twice the size of L2 on `stream`, run between timed
    launches so that no launch finds the previous one's data in L2."""
    if _inputs_mib(w) > L2_MIB:
        return None
    import torch
    buf = torch.empty(FLUSH_MIB << 20, dtype=torch.uint8, device=dev)

    def flush():
        with torch.cuda.stream(stream):
            buf.zero_()
    return flush


def _config(w):
    in_mib = _inputs_mib(w)
    l2 = (f"inputs larger than L2 (q+k+v {in_mib:.0f} MiB vs {L2_MIB} MiB L2)" if in_mib > L2_MIB
          else f"inputs fit in L2 (q+k+v {in_mib:.1f} MiB): L2 flushed before every timed "
               f"launch ({FLUSH_MIB} MiB write, outside the launch's events); value from "
               f"the launches' own events")
    return {"workload": w.name, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv, "S": w.S,
            "D": w.D, "P": w.P, "causal": w.causal, "order": w.order,
            "input_dist": f"N(0,{w.std}^2) {w.dtype}", "l2": l2,
            "parallelism": "replicas"}


def _e2e(args, w, q, k, v, qd, kd, vd, out, lse, step, dev, stream, dist, world):
    """Same metric through the public API with pinned host buffers. Every step
    copies its q, k, v host->device, runs the call and copies out and lse back.
    Steps are pipelined the way a serving loop would run them: two device
    buffer sets, host->device copies on one stream, the attention call on
    another, device->host copies on a third, so step i's copies overlap the
    neighbouring steps' compute."""
    import torch
    from sequence_exact_attention_gb300 import binding
    flop = w.flop
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    sets = [(qd, kd, vd, out, lse),
            (torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd),
             torch.empty_like(out), torch.empty_like(lse))]
    host_out = [(torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                 torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_cmp = stream
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def run(n):
        for i in range(n):
            bsel = i % 2
            qb, kb, vb, ob, lb = sets[bsel]
            if used[bsel]:
                s_in.wait_event(ev_cmp[bsel])      # inputs of step i-2 consumed
            with torch.cuda.stream(s_in):
                qb.copy_(qh, non_blocking=True)
                kb.copy_(kh, non_blocking=True)
                vb.copy_(vh, non_blocking=True)
                ev_in[bsel].record(s_in)
            s_cmp.wait_event(ev_in[bsel])
            if used[bsel]:
                s_cmp.wait_event(ev_out[bsel])     # outputs of step i-2 read back
            binding.ring_attn_fwd(qb, kb, vb, w.P, w.causal, w.scale, w.order, out=ob,
                                  lse=lb, stream=s_cmp)
            ev_cmp[bsel].record(s_cmp)
            s_out.wait_event(ev_cmp[bsel])
            with torch.cuda.stream(s_out):
                host_out[bsel][0].copy_(ob, non_blocking=True)
                host_out[bsel][1].copy_(lb, non_blocking=True)
                ev_out[bsel].record(s_out)
            used[bsel] = True

    run(2)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    run(args.steps)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_cmp)
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = _max_over_ranks(e2e_ms, dist, dev)
    e2e_val = _job_rate(world, flop, args.steps, e2e_ms) / 1e12
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    return {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "pipelined": "2 buffer sets; h2d, compute, d2h streams"}


def run_ours(args, w):
    import torch
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import make_qkv

    world, rank, local, dist = _dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    try:
        binding.load()
    except RuntimeError:
        from sequence_exact_attention_gb300 import build
        build.build()
        binding.load()

    q, k, v = make_qkv(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty(w.B, w.S, w.H_q, w.D, dtype=qd.dtype, device=dev)
    lse = torch.empty(w.B, w.H_q, w.S, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.ring_attn_fwd(qd, kd, vd, w.P, w.causal, w.scale, w.order, out=out,
                              lse=lse, dev_status=status, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError("device-side wait expired during warm-up")

    # ---- device-timed region: inputs resident in HBM
    clocks = ClockSampler(local)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if dist:
        dist.barrier()
    flush = _l2_flusher(w, dev, stream)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if flush is not None:
        # the flushes between launches are not the workload's time
        total_ms = sum(launch_ms)
    if int(status.item()) != 0:
        raise RuntimeError("device-side wait expired in the timed region")
    total_ms = _max_over_ranks(total_ms, dist, dev)
    flop = w.flop
    value = _job_rate(world, flop, args.steps, total_ms) / 1e12
    kernel_ms = statistics.mean(launch_ms)

    # ---- end to end through the public API, host buffers, copies timed
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(args, w, q, k, v, qd, kd, vd, out, lse, step, dev, stream, dist, world)

    if rank != 0:
        return 0

    peaks, peak_src = _peaks()
    achieved = flop / (kernel_ms / 1e3) / 1e12
    if w.dtype == "bf16":
        bound, peak = "tensor", float(peaks.get("bf16_tflops"))
        peak_note = f"{peak_src} bf16 dense (burst)"
        kname = f"attn_tc_kernel<{w.D},false,false>"
        traffic = _traffic("attn_tc", w.name)
    else:
        # exact fp32 FMA path: 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz
        bound, peak = "alu", 152 * 128 * 2 * 2.07e9 / 1e12
        peak_note = "fp32 FMA: SM count x lanes x 2 x max SM clock"
        kname = f"attn_simt_kernel<{w.D}>"
        traffic = None

    cpu, parity = None, None
    if world == 1 and not args.no_cpu_baseline:
        n_rows = min(args.cpu_rows, w.S)
        want = []
        rate, dt, rows = _oracle_sample_rate(w, q, k, v, n_rows, seed=7, want=want)
        cpu = {"value": rate, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
               "sample": f"{n_rows} random query rows x all {w.H_q} heads of the same "
                         f"workload, float64 NumPy oracle, {dt:.1f} s"}
        parity = _parity(w, out, lse, rows, want[0])

    line = {
        "metric": _fwd_metric(w), "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": _config(w),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_note, "kernel": kname, "kernel_ms": kernel_ms,
                     "kernel_ms_median": statistics.median(launch_ms),
                     "kernel_ms_min": min(launch_ms),
                     # one exponential per allowed (query, key) pair
                     "exp2_per_s": flop / (4.0 * w.D) / (kernel_ms / 1e3),
                     "frac_of_sustained_peak": (achieved / float(peaks["bf16_tflops_sustained"])
                                                if w.dtype == "bf16" else None)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clk,
        "gpu_launches": args.steps,
        "parity": parity,
        "device": _device_info(dev),
    }
    from sequence_exact_attention_gb300.workloads import HEADLINE
    if world == 1 and w.name == HEADLINE and not getattr(args, "no_configs", False):
        del qd, kd, vd
        torch.cuda.empty_cache()
        line["configs"] = _configs_sweep(dev, stream)
    print(json.dumps(line), flush=True)
    return 0


# Every other workload, measured in the same run as the headline
# (reported under "configs" of the headline line): kernel time by CUDA events,
# the roofline fraction, the stored DRAM traffic, clocks and parity against
# the float64 oracle on sampled rows.
CONFIG_SWEEP = ("fp32_s256", "bf16_s4k_causal", "bf16_s128k_gqa_causal", "merge_p8_s64k",
                "bf16_s16k_d64", "bf16_s32k_causal_zigzag_bwd", "bf16_varlen_32k_causal_zigzag",
                "bf16_ulysses_s16k_b2_causal", "bf16_s32760_uneven_causal_zigzag")


def _event_times(fn, warm, timed, stream, dev, between=None):
    """CUDA-event milliseconds of `timed` calls of fn after `warm` calls; with
    `between`, that call runs before every timed call, outside its events."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(timed)]
    for a, b in ev:
        if between is not None:
            between()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) for a, b in ev]


def _tol_check(errs, tol):
    """errs: dict of (max, mean) pairs; adds within_tolerance."""
    out = {k: {"max_abs_err": float(v[0]), "mean_abs_err": float(v[1])} for k, v in errs.items()}
    out["tolerance"] = tol
    out["within_tolerance"] = bool(all(v[0] <= tol["max"] and v[1] <= tol["mean"]
                                       for v in errs.values()))
    return out


def _sweep_fwd(w, dev, stream, peaks):
    import numpy as np
    import torch
    import oracle
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import make_qkv
    q, k, v = make_qkv(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty(w.B, w.S, w.H_q, w.D, dtype=qd.dtype, device=dev)
    lse = torch.empty(w.B, w.H_q, w.S, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        binding.ring_attn_fwd(qd, kd, vd, w.P, w.causal, w.scale, w.order, out=out, lse=lse,
                              dev_status=status, stream=stream)

    clocks = ClockSampler(dev.index)
    clocks.start()
    ms = _event_times(step, 2, 3 if w.flop > 5e13 else 10, stream, dev,
                      between=_l2_flusher(w, dev, stream))
    clk = clocks.stop()
    kernel_ms = statistics.mean(ms)
    achieved = w.flop / (kernel_ms / 1e3) / 1e12
    if w.dtype == "bf16":
        bound, peak, kname = "tensor", float(peaks["bf16_tflops"]), f"attn_tc_kernel<{w.D},false,false>"
        traffic = _traffic("attn_tc", w.name)
        tol = {"max": 2e-2, "mean": 2e-3}
    else:
        bound, peak, kname = "alu", 152 * 128 * 2 * 2.07e9 / 1e12, f"attn_simt_kernel<{w.D}>"
        traffic = None
        tol = {"max": 1e-4, "mean": 1e-4}
    # parity: every row when the oracle is quick, else seeded sampled rows
    n_rows = w.S if w.S <= 4096 else (16 if w.S > 65536 else 64)
    rows = np.sort(np.random.default_rng(11).choice(w.S, n_rows, replace=False))
    want_o, want_l = oracle.attention_rows(q, k, v, w.causal, w.scale, rows)
    eo = np.abs(out[:, rows].double().cpu().numpy() - want_o)
    el = np.abs(lse[:, :, rows].double().cpu().numpy() - want_l)
    parity = _tol_check({"out": (eo.max(), eo.mean()), "lse": (el.max(), el.mean())}, tol)
    parity["rows"] = int(n_rows)
    parity["status_word"] = int(status.item())
    return {"workload": w.name, "config": _config(w), "metric": _fwd_metric(w),
            "value": achieved, "unit": UNIT, "kernel": kname, "kernel_ms": kernel_ms,
            "kernel_ms_min": min(ms), "launches": len(ms),
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": traffic},
            "clocks": clk, "parity": parity}


def _layout_entry(w, cfg, metric, kname, ms, clk, parity, peaks):
    kernel_ms = statistics.mean(ms)
    achieved = w.flop / (kernel_ms / 1e3) / 1e12
    peak = float(peaks["bf16_tflops"])
    return {"workload": w.name, "config": cfg, "metric": metric, "value": achieved, "unit": UNIT,
            "kernel": kname, "kernel_ms": kernel_ms, "kernel_ms_min": min(ms),
            "launches": len(ms),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": _traffic("attn_tc", w.name)},
            "clocks": clk, "parity": parity}


def _sweep_varlen(w, dev, stream, peaks):
    """Packed batch: CUDA-event time of ring_attn_fwd_varlen, parity on 8
    sampled rows of every sequence against the oracle on that sequence alone."""
    import numpy as np
    import torch
    import oracle
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import make_varlen
    q, k, v, cu = make_varlen(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    cud = torch.tensor(cu, dtype=torch.int32, device=dev)
    out, lse = torch.empty_like(qd), torch.empty(w.H_q, w.total, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        binding.ring_attn_fwd_varlen(qd, kd, vd, cud, w.max_seqlen, w.P, w.causal, w.scale,
                                     w.order, out=out, lse=lse, dev_status=status, stream=stream)

    clocks = ClockSampler(dev.index)
    clocks.start()
    ms = _event_times(step, 2, 10, stream, dev)
    clk = clocks.stop()
    rng = np.random.default_rng(13)
    eo_max = eo_sum = el_max = el_sum = 0.0
    n_o = n_l = 0
    out_h, lse_h = out.double().cpu().numpy(), lse.double().cpu().numpy()
    for i, n in enumerate(w.lengths):
        lo = cu[i]
        rows = np.sort(rng.choice(n, min(8, n), replace=False))
        want_o, want_l = oracle.attention_rows(q[None, lo:lo + n], k[None, lo:lo + n],
                                               v[None, lo:lo + n], w.causal, w.scale, rows)
        eo = np.abs(out_h[lo + rows] - want_o[0])
        el = np.abs(lse_h[:, lo + rows] - want_l[0])
        eo_max, el_max = max(eo_max, eo.max()), max(el_max, el.max())
        eo_sum, el_sum = eo_sum + eo.sum(), el_sum + el.sum()
        n_o, n_l = n_o + eo.size, n_l + el.size
    parity = _tol_check({"out": (eo_max, eo_sum / n_o), "lse": (el_max, el_sum / n_l)},
                        {"max": 2e-2, "mean": 2e-3})
    parity["rows"] = "8 sampled rows of every sequence"
    parity["status_word"] = int(status.item())
    return _layout_entry(w, _varlen_config(w), VARLEN_METRIC, "attn_tc_kernel<128,false,true>",
                         ms, clk, parity, peaks)


def _sweep_ulysses(w, dev, stream, peaks):
    """Sequence-parallel layout: CUDA-event time of ring_attn_fwd_ulysses,
    parity on sampled positions against full attention over each sequence."""
    import numpy as np
    import torch
    import oracle
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import make_sharded_qkv
    q, k, v = make_sharded_qkv(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    P, B, C = q.shape[0], q.shape[1], q.shape[2]
    out = torch.empty_like(qd)
    lse = torch.empty(P, B, w.H_q, C, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        binding.ring_attn_fwd_ulysses(qd, kd, vd, w.S, w.causal, w.scale, out=out, lse=lse,
                                      dev_status=status, stream=stream)

    clocks = ClockSampler(dev.index)
    clocks.start()
    ms = _event_times(step, 2, 10, stream, dev)
    clk = clocks.stop()

    def seq(x):      # [P, B, C, H, D] -> [B, S, H, D]: shard p holds positions [pC, pC + C)
        return x.permute(1, 0, 2, 3, 4).reshape(B, P * C, x.shape[3], x.shape[4])[:, :w.S]

    rows = np.sort(np.random.default_rng(14).choice(w.S, 32, replace=False))
    want_o, want_l = oracle.attention_rows(seq(q), seq(k), seq(v), w.causal, w.scale, rows)
    p_idx, c_idx = torch.from_numpy(rows // C), torch.from_numpy(rows % C)
    got_o = out.cpu()[p_idx, :, c_idx].permute(1, 0, 2, 3).double().numpy()
    got_l = lse.cpu()[p_idx, :, :, c_idx].permute(1, 2, 0).double().numpy()
    eo, el = np.abs(got_o - want_o), np.abs(got_l - want_l)
    parity = _tol_check({"out": (eo.max(), eo.mean()), "lse": (el.max(), el.mean())},
                        {"max": 2e-2, "mean": 2e-3})
    parity["rows"] = 32
    parity["status_word"] = int(status.item())
    return _layout_entry(w, _ulysses_config(w), ULYSSES_METRIC, "attn_tc_kernel<128,false,false>",
                         ms, clk, parity, peaks)


def _sweep_merge(w, dev, stream, peaks):
    import numpy as np
    import torch
    import oracle
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import make_merge_parts
    os_, ls = make_merge_parts(w)
    od = [o.to(dev) for o in os_]
    ld = [l.to(dev) for l in ls]
    out = torch.empty_like(od[0])
    lse = torch.empty_like(ld[0])

    def step():
        binding.attn_lse_merge_n(od, ld, out=out, lse=lse, stream=stream)

    clocks = ClockSampler(dev.index)
    clocks.start()
    ms = _event_times(step, 2, 5, stream, dev)     # 9.7 GB a launch: inputs far above L2
    clk = clocks.stop()
    kernel_ms = statistics.mean(ms)
    gbs = w.bytes / (kernel_ms / 1e3) / 1e9
    pos = np.sort(np.random.default_rng(12).choice(w.S, 256, replace=False))
    want_o, want_l = oracle.lse_merge_n([o[:, pos].numpy() for o in os_],
                                        [l[:, :, pos].numpy() for l in ls])
    eo = np.abs(out[:, pos].double().cpu().numpy() - want_o)
    el = np.abs(lse[:, :, pos].double().cpu().numpy() - want_l)
    parity = _tol_check({"out": (eo.max(), eo.mean()), "lse": (el.max(), el.mean())},
                        {"max": 1e-4, "mean": 1e-4})
    parity["positions"] = 256
    return {"workload": w.name, "config": _merge_config(w), "metric": MERGE_METRIC,
            "value": gbs, "unit": "GB/s", "kernel": "lse_merge_kernel",
            "kernel_ms": kernel_ms, "kernel_ms_min": min(ms), "launches": len(ms),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]),
                         "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]),
                         "traffic": _traffic("merge", w.name)},
            "clocks": clk, "parity": parity}


def _sweep_bwd(w, dev, stream, peaks):
    import numpy as np
    import torch
    from oracle.backward import backward_rows
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import bwd_flop, make_dout, make_qkv
    q, k, v = make_qkv(w)
    dout = make_dout(w)
    qd, kd, vd, dd = (t.to(dev) for t in (q, k, v, dout))
    out, lse = binding.ring_attn_fwd(qd, kd, vd, w.P, w.causal, w.scale, w.order, stream=stream)
    ws = torch.empty(binding.bwd_workspace_bytes(w.B, w.H_q, w.S, w.D, w.P, w.order),
                     dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        binding.ring_attn_bwd(qd, kd, vd, out, lse, dd, w.P, w.causal, w.scale, w.order,
                              dq=dq, dk=dk, dv=dv, workspace=ws, dev_status=status,
                              stream=stream)

    clocks = ClockSampler(dev.index)
    clocks.start()
    ms = _event_times(step, 2, 5, stream, dev)
    clk = clocks.stop()
    kernel_ms = statistics.mean(ms)
    flop = bwd_flop(w)
    achieved = flop / (kernel_ms / 1e3) / 1e12
    peak = float(peaks["bf16_tflops"])
    # parity of dq on sampled rows of a causal prefix (dq_i depends on keys
    # j <= i only), query head 0, against the float64 chain rule
    n = min(w.S, 4096)
    rows = np.sort(np.random.default_rng(13).choice(n, 32, replace=False))
    want_dq, _, _ = backward_rows(q[:, :n], k[:, :n], v[:, :n], dout[:, :n], w.causal, w.scale,
                                  0, rows, np.zeros(0, dtype=np.int64))
    got = dq[:, rows, 0].double().cpu().numpy()
    e = np.abs(got - want_dq)
    rel_max = float(e.max() / max(np.abs(want_dq).max(), 1e-2))
    rel_mean = float(e.mean() / max(np.abs(want_dq).mean(), 1e-2))
    parity = {"dq_rows": 32, "head": 0, "rel_max_err": rel_max, "rel_mean_err": rel_mean,
              "tolerance": {"rel_max": 2e-2, "rel_mean": 1e-2},
              "within_tolerance": bool(rel_max <= 2e-2 and rel_mean <= 1e-2),
              "status_word": int(status.item())}
    return {"workload": w.name, "config": _config(w), "metric": BWD_METRIC,
            "value": achieved, "unit": UNIT, "kernel": "bwd_prep + bwd_dkdv + bwd_dq",
            "kernel_ms": kernel_ms, "kernel_ms_min": min(ms), "launches": 3 * len(ms),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": None},
            "clocks": clk, "parity": parity}


def _configs_sweep(dev, stream):
    """One entry per workload of CONFIG_SWEEP; a failing entry reports its error."""
    import torch
    from sequence_exact_attention_gb300.workloads import (BWD_WORKLOADS, MERGE_WORKLOADS,
                                                          ULYSSES_WORKLOADS, VARLEN_WORKLOADS,
                                                          WORKLOADS)
    peaks, _ = _peaks()
    res = []
    for name in CONFIG_SWEEP:
        try:
            if name in MERGE_WORKLOADS:
                e = _sweep_merge(MERGE_WORKLOADS[name], dev, stream, peaks)
            elif name in VARLEN_WORKLOADS:
                e = _sweep_varlen(VARLEN_WORKLOADS[name], dev, stream, peaks)
            elif name in ULYSSES_WORKLOADS:
                e = _sweep_ulysses(ULYSSES_WORKLOADS[name], dev, stream, peaks)
            elif name in BWD_WORKLOADS:
                e = _sweep_bwd(BWD_WORKLOADS[name], dev, stream, peaks)
            else:
                e = _sweep_fwd(WORKLOADS[name], dev, stream, peaks)
        except Exception as ex:          # reporting only: the headline line still prints
            e = {"workload": name, "error": repr(ex)}
        res.append(e)
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    return res


BWD_METRIC = "ring-attn bwd TFLOP/s (2.5x forward FLOP), bf16, causal, 1 GB300"


def _bwd_pairs(w):
    return w.B * w.H_q * w.S * w.S / (2.0 if w.causal else 1.0)


def _oracle_bwd_sample_rate(w, q, k, v, dout, n):
    """float64 backward oracle on a causal prefix: positions [0, n) of query
    head 0 and its kv head (a prefix of a causal problem is itself a whole
    problem). Returns (TFLOP/s by 10*D FLOP per allowed pair, seconds)."""
    from oracle.backward import attention_backward
    hk = 0
    t0 = time.perf_counter()
    attention_backward(q[:1, :n, :1], k[:1, :n, hk:hk + 1], v[:1, :n, hk:hk + 1],
                       dout[:1, :n, :1], w.causal, w.scale)
    dt = time.perf_counter() - t0
    pairs = n * (n + 1) / 2 if w.causal else float(n * n)
    return 10.0 * w.D * pairs / dt / 1e12, dt


def run_bwd(args, w):
    """The backward pass (prep, dK/dV, dQ kernels) on its workload."""
    import torch
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import bwd_flop, make_dout, make_qkv

    world, rank, local, dist = _dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load()
    q, k, v = make_qkv(w)
    dout = make_dout(w)
    qd, kd, vd, dd = (t.to(dev) for t in (q, k, v, dout))
    stream = torch.cuda.current_stream(dev)
    out, lse = binding.ring_attn_fwd(qd, kd, vd, w.P, w.causal, w.scale, w.order, stream=stream)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(binding.bwd_workspace_bytes(w.B, w.H_q, w.S, w.D, w.P, w.order),
                     dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    phases = (("bwd_prep_kernel", binding.BWD_PREP), ("bwd_dkdv_kernel", binding.BWD_DKDV),
              ("bwd_dq_kernel", binding.BWD_DQ))

    def step(ev=None):
        for i, (_, ph) in enumerate(phases):
            if ev is not None:
                ev[i][0].record(stream)
            binding.ring_attn_bwd(qd, kd, vd, out, lse, dd, w.P, w.causal, w.scale, w.order,
                                  dq=dq, dk=dk, dv=dv, workspace=ws, dev_status=status,
                                  stream=stream, phases=ph)
            if ev is not None:
                ev[i][1].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError("device-side wait expired during warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in phases] for _ in range(args.steps)]
    flush = _l2_flusher(w, dev, stream)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush()
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError("device-side wait expired in the timed region")
    total_ms = t0.elapsed_time(t1)
    if flush is not None:
        # each step from its first launch's start to its last launch's end,
        # without the flushes between steps
        total_ms = sum(e[0][0].elapsed_time(e[-1][1]) for e in evs)
    total_ms = _max_over_ranks(total_ms, dist, dev)
    flop = bwd_flop(w)
    value = _job_rate(world, flop, args.steps, total_ms) / 1e12
    phase_ms = {name: statistics.mean(e[i][0].elapsed_time(e[i][1]) for e in evs)
                for i, (name, _) in enumerate(phases)}

    # end to end: host buffers, inputs copied in and gradients copied out every step
    e2e = None
    if not args.no_e2e:
        hosts_in = [t.pin_memory() for t in (q, k, v, dout)]
        out_h, lse_h = out.cpu().pin_memory(), lse.cpu().pin_memory()
        hosts_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]

        def e2e_step():
            for hsrc, ddst in zip(hosts_in + [out_h, lse_h], (qd, kd, vd, dd, out, lse)):
                ddst.copy_(hsrc, non_blocking=True)
            step()
            for dsrc, hdst in zip((dq, dk, dv), hosts_out):
                hdst.copy_(dsrc, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b_ = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            e2e_step()
        b_.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = a.elapsed_time(b_)
        e_ms = _max_over_ranks(e_ms, dist, dev)
        e2e = {"value": _job_rate(world, flop, args.steps, e_ms) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": sum(t.numel() * t.element_size()
                                         for t in hosts_in + [out_h, lse_h]),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hosts_out),
               "pipelined": "no: copies and kernels in order on one stream"}
    if rank != 0:
        return 0

    peaks, peak_src = _peaks()
    pairs = _bwd_pairs(w)
    dkdv_flop = 8.0 * w.D * pairs      # S^T, dP^T, dV, dK
    dq_flop = 6.0 * w.D * pairs        # S, dP, dQ
    dom = max(("bwd_dkdv_kernel", "bwd_dq_kernel"), key=lambda n: phase_ms[n])
    dom_flop = dkdv_flop if dom == "bwd_dkdv_kernel" else dq_flop
    achieved = dom_flop / (phase_ms[dom] / 1e3) / 1e12
    peak = float(peaks["bf16_tflops"])
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        n = min(args.cpu_prefix, w.S)
        rate, dt = _oracle_bwd_sample_rate(w, q, k, v, dout, n)
        cpu = {"value": rate, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
               "sample": f"causal prefix of {n} positions, query head 0, float64 NumPy "
                         f"backward oracle, {dt:.1f} s"}
    line = {
        "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": _config(w),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_src} bf16 dense (burst)", "kernel": f"{dom}<{w.D}>",
                     "kernel_ms": phase_ms[dom],
                     "algorithmic_flop": "dK/dV kernel 8*D per allowed pair (S^T, dP^T, dV, "
                                         "dK); dQ kernel 6*D (S, dP, dQ)",
                     "phase_ms": phase_ms,
                     "frac_of_sustained_peak": achieved / float(peaks["bf16_tflops_sustained"])},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clk,
        "gpu_launches": 3 * args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_bwd_reference(args, w):
    world, rank, _, _ = _dist_setup(args.gpus)
    if rank != 0:
        return 0
    from sequence_exact_attention_gb300.workloads import make_dout, make_qkv
    q, k, v = make_qkv(w)
    dout = make_dout(w)
    n = min(args.cpu_prefix, w.S)
    for _ in range(args.warmup):
        _oracle_bwd_sample_rate(w, q, k, v, dout, n)
    flops, secs = 0.0, 0.0
    for _ in range(args.steps):
        rate, dt = _oracle_bwd_sample_rate(w, q, k, v, dout, n)
        flops += rate * dt * 1e12
        secs += dt
    value = flops / secs / 1e12
    sample = f"causal prefix of {n} positions, query head 0, per step (float64 NumPy oracle)"
    print(json.dumps({
        "impl": "reference", "metric": BWD_METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": _config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


def _timed_launches(args, step, dev, stream, dist):
    """Warm-up, then args.steps steps bracketed by barriers and syncs; returns
    (total ms, mean per-launch ms from events on the launching stream, clocks)."""
    import torch
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    total_ms = _max_over_ranks(total_ms, dist, dev)
    return total_ms, statistics.mean(a.elapsed_time(b) for a, b in ev), clk


def _layout_line(args, world, metric, w, cfg, flop, total_ms, kernel_ms, clk, cpu):
    peaks, peak_src = _peaks()
    achieved = flop / (kernel_ms / 1e3) / 1e12
    peak = float(peaks["bf16_tflops"])
    return {
        "metric": metric, "value": _job_rate(world, flop, args.steps, total_ms) / 1e12,
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": cfg,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": _traffic("attn_tc", w.name),
                     "peak_source": f"{peak_src} bf16 dense (burst)",
                     "kernel": f"attn_tc_kernel<{w.D},false,...>", "kernel_ms": kernel_ms,
                     "frac_of_sustained_peak": achieved / float(peaks["bf16_tflops_sustained"])},
        "cpu_baseline": cpu, "clocks": clk, "gpu_launches": args.steps,
    }


def run_varlen(args, w):
    """Packed variable-length batch through ring_attn_fwd_varlen."""
    import numpy as np
    import torch
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import make_varlen

    world, rank, local, dist = _dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load()
    q, k, v, cu = make_varlen(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    cud = torch.tensor(cu, dtype=torch.int32, device=dev)
    out, lse = torch.empty_like(qd), torch.empty(w.H_q, w.total, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.ring_attn_fwd_varlen(qd, kd, vd, cud, w.max_seqlen, w.P, w.causal, w.scale,
                                     w.order, out=out, lse=lse, dev_status=status, stream=stream)

    total_ms, kernel_ms, clk = _timed_launches(args, step, dev, stream, dist)
    if int(status.item()) != 0:
        raise RuntimeError("device-side wait expired")
    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        n = w.lengths[0]
        rows = np.sort(np.random.default_rng(7).choice(n, 256, replace=False))
        t0 = time.perf_counter()
        oracle.attention_rows(q[None, :n], k[None, :n], v[None, :n], w.causal, w.scale, rows)
        dt = time.perf_counter() - t0
        pairs = float((rows + 1).sum()) if w.causal else 256.0 * n
        cpu = {"value": 4.0 * w.D * pairs * w.H_q / dt / 1e12, "unit": UNIT,
               "cores": _blas_threads(), "kind": "oracle",
               "sample": f"256 random query rows of the first sequence ({n} tokens), all "
                         f"heads, float64 NumPy oracle, {dt:.1f} s"}
    cfg = _varlen_config(w)
    line = _layout_line(args, world, VARLEN_METRIC, w, cfg, w.flop, total_ms, kernel_ms, clk,
                        cpu)
    print(json.dumps(line), flush=True)
    return 0


def run_ulysses(args, w):
    """Sequence-parallel (Ulysses) layout through ring_attn_fwd_ulysses."""
    import torch
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import make_sharded_qkv

    world, rank, local, dist = _dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load()
    q, k, v = make_sharded_qkv(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    C = q.shape[2]
    out = torch.empty_like(qd)
    lse = torch.empty(w.P, w.B, w.H_q, C, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.ring_attn_fwd_ulysses(qd, kd, vd, w.S, w.causal, w.scale, out=out, lse=lse,
                                      dev_status=status, stream=stream)

    total_ms, kernel_ms, clk = _timed_launches(args, step, dev, stream, dist)
    if int(status.item()) != 0:
        raise RuntimeError("device-side wait expired")
    if rank != 0:
        return 0
    line = _layout_line(args, world, ULYSSES_METRIC, w, _ulysses_config(w), w.flop, total_ms,
                        kernel_ms, clk, None)
    print(json.dumps(line), flush=True)
    return 0


def run_merge(args, w):
    """The standalone n-way LSE merge on its workload; HBM-bound, GB/s."""
    import torch
    from sequence_exact_attention_gb300 import binding
    from sequence_exact_attention_gb300.workloads import make_merge_parts

    world, rank, local, dist = _dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.load()
    os_, ls = make_merge_parts(w)
    od = [o.to(dev) for o in os_]
    ld = [l.to(dev) for l in ls]
    out = torch.empty_like(od[0])
    lse = torch.empty_like(ld[0])
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        binding.attn_lse_merge_n(od, ld, out=out, lse=lse, stream=stream)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        dist.barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        binding.attn_lse_merge_n(od, ld, out=out, lse=lse, stream=stream)
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    total_ms = _max_over_ranks(total_ms, dist, dev)
    if rank != 0:
        return 0
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    peaks, src = _peaks()
    gbs = w.bytes / (kernel_ms / 1e3) / 1e9
    line = {
        "metric": MERGE_METRIC, "value":
            _job_rate(world, w.bytes, args.steps, total_ms) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if w.dtype == "f32" else "bf16",
        "data": "synthetic",
        "config": _merge_config(w),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]),
                     "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]),
                     "traffic": _traffic("merge", w.name),
                     "peak_source": f"{src} HBM copy", "kernel": "lse_merge_kernel",
                     "kernel_ms": kernel_ms},
        "clocks": clk, "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def _varlen_config(w):
    return {"workload": w.name, "lengths": list(w.lengths), "total": w.total, "H_q": w.H_q,
            "H_kv": w.H_kv, "D": w.D, "P": w.P, "causal": w.causal, "order": w.order,
            "layout": "packed [total, H, D], cu_seqlens on the device",
            "l2": "inputs larger than L2", "parallelism": "replicas"}


def _ulysses_config(w):
    return dict(_config(w), layout="sequence-parallel [P, B, C, H, D], C = S/P",
                parallelism="replicas (P virtual ranks inside one launch)")


def _merge_config(w):
    return {"workload": w.name, "n": w.n, "B": w.B, "H": w.H, "S": w.S, "D": w.D,
            "l2": "inputs larger than L2 (8 GiB of partials)"}


def _reference_line(args, metric, unit, value, total_t, cfg, sample):
    """The reference arm's JSON line: the float64 oracle on the host cores."""
    return {
        "impl": "reference", "metric": metric, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": unit, "cores": _blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _timed_samples(args, sample):
    """args.warmup untimed and args.steps timed calls of sample(seed) ->
    (work, seconds); returns (work per second, total seconds)."""
    for i in range(args.warmup):
        sample(100 + i)
    work, total_t = 0.0, 0.0
    for i in range(args.steps):
        wk, dt = sample(1000 + i)
        work += wk
        total_t += dt
    return work / total_t, total_t


def run_varlen_reference(args, w):
    """The oracle on sampled rows of the packed batch, each row within its
    own sequence."""
    import numpy as np
    import oracle
    from sequence_exact_attention_gb300.workloads import make_varlen
    world, rank, _, _ = _dist_setup(args.gpus)
    if rank != 0:
        return 0
    q, k, v, cu = make_varlen(w)
    cu = np.asarray(cu)
    n_rows = min(args.ref_rows, w.total)

    def sample(seed):
        rows = np.sort(np.random.default_rng(seed).choice(w.total, n_rows, replace=False))
        seq = np.searchsorted(cu, rows, side="right") - 1
        pairs, dt = 0.0, 0.0
        for b in np.unique(seq):
            lo, hi = int(cu[b]), int(cu[b + 1])
            local = rows[seq == b] - lo
            t0 = time.perf_counter()
            oracle.attention_rows(q[None, lo:hi], k[None, lo:hi], v[None, lo:hi], w.causal,
                                  w.scale, local)
            dt += time.perf_counter() - t0
            pairs += float((local + 1).sum()) if w.causal else float(len(local) * (hi - lo))
        return 4.0 * w.D * w.H_q * pairs, dt

    rate, total_t = _timed_samples(args, sample)
    line = _reference_line(args, VARLEN_METRIC, UNIT, rate / 1e12, total_t, _varlen_config(w),
                           f"{n_rows} random rows of the packed batch x all {w.H_q} heads per "
                           "step, each over its own sequence (float64 NumPy oracle)")
    print(json.dumps(line), flush=True)
    return 0


def run_ulysses_reference(args, w):
    """The oracle on sampled rows of the same attention: the Ulysses method's
    result is full attention over the whole sequence."""
    import numpy as np
    import oracle
    from sequence_exact_attention_gb300.workloads import make_sharded_qkv
    world, rank, _, _ = _dist_setup(args.gpus)
    if rank != 0:
        return 0
    qs, ks, vs = make_sharded_qkv(w)

    def unshard(x):      # [P, B, C, H, D] -> [B, S, H, D]
        P, B, C, H, D = x.shape
        return x.permute(1, 0, 2, 3, 4).reshape(B, P * C, H, D)[:, :w.S]

    q, k, v = unshard(qs), unshard(ks), unshard(vs)
    n_rows = min(args.ref_rows, w.S)

    def sample(seed):
        rate, dt, _ = _oracle_sample_rate(w, q, k, v, n_rows, seed)
        return rate * dt * 1e12, dt

    rate, total_t = _timed_samples(args, sample)
    line = _reference_line(args, ULYSSES_METRIC, UNIT, rate / 1e12, total_t, _ulysses_config(w),
                           f"{n_rows} random query rows x all {w.H_q} heads x {w.B} sequences "
                           "per step, full key range (float64 NumPy oracle)")
    print(json.dumps(line), flush=True)
    return 0


def run_merge_reference(args, w):
    """The oracle's n-way merge on a slice of the workload's rows."""
    import dataclasses
    import oracle
    from sequence_exact_attention_gb300.workloads import make_merge_parts
    world, rank, _, _ = _dist_setup(args.gpus)
    if rank != 0:
        return 0
    ws = dataclasses.replace(w, S=min(w.S, 16 * args.ref_rows))
    os_, ls = make_merge_parts(ws)

    def sample(seed):
        t0 = time.perf_counter()
        oracle.lse_merge_n(os_, ls)
        return float(ws.bytes), time.perf_counter() - t0

    rate, total_t = _timed_samples(args, sample)
    line = _reference_line(args, MERGE_METRIC, "GB/s", rate / 1e9, total_t, _merge_config(w),
                           f"all {ws.n} partials of S={ws.S} positions (same B, H, D, drawn "
                           "the same way) per step (float64 NumPy oracle)")
    print(json.dumps(line), flush=True)
    return 0


def main():
    from sequence_exact_attention_gb300.workloads import (BWD_WORKLOADS, HEADLINE,
                                                          MERGE_WORKLOADS, ULYSSES_WORKLOADS,
                                                          VARLEN_WORKLOADS, WORKLOADS)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=sorted(WORKLOADS) + sorted(MERGE_WORKLOADS) + sorted(BWD_WORKLOADS)
                    + sorted(VARLEN_WORKLOADS) + sorted(ULYSSES_WORKLOADS))
    ap.add_argument("--cpu-rows", type=int, default=768)
    ap.add_argument("--ref-rows", type=int, default=24)
    ap.add_argument("--cpu-prefix", type=int, default=16384,
                    help="backward workloads: causal prefix length of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="headline only: skip the sweep of the other workloads")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override S (smaller profiling cases of the same shape)")
    args = ap.parse_args()
    ref = args.impl == "reference"
    if args.workload in MERGE_WORKLOADS:
        w = MERGE_WORKLOADS[args.workload]
        if args.seq_len:
            w = dataclasses.replace(w, S=args.seq_len, name=f"{w.name}@S={args.seq_len}")
        return run_merge_reference(args, w) if ref else run_merge(args, w)
    if args.workload in VARLEN_WORKLOADS:
        w = VARLEN_WORKLOADS[args.workload]
        return run_varlen_reference(args, w) if ref else run_varlen(args, w)
    if args.workload in ULYSSES_WORKLOADS:
        w = ULYSSES_WORKLOADS[args.workload]
        return run_ulysses_reference(args, w) if ref else run_ulysses(args, w)
    if args.workload in BWD_WORKLOADS:
        w = BWD_WORKLOADS[args.workload]
        if args.seq_len:
            w = w.scaled(S=args.seq_len, name=f"{w.name}@S={args.seq_len}")
        return run_bwd_reference(args, w) if args.impl == "reference" else run_bwd(args, w)
    w = WORKLOADS[args.workload]
    if args.seq_len:
        w = w.scaled(S=args.seq_len, name=f"{w.name}@S={args.seq_len}")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
