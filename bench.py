#!/usr/bin/env python
"""Benchmark of the K3 DFlash drafter block attention; prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long_context|mixed_8x8|heads_24_4|tiny|w6_8x6|single_w6|...]
                    [--yarn] [--op attn|qk_norm_rope] [--warm-l2] [--no-e2e] [--no-cpu-baseline]
                    [--sweep]

Metric: drafter block-attention microseconds per call (lower is better) on
one of the op's workloads, default the long-context one (8 requests x 8 draft
tokens, 24/4 heads, contexts U{16384..131072}, a 20,000-page bf16 pool,
fused RMSNorm + RoPE, int64 positions), with the achieved HBM bandwidth of
the dominant kernel against the measured copy bandwidth in "roofline".

ours:       the CUDA library through its Python binding.  Inputs are resident
            in HBM; L2 is flushed (512 MB written, then 512 MB read) before
            every timed call; each call is timed with CUDA events on the
            launching stream.  "e2e" times the same call handed the per-step
            inputs (qkv, page table, lengths, positions) and the output in
            pinned host memory: the kernels read and write them across the
            host link inside the timed region.  "e2e_copies" times it with
            the inputs copied to device memory in one packed copy and the
            output copied back instead.  --warm-l2 skips the flush (a warm-cache line,
            labelled in "config").  "cpu_baseline" is one whole call of the
            fp64 oracle on one host thread; "cpu_all_cores" is one whole call
            of it on all host cores.
reference:  the fp64 CPU oracle (test infrastructure, timed as it stands on
            the host cores), each step one whole call of the same workload on
            all host threads.

Multi-GPU: the op does not shard across GPUs in a way that needs any
exchange; N ranks run N independent replicas ("replicas only") and value is
the job's aggregate time per call (max-over-ranks time / calls of all ranks).
"""
from __future__ import annotations

import argparse
import functools
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "drafter block-attn µs/call and HBM GB/s (% of GB300 peak) at 8 req × 8 tok"
UNIT = "us/call"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20   # written, then a second buffer of this size is read
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCE = os.path.join(ROOT, "speculative_decoding_drafter_k3_gb300", "csrc", "k3da.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_context")
    ap.add_argument("--op", choices=["attn", "qk_norm_rope"], default="attn",
                    help="attn: the block attention (headline); qk_norm_rope: the standalone "
                         "fused q/k norm + RoPE call on --tokens tokens of --heads heads")
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--yarn", action="store_true",
                    help="YaRN RoPE (factor 4, original context 4096, beta 32/1, mscale 0.1 ln 4 + 1)")
    ap.add_argument("--heads", choices=["6/1", "24/4"], default="24/4")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-small", action="store_true",
                    help="skip the extra timing of the small workloads on the default line")
    ap.add_argument("--warm-l2", action="store_true",
                    help="do not flush L2 between timed calls (a labelled warm-cache line, "
                         "never the headline)")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the headline: time every other configuration (tiny, the "
                         "8x8 and W=6 shapes, each request x token split) with L2 flushed and "
                         "warm, one JSON line")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            data = json.load(open(path))

            def find(d):
                if isinstance(d, dict):
                    for k, v in d.items():
                        if k == "hbm_gbs" and isinstance(v, (int, float)):
                            return float(v)
                        r = find(v)
                        if r:
                            return r
                return None

            v = find(data)
            if v:
                return v, "measured (MEASURED_PEAKS.json hbm_gbs)"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 copy measurement)"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={device_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def samples(self) -> int:
        if self.proc is None:
            return 0
        try:
            return sum(1 for _ in open(self.path))
        except OSError:
            return 0

    def settle(self, busy, seconds: float = 0.8):
        """Keeps the GPU busy (untimed calls of ``busy``) until nvidia-smi has
        been sampling for ``seconds``, so its start-up never overlaps the
        timed region and the samples it takes are under load."""
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds or (self.proc is not None and self.samples() < 2
                                                      and time.perf_counter() - t0 < 5.0):
            busy()
            torch.cuda.synchronize()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def kernel_source_hash() -> str:
    return hashlib.sha256(open(KERNEL_SOURCE, "rb").read()).hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the split kernel from a committed ncu capture,
    or None when absent or taken on a different kernel source."""
    try:
        data = json.load(open(PROFILE_TRAFFIC))
    except (OSError, ValueError):
        return None
    entry = data.get(workload)
    if not entry or entry.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


# ------------------------------------------------------------- CPU oracle --

def cpu_baseline(case):
    """One whole call of the fp64 oracle on one host thread (its R x Hkv
    independent (request, kv head) units one after another), wall clock."""
    from oracle import units as ou

    us = ou.units_of(case)
    _, wall, n = ou.run_units(us, threads=1)
    return {"value": wall * 1e6, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"whole call: fp64 C oracle, {len(us)} (request, kv head) units on 1 thread, wall clock"}


def cpu_all_cores(case, threads: int = 0):
    """One whole call of the oracle on all host cores: the R x Hkv
    independent (request, kv head) units, longest first, on a pool of
    threads (the C oracle keeps no global state and ctypes releases the GIL
    during each call).  Wall-clock time of the pool; inputs marshalled
    before the clock starts."""
    from oracle import units as ou

    us = ou.units_of(case)
    _, wall, n = ou.run_units(us, threads=threads)
    return {"value": wall * 1e6, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": (f"whole call: fp64 C oracle, {len(us)} (request, kv head) units on "
                       f"{n} threads, wall clock")}


# ------------------------------------------------------------------ arms --

def config_of(case, extra=None):
    cfg = {"workload": case.name, "requests": case.R, "block_tokens": case.B,
           "heads": f"{case.Hq}/{case.Hkv}", "head_dim": case.D, "page_size": case.P,
           "pool_pages": case.num_pages, "page_stride": case.page_stride,
           "qknorm_rope": case.qknorm, "positions": str(case.pos_dtype).replace("torch.", ""),
           "context_tokens": case.context_tokens(), "ctx_lens": case.lens_list(),
           "algorithmic_bytes_per_call": case.algorithmic_bytes(),
           "l2": "flushed before every timed call (512 MB written, then 512 MB read)"}
    if extra:
        cfg.update(extra)
    return cfg


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host
    cores.  Each step is one whole call of the workload (its (request, kv
    head) units on a pool of all host threads), wall clock."""
    from speculative_decoding_drafter_k3_gb300 import workloads
    from oracle import units as ou

    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = workloads.WORKLOADS[args.workload](device=dev)
    us = ou.units_of(case)
    for _ in range(args.warmup):
        ou.run_units(us)
    times, n = [], 0
    for _ in range(args.steps):
        _, wall, n = ou.run_units(us)
        times.append(wall)
    us_call = statistics.mean(times) * 1e6
    sample = (f"whole call per step: fp64 C oracle, {len(us)} (request, kv head) units on {n} host "
              f"threads, wall clock")
    line = {"impl": "reference", "metric": METRIC, "value": us_call, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us_call / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(case),
            "cpu_baseline": {"value": us_call, "unit": UNIT, "cores": n, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": us_call, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_sweep(args, k3da, workloads, dev, status, flush, timed_calls):
    """Every configuration but the long-context one, whole calls timed as
    the headline is (events on the launching stream, K calls), once with L2
    flushed before each call and once warm (the previous call's inputs left
    in L2, a spin kernel in front of each call): one JSON line."""
    cases = [("tiny", workloads.tiny), ("mixed_8x8", workloads.mixed_8x8),
             ("heads_24_4", workloads.heads_24_4), ("w6_8x6", workloads.w6_8x6),
             ("single_w6", workloads.single_w6), ("single_w6_long", workloads.single_w6_long)]
    cases += [(f"split_{r}x{b}", functools.partial(workloads.split_sweep, r, b))
              for r, b in workloads.SPLITS]
    rows = {}
    for name, make in cases:
        c = make(device=dev)
        o = torch.empty(c.T, c.Hq * c.D, dtype=torch.bfloat16, device=dev)
        w = k3da.case_workspace(c)
        row = {"algorithmic_bytes": c.algorithmic_bytes()}
        for warm in (False, True):
            flush.warm = warm
            ms = sorted(timed_calls(c, o, w, args.steps))
            row["warm" if warm else "cold"] = {
                "us_mean": statistics.mean(ms) * 1e3, "us_median": statistics.median(ms) * 1e3,
                "us_p10": ms[len(ms) // 10] * 1e3, "us_p90": ms[(9 * len(ms)) // 10] * 1e3}
        rows[name] = row
    flush.warm = args.warm_l2
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    print(json.dumps({"sweep": rows, "unit": UNIT, "steps": args.steps, "warmup": args.warmup,
                      "timing": "whole calls, CUDA events on the launching stream; cold = L2 "
                                "flushed before each call, warm = previous call's inputs in L2"}),
          flush=True)


def run_ours(args, world, rank):
    import speculative_decoding_drafter_k3_gb300 as k3da
    from speculative_decoding_drafter_k3_gb300 import build as kbuild, workloads

    kbuild.build()
    k3da.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workloads.WORKLOADS[args.workload](device=dev)
    out = torch.empty(case.T, case.Hq * case.D, dtype=torch.bfloat16, device=dev)
    ws = k3da.case_workspace(case)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    class _Flush:
        warm = args.warm_l2

        def zero_(self):
            # Write a buffer larger than L2, then read another one: L2 ends
            # up holding clean lines of neither input, so the timed call
            # neither hits in L2 nor pays for writing back the flush.
            if self.warm:
                # No flush: a spin kernel that touches no memory keeps the
                # GPU busy while the host enqueues the call, so the timed
                # call is not waiting for its own launch.
                torch.cuda._sleep(200_000)
                return
            flush_w.zero_()
            torch.sum(flush_r, dim=0, out=sink)

    flush = _Flush()

    yarn = k3da.Yarn.of(4.0, 4096.0) if args.yarn and case.qknorm else None

    def timed_calls(c, o, w, K, clocks=None):
        """K calls of case c, each after an L2 flush, each bracketed by CUDA
        events on the launching stream; returns the per-call times in ms.
        Python's garbage collector is off while the calls are enqueued, so
        no host pause can open a gap between an event and its call."""
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            k3da.run_case(c, out=o, workspace=w, status=status, yarn=yarn)
        torch.cuda.synchronize()
        if clocks is not None:
            def busy():
                for _ in range(20):
                    flush.zero_()
                    k3da.run_case(c, out=o, workspace=w, status=status, yarn=yarn)
            clocks.settle(busy)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        barrier(world)
        torch.cuda.synchronize()
        gc.disable()
        try:
            for i in range(K):
                flush.zero_()
                ev[i][0].record()
                k3da.run_case(c, out=o, workspace=w, status=status, yarn=yarn)
                ev[i][1].record()
            torch.cuda.synchronize()
        finally:
            gc.enable()
        barrier(world)
        return [e[0].elapsed_time(e[1]) for e in ev]

    K = args.steps
    if args.sweep:
        run_sweep(args, k3da, workloads, dev, status, flush, timed_calls)
        return
    # Headline: whole calls (split pass + combine), one event pair per call.
    clocks = ClockSampler(dev.index) if rank == 0 else None
    call_ms = timed_calls(case, out, ws, K, clocks)
    clock_info = clocks.stop() if clocks else None
    total_ms = max_over_ranks(sum(call_ms), world)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    value = total_ms * 1e3 / (K * world)

    # Roofline: the split pass alone, bracketed by an event the library
    # records between its two kernels.
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for e in pev:
        e[1].record()  # torch creates its events lazily: create the one the library records
    torch.cuda.synchronize()
    gc.disable()
    for i in range(K):
        flush.zero_()
        pev[i][0].record()
        k3da.set_phase_event(pev[i][1])
        k3da.run_case(case, out=out, workspace=ws, status=status, yarn=yarn)
        pev[i][2].record()
    torch.cuda.synchronize()
    gc.enable()
    k3da.set_phase_event(None)
    split_ms = [e[0].elapsed_time(e[1]) for e in pev]
    combine_ms = [e[1].elapsed_time(e[2]) for e in pev]  # combine after the event: no launch overlap

    # The drafter's deployed shapes (8x8 mixed lengths, 24/4 heads, the W=6
    # block), timed the same way in the same process.
    small = None
    if args.workload == "long_context" and not args.no_small:
        small = {}
        for name in ("mixed_8x8", "heads_24_4", "w6_8x6"):
            c = workloads.WORKLOADS[name](device=dev)
            o = torch.empty(c.T, c.Hq * c.D, dtype=torch.bfloat16, device=dev)
            ms = timed_calls(c, o, k3da.case_workspace(c), K)
            small[name] = {"us_per_call": statistics.mean(ms) * 1e3,
                           "median_us": statistics.median(ms) * 1e3,
                           "algorithmic_bytes": c.algorithmic_bytes()}
        assert int(status.item()) == 0, f"device status {int(status.item())}"

    # End to end through the public binding with host buffers, two ways.
    # Host-resident ("e2e"): the call is handed the pinned host tensors
    # themselves (qkv, page table, lengths, positions, output); its kernels
    # read the inputs and write the output across the host link, with no
    # copy.  Copies ("e2e_copies"): the inputs travel from pinned host memory
    # in one packed copy, the call reads them in device memory, and the
    # output comes back in one copy.
    e2e = e2e_copies = None
    if not args.no_e2e:
        import dataclasses
        inputs = [case.qkv, case.page_table, case.ctx_lens] + ([case.positions] if case.qknorm else [])
        offs, total = [], 0
        for t in inputs:
            total = (total + 15) // 16 * 16
            offs.append(total)
            total += t.numel() * t.element_size()
        dev_pack = torch.empty(total, dtype=torch.uint8, device=dev)
        host_pack = torch.zeros(total, dtype=torch.uint8).pin_memory()
        views, host_views = [], []
        for t, o in zip(inputs, offs):
            n = t.numel() * t.element_size()
            host_pack[o:o + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
            views.append(dev_pack[o:o + n].view(t.dtype).view(t.shape))
            host_views.append(host_pack[o:o + n].view(t.dtype).view(t.shape))
        case_e2e = dataclasses.replace(case, qkv=views[0], page_table=views[1], ctx_lens=views[2],
                                       positions=views[3] if case.qknorm else None)
        case_host = dataclasses.replace(case, qkv=host_views[0], page_table=host_views[1],
                                        ctx_lens=host_views[2], positions=host_views[3] if case.qknorm else None)
        host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        def step_copies():
            dev_pack.copy_(host_pack, non_blocking=True)
            k3da.run_case(case_e2e, out=out, workspace=ws, status=status, yarn=yarn)
            host_out.copy_(out, non_blocking=True)

        def step_host():
            k3da.run_case(case_host, out=host_out, workspace=ws, status=status, yarn=yarn)

        def time_steps(step):
            for _ in range(3):
                step()
            torch.cuda.synchronize()
            eev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
            barrier(world)
            torch.cuda.synchronize()
            gc.disable()
            for i in range(K):
                flush.zero_()
                eev[i][0].record()
                step()
                eev[i][1].record()
            torch.cuda.synchronize()
            gc.enable()
            barrier(world)
            return max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in eev), world) * 1e3 / (K * world)

        h2d = sum(t.numel() * t.element_size() for t in inputs)
        d2h = out.numel() * out.element_size()
        e2e = {"value": time_steps(step_host), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "copies_per_step": {"h2d": 0, "d2h": 0},
               "transfer": "host-resident: the call is handed the pinned host tensors; its kernels "
                           "read the inputs and write the output across the host link"}
        e2e_copies = {"value": time_steps(step_copies), "unit": UNIT, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "copies_per_step": {"h2d": 1, "d2h": 1},
                      "transfer": "one packed cudaMemcpyAsync of the inputs to device memory, the "
                                  "call, one copy of the output back"}
        assert int(status.item()) == 0, f"device status {int(status.item())}"

    out_bytes = case.T * case.Hq * case.D * 2
    split_bytes = case.algorithmic_bytes() - out_bytes
    split_us = statistics.mean(split_ms) * 1e3
    peak, peak_src = measured_hbm_peak()
    achieved = split_bytes / (split_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profiled_traffic(args.workload),
                "kernel": "k3da_tc_kernel (split pass; combine excluded)",
                "algorithmic_bytes_per_launch": split_bytes, "launch_us": split_us,
                "peak_source": peak_src,
                "combine_us_unoverlapped": statistics.mean(combine_ms) * 1e3,
                "whole_call_gbs": case.algorithmic_bytes() / (value * 1e-6) / 1e9,
                "whole_call_frac": case.algorithmic_bytes() / (value * 1e-6) / 1e9 / peak}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)",
            "data": "synthetic (seeded N(0,1) bf16 pool/qkv, random page permutation)",
            "config": config_of(case, {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                       **({"l2": "warm: not flushed between timed calls (inputs stay "
                                                 "in L2 from the previous call)"} if args.warm_l2 else {}),
                                       "rope": "yarn(4.0, 4096, 32, 1)" if yarn is not None else "neox",
                                       "split_ctas": k3da.split_grid(dev.index)}),
            "roofline": roofline, "e2e": e2e, "e2e_copies": e2e_copies, "gpu_launches": 2 * K, "clocks": clock_info,
            "small_workloads": small,
            "median_call_us": statistics.median(call_ms) * 1e3,
            "p10_p90_call_us": [sorted(call_ms)[int(0.1 * (K - 1))] * 1e3,
                                sorted(call_ms)[int(0.9 * (K - 1))] * 1e3]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
        line["cpu_all_cores"] = cpu_all_cores(case)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_norm_rope(args, world, rank):
    """The standalone q/k norm + RoPE call: µs per call on T tokens, L2
    flushed before each call; bytes = q and k heads read and written,
    positions, weights."""
    import speculative_decoding_drafter_k3_gb300 as k3da
    from speculative_decoding_drafter_k3_gb300 import build as kbuild

    kbuild.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    Hq, Hkv = (24, 4) if args.heads == "24/4" else (6, 1)
    T, D = args.tokens, 64
    g = torch.Generator().manual_seed(12)
    qkv = torch.randn(T, (Hq + 2 * Hkv) * D, generator=g).to(torch.bfloat16).to(dev)
    qw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16).to(dev)
    kw = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16).to(dev)
    pos = torch.randint(0, 1 << 17, (T,), generator=g, dtype=torch.int64).to(dev)
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    yarn = k3da.Yarn.of(4.0, 4096.0) if args.yarn else None

    def call():
        k3da.k3da_qk_norm_rope(qkv, pos, qw, kw, num_q_heads=Hq, num_kv_heads=Hkv, yarn=yarn)

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(dev.index) if rank == 0 else None
    barrier(world)
    for i in range(K):
        flush_w.zero_()
        ev[i][0].record()
        call()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    clock_info = clocks.stop() if clocks else None
    ms = [e[0].elapsed_time(e[1]) for e in ev]
    us = max_over_ranks(sum(ms), world) * 1e3 / (K * world)
    nbytes = 2 * T * (Hq + Hkv) * D * 2 + T * 8 + 2 * D * 2
    peak, peak_src = measured_hbm_peak()
    achieved = nbytes / (us * 1e-6) / 1e9
    # CPU baseline: the fp64 oracle of the cell on the same tokens.
    import oracle
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < 2.0 or n < 3:
        oracle.qk_norm_rope(qkv.cpu(), pos.cpu(), qw.cpu(), kw.cpu(), num_q_heads=Hq, num_kv_heads=Hkv)
        n += 1
    cpu_us = (time.perf_counter() - t0) / n * 1e6
    line = {"metric": "fused q/k RMSNorm + NeoX RoPE µs/call", "value": us, "unit": "us/call",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 math)",
            "data": "synthetic (seeded N(0,1) bf16 qkv)",
            "config": {"workload": f"qk_norm_rope_T{T}_{args.heads}", "tokens": T, "heads": args.heads,
                       "head_dim": D, "positions": "int64",
                       "l2": "flushed before every timed call (512 MB written)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "kernel": "k3da_norm_rope_kernel",
                         "algorithmic_bytes_per_launch": nbytes, "launch_us": us, "peak_source": peak_src},
            "e2e": None, "gpu_launches": K, "clocks": clock_info,
            "cpu_baseline": {"value": cpu_us, "unit": "us/call", "cores": 1, "kind": "oracle",
                             "sample": f"the whole call ({T} tokens), {n} runs"}}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank = dist_setup(args)
    if args.op == "qk_norm_rope" and args.impl == "ours":
        run_norm_rope(args, world, rank)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
