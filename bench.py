"""Benchmark: exact attention forward TFLOP/s (causal-adjusted) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (the one the headline metric is quoted on): exact attention forward, B=1, H=8, N=32768,
d=64, fp16 Q/K/V i.i.d. N(0,1) (seeded synthetic inputs), causal, scale 1/sqrt(64), device-resident,
monolithic path (cqsa_attn_fwd). A step is one forward over that input. Causal-adjusted FLOP per
step = 4*B*H*N^2*d/2.

- value: device time of the K timed steps, each bracketed by CUDA events on the launch stream, with
  the 129 MB L2 flushed (256 MiB write) before every step outside the events; whole-job throughput
  over N ranks (weak scaling: every rank runs the full workload; max time over ranks).
- e2e: the same metric through the C ABI with HOST buffers: cqsa_stream_attn_fwd with pinned host
  Q/K/V and a pinned host output (16,384-token chunks), host<->device copies inside the timed region.
- roofline: achieved algorithmic FLOP/s of the attention kernel vs the measured dense fp16/bf16 tensor
  peak (MEASURED_PEAKS.json; else the fallback figure, labelled so).
- cpu_baseline: the FP64 oracle on a bounded sample of the workload's rows on this host's cores.
- --impl reference: the oracle itself as the reference arm, on a bounded row sample per step.

Secondary measurements (one JSON line each, not the headline; `--measure NAME`):
- merge: the LSE merge of the 131,072-token chunked workload (16,384-token chunks, Q chunk i merges
  i+1 fp32 partials), achieved HBM GB/s of the algorithmic bytes vs the measured copy bandwidth.
- link: pinned host <-> device copy probe (1 GiB cudaMemcpyAsync each way), the link roofline.
- stream: the host-resident streaming driver (token-major pinned Q/K/V, 262,144-token chunks; N from
  --n, default 4,000,000): TFLOP/s, copy rate while overlapped vs the link probe, stall time.
- bf16: B=2 H=32 N=16384 d=128 bf16 non-causal monolithic forward (K scaled by 3), TFLOP/s and the
  fraction of the tensor peak (algorithmic FLOP; the hi/lo split of P costs 1.5x the MMA work).
- bwd: the attention backward (dq, dk, dv from the saved LSE) on the headline shape, TFLOP/s of the
  five products vs the tensor peak.
- quorum: the cyclic quorum-set decomposition on the pages' 4,000,000-token example (B=1 H=8 d=64
  fp16 causal, c=31, interest set (0,1,3,8,12,18), itr=1: 31 subproblems), token-major pinned host
  Q/K/V/out (N from --n); TFLOP/s, kernel time, staging copies.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

B, H, N, D = 1, 8, 32768, 64
CAUSAL = True
FLOP_PER_STEP = 4.0 * B * H * N * N * D / 2.0
E2E_CHUNK = N // 8  # 4,096 tokens: the first copy is small and 8 launches overlap over the driver's streams
WORKLOAD = "exact attention forward, B=1 H=8 N=32768 d=64 fp16 causal, scale 1/sqrt(64), device-resident, monolithic"
METRIC = "exact attention fwd TFLOP/s (causal-adjusted) at 1 GB300; % of tensor-core peak"
FALLBACK_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        for key in ("bf16_tflops", "bf16_dense_tflops", "tflops_bf16"):
            if key in pk:
                return float(pk[key]), "measured (MEASURED_PEAKS.json %s)" % key, pk
    return FALLBACK_TFLOPS, "fallback (1.9 PFLOP/s bf16 burst, earlier GB300 measurement)", None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Weak scaling: every rank runs `steps` full steps; the job takes the slowest rank's time."""
    return world * flop_per_step * steps / (max_ms / 1000.0) / 1e12


def oracle_sample(rows: int, seed: int = 1, want=False):
    """Time the FP64 oracle on `rows` seeded rows of the workload; returns (seconds, FLOP, threads), and
    with `want` also (rows, out, lse) of the oracle."""
    import oracle
    import synthetic as syn
    qn, kn, vn = syn.qkv(B, H, N, D, seed=0)
    sel = syn.sample_rows(B, H, N, rows, seed=seed)[:rows]
    t0 = time.perf_counter()
    ro, rl, _ = oracle.attn_rows(qn, kn, vn, B=B, H=H, Nq=N, d=D, causal=CAUSAL, rows=sel)
    dt = time.perf_counter() - t0
    flop = float(np.sum(4.0 * D * (sel[:, 2] + 1)))  # causal: row i sees i+1 keys
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    if want:
        return dt, flop, threads, (sel, ro, rl)
    return dt, flop, threads


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


def cpu_baseline(target_s: float = 12.0, out=None, lse=None):
    """The oracle timed on a bounded row sample of the workload on this host's cores. Given the bench's
    output (device tensors of the last timed step), its rows are also compared with the oracle's."""
    dt, flop, thr = oracle_sample(256)
    rows = int(min(65536, max(256, 256 * target_s / max(dt, 1e-3))))
    dt, flop, thr, (sel, ro, rl) = oracle_sample(rows, seed=2, want=True)
    res = {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
           "sample": f"{rows} seeded query rows (b,h,i uniform) of the workload, each in full over its causal "
                     f"keys, FP64, {dt:.1f} s",
           "cpu_model": _cpu_model(), "rows_per_s": rows / dt,
           "extrapolated_full_s": FLOP_PER_STEP / (flop / dt)}
    if out is not None:
        import torch
        b, h, i = (torch.as_tensor(sel[:, j], device=out.device) for j in range(3))
        o = out[b, h, i].float().cpu().numpy().astype(np.float64)
        e = np.abs(o - ro)
        le = np.abs(lse[b, h, i].cpu().numpy().astype(np.float64) - rl)
        res["output_check"] = {"rows": int(len(sel)), "max_abs": float(e.max()), "mean_abs": float(e.mean()),
                               "lse_max_abs": float(le.max()),
                               "within_tolerance": bool(e.max() <= 4e-3 and e.mean() <= 2e-4 and le.max() <= 1e-3),
                               "tolerance": "max abs 4e-3, mean abs 2e-4, LSE 1e-3 (fp16 output vs FP64 oracle)"}
    return res


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    # size one step to ~1/ (steps+warmup) of ~2 minutes of oracle time
    dt, flop, thr = oracle_sample(128)
    per_step_rows = int(max(64, min(8192, 128 * (90.0 / (args.steps + args.warmup)) / max(dt, 1e-3))))
    for w in range(args.warmup):
        oracle_sample(per_step_rows, seed=100 + w)
    tot_t, tot_f = 0.0, 0.0
    for s in range(args.steps):
        dt, flop, thr = oracle_sample(per_step_rows, seed=200 + s)
        tot_t += dt
        tot_f += flop
    value = tot_f / tot_t / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "sample_rows_per_step": per_step_rows},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": f"{per_step_rows} seeded query rows per step, FP64 oracle"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import exact_long_context_tcgen05_gb300 as cq
    import synthetic as syn

    qn, kn, vn = syn.qkv(B, H, N, D, seed=0)
    dev = torch.device("cuda", local)
    q, k, v = (torch.from_numpy(x.view(np.int16)).view(torch.float16).to(dev) for x in (qn, kn, vn))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        cq.cqsa_attn_fwd(q, k, v, out, lse, B, H, N, D, CAUSAL, 0.0, cq.CQSA_F16, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    rc, code, _ = cq.cqsa_device_error()
    if rc != cq.CQSA_OK:
        raise SystemExit(f"device error after warm-up: {code}")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)  # evict L2 (129 MB) between timed steps, outside the events
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    ms = [a.elapsed_time(b) for a, b in ev]
    dev_ms = max_over_ranks(sum(ms), world, dev)
    value = whole_job_tflops(FLOP_PER_STEP, args.steps, world, dev_ms)
    kernel_tflops = FLOP_PER_STEP / (statistics.mean(ms) / 1000.0) / 1e12

    # end to end: host (pinned) buffers in and out through the C ABI
    hq, hk, hv = (torch.from_numpy(x.view(np.int16)).view(torch.float16).pin_memory() for x in (qn, kn, vn))
    hout = torch.empty((B, H, N, D), dtype=torch.float16).pin_memory()
    hlse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    st = cq.cqsa_stream_stats()

    def e2e_step():
        cq.cqsa_stream_attn_fwd(hq, hk, hv, cq.CQSA_LAYOUT_BHND, hout, hlse, True, B, H, N, D, CAUSAL, 0.0,
                                cq.CQSA_F16, E2E_CHUNK, st, stream)

    for _ in range(2):
        e2e_step()
    e2e_steps = max(3, min(args.steps, 10))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_val = world * FLOP_PER_STEP / e2e_s / 1e12

    # no bounded device wait gave up during the timed steps (the device error word is clear)
    rc, code, _ = cq.cqsa_device_error()
    ok = rc == cq.CQSA_OK
    peak, peak_src, _ = _peaks()
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": dev_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f16",
                "data": "synthetic (seeded N(0,1) Q/K/V, SplitMix64 + Box-Muller)",
                "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "d": D, "causal": CAUSAL,
                           "l2": "flushed before every timed step (256 MiB device write outside the events)",
                           "parallelism": f"weak scaling, {world} independent rank(s)"},
                "roofline": {"bound": "tensor", "achieved": kernel_tflops, "peak": peak, "unit": "TFLOP/s",
                             "frac": kernel_tflops / peak, "traffic": _traffic_per_launch(),
                             "peak_source": peak_src + "; dense fp16 rate = bf16 rate"},
                "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": int(st.h2d_bytes),
                        "d2h_bytes_per_step": int(st.d2h_bytes),
                        "path": f"cqsa_stream_attn_fwd, pinned host Q/K/V/out, {E2E_CHUNK}-token chunks, inputs "
                                "resident on the device (each chunk copied once, beside the launches of the "
                                "chunks before it; one launch per query chunk over its key prefix)"},
                "gpu_launches": args.steps, "wall_s_timed_region": wall,
                "clocks": clk.summary(), "device_error_free": ok}
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(out=out, lse=lse)
        if args.secondary != "none":
            line["secondary"] = run_secondary(cq, dev, args)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def kernel_code_hash(path: str) -> str:
    """sha256[:16] of a source file's code: // comments and all white space removed, so comment and
    layout edits keep a profile's counters attached to the code they were taken on."""
    import hashlib
    with open(path) as f:
        lines = []
        for line in f.read().splitlines():
            i = line.find("//")
            if i >= 0:
                line = line[:i]
            line = "".join(line.split())
            if line:
                lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def _traffic_per_launch():
    """DRAM bytes per attention launch from the committed ncu summary of this workload, or None when
    the kernel code has changed since those counters were taken (the summary records its code hash)."""
    import re
    path = os.path.join(ROOT, "profiles", "attn_fwd_f16_d64_causal_N32768.md")
    src = os.path.join(ROOT, "exact_long_context_tcgen05_gb300", "csrc", "attn_fwd.cu")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        text = f.read()
    m_sha = re.search(r"code hash `([0-9a-f]{16})`", text)
    m_b = re.search(r"\| dram_bytes_per_launch \| (\d+) \|", text)
    if not m_sha or not m_b or m_sha.group(1) != kernel_code_hash(src):
        return None
    return int(m_b.group(1))


def _hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        for key in ("hbm_gbs", "hbm_GBps", "copy_gbs"):
            if key in pk:
                return float(pk[key]), "measured (MEASURED_PEAKS.json %s)" % key
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 copy measurement)"


def _time_events(fn, reps, stream):
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def measure_merge(cq, dev, reps):
    """LSE merge of the chunked 131,072-token workload: for Q chunk i (of 8), i+1 fp32 partials
    [1,8,16384,64] + LSE are merged into fp16 out + fp32 LSE. Partials are seeded on the device (the
    merge's speed does not depend on their values); 1.2 GB of partials, far above L2."""
    import torch
    Bm, Hm, C, Dm, nch = 1, 8, 16384, 64, 8
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    parts_o = [torch.randn((Bm, Hm, C, Dm), generator=g, device=dev) for _ in range(nch * (nch + 1) // 2)]
    parts_l = [torch.randn((Bm, Hm, C), generator=g, device=dev) for _ in range(nch * (nch + 1) // 2)]
    outs = [torch.empty((Bm, Hm, C, Dm), dtype=torch.float16, device=dev) for _ in range(nch)]
    lses = [torch.empty((Bm, Hm, C), dtype=torch.float32, device=dev) for _ in range(nch)]
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    offs = [i * (i + 1) // 2 for i in range(nch)]

    def step():
        # the query chunks' merges are independent: the four largest on the timed stream, the four
        # smallest (1-4 partials, each too small to fill the GPU alone) beside them on a second stream
        side.wait_stream(stream)
        for i in range(nch):
            s = stream if i >= nch // 2 else side
            cq.cqsa_merge_partials(parts_o[offs[i]:offs[i] + i + 1], parts_l[offs[i]:offs[i] + i + 1], i + 1,
                                   outs[i], lses[i], Bm, Hm, C, Dm, cq.CQSA_F16, s)
        stream.wait_stream(side)

    for _ in range(3):
        step()
    ms = statistics.median(_time_events(step, reps, stream))
    rows = Bm * Hm * C
    nparts = nch * (nch + 1) // 2
    algo = nparts * rows * (Dm * 4 + 4) + nch * rows * (Dm * 2 + 4)
    peak, src = _hbm_peak()
    gbs = algo / (ms / 1000.0) / 1e9
    return {"measure": "merge", "workload": "LSE merge, 131,072 tokens in 16,384-token chunks (36 partials, 8 merges), "
            "B=1 H=8 d=64, fp32 partials -> fp16 out + fp32 LSE", "ms_per_step": ms, "algorithmic_bytes": algo,
            "launches_per_step": nch, "streams": 2,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "peak_source": src}}


def measure_link(dev, reps):
    import torch
    nbytes = 1 << 30
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    h2d = _time_events(lambda: d.copy_(h, non_blocking=True), reps, stream)
    d2h = _time_events(lambda: h.copy_(d, non_blocking=True), reps, stream)
    return {"measure": "link", "bytes": nbytes, "h2d_gbs": nbytes / (statistics.median(h2d) / 1e3) / 1e9,
            "d2h_gbs": nbytes / (statistics.median(d2h) / 1e3) / 1e9,
            "method": "1 GiB pinned host buffer, cudaMemcpyAsync, CUDA events, median of %d" % reps}


def measure_stream(cq, dev, n_tokens, link_h2d_gbs, host=None, accumulating=False):
    """Host-resident streaming forward. By default the driver keeps the inputs resident on the device
    (they fit) and runs one launch per query chunk; accumulating=True forces the memory-bounded schedule
    (every chunk pair through the fp32 accumulator, K/V chunks double-buffered)."""
    import torch
    Bs, Hs, Ds, C = 1, 8, 64, 262_144
    shape = (Bs, n_tokens, Hs, Ds)
    if host is None:
        host = _host_qkv_token_major(n_tokens, Hs, Ds)
    out = torch.empty(shape, dtype=torch.float16).pin_memory()
    lse = torch.empty((Bs, Hs, n_tokens), dtype=torch.float32).pin_memory()
    st = cq.cqsa_stream_stats()
    stream = torch.cuda.current_stream(dev)
    cq.cqsa_set_stream_kv_resident_bytes(0 if accumulating else -1)
    try:
        t0 = time.perf_counter()
        cq.cqsa_stream_attn_fwd(host[0], host[1], host[2], cq.CQSA_LAYOUT_BNHD, out, lse, True, Bs, Hs, n_tokens, Ds,
                                True, 0.0, cq.CQSA_F16, C, st, stream)
        wall = time.perf_counter() - t0
    finally:
        cq.cqsa_set_stream_kv_resident_bytes(-1)
    n_q = -(-n_tokens // C)
    flop = 4.0 * Bs * Hs * n_tokens * n_tokens * Ds / 2.0
    copy_gbs = st.h2d_bytes / (st.h2d_ms / 1e3) / 1e9 if st.h2d_ms > 0 else None
    peak, src, _ = _peaks()
    return {"measure": "stream", "workload": f"host-resident streaming, B=1 H=8 N={n_tokens} d=64 fp16 causal, "
            f"token-major pinned Q/K/V/out, {C}-token chunks",
            "schedule": "resident inputs, one launch per query chunk" if st.n_chunks == n_q else
                        "accumulating chunk pairs",
            "wall_s": wall, "tflops": flop / wall / 1e12,
            "compute_s": st.compute_ms / 1e3, "stall_ms": st.stall_ms, "h2d_bytes": st.h2d_bytes,
            "d2h_bytes": st.d2h_bytes, "copy_gbs_overlapped": copy_gbs, "link_h2d_gbs": link_h2d_gbs,
            "copy_frac_of_link": (copy_gbs / link_h2d_gbs) if (copy_gbs and link_h2d_gbs) else None,
            "overlap_wall_over_compute": wall / (st.compute_ms / 1e3) if st.compute_ms > 0 else None,
            "peak_device_bytes": st.peak_device_bytes, "n_units": st.n_chunks,
            "roofline": {"bound": "tensor", "achieved": flop / wall / 1e12, "peak": peak, "unit": "TFLOP/s",
                         "frac": flop / wall / 1e12 / peak, "peak_source": src},
            "link_or_tensor_roofline_frac": (max(st.h2d_bytes / (link_h2d_gbs * 1e9), flop / (peak * 1e12)) / wall
                                             if link_h2d_gbs else None)}


def _host_qkv_token_major(n_tokens, Hs=8, Ds=64):
    import torch
    import synthetic as syn
    shape = (1, n_tokens, Hs, Ds)
    host = [torch.empty(shape, dtype=torch.float16).pin_memory() for _ in range(3)]
    for tid, t in enumerate(host):
        syn.normal(1, Hs, n_tokens, Ds, seed=0, tensor_id=tid, layout=syn.LAYOUT_BNHD, out=t.numpy().view(np.uint16))
    return host


def measure_quorum(cq, dev, n_tokens, acc_on_host=False, npar=1, engine="classic", device_inputs=False):
    """The quorum decomposition; with device_inputs, Q/K/V and the output are device-resident (the chunks
    are read in place) and the call is timed with CUDA events, after one untimed call."""
    import torch
    Hs, Ds, c, D, itr = 8, 64, 31, (0, 1, 3, 8, 12, 18), 1
    host = _host_qkv_token_major(n_tokens, Hs, Ds)
    eng = cq.CQSA_ENGINE_WAVE if engine == "wave" else cq.CQSA_ENGINE_CLASSIC
    if device_inputs:
        qkv = [t.to(dev) for t in host]
        out = torch.empty((1, n_tokens, Hs, Ds), dtype=torch.float16, device=dev)
        lse = torch.empty((1, Hs, n_tokens), dtype=torch.float32, device=dev)
    else:
        qkv = host
        out = torch.empty((1, n_tokens, Hs, Ds), dtype=torch.float16).pin_memory()
        lse = torch.empty((1, Hs, n_tokens), dtype=torch.float32).pin_memory()
    st = cq.cqsa_quorum_stats()
    stream = torch.cuda.current_stream(dev)

    def call():
        cq.cqsa_quorum_attn_fwd_ex(qkv[0], qkv[1], qkv[2], cq.CQSA_LAYOUT_BNHD, not device_inputs, out, lse,
                                   not device_inputs, 1, Hs, n_tokens, Ds, True, 0.0, cq.CQSA_F16, c, D, itr,
                                   acc_on_host=acc_on_host, max_parallel=npar, engine=eng, stats=st, stream=stream)

    mono_s = None
    if device_inputs:
        # the call returns after its own streams drain, so each interval also holds its host-side work
        # (schedule, pool, launches); median of 7
        call()
        samples = _time_events(call, 7, stream)
        ms = statistics.median(samples)
        wall = ms / 1e3
        # the monolithic call on the same problem ([B,H,N,d] copies of the same device inputs)
        qb, kb, vb = (x.permute(0, 2, 1, 3).contiguous() for x in qkv)
        ob = torch.empty_like(qb)
        lb = torch.empty((1, Hs, n_tokens), dtype=torch.float32, device=dev)

        def mono_call():
            cq.cqsa_attn_fwd(qb, kb, vb, ob, lb, 1, Hs, n_tokens, Ds, True, 0.0, cq.CQSA_F16, stream)

        mono_call()
        mono_s = statistics.median(_time_events(mono_call, 7, stream)) / 1e3
        del qb, kb, vb, ob
    else:
        t0 = time.perf_counter()
        call()
        wall = time.perf_counter() - t0
    flop = 4.0 * Hs * n_tokens * n_tokens * Ds / 2.0
    where = "device-resident token-major Q/K/V/out" if device_inputs else "token-major pinned host Q/K/V/out"
    extra = {}
    if mono_s:
        extra = {"mono_tflops": flop / mono_s / 1e12, "over_mono": mono_s / wall,
                 "ms_samples": [round(x, 3) for x in samples]}
    return {"measure": "quorum", "workload": f"cyclic quorum decomposition, B=1 H=8 N={n_tokens} d=64 fp16 causal, "
            f"c={c} interest_set={D} itr={itr}, {where}", "wall_s": wall, **extra,
            "tflops": flop / wall / 1e12, "compute_s": st.compute_ms / 1e3, "copy_s": st.copy_ms / 1e3,
            "copy_bytes": st.copy_bytes, "chunk_tokens": st.chunk_tokens, "subproblems": st.n_subproblems,
            "pairs": st.n_pairs, "chunk_loads": st.n_chunk_loads, "peak_device_bytes": st.peak_device_bytes,
            "accumulator": "host (pinned)" if acc_on_host else "device", "acc_host_bytes": st.acc_host_bytes,
            "max_parallel": npar, "engine": engine, "launches": st.n_launches,
            "inputs": "device-resident (read in place), CUDA events" if device_inputs else "pinned host, wall clock",
            "context": "the pages' own run of this example (unnamed GPU): 2 min 06 s, 31 subproblems"}


def measure_bf16(cq, dev, reps):
    import torch
    import synthetic as syn
    Bb, Hb, Nb, Db = 2, 32, 16384, 128
    qn, kn, vn = syn.qkv(Bb, Hb, Nb, Db, seed=0, dtype=syn.BF16, k_mul=3.0)
    q, k, v = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev) for x in (qn, kn, vn))
    out = torch.empty_like(q)
    lse = torch.empty((Bb, Hb, Nb), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        cq.cqsa_attn_fwd(q, k, v, out, lse, Bb, Hb, Nb, Db, False, 0.0, cq.CQSA_BF16, stream)

    for _ in range(3):
        step()
    ms = []
    for i in range(reps):
        flush.fill_(i & 0xFF)
        ms += _time_events(step, 1, stream)
    flop = 4.0 * Bb * Hb * Nb * Nb * Db
    tf = flop / (statistics.median(ms) / 1e3) / 1e12
    peak, src, _ = _peaks()
    return {"measure": "bf16", "workload": "B=2 H=32 N=16384 d=128 bf16 non-causal, K x3, monolithic",
            "ms_per_step": statistics.median(ms), "tflops": tf,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "peak_source": src, "note": "algorithmic FLOP; the P hi/lo split issues 1.5x the MMA work"}}


def measure_bwd(cq, dev, reps, N=32768, H=8, B=1, D=64, causal=True, bf16=False, k_mul=1.0):
    """Attention backward, by default on the headline shape (B=1 H=8 N=32768 d=64 fp16 causal): the whole
    cqsa_attn_bwd call (D = rowsum(dO * O), zeroing the dQ accumulator, the tcgen05 kernel, the dQ
    conversion) timed with CUDA events, inputs and forward outputs resident. Algorithmic FLOP: five
    products of 2*N*N*d per head (S, dP, dV, dK, dQ), halved by the causal mask = 2.5x the forward."""
    import torch
    import synthetic as syn
    dt = syn.BF16 if bf16 else syn.F16
    tdt = torch.bfloat16 if bf16 else torch.float16
    code = cq.CQSA_BF16 if bf16 else cq.CQSA_F16
    qn, kn, vn = syn.qkv(B, H, N, D, seed=0, dtype=dt, k_mul=k_mul)
    gn = syn.normal(B, H, N, D, seed=0, tensor_id=syn.TID_DO, dtype=dt)
    q, k, v, g = (torch.from_numpy(x.view(np.int16)).view(tdt).to(dev) for x in (qn, kn, vn, gn))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    cq.cqsa_attn_fwd(q, k, v, out, lse, B, H, N, D, causal, 0.0, code, stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = cq.cqsa_attn_bwd_workspace_size(B, H, N, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        cq.cqsa_attn_bwd(q, k, v, out, g, lse, dq, dk, dv, ws, ws_bytes, B, H, N, D, causal, 0.0, code, stream)

    for _ in range(3):
        step()
    ms = []
    for i in range(reps):
        flush.fill_(i & 0xFF)
        ms += _time_events(step, 1, stream)
    flop = 2.5 * 4.0 * B * H * N * N * D / (2 if causal else 1)
    tf = flop / (statistics.median(ms) / 1e3) / 1e12
    peak, src, _ = _peaks()
    kind = ("bf16" if bf16 else "fp16") + (" causal" if causal else " non-causal")
    kind += f", K x{k_mul:g}" if k_mul != 1.0 else ""
    return {"measure": "bwd", "workload": f"B={B} H={H} N={N} d={D} {kind} backward (dq, dk, dv)",
            "ms_per_step": statistics.median(ms), "ms_min": min(ms), "tflops": tf,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "peak_source": src, "note": "algorithmic FLOP of the five products, whole call"}}


def measure_copy_series(dev, seconds=15.0):
    """Host-to-device copy rate over time: 256 MiB copies alternating between a freshly pinned buffer and
    pinned buffers filled by the synthetic generator (as the streaming workload's are), to tell host-side
    contention (both move together) from an effect of the buffers (they differ)."""
    import torch
    import synthetic as syn
    reg = 256 << 20
    dbuf = torch.empty(reg, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream(dev)
    fresh = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    fresh.numpy()[:] = 7
    gen = []
    for tid in range(3):
        t = torch.empty((1, 1 << 20, 8, 64), dtype=torch.float16).pin_memory()
        syn.normal(1, 8, 1 << 20, 64, seed=0, tensor_id=tid, layout=syn.LAYOUT_BNHD, out=t.numpy().view(np.uint16))
        gen.append(t.view(-1).view(torch.uint8))

    def rate(src):
        with torch.cuda.stream(side):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(side)
            dbuf.copy_(src, non_blocking=True)
            b.record(side)
        side.synchronize()
        return reg / (a.elapsed_time(b) / 1e3) / 1e9

    t0 = time.perf_counter()
    f, g = [], []
    i = 0
    while time.perf_counter() - t0 < seconds:
        off = (i % 4) * reg
        f.append(rate(fresh[off:off + reg]))
        g.append(rate(gen[i % 3][off:off + reg]))
        i += 1
    fa, ga = np.array(f), np.array(g)
    return {"measure": "copy_series", "copies_each": len(f), "seconds": seconds,
            "fresh_gbs": {"median": float(np.median(fa)), "min": float(fa.min()), "max": float(fa.max()),
                          "frac_above_150": float(np.mean(fa > 150))},
            "generated_gbs": {"median": float(np.median(ga)), "min": float(ga.min()), "max": float(ga.max()),
                              "frac_above_150": float(np.mean(ga > 150))},
            "correlation": float(np.corrcoef(fa, ga)[0, 1]) if len(f) > 2 else None,
            "method": "alternating 256 MiB cudaMemcpyAsync copies, CUDA events per copy"}


def measure_stream_bwd(cq, dev, N=131072, C=16384, H=8):
    """The host-resident backward (cqsa_stream_attn_bwd: pinned host q, k, v, out, dout, lse in, dq, dk, dv
    out, 16,384-token chunks, copies double-buffered beside the kernels) against the device-resident
    backward of the same problem (cqsa_attn_bwd, CUDA events): wall time, TFLOP/s and their ratio."""
    import torch
    import synthetic as syn
    B, D = 1, 64
    qn, kn, vn = syn.qkv(B, H, N, D, seed=0)
    gn = syn.normal(B, H, N, D, seed=0, tensor_id=syn.TID_DO)
    q, k, v, g = (torch.from_numpy(x.view(np.int16)).view(torch.float16).to(dev) for x in (qn, kn, vn, gn))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    cq.cqsa_attn_fwd(q, k, v, out, lse, B, H, N, D, True, 0.0, cq.CQSA_F16, stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = cq.cqsa_attn_bwd_workspace_size(B, H, N, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def dev_step():
        cq.cqsa_attn_bwd(q, k, v, out, g, lse, dq, dk, dv, ws, ws_bytes, B, H, N, D, True, 0.0, cq.CQSA_F16, stream)

    dev_step()
    dev_ms = statistics.median(_time_events(dev_step, 3, stream))
    host = [t.cpu().pin_memory() for t in (q, k, v, out, g, lse)]
    grads = [torch.empty((B, H, N, D), dtype=torch.float16).pin_memory() for _ in range(3)]

    def host_step():
        return cq.cqsa_stream_attn_bwd_ex(*host, *grads, B, H, N, D, True, 0.0, cq.CQSA_F16, C, None, stream)

    host_step()
    runs = []
    for _ in range(3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        st = host_step()
        runs.append((time.perf_counter() - t0, st))
    runs.sort(key=lambda r: r[0])
    wall, st = runs[len(runs) // 2]
    flop = 2.5 * 4.0 * B * H * N * N * D / 2
    comp_s = st.compute_ms / 1e3
    return {"measure": "stream_bwd", "workload": f"host-resident backward, B=1 H={H} N={N} d=64 fp16 causal, "
            f"{C}-token chunks, pinned host tensors", "wall_s": wall, "tflops": flop / wall / 1e12,
            "compute_s": comp_s, "wall_over_compute": wall / comp_s if comp_s > 0 else None,
            "stall_ms": st.stall_ms, "h2d_bytes": st.h2d_bytes, "d2h_bytes": st.d2h_bytes,
            "copy_gbs": st.h2d_bytes / (st.h2d_ms / 1e3) / 1e9 if st.h2d_ms > 0 else None,
            "n_pairs": st.n_chunks, "peak_device_bytes": st.peak_device_bytes,
            "device_resident_ms": dev_ms, "device_resident_tflops": flop / (dev_ms / 1e3) / 1e12,
            "wall_over_device_resident": wall / (dev_ms / 1e3),
            "numa_nodes_of_host_pages": _numa_nodes(host[0]),
            "note": "resident schedule (inputs copied once and kept): one chunk-pair launch per key chunk over "
                    "every query it meets, on up to four streams; n_pairs counts those launches, compute_s is "
                    "the union of the call's kernel intervals (D, launches, output casts)"}


def _numa_nodes(t, samples=64):
    """NUMA nodes of a sample of a host tensor's pages (move_pages with no target nodes reports them);
    {} where the system call is unavailable."""
    import ctypes
    import platform
    nr = {"aarch64": 239, "x86_64": 279}.get(platform.machine())
    if nr is None:
        return {}
    try:
        libc = ctypes.CDLL(None, use_errno=True)
        page = os.sysconf("SC_PAGE_SIZE")
        base, nbytes = t.data_ptr(), t.numel() * t.element_size()
        addrs = [(base + (nbytes - 1) * k // max(1, samples - 1)) & ~(page - 1) for k in range(samples)]
        pages = (ctypes.c_void_p * samples)(*addrs)
        status = (ctypes.c_int * samples)()
        if libc.syscall(nr, 0, samples, pages, None, status, 0) != 0:
            return {}
        nodes = {}
        for st in status:
            nodes[str(st)] = nodes.get(str(st), 0) + 1
        return nodes
    except (OSError, AttributeError, ValueError):
        return {}


def measure_link_driver_shaped(cq, dev, host, chunk_tokens, reps=6):
    """Host-to-device copies shaped like the streaming driver's: one contiguous chunk of the token-major
    host tensors (chunk_tokens x 8 heads x 64 x 2 bytes) per cudaMemcpyAsync on a non-blocking stream,
    from the workload's own pinned buffers, alone and while attention kernels run on another stream."""
    import torch
    per_tok = 8 * 64 * 2
    nbytes = chunk_tokens * per_tok
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream(dev)
    n_chunks = host[1].shape[1] // chunk_tokens
    flat = [t.view(-1).view(torch.uint8) for t in host[1:]]

    def copies():
        res = []
        for r in range(reps):
            src = flat[r % 2][(r % n_chunks) * nbytes:(r % n_chunks + 1) * nbytes]
            res += _time_events(lambda: dbuf.copy_(src, non_blocking=True), 1, side)
        return res

    with torch.cuda.stream(side):
        alone = copies()
    # the same copies beside the headline attention kernel on the default stream
    import synthetic as syn
    qn, kn, vn = syn.qkv(1, 8, 32768, 64, seed=0)
    q, k, v = (torch.from_numpy(x.view(np.int16)).view(torch.float16).to(dev) for x in (qn, kn, vn))
    out = torch.empty_like(q)
    lse = torch.empty((1, 8, 32768), dtype=torch.float32, device=dev)
    main = torch.cuda.current_stream(dev)
    for _ in range(3 * reps):
        cq.cqsa_attn_fwd(q, k, v, out, lse, 1, 8, 32768, 64, True, 0.0, cq.CQSA_F16, main)
    with torch.cuda.stream(side):
        busy = copies()
    torch.cuda.synchronize()
    gbs = lambda ms: [nbytes / (m / 1e3) / 1e9 for m in ms]  # noqa: E731
    return {"copy_bytes": nbytes, "h2d_gbs_alone": gbs(alone), "h2d_gbs_beside_attention": gbs(busy),
            "numa_nodes_of_host_pages": _numa_nodes(host[1]),
            "method": f"{reps} plain cudaMemcpyAsync copies of one {chunk_tokens}-token chunk each from the "
                      "workload's pinned token-major K/V, non-blocking stream, CUDA events per copy"}


def run_secondary(cq, dev, args):
    """Secondary lines of the other workloads (each with its own CUDA-event timing, clocks and roofline):
    the bf16 d=128 forward, the LSE merge of the chunked workload, the backward, the host link probed
    as a 1 GiB copy and as the streaming driver's copies, and the host-resident streaming workload."""
    import torch
    res = {}
    reps = 10

    def run(name, fn):
        t0 = time.perf_counter()
        with ClockSampler(dev.index if dev.index is not None else 0) as clk:
            try:
                r = fn()
            except Exception as e:  # noqa: BLE001  (a failed secondary line must not hide the headline)
                r = {"error": f"{type(e).__name__}: {e}"}
        r["clocks"] = clk.summary()
        r["host_s"] = time.perf_counter() - t0
        res[name] = r
        torch.cuda.empty_cache()

    run("bf16_d128", lambda: measure_bf16(cq, dev, reps))
    run("merge_131k", lambda: measure_merge(cq, dev, reps))
    run("bwd_32k", lambda: measure_bwd(cq, dev, reps))
    run("bwd_bf16_d128", lambda: measure_bwd(cq, dev, max(3, reps // 2), N=16384, H=32, B=2, D=128, causal=False,
                                             bf16=True, k_mul=3.0))
    run("stream_bwd_131k", lambda: measure_stream_bwd(cq, dev))
    run("quorum_wave_262k", lambda: measure_quorum(cq, dev, 262_144, engine="wave", device_inputs=True))
    run("link_1gib", lambda: measure_link(dev, 5))
    if args.secondary == "all":
        link = res["link_1gib"].get("h2d_gbs")
        host = _host_qkv_token_major(args.n)
        run("link_driver_shaped", lambda: measure_link_driver_shaped(cq, dev, host, 262_144))
        run("stream_4m", lambda: measure_stream(cq, dev, args.n, link, host=host))
        del host
    rc, code, _ = cq.cqsa_device_error()
    res["device_error_free"] = rc == cq.CQSA_OK
    return res


def run_measure(args):
    import torch
    world, rank, local = _dist()
    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_long_context_tcgen05_gb300 as cq
    reps = max(5, min(args.steps, 20))
    if args.measure == "merge":
        line = measure_merge(cq, dev, reps)
    elif args.measure == "link":
        line = measure_link(dev, reps)
    elif args.measure == "stream":
        link = measure_link(dev, 5)
        line = measure_stream(cq, dev, args.n, link["h2d_gbs"])
    elif args.measure == "quorum":
        line = measure_quorum(cq, dev, args.n, acc_on_host=args.acc_on_host, npar=args.max_parallel,
                              engine=args.engine, device_inputs=args.device_inputs)
    elif args.measure == "bwd":
        line = measure_bwd(cq, dev, reps, N=args.bwd_n, H=args.bwd_h, B=args.bwd_b, D=args.bwd_d,
                           causal=not args.bwd_noncausal, bf16=args.bwd_bf16, k_mul=args.bwd_kmul)
    elif args.measure == "stream-bwd":
        line = measure_stream_bwd(cq, dev)
    elif args.measure == "copy-series":
        line = measure_copy_series(dev)
    else:
        line = measure_bf16(cq, dev, reps)
    rc, code, _ = cq.cqsa_device_error()
    line["device_error_free"] = rc == cq.CQSA_OK
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--measure", choices=("merge", "link", "stream", "bf16", "quorum", "bwd", "stream-bwd",
                                          "copy-series"),
                    default=None)
    ap.add_argument("--n", type=int, default=4_000_000, help="tokens for --measure stream / quorum")
    ap.add_argument("--acc-on-host", action="store_true", help="--measure quorum with the host accumulator")
    ap.add_argument("--max-parallel", type=int, default=1, help="--measure quorum: parallel subproblem lanes")
    ap.add_argument("--engine", choices=("classic", "wave"), default="classic", help="--measure quorum: engine")
    ap.add_argument("--device-inputs", action="store_true", help="--measure quorum: device-resident Q/K/V/out")
    ap.add_argument("--bwd-n", type=int, default=32768, help="--measure bwd: tokens")
    ap.add_argument("--bwd-h", type=int, default=8, help="--measure bwd: heads")
    ap.add_argument("--bwd-b", type=int, default=1, help="--measure bwd: batch")
    ap.add_argument("--bwd-d", type=int, default=64, choices=(64, 128), help="--measure bwd: head dim")
    ap.add_argument("--bwd-bf16", action="store_true", help="--measure bwd: bf16 instead of fp16")
    ap.add_argument("--bwd-noncausal", action="store_true", help="--measure bwd: no causal mask")
    ap.add_argument("--bwd-kmul", type=float, default=1.0, help="--measure bwd: scale of K (peaked rows)")
    ap.add_argument("--secondary", choices=("all", "fast", "none"), default="all",
                    help="secondary lines in the headline JSON: all, fast (no host-streaming workload), none")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.measure:
        return run_measure(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
