"""Benchmark of the GB300 logprob / greedy-acceptance epilogue.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config large|spec|decode|wide|tiny]
                [--impl reference] [--no-cpu-baseline] [--no-per-workload]

One step = one lp_run (prepare, persistent stream and record kernels) over the whole
logit block of the chosen workload, inputs resident in HBM.  L2 is flushed
(a 256 MiB device write) before every timed step, outside the timed events.
Rank 0 prints one JSON line.  ``--impl reference`` times the CPU oracle (the
reference arm) on the host cores instead.
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

import workloads as W  # noqa: E402

DESCRIPTIONS = {
    "tiny": "tiny: 6 rows, V=1,000 (stride 1,024) FP32, one k=3 verify group + an explicit-id row + an unrequested row",
    "decode": "decode: 64 rows x V=151,936 (stride 152,064) BF16, k=0, K=20, sampled tokens",
    "spec": "spec verify: 128 groups x (k=3 + 1) = 512 rows x V=248,320 (stride 248,448) BF16, p_accept 0.7, "
            "half K=20 / half 128 explicit ids",
    "large": "large verify: 256 groups x (k=7 + 1) = 2,048 rows x V=262,144 FP32 (BF16-rounded N(0,4)), p_accept 0.6, "
             "64 natural K~U{0..20}, 64 explicit ids U{1..128}, 128 unrequested",
    "wide": "wide-vocab: 4 rows x V=1,048,576 (stride 1,048,704) BF16, one k=3 group, 64-way tie at the max, K=20",
}
FLUSH_BYTES = 256 << 20
METRIC = "verify-epilogue logit rows/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (about 8 TB/s); the roofline's peak is the measured copy


def kernel_source_hash() -> str:
    """SHA-256 of the stream kernel's sources: a DRAM-traffic figure taken by ncu is
    only reported while the kernel is unchanged since the capture."""
    import hashlib
    h = hashlib.sha256()
    for rel in ("logprob_epilogue_gb300/csrc/lp_kernels.cu", "logprob_epilogue_gb300/csrc/lp_internal.h"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(config: str):
    """DRAM bytes per launch of lp_stream_kernel from the committed ncu summary of
    this workload (profiles/lp_stream_kernel_<config>_dram.txt), or None when there
    is none or the kernel changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"lp_stream_kernel_{config}_dram.txt")
    try:
        fields = {}
        for ln in open(path):
            if ":" in ln and not ln.startswith("#"):
                k, v = ln.split(":", 1)
                fields[k.strip()] = v.strip()
        if fields.get("kernel_source_sha256") != kernel_source_hash():
            return None
        return int(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def algorithmic_bytes(w: W.Workload, accepted: np.ndarray) -> dict:
    """Bytes the epilogue must move for one run, given the accepted counts.

    Logit rows actually read (V * element size each), one 32-byte sector per
    gathered logit (chosen token and explicit ids of emitted requested rows),
    the 258-word record of each emitted requested row, and the small per-group
    and per-row inputs and outputs.
    """
    rows_read = 0
    rec_rows = 0
    gathers = 0
    G = w.groups
    for g in range(G):
        r0, r1 = int(w.group_indptr[g]), int(w.group_indptr[g + 1])
        k = r1 - r0 - 1
        req = int(w.requested[g]) != 0
        need = req or k >= 1 or int(w.sampled_tokens[g]) < 0
        if not need:
            continue
        emitted = int(accepted[g]) + 1
        rows_read += emitted
        if req:
            rec_rows += emitted
            cnt = int(w.id_counts[g])
            gathers += emitted * (1 + (cnt if cnt > 0 else 0))
    logit_bytes = rows_read * w.V * w.elt
    small = 4 * (G + 1) + 4 * w.rows * 2 + 4 * G * 6 + 4 * 128 * int((w.id_counts > 0).sum())
    total = logit_bytes + gathers * 32 + rec_rows * 258 * 4 + small
    return {"total": total, "logit_bytes": logit_bytes, "rows_read": rows_read, "records": rec_rows,
            "gathers": gathers}


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.idx)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

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
        if self._t:
            self._t.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl != "reference" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device])
        else:
            pg.barrier()


def max_over_ranks(pg, value: float, device=None) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def time_oracle(w: W.Workload, threads: int, min_seconds: float = 10.0, max_passes: int = 400):
    """Times the oracle as it stands on whole-block passes over the workload,
    repeated until about `min_seconds` of host time (at least one pass)."""
    import oracle
    x = w.logits_f32()
    passes = 0
    t0 = time.perf_counter()
    while True:
        oracle.epilogue(x, w.V, **w.inputs(), k_max=w.k_max, threads=threads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            break
    return passes * w.rows / dt, dt, f"{passes} whole-block passes ({w.rows} rows, {w.groups} groups each)"


def run_reference(args, world, rank, local, pg):
    if rank != 0:
        return 0
    w = W.make(args.config)
    cores = os.cpu_count() or 1
    import oracle
    oracle.build()
    x = w.logits_f32()
    for _ in range(max(args.warmup, 0) and 1):
        oracle.epilogue(x, w.V, **w.inputs(), k_max=w.k_max, threads=cores)
    times = []
    steps = max(1, min(args.steps, 5))
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.epilogue(x, w.V, **w.inputs(), k_max=w.k_max, threads=cores)
        times.append(time.perf_counter() - t0)
    per = sum(times) / len(times)
    value = w.rows / per
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.config]},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"whole block per step ({w.rows} rows), {steps} steps"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class Flusher:
    """Evicts the inputs from L2 before a timed step: writes a 256 MiB buffer, then
    (mode "write+read", the default) reads another 256 MiB buffer so that the
    dirty lines of that write are written back before the step, not during it."""

    MODE = os.environ.get("LP_BENCH_FLUSH", "write+read")

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.clean = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)  # summed without a cast

    def __call__(self, i):
        import torch
        if self.MODE == "none":
            return
        self.buf.fill_(i)
        if self.MODE == "write+read":
            self.last = self.clean.sum()


def bench_device(w: W.Workload, steps: int, warmup: int, device: int, staging: bool = True, clip=None):
    """Times lp_run on device-resident inputs; returns per-step durations (s) and outputs.
    ``clip``: optional (eos_tokens, budgets) commit-clipping inputs."""
    import torch
    import logprob_epilogue_gb300 as lpe
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    dev = torch.device("cuda", device)
    plan = lpe.Plan(max_rows=w.rows, max_groups=w.groups, k_max=w.k_max, V=w.V, V_padded=w.Vp, dtype=w.dtype,
                    k_alt_max=20, max_ids=128, device=device, host_staging=staging)
    if w.dtype == "bf16":
        logits = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16)
    else:
        logits = torch.from_numpy(w.logits)
    ti = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)  # noqa: E731
    ins = dict(logits=logits.to(dev), group_indptr=ti(w.group_indptr), draft_tokens=ti(w.draft_tokens),
               sampled_tokens=ti(w.sampled_tokens), requested=ti(w.requested), top_k=ti(w.top_k),
               token_ids=ti(w.token_ids.reshape(-1)), id_counts=ti(w.id_counts))
    outs = dict(records=torch.zeros((w.rows, 258), dtype=torch.int32, device=dev),
                accepted=torch.zeros(w.groups, dtype=torch.int32, device=dev),
                emitted_tokens=torch.zeros(w.rows, dtype=torch.int32, device=dev),
                lse_out=torch.zeros(w.rows, dtype=torch.float32, device=dev),
                status=torch.zeros(1, dtype=torch.int32, device=dev))
    plan.bind(**ins, **outs)
    if clip is not None:
        ins["eos_tokens"], ins["budgets"] = ti(clip[0]), ti(clip[1])
        plan.bind_clip(eos_tokens=ins["eos_tokens"], budgets=ins["budgets"])
    flush = Flusher(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        flush(1)
        plan.run(stream)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    return plan, ins, outs, flush, starts, ends, stream


def bench_score(device: int, peak: float, steps: int = 200, warmup: int = 5) -> dict:
    """Times prompt scoring (lp_score) of the 512 x 151,936 BF16 prompt workload
    on device-resident inputs; algorithmic bytes = the logits of the rows with a
    valid target + the targets + the 43-word records."""
    import torch
    import logprob_epilogue_gb300 as lpe
    w = W.prompt()
    dev = torch.device("cuda", device)
    tg_np = np.asarray(w.meta["targets"], np.int32)
    plan = lpe.Plan(max_rows=w.rows, max_groups=w.rows, k_max=0, V=w.V, V_padded=w.Vp, dtype=w.dtype,
                    k_alt_max=20, max_ids=128, device=device)
    logits = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16).to(dev)
    tg = torch.from_numpy(tg_np).to(dev)
    rec = torch.zeros((w.rows, lpe.SCORE_WORDS), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = Flusher(dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        flush(i)
        plan.score(logits=logits, target_tokens=tg, records=rec, status=st, stream=stream)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush(i)
        starts[i].record(stream)
        plan.score(logits=logits, target_tokens=tg, records=rec, status=st, stream=stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if int(st.item()) != 0:
        raise RuntimeError(f"prompt scoring status {int(st.item()):#x}")
    m = statistics.mean(a.elapsed_time(b) * 1e-3 for a, b in zip(starts, ends))
    valid = int(((tg_np >= 0) & (tg_np < w.V)).sum())
    nbytes = valid * w.V * 2 + w.rows * 4 + w.rows * lpe.SCORE_WORDS * 4
    plan.close()
    return {"rows_per_s": w.rows / m, "us_per_step": m * 1e6, "hbm_gbs": nbytes / m / 1e9,
            "frac": nbytes / m / 1e9 / peak, "frac_of_nominal": nbytes / m / 1e9 / NOMINAL_HBM_GBS,
            "rows_read": valid, "dtype": w.dtype}


def bench_chain(device: int, peak: float, steps: int = 100, warmup: int = 5) -> dict:
    """Times stochastic chain verification (lp_chain_verify) of the chain
    workload: 128 groups x (3 drafts + 1) rows x 248,320 BF16, with FP32 draft
    laws.  Algorithmic bytes: every row read once for its lse, and the drawn row
    of each group read again for its weights (logits, plus the draft law when
    the draw is from the residual), plus the small per-row and per-group
    vectors."""
    import torch
    import logprob_epilogue_gb300 as lpe
    w = W.chain()
    dev = torch.device("cuda", device)
    plan = lpe.Plan(max_rows=w.rows, max_groups=w.groups, k_max=w.k_max, V=w.V, V_padded=w.Vp, dtype=w.dtype,
                    device=device)
    ti = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)  # noqa: E731
    tf = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)  # noqa: E731
    m = w.meta
    ins = dict(logits=torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16).to(dev),
               group_indptr=ti(w.group_indptr), draft_tokens=ti(w.draft_tokens), draft_probs=tf(m["draft_probs"]),
               temperature=tf(m["temperature"]), u=tf(m["u"]), r=tf(m["r"]))
    outs = dict(accepted=torch.zeros(w.groups, dtype=torch.int32, device=dev),
                emitted=torch.zeros(w.rows, dtype=torch.int32, device=dev),
                status=torch.zeros(1, dtype=torch.int32, device=dev))
    flush = Flusher(dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        flush(i)
        plan.chain_verify(**ins, **outs, stream=stream)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush(i)
        starts[i].record(stream)
        plan.chain_verify(**ins, **outs, stream=stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if int(outs["status"].item()) != 0:
        raise RuntimeError(f"chain verification status {int(outs['status'].item()):#x}")
    t = statistics.median(a.elapsed_time(b) * 1e-3 for a, b in zip(starts, ends))
    acc = outs["accepted"].cpu().numpy()
    k = w.k_max
    rows_read = int((acc + 1).sum())
    residual = int((acc < k).sum())
    nbytes = (rows_read + w.groups) * w.V * 2 + residual * w.V * 4 + w.rows * 16 + w.groups * 16
    plan.close()
    return {"rows_per_s": w.rows / t, "us_per_step": t * 1e6, "hbm_gbs": nbytes / t / 1e9,
            "frac": nbytes / t / 1e9 / peak, "frac_of_nominal": nbytes / t / 1e9 / NOMINAL_HBM_GBS,
            "rows_read": rows_read, "dtype": w.dtype,
            "accepted_mean": float(acc.mean())}


def run_e2e(args, w, plan, stream, dev, pg, local, world, accepted):
    """Same metric through lp_run_host: pinned host buffers, H2D and D2H inside the timed region."""
    import torch
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731

    harr = dict(logits=pin(w.logits), group_indptr=pin(w.group_indptr), draft_tokens=pin(w.draft_tokens),
                sampled_tokens=pin(w.sampled_tokens), requested=pin(w.requested), top_k=pin(w.top_k),
                token_ids=pin(w.token_ids), id_counts=pin(w.id_counts),
                records=pin(np.zeros((w.rows, 258), np.int32)), accepted=pin(np.zeros(w.groups, np.int32)),
                emitted_tokens=pin(np.zeros(w.rows, np.int32)), lse_out=pin(np.zeros(w.rows, np.float32)),
                status=pin(np.zeros(1, np.int32)))
    h2d, d2h = plan.host_bytes(harr)
    # pinned logits are read in place: what crosses the link is the rows the
    # run reads and the gathered logits, not the whole block
    in_place = h2d < w.rows * w.Vp * w.elt
    if in_place:
        ab = algorithmic_bytes(w, accepted)
        h2d += ab["logit_bytes"] + ab["gathers"] * 32
    for _ in range(3):
        plan.run_host(harr, stream)
    torch.cuda.synchronize(dev)
    barrier(pg, local if pg else None)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        plan.run_host(harr, stream)
        stream.synchronize()
    e2e_t = (time.perf_counter() - t0) / args.e2e_steps
    e2e_t = max_over_ranks(pg, e2e_t, dev if pg else None)
    e2e_ok = np.array_equal(harr["accepted"].numpy(), accepted)
    del harr
    return {"value": world * w.rows / e2e_t, "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_t * 1e3, "matches_device_run": bool(e2e_ok),
            "logits": "read in place from pinned host memory (the rows the run reads)" if in_place
                      else "copied to device staging"}



def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="large", choices=list(DESCRIPTIONS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--groups", type=int, default=0,
                    help="verify groups of the timed workload (0: its own count); a smaller block for profiling")
    args = ap.parse_args()
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, world, rank, local, pg)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import logprob_epilogue_gb300 as lpe
    from logprob_epilogue_gb300 import build as B
    if rank == 0 or world == 1:
        B.build()
    barrier(pg, local if pg else None)
    lpe.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    w = W.make(args.config, **({"groups": args.groups} if args.groups > 0 and args.config in ("spec", "large") else {}))
    plan, ins, outs, flush, starts, ends, stream = bench_device(w, args.steps, args.warmup, local,
                                                               staging=not args.no_e2e)

    # ---- timed region: device-resident inputs, L2 flushed before each step
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES", "").isdigit() else local)
    barrier(pg, local if pg else None)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.2)
    for i in range(args.steps):
        flush(i)
        starts[i].record(stream)
        plan.run(stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(pg, local if pg else None)
    durs = [s.elapsed_time(e) * 1e-3 for s, e in zip(starts, ends)]
    total = sum(durs)
    total = max_over_ranks(pg, total, dev if pg else None)
    per_step = total / args.steps
    value = world * w.rows / per_step

    accepted = outs["accepted"].cpu().numpy()
    status = int(outs["status"].cpu().numpy().view(np.uint32)[0])
    ab = algorithmic_bytes(w, accepted)
    mean_launch = statistics.mean(durs)
    achieved_gbs = ab["total"] / mean_launch / 1e9
    peak, peak_kind = peaks()

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, plan, stream, dev, pg, local, world, accepted)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.config], "logits_dtype": w.dtype,
                   "l2": f"flushed before every timed step, outside the events ({Flusher.MODE}: 256 MiB write"
                         + (", then a 256 MiB read so its write-back completes before the step)" if Flusher.MODE == "write+read" else ")"),
                   "rows_read_per_step": ab["rows_read"], "parallelism": f"replicas x{world}"},
        "hbm_gbs": achieved_gbs,
        "rows_read_per_s": world * ab["rows_read"] / per_step,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak, "frac_of_nominal": achieved_gbs / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS, "traffic": measured_traffic(args.config),
                     "kernel": "lp_stream_kernel (timed with lp_prepare_kernel: one lp_run)",
                     "algorithmic_bytes_per_launch": ab["total"], "peak_source": peak_kind},
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,  # lp_prepare_kernel, lp_stream_kernel and lp_record_kernel per lp_run
        "clocks": clocks,
        "status": status,
        "median_launch_us": statistics.median(durs) * 1e6,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        v, dt, sample = time_oracle(w, cores)
        v1, dt1, sample1 = time_oracle(w, 1, min_seconds=2.0, max_passes=1)
        line["cpu_baseline"] = {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle",
                                "sample": sample, "seconds": dt,
                                "single_thread": {"value": v1, "unit": "rows/s", "cores": 1, "sample": sample1,
                                                  "seconds": dt1}}
    plan.close()
    del ins, outs
    if rank == 0 and not args.no_per_workload:
        per = {}
        # the other workloads, and the spec block with commit clipping (seeded
        # EOS tokens and output budgets, every case of the rule)
        cases = [(name, name, None) for name in DESCRIPTIONS if name != args.config]
        cases.append(("spec_clipped", "spec", 5))
        for name, base, clip_seed in cases:
            wn = W.make(base)
            clip = None if clip_seed is None else W.commit_clip(wn, clip_seed)
            p2, i2, o2, fl2, st2, en2, s2 = bench_device(wn, 200, 5, local, staging=False, clip=clip)
            for i in range(200):
                fl2(i)
                st2[i].record(s2)
                p2.run(s2)
                en2[i].record(s2)
            torch.cuda.synchronize(dev)
            d2 = [a.elapsed_time(b) * 1e-3 for a, b in zip(st2, en2)]
            abn = algorithmic_bytes(wn, o2["accepted"].cpu().numpy())
            m2 = statistics.mean(d2)
            per[name] = {"rows_per_s": wn.rows / m2, "us_per_step": m2 * 1e6,
                         "hbm_gbs": abn["total"] / m2 / 1e9, "frac": abn["total"] / m2 / 1e9 / peak,
                         "frac_of_nominal": abn["total"] / m2 / 1e9 / NOMINAL_HBM_GBS,
                         "rows_read": abn["rows_read"], "dtype": wn.dtype}
            p2.close()
            del i2, o2, fl2
        per["prompt_score"] = bench_score(local, peak)
        per["chain"] = bench_chain(local, peak)
        line["per_workload"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
