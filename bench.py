"""Benchmark of the fused KIVI decode step on one GPU (or N replicas).

A step is one serving decode step over the pages' decode shape (VeloxQuant-MLX
changelog v0.42.0 "Added": B=1, H=32, D=128, b=2, g=32, S_q=1; S_kv=65536,
the long end of its sweep) with the KIVI cache of changelog v0.8.0 (fp16
residual window of 32 tokens): append the new token's K/V to every sequence
(flushing a group to 2-bit codes whenever the residual fills) and run the
fused decode-attend over the whole cache.

Prints one JSON line.  `value` is microseconds per step (lower is better),
device-timed with CUDA events over K back-to-back steps that rotate over
enough identical cache copies to exceed 4x L2, so every step streams its
cache from HBM.  The roofline object reports the decode kernel's achieved
HBM bandwidth over the algorithmic bytes (packed codes + fp16 scale/zero
planes + fp16 residual + q + out).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --report [WORKLOAD ...]    # secondary figures, see run_report
  python bench.py --profile-decode WORKLOAD N  # N decodes of one cache (ncu)

The timed region repeats passes of exactly K steps until about 0.6 s of
device time has elapsed (so that the clock sampler sees the load); `value` is
the median pass's time per step, with the 10th and 90th percentiles beside
it.  The same line carries `targets`: the decode (and, for the 4-bit
workload, the 512-token append) of every workload with S_kv >= 32768 or
served in batches, each with its algorithmic bytes and HBM fraction.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused 2-bit KV decode-attend: µs/step and HBM GB/s (% of GB300 peak)"
UNIT = "us/step"
DEFAULT_WORKLOAD = "pages_S65536"
# GB300's nominal HBM3e bandwidth (about 8 TB/s); fractions against it are
# reported beside the ones against the measured copy bandwidth
NOMINAL_HBM_GBS = 8000.0
# device seconds the sustained timed region lasts at least
SUSTAIN_S = 0.6
# the decode workloads reported in `targets` (S_kv >= 32768 or batched)
TARGET_WORKLOADS = ("pages_S32768", "gqa_serving", "int4_append",
                    "ragged_long")


# ---------------------------------------------------------------------------
# byte accounting (the roofline numerator)
# ---------------------------------------------------------------------------

def decode_bytes(w, seq_lens):
    """Algorithmic bytes of one fused decode over caches of the given lengths:
    per (b, h_kv): T_q * (2 packed rows + fp16 K scale/zero per token + fp16
    V scale/zero per token) + n_res * fp16 K and V rows + q + out."""
    D, g, bits, R = w.D, w.group, w.bits, w.residual
    row = D * bits // 8
    per_q_tok = 2 * row + (2 * D * 2) / g + 2 * (D // g) * 2
    gq = w.H_q // w.H_kv
    total = 0.0
    for S in seq_lens:
        Tq = 0 if S < R else g * ((S - R) // g)
        nres = S - Tq
        total += w.H_kv * (Tq * per_q_tok + nres * D * 4 + gq * D * 2 + gq * D * 4)
    return int(total)


def append_bytes(w, n_new):
    """Algorithmic bytes of appending n_new tokens per sequence without a
    flush: read the new fp16 K/V rows, write them to the residual ring."""
    return w.B * w.H_kv * n_new * w.D * 2 * 2 * 2


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index, self.period_ms = index, period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        time.sleep(0.1)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


DECODE_KERNEL_SOURCES = ("bit_kv_cache_05_gb300/csrc/decode_mma.cuh",
                         "bit_kv_cache_05_gb300/csrc/decode_mma.cu",
                         "bit_kv_cache_05_gb300/csrc/bulk_pipe.cuh")


def decode_kernel_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes (read + write) of one decode launch from the committed ncu
    summary, or None when there is none for this workload or the kernel
    source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_source_sha") != decode_kernel_hash():
        return None
    return int(entry["dram_bytes_per_launch"])


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_steps(w, budget_s: float = 12.0, max_steps: int = 8, inputs=None):
    """Time the CPU oracle on the same step (append one token per sequence,
    then decode-attend every head) on a bounded sample: whole steps until
    `budget_s` seconds of stepping or `max_steps` steps.  Returns
    (us_per_step, steps, setup_s)."""
    import numpy as np
    import torch
    import oracle
    from bit_kv_cache_05_gb300 import synth
    t0 = time.perf_counter()
    if inputs is None:
        inputs = synth.make_inputs(w, device="cpu")
    K = inputs["K"].cpu().numpy()
    V = inputs["V"].cpu().numpy()
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, w.bits, w.group,
                            w.residual, w.max_seq + max_steps + 1)
    oc.quantize(K, V, w.seq_lens)
    K1, V1, q = synth.decode_tokens(w, max_steps, device="cpu")
    K1, V1, q = K1.numpy(), V1.numpy(), q.numpy()
    setup = time.perf_counter() - t0
    times = []
    start = time.perf_counter()
    for i in range(max_steps):
        a = time.perf_counter()
        oc.append(K1[i], V1[i], [1] * w.B)
        oc.attend(q[i])
        times.append(time.perf_counter() - a)
        if time.perf_counter() - start > budget_s:
            break
    del oc
    return 1e6 * sum(times) / len(times), len(times), setup


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def oracle_whole_steps(w, warmup: int, steps: int, budget_s: float = 200.0):
    """The CPU oracle on `warmup` + `steps` steps of the workload: each step
    appends one token per sequence and runs the decode-attend of every query
    head (a whole step).  The first warm-up step is timed to project the
    run; if whole steps would take longer than `budget_s`, each step instead
    runs the decode-attend of a rotating subset of the query heads, its time
    scaled to all of them (said in the returned sample text).  Returns
    (us_per_step over the timed steps, setup_s, sample)."""
    import oracle
    from bit_kv_cache_05_gb300 import synth
    t0 = time.perf_counter()
    inputs = synth.make_inputs(w, device="cpu")
    oc = oracle.OracleCache(w.B, w.H_q, w.H_kv, w.D, w.bits, w.group,
                            w.residual, w.max_seq + warmup + steps + 1)
    oc.quantize(inputs["K"].numpy(), inputs["V"].numpy(), w.seq_lens)
    K1, V1, q = synth.decode_tokens(w, warmup + steps, device="cpu")
    K1, V1, q = K1.numpy(), V1.numpy(), q.numpy()
    setup = time.perf_counter() - t0
    heads = w.B * w.H_q
    per_step = heads                   # query heads attended per step
    total, cursor = 0.0, 0
    for i in range(warmup + steps):
        a = time.perf_counter()
        oc.append(K1[i], V1[i], [1] * w.B)
        b = time.perf_counter()
        if per_step == heads:
            oc.attend(q[i])
        else:
            for _ in range(per_step):
                j = cursor % heads
                cursor += 1
                oc.attend_one(j // w.H_q, j % w.H_q, q[i, j // w.H_q, j % w.H_q])
        c = time.perf_counter()
        if i == 0:
            full = (b - a) + (c - b) * heads / per_step
            left = warmup + steps - 1
            if left * full > budget_s:
                per_step = max(1, int(heads * budget_s / (left * full)))
        if i >= warmup:
            total += (b - a) + (c - b) * heads / per_step
    del oc
    if per_step == heads:
        sample = (f"{warmup} untimed + {steps} timed whole steps (append one "
                  f"token per sequence, decode-attend all {heads} query "
                  f"heads) after an untimed {setup:.1f}s prefill")
    else:
        sample = (f"{warmup} untimed + {steps} timed steps after an untimed "
                  f"{setup:.1f}s prefill; each appends one token per sequence "
                  f"and attends {per_step} of the {heads} query heads "
                  f"(rotating), scaled to all (whole steps would exceed "
                  f"{budget_s:.0f}s)")
    return 1e6 * total / max(steps, 1), setup, sample


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    us, setup, sample = oracle_whole_steps(w, args.warmup, args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 3),
        "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, N(0,1) fp16 K/V/q)",
        "config": config_of(w),
        "cpu_baseline": {"kind": "oracle", "value": round(us, 3), "unit": UNIT,
                         "cores": 1, "sample": sample},
        "e2e": {"value": round(us, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w):
    """The workload as both arms name it (identical keys and values)."""
    return {"workload": w.name, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv,
            "D": w.D, "bits": w.bits, "group": w.group,
            "residual": w.residual, "S_kv": w.seq_lens[0] if w.B == 1
            else w.seq_lens, "S_q": 1,
            "step": "append 1 token per sequence + fused decode-attend",
            "l2": "inputs larger than L2 (the GPU arm rotates cache copies "
                  "totalling more than 4x L2)",
            "parallelism": "replicas (one independent cache per GPU)"}


def _pct(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, int(q * len(xs)))]


def run_ours(args, w, rank, world, local):
    import torch
    from bit_kv_cache_05_gb300 import _lib, synth
    from bit_kv_cache_05_gb300.cache import KiviCache

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _lib.load()
    K_steps = args.steps
    W = args.warmup
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20
    step_bytes = decode_bytes(w, w.seq_lens)
    n_copies = max(2, -(-4 * l2 // step_bytes))
    # appending steps the run may take: warm-up, one sizing pass, the
    # sustained passes (at most max_sustain steps) and the end-to-end loop
    # (the decode-alone loops append nothing)
    max_sustain = max(K_steps, 16384)
    n_total = W + K_steps + max_sustain + K_steps
    inp = synth.make_inputs(w, device=dev)
    K1, V1, q = synth.decode_tokens(w, 64, device=dev)
    headroom = -(-n_total // n_copies) + 64
    caches = [KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q,
                        bits=w.bits, group=w.group, residual=w.residual,
                        max_seq=w.max_seq + headroom)
              for _ in range(n_copies)]
    del inp
    out = torch.empty(w.B, w.H_q, w.D, dtype=torch.float32, device=dev)
    ones = [1] * w.B
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    cursor = [0]

    def step():
        i = cursor[0]
        cursor[0] += 1
        c = caches[i % n_copies]
        c.append(K1[i % 64], V1[i % 64], ones)
        c.decode_attend(q[i % 64], out)

    # warm-up, timed as a whole to size the sustained region
    wa = torch.cuda.Event(enable_timing=True)
    wb = torch.cuda.Event(enable_timing=True)
    wa.record(stream)
    for _ in range(W):
        step()
    wb.record(stream)
    torch.cuda.synchronize(dev)
    # one more untimed pass of K steps sizes the sustained region (the
    # warm-up carries the first calls' one-time costs)
    wa.record(stream)
    for _ in range(K_steps):
        step()
    wb.record(stream)
    torch.cuda.synchronize(dev)
    est_ms = max(wa.elapsed_time(wb) / K_steps, 1e-3)
    passes = int(max(1, min(max_sustain // K_steps,
                            -(-SUSTAIN_S * 1e3 // (est_ms * K_steps)))))
    passes = int(max_over_ranks(passes, world, dev))

    peak, peak_kind = measured_peak_gbs()
    with ClockSampler(local) as clk:
        # (1) the timed region: `passes` passes of exactly K steps each
        barrier(world)
        torch.cuda.synchronize(dev)
        l0 = _lib.launch_count()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(passes + 1)]
        ev[0].record(stream)
        for p in range(passes):
            for _ in range(K_steps):
                step()
            ev[p + 1].record(stream)
        torch.cuda.synchronize(dev)
        launches = (_lib.launch_count() - l0) / passes
        pass_ms = [ev[p].elapsed_time(ev[p + 1]) / K_steps for p in range(passes)]
        device_s = ev[0].elapsed_time(ev[passes]) / 1e3
        ms = statistics.median(pass_ms)
        ms = max_over_ranks(ms, world, dev)
        barrier(world)

        # (2) the decode call alone (its decode and merge kernels), rotating
        # over the copies: (a) each call between its own pair of events (the
        # launch duration; the roofline uses its median), (b) passes of K
        # calls back to back between two events (where the merge of one call
        # and the decode of the next do not overlap)
        n_d = max(3 * K_steps, 60)
        dv = [(torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(n_d)]
        j = cursor[0]
        for i in range(n_d):
            dv[i][0].record(stream)
            caches[j % n_copies].decode_attend(q[j % 64], out)
            dv[i][1].record(stream)
            j += 1
        torch.cuda.synchronize(dev)
        dec_ms = sorted(a.elapsed_time(b) for a, b in dv)
        dec_avg = statistics.median(dec_ms)
        n_dp = max(5, min(50, passes // 4))
        pv = [torch.cuda.Event(enable_timing=True) for _ in range(n_dp + 1)]
        pv[0].record(stream)
        for p in range(n_dp):
            for i in range(K_steps):
                caches[j % n_copies].decode_attend(q[j % 64], out)
                j += 1
            pv[p + 1].record(stream)
        torch.cuda.synchronize(dev)
        dec_b2b = statistics.median(pv[p].elapsed_time(pv[p + 1]) / K_steps
                                    for p in range(n_dp))

        # (3) end to end through the public API from pinned host memory:
        # vq_kivi_step_host takes the new token's K and V and the query in
        # pinned host memory (copied into device slots on the cache's copy
        # stream, overlapping the previous step) and stores the output into
        # pinned host memory from the decode kernel
        hK = K1.reshape(-1, w.B, w.H_kv, w.D).cpu().pin_memory()
        hV = V1.reshape(-1, w.B, w.H_kv, w.D).cpu().pin_memory()
        hq = q.reshape(-1, w.B, w.H_q, w.D).cpu().pin_memory()
        hout = torch.empty(K_steps, w.B, w.H_q, w.D, dtype=torch.float32
                           ).pin_memory()
        views = [(hK[i % 64], hV[i % 64], hq[i % 64], hout[i]) for i in range(K_steps)]
        for c in caches:          # each cache's slots, stream and events
            c.step_host(*views[0])
        cursor[0] += 1
        torch.cuda.synchronize(dev)
        barrier(world)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        h0 = time.perf_counter()
        t0.record(stream)
        for i in range(K_steps):
            caches[(cursor[0] + i) % n_copies].step_host(*views[i])
        t1.record(stream)
        host_us = (time.perf_counter() - h0) * 1e6 / K_steps
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(t0.elapsed_time(t1) / K_steps, world, dev)
        ref = caches[(cursor[0] + K_steps - 1) % n_copies]
        cursor[0] += K_steps
        # the last step's output in host memory against a device decode of
        # the same cache and query (the same kernels: equal bit for bit)
        last_ok = bool(torch.equal(
            hout[K_steps - 1],
            ref.decode_attend(hq[(K_steps - 1) % 64].cuda(), None).cpu()))

    clocks = clk.summary()
    S_dec = caches[cursor[0] % n_copies].lengths()[0]
    dec_bytes = decode_bytes(w, S_dec)
    achieved = dec_bytes / (dec_avg * 1e-3) / 1e9
    h2d = (K1[0].numel() + V1[0].numel() + q[0].numel()) * 2
    d2h = out.numel() * 4
    for c in caches:
        c.close()
    del caches
    torch.cuda.empty_cache()

    targets = None
    if rank == 0 and not args.no_targets:
        targets = {}
        for name in TARGET_WORKLOADS:
            if name == w.name:
                continue
            targets[name] = measure_workload(synth.workload(name), peak,
                                             full=False)
            torch.cuda.empty_cache()
        # KIVI-Sink decode at the pages' shape (5 sinks per head, the
        # pages' default n_sink_tokens)
        targets["pages_S32768_sink5"] = dict(
            measure_workload(synth.workload("pages_S32768"), peak, full=False,
                             n_sink=5), n_sink=5)
        torch.cuda.empty_cache()
        # Kitty decode at the pages' shape (a quarter of the key channels in
        # 4 bits, the pages' default kitty_hi_fraction)
        targets["pages_S32768_kitty"] = dict(
            measure_workload(synth.workload("pages_S32768"), peak, full=False,
                             kitty_hi=32), kitty_hi=32)
        torch.cuda.empty_cache()
        # AgeTieredKV decode at the pages' shape, the pages' default tiers
        # (8 / 4 / 2 bits below 128 / 1024 tokens of age); 8-bit row capacity
        age = (128, 1024, 8, 4, 2)
        wa = synth.dataclasses.replace(synth.workload("pages_S32768"), bits=8,
                                       residual=0)
        targets["pages_S32768_age"] = dict(
            measure_workload(wa, peak, full=False, age=age), age=list(age))
        torch.cuda.empty_cache()
        tpk, tpk_kind = measured_peak_tflops()
        targets["int4_append_prefill_attend"] = dict(
            measure_multi(synth.workload("int4_append"), 512, tpk),
            peak_kind=tpk_kind)
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        us, n, setup = oracle_steps(w)
        cpu = {"kind": "oracle", "value": round(us, 3), "unit": UNIT,
               "cores": 1,
               "sample": f"{n} whole steps (append 1 token/seq + decode-attend "
                         f"all heads) after an untimed {setup:.1f}s prefill"}
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(ms * 1e3, 3), "unit": UNIT,
        "n_gpus": world, "steps": K_steps, "warmup": W,
        "ms_per_step": round(ms, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, N(0,1) fp16 K/V/q)",
        "config": config_of(w),
        "timing": {"passes": passes, "steps_per_pass": K_steps,
                   "stat": "median over passes of the pass time / K",
                   "p10_us": round(_pct(pass_ms, 0.1) * 1e3, 3),
                   "p90_us": round(_pct(pass_ms, 0.9) * 1e3, 3),
                   "device_s": round(device_s, 3),
                   "l2": f"rotating {n_copies} cache copies "
                         f"({n_copies * step_bytes / 1e6:.0f} MB > 4x L2)"},
        "decode_us": round(dec_avg * 1e3, 3),
        "decode_p10_p90_us": [round(_pct(dec_ms, 0.1) * 1e3, 3),
                              round(_pct(dec_ms, 0.9) * 1e3, 3)],
        "decode_back_to_back_us": round(dec_b2b * 1e3, 3),
        "decode_gbs": round(achieved, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": measured_traffic(w.name),
                     "peak_kind": peak_kind,
                     "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "kernel": "fused decode-attend + partial merge "
                               "(k_decode_mma, k_merge_mma; one call between "
                               "two events, median)",
                     "algorithmic_bytes": dec_bytes},
        "targets": targets,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_ms * 1e3, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "KiviCache.step_host (vq_kivi_step_host): pinned "
                       "host K, V, q in, pinned host output",
                "last_output_matches_device_decode": last_ok,
                "breakdown": {
                    "host_issue_us": round(host_us, 2),
                    "step_device_us": round(ms * 1e3, 2),
                    "reading": "the kernels read a step's inputs from "
                               "the pinned buffers through their device "
                               "mappings (a step that quantizes a group "
                               "stages them first); the step time is the "
                               "larger of the device step and the host's "
                               "time to issue it"}},
        "gpu_launches": int(round(launches)),
        "gpu_launches_per": "pass of K steps",
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def measure_workload(w, peak, full=True, n_sink=0, kitty_hi=None, age=None):
    """The decode of workload `w` from HBM (rotating over cache copies larger
    than 4x L2, the median of 100 launches), and the append of the
    workload's appended tokens per sequence (one token when it appends none)
    timed over at least 8 caches.  With `full`, also the decode hot (one
    cache, repeated), the prefill (the quantize call) and the unfused path
    the pages compare the fused decode against: this library's dequantize
    to fp16 K_hat / V_hat in memory, then torch's
    scaled_dot_product_attention over them (a context row, not a target)."""
    import torch
    import torch.nn.functional as F
    from bit_kv_cache_05_gb300 import synth
    from bit_kv_cache_05_gb300.cache import KiviCache
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    inp = synth.make_inputs(w, device="cuda")
    n_app = w.n_append if w.n_append else 1
    S_dec = [s + n_app for s in w.seq_lens]
    nb = decode_bytes(w, S_dec)
    ncp = max(2, -(-4 * l2 // nb))
    if nb * ncp > 8e9:
        ncp = 2
    caches = []

    def make(i):
        caches.append(KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q,
                                bits=w.bits, group=w.group,
                                residual=w.residual,
                                max_seq=w.max_seq + n_app + 8, n_sink=n_sink,
                                kitty_hi=kitty_hi, age=age))
    # prefill and append are timed over at least 8 caches; the decode
    # rotates over the first ncp
    na = max(ncp, 8)
    prefill = _ev_times(make, na)
    K1, V1, _ = synth.decode_tokens(w, 1, device="cuda")
    if w.n_append:
        Kn = inp["K_new"]
        Vn = inp["V_new"]
    else:
        Kn, Vn = K1[0], V1[0]
    app = _ev_times(lambda i: caches[i].append(Kn, Vn, [n_app] * w.B), na)
    for c in caches[ncp:]:
        c.close()
    del caches[ncp:]
    del inp["K"], inp["V"]
    q = inp["q"]
    out = torch.empty(w.B, w.H_q, w.D, device="cuda")
    for i in range(2 * ncp):
        caches[i % ncp].decode_attend(q, out)
    flushed = _ev_times(lambda i: caches[i % ncp].decode_attend(q, out), 100)
    caches[0].device_status()
    # KIVI-Sink: the fp16 rows of the sinks of the quantized region
    cb = caches[0].cache_bytes()
    nb += cb["sink_bytes"]
    if kitty_hi is not None or age is not None:
        # Kitty: mixed-width key rows + key scale/zero + channel masks, fp16
        # values and residual window, q and out; AgeTieredKV: codes at each
        # group's width + scales / zeros + residual, q and out
        gq = w.H_q // w.H_kv
        nb = (cb["code_bytes"] + cb["meta_bytes"] + cb["value_fp16_bytes"] +
              cb["residual_bytes"] + w.B * w.H_q * w.D * (2 + 4))
    ab = (append_bytes(w, n_app) if not w.n_append
          else flush_append_bytes(w, n_app))
    res = {
        "config": {"B": w.B, "H_q": w.H_q, "H_kv": w.H_kv, "D": w.D,
                   "bits": w.bits, "group": w.group, "residual": w.residual,
                   "S_kv": S_dec[0] if len(set(S_dec)) == 1 else S_dec},
        "decode_us": round(flushed[0], 2),
        "decode_p10_p90_us": [round(flushed[1], 2), round(flushed[2], 2)],
        "decode_bytes": nb,
        "decode_frac": round(nb / (flushed[0] * 1e-6) / 1e9 / peak, 4),
        "decode_frac_nominal": round(nb / (flushed[0] * 1e-6) / 1e9
                                     / NOMINAL_HBM_GBS, 4),
        "cache_copies": ncp,
        "append_tokens_per_seq": n_app, "append_us": round(app[0], 2),
        "append_bytes": ab,
        "append_frac": round(ab / (app[0] * 1e-6) / 1e9 / peak, 4),
    }
    if full:
        hot = _ev_times(lambda i: caches[0].decode_attend(q, out), 100)
        fused = out.clone()
        smax = max(S_dec)
        shape = (w.B, w.H_kv, smax, w.D)
        # zeroed: padding rows of short sequences stay finite under the mask
        Kh = torch.zeros(shape, dtype=torch.float16, device="cuda")
        Vh = torch.zeros(shape, dtype=torch.float16, device="cuda")
        caches[0].dequantize(out=(Kh, Vh))
        dq = _ev_times(lambda i: caches[0].dequantize(out=(Kh, Vh)), 10)
        q4 = q.view(w.B, w.H_q, 1, w.D)
        g = w.H_q // w.H_kv
        kw = {"enable_gqa": True} if g > 1 else {}

        def sdpa(i):
            if min(S_dec) == smax:
                return F.scaled_dot_product_attention(q4, Kh, Vh, **kw)
            # ragged: one call per sequence over its own length (no mask)
            return torch.cat([F.scaled_dot_product_attention(
                q4[b:b + 1], Kh[b:b + 1, :, :S_dec[b]], Vh[b:b + 1, :, :S_dec[b]],
                **kw) for b in range(w.B)])
        ref = sdpa(0).float().view(w.B, w.H_q, w.D)
        at = _ev_times(sdpa, 10)
        res.update({
            "decode_hot_us": round(hot[0], 2),
            "prefill_us": round(prefill[0], 1),
            "unfused": {"dequantize_us": round(dq[0], 1),
                        "sdpa_us": round(at[0], 1),
                        "total_us": round(dq[0] + at[0], 1),
                        "fused_speedup": round((dq[0] + at[0]) / flushed[0], 2),
                        "max_abs_diff_vs_fused": float((ref - fused).abs().max())},
        })
        del Kh, Vh, ref
    for c in caches:
        c.close()
    del caches, inp
    return res


def multi_flops(w, seq_lens, S_q):
    """Algorithmic FLOPs of causal multi-query attention: per query head and
    query i (position S - S_q + i), 2 D multiply-adds per visible token for
    q . k and again for p v, i.e. 4 D (pos + 1)."""
    tot = 0
    for S in seq_lens:
        vis = sum(S - S_q + i + 1 for i in range(S_q))
        tot += w.H_q * 4 * w.D * vis
    return tot


def measure_multi(w, S_q, peak_tflops, reps=5):
    """Chunked prefill attend: append S_q tokens to every sequence of the
    workload's cache, then attend them causally over the whole cache
    (vq_kivi_attend_multi), timed over `reps` caches (each larger than L2
    rotates the cache out between launches)."""
    import torch
    from bit_kv_cache_05_gb300 import synth
    from bit_kv_cache_05_gb300.cache import KiviCache
    inp = synth.make_inputs(w, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(7)
    Kn = torch.randn(w.B, w.H_kv, S_q, w.D, generator=g, device="cuda").half()
    Vn = torch.randn(w.B, w.H_kv, S_q, w.D, generator=g, device="cuda").half()
    q = torch.randn(w.B, w.H_q, S_q, w.D, generator=g, device="cuda").half()
    caches = []
    for _ in range(2):
        c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=w.bits,
                      group=w.group, residual=w.residual,
                      max_seq=w.max_seq + S_q)
        c.append(Kn, Vn, [S_q] * w.B)
        caches.append(c)
    del inp
    out = torch.empty(w.B, w.H_q, S_q, w.D, device="cuda")
    for c in caches:
        c.attend_multi(q, out)
    t = _ev_times(lambda i: caches[i % 2].attend_multi(q, out), reps)
    caches[0].device_status()
    S_now = [s + S_q for s in w.seq_lens]
    fl = multi_flops(w, S_now, S_q)
    for c in caches:
        c.close()
    tf = fl / (t[0] * 1e-6) / 1e12
    return {"S_q": S_q, "S_kv": S_now[0] if len(set(S_now)) == 1 else S_now,
            "us": round(t[0], 1), "p10_p90_us": [round(t[1], 1), round(t[2], 1)],
            "algorithmic_flops": fl, "tflops": round(tf, 2),
            "peak_tflops": peak_tflops, "frac": round(tf / peak_tflops, 4),
            "kernel": "k_attend_multi (tcgen05, TMEM accumulators)"}


def measured_peak_tflops():
    """Dense fp16 tensor peak: the measured bf16 GEMM rate (fp16 and bf16
    run at the same nominal rate on the tensor cores)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def flush_append_bytes(w, n_new):
    """Algorithmic bytes of appending n_new tokens per sequence to a cache
    whose residual holds w.residual tokens (the workload's state): read the
    old residual and the new fp16 K/V rows, write the flushed groups as
    packed codes plus fp16 scale/zero, and the tokens left in the ring."""
    D, g, bits, R = w.D, w.group, w.bits, w.residual
    row = D * bits // 8
    tot = 0
    for S in w.seq_lens:
        Tq0 = 0 if S < R else g * ((S - R) // g)
        S1 = S + n_new
        Tq1 = 0 if S1 < R else g * ((S1 - R) // g)
        nres0, nres1 = S - Tq0, S1 - Tq1
        flushed = Tq1 - Tq0
        rd = (nres0 + n_new) * D * 2 * 2
        wr = flushed * (2 * row + (2 * D * 2) / g + 2 * (D // g) * 2)
        # tokens that stay fp16: the new ones written to the ring
        wr += min(nres1, n_new) * D * 2 * 2
        tot += w.H_kv * (rd + wr)
    return int(tot)


REPORT_WORKLOADS = ("pages_S8192", "pages_S32768", "pages_S65536",
                    "gqa_serving", "int4_append", "ragged_long")


def _ev_times(fn, n):
    """Median, p10 and p90 in us of n CUDA-event-timed calls fn(i), device
    time: a spin kernel queued first keeps the device busy while the host
    queues the calls, so no host launch time falls between the events."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(n * 1e5))   # ~50 us of spinning per queued call
    for i in range(n):
        ev[i][0].record()
        fn(i)
        ev[i][1].record()
    torch.cuda.synchronize()
    ts = sorted(1e3 * a.elapsed_time(b) for a, b in ev)
    return ts[n // 2], ts[n // 10], ts[(9 * n) // 10]


def run_report(names):
    """Secondary figures, one JSON line per workload (measure_workload with
    the hot decode, the prefill and the unfused context path)."""
    import torch
    from bit_kv_cache_05_gb300 import synth
    peak, peak_kind = measured_peak_gbs()
    for name in names:
        res = measure_workload(synth.workload(name), peak, full=True)
        print(json.dumps(dict(workload=name, peak_gbs=peak, peak_kind=peak_kind,
                              **res)), flush=True)
        torch.cuda.empty_cache()


def run_profile_decode(name: str, n: int):
    """One cache of a named workload and n decode launches on it, for ncu
    captures of the decode kernels (and of the prefill's k_flush).  A
    suffix picks the variant the benchmark times beside the plain cache:
    ":sink5" (5 sink tokens), ":kitty" (32 of 128 key channels in 4 bits),
    ":age" (8 / 4 / 2-bit tiers below 128 / 1024 tokens of age)."""
    import torch
    from bit_kv_cache_05_gb300 import synth
    from bit_kv_cache_05_gb300.cache import KiviCache
    name, _, variant = name.partition(":")
    w = synth.workload(name)
    extra = {}
    if variant == "sink5":
        extra = dict(n_sink=5)
    elif variant == "kitty":
        extra = dict(kitty_hi=w.D // 4)
    elif variant == "age":
        w = synth.dataclasses.replace(w, bits=8, residual=0)
        extra = dict(age=(128, 1024, 8, 4, 2))
    elif variant:
        raise SystemExit(f"unknown decode variant {variant!r}")
    inp = synth.make_inputs(w, device="cuda")
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=w.bits,
                  group=w.group, residual=w.residual, max_seq=w.max_seq,
                  **extra)
    del inp["K"], inp["V"]
    torch.cuda.synchronize()
    out = None
    for _ in range(n):
        out = c.decode_attend(inp["q"])
    torch.cuda.synchronize()
    c.device_status()
    print("ok", name, c.decode_kernel(),
          float(out.abs().max()) if out is not None else 0.0)
    c.close()


def run_profile_multi(name: str, B: str, S_q: str, n: str):
    import torch
    from bit_kv_cache_05_gb300 import synth
    from bit_kv_cache_05_gb300.cache import KiviCache
    w0 = synth.workload(name)
    w = synth.shrink(w0, w0.seq_lens[:int(B)], n_append=0)
    S_q, n = int(S_q), int(n)
    inp = synth.make_inputs(w, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(7)
    Kn = torch.randn(w.B, w.H_kv, S_q, w.D, generator=g, device="cuda").half()
    Vn = torch.randn(w.B, w.H_kv, S_q, w.D, generator=g, device="cuda").half()
    q = torch.randn(w.B, w.H_q, S_q, w.D, generator=g, device="cuda").half()
    c = KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q, bits=w.bits,
                  group=w.group, residual=w.residual, max_seq=w.max_seq + S_q)
    c.append(Kn, Vn, [S_q] * w.B)
    del inp
    out = None
    for _ in range(n):
        out = c.attend_multi(q)
    torch.cuda.synchronize()
    c.device_status()
    print("ok", name, w.B, S_q, float(out.abs().max()) if out is not None else 0.0)
    c.close()


def _respawn_under_torchrun(args, argv):
    """`--gpus N` (N > 1) without a torch.distributed launcher: start N local
    ranks with torch.distributed.run (rendezvous on 127.0.0.1) and return
    its exit status."""
    import socket
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-targets", action="store_true",
                    help="leave out the decode of the other target workloads")
    ap.add_argument("--report", nargs="*", default=None,
                    help="secondary figures for these workloads (all when "
                         "none are named) instead of the benchmark line")
    ap.add_argument("--profile-decode", nargs=2, metavar=("WORKLOAD", "N"),
                    default=None,
                    help="build one cache and run N decodes (for ncu)")
    ap.add_argument("--profile-multi", nargs=4, metavar=("WORKLOAD", "B", "S_Q", "N"),
                    default=None,
                    help="append S_Q tokens to the first B sequences of a "
                         "workload's cache and attend them N times (for ncu)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1 or args.gpus < 1:
        ap.error("--steps and --gpus must be >= 1")
    if args.profile_multi is not None:
        run_profile_multi(*args.profile_multi)
        return 0
    if args.profile_decode is not None:
        run_profile_decode(args.profile_decode[0], int(args.profile_decode[1]))
        return 0
    if args.report is not None:
        run_report(args.report or list(REPORT_WORKLOADS))
        return 0
    rank, world, local = dist_env()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return _respawn_under_torchrun(args, argv)
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch "
              f"one rank per GPU (or run without a launcher and let bench.py "
              f"start the ranks)", file=sys.stderr)
        return 2
    from bit_kv_cache_05_gb300 import synth
    w = synth.workload(args.workload)
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, w, rank, world)
        else:
            run_ours(args, w, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
