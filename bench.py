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
                         "bit_kv_cache_05_gb300/csrc/decode_mma.cu")


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

def oracle_sampled_steps(w, warmup: int, steps: int):
    """The CPU oracle on `warmup` + `steps` steps of the workload, each one a
    bounded sample: the whole append (one token per sequence), then the
    decode-attend of ONE query head (rotating over all B * H_q of them),
    its time scaled by B * H_q to the full step.  Returns
    (us_per_step over the timed steps, setup_s)."""
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
    total = 0.0
    for i in range(warmup + steps):
        a = time.perf_counter()
        oc.append(K1[i], V1[i], [1] * w.B)
        b = time.perf_counter()
        j = i % heads
        oc.attend_one(j // w.H_q, j % w.H_q, q[i, j // w.H_q, j % w.H_q])
        c = time.perf_counter()
        if i >= warmup:
            total += (b - a) + (c - b) * heads
    del oc
    return 1e6 * total / max(steps, 1), setup


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    us, setup = oracle_sampled_steps(w, args.warmup, args.steps)
    sample = (f"{args.warmup} untimed + {args.steps} timed steps after an "
              f"untimed {setup:.1f}s prefill; each step appends one token per "
              f"sequence and runs the decode-attend of one query head "
              f"(rotating), scaled by B*H_q = {w.B * w.H_q}")
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
    return {"workload": w.name, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv,
            "D": w.D, "bits": w.bits, "group": w.group,
            "residual": w.residual, "S_kv": w.seq_lens[0] if w.B == 1
            else w.seq_lens, "S_q": 1,
            "step": "append 1 token per sequence + fused decode-attend"}


def run_ours(args, w, rank, world, local):
    import torch
    from bit_kv_cache_05_gb300 import _lib, synth
    from bit_kv_cache_05_gb300.cache import KiviCache

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _lib.load()
    K_steps = args.steps
    W = args.warmup
    n_total = W + K_steps
    inp = synth.make_inputs(w, device=dev)
    K1, V1, q = synth.decode_tokens(w, max(n_total, 1), device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20
    step_bytes = decode_bytes(w, w.seq_lens)
    n_copies = max(2, -(-4 * l2 // step_bytes))
    headroom = n_total + 64
    caches = [KiviCache(inp["K"], inp["V"], w.seq_lens, H_q=w.H_q,
                        bits=w.bits, group=w.group, residual=w.residual,
                        max_seq=w.max_seq + 3 * headroom)
              for _ in range(n_copies)]
    del inp
    out = torch.empty(w.B, w.H_q, w.D, dtype=torch.float32, device=dev)
    ones = [1] * w.B
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    def step(i):
        c = caches[i % n_copies]
        c.append(K1[i], V1[i], ones)
        c.decode_attend(q[i], out)

    # warm-up
    for i in range(W):
        step(i)
    torch.cuda.synchronize(dev)

    peak, peak_kind = measured_peak_gbs()
    with ClockSampler(local) as clk:
        # (1) the timed steps
        barrier(world)
        torch.cuda.synchronize(dev)
        l0 = _lib.launch_count()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(W, n_total):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        launches = _lib.launch_count() - l0
        ms = e0.elapsed_time(e1) / K_steps
        ms = max_over_ranks(ms, world, dev)
        barrier(world)

        # (2) the decode launch alone, per-launch events, rotating copies
        ev = [(torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(K_steps)]
        for i in range(K_steps):
            c = caches[(i + 1) % n_copies]
            ev[i][0].record(stream)
            c.decode_attend(q[i], out)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        dec_ms = [a.elapsed_time(b) for a, b in ev]
        dec_avg = sum(dec_ms) / len(dec_ms)

        # (3) end to end through the public API from pinned host memory
        # a step's inputs (the new token's K and V, the query) sit packed in
        # one pinned buffer, so that they cross in one copy; the cache calls
        # take views of the device copy
        nK, nV, nq = K1[0].numel(), V1[0].numel(), q[0].numel()
        hin = torch.cat([K1.reshape(n_total, nK), V1.reshape(n_total, nV),
                         q.reshape(n_total, nq)], dim=1).cpu().pin_memory()
        hout = torch.empty(K_steps, w.B, w.H_q, w.D, dtype=torch.float32
                           ).pin_memory()
        din = torch.empty(nK + nV + nq, dtype=K1.dtype, device=dev)
        dK = din[:nK].view(K1[0].shape)
        dV = din[nK:nK + nV].view(V1[0].shape)
        dq = din[nK + nV:].view(q[0].shape)
        torch.cuda.synchronize(dev)
        barrier(world)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(K_steps):
            c = caches[(i + 2) % n_copies]
            din.copy_(hin[W + i], non_blocking=True)
            c.append(dK, dV, ones)
            c.decode_attend(dq, out)
            hout[i].copy_(out, non_blocking=True)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(t0.elapsed_time(t1) / K_steps, world, dev)

    clocks = clk.summary()
    S_now = [s + n_total for s in w.seq_lens]
    dec_bytes = decode_bytes(w, S_now)
    achieved = dec_bytes / (dec_avg * 1e-3) / 1e9
    h2d = (K1[0].numel() + V1[0].numel() + q[0].numel()) * 2
    d2h = out.numel() * 4

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        us, n, setup = oracle_steps(w)
        cpu = {"kind": "oracle", "value": round(us, 3), "unit": UNIT,
               "cores": 1,
               "sample": f"{n} whole steps (append 1 token/seq + decode-attend "
                         f"all heads) after an untimed {setup:.1f}s prefill"}
    for c in caches:
        c.close()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(ms * 1e3, 3), "unit": UNIT,
        "n_gpus": world, "steps": K_steps, "warmup": W,
        "ms_per_step": round(ms, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, N(0,1) fp16 K/V/q)",
        "config": dict(config_of(w), l2=f"rotating {n_copies} cache copies "
                       f"({n_copies * step_bytes / 1e6:.0f} MB > 4x L2)",
                       parallelism=f"replicas x{world}"),
        "decode_us": round(dec_avg * 1e3, 3),
        "decode_gbs": round(achieved, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": measured_traffic(w.name),
                     "peak_kind": peak_kind,
                     "kernel": "fused decode-attend + partial merge "
                               "(k_decode_mma, k_merge_mma; timed together)",
                     "algorithmic_bytes": dec_bytes},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_ms * 1e3, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


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
    """Secondary figures, one JSON line per workload: the decode from HBM
    (rotating over cache copies larger than 4x L2) and hot (one cache,
    repeated), the append (the workload's appended tokens per sequence, else
    one), the quantize of the initial cache (prefill), and the unfused path
    the pages compare the fused decode against: this library's dequantize to
    fp16 K_hat / V_hat in memory, then torch's scaled_dot_product_attention
    over them (a context row, not a target)."""
    import torch
    import torch.nn.functional as F
    from bit_kv_cache_05_gb300 import synth
    from bit_kv_cache_05_gb300.cache import KiviCache
    peak, peak_kind = measured_peak_gbs()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    for name in names:
        w = synth.workload(name)
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
                                    max_seq=w.max_seq + n_app + 8))
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
        hot = _ev_times(lambda i: caches[0].decode_attend(q, out), 100)
        caches[0].device_status()
        fused = out.clone()
        # the unfused context path
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
        line = {
            "workload": name, "peak_gbs": peak, "peak_kind": peak_kind,
            "decode_bytes": nb, "cache_copies": ncp,
            "decode_us": round(flushed[0], 2),
            "decode_p10_p90_us": [round(flushed[1], 2), round(flushed[2], 2)],
            "decode_frac": round(nb / (flushed[0] * 1e-6) / 1e9 / peak, 3),
            "decode_hot_us": round(hot[0], 2),
            "append_tokens_per_seq": n_app, "append_us": round(app[0], 2),
            "prefill_us": round(prefill[0], 1),
            "unfused": {"dequantize_us": round(dq[0], 1),
                        "sdpa_us": round(at[0], 1),
                        "total_us": round(dq[0] + at[0], 1),
                        "fused_speedup": round((dq[0] + at[0]) / flushed[0], 2),
                        "max_abs_diff_vs_fused": float((ref - fused).abs().max())},
        }
        print(json.dumps(line), flush=True)
        for c in caches:
            c.close()
        del caches, Kh, Vh, inp, ref
        torch.cuda.empty_cache()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--report", nargs="*", default=None,
                    help="secondary figures for these workloads (all when "
                         "none are named) instead of the benchmark line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.report is not None:
        run_report(args.report or list(REPORT_WORKLOADS))
        return
    from bit_kv_cache_05_gb300 import synth
    w = synth.workload(args.workload)
    rank, world, local = dist_env()
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


if __name__ == "__main__":
    main()
