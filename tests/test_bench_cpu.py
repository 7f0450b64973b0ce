"""bench.py on the CPU: the roofline numerator (algorithmic bytes of one
decode) against the per-unit byte counts, and the reference arm's JSON line.

Per (sequence, kv head) a decode reads T_q quantized token-heads — two
packed code rows plus the fp16 key scale/zero (amortized over the g tokens of
a key group) and the fp16 value scale/zero of the token: 48 B at D=64 b=2
g=32, 96 B at D=128 b=2 g=32, 144 B at D=128 b=4 g=64 — and n_res fp16 key
and value rows (4 D bytes each), and per query head reads q (2 D bytes) and
writes out (4 D bytes).  The residual rule gives T_q = g * floor((S - R) / g).
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.mark.parametrize("name,lens,expect", [
    ("tiny", [256], 4 * (224 * 48 + 32 * 256 + 64 * 2 + 64 * 4)),
    ("pages_S512", [512], 32 * (480 * 96 + 32 * 512 + 768)),
    ("pages_S2048", [2048], 32 * (2016 * 96 + 32 * 512 + 768)),
    ("pages_S8192", [8192], 32 * (8160 * 96 + 32 * 512 + 768)),
    ("pages_S32768", [32768], 32 * (32736 * 96 + 32 * 512 + 768)),
    ("pages_S65536", [65536], 32 * (65504 * 96 + 32 * 512 + 768)),
    # 4 query heads per kv head: q and out four times per (b, kv head)
    ("gqa_serving", [8192] * 16, 16 * 8 * (8160 * 96 + 32 * 512 + 4 * 768)),
    # 4-bit, g = 64, R = 64, after the 512-token append: S = 33280
    ("int4_append", [33280] * 8, 8 * 32 * (33216 * 144 + 64 * 512 + 768)),
])
def test_decode_bytes_match_the_per_unit_counts(name, lens, expect):
    import bench
    from bit_kv_cache_05_gb300 import synth
    assert bench.decode_bytes(synth.workload(name), lens) == expect


def test_pages_shape_totals():
    """The pages' sweep at S_kv = 512 ... 65536, as whole-decode totals."""
    import bench
    from bit_kv_cache_05_gb300 import synth
    got = [bench.decode_bytes(synth.workload(f"pages_S{s}"), [s])
           for s in (512, 2048, 8192, 32768, 65536)]
    assert got == [2023424, 6742016, 25616384, 101113856, 201777152]


def test_reference_arm_prints_one_json_line():
    """--impl reference times the oracle on the host cores and prints the
    benchmark's line with impl, cpu_baseline and a zero-copy e2e."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
         "--workload", "tiny", "--steps", "1", "--warmup", "3"],
        capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "us/step"
    assert d["higher_is_better"] is False
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["e2e"]["d2h_bytes_per_step"] == 0
    # whole steps (every query head attended), and the same config as the
    # GPU arm names (both come from config_of)
    assert "whole steps" in d["cpu_baseline"]["sample"]
    import bench
    from bit_kv_cache_05_gb300 import synth
    assert d["config"] == json.loads(json.dumps(bench.config_of(synth.workload("tiny"))))


def _run_bench(args, env_extra=None, drop=("RANK", "WORLD_SIZE", "LOCAL_RANK")):
    env = {k: v for k, v in os.environ.items() if k not in drop}
    env["CUDA_VISIBLE_DEVICES"] = ""
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=900, env=env,
                          cwd=ROOT)


def test_gpus_without_a_launcher_starts_the_ranks():
    """--gpus 2 with no torch.distributed launcher: bench.py starts two local
    ranks itself (torch.distributed.run on 127.0.0.1); for the reference arm
    rank 0 alone prints its line and the other rank exits 0."""
    r = _run_bench(["--impl", "reference", "--gpus", "2", "--workload", "tiny",
                    "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_gpus_that_disagree_with_the_launcher_fail():
    """A launcher that started a different number of ranks than --gpus asks
    for is an error (exit status 2), not a silent single replica."""
    r = _run_bench(["--impl", "reference", "--gpus", "2", "--workload", "tiny",
                    "--steps", "1", "--warmup", "3"],
                   env_extra={"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode == 2
    assert "WORLD_SIZE" in r.stderr


def test_flush_append_bytes_of_the_4bit_workload():
    """The 512-token append of the 4-bit workload (R = 64 tokens in the
    residual before it, 64 after): per (b, kv head) read 64 + 512 fp16 K and V
    rows, write 512 quantized token-heads of 144 B and 64 fp16 K and V rows."""
    import bench
    from bit_kv_cache_05_gb300 import synth
    w = synth.workload("int4_append")
    per_head = (64 + 512) * 512 + 512 * 144 + 64 * 512
    assert per_head == 401408
    assert bench.flush_append_bytes(w, 512) == 8 * 32 * per_head


def test_multi_query_flops_per_unit():
    """Causal multi-query FLOPs: 4 D per (query head, query, visible token);
    with S = 5 and S_q = 2 the two queries see 4 and 5 tokens."""
    import bench
    from bit_kv_cache_05_gb300 import synth
    w = synth.Workload("t", 1, 2, 1, 4, 2, 4, 4, [5])
    assert bench.multi_flops(w, [5], 2) == 2 * 4 * 4 * (4 + 5)
    w4 = synth.workload("int4_append")
    S = 33280
    per_head = 4 * 128 * sum(S - 512 + i + 1 for i in range(512))
    assert bench.multi_flops(w4, [S] * 8, 512) == 8 * 32 * per_head
