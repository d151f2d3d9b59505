"""CPU checks of the benchmark's byte accounting and of its reference arm."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_kv_bytes_per_token_llama3_70b():
    """'LLM Serving Engine Shootout', 2.1 KV Cache Memory Equation: K and V of
    one token over 80 layers, 8 KV heads, d 128, 2-byte elements.  The page
    prints 655,360 bytes because it counts the 2-byte element size twice; the
    equation's own terms give 327,680 bytes (320 KiB)."""
    assert bench.kv_bytes_per_token(80, 8, 128, 2) == 327680
    assert bench.kv_bytes_per_token(80, 8, 128, 2) * 2 == 655360


def test_algorithmic_bytes_by_hand():
    w = W.make("tiny_mha", 0, lens=[1, 16, 17, 0])
    ab = bench.algorithmic_bytes(w)
    d, H, s = 64, 4, 2
    assert ab["kv"] == 2 * (1 + 16 + 17) * H * d * s
    assert ab["qo"] == 2 * 4 * H * d * s
    assert ab["tables"] == 4 * (1 + 1 + 2 + 0) + 4 * 4
    assert ab["scatter"] == 4 * 3 * H * d * s + 8 * 4       # three tokens have a slot
    assert ab["step"] == ab["kv"] + ab["qo"] + ab["tables"] + ab["scatter"]


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_mha", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_prefill_flops_by_hand():
    pw = W.make_prefill("tiny_mha", 0, lens=[10, 4], q_lens=[3, 4])
    # seq 0: positions 7, 8, 9 -> 8 + 9 + 10 keys; seq 1: positions 0..3 -> 1+2+3+4 keys
    keys = (8 + 9 + 10) + (1 + 2 + 3 + 4)
    assert bench.prefill_flops(pw) == 4 * 64 * 4 * keys
