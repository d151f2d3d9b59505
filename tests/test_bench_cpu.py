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


def test_shared_prefix_groups_and_unique_bytes_by_hand():
    """The copy-on-write batch records its groups (runs of consecutive
    sequences) and each sequence's shared prefix (whole shared blocks only: a
    partial last prefix block is copied per sequence, so it is not shared);
    the distinct-slot byte count takes each group's shared rows once."""
    ng, gs, P, bs = 3, 4, 40, 16
    w = W.make("shared_prefix_cow", 2, groups=ng, group_size=gs, prefix_len=P, max_len=30,
               num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=bs)
    assert w.group_start.tolist() == [0, 4, 8, 12]
    shared = (P // bs) * bs                                  # 32 tokens in shared blocks
    assert w.prefix_lens.tolist() == [shared] * (ng * gs)
    assert w.max_group_size == gs
    bt = w.block_tables.numpy()
    for g in range(ng):
        rows = bt[g * gs:(g + 1) * gs, : P // bs]
        assert (rows == rows[0]).all()                       # the group's shared blocks
        assert len(set(bt[g * gs:(g + 1) * gs, P // bs].tolist())) == gs   # copied block
    ctx = w.context_lens.numpy().astype(np.int64)
    unique_tokens = ng * shared + int((ctx - shared).sum())
    ab = bench.algorithmic_bytes(w)
    assert ab["kv_unique"] == 2 * unique_tokens * 2 * 64 * 2
    assert ab["kv"] == 2 * int(ctx.sum()) * 2 * 64 * 2
    assert ab["decode_unique"] == ab["kv_unique"] + ab["qo"] + ab["tables"]
    # layout changes keep or drop the description consistently
    assert w.permuted(1).group_start.tolist() == [0, 4, 8, 12]
    assert w.unshared().group_start is None and w.unshared().prefix_lens is None
    assert "kv_unique" not in bench.algorithmic_bytes(W.make("tiny_mha", 0))
