"""GPU parity of chunked prefill over FP8 E4M3 caches (pa_prefill_fp8) against
the fp64 oracle reading the same codes: |gpu - oracle| <= 2e-3 + 1e-2 |oracle|
per element.  The chunk's K/V go into the pool through
pa_reshape_and_cache_fp8 first, and the pool must then hold exactly the codes
the oracle's encoder picks.  Unowned slots hold the E4M3 NaN code, so a slot
read by mistake shows up as a non-finite output."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
RTOL, ATOL = 1e-2, 2e-3


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from pagedattention_kv_cache_attention_gb300 import build
    build.build()
    import pagedattention_kv_cache_attention_gb300 as pa
    pa._load()
    assert pa.pa_device_errors() == 0
    return pa


def run(pa, pw):
    dev = torch.device("cuda")
    kc, vc = pw.k_cache.to(dev), pw.v_cache.to(dev)
    pa.pa_reshape_and_cache_fp8(pw.key.to(dev), pw.value.to(dev), kc, vc,
                                pw.slot_mapping.to(dev), pw.k_scale, pw.v_scale)
    q = pw.query.to(dev)
    out = torch.full_like(q, float("nan"))
    pa.pa_prefill_fp8(out, q, pw.query_start.to(dev), kc, vc, pw.block_tables.to(dev),
                      pw.context_lens.to(dev), pw.scale, pw.k_scale, pw.v_scale, pw.max_q_len)
    torch.cuda.synchronize()
    return kc, vc, out, pa.pa_device_errors()


def host_pool(pw):
    kh, vh = pw.k_cache.numpy().copy(), pw.v_cache.numpy().copy()
    oracle.reshape_and_cache_fp8(pw.key, pw.value, kh, vh, pw.slot_mapping, pw.dtype,
                                 pw.k_scale, pw.v_scale)
    return kh, vh


def check(pw, kc, vc, out, rows=None):
    kh, vh = host_pool(pw)
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)
    ref = oracle.prefill(pw.query, pw.query_start, kh, vh, pw.block_tables, pw.context_lens,
                         pw.scale, pw.dtype, kv_dtype="e4m3", k_scale=pw.k_scale,
                         v_scale=pw.v_scale)
    got = out.float().cpu().double().numpy()
    if rows is not None:
        ref, got = ref[rows], got[rows]
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{int(bad.sum())} elements outside tolerance, max err {err.max():.3g}"


CASES = [
    ("tiny_mha", dict(lens=[20, 37, 1, 64], chunk=9)),
    ("tiny_mha", dict(lens=[30, 17], chunk=10**6)),                              # whole prompts
    ("tiny_mha", dict(lens=[50, 3, 100], q_lens=[1, 1, 1])),                    # decode-like
    ("tiny_mha", dict(lens=[70, 33], chunk=40, head_dim=128, dtype="bf16")),
    ("llama3_8b_gqa", dict(lens=[600, 1500, 33], chunk=300)),                     # G 4, two tiles
    ("llama3_8b_gqa", dict(lens=[200, 90], chunk=77, num_q_heads=24, num_kv_heads=8)),  # G 3
    ("llama3_70b_cb", dict(lens=[130, 1000, 31], chunk=65)),                      # G 8, bs 32
    ("llama3_70b_cb", dict(lens=[300, 64], chunk=10**6, head_dim=64, dtype="bf16")),
    ("llama3_8b_gqa", dict(lens=[100, 40], chunk=10**6, num_q_heads=8, num_kv_heads=8)),  # G 1
    ("llama3_8b_gqa", dict(lens=[500, 64], chunk=50, num_q_heads=16, num_kv_heads=8,
                           dtype="bf16")),                                  # G 2, one tile
    ("llama3_70b_cb", dict(lens=[700, 1200], chunk=150, dtype="bf16")),     # G 8, bf16, bs 32
    ("llama3_70b_cb", dict(lens=[400, 900, 61], chunk=140, num_q_heads=40, num_kv_heads=8)),  # G 5
    ("llama3_8b_gqa", dict(lens=[260, 45, 700], chunk=37, num_q_heads=28, num_kv_heads=4)),  # G 7
    ("llama3_8b_gqa", dict(lens=[900, 300, 1700], chunk=256, head_dim=64)),              # d 64
    ("llama3_8b_gqa", dict(lens=[500, 64], chunk=20, head_dim=64, dtype="bf16")),        # one tile
]


@pytest.mark.parametrize("name,kw", CASES, ids=[f"{n}-{i}" for i, (n, _) in enumerate(CASES)])
def test_prefill_fp8_cases(pa, name, kw):
    pw = W.to_fp8(W.make_prefill(name, 81, **kw))
    kc, vc, out, err = run(pa, pw)
    assert err == 0
    check(pw, kc, vc, out)


def test_prefill_fp8_scales(pa):
    """Scales other than the workloads' default (K and V differ)."""
    pw = W.to_fp8(W.make_prefill("llama3_8b_gqa", 82, lens=[400, 123], chunk=90, dtype="bf16"),
                  k_scale=0.0131, v_scale=0.047)
    kc, vc, out, err = run(pa, pw)
    assert err == 0
    check(pw, kc, vc, out)


def test_prefill_fp8_llama3_8b_chunks_sampled(pa):
    """Llama-3-8B shape: 16 sequences, 512-token chunks at the end of contexts
    up to 4096; a seeded sample of rows is checked."""
    pw = W.to_fp8(W.make_prefill("llama3_8b_gqa", 83, batch=16, chunk=512))
    kc, vc, out, err = run(pa, pw)
    assert err == 0
    rows = np.random.default_rng(0).choice(pw.total_q, 400, replace=False)
    check(pw, kc, vc, out, rows=np.sort(rows))


@pytest.mark.parametrize("i", range(16))
def test_prefill_fp8_random_shapes(pa, i):
    """Seeded random shapes: batch 1-4, contexts up to 1500, chunk 1-600, group
    1-8, head_dim 64 or 128, block size 16 or 32, fp16 or bf16 queries."""
    rng = np.random.default_rng(1100 + i)
    G, hkv = int(rng.integers(1, 9)), int(rng.choice([1, 2, 4]))
    lens = [int(x) for x in rng.integers(1, 1501, int(rng.integers(1, 5)))]
    kw = dict(lens=lens, chunk=int(rng.choice([1, 7, 33, 64, 100, 257, 600])),
              num_q_heads=G * hkv, num_kv_heads=hkv, head_dim=int(rng.choice([64, 128])),
              block_size=int(rng.choice([16, 32])), dtype=str(rng.choice(["fp16", "bf16"])))
    pw = W.to_fp8(W.make_prefill("llama3_8b_gqa", 90 + i, **kw))
    kc, vc, out, err = run(pa, pw)
    assert err == 0
    check(pw, kc, vc, out)


@pytest.mark.parametrize("chunk,head_dim", [(300, 128), (20, 128), (40, 64), (10, 64)],
                         ids=["two-tile", "one-tile", "two-tile-d64", "one-tile-d64"])
def test_prefill_fp8_bad_block_flagged_others_exact(pa, chunk, head_dim):
    """An out-of-range block id in one sequence's table: the call flags it,
    reads nothing through it (the sub-tile's codes are never copied, its V rows
    are cleared after the widening, so that sequence's rows stay finite), and
    every other sequence's rows still match the oracle."""
    pw = W.to_fp8(W.make_prefill("llama3_8b_gqa", 85, lens=[700, 1400, 900], chunk=chunk,
                                 head_dim=head_dim))
    dev = torch.device("cuda")
    kc, vc = pw.k_cache.to(dev), pw.v_cache.to(dev)
    pa.pa_reshape_and_cache_fp8(pw.key.to(dev), pw.value.to(dev), kc, vc,
                                pw.slot_mapping.to(dev), pw.k_scale, pw.v_scale)
    bt = pw.block_tables.clone()
    bt[1, 5] = pw.num_blocks + 7          # a block well inside sequence 1's context
    q, qs = pw.query.to(dev), pw.query_start.to(dev)
    out = torch.full_like(q, float("nan"))
    pa.pa_prefill_fp8(out, q, qs, kc, vc, bt.to(dev), pw.context_lens.to(dev), pw.scale,
                      pw.k_scale, pw.v_scale, pw.max_q_len)
    torch.cuda.synchronize()
    assert pa.pa_device_errors() & pa.DEVERR_BAD_BLOCK
    qs_h = pw.query_start.numpy()
    a1, b1 = int(qs_h[1]), int(qs_h[2])
    assert torch.isfinite(out[a1:b1].float()).all()
    kh, vh = host_pool(pw)
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)
    for i in (0, 2):
        a, b = int(qs_h[i]), int(qs_h[i + 1])
        ref = oracle.prefill(pw.query[a:b], np.array([0, b - a], dtype=np.int32), kh, vh,
                             pw.block_tables[i:i + 1], pw.context_lens[i:i + 1], pw.scale,
                             pw.dtype, kv_dtype="e4m3", k_scale=pw.k_scale, v_scale=pw.v_scale)
        got = out[a:b].float().cpu().double().numpy()
        err = np.abs(got - ref)
        assert not (err > ATOL + RTOL * np.abs(ref)).any(), f"seq {i}: max err {err.max():.3g}"
