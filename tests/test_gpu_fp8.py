"""GPU parity of the FP8 E4M3 KV cache against the oracle.

pa_reshape_and_cache_fp8 must store exactly the codes the oracle's encoder
picks (nearest, ties to even, saturating), compared over the whole pool;
pa_decode_fp8 must satisfy |gpu - oracle| <= 2e-3 + 1e-2 |oracle| where the
oracle attends over the exactly dequantised cache in fp64."""
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


def run_fp8(pa, w, partition_sizes):
    dev = torch.device("cuda")
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    pa.pa_reshape_and_cache_fp8(w.key.to(dev), w.value.to(dev), kc, vc, w.slot_mapping.to(dev),
                                w.k_scale, w.v_scale)
    q, bt, cl = w.query.to(dev), w.block_tables.to(dev), w.context_lens.to(dev)
    outs = {}
    for ps in partition_sizes:
        out = torch.empty_like(q)
        pa.pa_decode_fp8(out, q, kc, vc, bt, cl, w.scale, w.k_scale, w.v_scale,
                         w.max_context_len, ps)
        outs[ps] = out
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
    return kc, vc, outs


def host_pool(w):
    kh, vh = w.k_cache.numpy().copy(), w.v_cache.numpy().copy()
    oracle.reshape_and_cache_fp8(w.key, w.value, kh, vh, w.slot_mapping, w.dtype, w.k_scale,
                                 w.v_scale)
    return kh, vh


def check(w, kh, vh, outs, pairs=None):
    ref = oracle.decode(w.query, kh, vh, w.block_tables, w.context_lens, w.scale, w.dtype,
                        pairs=pairs, kv_dtype="e4m3", k_scale=w.k_scale, v_scale=w.v_scale)
    for ps, out in outs.items():
        got = out.float().cpu().double().numpy()
        if pairs is not None:
            pr = np.asarray(pairs).reshape(-1, 2)
            got = got[pr[:, 0], pr[:, 1]]
        assert np.isfinite(got).all(), ps
        err = np.abs(got - ref)
        bad = err > ATOL + RTOL * np.abs(ref)
        assert not bad.any(), f"partition {ps}: {int(bad.sum())} bad, max err {err.max():.3g}"


CASES = [("llama3_8b_gqa", dict(lens=[1, 15, 16, 17, 100, 513, 2049], num_q_heads=32)),
         ("llama3_70b_cb", dict(lens=[1, 31, 32, 33, 700, 3000])),
         ("llama3_8b_gqa", dict(lens=[40, 300], num_q_heads=8, num_kv_heads=8)),     # G = 1
         ("long_context", dict(lens=[9000, 3], dtype="fp16")),
         # bf16 queries (carried in fp16 under a power-of-two rescale)
         ("llama3_70b_cb", dict(lens=[1, 31, 32, 33, 700, 3000], dtype="bf16")),
         ("long_context", dict(lens=[9000, 3])),
         ("llama3_8b_gqa", dict(lens=[5, 600], num_q_heads=24, num_kv_heads=8, block_size=32,
                                dtype="bf16")),
         # head_dim 64: 64-byte rows, staged with the 64-byte swizzle
         ("tiny_mha", dict(lens=[1, 15, 16, 17, 100, 200])),
         ("llama3_8b_gqa", dict(lens=[1, 33, 700, 2049], head_dim=64)),
         ("llama3_8b_gqa", dict(lens=[5, 600, 1500], head_dim=64, num_q_heads=64, num_kv_heads=8,
                                block_size=32, dtype="bf16"))]


@pytest.mark.parametrize("name,kw", CASES, ids=[f"{n}-{i}" for i, (n, _) in enumerate(CASES)])
def test_fp8_small_cases(pa, name, kw):
    w = W.to_fp8(W.make(name, 41, **kw))
    kc, vc, outs = run_fp8(pa, w, [0, 16, 512, 1024])
    kh, vh = host_pool(w)
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)
    check(w, kh, vh, outs)


@pytest.mark.parametrize("name,dtype", [("llama3_8b_gqa", "fp16"), ("llama3_70b_cb", "fp16"),
                                        ("llama3_70b_cb", "bf16"), ("long_context", "bf16")])
def test_fp8_full_size(pa, name, dtype):
    w = W.to_fp8(W.make(name, 0, dtype=dtype))
    kc, vc, outs = run_fp8(pa, w, [w.partition_size])
    kh, vh = host_pool(w)
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)
    rng = np.random.default_rng(0)
    n = 2 if name == "long_context" else 16   # the long sequences are slow in the oracle
    seqs = sorted(set(rng.choice(w.num_seqs, n, replace=False).tolist()) |
                  {int(w.context_lens.argmax())})
    check(w, kh, vh, outs, pairs=[(i, h) for i in seqs for h in range(w.num_q_heads)])


@pytest.mark.parametrize("i", range(12))
def test_fp8_random_shapes(pa, i):
    """Seeded random FP8 decode shapes: batch 1-8, contexts 0-3000, group 1-8,
    1-8 KV heads, head_dim 64 or 128, block size 16 or 32, one partition size
    each."""
    rng = np.random.default_rng(4000 + i)
    G, hkv = int(rng.integers(1, 9)), int(rng.choice([1, 2, 4, 8]))
    lens = [int(x) for x in rng.integers(0, 3001, int(rng.integers(1, 9)))]
    w = W.to_fp8(W.make("llama3_8b_gqa", 120 + i, lens=lens, num_q_heads=G * hkv,
                        num_kv_heads=hkv, block_size=int(rng.choice([16, 32])),
                        head_dim=int(rng.choice([64, 128])),
                        dtype=str(rng.choice(["fp16", "bf16"]))))
    ps = int(rng.choice([0, 16, 48, 160, 512]))
    kc, vc, outs = run_fp8(pa, w, [ps])
    kh, vh = host_pool(w)
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)
    check(w, kh, vh, outs)


@pytest.mark.parametrize("scales", [(3e4, 3e4), (1e-6, 1e-6), (1e3, 1e-7), (1.0, 0.0)],
                         ids=["large", "tiny", "mixed", "one-head-zero"])
def test_fp8_bf16_query_magnitudes(pa, scales):
    """bf16 queries far from 1, and heads of very different magnitude in one
    query group (the power-of-two rescale is per sequence and KV head)."""
    w = W.to_fp8(W.make("llama3_8b_gqa", 46, lens=[300, 1000, 17], dtype="bf16"))
    q = w.query.float()
    q[:, 0::4] *= scales[0]
    q[:, 1::4] *= scales[1]
    w.query = q.to(torch.bfloat16)
    kc, vc, outs = run_fp8(pa, w, [0, 512])
    kh, vh = host_pool(w)
    check(w, kh, vh, outs)


def test_fp8_scatter_from_bf16_and_saturation(pa):
    """bf16 source rows, and values far past the E4M3 range, quantise exactly
    as the oracle does (saturating at +-448)."""
    w = W.to_fp8(W.make("llama3_8b_gqa", 42, batch=6))
    dev = torch.device("cuda")
    key = (torch.randn(w.num_seqs, w.num_kv_heads, w.head_dim) * 3).to(torch.bfloat16)
    value = torch.randn(w.num_seqs, w.num_kv_heads, w.head_dim).to(torch.bfloat16)
    key[0, 0, :4] = torch.tensor([1e4, -1e4, 5.0, -6.0]).to(torch.bfloat16)
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    pa.pa_reshape_and_cache_fp8(key.to(dev), value.to(dev), kc, vc, w.slot_mapping.to(dev),
                                w.k_scale, w.v_scale)
    torch.cuda.synchronize()
    kh, vh = w.k_cache.numpy().copy(), w.v_cache.numpy().copy()
    oracle.reshape_and_cache_fp8(key, value, kh, vh, w.slot_mapping, "bf16", w.k_scale,
                                 w.v_scale)
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)
    s = int(w.slot_mapping[0])
    row = kh[s // w.block_size, 0, s % w.block_size, :2]
    assert row.tolist() == [0x7E, 0xFE]


def test_fp8_permutation_bitwise(pa):
    w = W.to_fp8(W.make("llama3_70b_cb", 43, batch=20, max_len=2500))
    _, _, a = run_fp8(pa, w, [0, 1024])
    _, _, b = run_fp8(pa, w.permuted(3), [0, 1024])
    for ps in (0, 1024):
        assert torch.equal(a[ps].view(torch.int16), b[ps].view(torch.int16))
