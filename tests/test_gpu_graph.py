"""The decode step captured in a CUDA graph ("Inference Engines": CUDA graphs
cut launch overhead).  Every library call only validates on the host and
enqueues kernels, so a captured step replayed with new inputs written into the
captured buffers must give the bit-identical result of the same calls made
eagerly -- and, like every GPU result here, match the fp64 oracle: the
replayed pools bit for bit (the oracle's scatter), the replayed output within
|gpu - oracle| <= 2e-3 + 1e-2 |oracle|, for both input sets."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

RTOL, ATOL = 1e-2, 2e-3

pytestmark = pytest.mark.gpu


def bits(t):
    """Raw bits of a cache (its unowned slots hold NaN, which compares unequal)."""
    return t.view(torch.uint8)


def oracle_step(w, fp8):
    """The oracle's pools after the step's scatter, and its fp64 output."""
    if fp8:
        kh, vh = w.k_cache.numpy().copy(), w.v_cache.numpy().copy()
        oracle.reshape_and_cache_fp8(w.key, w.value, kh, vh, w.slot_mapping, w.dtype,
                                     w.k_scale, w.v_scale)
    else:
        kh = w.k_cache.view(torch.int16).numpy().view(np.uint16).copy()
        vh = w.v_cache.view(torch.int16).numpy().view(np.uint16).copy()
        oracle.reshape_and_cache(w.key, w.value, kh, vh, w.slot_mapping)
    ref = oracle.decode(w.query, kh, vh, w.block_tables, w.context_lens, w.scale, w.dtype,
                        kv_dtype="e4m3" if fp8 else None, k_scale=w.k_scale, v_scale=w.v_scale)
    return kh, vh, ref


def assert_matches_oracle(static, w, fp8, what):
    kh, vh, ref = oracle_step(w, fp8)
    for name, host in (("kc", kh), ("vc", vh)):
        dev = static[name].cpu()
        got = (dev.numpy() if fp8 else dev.view(torch.int16).numpy().view(np.uint16))
        assert np.array_equal(got[:w.num_blocks], host), f"{what}: {name} differs from the oracle"
    got = static["out"].float().cpu().double().numpy()
    assert np.isfinite(got).all(), what
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside tolerance, max {err.max():.3g}"


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


@pytest.mark.parametrize("fp8", [False, True])
def test_captured_step_replays_bitwise(pa, fp8):
    base = W.make("llama3_8b_gqa", 51, batch=16)
    other = W.make("llama3_8b_gqa", 52, batch=16)   # same shapes, new values and lengths
    if fp8:
        base, other = W.to_fp8(base), W.to_fp8(other)
    dev = torch.device("cuda")
    maxctx = max(base.max_context_len, other.max_context_len)
    NB = max(base.num_blocks, other.num_blocks)
    ps = 512

    def buffers(w):
        kc = torch.zeros((NB,) + tuple(w.k_cache.shape[1:]), dtype=w.k_cache.dtype, device=dev)
        vc = torch.zeros_like(kc)
        kc[:w.num_blocks] = w.k_cache.to(dev)
        vc[:w.num_blocks] = w.v_cache.to(dev)
        return dict(kc=kc, vc=vc, key=w.key.to(dev), value=w.value.to(dev),
                    sm=w.slot_mapping.to(dev), q=w.query.to(dev), bt=w.block_tables.to(dev),
                    cl=w.context_lens.to(dev), out=torch.empty_like(w.query, device=dev))

    ws = pa.new_decode_workspace(base.num_seqs, base.num_q_heads, base.head_dim, maxctx, ps)

    def step(b, w, stream=None):
        if fp8:
            pa.pa_reshape_and_cache_fp8(b["key"], b["value"], b["kc"], b["vc"], b["sm"],
                                        w.k_scale, w.v_scale, stream=stream)
            pa.pa_decode_fp8(b["out"], b["q"], b["kc"], b["vc"], b["bt"], b["cl"], w.scale,
                             w.k_scale, w.v_scale, maxctx, ps, workspace=ws, stream=stream)
        else:
            pa.pa_reshape_and_cache(b["key"], b["value"], b["kc"], b["vc"], b["sm"],
                                    stream=stream)
            pa.pa_decode(b["out"], b["q"], b["kc"], b["vc"], b["bt"], b["cl"], w.scale, maxctx,
                         ps, workspace=ws, stream=stream)

    # eager reference results for both input sets
    eager = {}
    for name, w in (("base", base), ("other", other)):
        b = buffers(w)
        step(b, w)
        torch.cuda.synchronize()
        eager[name] = (b["out"].clone(), b["kc"].clone(), b["vc"].clone())

    # capture with the base inputs in static buffers
    static = buffers(base)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(static, base, stream=side)        # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    fresh = buffers(base)
    for k in ("kc", "vc"):
        static[k].copy_(fresh[k])
    with torch.cuda.graph(g):
        step(static, base, stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    out, kc, vc = eager["base"]
    assert torch.equal(static["out"].view(torch.int16), out.view(torch.int16))
    assert torch.equal(bits(static["kc"]), bits(kc)) and torch.equal(bits(static["vc"]), bits(vc))
    assert_matches_oracle(static, base, fp8, "first replay")

    # new inputs in the same buffers, replay
    nb = buffers(other)
    for k in ("kc", "vc", "key", "value", "sm", "q", "bt", "cl"):
        static[k].copy_(nb[k])
    g.replay()
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
    out, kc, vc = eager["other"]
    assert torch.equal(static["out"].view(torch.int16), out.view(torch.int16))
    assert torch.equal(bits(static["kc"]), bits(kc)) and torch.equal(bits(static["vc"]), bits(vc))
    assert_matches_oracle(static, other, fp8, "replay with new inputs")


def test_captured_shared_prefix_step(pa):
    """The copy-on-write step through pa_decode_shared_prefix (scatter, the
    shared pass, the decode and its join) captured once and replayed with a
    second batch of the same shapes written into the captured buffers: the
    same bits as the eager calls, and the oracle's per-sequence attention."""
    kw = dict(groups=4, group_size=4, prefix_len=256, max_len=64, partition_size=64)
    base = W.make("shared_prefix_cow", 53, **kw)
    other = W.make("shared_prefix_cow", 54, **kw)
    assert torch.equal(base.group_start, other.group_start)
    dev = torch.device("cuda")
    maxctx = max(base.max_context_len, other.max_context_len)
    NB = max(base.num_blocks, other.num_blocks)
    ps, mgs = 64, base.max_group_size

    def buffers(w):
        kc = torch.zeros((NB,) + tuple(w.k_cache.shape[1:]), dtype=w.k_cache.dtype, device=dev)
        vc = torch.zeros_like(kc)
        kc[:w.num_blocks] = w.k_cache.to(dev)
        vc[:w.num_blocks] = w.v_cache.to(dev)
        return dict(kc=kc, vc=vc, key=w.key.to(dev), value=w.value.to(dev),
                    sm=w.slot_mapping.to(dev), q=w.query.to(dev), bt=w.block_tables.to(dev),
                    cl=w.context_lens.to(dev), gs=w.group_start.to(dev),
                    pl=w.prefix_lens.to(dev), out=torch.empty_like(w.query, device=dev))

    ws = pa.new_decode_workspace(base.num_seqs, base.num_q_heads, base.head_dim, maxctx, ps)

    def step(b, w, stream=None):
        pa.pa_reshape_and_cache(b["key"], b["value"], b["kc"], b["vc"], b["sm"], stream=stream)
        pa.pa_decode_shared_prefix(b["out"], b["q"], b["kc"], b["vc"], b["bt"], b["cl"], b["gs"],
                                   b["pl"], mgs, w.scale, maxctx, ps, workspace=ws,
                                   stream=stream)

    eager = {}
    for name, w in (("base", base), ("other", other)):
        b = buffers(w)
        step(b, w)
        torch.cuda.synchronize()
        eager[name] = (b["out"].clone(), b["kc"].clone(), b["vc"].clone())

    static = buffers(base)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(static, base, stream=side)        # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    fresh = buffers(base)
    for k in ("kc", "vc"):
        static[k].copy_(fresh[k])
    with torch.cuda.graph(g):
        step(static, base, stream=torch.cuda.current_stream())
    for name, w, copy_in in (("base", base, False), ("other", other, True)):
        if copy_in:
            nb = buffers(w)
            for k in ("kc", "vc", "key", "value", "sm", "q", "bt", "cl", "gs", "pl"):
                static[k].copy_(nb[k])
        g.replay()
        torch.cuda.synchronize()
        assert pa.pa_device_errors() == 0
        out, kc, vc = eager[name]
        assert torch.equal(static["out"].view(torch.int16), out.view(torch.int16)), name
        assert torch.equal(bits(static["kc"]), bits(kc)) and torch.equal(bits(static["vc"]), bits(vc))
        assert_matches_oracle(static, w, False, f"shared-prefix replay ({name})")
