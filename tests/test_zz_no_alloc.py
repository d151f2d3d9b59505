"""pa_decode_static_workspace: paged decode for callers that may not allocate
device memory (a framework that has reserved nearly all device memory for its
own KV pool, a plugin whose host runtime owns every allocation, a real-time
enqueue path that cannot risk an allocation's device-wide synchronisation).

The entry point is called through the C ABI with no workspace argument.  On two
calls in a row, with different inputs, its output must agree with pa_decode's
(which takes a caller-allocated workspace) and with the fp64 oracle, within
the parity tolerance used by every GPU test here.  The library's array keeps
the previous call's partials, so a sequence whose length the kernels refuse
must come out as zeros, not as a join of those stale partials.  Bad arguments
get the statuses pa_decode gives them, and a shape needing more scratch than
the array is refused before anything runs.  This file is collected last, and
it builds and loads the library itself, so it also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-2, 2e-3
STATIC_BYTES = 64 * 1024 * 1024  # PA_STATIC_WORKSPACE_BYTES in include/pa.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from pagedattention_kv_cache_attention_gb300 import build
    build.build()
    import pagedattention_kv_cache_attention_gb300 as pa
    L = pa._load()
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    L.pa_decode_static_workspace.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64,
                                             ctypes.c_float, i32, i32, i32, P]
    L.pa_decode_static_workspace.restype = i32
    L.pa_decode.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64,
                            ctypes.c_float, i32, i32, P, sz, i32, P]
    L.pa_decode.restype = i32
    assert pa.pa_device_errors() == 0
    return L


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _inputs(w):
    """Device copies of a workload with each sequence's newest token already
    written to its slot (until then that slot holds the generator's NaN)."""
    import pagedattention_kv_cache_attention_gb300 as pa
    dev = torch.device("cuda")
    t = dict(q=w.query.to(dev), kc=w.k_cache.to(dev), vc=w.v_cache.to(dev),
             bt=w.block_tables.to(dev), cl=w.context_lens.to(dev))
    pa.pa_reshape_and_cache(w.key.to(dev), w.value.to(dev), t["kc"], t["vc"],
                            w.slot_mapping.to(dev))
    return t


def _oracle(w, context_lens=None):
    kh, vh = _u16(w.k_cache).copy(), _u16(w.v_cache).copy()
    oracle.reshape_and_cache(w.key, w.value, kh, vh, w.slot_mapping)
    cl = w.context_lens if context_lens is None else context_lens
    return oracle.decode(w.query, kh, vh, w.block_tables, cl, w.scale, w.dtype)


def _static_call(L, w, t, out, max_ctx, ps, cl=None):
    return L.pa_decode_static_workspace(
        out.data_ptr(), t["q"].data_ptr(), t["kc"].data_ptr(), t["vc"].data_ptr(),
        t["bt"].data_ptr(), w.max_blocks_per_seq, (cl if cl is not None else t["cl"]).data_ptr(),
        w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks,
        w.scale, max_ctx, ps, 0 if w.dtype == "fp16" else 1,
        torch.cuda.current_stream().cuda_stream)


def _close(got, ref):
    got = np.asarray(got, dtype=np.float64)
    return np.isfinite(got).all() and np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))


def test_static_workspace_matches_pa_decode_and_oracle_on_two_calls(lib):
    import pagedattention_kv_cache_attention_gb300 as pa
    # 8 partitions (joined inside the decode kernel, fp16), then 59 partitions
    # (joined by the reduce kernel, bf16): two calls in a row on one array
    cases = [W.make("llama3_8b_gqa", 21, batch=12),
             W.make("long_context", 22, lens=[30000, 7, 12000], dtype="bf16")]
    for w in cases:
        t = _inputs(w)
        ps = 512
        assert pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.head_dim,
                                           w.max_context_len, ps) > 0
        ref = torch.empty_like(t["q"])
        pa.pa_decode(ref, t["q"], t["kc"], t["vc"], t["bt"], t["cl"], w.scale,
                     w.max_context_len, ps)
        out = torch.full_like(t["q"], float("nan"))
        assert _static_call(lib, w, t, out, w.max_context_len, ps) == 0
        torch.cuda.synchronize()
        assert pa.pa_device_errors() == 0
        got = out.float().cpu().double().numpy()
        assert _close(got, ref.float().cpu().double().numpy()), w.name
        assert _close(got, _oracle(w)), w.name


@pytest.mark.parametrize("ps", [64, 16], ids=["join-in-kernel", "join-by-reduce"])
def test_static_workspace_ignores_stale_partials(lib, ps):
    """A context length inside max_context_len but beyond the block table is
    refused by the decode kernel; the join must then take no partition, even
    though the array still holds the previous call's partials for that row."""
    import pagedattention_kv_cache_attention_gb300 as pa
    w = W.make("tiny_mha", 24, lens=[150, 190, 60, 120])
    t = _inputs(w)
    cap = w.max_blocks_per_seq * w.block_size                # 208 tokens
    max_ctx = cap + 400
    assert pa.pa_decode_num_partitions(max_ctx, ps) == (10 if ps == 64 else 38)
    # first call: every row's partials land in the array
    out = torch.empty_like(t["q"])
    assert _static_call(lib, w, t, out, max_ctx, ps) == 0
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
    assert _close(out.float().cpu().double().numpy(), _oracle(w))
    # second call: sequence 1 claims more tokens than its table can hold
    cl = w.context_lens.clone()
    cl[1] = cap + 50
    out2 = torch.full_like(t["q"], float("nan"))
    assert _static_call(lib, w, t, out2, max_ctx, ps, cl=cl.cuda()) == 0
    torch.cuda.synchronize()
    assert pa.pa_device_errors() & pa.DEVERR_BAD_LEN
    got = out2.float().cpu().double().numpy()
    assert np.all(got[1] == 0.0)                            # a refused length gives zeros
    ref = _oracle(w)
    keep = [0, 2, 3]
    assert _close(got[keep], ref[keep])


def test_static_workspace_statuses_match_pa_decode(lib):
    """Bad arguments get pa_decode's status even when the shape is too large
    for the array; a valid shape that is too large is refused as unsupported."""
    import pagedattention_kv_cache_attention_gb300 as pa
    w = W.make("tiny_mha", 23)
    t = _inputs(w)
    B, Hq, d = 4096, 64, 128
    max_ctx, ps = 16384, 512
    assert pa.pa_decode_workspace_size(B, Hq, d, max_ctx, ps) > STATIC_BYTES
    p = {k: v.data_ptr() for k, v in t.items()}
    out = torch.empty_like(t["q"])

    def both(**over):
        a = dict(Hkv=8, d=d, ps=ps, scale=w.scale)
        a.update(over)
        s_static = lib.pa_decode_static_workspace(
            out.data_ptr(), p["q"], p["kc"], p["vc"], p["bt"], w.max_blocks_per_seq, p["cl"], B,
            Hq, a["Hkv"], a["d"], 16, w.num_blocks, a["scale"], max_ctx, a["ps"], 0, None)
        s_decode = lib.pa_decode(
            out.data_ptr(), p["q"], p["kc"], p["vc"], p["bt"], w.max_blocks_per_seq, p["cl"], B,
            Hq, a["Hkv"], a["d"], 16, w.num_blocks, a["scale"], max_ctx, a["ps"], None, 0, 0,
            None)
        return s_static, s_decode

    assert both(ps=500) == (1, 1)                 # partition not a multiple of 16: invalid
    assert both(Hkv=7) == (1, 1)                  # heads not divisible: invalid
    assert both(scale=float("inf")) == (1, 1)     # non-finite scale: invalid
    assert both(d=96) == (2, 2)                   # head_dim 96: unsupported
    # a valid shape: pa_decode wants a workspace (invalid without one); the
    # array is too small for it (unsupported); nothing was enqueued
    assert both() == (2, 1)
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
