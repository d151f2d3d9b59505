"""pa_decode_static_workspace: paged decode for callers that may not allocate
device memory (work enqueued during CUDA-graph capture, frameworks that have
reserved the whole device for their own KV pool, enqueue paths that cannot
afford an allocation's implicit device synchronisation).

The entry point is called through the C ABI with no workspace argument.  On two
calls in a row, with different inputs, its output must agree with pa_decode's
(which takes a caller-allocated workspace) within the parity tolerance used by
every GPU test here; a shape needing more scratch than the library's fixed
array is refused before anything runs.  This file is collected last, and it
builds and loads the library itself, so it also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

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
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.pa_decode_static_workspace.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64,
                                             ctypes.c_float, i32, i32, i32, P]
    L.pa_decode_static_workspace.restype = i32
    return L


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


def _static_call(L, w, t, out, max_ctx, ps):
    return L.pa_decode_static_workspace(
        out.data_ptr(), t["q"].data_ptr(), t["kc"].data_ptr(), t["vc"].data_ptr(),
        t["bt"].data_ptr(), w.max_blocks_per_seq, t["cl"].data_ptr(), w.num_seqs,
        w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.scale, max_ctx,
        ps, 0 if w.dtype == "fp16" else 1, torch.cuda.current_stream().cuda_stream)


def test_static_workspace_matches_pa_decode_on_two_calls(lib):
    import pagedattention_kv_cache_attention_gb300 as pa
    cases = [W.make("llama3_8b_gqa", 21, batch=12),                        # 8 partitions, fp16
             W.make("long_context", 22, lens=[30000, 7, 12000], dtype="bf16")]  # 59 partitions
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
        exp = ref.float().cpu().double().numpy()
        assert np.isfinite(got).all()
        assert np.all(np.abs(got - exp) <= ATOL + RTOL * np.abs(exp))


def test_static_workspace_refuses_oversized_shapes(lib):
    import pagedattention_kv_cache_attention_gb300 as pa
    w = W.make("tiny_mha", 23)
    t = _inputs(w)
    B, Hq, d = 4096, 64, 128
    max_ctx, ps = 16384, 512
    assert pa.pa_decode_workspace_size(B, Hq, d, max_ctx, ps) > STATIC_BYTES
    out = torch.empty_like(t["q"])
    status = lib.pa_decode_static_workspace(
        out.data_ptr(), t["q"].data_ptr(), t["kc"].data_ptr(), t["vc"].data_ptr(),
        t["bt"].data_ptr(), w.max_blocks_per_seq, t["cl"].data_ptr(), B, Hq, 8, d, 16,
        w.num_blocks, w.scale, max_ctx, ps, 0, None)
    assert status == 2   # PA_ERR_UNSUPPORTED, nothing enqueued
