"""CPU oracle for PagedAttention decode (fp64, plain C + OpenMP).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package; the CUDA
library and its Python binding never do, and the two share no code.  The C
source ``pa_oracle.c`` states what is computed and which page and section each
step follows; this module only marshals numpy / torch CPU arrays into it.

Every function here is pinned by ``tests/test_oracle.py`` against facts the
pages or mathematics fix (the block-table worked example, brute-force
non-paged attention and torch's fp64 SDPA on tiny inputs, permutation and
copy-on-write invariance, closed forms), so no part is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_OUT = os.path.join(_HERE, "_build", "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

FP16, BF16, E4M3 = 0, 1, 2
DT = {"fp16": FP16, "bf16": BF16, "e4m3": E4M3}


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no fast-math: IEEE fp64)."""
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OUT)
    return _OUT


def _load(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int, ctypes.c_int64
    L.pa_oracle_fp16_to_f64.argtypes = [ctypes.c_uint16]
    L.pa_oracle_fp16_to_f64.restype = ctypes.c_double
    L.pa_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.pa_oracle_bf16_to_f64.restype = ctypes.c_double
    L.pa_oracle_reshape_and_cache.argtypes = [P, P, i64, i64, P, P, P, i32, i32, i32, i32, i64]
    L.pa_oracle_reshape_and_cache.restype = i32
    L.pa_oracle_gather.argtypes = [P, P, i32, ctypes.c_double, P, i32, i32, i32, i32, i32,
                                   i32, i64]
    L.pa_oracle_gather.restype = i32
    L.pa_oracle_decode.argtypes = [P, P, P, P, i32, P, P, P, P, i32, P, i32, i32, i32,
                                   i32, i32, i64, ctypes.c_float, i32, i32, ctypes.c_double,
                                   ctypes.c_double, P, i32, i32, i32]
    L.pa_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    L.pa_oracle_e4m3_to_f64.restype = ctypes.c_double
    L.pa_oracle_e4m3_from_f32.argtypes = [ctypes.c_float]
    L.pa_oracle_e4m3_from_f32.restype = ctypes.c_uint8
    L.pa_oracle_reshape_and_cache_fp8.argtypes = [P, P, i64, i64, P, P, P, i32, i32, i32, i32,
                                                  i64, i32, ctypes.c_float, ctypes.c_float]
    L.pa_oracle_reshape_and_cache_fp8.restype = i32
    L.pa_oracle_decode.restype = i32
    L.pa_oracle_lse_combine.argtypes = [P, P, P, P, P, i32, i32, i32]
    L.pa_oracle_lse_combine.restype = None
    L.pa_oracle_max_threads.restype = i32
    L.pa_oracle_prefill.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64,
                                    ctypes.c_float, i32, i32, ctypes.c_double, ctypes.c_double,
                                    i32]
    L.pa_oracle_prefill.restype = i32
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(build())
    return _lib


def _u16(x) -> np.ndarray:
    """Raw 16-bit words of an fp16/bf16 torch tensor or a uint16 numpy array."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(x).view(np.uint16)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def to_f64(raw, dtype: str) -> np.ndarray:
    """Exact fp64 value of each fp16/bf16 word (the oracle's own conversion)."""
    r = _u16(raw)
    f = lib().pa_oracle_bf16_to_f64 if dtype == "bf16" else lib().pa_oracle_fp16_to_f64
    flat = np.fromiter((f(int(v)) for v in r.ravel()), dtype=np.float64, count=r.size)
    return flat.reshape(r.shape)


def reshape_and_cache(key, value, k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping,
                      key_stride: int = -1, value_stride: int = -1) -> None:
    """Scatter the new tokens' K/V rows into the (uint16 numpy) caches in place.
    key/value: [T, Hkv, d]; caches: [NB, Hkv, bs, d]."""
    k = _u16(key)
    v = _u16(value)
    T, Hkv, d = k.shape
    NB, _, bs, _ = k_cache.shape
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
    sm = np.ascontiguousarray(slot_mapping.detach().numpy() if hasattr(slot_mapping, "detach")
                              else slot_mapping, dtype=np.int64)
    rc = lib().pa_oracle_reshape_and_cache(
        _p(k), _p(v), key_stride if key_stride >= 0 else Hkv * d,
        value_stride if value_stride >= 0 else Hkv * d, _p(k_cache), _p(v_cache), _p(sm),
        T, Hkv, d, bs, NB)
    if rc:
        raise IndexError(f"oracle reshape_and_cache: status {rc}")


def _kv(x, dtype: str) -> np.ndarray:
    """Raw storage of a cache: uint8 codes for E4M3, 16-bit words otherwise."""
    if dtype == "e4m3":
        if hasattr(x, "detach"):
            import torch
            x = x.detach().contiguous().view(torch.uint8).numpy()
        return np.ascontiguousarray(x).view(np.uint8)
    return _u16(x)


def gather(cache, block_table_row, ctx: int, kv_head: int, dtype: str,
           mult: float = 1.0) -> np.ndarray:
    """Contiguous fp64 [ctx, d] rows of one sequence's KV head, read through its
    block table (each element times ``mult``, the FP8 dequantisation scale)."""
    c = _kv(cache, dtype)
    NB, Hkv, bs, d = c.shape
    bt = _i32(block_table_row)
    out = np.empty((max(ctx, 0), d), dtype=np.float64)
    rc = lib().pa_oracle_gather(_p(out), _p(c), DT[dtype], float(mult), _p(bt), bt.shape[0],
                                ctx, Hkv, kv_head, d, bs, NB)
    if rc:
        raise IndexError(f"oracle gather: status {rc}")
    return out


def decode(query, k_cache, v_cache, block_tables, context_lens, scale: float, dtype: str,
           pairs=None, partition_size: int = 0, threads: int = 0, return_partials: bool = False,
           kv_dtype: str = None, k_scale: float = 1.0, v_scale: float = 1.0):
    """fp64 decode attention.  Returns out [n, d] for the (seq, head) ``pairs``
    (default: all, shaped [B, Hq, d]).  With ``partition_size`` > 0 the
    result is computed partition-wise and joined by log-sum-exp; with
    ``return_partials`` also returns (m, l, o) per partition.  ``kv_dtype``
    "e4m3" reads uint8 caches whose codes stand for k_scale*e / v_scale*e."""
    kv_dtype = kv_dtype or dtype
    q = _u16(query)
    kc = _kv(k_cache, kv_dtype)
    vc = _kv(v_cache, kv_dtype)
    bt = _i32(block_tables)
    cl = _i32(context_lens)
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = kc.shape
    MB = bt.shape[1] if bt.ndim == 2 else 0
    pr = None if pairs is None else np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    n = B * Hq if pr is None else pr.shape[0]
    out = np.empty((n, d), dtype=np.float64)
    maxp = 0
    pm = pl = po = None
    if return_partials:
        assert partition_size > 0
        maxp = max(1, int((cl.max() + partition_size - 1) // partition_size)) if cl.size else 1
        pm = np.empty((n, maxp), dtype=np.float64)
        pl = np.empty((n, maxp), dtype=np.float64)
        po = np.empty((n, maxp, d), dtype=np.float64)
    rc = lib().pa_oracle_decode(
        _p(out), _p(pm) if pm is not None else None, _p(pl) if pl is not None else None,
        _p(po) if po is not None else None, maxp, _p(q), _p(kc), _p(vc), _p(bt), MB, _p(cl),
        B, Hq, Hkv, d, bs, NB, float(scale), DT[dtype], DT[kv_dtype], float(k_scale),
        float(v_scale), _p(pr) if pr is not None else None, n, partition_size, threads)
    if rc:
        raise IndexError(f"oracle decode: status {rc}")
    if pr is None:
        out = out.reshape(B, Hq, d)
    if return_partials:
        return out, pm, pl, po
    return out


def prefill(query, query_start, k_cache, v_cache, block_tables, context_lens, scale: float,
            dtype: str, threads: int = 0, kv_dtype: str = None, k_scale: float = 1.0,
            v_scale: float = 1.0) -> np.ndarray:
    """fp64 causal attention of each chunk row (position ctx - q_len + t) over
    tokens 0 .. its position.  query [total_q, Hq, d]; returns the same shape.
    ``kv_dtype`` "e4m3" reads uint8 caches whose codes stand for k_scale*e /
    v_scale*e, as in ``decode``."""
    kv_dtype = kv_dtype or dtype
    q = _u16(query)
    qs = _i32(query_start)
    kc = _kv(k_cache, kv_dtype)
    vc = _kv(v_cache, kv_dtype)
    bt = _i32(block_tables)
    cl = _i32(context_lens)
    total_q, Hq, d = q.shape
    NB, Hkv, bs, _ = kc.shape
    B = cl.shape[0]
    assert qs.shape[0] == B + 1 and int(qs[-1]) == total_q
    out = np.empty((total_q, Hq, d), dtype=np.float64)
    rc = lib().pa_oracle_prefill(_p(out), _p(q), _p(qs), _p(kc), _p(vc), _p(bt), bt.shape[1],
                                 _p(cl), B, Hq, Hkv, d, bs, NB, float(scale), DT[dtype],
                                 DT[kv_dtype], float(k_scale), float(v_scale), threads)
    if rc:
        raise IndexError(f"oracle prefill: status {rc}")
    return out


def e4m3_to_f64(codes) -> np.ndarray:
    """Exact value of each E4M3 code (the oracle's own decoder)."""
    c = np.asarray(codes, dtype=np.uint8)
    f = lib().pa_oracle_e4m3_to_f64
    return np.fromiter((f(int(v)) for v in c.ravel()), dtype=np.float64,
                       count=c.size).reshape(c.shape)


def e4m3_from_f32(x) -> np.ndarray:
    """Nearest E4M3 code of each float32 (ties to even, saturating at 448)."""
    a = np.asarray(x, dtype=np.float32)
    f = lib().pa_oracle_e4m3_from_f32
    return np.fromiter((f(float(v)) for v in a.ravel()), dtype=np.uint8,
                       count=a.size).reshape(a.shape)


def reshape_and_cache_fp8(key, value, k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping,
                          dtype: str, k_scale: float, v_scale: float) -> None:
    """Scatter the new tokens' rows into uint8 E4M3 caches in place, each
    element stored as the code of float32(x) / scale."""
    k = _u16(key)
    v = _u16(value)
    T, Hkv, d = k.shape
    NB, _, bs, _ = k_cache.shape
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    sm = np.ascontiguousarray(slot_mapping.detach().numpy() if hasattr(slot_mapping, "detach")
                              else slot_mapping, dtype=np.int64)
    rc = lib().pa_oracle_reshape_and_cache_fp8(
        _p(k), _p(v), Hkv * d, Hkv * d, _p(k_cache), _p(v_cache), _p(sm), T, Hkv, d, bs, NB,
        DT[dtype], float(k_scale), float(v_scale))
    if rc:
        raise IndexError(f"oracle reshape_and_cache_fp8: status {rc}")


def lse_combine(m: np.ndarray, l: np.ndarray, o: np.ndarray, nparts) -> np.ndarray:
    """Join per-partition (m, l, o) by log-sum-exp (natural-log m)."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    n, P, d = o.shape
    npt = np.ascontiguousarray(nparts, dtype=np.int32)
    out = np.empty((n, d), dtype=np.float64)
    lib().pa_oracle_lse_combine(_p(out), _p(m), _p(l), _p(o), _p(npt), n, P, d)
    return out


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, block_mapping) -> None:
    """Copy-on-write fork ("Serving engines", How vLLM works: a write forks
    only the block being written): for every (src, dst) row of block_mapping,
    physical block dst of both caches becomes a copy of block src, all heads
    and rows.  Every source is read before any destination is written."""
    m = np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    for cache in (k_cache, v_cache):
        cache[m[:, 1]] = cache[m[:, 0]].copy()


def swap_blocks(src: np.ndarray, dst: np.ndarray, block_mapping) -> None:
    """Preemption by swapping ("Serving engines", How vLLM works: blocks move
    to host memory and back): dst block m[k, 1] = src block m[k, 0]."""
    m = np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    dst[m[:, 1]] = src[m[:, 0]]


def max_threads() -> int:
    return int(lib().pa_oracle_max_threads())
