"""PagedAttention decode for GB300 (sm_103a): Python binding of libpa.

The functions here carry the names of the C ABI in ``include/pa.h`` and do
argument marshalling only: they check tensor devices, dtypes, shapes and
contiguity, pass ``data_ptr()`` values, sizes and the current CUDA stream to
the library, and turn a non-zero status into an exception.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback path, and
importing a function fails loudly when ``libpa.so`` has not been built.

PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "pa_reshape_and_cache", "pa_decode", "pa_decode_reduce", "pa_decode_workspace_size",
    "pa_decode_num_partitions", "pa_device_errors", "pa_status_string", "library_path",
    "pa_decode_static_workspace", "STATIC_WORKSPACE_BYTES", "pa_copy_blocks", "pa_swap_blocks",
    "pa_reshape_and_cache_fp8", "pa_decode_fp8", "pa_prefill", "pa_selftest_bounded_wait",
    "PaError", "DEVERR_BAD_BLOCK", "DEVERR_BAD_SLOT", "DEVERR_BAD_LEN", "DEVERR_TIMEOUT",
    "DEVERR_WORKSPACE", "DEVERR_PREFIX", "DECODE_COUNTER_BYTES", "new_decode_workspace",
    "pa_decode_shared_prefix", "pa_decode_shared_prefix_fp8", "pa_prefill_fp8",
    "pa_copy_blocks_fp8",
]

PA_FP16, PA_BF16 = 0, 1
DEVERR_BAD_BLOCK, DEVERR_BAD_SLOT, DEVERR_BAD_LEN, DEVERR_TIMEOUT = 1, 2, 4, 8
DEVERR_WORKSPACE = 16
DEVERR_PREFIX = 32
# Bytes of join counters at the start of a split-context workspace
# (PA_DECODE_COUNTER_BYTES in include/pa.h); they must be zero when a
# workspace is first used, and every pa_decode call leaves them zero.
DECODE_COUNTER_BYTES = 256 * 1024
_DT = {torch.float16: PA_FP16, torch.bfloat16: PA_BF16}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class PaError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call}: {pa_status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def _load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise ImportError(
                    f"libpa.so is not built ({_build.LIB} missing): run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            L = ctypes.CDLL(_build.LIB)
            P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            L.pa_reshape_and_cache.argtypes = [P, P, i64, i64, P, P, P, i32, i32, i32, i32, i64,
                                               i32, P]
            L.pa_reshape_and_cache.restype = i32
            L.pa_decode_num_partitions.argtypes = [i32, i32]
            L.pa_decode_num_partitions.restype = i32
            L.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
            L.pa_decode_workspace_size.restype = sz
            L.pa_decode.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64,
                                    ctypes.c_float, i32, i32, P, sz, i32, P]
            L.pa_decode.restype = i32
            L.pa_decode_reduce.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P]
            L.pa_decode_reduce.restype = i32
            L.pa_device_errors.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
            L.pa_selftest_bounded_wait.argtypes = [P]
            L.pa_selftest_bounded_wait.restype = i32
            L.pa_device_errors.restype = i32
            L.pa_status_string.argtypes = [i32]
            L.pa_status_string.restype = ctypes.c_char_p
            L.pa_version.restype = i32
            _lib = L
    return _lib


def pa_status_string(status: int) -> str:
    return _load().pa_status_string(int(status)).decode()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(call: str, status: int) -> None:
    if status != 0:
        raise PaError(call, status)


def _cuda(name: str, t: torch.Tensor, dtype=None) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.get_device() != torch.cuda.current_device():
        raise ValueError(f"{name} is on cuda:{t.get_device()}, but the calls run on the current "
                         f"device cuda:{torch.cuda.current_device()}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}: fp16 or bf16")
    return _DT[t.dtype]


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """Write key/value [T, Hkv, d] rows into k_cache/v_cache [NB, Hkv, bs, d]
    at slot_mapping[t] (int64; negative = skip), in place."""
    for n, t in (("key", key), ("value", value), ("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda(n, t, k_cache.dtype)
    _cuda("slot_mapping", slot_mapping, torch.int64)
    if not (k_cache.is_contiguous() and v_cache.is_contiguous() and slot_mapping.is_contiguous()):
        raise ValueError("caches and slot_mapping must be contiguous")
    T, Hkv, d = key.shape
    NB, Hkv2, bs, d2 = k_cache.shape
    if (Hkv, d) != (Hkv2, d2) or value.shape != key.shape or v_cache.shape != k_cache.shape:
        raise ValueError("key/value/cache shapes disagree")
    if slot_mapping.numel() != T:
        raise ValueError("slot_mapping must have one entry per token")
    for n, t in (("key", key), ("value", value)):
        if t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{n}: heads must be contiguous inside a token row")
    _check("pa_reshape_and_cache", _load().pa_reshape_and_cache(
        key.data_ptr(), value.data_ptr(), key.stride(0), value.stride(0), k_cache.data_ptr(),
        v_cache.data_ptr(), slot_mapping.data_ptr(), T, Hkv, d, bs, NB, _dtype_code(k_cache),
        _stream(stream)))


def pa_decode_num_partitions(max_context_len: int, partition_size: int) -> int:
    return int(_load().pa_decode_num_partitions(max_context_len, partition_size))


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, head_dim: int,
                             max_context_len: int, partition_size: int) -> int:
    return int(_load().pa_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len,
                                                partition_size))


def new_decode_workspace(num_seqs: int, num_q_heads: int, head_dim: int, max_context_len: int,
                         partition_size: int, device=None) -> torch.Tensor:
    """A zero-filled workspace (CUDA uint8 tensor) of pa_decode_workspace_size
    bytes, at least one byte; its join counters start at zero as pa_decode
    requires, and every pa_decode call leaves them zero, so it can be reused
    for any later call it is large enough for."""
    need = pa_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len,
                                    partition_size)
    return torch.zeros(max(1, need), dtype=torch.uint8,
                       device=device if device is not None else torch.cuda.current_device())


def pa_decode(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
              scale: float, max_context_len: int, partition_size: int = 0,
              workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Paged decode attention into ``out`` [B, Hq, d].  ``workspace`` (a CUDA
    uint8 tensor of at least pa_decode_workspace_size bytes whose first
    DECODE_COUNTER_BYTES were zero when it was first used, e.g. from
    new_decode_workspace) is allocated here, zero-filled, with torch when it
    is needed and not given."""
    dt = k_cache.dtype
    for n, t in (("out", out), ("query", query), ("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda(n, t, dt)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _cuda("block_tables", block_tables, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    if not (block_tables.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("block_tables and context_lens must be contiguous")
    B, Hq, d = query.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if out.shape != query.shape or v_cache.shape != k_cache.shape or d2 != d:
        raise ValueError("out/query/cache shapes disagree")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    need = pa_decode_workspace_size(B, Hq, d, max_context_len, partition_size)
    ws_ptr, ws_bytes = 0, 0
    if need:
        if workspace is None:
            workspace = torch.zeros(need, dtype=torch.uint8, device=query.device)
        _cuda("workspace", workspace)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check("pa_decode", _load().pa_decode(
        out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), B, Hq, Hkv, d,
        bs, NB, float(scale), int(max_context_len), int(partition_size), ws_ptr or None,
        ws_bytes, _dtype_code(k_cache), _stream(stream)))
    return out


def _shared_prefix(name, out, query, k_cache, v_cache, block_tables, context_lens, group_start,
                   prefix_lens, max_group_size, scale, scales, max_context_len, partition_size,
                   workspace, stream):
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    fp8 = scales is not None
    f = _blocks_fn(name, [P, P, P, P, P, i32, P, P, P, i32, i32, i32, i32, i32, i32, i32, i64, f32]
                   + ([f32, f32] if fp8 else []) + [i32, i32, P, ctypes.c_size_t, i32, P])
    for n, t in (("out", out), ("query", query)):
        _cuda(n, t, query.dtype)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda(n, t, torch.uint8 if fp8 else query.dtype)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for n, t in (("block_tables", block_tables), ("context_lens", context_lens),
                 ("group_start", group_start), ("prefix_lens", prefix_lens)):
        _cuda(n, t, torch.int32)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, Hq, d = query.shape
    NB, Hkv, bs, d2 = k_cache.shape
    if out.shape != query.shape or v_cache.shape != k_cache.shape or d2 != d:
        raise ValueError("out/query/cache shapes disagree")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    if prefix_lens.numel() != B or group_start.dim() != 1 or group_start.numel() < 2:
        raise ValueError("prefix_lens must be [B] and group_start [num_groups + 1]")
    need = pa_decode_workspace_size(B, Hq, d, max_context_len, partition_size)
    ws_ptr, ws_bytes = 0, 0
    if need:
        if workspace is None:
            workspace = torch.zeros(need, dtype=torch.uint8, device=query.device)
        _cuda("workspace", workspace)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(name, f(
        out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(),
        group_start.data_ptr(), prefix_lens.data_ptr(), group_start.numel() - 1,
        int(max_group_size), B, Hq, Hkv, d, bs, NB, float(scale),
        *([float(scales[0]), float(scales[1])] if fp8 else []), int(max_context_len),
        int(partition_size), ws_ptr or None, ws_bytes, _dtype_code(query), _stream(stream)))
    return out


def pa_decode_shared_prefix(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, group_start: torch.Tensor,
                            prefix_lens: torch.Tensor, max_group_size: int, scale: float,
                            max_context_len: int, partition_size: int,
                            workspace: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """pa_decode over groups of sequences sharing a prefix in the same
    physical blocks: ``group_start`` (int32 [num_groups + 1], runs of
    consecutive sequences covering the batch) and ``prefix_lens`` (int32 [B],
    shared leading tokens of each sequence, equal within a group) on the
    device; ``max_group_size`` bounds the groups' sizes.  The shared prefix's
    K/V is read once per group.  ``workspace`` as for pa_decode."""
    return _shared_prefix("pa_decode_shared_prefix", out, query, k_cache, v_cache, block_tables,
                          context_lens, group_start, prefix_lens, max_group_size, scale, None,
                          max_context_len, partition_size, workspace, stream)


def pa_decode_shared_prefix_fp8(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                                v_cache: torch.Tensor, block_tables: torch.Tensor,
                                context_lens: torch.Tensor, group_start: torch.Tensor,
                                prefix_lens: torch.Tensor, max_group_size: int, scale: float,
                                k_scale: float, v_scale: float, max_context_len: int,
                                partition_size: int, workspace: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """pa_decode_shared_prefix over uint8 FP8 E4M3 caches (codes times
    k_scale / v_scale), fp16 or bf16 queries and output."""
    return _shared_prefix("pa_decode_shared_prefix_fp8", out, query, k_cache, v_cache,
                          block_tables, context_lens, group_start, prefix_lens, max_group_size,
                          scale, (k_scale, v_scale), max_context_len, partition_size, workspace,
                          stream)


def pa_decode_reduce(out: torch.Tensor, workspace: torch.Tensor, context_lens: torch.Tensor,
                     max_context_len: int, partition_size: int, stream=None) -> torch.Tensor:
    """Join split-context partials in ``workspace`` into ``out`` [B, Hq, d]."""
    _cuda("out", out)
    _cuda("workspace", workspace)
    _cuda("context_lens", context_lens, torch.int32)
    if not (out.is_contiguous() and workspace.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("out, workspace and context_lens must be contiguous")
    B, Hq, d = out.shape
    _check("pa_decode_reduce", _load().pa_decode_reduce(
        out.data_ptr(), workspace.data_ptr(), context_lens.data_ptr(), B, Hq, d,
        int(max_context_len), int(partition_size), _dtype_code(out), _stream(stream)))
    return out


# Size of the library's own scratch array used by pa_decode_static_workspace
# (PA_STATIC_WORKSPACE_BYTES in include/pa.h).
STATIC_WORKSPACE_BYTES = 64 * 1024 * 1024


def pa_decode_static_workspace(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                               v_cache: torch.Tensor, block_tables: torch.Tensor,
                               context_lens: torch.Tensor, scale: float, max_context_len: int,
                               partition_size: int = 0, stream=None) -> torch.Tensor:
    """pa_decode for callers that may not allocate device memory (a framework
    that has reserved nearly all device memory for its own KV pool, a plugin
    whose host runtime owns every allocation, a real-time enqueue path that
    cannot risk an allocation's device-wide synchronisation): the
    split-context partials and join counters go to a fixed 64 MiB array the
    library carries, so neither this binding nor the library allocates.
    Shapes needing more scratch than that raise PaError (unsupported shape).
    All calls on a device share the array; calls that overlap on the GPU race."""
    L = _load()
    if not getattr(L.pa_decode_static_workspace, "argtypes", None):
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.pa_decode_static_workspace.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                                 i64, ctypes.c_float, i32, i32, i32, P]
        L.pa_decode_static_workspace.restype = i32
    dt = k_cache.dtype
    for n, t in (("out", out), ("query", query), ("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda(n, t, dt)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _cuda("block_tables", block_tables, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    B, Hq, d = query.shape
    NB, Hkv, bs, _ = k_cache.shape
    _check("pa_decode_static_workspace", L.pa_decode_static_workspace(
        out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), B, Hq, Hkv, d,
        bs, NB, float(scale), int(max_context_len), int(partition_size), _dtype_code(k_cache),
        _stream(stream)))
    return out


def _blocks_fn(name: str, argtypes):
    L = _load()
    f = getattr(L, name)
    if not getattr(f, "argtypes", None):
        f.argtypes = argtypes
        f.restype = ctypes.c_int32
    return f


def _copy_blocks(name, k_cache, v_cache, block_mapping, dtypes, stream):
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f = _blocks_fn(name, [P, P, P, i32, i32, i32, i32, i64, P])
    if k_cache.dtype not in dtypes:
        raise ValueError(f"{name}: caches must be {' or '.join(str(d) for d in dtypes)}")
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda(n, t, k_cache.dtype)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _cuda("block_mapping", block_mapping, torch.int64)
    if block_mapping.dim() != 2 or block_mapping.shape[1] != 2 or not block_mapping.is_contiguous():
        raise ValueError("block_mapping must be a contiguous [n, 2] tensor")
    NB, Hkv, bs, d = k_cache.shape
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    _check(name, f(k_cache.data_ptr(), v_cache.data_ptr(), block_mapping.data_ptr(),
                   block_mapping.shape[0], Hkv, d, bs, NB, _stream(stream)))


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, block_mapping: torch.Tensor,
                   stream=None) -> None:
    """Copy-on-write fork: for each row (src, dst) of ``block_mapping`` (CUDA
    int64 [n, 2]), physical block dst of both caches (fp16 or bf16) becomes a
    copy of block src.  Destinations distinct and not also sources."""
    _copy_blocks("pa_copy_blocks", k_cache, v_cache, block_mapping,
                 (torch.float16, torch.bfloat16), stream)


def pa_copy_blocks_fp8(k_cache: torch.Tensor, v_cache: torch.Tensor, block_mapping: torch.Tensor,
                       stream=None) -> None:
    """pa_copy_blocks over uint8 FP8 E4M3 caches."""
    _copy_blocks("pa_copy_blocks_fp8", k_cache, v_cache, block_mapping, (torch.uint8,), stream)


def pa_swap_blocks(src: torch.Tensor, dst: torch.Tensor, block_mapping: torch.Tensor,
                   stream=None) -> None:
    """Move whole blocks between pools [NB, ...] (one cache): dst block
    mapping[k, 1] = src block mapping[k, 0].  Each of src, dst is a CUDA tensor
    or a pinned CPU tensor; ``block_mapping`` is int64 [n, 2] on the GPU or in
    pinned CPU memory.  The copy runs as one kernel on ``stream``."""
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f = _blocks_fn("pa_swap_blocks", [P, P, P, i32, i64, i64, i64, P])
    for n, t in (("src", src), ("dst", dst), ("block_mapping", block_mapping)):
        if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{n} must be a CUDA tensor or a pinned CPU tensor")
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if block_mapping.dtype != torch.int64 or block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be int64 [n, 2]")
    if src.dtype != dst.dtype or src.shape[1:] != dst.shape[1:]:
        raise ValueError("src and dst must have the same dtype and block shape")
    block_bytes = src[0].numel() * src.element_size() if src.shape[0] else 0
    _check("pa_swap_blocks", f(src.data_ptr(), dst.data_ptr(), block_mapping.data_ptr(),
                               block_mapping.shape[0], block_bytes, src.shape[0], dst.shape[0],
                               _stream(stream)))


def pa_reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                             v_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                             v_scale: float, stream=None) -> None:
    """Write key/value [T, Hkv, d] (fp16/bf16) into uint8 FP8 E4M3 caches
    [NB, Hkv, bs, d] at slot_mapping[t], each element as the code of x/scale."""
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f = _blocks_fn("pa_reshape_and_cache_fp8", [P, P, i64, i64, P, P, P, i32, i32, i32, i32,
                                                 i64, i32, f32, f32, P])
    for n, t in (("key", key), ("value", value)):
        _cuda(n, t, key.dtype)
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n}: heads must be contiguous inside a token row")
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda(n, t, torch.uint8)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _cuda("slot_mapping", slot_mapping, torch.int64)
    T, Hkv, d = key.shape
    NB, Hkv2, bs, d2 = k_cache.shape
    if (Hkv, d) != (Hkv2, d2) or value.shape != key.shape or v_cache.shape != k_cache.shape:
        raise ValueError("key/value/cache shapes disagree")
    _check("pa_reshape_and_cache_fp8", f(
        key.data_ptr(), value.data_ptr(), key.stride(0), value.stride(0), k_cache.data_ptr(),
        v_cache.data_ptr(), slot_mapping.data_ptr(), T, Hkv, d, bs, NB, _dtype_code(key),
        float(k_scale), float(v_scale), _stream(stream)))


def pa_decode_fp8(out: torch.Tensor, query: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                  scale: float, k_scale: float, v_scale: float, max_context_len: int,
                  partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """Paged decode attention over uint8 FP8 E4M3 caches (codes times
    k_scale / v_scale) into ``out`` [B, Hq, d] (fp16 or bf16 queries and output)."""
    P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    f = _blocks_fn("pa_decode_fp8", [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64, f32,
                                     f32, f32, i32, i32, P, sz, i32, P])
    for n, t in (("out", out), ("query", query)):
        _cuda(n, t, query.dtype)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda(n, t, torch.uint8)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _cuda("block_tables", block_tables, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    B, Hq, d = query.shape
    NB, Hkv, bs, _ = k_cache.shape
    need = pa_decode_workspace_size(B, Hq, d, max_context_len, partition_size)
    ws_ptr, ws_bytes = 0, 0
    if need:
        if workspace is None:
            workspace = torch.zeros(need, dtype=torch.uint8, device=query.device)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check("pa_decode_fp8", f(
        out.data_ptr(), query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), B, Hq, Hkv, d,
        bs, NB, float(scale), float(k_scale), float(v_scale), int(max_context_len),
        int(partition_size), ws_ptr or None, ws_bytes, _dtype_code(query), _stream(stream)))
    return out


def _prefill(name, out, query, query_start, k_cache, v_cache, block_tables, context_lens, scale,
             scales, max_q_len, stream):
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    fp8 = scales is not None
    f = _blocks_fn(name, [P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i64, f32]
                   + ([f32, f32] if fp8 else []) + [i32, P])
    for n, t in (("out", out), ("query", query)):
        _cuda(n, t, query.dtype)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _cuda(n, t, torch.uint8 if fp8 else query.dtype)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for n, t in (("query_start", query_start), ("block_tables", block_tables),
                 ("context_lens", context_lens)):
        _cuda(n, t, torch.int32)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    total_q, Hq, d = query.shape
    NB, Hkv, bs, _ = k_cache.shape
    B = context_lens.numel()
    if query_start.numel() != B + 1 or out.shape != query.shape:
        raise ValueError("query_start must have num_seqs + 1 entries; out must match query")
    _check(name, f(out.data_ptr(), query.data_ptr(), query_start.data_ptr(), k_cache.data_ptr(),
                   v_cache.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
                   context_lens.data_ptr(), B, int(max_q_len), Hq, Hkv, d, bs, NB, float(scale),
                   *([float(scales[0]), float(scales[1])] if fp8 else []), _dtype_code(query),
                   _stream(stream)))
    return out


def pa_prefill(out: torch.Tensor, query: torch.Tensor, query_start: torch.Tensor,
               k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
               context_lens: torch.Tensor, scale: float, max_q_len: int,
               stream=None) -> torch.Tensor:
    """Causal chunked-prefill attention into ``out`` [total_q, Hq, d]: row t of
    sequence i's chunk (rows query_start[i]..query_start[i+1]-1) sits at
    position context_lens[i] - q_len_i + t and attends to tokens 0..that."""
    return _prefill("pa_prefill", out, query, query_start, k_cache, v_cache, block_tables,
                    context_lens, scale, None, max_q_len, stream)


def pa_prefill_fp8(out: torch.Tensor, query: torch.Tensor, query_start: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                   context_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float,
                   max_q_len: int, stream=None) -> torch.Tensor:
    """pa_prefill over uint8 FP8 E4M3 caches (codes times k_scale / v_scale),
    fp16 or bf16 queries and output."""
    return _prefill("pa_prefill_fp8", out, query, query_start, k_cache, v_cache, block_tables,
                    context_lens, scale, (k_scale, v_scale), max_q_len, stream)


def pa_selftest_bounded_wait(stream=None) -> None:
    """Launch the wait-limit self-test: one CTA waits on a barrier nothing
    completes, gives up after about a second and sets DEVERR_TIMEOUT."""
    _check("pa_selftest_bounded_wait", _load().pa_selftest_bounded_wait(_stream(stream)))


def pa_device_errors(stream=None) -> int:
    """Wait for ``stream`` and return (and clear) the device error bits."""
    flags = ctypes.c_uint32(0)
    _check("pa_device_errors", _load().pa_device_errors(_stream(stream), ctypes.byref(flags)))
    return int(flags.value)
