"""CPU checks of the C ABI: the library builds, loads without a GPU, exports
every function include/pa.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    import pagedattention_kv_cache_attention_gb300 as pa
    from pagedattention_kv_cache_attention_gb300 import build
    build.build()
    return pa._load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_decode_reduce", "pa_decode_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from pagedattention_kv_cache_attention_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pa_[a-z_]+)\b", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared in pa.h but not exported: {missing}"
    for n in declared_functions():
        assert hasattr(lib, n)


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "pa.h"\nint main(void){return pa_version() == 4 ? 0 : 1;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only",
                    "-I", os.path.join(ROOT, "include"), str(src)], check=True)


def test_status_strings(lib):
    lib.pa_status_string.restype = ctypes.c_char_p
    assert lib.pa_status_string(0) == b"ok"
    assert lib.pa_status_string(1) == b"invalid argument"
    assert lib.pa_status_string(2) == b"unsupported shape"
    assert lib.pa_status_string(3) == b"CUDA error"
    assert lib.pa_status_string(99) == b"unknown status"


def test_partition_count_and_workspace_size(lib):
    import pagedattention_kv_cache_attention_gb300 as pa
    assert pa.pa_decode_num_partitions(1000, 0) == 1
    assert pa.pa_decode_num_partitions(512, 512) == 1
    assert pa.pa_decode_num_partitions(513, 512) == 2
    assert pa.pa_decode_num_partitions(131072, 512) == 256
    assert pa.pa_decode_workspace_size(8, 32, 128, 512, 512) == 0
    # the join counters (a fixed 256 KiB), then m, l [R, P] and o [R, P, d],
    # each 256-byte aligned
    R, P, d = 8 * 32, 256, 128
    ml = (R * P * 4 + 255) // 256 * 256
    assert pa.DECODE_COUNTER_BYTES == 256 * 1024
    assert pa.pa_decode_workspace_size(8, 32, 128, 131072, 512) == (
        pa.DECODE_COUNTER_BYTES + 2 * ml + R * P * d * 4)


def _decode_status(lib, **over):
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: every case below fails host checks first
    args = dict(out=fake, query=fake, k=fake, v=fake, bt=fake, mb=13, cl=fake, B=4, Hq=4, Hkv=4,
                d=64, bs=16, NB=64, scale=0.125, maxctx=200, ps=0, ws=None, wsb=0, dt=0, st=None)
    args.update(over)
    lib.pa_decode.argtypes = [P, P, P, P, P, ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32,
                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                              ctypes.c_float, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_size_t,
                              ctypes.c_int32, P]
    return lib.pa_decode(*args.values())


@pytest.mark.parametrize("over,status", [
    (dict(d=96), 2), (dict(d=256), 2), (dict(bs=8), 2), (dict(bs=64), 2),
    (dict(Hq=32, Hkv=2), 2),                      # group of 16
    (dict(Hq=6, Hkv=4), 1),                       # not a multiple
    (dict(dt=7), 1), (dict(ps=24), 1), (dict(ps=-16), 1), (dict(maxctx=-1), 1),
    (dict(out=None), 1), (dict(k=ctypes.c_void_p(0x10008)), 1),   # null, misaligned
    (dict(scale=float("nan")), 1), (dict(NB=0), 1), (dict(mb=0), 1),
    (dict(ps=64, ws=None, wsb=0), 1),             # split needs a workspace
    (dict(B=0), 0),                               # empty batch: nothing to do
])
def test_decode_host_validation(lib, over, status):
    assert _decode_status(lib, **over) == status


def test_reshape_host_validation(lib):
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.pa_reshape_and_cache.argtypes = [P, P, i64, i64, P, P, P, i32, i32, i32, i32, i64, i32, P]
    f = P(0x10000)
    call = lambda **o: lib.pa_reshape_and_cache(*{**dict(
        k=f, v=f, ks=512, vs=512, kc=f, vc=f, sm=f, T=4, H=4, d=128, bs=16, NB=64, dt=0, st=None),
        **o}.values())
    assert call(T=0) == 0
    assert call(d=80) == 2
    assert call(bs=48) == 2
    assert call(ks=256) == 1          # stride shorter than a row
    assert call(vs=516) == 1          # stride not a multiple of 8
    assert call(sm=None) == 1
    assert call(kc=P(0x10002)) == 1
    assert call(dt=3) == 1


def test_version(lib):
    assert lib.pa_version() == 4


def _shared_prefix_status(lib, **over):
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    fake = P(0x10000)  # never dereferenced: every case below fails host checks first
    args = dict(out=fake, query=fake, k=fake, v=fake, bt=fake, mb=160, cl=fake, gs=fake, pl=fake,
                ng=4, mgs=8, B=32, Hq=32, Hkv=8, d=128, bs=16, NB=4096, scale=0.088, maxctx=2560,
                ps=512, ws=fake, wsb=1 << 30, dt=0, st=None)
    args.update(over)
    lib.pa_decode_shared_prefix.argtypes = [P, P, P, P, P, i32, P, P, P, i32, i32, i32, i32, i32,
                                            i32, i32, ctypes.c_int64, ctypes.c_float, i32, i32, P,
                                            ctypes.c_size_t, i32, P]
    return lib.pa_decode_shared_prefix(*args.values())


@pytest.mark.parametrize("over,status", [
    (dict(gs=None), 1), (dict(pl=None), 1),                 # group arrays missing
    (dict(ng=0), 1), (dict(ng=33), 1),                      # 1 <= num_groups <= num_seqs
    (dict(mgs=0), 1), (dict(mgs=33), 1),                    # 1 <= max_group_size <= num_seqs
    (dict(ps=0), 1),                                        # sharing needs partitions
    (dict(ps=16384, maxctx=65536), 2),                      # partition beyond the kernel's table
    (dict(d=96), 2), (dict(ps=24), 1),                      # pa_decode's own checks come first
    (dict(B=65535, ng=1, mgs=65535, Hq=8, Hkv=1, maxctx=1 << 30, ps=16, mb=1 << 26),
     2),                                                    # grid x too large
    (dict(ws=None, wsb=0), 1),                              # a split needs a workspace
    (dict(B=0, ng=1, mgs=1), 0),                            # empty batch: nothing to do
])
def test_shared_prefix_host_validation(lib, over, status):
    assert _shared_prefix_status(lib, **over) == status


def _fp8_status(lib, name, **over):
    """Host checks of the FP8 entry points (bad scales, then the checks of
    their 16-bit forms); nothing is dereferenced."""
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    fake = P(0x10000)
    if name == "pa_prefill_fp8":
        args = dict(out=fake, q=fake, qs=fake, k=fake, v=fake, bt=fake, mb=64, cl=fake, B=4,
                    mq=64, Hq=32, Hkv=8, d=128, bs=16, NB=1024, scale=0.088, ks=0.5, vs=0.5, dt=0,
                    st=None)
        types = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i64, f32, f32, f32, i32, P]
    elif name == "pa_decode_shared_prefix_fp8":
        args = dict(out=fake, q=fake, k=fake, v=fake, bt=fake, mb=160, cl=fake, gs=fake, pl=fake,
                    ng=4, mgs=8, B=32, Hq=32, Hkv=8, d=128, bs=16, NB=4096, scale=0.088, ks=0.5,
                    vs=0.5, maxctx=2560, ps=512, ws=fake, wsb=1 << 30, dt=0, st=None)
        types = [P, P, P, P, P, i32, P, P, P, i32, i32, i32, i32, i32, i32, i32, i64, f32, f32, f32,
                 i32, i32, P, ctypes.c_size_t, i32, P]
    else:  # pa_copy_blocks_fp8
        args = dict(k=fake, v=fake, m=fake, n=2, Hkv=8, d=128, bs=16, NB=1024, st=None)
        types = [P, P, P, i32, i32, i32, i32, i64, P]
    args.update(over)
    f = getattr(lib, name)
    f.argtypes = types
    f.restype = i32
    return f(*args.values())


@pytest.mark.parametrize("name,over,status", [
    ("pa_prefill_fp8", dict(ks=0.0), 1), ("pa_prefill_fp8", dict(vs=float("nan")), 1),
    ("pa_prefill_fp8", dict(ks=float("inf")), 1), ("pa_prefill_fp8", dict(dt=2), 1),
    ("pa_prefill_fp8", dict(d=96), 2), ("pa_prefill_fp8", dict(Hq=72, Hkv=8), 2),
    ("pa_prefill_fp8", dict(B=0), 0),
    ("pa_decode_shared_prefix_fp8", dict(vs=-1.0), 1),
    ("pa_decode_shared_prefix_fp8", dict(ks=float("nan")), 1),
    ("pa_decode_shared_prefix_fp8", dict(dt=5), 1),
    ("pa_decode_shared_prefix_fp8", dict(gs=None), 1),
    ("pa_decode_shared_prefix_fp8", dict(ps=16384, maxctx=65536), 2),
    ("pa_decode_shared_prefix_fp8", dict(B=0, ng=1, mgs=1), 0),
    ("pa_copy_blocks_fp8", dict(d=96), 2), ("pa_copy_blocks_fp8", dict(m=None), 1),
    ("pa_copy_blocks_fp8", dict(n=0), 0),
])
def test_fp8_entry_points_host_validation(lib, name, over, status):
    assert _fp8_status(lib, name, **over) == status


def test_binding_matches_cache_type_to_entry_point(lib):
    """The Python block copies check the cache type before anything reaches
    the library: the 16-bit form refuses uint8 (FP8) caches, whose blocks are
    half the bytes, and the FP8 form refuses 16-bit caches."""
    import torch
    import pagedattention_kv_cache_attention_gb300 as pa
    m = torch.zeros(1, 2, dtype=torch.int64)
    f8 = torch.zeros(4, 2, 16, 64, dtype=torch.uint8)
    f16 = torch.zeros(4, 2, 16, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="caches must be"):
        pa.pa_copy_blocks(f8, f8, m)
    with pytest.raises(ValueError, match="caches must be"):
        pa.pa_copy_blocks_fp8(f16, f16, m)
