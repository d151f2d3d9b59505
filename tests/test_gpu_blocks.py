"""GPU parity of the whole-block moves against the oracle: copy-on-write fork
(pa_copy_blocks) and swap to a pinned host pool and back (pa_swap_blocks).
Every pool is compared bit for bit; decode after a fork or a swap round trip
must give the bit-identical output the untouched sequences had before."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


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


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _pairs(rng, nb, n, exclude=()):
    """n (src, dst) pairs: distinct destinations, none of them a source."""
    ids = rng.permutation([b for b in range(nb) if b not in set(exclude)])
    src, dst = ids[:n], ids[n:2 * n]
    return np.stack([src, dst], 1).astype(np.int64)


@pytest.mark.parametrize("name,kw", [("llama3_8b_gqa", dict(batch=8)),
                                     ("llama3_70b_cb", dict(batch=16, dtype="bf16")),
                                     ("tiny_mha", {})])
def test_copy_blocks_bitexact(pa, name, kw):
    w = W.make(name, 31, **kw)
    rng = np.random.default_rng(0)
    m = _pairs(rng, w.num_blocks, min(40, w.num_blocks // 2))
    kc, vc = w.k_cache.cuda(), w.v_cache.cuda()
    pa.pa_copy_blocks(kc, vc, torch.from_numpy(m).cuda())
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
    kh, vh = u16(w.k_cache).copy(), u16(w.v_cache).copy()
    oracle.copy_blocks(kh, vh, m)
    assert np.array_equal(u16(kc), kh) and np.array_equal(u16(vc), vh)


@pytest.mark.parametrize("name,kw", [("llama3_70b_cb", dict(batch=16)),
                                     ("llama3_8b_gqa", dict(batch=8, head_dim=64))])
def test_copy_blocks_fp8_bitexact(pa, name, kw):
    """FP8 caches (one byte per element): every pair is copied whole and no
    byte outside the destination blocks changes -- in particular the last
    blocks of the pool, which a copy sized for two-byte elements would run
    past."""
    w = W.to_fp8(W.make(name, 33, **kw))
    rng = np.random.default_rng(1)
    m = _pairs(rng, w.num_blocks, min(40, w.num_blocks // 2))
    m[0] = [w.num_blocks - 1, m[0, 1]]          # the pool's last block as a source ...
    m[1] = [m[1, 0], w.num_blocks - 2]          # ... and a block near the end as a destination
    assert len(set(m[:, 1])) == len(m) and not set(m[:, 1]) & set(m[:, 0])
    kc, vc = w.k_cache.cuda(), w.v_cache.cuda()
    pa.pa_copy_blocks_fp8(kc, vc, torch.from_numpy(m).cuda())
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
    kh, vh = w.k_cache.numpy().copy(), w.v_cache.numpy().copy()
    oracle.copy_blocks(kh, vh, m)
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)
    with pytest.raises(ValueError):
        pa.pa_copy_blocks(kc, vc, torch.from_numpy(m).cuda())   # the 16-bit form refuses uint8


def test_fork_then_write_leaves_sharer_unchanged(pa):
    """Sequences of a group share their prefix blocks.  Sequence 1 forks one
    shared block into a free block: with the same data behind a new id every
    output is bit-identical.  Then it writes a row of the fork only: every
    other sequence's output stays bit-identical, and sequence 1's matches the
    oracle."""
    w = W.make("shared_prefix_cow", 32, groups=2, group_size=4, prefix_len=2040, max_len=40)
    dev = torch.device("cuda")
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    pa.pa_reshape_and_cache(w.key.to(dev), w.value.to(dev), kc, vc, w.slot_mapping.to(dev))
    q, cl = w.query.to(dev), w.context_lens.to(dev)
    before = torch.empty_like(q)
    pa.pa_decode(before, q, kc, vc, w.block_tables.to(dev), cl, w.scale, w.max_context_len, 512)
    # fork: sequence 1 copies shared logical block 5 into a free block
    owned = set(w.block_tables.numpy().ravel().tolist())
    free = [b for b in range(w.num_blocks) if b not in owned][0]
    src = int(w.block_tables[1, 5])
    assert src == int(w.block_tables[0, 5])
    m = torch.tensor([[src, free]], dtype=torch.int64)
    pa.pa_copy_blocks(kc, vc, m.to(dev))
    bt = w.block_tables.clone()
    bt[1, 5] = free
    after = torch.empty_like(q)
    pa.pa_decode(after, q, kc, vc, bt.to(dev), cl, w.scale, w.max_context_len, 512)
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
    # same data behind a new physical id: every output bit-identical
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))
    # now the fork diverges: overwrite one row of the forked block only
    key = torch.randn(1, w.num_kv_heads, w.head_dim).to(w.torch_dtype())
    slot = torch.tensor([free * w.block_size + 3], dtype=torch.int64)
    pa.pa_reshape_and_cache(key.to(dev), key.to(dev), kc, vc, slot.to(dev))
    after2 = torch.empty_like(q)
    pa.pa_decode(after2, q, kc, vc, bt.to(dev), cl, w.scale, w.max_context_len, 512)
    torch.cuda.synchronize()
    others = [i for i in range(w.num_seqs) if i != 1]
    assert torch.equal(after2[others].view(torch.int16), before[others].view(torch.int16))
    assert not torch.equal(after2[1].view(torch.int16), before[1].view(torch.int16))
    # the oracle's own pools through the same steps: scatter, fork, write
    kh, vh = u16(w.k_cache).copy(), u16(w.v_cache).copy()
    oracle.reshape_and_cache(w.key, w.value, kh, vh, w.slot_mapping)
    oracle.copy_blocks(kh, vh, m.numpy())
    oracle.reshape_and_cache(key, key, kh, vh, slot)
    assert np.array_equal(u16(kc), kh) and np.array_equal(u16(vc), vh)
    ref = oracle.decode(w.query, kh, vh, bt, w.context_lens, w.scale, w.dtype,
                        pairs=[(1, h) for h in range(w.num_q_heads)])
    got = after2[1].float().cpu().double().numpy()
    assert np.all(np.abs(got - ref) <= 2e-3 + 1e-2 * np.abs(ref))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_swap_out_and_back_in(pa, dtype):
    """Preempt sequences 0-3: their blocks go to a pinned host pool, their
    device blocks are overwritten, then they come back into other ids."""
    w = W.make("llama3_70b_cb", 33, batch=12, dtype=dtype, max_len=2000)
    dev = torch.device("cuda")
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    pa.pa_reshape_and_cache(w.key.to(dev), w.value.to(dev), kc, vc, w.slot_mapping.to(dev))
    q, cl, bt = w.query.to(dev), w.context_lens.to(dev), w.block_tables.to(dev)
    before = torch.empty_like(q)
    pa.pa_decode(before, q, kc, vc, bt, cl, w.scale, w.max_context_len, 1024)
    nblk = w.blocks_used()
    victims = [(i, lb) for i in range(4) for lb in range(int(nblk[i]))]
    dev_ids = np.array([int(w.block_tables[i, lb]) for i, lb in victims], np.int64)
    n = len(victims)
    host_k = torch.zeros((n + 5,) + tuple(kc.shape[1:]), dtype=kc.dtype).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    out_map = torch.from_numpy(np.stack([dev_ids, np.arange(n) + 5], 1)).pin_memory()
    pa.pa_swap_blocks(kc, host_k, out_map)
    pa.pa_swap_blocks(vc, host_v, out_map)
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
    # host pool bit-exact against the oracle's swap of the same blocks out of
    # the oracle's own pool (after its scatter) into a zeroed pool
    kh = u16(w.k_cache).copy()
    vh = u16(w.v_cache).copy()
    oracle.reshape_and_cache(w.key, w.value, kh, vh, w.slot_mapping)
    assert np.array_equal(u16(kc), kh)
    exp = np.zeros((n + 5,) + tuple(kc.shape[1:]), np.uint16)
    oracle.swap_blocks(kh, exp, out_map.numpy())
    assert np.array_equal(u16(host_k), exp)
    # the freed device blocks get reused (garbage), the victims come back elsewhere
    kc[torch.from_numpy(dev_ids).to(dev)] = float("nan")
    vc[torch.from_numpy(dev_ids).to(dev)] = float("nan")
    perm = np.random.default_rng(1).permutation(dev_ids)
    in_map = torch.from_numpy(np.stack([np.arange(n) + 5, perm], 1)).to(dev)
    pa.pa_swap_blocks(host_k, kc, in_map)
    pa.pa_swap_blocks(host_v, vc, in_map)
    bt2 = w.block_tables.clone()
    for (i, lb), new in zip(victims, perm):
        bt2[i, lb] = int(new)
    after = torch.empty_like(q)
    pa.pa_decode(after, q, kc, vc, bt2.to(dev), cl, w.scale, w.max_context_len, 1024)
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))


def test_bad_block_ids_and_pageable_memory(pa):
    w = W.make("tiny_mha", 34)
    kc, vc = w.k_cache.cuda(), w.v_cache.cuda()
    m = torch.tensor([[0, w.num_blocks], [-1, 3], [2, 5]], dtype=torch.int64).cuda()
    pa.pa_copy_blocks(kc, vc, m)
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == pa.DEVERR_BAD_BLOCK
    kh, vh = u16(w.k_cache).copy(), u16(w.v_cache).copy()
    oracle.copy_blocks(kh, vh, [[2, 5]])   # only the valid pair is applied
    assert np.array_equal(u16(kc), kh) and np.array_equal(u16(vc), vh)
    import ctypes
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L = pa._load()
    L.pa_swap_blocks.argtypes = [P, P, P, i32, i64, i64, i64, P]
    L.pa_swap_blocks.restype = i32
    pageable = np.zeros((4, 4096), np.uint16)
    status = L.pa_swap_blocks(kc.data_ptr(), ctypes.c_void_p(pageable.ctypes.data),
                              m.data_ptr(), 1, 4096, w.num_blocks, 4, None)
    assert status == 1  # PA_ERR_INVALID_ARG: the device cannot reach pageable memory
