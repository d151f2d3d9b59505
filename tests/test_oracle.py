"""Pins for the CPU oracle: each test ties the oracle to something other than
itself -- a fact the pages print, a closed form, an invariant the pages imply,
a library routine, or brute force on tiny inputs.  CPU only.

Pages cited (title, section):
  [SHOOT]  "LLM Serving Engine Shootout", 3.1 PagedAttention Mechanics
           (block table, A_ij = q_i.k_j / sqrt(d_head), k_j via BlockTable[floor(j/B)])
  [ZHI]    zhichai.net Chinese original, section 1 block-table diagram
           (tokens 0-15 -> physical #7, tokens 16-31 -> physical #2)
  [RAGY]   "Inference Engines" (ragyfied.com), PagedAttention (waste under one
           block per sequence; two sequences may point at the same block)
  [ENG]    "Serving engines", How vLLM works (block table + slot mapping,
           physical placement anywhere in the pool, copy-on-write)
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _after_scatter(w):
    kc = w.k_cache.clone().view(torch.int16).numpy().view(np.uint16)
    vc = w.v_cache.clone().view(torch.int16).numpy().view(np.uint16)
    oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slot_mapping)
    return kc, vc


def _decode(w, **kw):
    kc, vc = _after_scatter(w)
    return oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype, **kw)


def _contiguous_np(cache_u16, bt_row, ctx, kvh, dtype):
    """Independent gather for brute force: numpy fancy indexing on the block table."""
    bs = cache_u16.shape[2]
    j = np.arange(ctx)
    phys = np.asarray(bt_row)[j // bs]
    rows = cache_u16[phys, kvh, j % bs, :]
    if dtype == "fp16":
        return rows.view(np.float16).astype(np.float64)
    return (rows.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- conversions

def pin_fp16_conversion():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.to_f64(bits, "fp16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def pin_bf16_conversion():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.to_f64(bits, "bf16")
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


# ------------------------------------------------------------- paging facts

def pin_block_table_worked_example():
    """[ZHI]: logical block 0 -> physical #7, logical block 1 -> physical #2."""
    g = json.load(open(os.path.join(GOLDEN, "block_table_worked_example.json")))
    bs, d, NB = g["block_size"], 8, 8
    # every cache row holds its own (block, row) address, so a gathered row names its source
    cache = np.zeros((NB, 1, bs, d), dtype=np.float16)
    for b in range(NB):
        for r in range(bs):
            cache[b, 0, r, 0] = b
            cache[b, 0, r, 1] = r
    out = oracle.gather(cache.view(np.uint16), np.array(g["block_table"]), g["context_len"], 0, "fp16")
    got = [[int(x[0]), int(x[1])] for x in out]
    assert got == g["expected_physical_rows"]


def pin_scatter_slot_placement():
    """[ENG] slot mapping, plain reading: slot = physical_block * bs + offset.
    Token written at slot 7*16+5 lands in physical block 7, row 5, every KV
    head, and nothing else changes."""
    NB, Hkv, bs, d = 8, 2, 16, 8
    kc = np.zeros((NB, Hkv, bs, d), dtype=np.uint16)
    vc = np.zeros((NB, Hkv, bs, d), dtype=np.uint16)
    key = np.arange(1, 1 + 2 * Hkv * d, dtype=np.uint16).reshape(2, Hkv, d)
    val = key + 1000
    slots = np.array([7 * 16 + 5, -1], dtype=np.int64)
    oracle.reshape_and_cache(key, val, kc, vc, slots)
    exp_k = np.zeros_like(kc)
    exp_k[7, :, 5, :] = key[0]
    exp_v = np.zeros_like(vc)
    exp_v[7, :, 5, :] = val[0]
    assert np.array_equal(kc, exp_k) and np.array_equal(vc, exp_v)


def pin_scatter_roundtrip_workload():
    """The new token written through its slot is the last row the sequence's
    block table reaches ([SHOOT] gather rule, [ENG] slot mapping)."""
    w = W.make("llama3_70b_cb", 3, batch=6, max_len=300)
    kc, vc = _after_scatter(w)
    for i in range(w.num_seqs):
        c = int(w.context_lens[i])
        for h in range(w.num_kv_heads):
            rows = oracle.gather(kc, w.block_tables[i], c, h, w.dtype)
            ref = w.key[i, h].float().double().numpy()
            assert np.array_equal(rows[c - 1], ref)


def pin_identity_v_probe():
    """Equal keys + one-hot V per physical slot: the output times ctx is the
    indicator of exactly the slots the block table reaches ([SHOOT], [ZHI])."""
    NB, bs, d = 4, 16, 64
    rng = np.random.default_rng(1)
    perm = rng.permutation(NB)
    kc = np.ones((NB, 1, bs, d), dtype=np.float16)
    vc = np.zeros((NB, 1, bs, d), dtype=np.float16)
    for b in range(NB):
        for r in range(bs):
            vc[b, 0, r, b * bs + r] = 1.0
    for ctx in (1, 15, 16, 17, 40, 64):
        bt = perm[: (ctx + bs - 1) // bs].astype(np.int32)[None, :]
        q = np.full((1, 1, d), 0.25, dtype=np.float16)
        out = oracle.decode(q.view(np.uint16), kc.view(np.uint16), vc.view(np.uint16), bt,
                            np.array([ctx], np.int32), 0.125, "fp16")[0, 0]
        expect = np.zeros(d)
        for j in range(ctx):
            expect[bt[0, j // bs] * bs + j % bs] = 1.0
        assert np.allclose(out * ctx, expect, rtol=0, atol=1e-12)


# ------------------------------------------------------- attention vs brute force

def _brute(w, kc, vc):
    """Textbook non-paged attention on contiguous copies (numpy fp64)."""
    G = w.num_q_heads // w.num_kv_heads
    raw = w.query.view(torch.int16).numpy().view(np.uint16)
    q = raw.view(np.float16).astype(np.float64) if w.dtype == "fp16" else \
        (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = np.zeros((w.num_seqs, w.num_q_heads, w.head_dim))
    for i in range(w.num_seqs):
        c = int(w.context_lens[i])
        for h in range(w.num_q_heads):
            if c == 0:
                continue
            K = _contiguous_np(kc, w.block_tables[i].numpy(), c, h // G, w.dtype)
            V = _contiguous_np(vc, w.block_tables[i].numpy(), c, h // G, w.dtype)
            s = float(np.float32(w.scale)) * (K @ q[i, h])
            p = np.exp(s - s.max())
            out[i, h] = (p[:, None] * V).sum(0) / p.sum()
    return out


def _tiny_cases():
    return [W.make("tiny_mha", 0, head_dim=64),
            W.make("tiny_mha", 1, lens=[1, 16, 17, 33], head_dim=64),
            W.make("llama3_8b_gqa", 2, batch=3, lens=[5, 40, 77], head_dim=64, num_q_heads=8,
                   num_kv_heads=2),
            W.make("llama3_70b_cb", 4, lens=[31, 32, 33], head_dim=64, num_q_heads=16,
                   num_kv_heads=2, dtype="bf16")]


def pin_brute_force_textbook():
    for w in _tiny_cases():
        kc, vc = _after_scatter(w)
        got = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
        ref = _brute(w, kc, vc)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def pin_torch_sdpa_fp64():
    """Library routine: torch scaled_dot_product_attention in fp64 on CPU over
    the contiguous K/V, KV heads repeated for each query head group."""
    F = torch.nn.functional
    for w in _tiny_cases():
        kc, vc = _after_scatter(w)
        got = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
        G = w.num_q_heads // w.num_kv_heads
        for i in range(w.num_seqs):
            c = int(w.context_lens[i])
            Ks = np.stack([_contiguous_np(kc, w.block_tables[i].numpy(), c, h, w.dtype)
                           for h in range(w.num_kv_heads)])
            Vs = np.stack([_contiguous_np(vc, w.block_tables[i].numpy(), c, h, w.dtype)
                           for h in range(w.num_kv_heads)])
            K = torch.from_numpy(Ks).repeat_interleave(G, 0)[None]
            V = torch.from_numpy(Vs).repeat_interleave(G, 0)[None]
            q = w.query[i].to(torch.float64)[None, :, None, :]
            ref = F.scaled_dot_product_attention(q, K, V, scale=float(np.float32(w.scale)))
            assert np.allclose(got[i], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ invariants

def pin_permutation_invariance():
    """[ENG]/[ZHI]: a block may sit anywhere in the pool; relabelling physical
    ids (pool and tables together) leaves every output bit-identical."""
    for w in _tiny_cases()[:3]:
        a = _decode(w)
        b = _decode(w.permuted(11))
        assert np.array_equal(a, b)


def pin_copy_on_write_sharing():
    """[RAGY]/[ENG]: sequences pointing at the same physical prefix blocks give
    bit-identical results to the same data copied into private blocks."""
    for P in (64, 40):  # full shared blocks; and a partial prefix block copied per sequence
        w = W.make("shared_prefix_cow", 5, groups=2, group_size=3, prefix_len=P, max_len=20,
                   head_dim=64)
        u = w.unshared()
        assert u.num_blocks > w.num_blocks
        assert np.array_equal(_decode(w), _decode(u))


def pin_gqa_equals_repeated_mha():
    """Query head h of a GQA layout reads KV head h // G: same result as MHA
    with every KV head stored G times."""
    w = W.make("llama3_8b_gqa", 6, lens=[3, 50, 96], head_dim=64, num_q_heads=8, num_kv_heads=2)
    kc, vc = _after_scatter(w)
    got = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    G = 4
    kcm = np.repeat(kc, G, axis=1)
    vcm = np.repeat(vc, G, axis=1)
    ref = oracle.decode(w.query, kcm, vcm, w.block_tables, w.context_lens, w.scale, w.dtype)
    assert np.array_equal(got, ref)


def pin_equal_keys_give_mean():
    """Closed form: equal logits -> uniform softmax -> arithmetic mean of V."""
    w = W.make("tiny_mha", 7, lens=[1, 9, 40, 200])
    kc, vc = _after_scatter(w)
    kc[:] = np.float16(0.5).view(np.uint16)
    out = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    for i in range(w.num_seqs):
        c = int(w.context_lens[i])
        for h in range(w.num_q_heads):
            V = _contiguous_np(vc, w.block_tables[i].numpy(), c, h, "fp16")
            assert np.allclose(out[i, h], V.mean(0), rtol=1e-13, atol=1e-15)


def pin_single_token_returns_its_value():
    """ctx = 1: the softmax weight is exactly 1, so o = v_0."""
    w = W.make("tiny_mha", 8, lens=[1, 1, 1, 1])
    kc, vc = _after_scatter(w)
    out = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    ref = w.value.double().numpy()
    assert np.array_equal(out, ref)


def pin_logit_shift_invariance():
    """Adding one constant to every logit of a row leaves the output unchanged:
    a K column that is constant over tokens makes q's entry there a shift."""
    w = W.make("tiny_mha", 9, lens=[5, 60, 120, 177])
    kc, vc = _after_scatter(w)
    kc[..., -1] = np.float16(1.0).view(np.uint16)
    q1 = w.query.clone()
    q2 = w.query.clone()
    q1[..., -1] = 0.0
    q2[..., -1] = 3.0
    a = oracle.decode(q1, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    b = oracle.decode(q2, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-13)
    assert not np.array_equal(q1, q2)


def pin_dominant_key():
    """A key whose logit exceeds the others by > 40 takes all the weight:
    o = its V row to within e^-40 relative."""
    w = W.make("tiny_mha", 10, lens=[30, 30, 30, 30])
    kc, vc = _after_scatter(w)
    j = 17
    for i in range(w.num_seqs):
        phys = int(w.block_tables[i, j // 16])
        for h in range(w.num_q_heads):
            qv = w.query[i, h].float().numpy()
            kc[phys, h, j % 16, :] = (np.sign(qv) * 60.0).astype(np.float16).view(np.uint16)
    out = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    for i in range(w.num_seqs):
        phys = int(w.block_tables[i, j // 16])
        for h in range(w.num_q_heads):
            v = vc[phys, h, j % 16, :].view(np.float16).astype(np.float64)
            assert np.allclose(out[i, h], v, rtol=0, atol=1e-12)


def pin_golden_closed_form():
    g = json.load(open(os.path.join(GOLDEN, "closed_form_two_keys.json")))
    d, bs, NB = g["head_dim"], g["block_size"], g["num_blocks"]
    kc = np.zeros((NB, 1, bs, d), np.float16)
    vc = np.zeros((NB, 1, bs, d), np.float16)
    phys = g["block_table"][0]
    for j, row in enumerate(g["k_rows_nonzero"]):
        kc[phys, 0, j, : len(row)] = row
    for j, row in enumerate(g["v_rows_nonzero"]):
        vc[phys, 0, j, : len(row)] = row
    q = np.zeros((1, 1, d), np.float16)
    q[0, 0, : len(g["q_nonzero"])] = g["q_nonzero"]
    out = oracle.decode(q.view(np.uint16), kc.view(np.uint16), vc.view(np.uint16),
                        np.array([g["block_table"]], np.int32), np.array([2], np.int32),
                        g["scale"], "fp16")[0, 0]
    exp = np.zeros(d)
    exp[:2] = g["expected_out_nonzero"]
    assert np.allclose(out, exp, rtol=1e-15, atol=1e-16)


def pin_zero_context():
    """Reading taken: a sequence with no tokens gives a zero output."""
    w = W.make("tiny_mha", 12, lens=[0, 5, 0, 16])
    out = _decode(w)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isfinite(out))


def pin_partitions_join_to_unsplit():
    """Split-context reading: partition-wise softmax joined by log-sum-exp
    equals the unsplit result (fp64, 1e-12), for several partition sizes."""
    w = W.make("llama3_8b_gqa", 13, lens=[1, 16, 100, 513, 1100], head_dim=64, num_q_heads=8,
               num_kv_heads=2)
    kc, vc = _after_scatter(w)
    ref = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    for ps in (16, 64, 512, 2048):
        got, m, l, o = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale,
                                     w.dtype, partition_size=ps, return_partials=True)
        assert np.allclose(got.reshape(ref.shape), ref, rtol=1e-12, atol=1e-13)
        nparts = np.repeat((w.context_lens.numpy() + ps - 1) // ps, w.num_q_heads)
        joined = oracle.lse_combine(m, l, o, nparts)
        assert np.allclose(joined.reshape(ref.shape), ref, rtol=1e-12, atol=1e-13)


def pin_poison_never_read():
    """Free blocks and tail slots hold NaN; every oracle output is finite, so
    the oracle reads no slot outside a sequence's tokens."""
    for name, kw in (("tiny_mha", {}), ("llama3_70b_cb", dict(batch=5, max_len=200)),
                     ("shared_prefix_cow", dict(groups=2, group_size=2, prefix_len=40, max_len=30,
                                                head_dim=64))):
        out = _decode(W.make(name, 14, **kw))
        assert np.all(np.isfinite(out))


def pin_waste_under_one_block():
    """[RAGY]: waste is under one block per sequence."""
    for name in W.NAMES:
        kw = dict(batch=16, max_len=3000) if name in ("llama3_8b_gqa", "llama3_70b_cb") else {}
        if name == "long_context":
            kw = dict(lens=[100, 2000])
        if name == "shared_prefix_cow":
            kw = dict(groups=2, group_size=2)
        w = W.make(name, 15, **kw)
        ctx = w.context_lens.numpy().astype(np.int64)
        waste = w.blocks_used() * w.block_size - ctx
        assert np.all(waste < w.block_size) and np.all(waste >= 0)


def _fork_case():
    """Two sequences of one tiny pool share every physical block; the second
    then forks its last block into a free block and writes its new token there."""
    w = W.make("tiny_mha", 16, lens=[40, 40], num_q_heads=2, num_kv_heads=2)
    w.block_tables[1] = w.block_tables[0]
    w.slot_mapping[1] = -1  # the shared slot of token 39 is written once, by sequence 0
    kc, vc = _after_scatter(w)
    return w, kc, vc


def pin_copy_on_write_fork():
    """[ENG] copy-on-write: the second sequence forks the shared block it is
    about to write and writes its new token (position 40) into the fork.  The
    other sequence's output is bit-identical to before, and the writer reads
    the shared rows followed by its own new token."""
    w, kc, vc = _fork_case()
    before = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    last = int(w.block_tables[1, 2])
    owned = set(w.block_tables[0].numpy().tolist())
    free = next(b for b in range(w.num_blocks) if b not in owned)
    oracle.copy_blocks(kc, vc, [[last, free]])
    w.block_tables[1, 2] = free
    new_k = (np.arange(2 * 64) % 7).astype(np.float16).reshape(1, 2, 64)
    oracle.reshape_and_cache(new_k.view(np.uint16), new_k.view(np.uint16), kc, vc,
                             np.array([free * 16 + 8], np.int64))
    w.context_lens[1] = 41
    after = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    assert np.array_equal(after[0], before[0])
    for h in range(2):
        rows0 = oracle.gather(kc, w.block_tables[0], 40, h, "fp16")
        rows1 = oracle.gather(kc, w.block_tables[1], 41, h, "fp16")
        assert np.array_equal(rows1[:40], rows0)
        assert np.array_equal(rows1[40], new_k[0, h].astype(np.float64))


def pin_swap_out_and_back():
    """[ENG] preemption by swapping: a sequence's blocks moved to a host pool
    and back into other physical ids, with its table remapped, decode to the
    bit-identical output."""
    w = W.make("llama3_70b_cb", 17, lens=[70, 5, 33, 300, 200], head_dim=64, num_q_heads=4,
               num_kv_heads=2)
    kc, vc = _after_scatter(w)
    before = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    used = w.block_tables[0, :3].numpy().astype(np.int64)
    host_k = np.zeros((8,) + kc.shape[1:], np.uint16)
    host_v = np.zeros_like(host_k)
    oracle.swap_blocks(kc, host_k, np.stack([used, np.arange(3)], 1))
    oracle.swap_blocks(vc, host_v, np.stack([used, np.arange(3)], 1))
    kc[used] = 0xFFFF  # the freed blocks are reused by someone else
    vc[used] = 0xFFFF
    owned = set(w.block_tables.numpy().ravel().tolist())
    fresh = np.array([b for b in range(w.num_blocks) if b not in owned][:3], np.int64)
    oracle.swap_blocks(host_k, kc, np.stack([np.arange(3), fresh], 1))
    oracle.swap_blocks(host_v, vc, np.stack([np.arange(3), fresh], 1))
    w.block_tables[0, :3] = torch.from_numpy(fresh.astype(np.int32))
    after = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
    assert np.array_equal(after, before)


# --------------------------------------------------------------- FP8 caches

def pin_e4m3_decode_all_codes():
    """The oracle's E4M3 decoder against torch's float8_e4m3fn on all 256 codes."""
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and nan.sum() == 2
    assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def pin_e4m3_encode_matches_torch():
    """Nearest code, ties to even: equal to torch's cast for every fp16 value
    below the first magnitude torch turns into NaN (464), and for random
    float32 values in range."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float32)
    rng = np.random.default_rng(0)
    x = np.concatenate([x, rng.uniform(-463, 463, 20000).astype(np.float32),
                        rng.standard_normal(20000).astype(np.float32) * 1e-2])
    x = x[np.isfinite(x) & (np.abs(x) < 464)]
    mine = oracle.e4m3_from_f32(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def pin_e4m3_saturates():
    """Beyond the largest magnitude the encoder clamps to +-448 (saturating
    conversion), NaN stays NaN."""
    x = np.array([464.0, 470.0, 479.9, 480.0, 1e6, np.inf, -500.0, -np.inf, np.nan],
                 dtype=np.float32)
    got = oracle.e4m3_from_f32(x)
    assert got.tolist()[:8] == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert got[8] & 0x7F == 0x7F


def pin_fp8_scatter_codes():
    """reshape_and_cache into FP8 caches stores code(float32(x) / scale) at the
    slot (checked against torch's cast), and nothing else changes."""
    w = W.make("llama3_8b_gqa", 18, batch=3, max_len=700)
    f8 = W.to_fp8(w)
    kc, vc = f8.k_cache.numpy().copy(), f8.v_cache.numpy().copy()
    oracle.reshape_and_cache_fp8(w.key, w.value, kc, vc, w.slot_mapping, "fp16", f8.k_scale,
                                 f8.v_scale)
    changed = np.argwhere(kc != f8.k_cache.numpy())
    for i in range(w.num_seqs):
        s = int(w.slot_mapping[i])
        blk, off = s // w.block_size, s % w.block_size
        exp_k = (w.key[i].float() / torch.tensor(f8.k_scale, dtype=torch.float32)).clamp(-448, 448)
        exp_k = exp_k.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(kc[blk, :, off, :], exp_k)
        exp_v = (w.value[i].float() / torch.tensor(f8.v_scale, dtype=torch.float32)).clamp(-448, 448)
        assert np.array_equal(vc[blk, :, off, :],
                              exp_v.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    slots = {(int(s) // w.block_size, int(s) % w.block_size) for s in w.slot_mapping}
    assert all((int(b), int(o)) in slots for b, _, o, _ in changed)


def pin_fp8_decode_equals_16bit_when_exact():
    """With power-of-two scales every dequantised element is exactly an fp16
    value, so the FP8 decode must equal the fp16 decode of those values bit
    for bit; a V scale multiplies the output; a K scale is a logit scale."""
    w = W.make("llama3_8b_gqa", 19, lens=[3, 70, 260], head_dim=64, num_q_heads=8,
               num_kv_heads=2)
    f8 = W.to_fp8(w, k_scale=0.25, v_scale=0.5)
    kc, vc = f8.k_cache.numpy().copy(), f8.v_cache.numpy().copy()
    oracle.reshape_and_cache_fp8(w.key, w.value, kc, vc, w.slot_mapping, "fp16", 0.25, 0.5)
    k16 = (torch.from_numpy(kc).view(torch.float8_e4m3fn).float() * 0.25).half()
    v16 = (torch.from_numpy(vc).view(torch.float8_e4m3fn).float() * 0.5).half()
    got = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, "fp16",
                        kv_dtype="e4m3", k_scale=0.25, v_scale=0.5)
    ref = oracle.decode(w.query, k16, v16, w.block_tables, w.context_lens, w.scale, "fp16")
    assert np.array_equal(got, ref)
    a = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, "fp16",
                      kv_dtype="e4m3", k_scale=2.0, v_scale=3.0)
    b = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale * 2.0, "fp16",
                      kv_dtype="e4m3", k_scale=1.0, v_scale=1.0)
    assert np.allclose(a, 3.0 * b, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------- chunked prefill

def _prefill_pool(pw):
    kc = pw.k_cache.clone().view(torch.int16).numpy().view(np.uint16)
    vc = pw.v_cache.clone().view(torch.int16).numpy().view(np.uint16)
    oracle.reshape_and_cache(pw.key, pw.value, kc, vc, pw.slot_mapping)
    return kc, vc


def pin_prefill_single_token_is_decode():
    """A chunk of one token is a decode step: bit-identical outputs."""
    pw = W.make_prefill("llama3_8b_gqa", 20, lens=[5, 17, 40, 333], head_dim=64,
                        num_q_heads=8, num_kv_heads=2, q_lens=[1, 1, 1, 1])
    kc, vc = _prefill_pool(pw)
    got = oracle.prefill(pw.query, pw.query_start, kc, vc, pw.block_tables, pw.context_lens,
                         pw.scale, pw.dtype)
    ref = oracle.decode(pw.query, kc, vc, pw.block_tables, pw.context_lens, pw.scale, pw.dtype)
    assert np.array_equal(got, ref)


def pin_prefill_rows_are_truncated_decodes():
    """Row t of a chunk attends to exactly the tokens up to its position."""
    pw = W.make_prefill("tiny_mha", 21, lens=[20, 37], chunk=9)
    kc, vc = _prefill_pool(pw)
    got = oracle.prefill(pw.query, pw.query_start, kc, vc, pw.block_tables, pw.context_lens,
                         pw.scale, pw.dtype)
    for i in range(pw.num_seqs):
        ql = int(pw.q_lens[i])
        for t in range(ql):
            row = int(pw.query_start[i]) + t
            pos = int(pw.context_lens[i]) - ql + t
            ref = oracle.decode(pw.query[row:row + 1], kc, vc, pw.block_tables[i:i + 1],
                                np.array([pos + 1], np.int32), pw.scale, pw.dtype)
            assert np.array_equal(got[row], ref[0])


def pin_prefill_vs_torch_causal_sdpa():
    """Whole-prompt prefill (chunk = context) against torch's fp64
    scaled_dot_product_attention with a causal mask on contiguous K/V."""
    F = torch.nn.functional
    pw = W.make_prefill("llama3_70b_cb", 22, lens=[50, 33], head_dim=64, num_q_heads=8,
                        num_kv_heads=2, chunk=10**6)
    kc, vc = _prefill_pool(pw)
    got = oracle.prefill(pw.query, pw.query_start, kc, vc, pw.block_tables, pw.context_lens,
                         pw.scale, pw.dtype)
    G = 4
    for i in range(pw.num_seqs):
        c = int(pw.context_lens[i])
        K = torch.from_numpy(np.stack([_contiguous_np(kc, pw.block_tables[i].numpy(), c, h, "fp16")
                                       for h in range(2)])).repeat_interleave(G, 0)
        V = torch.from_numpy(np.stack([_contiguous_np(vc, pw.block_tables[i].numpy(), c, h, "fp16")
                                       for h in range(2)])).repeat_interleave(G, 0)
        q0 = int(pw.query_start[i])
        Q = pw.query[q0:q0 + c].double().permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(Q[None], K[None], V[None], is_causal=True,
                                             scale=float(np.float32(pw.scale)))[0]
        assert np.allclose(got[q0:q0 + c], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def pin_prefill_chunks_compose():
    """Prefilling a prompt in two chunks gives, row for row, the outputs of
    prefilling it in one (bit-identical)."""
    full = W.make_prefill("tiny_mha", 23, lens=[45, 30, 60, 17], chunk=10**6)
    kc, vc = _prefill_pool(full)
    one = oracle.prefill(full.query, full.query_start, kc, vc, full.block_tables,
                         full.context_lens, full.scale, full.dtype)
    ctx = full.context_lens.numpy()
    cut = ctx // 2
    for part in range(2):
        lens = cut if part == 0 else ctx
        ql = cut if part == 0 else ctx - cut
        rows = np.concatenate([np.arange(int(full.query_start[i]) + (0 if part == 0 else cut[i]),
                                         int(full.query_start[i]) + (cut[i] if part == 0 else ctx[i]))
                               for i in range(full.num_seqs)])
        qs = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        two = oracle.prefill(full.query[torch.from_numpy(rows)], qs, kc, vc, full.block_tables,
                             lens.astype(np.int32), full.scale, full.dtype)
        assert np.array_equal(two, one[rows])


def _prefill_pool_fp8(pw):
    kh, vh = pw.k_cache.numpy().copy(), pw.v_cache.numpy().copy()
    oracle.reshape_and_cache_fp8(pw.key, pw.value, kh, vh, pw.slot_mapping, pw.dtype,
                                 pw.k_scale, pw.v_scale)
    return kh, vh


def pin_prefill_fp8_single_token_is_decode():
    """FP8 caches: a chunk of one token is an FP8 decode step (bit-identical)."""
    pw = W.to_fp8(W.make_prefill("llama3_8b_gqa", 24, lens=[5, 17, 40, 333], num_q_heads=8,
                                 num_kv_heads=2, q_lens=[1, 1, 1, 1], dtype="bf16"))
    kh, vh = _prefill_pool_fp8(pw)
    fp8 = dict(kv_dtype="e4m3", k_scale=pw.k_scale, v_scale=pw.v_scale)
    got = oracle.prefill(pw.query, pw.query_start, kh, vh, pw.block_tables, pw.context_lens,
                         pw.scale, pw.dtype, **fp8)
    ref = oracle.decode(pw.query, kh, vh, pw.block_tables, pw.context_lens, pw.scale, pw.dtype,
                        **fp8)
    assert np.array_equal(got, ref)


def pin_prefill_fp8_vs_torch_dequantised_sdpa():
    """FP8 caches: whole-prompt prefill against torch's fp64 causal SDPA over
    contiguous K/V whose codes are decoded by torch's own float8_e4m3fn type
    and multiplied by the scales (not the oracle's decoder)."""
    F = torch.nn.functional
    ks, vs = 0.037, 0.11
    pw = W.to_fp8(W.make_prefill("llama3_70b_cb", 25, lens=[50, 33], head_dim=64, num_q_heads=8,
                                 num_kv_heads=2, chunk=10**6), k_scale=ks, v_scale=vs)
    kh, vh = _prefill_pool_fp8(pw)
    got = oracle.prefill(pw.query, pw.query_start, kh, vh, pw.block_tables, pw.context_lens,
                         pw.scale, pw.dtype, kv_dtype="e4m3", k_scale=ks, v_scale=vs)
    G, bs = 4, pw.block_size
    for i in range(pw.num_seqs):
        c = int(pw.context_lens[i])
        bt = pw.block_tables[i].numpy()
        idx = [(int(bt[j // bs]), j % bs) for j in range(c)]

        def contiguous(cache, scale):
            codes = np.stack([np.stack([cache[b, h, o] for b, o in idx]) for h in range(2)])
            vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double() * scale
            return vals.repeat_interleave(G, 0)
        K, V = contiguous(kh, ks), contiguous(vh, vs)
        q0 = int(pw.query_start[i])
        Q = pw.query[q0:q0 + c].double().permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(Q[None], K[None], V[None], is_causal=True,
                                             scale=float(np.float32(pw.scale)))[0]
        assert np.allclose(got[q0:q0 + c], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def pin_random_shapes_vs_brute_force():
    """Seeded sweep of small random shapes (group 1-8, 1/2/4 KV heads, head_dim
    64/128, block size 16/32, fp16/bf16, contexts 0-300): the oracle's decode
    equals the textbook non-paged attention (numpy gather + softmax) to 1e-12,
    and its prefill of each sequence's last rows equals the decode of the
    sequence cut at each row's position (bit for bit)."""
    for i in range(16):
        rng = np.random.default_rng(5000 + i)
        G, hkv = int(rng.integers(1, 9)), int(rng.choice([1, 2, 4]))
        lens = [int(x) for x in rng.integers(0, 301, int(rng.integers(1, 5)))]
        kw = dict(lens=lens, num_q_heads=G * hkv, num_kv_heads=hkv,
                  head_dim=int(rng.choice([64, 128])), block_size=int(rng.choice([16, 32])),
                  dtype=str(rng.choice(["fp16", "bf16"])))
        w = W.make("llama3_8b_gqa", 200 + i, **kw)
        kc, vc = _after_scatter(w)
        got = oracle.decode(w.query, kc, vc, w.block_tables, w.context_lens, w.scale, w.dtype)
        assert np.allclose(got, _brute(w, kc, vc), rtol=1e-12, atol=1e-13), i
        pw = W.make_prefill("llama3_8b_gqa", 300 + i, chunk=int(rng.integers(1, 40)),
                            **dict(kw, lens=[max(1, x) for x in lens]))
        pkc, pvc = _prefill_pool(pw)
        rows = oracle.prefill(pw.query, pw.query_start, pkc, pvc, pw.block_tables,
                              pw.context_lens, pw.scale, pw.dtype)
        for s in range(pw.num_seqs):
            ql = int(pw.query_start[s + 1] - pw.query_start[s])
            for t in range(ql):
                row = int(pw.query_start[s]) + t
                pos = int(pw.context_lens[s]) - ql + t
                ref = oracle.decode(pw.query[row:row + 1], pkc, pvc, pw.block_tables[s:s + 1],
                                    np.array([pos + 1], np.int32), pw.scale, pw.dtype)
                assert np.array_equal(rows[row], ref[0]), (i, s, t)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


def test_generator_slots_are_distinct():
    """Every generated batch honours the scatter's contract (no two new tokens
    in one slot), and the check rejects a duplicate."""
    for name in W.NAMES:
        W.check_distinct_slots(W.make(name, 3).slot_mapping)
    W.check_distinct_slots(W.make_prefill("llama3_8b_gqa", 3, batch=4, chunk=100).slot_mapping)
    W.check_distinct_slots([5, -1, -1, 7])
    with pytest.raises(ValueError):
        W.check_distinct_slots([5, 9, 5])
