"""GPU parity: the CUDA library (through its C ABI) against the fp64 CPU oracle.

reshape_and_cache and all gathering must match bit-exactly; attention output
must satisfy |gpu - oracle| <= 2e-3 + 1e-2 |oracle| per element.  Small cases
compare every output; the full-size workloads compare every output where the
oracle finishes in seconds and a seeded sample of (sequence, head) rows
otherwise.  Layout changes (physical-block permutation, copy-on-write sharing)
must leave the GPU output bit-identical.
"""
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


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Run:
    """One workload on the GPU: pool after the scatter, decode output(s)."""

    def __init__(self, pa, w, partition_sizes=None):
        self.w = w
        dev = torch.device("cuda")
        self.kc, self.vc = w.k_cache.to(dev), w.v_cache.to(dev)
        pa.pa_reshape_and_cache(w.key.to(dev), w.value.to(dev), self.kc, self.vc,
                                w.slot_mapping.to(dev))
        self.q = w.query.to(dev)
        self.bt = w.block_tables.to(dev)
        self.cl = w.context_lens.to(dev)
        self.outs = {}
        for ps in (partition_sizes if partition_sizes is not None else [w.partition_size]):
            out = torch.empty_like(self.q)
            pa.pa_decode(out, self.q, self.kc, self.vc, self.bt, self.cl, w.scale,
                         max(w.max_context_len, 0), ps)
            self.outs[ps] = out
        torch.cuda.synchronize()
        self.err = pa.pa_device_errors()

    def host_pool(self):
        kh, vh = u16(self.w.k_cache).copy(), u16(self.w.v_cache).copy()
        oracle.reshape_and_cache(self.w.key, self.w.value, kh, vh, self.w.slot_mapping)
        return kh, vh


def assert_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} elements outside tolerance; "
                           f"max abs err {err.max():.3g}")


def check_decode(run, pairs=None):
    w = run.w
    kh, vh = run.host_pool()
    ref = oracle.decode(w.query, kh, vh, w.block_tables, w.context_lens, w.scale, w.dtype,
                        pairs=pairs)
    for ps, out in run.outs.items():
        got = out.float().cpu().double().numpy()
        if pairs is not None:
            pr = np.asarray(pairs).reshape(-1, 2)
            got = got[pr[:, 0], pr[:, 1]]
        assert_close(got, ref, f"{w.name} partition_size={ps}")


def sample_pairs(w, n_seqs, seed=0):
    """All heads of a seeded sample of sequences, always including the longest
    and the shortest."""
    rng = np.random.default_rng(seed)
    ctx = w.context_lens.numpy()
    seqs = set(rng.choice(w.num_seqs, size=min(n_seqs, w.num_seqs), replace=False).tolist())
    seqs |= {int(ctx.argmax()), int(ctx.argmin())}
    return [(i, h) for i in sorted(seqs) for h in range(w.num_q_heads)]


# ------------------------------------------------------------------ full sizes

FULL = [("tiny_mha", {}), ("llama3_8b_gqa", {}), ("shared_prefix_cow", {}),
        ("long_context", {}), ("llama3_70b_cb", {}), ("llama3_70b_cb", dict(dtype="bf16"))]


@pytest.mark.parametrize("name,kw", FULL, ids=[f"{n}-{k.get('dtype', 'default')}" for n, k in FULL])
def test_full_size_workload(pa, name, kw):
    w = W.make(name, 0, **kw)
    run = Run(pa, w)
    assert run.err == 0
    kh, vh = run.host_pool()
    # scatter: the whole pool, bit for bit (untouched and poisoned slots included)
    assert np.array_equal(u16(run.kc), kh) and np.array_equal(u16(run.vc), vh)
    if name in ("long_context", "llama3_70b_cb"):
        check_decode(run, sample_pairs(w, 2 if name == "long_context" else 24))
    else:
        check_decode(run)


# ---------------------------------------------------------- shapes and edges

SMALL = [
    ("tiny_mha", dict(lens=[0, 1, 2, 15])),
    ("tiny_mha", dict(lens=[16, 17, 31, 32], head_dim=128)),
    ("tiny_mha", dict(lens=[33, 47, 48, 49], dtype="bf16")),
    ("tiny_mha", dict(lens=[5, 64, 100, 200], num_q_heads=8, num_kv_heads=4)),     # G = 2
    ("llama3_8b_gqa", dict(lens=[1, 100, 513, 1000, 2049], head_dim=64)),            # G = 4
    ("llama3_8b_gqa", dict(lens=[700, 3], num_q_heads=24, num_kv_heads=8)),          # G = 3
    ("llama3_70b_cb", dict(lens=[1, 31, 32, 33, 64, 65, 1023], head_dim=64)),        # G = 8, bs 32
    ("llama3_70b_cb", dict(lens=[2, 300, 4000], dtype="bf16")),
    ("llama3_70b_cb", dict(lens=[7, 70], num_q_heads=40, num_kv_heads=8)),           # G = 5
    ("long_context", dict(lens=[20000, 1, 5000])),
    ("shared_prefix_cow", dict(groups=3, group_size=4, prefix_len=2040, max_len=100)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(SMALL)])
def test_small_cases_all_partition_sizes(pa, name, kw):
    w = W.make(name, 1, **kw)
    run = Run(pa, w, partition_sizes=[0, 16, 64, 128, 512, 1 << 20])
    assert run.err == 0
    kh, vh = run.host_pool()
    assert np.array_equal(u16(run.kc), kh) and np.array_equal(u16(run.vc), vh)
    check_decode(run)


def _random_decode(i):
    """Seeded random decode shape: batch 1-8, contexts 0-3000, group 1-8,
    1-8 KV heads, head_dim 64 or 128, block size 16 or 32, fp16 or bf16."""
    rng = np.random.default_rng(2000 + i)
    G = int(rng.integers(1, 9))
    hkv = int(rng.choice([1, 2, 4, 8]))
    lens = [int(x) for x in rng.integers(0, 3001, int(rng.integers(1, 9)))]
    return dict(lens=lens, num_q_heads=G * hkv, num_kv_heads=hkv,
                head_dim=int(rng.choice([64, 128])), block_size=int(rng.choice([16, 32])),
                dtype=str(rng.choice(["fp16", "bf16"])))


@pytest.mark.parametrize("i", range(30))
def test_decode_random_shapes(pa, i):
    w = W.make("llama3_8b_gqa", 90 + i, **_random_decode(i))
    ps = int(np.random.default_rng(3000 + i).choice([0, 16, 48, 160, 512]))
    run = Run(pa, w, partition_sizes=[ps])
    assert run.err == 0
    kh, vh = run.host_pool()
    assert np.array_equal(u16(run.kc), kh) and np.array_equal(u16(run.vc), vh)
    check_decode(run)


def test_empty_batch(pa):
    dev = torch.device("cuda")
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device=dev)
    q = torch.zeros(0, 2, 64, dtype=torch.float16, device=dev)
    out = torch.empty_like(q)
    pa.pa_decode(out, q, kc, kc.clone(), torch.zeros(0, 1, dtype=torch.int32, device=dev),
                 torch.zeros(0, dtype=torch.int32, device=dev), 0.125, 0, 0)
    pa.pa_reshape_and_cache(q.view(0, 2, 64), q.view(0, 2, 64), kc, kc.clone(),
                            torch.zeros(0, dtype=torch.int64, device=dev))
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0


def test_skipped_slots_and_strided_key(pa):
    """slot < 0 writes nothing; key/value may be row-strided views (e.g. of a
    fused QKV buffer)."""
    w = W.make("llama3_70b_cb", 2, lens=[10, 40, 90, 33])
    dev = torch.device("cuda")
    sm = w.slot_mapping.clone()
    sm[1] = -1
    fused = torch.randn(w.num_seqs, 3, w.num_kv_heads, w.head_dim,
                        generator=torch.Generator().manual_seed(3)).to(w.torch_dtype())
    key, value = fused[:, 1], fused[:, 2]
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    fd = fused.to(dev)
    pa.pa_reshape_and_cache(fd[:, 1], fd[:, 2], kc, vc, sm.to(dev))
    torch.cuda.synchronize()
    kh, vh = u16(w.k_cache).copy(), u16(w.v_cache).copy()
    oracle.reshape_and_cache(key.contiguous(), value.contiguous(), kh, vh, sm)
    assert np.array_equal(u16(kc), kh) and np.array_equal(u16(vc), vh)
    assert pa.pa_device_errors() == 0


# ------------------------------------------------------------------ invariants

def test_permutation_invariance_bitwise(pa):
    w = W.make("llama3_70b_cb", 4, batch=24, max_len=3000)
    a = Run(pa, w, partition_sizes=[0, 512])
    b = Run(pa, w.permuted(9), partition_sizes=[0, 512])
    for ps in (0, 512):
        assert torch.equal(a.outs[ps].view(torch.int16), b.outs[ps].view(torch.int16))


def test_copy_on_write_bitwise(pa):
    for P in (2048, 2040):
        w = W.make("shared_prefix_cow", 5, groups=2, group_size=4, prefix_len=P, max_len=300)
        a = Run(pa, w, partition_sizes=[0, 512])
        b = Run(pa, w.unshared(), partition_sizes=[0, 512])
        for ps in (0, 512):
            assert torch.equal(a.outs[ps].view(torch.int16), b.outs[ps].view(torch.int16))


def test_identity_v_probe(pa):
    """Equal keys, one-hot V per physical slot: out * ctx marks exactly the
    slots the block table reaches."""
    NB, bs, d = 4, 16, 64
    dev = torch.device("cuda")
    perm = np.random.default_rng(1).permutation(NB)
    kc = torch.ones(NB, 1, bs, d, dtype=torch.float16)
    vc = torch.zeros(NB, 1, bs, d, dtype=torch.float16)
    for b in range(NB):
        for r in range(bs):
            vc[b, 0, r, b * bs + r] = 1.0
    for ctx in (1, 15, 16, 17, 40, 64):
        bt = torch.from_numpy(perm[: (ctx + bs - 1) // bs].astype(np.int32))[None].to(dev)
        q = torch.full((1, 1, d), 0.25, dtype=torch.float16, device=dev)
        out = torch.empty_like(q)
        pa.pa_decode(out, q, kc.to(dev), vc.to(dev), bt,
                     torch.tensor([ctx], dtype=torch.int32, device=dev), 0.125, ctx, 0)
        got = out.float().cpu().numpy()[0, 0] * ctx
        expect = np.zeros(d)
        for j in range(ctx):
            expect[perm[j // bs] * bs + j % bs] = 1.0
        assert np.allclose(got, expect, atol=2e-3 * ctx), ctx


def test_reduce_alone_against_oracle_partials(pa):
    """pa_decode_reduce on partials the oracle computed (rounded to fp32, m
    converted to base 2) matches the oracle's log-sum-exp join."""
    w = W.make("llama3_8b_gqa", 6, lens=[1, 40, 600, 1500], head_dim=128)
    ps = 128
    kh = u16(w.k_cache).copy()
    vh = u16(w.v_cache).copy()
    oracle.reshape_and_cache(w.key, w.value, kh, vh, w.slot_mapping)
    ref, m, l, o = oracle.decode(w.query, kh, vh, w.block_tables, w.context_lens, w.scale,
                                 w.dtype, partition_size=ps, return_partials=True)
    B, Hq, d = w.num_seqs, w.num_q_heads, w.head_dim
    P = pa.pa_decode_num_partitions(w.max_context_len, ps)
    assert m.shape[1] == P
    size = pa.pa_decode_workspace_size(B, Hq, d, w.max_context_len, ps)
    ws = torch.zeros(size, dtype=torch.uint8)
    R = B * Hq
    ml = (R * P * 4 + 255) // 256 * 256
    c0 = pa.DECODE_COUNTER_BYTES          # m, l, o follow the join counters
    ws[c0:c0 + R * P * 4].view(torch.float32).copy_(
        torch.from_numpy((m * np.log2(np.e)).astype(np.float32).ravel()))
    ws[c0 + ml:c0 + ml + R * P * 4].view(torch.float32).copy_(
        torch.from_numpy(l.astype(np.float32).ravel()))
    ws[c0 + 2 * ml:c0 + 2 * ml + R * P * d * 4].view(torch.float32).copy_(
        torch.from_numpy(o.astype(np.float32).ravel()))
    out = torch.empty(B, Hq, d, dtype=torch.float16, device="cuda")
    pa.pa_decode_reduce(out, ws.cuda(), w.context_lens.cuda(), w.max_context_len, ps)
    got = out.float().cpu().double().numpy()
    assert_close(got, ref.reshape(B, Hq, d), "reduce")


def test_join_counters_return_to_zero_across_shapes(pa):
    """Split calls joined inside the decode kernel (at most 32 partitions) leave
    the workspace's counter words zero, so one zero-filled workspace serves
    successive calls of different shapes; every output matches the oracle."""
    cases = [(W.make("llama3_8b_gqa", 31, lens=[900, 1500, 300, 2000]), 512),
             (W.make("llama3_70b_cb", 32, lens=[1, 700, 64, 65, 2000, 33]), 64),
             (W.make("tiny_mha", 33, lens=[0, 17, 200, 99]), 16),
             (W.make("llama3_8b_gqa", 34, lens=[4000, 10, 512, 513], dtype="bf16"), 128)]
    need = max(pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.head_dim,
                                           w.max_context_len, ps) for w, ps in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for w, ps in cases:
            P = pa.pa_decode_num_partitions(w.max_context_len, ps)
            assert 1 < P <= 32
            run = Run(pa, w, partition_sizes=[])
            out = torch.empty_like(run.q)
            pa.pa_decode(out, run.q, run.kc, run.vc, run.bt, run.cl, w.scale, w.max_context_len,
                         ps, workspace=ws)
            torch.cuda.synchronize()
            assert pa.pa_device_errors() == 0
            assert int(ws[:pa.DECODE_COUNTER_BYTES].count_nonzero()) == 0
            run.outs = {ps: out}
            check_decode(run)


def test_join_counter_not_zero_is_flagged(pa):
    """A workspace whose counter words were not cleared is reported as
    PA_DEVERR_WORKSPACE, without a fault; a sequence short enough for one
    partition is still exact (it never uses a counter); once the counters are
    cleared, the same call matches the oracle."""
    w = W.make("llama3_8b_gqa", 35, lens=[900, 1500, 300])
    ps = 512
    run = Run(pa, w, partition_sizes=[])
    size = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.head_dim,
                                       w.max_context_len, ps)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    ws[:4 * w.num_seqs * w.num_kv_heads].view(torch.int32).fill_(5)
    out = torch.zeros_like(run.q)
    pa.pa_decode(out, run.q, run.kc, run.vc, run.bt, run.cl, w.scale, w.max_context_len, ps,
                 workspace=ws)
    torch.cuda.synchronize()
    assert pa.pa_device_errors() & pa.DEVERR_WORKSPACE
    kh, vh = run.host_pool()
    ref = oracle.decode(w.query, kh, vh, w.block_tables, w.context_lens, w.scale, w.dtype)
    assert_close(out[2:].float().cpu().double().numpy(), ref[2:], "one-partition sequence")
    ws.zero_()
    pa.pa_decode(out, run.q, run.kc, run.vc, run.bt, run.cl, w.scale, w.max_context_len, ps,
                 workspace=ws)
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
    assert_close(out.float().cpu().double().numpy(), ref, "after clearing the counters")


# ------------------------------------------------------------ device errors

def test_bad_block_entry_is_flagged_not_read(pa):
    w = W.make("llama3_70b_cb", 7, lens=[100, 200, 64])
    run_ok = Run(pa, w, partition_sizes=[0, 64])
    assert run_ok.err == 0
    bad = w.clone()
    bad.block_tables[1, 2] = w.num_blocks + 5      # outside the pool
    bad.block_tables[2, 0] = -3
    run = Run(pa, bad, partition_sizes=[0, 64])
    assert run.err & pa.DEVERR_BAD_BLOCK
    for ps, out in run.outs.items():
        assert torch.isfinite(out.float()).all()
        # the untouched sequence is bit-identical to the good run's
        assert torch.equal(out[0].view(torch.int16), run_ok.outs[ps][0].view(torch.int16))


def test_bad_slot_and_length_flags(pa):
    w = W.make("tiny_mha", 8)
    dev = torch.device("cuda")
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    sm = w.slot_mapping.clone()
    sm[0] = w.num_blocks * w.block_size     # one past the pool
    pa.pa_reshape_and_cache(w.key.to(dev), w.value.to(dev), kc, vc, sm.to(dev))
    assert pa.pa_device_errors() == pa.DEVERR_BAD_SLOT
    q = w.query.to(dev)
    out = torch.empty_like(q)
    cl = w.context_lens.clone()
    cl[1] = w.max_blocks_per_seq * w.block_size + 1   # longer than the table
    pa.pa_decode(out, q, kc, vc, w.block_tables.to(dev), cl.to(dev), w.scale, int(cl.max()), 0)
    assert pa.pa_device_errors() & pa.DEVERR_BAD_LEN
    assert torch.all(out[1] == 0)
    assert pa.pa_device_errors() == 0   # the word was cleared


def test_bounded_wait_gives_up_and_context_survives(pa):
    """The wait limit every staged-data wait uses: a CTA waiting on a barrier
    nothing completes gives up after about a second and reports
    PA_DEVERR_TIMEOUT, without a fault; the context then still runs a decode
    that matches the oracle."""
    import time
    assert pa.pa_device_errors() == 0
    t0 = time.perf_counter()
    pa.pa_selftest_bounded_wait()
    flags = pa.pa_device_errors()          # waits for the stream
    dt = time.perf_counter() - t0
    assert flags & pa.DEVERR_TIMEOUT
    assert 0.5 < dt < 30, dt
    run = Run(pa, W.make("tiny_mha", 7))
    assert run.err == 0
    check_decode(run)


def test_binding_rejects_bad_tensors_before_launch(pa):
    """The Python binding refuses strided views, wrong dtypes and wrong shapes
    with ValueError before anything is launched."""
    w = W.make("tiny_mha", 8)
    dev = torch.device("cuda")
    q, kc, vc = w.query.to(dev), w.k_cache.to(dev), w.v_cache.to(dev)
    bt, cl = w.block_tables.to(dev), w.context_lens.to(dev)
    out = torch.empty_like(q)
    bad = [
        dict(query=q.transpose(0, 1).contiguous().transpose(0, 1)),   # strided view
        dict(block_tables=bt.to(torch.int64)),                        # wrong dtype
        dict(out=torch.empty(q.shape[0], q.shape[1] + 1, q.shape[2], dtype=q.dtype, device=dev)),
        dict(query=w.query),                                          # host tensor
    ]
    for kw in bad:
        args = dict(out=out, query=q, k_cache=kc, v_cache=vc, block_tables=bt, context_lens=cl)
        args.update(kw)
        with pytest.raises(ValueError):
            pa.pa_decode(args["out"], args["query"], args["k_cache"], args["v_cache"],
                         args["block_tables"], args["context_lens"], w.scale, w.max_context_len, 0)
    torch.cuda.synchronize()
    assert pa.pa_device_errors() == 0
