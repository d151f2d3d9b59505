"""GPU parity of pa_decode_shared_prefix (through the C ABI) against the fp64
CPU oracle.

The oracle knows nothing of prefix groups: it attends every sequence over its
own tokens through its own block table, exactly as for pa_decode.  The shared
pass must therefore reproduce per-sequence attention while reading each group's
shared prefix once.  Cases span several partitions, group chunks (groups with
more than one CTA's 128 query rows), members shorter than the shared prefix,
partitions joined inside the decode kernel and by the reduce kernel, and the
device-side checks of the group description.
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


def assert_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} elements outside tolerance; "
                           f"max abs err {err.max():.3g}")


class SharedRun:
    """Scatter the new tokens, then decode the batch both ways."""

    def __init__(self, pa, w, ps, context_lens=None, group_start=None, prefix_lens=None,
                 max_group_size=None, block_tables=None, plain=True):
        dev = torch.device("cuda")
        self.w = w
        self.fp8 = w.kv_dtype == "e4m3"
        self.cl_host = w.context_lens if context_lens is None else context_lens
        self.bt_host = w.block_tables if block_tables is None else block_tables
        self.kc, self.vc = w.k_cache.to(dev), w.v_cache.to(dev)
        if self.fp8:
            pa.pa_reshape_and_cache_fp8(w.key.to(dev), w.value.to(dev), self.kc, self.vc,
                                        w.slot_mapping.to(dev), w.k_scale, w.v_scale)
        else:
            pa.pa_reshape_and_cache(w.key.to(dev), w.value.to(dev), self.kc, self.vc,
                                    w.slot_mapping.to(dev))
        q, bt, cl = w.query.to(dev), self.bt_host.to(dev), self.cl_host.to(dev)
        gs = (w.group_start if group_start is None else group_start).to(dev)
        pl = (w.prefix_lens if prefix_lens is None else prefix_lens).to(dev)
        mgs = w.max_group_size if max_group_size is None else max_group_size
        self.maxctx = max(int(self.cl_host.max().item()), 1)
        ws = pa.new_decode_workspace(w.num_seqs, w.num_q_heads, w.head_dim, self.maxctx, ps)
        def shared(out):
            if self.fp8:
                pa.pa_decode_shared_prefix_fp8(out, q, self.kc, self.vc, bt, cl, gs, pl, mgs,
                                               w.scale, w.k_scale, w.v_scale, self.maxctx, ps,
                                               workspace=ws)
            else:
                pa.pa_decode_shared_prefix(out, q, self.kc, self.vc, bt, cl, gs, pl, mgs,
                                           w.scale, self.maxctx, ps, workspace=ws)
        self.out = torch.empty_like(q)
        shared(self.out)
        # a second call on the same workspace (its join counters left at zero)
        self.out2 = torch.empty_like(q)
        shared(self.out2)
        self.plain = None
        if plain:
            self.plain = torch.empty_like(q)
            if self.fp8:
                pa.pa_decode_fp8(self.plain, q, self.kc, self.vc, bt, cl, w.scale, w.k_scale,
                                 w.v_scale, self.maxctx, ps)
            else:
                pa.pa_decode(self.plain, q, self.kc, self.vc, bt, cl, w.scale, self.maxctx, ps)
        torch.cuda.synchronize()
        self.err = pa.pa_device_errors()

    def oracle_out(self, pairs=None):
        w = self.w
        if self.fp8:
            kh, vh = w.k_cache.numpy().copy(), w.v_cache.numpy().copy()
            oracle.reshape_and_cache_fp8(w.key, w.value, kh, vh, w.slot_mapping, w.dtype,
                                         w.k_scale, w.v_scale)
            return oracle.decode(w.query, kh, vh, self.bt_host, self.cl_host, w.scale, w.dtype,
                                 pairs=pairs, kv_dtype="e4m3", k_scale=w.k_scale,
                                 v_scale=w.v_scale)
        kh, vh = u16(w.k_cache).copy(), u16(w.v_cache).copy()
        oracle.reshape_and_cache(w.key, w.value, kh, vh, w.slot_mapping)
        return oracle.decode(w.query, kh, vh, self.bt_host, self.cl_host, w.scale, w.dtype,
                             pairs=pairs)

    def check(self, what, pairs=None):
        ref = self.oracle_out(pairs)
        for name, out in (("shared", self.out), ("shared, second call", self.out2),
                          ("plain", self.plain)):
            if out is None:
                continue
            got = out.float().cpu().double().numpy()
            if pairs is not None:
                pr = np.asarray(pairs).reshape(-1, 2)
                got = got[pr[:, 0], pr[:, 1]]
            assert_close(got, ref, f"{what} ({name})")
        assert torch.equal(self.out, self.out2), f"{what}: two calls differ"


# (groups, group size, prefix tokens, suffix max, partition size, q heads, kv heads, d, bs, dtype)
CASES = [
    (3, 2, 256, 40, 64, 32, 8, 128, 16, "fp16"),     # G 4, 4 shared partitions
    (2, 5, 300, 64, 64, 32, 8, 128, 16, "bf16"),     # prefix not a multiple of the partition
    (1, 37, 128, 30, 32, 32, 8, 128, 16, "fp16"),    # 37 members at G 4: two CTA chunks (32 + 5)
    (2, 18, 192, 50, 64, 64, 8, 128, 32, "fp16"),    # G 8, bs 32: 16 members per chunk, two chunks
    (3, 4, 160, 20, 32, 8, 8, 64, 16, "bf16"),       # MHA (G 1), head_dim 64
    (2, 11, 96, 33, 32, 12, 4, 64, 32, "fp16"),      # G 3: columns cut across members
    (4, 3, 40, 16, 16, 32, 8, 128, 16, "fp16"),      # partial prefix block (copied, not shared)
    (2, 3, 64, 8, 64, 32, 8, 128, 16, "bf16"),       # prefix = one partition
    (5, 1, 128, 40, 32, 32, 8, 128, 16, "fp16"),     # groups of one
    (2, 27, 144, 30, 48, 40, 8, 128, 16, "bf16"),    # G 5 (125 of 128 rows, 25 + 2 members); 48-token partitions
    (3, 5, 112, 24, 16, 56, 8, 64, 32, "fp16"),      # G 7 (35 of 128 rows), 16-token partitions
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_shared_prefix_matches_oracle(pa, case):
    ng, gs, P, smax, ps, hq, hkv, d, bs, dt = case
    w = W.make("shared_prefix_cow", seed=11 + ng * gs, groups=ng, group_size=gs, prefix_len=P,
               max_len=smax, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
               dtype=dt, partition_size=ps)
    r = SharedRun(pa, w, ps)
    assert r.err == 0
    r.check(f"groups {ng}x{gs} prefix {P} ps {ps} G {hq // hkv} d {d} bs {bs} {dt}")


FP8_CASES = [
    (3, 2, 256, 40, 64, 32, 8, 128, 16, "fp16"),     # G 4
    (2, 5, 300, 64, 64, 32, 8, 128, 16, "bf16"),     # two own partitions: the counter join
    (2, 18, 192, 50, 64, 64, 8, 128, 32, "fp16"),    # G 8, bs 32, two chunks
    (3, 4, 160, 20, 32, 8, 8, 64, 16, "bf16"),       # MHA, head_dim 64
    (2, 27, 144, 30, 48, 40, 8, 128, 16, "bf16"),    # G 5, 48-token partitions
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[f"fp8-case{i}" for i in range(len(FP8_CASES))])
def test_shared_prefix_fp8_matches_oracle(pa, case):
    """FP8 caches: the shared pass widens the prefix codes in shared memory;
    every output against the oracle reading the same codes, and against
    pa_decode_fp8."""
    ng, gs, P, smax, ps, hq, hkv, d, bs, dt = case
    w = W.to_fp8(W.make("shared_prefix_cow", seed=51 + ng * gs, groups=ng, group_size=gs,
                        prefix_len=P, max_len=smax, num_q_heads=hq, num_kv_heads=hkv,
                        head_dim=d, block_size=bs, dtype=dt, partition_size=ps))
    r = SharedRun(pa, w, ps)
    assert r.err == 0
    r.check(f"FP8 groups {ng}x{gs} prefix {P} ps {ps} G {hq // hkv} d {d} bs {bs} {dt}")


def test_full_size_shared_prefix_batch_fp8(pa):
    """The copy-on-write batch at full size over FP8 caches, bf16 queries: a
    sample of sequences against the oracle, every output against
    pa_decode_fp8."""
    w = W.to_fp8(W.make("shared_prefix_cow", dtype="bf16"))
    r = SharedRun(pa, w, w.partition_size)
    assert r.err == 0
    seqs = [0, 9, 64, 127]
    r.check("full-size FP8 shared-prefix batch",
            pairs=[(i, h) for i in seqs for h in range(w.num_q_heads)])
    diff = (r.out.float() - r.plain.float()).abs()
    assert (diff <= ATOL + RTOL * r.plain.float().abs()).all()


def test_members_shorter_than_the_prefix(pa):
    """Members whose context ends inside the shared prefix (at, before and
    after partition boundaries) take fewer partitions from the shared pass."""
    w = W.make("shared_prefix_cow", seed=5, groups=2, group_size=6, prefix_len=256, max_len=40,
               partition_size=64)
    cl = w.context_lens.clone()
    cl[0:6] = torch.tensor([1, 63, 64, 65, 200, 255], dtype=torch.int32)
    cl[8] = 128
    r = SharedRun(pa, w, 64, context_lens=cl)
    assert r.err == 0
    r.check("members shorter than the prefix")


def test_many_partitions_join_in_the_reduce_kernel(pa):
    """More than 32 partitions: the decode runs warp partitions and the
    separate log-sum-exp reduce joins the shared pass's partials too."""
    w = W.make("shared_prefix_cow", seed=6, groups=2, group_size=3, prefix_len=1536, max_len=200,
               partition_size=32)
    r = SharedRun(pa, w, 32)
    assert pa.pa_decode_num_partitions(r.maxctx, 32) > 32
    assert r.err == 0
    r.check("reduce-kernel join")


def test_loose_group_size_bound(pa):
    """max_group_size above every group's size: the extra chunks find no
    members and leave."""
    w = W.make("shared_prefix_cow", seed=13, groups=4, group_size=5, prefix_len=128, max_len=40,
               num_q_heads=64, num_kv_heads=8, partition_size=32)
    r = SharedRun(pa, w, 32, max_group_size=w.num_seqs)   # 16 members per CTA: a second chunk
    assert r.err == 0
    r.check("loose group-size bound")


def test_zero_prefix_is_plain_decode(pa):
    w = W.make("shared_prefix_cow", seed=7, groups=3, group_size=2, prefix_len=128, max_len=64,
               partition_size=32)
    pl = torch.zeros_like(w.prefix_lens)
    r = SharedRun(pa, w, 32, prefix_lens=pl)
    assert r.err == 0
    r.check("no shared prefix")


def test_one_partition_is_plain_decode(pa):
    """max_context_len <= partition_size: nothing to share, the call is pa_decode."""
    w = W.make("shared_prefix_cow", seed=8, groups=2, group_size=4, prefix_len=128, max_len=32,
               partition_size=512)
    r = SharedRun(pa, w, 512)
    assert r.err == 0
    r.check("one partition")
    assert torch.equal(r.out, r.plain)


@pytest.mark.parametrize("heads", [(32, 8), (64, 8)], ids=["G4", "G8"])
def test_full_size_shared_prefix_batch(pa, heads):
    """The copy-on-write batch at full size (16 groups x 8 sequences, 2048-token
    prefix, the batch's 1024-token partitions), with its own head shape and the
    70B one: every sequence of a sample against the oracle, and every output
    against pa_decode."""
    w = W.make("shared_prefix_cow", num_q_heads=heads[0], num_kv_heads=heads[1])
    r = SharedRun(pa, w, w.partition_size)
    assert r.err == 0
    rng = np.random.default_rng(0)
    seqs = sorted(set(rng.choice(w.num_seqs, size=12, replace=False).tolist()) | {0, 127})
    pairs = [(i, h) for i in seqs for h in range(w.num_q_heads)]
    r.check("full-size shared-prefix batch", pairs=pairs)
    diff = (r.out.float() - r.plain.float()).abs()
    assert (diff <= ATOL + RTOL * r.plain.float().abs()).all()


# ------------------------------------------------------------ device checks

def _free_block(w):
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    return next(b for b in range(w.num_blocks) if b not in used)


def test_table_mismatch_is_flagged(pa):
    """A member whose table names a copy of a shared block (same data, other
    block id) breaks the group's contract: PA_DEVERR_PREFIX."""
    w = W.make("shared_prefix_cow", seed=9, groups=2, group_size=4, prefix_len=128, max_len=32,
               partition_size=32)
    src = int(w.block_tables[5, 3])
    dst = _free_block(w)
    w.k_cache[dst] = w.k_cache[src]
    w.v_cache[dst] = w.v_cache[src]
    bt = w.block_tables.clone()
    bt[5, 3] = dst
    r = SharedRun(pa, w, 32, block_tables=bt, plain=False)
    assert r.err & pa.DEVERR_PREFIX
    # the copy holds the same data, so every output still matches
    r.check("table mismatch (same data)")


def test_prefix_length_mismatch_is_flagged(pa):
    w = W.make("shared_prefix_cow", seed=10, groups=2, group_size=3, prefix_len=128, max_len=32,
               partition_size=32)
    pl = w.prefix_lens.clone()
    pl[4] = 64
    r = SharedRun(pa, w, 32, prefix_lens=pl, plain=False)
    assert r.err & pa.DEVERR_PREFIX


@pytest.mark.parametrize("bad", ["short", "unordered", "too_big"])
def test_bad_groups_are_flagged(pa, bad):
    w = W.make("shared_prefix_cow", seed=12, groups=3, group_size=3, prefix_len=96, max_len=32,
               partition_size=32)
    gs = w.group_start.clone()
    mgs = w.max_group_size
    if bad == "short":
        gs[-1] = w.num_seqs - 1      # the last sequence is in no group
    elif bad == "unordered":
        gs[1], gs[2] = gs[2].item(), gs[1].item()
    else:
        mgs = 2                      # groups of 3 with a bound of 2
    r = SharedRun(pa, w, 32, group_start=gs, max_group_size=mgs, plain=False)
    assert r.err & pa.DEVERR_PREFIX
