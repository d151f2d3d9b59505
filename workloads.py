"""Seeded synthetic inputs for PagedAttention decode.

This module builds the inputs that both the CUDA library and the CPU oracle
consume, and nothing else: it holds none of the attention arithmetic.  It
plays the part a block manager plays in a serving engine ("Serving engines",
How vLLM works): physical blocks of one shared pool are handed out from a
seeded, shuffled free list, each sequence gets a block table (logical block ->
physical block, unused entries -1), and the newest token of each sequence gets
a slot (physical block * block_size + offset) in its last block.

Values: query, the new token's key/value and every owned cache slot are N(0,1)
in the workload's dtype.  Every slot no sequence owns (free blocks, the unused
tail of each last block) and the slot the new token is about to be written to
hold a poison value (NaN by default), so that any read outside a sequence's
tokens shows up in the output.

Workloads (sizes as the decode batches they stand in for):

  tiny_mha           4 seqs, 4 q = 4 kv heads, d 64,  bs 16, ctx U[1,200], 64-block pool
  llama3_8b_gqa      64 seqs, 32 q / 8 kv heads, d 128, bs 16, ctx U[512,4096], pool +10%,
                     1024-token partitions
  shared_prefix_cow  16 groups x 8 seqs sharing a 2048-token prefix, suffix U[1,512],
                     1024-token partitions
  long_context       8 seqs, 32/8 heads, d 128, bs 16, ctx {32768 x6, 65536, 131072}, bf16
  llama3_70b_cb      256 seqs, 64/8 heads, d 128, bs 32, ctx lognormal(ln 1024, 1.0)
                     clipped to [1,16384], pool +20%, fp16 or bf16, 2048-token partitions
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}
POISON_BITS = {"fp16": 0x7E00, "bf16": 0x7FC0}  # quiet NaN in each format


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                      # "fp16" | "bf16"
    num_seqs: int                   # B
    num_q_heads: int                # Hq
    num_kv_heads: int               # Hkv
    head_dim: int                   # d
    block_size: int                 # bs
    num_blocks: int                 # NB
    scale: float                    # fp32 value of 1/sqrt(d)
    partition_size: int             # split-context partition the workload is run with (0 = none)
    context_lens: torch.Tensor      # int32 [B]
    block_tables: torch.Tensor      # int32 [B, MB], -1 = unused
    slot_mapping: torch.Tensor      # int64 [B], slot of token ctx-1 (-1 if ctx == 0)
    query: torch.Tensor             # [B, Hq, d]
    key: torch.Tensor               # [B, Hkv, d]  new token's key
    value: torch.Tensor             # [B, Hkv, d]  new token's value
    k_cache: torch.Tensor           # [NB, Hkv, bs, d] before the new token is written
    v_cache: torch.Tensor           # [NB, Hkv, bs, d]
    seed: int = 0
    kv_dtype: str = ""              # "" = same as dtype; "e4m3": uint8 FP8 caches
    k_scale: float = 1.0            # FP8 caches: code e stands for k_scale * e
    v_scale: float = 1.0
    # prefix sharing (copy-on-write batches): groups are runs of consecutive
    # sequences, group g = sequences group_start[g] .. group_start[g+1]-1;
    # prefix_lens[i] = leading tokens of sequence i held in blocks shared with
    # its whole group (None: no sharing described)
    group_start: Optional[torch.Tensor] = None   # int32 [num_groups + 1]
    prefix_lens: Optional[torch.Tensor] = None   # int32 [B]

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.num_seqs else 0

    @property
    def elem_bytes(self) -> int:
        """Bytes per cached K/V element."""
        return 1 if self.kv_dtype == "e4m3" else 2

    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def blocks_used(self) -> np.ndarray:
        ctx = self.context_lens.numpy().astype(np.int64)
        return (ctx + self.block_size - 1) // self.block_size

    def internal_fragmentation(self) -> float:
        """Share of the allocated token slots that hold no token (waste)."""
        alloc = int((self.blocks_used() * self.block_size).sum())
        return 0.0 if alloc == 0 else 1.0 - float(self.context_lens.sum().item()) / alloc

    def clone(self) -> "Workload":
        return dataclasses.replace(
            self, **{f.name: getattr(self, f.name).clone()
                     for f in dataclasses.fields(self)
                     if isinstance(getattr(self, f.name), torch.Tensor)})

    def permuted(self, seed: int) -> "Workload":
        """Same logical content with every physical block id relabelled by a
        seeded random permutation of the pool."""
        rng = np.random.default_rng(seed)
        perm = torch.from_numpy(rng.permutation(self.num_blocks).astype(np.int64))
        w = self.clone()
        kc = torch.empty_like(self.k_cache)
        vc = torch.empty_like(self.v_cache)
        kc[perm] = self.k_cache
        vc[perm] = self.v_cache
        w.k_cache, w.v_cache = kc, vc
        bt = self.block_tables.to(torch.int64)
        w.block_tables = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).to(torch.int32)
        sm = self.slot_mapping
        blk = torch.div(sm.clamp(min=0), self.block_size, rounding_mode="floor")
        w.slot_mapping = torch.where(sm >= 0, perm[blk] * self.block_size + sm.clamp(min=0) % self.block_size, sm)
        return w

    def unshared(self) -> "Workload":
        """Same logical content with every physical block that more than one
        sequence references copied into a private block per extra sequence."""
        bt = self.block_tables.numpy().copy()
        owners = {}
        for i in range(self.num_seqs):
            for lb in range(bt.shape[1]):
                p = int(bt[i, lb])
                if p >= 0:
                    owners.setdefault(p, []).append((i, lb))
        extra = sum(len(v) - 1 for v in owners.values())
        nb = self.num_blocks + extra
        shape = (nb,) + tuple(self.k_cache.shape[1:])
        kc = torch.empty(shape, dtype=self.k_cache.dtype)
        vc = torch.empty(shape, dtype=self.v_cache.dtype)
        kc[: self.num_blocks] = self.k_cache
        vc[: self.num_blocks] = self.v_cache
        nxt = self.num_blocks
        for p, refs in owners.items():
            for (i, lb) in refs[1:]:
                kc[nxt] = self.k_cache[p]
                vc[nxt] = self.v_cache[p]
                bt[i, lb] = nxt
                nxt += 1
        w = self.clone()
        w.k_cache, w.v_cache, w.num_blocks = kc, vc, nb
        w.block_tables = torch.from_numpy(bt)
        w.group_start = w.prefix_lens = None  # nothing is shared any more
        # the new token's slot is always in a private block, so slots stay valid
        return w

    @property
    def max_group_size(self) -> int:
        if self.group_start is None:
            return 1
        return int((self.group_start[1:] - self.group_start[:-1]).max().item())


def _poison(t: torch.Tensor, dtype: str) -> None:
    t.view(torch.int16).fill_(POISON_BITS[dtype])  # both patterns fit a positive int16


def _randn(shape, gen: torch.Generator, dtype: str) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(DTYPES[dtype])


def _build(name, seed, dtype, B, Hq, Hkv, d, bs, ctx: np.ndarray, pool_slack: float,
           partition_size: int, rng: np.random.Generator, gen: torch.Generator,
           min_blocks: int = 0, prefix_groups: Optional[List[List[int]]] = None,
           prefix_len: int = 0, poison: str = "nan", table_len: int = 0) -> Workload:
    ctx = np.asarray(ctx, dtype=np.int64)
    nblk = (ctx + bs - 1) // bs
    shared_full = prefix_len // bs if prefix_groups else 0
    # blocks the pool must hold: shared prefix blocks once per group, the rest per sequence
    need = int(nblk.sum())
    if prefix_groups:
        need -= sum((len(g) - 1) * shared_full for g in prefix_groups)
    NB = max(int(math.ceil(pool_slack * need)), need, min_blocks)
    # block-table width: the workload's longest possible sequence, in blocks
    MB = max(1, int(nblk.max()) if len(nblk) else 1, (table_len + bs - 1) // bs)
    free_list = list(rng.permutation(NB))
    bt = np.full((B, MB), -1, dtype=np.int32)
    group_of = {}
    if prefix_groups:
        for gi, g in enumerate(prefix_groups):
            shared = [free_list.pop() for _ in range(shared_full)]
            for i in g:
                group_of[i] = gi
                bt[i, :shared_full] = shared
    for i in range(B):
        start = shared_full if i in group_of else 0
        for lb in range(start, int(nblk[i])):
            bt[i, lb] = free_list.pop()

    k_cache = _randn((NB, Hkv, bs, d), gen, dtype)
    v_cache = _randn((NB, Hkv, bs, d), gen, dtype)
    # copy-on-write: a partial last prefix block is copied into each sequence's
    # own block, so its prefix rows equal those of the group's first sequence
    if prefix_groups and prefix_len % bs:
        rows = prefix_len % bs
        for g in prefix_groups:
            src = int(bt[g[0], shared_full])
            for i in g[1:]:
                dst = int(bt[i, shared_full])
                k_cache[dst, :, :rows] = k_cache[src, :, :rows]
                v_cache[dst, :, :rows] = v_cache[src, :, :rows]
    owned = np.zeros(NB, dtype=bool)
    owned[bt[bt >= 0]] = True
    free_idx = torch.from_numpy(np.nonzero(~owned)[0])
    if len(free_idx):
        for cache in (k_cache, v_cache):
            tmp = cache[free_idx]
            _poison(tmp, dtype)
            cache[free_idx] = tmp
    # tail slots of each last block, and the slot the new token goes to
    slots = np.full(B, -1, dtype=np.int64)
    for i in range(B):
        c = int(ctx[i])
        if c == 0:
            continue
        last = int(bt[i, (c - 1) // bs])
        first_bad = (c - 1) % bs  # the new token's row and every row after it
        for cache in (k_cache, v_cache):
            _poison(cache[last, :, first_bad:], dtype)
        slots[i] = last * bs + (c - 1) % bs
    if poison != "nan":
        raise ValueError("only NaN poison is supported")

    query = _randn((B, Hq, d), gen, dtype)
    key = _randn((B, Hkv, d), gen, dtype)
    value = _randn((B, Hkv, d), gen, dtype)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    check_distinct_slots(slots)
    group_start = prefix_lens = None
    if prefix_groups:
        # every sequence in one run of consecutive sequences (a sequence in no
        # listed group is a group of its own, sharing nothing)
        starts, pl = [0], np.zeros(B, dtype=np.int32)
        for i in range(1, B + 1):
            if i == B or group_of.get(i, -1 - i) != group_of.get(i - 1, -2 - i):
                starts.append(i)
        for g in prefix_groups:
            if sorted(g) != list(range(min(g), max(g) + 1)):
                raise ValueError("prefix groups must be runs of consecutive sequences")
            pl[g] = shared_full * bs
        group_start = torch.tensor(starts, dtype=torch.int32)
        prefix_lens = torch.from_numpy(pl)
    return Workload(name=name, dtype=dtype, num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv,
                    head_dim=d, block_size=bs, num_blocks=NB, scale=scale,
                    partition_size=partition_size,
                    context_lens=torch.from_numpy(ctx.astype(np.int32)),
                    block_tables=torch.from_numpy(bt), slot_mapping=torch.from_numpy(slots),
                    query=query, key=key, value=value, k_cache=k_cache, v_cache=v_cache,
                    seed=seed, group_start=group_start, prefix_lens=prefix_lens)


def check_distinct_slots(slots) -> None:
    """The scatter's contract: no two new tokens of one call share a slot
    (slot < 0 = no token).  Raises ValueError on a duplicate."""
    s = np.asarray(slots, dtype=np.int64)
    s = s[s >= 0]
    if np.unique(s).size != s.size:
        raise ValueError("duplicate slot in slot_mapping")


NAMES = ("tiny_mha", "llama3_8b_gqa", "shared_prefix_cow", "long_context", "llama3_70b_cb")

FP8_POISON = 0x7F  # an E4M3 NaN code
FP8_SCALE = float(np.float32(4.0 / 448.0))  # N(0,1) values up to 4 sigma fit the E4M3 range


def to_fp8(w: Workload, k_scale: float = FP8_SCALE, v_scale: float = FP8_SCALE) -> Workload:
    """The same workload with FP8 E4M3 caches: every owned slot holds the
    nearest code (torch's float8_e4m3fn cast, after clamping to +-448) of its
    N(0,1) value divided by the scale; unowned slots hold the NaN code.  The
    query and the new token's K/V stay 16-bit (the scatter quantises them)."""
    out = w.clone()

    def quant(c, s):
        x = (c.float() / s).clamp(-448.0, 448.0)
        q = x.to(torch.float8_e4m3fn).view(torch.uint8)
        q[torch.isnan(c)] = FP8_POISON
        return q
    out.k_cache = quant(w.k_cache, k_scale)
    out.v_cache = quant(w.v_cache, v_scale)
    out.kv_dtype, out.k_scale, out.v_scale = "e4m3", float(k_scale), float(v_scale)
    return out


def make(name: str, seed: int = 0, *, dtype: Optional[str] = None, batch: Optional[int] = None,
         lens: Optional[Sequence[int]] = None, num_q_heads: Optional[int] = None,
         num_kv_heads: Optional[int] = None, head_dim: Optional[int] = None,
         block_size: Optional[int] = None, partition_size: Optional[int] = None,
         prefix_len: Optional[int] = None, groups: Optional[int] = None,
         group_size: Optional[int] = None, max_len: Optional[int] = None) -> Workload:
    """Build one of the named workloads.  Keyword overrides shrink or reshape a
    workload for tests (``batch``, ``lens``, heads, ``head_dim``, ...)."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    if name == "tiny_mha":
        B = batch or 4
        ctx = np.asarray(lens) if lens is not None else rng.integers(1, (max_len or 200) + 1, size=B)
        B = len(ctx)
        bs = block_size or 16
        Hq = num_q_heads or 4
        Hkv = num_kv_heads or Hq
        return _build(name, seed, dtype or "fp16", B, Hq, Hkv, head_dim or 64, bs, ctx, 1.0,
                      partition_size if partition_size is not None else 0, rng, gen,
                      min_blocks=64, table_len=max_len or 200)
    if name == "llama3_8b_gqa":
        B = batch or 64
        ctx = np.asarray(lens) if lens is not None else rng.integers(512, (max_len or 4096) + 1, size=B)
        B = len(ctx)
        return _build(name, seed, dtype or "fp16", B, num_q_heads or 32, num_kv_heads or 8,
                      head_dim or 128, block_size or 16, ctx, 1.1,
                      partition_size if partition_size is not None else 1024, rng, gen,
                      table_len=max_len or 4096)
    if name == "shared_prefix_cow":
        ng = groups or 16
        gs = group_size or 8
        P = 2048 if prefix_len is None else prefix_len
        B = ng * gs
        suffix = rng.integers(1, (max_len or 512) + 1, size=B)
        ctx = P + suffix
        grp = [list(range(g * gs, (g + 1) * gs)) for g in range(ng)]
        return _build(name, seed, dtype or "fp16", B, num_q_heads or 32, num_kv_heads or 8,
                      head_dim or 128, block_size or 16, ctx, 1.1,
                      partition_size if partition_size is not None else 1024, rng, gen,
                      prefix_groups=grp, prefix_len=P, table_len=P + (max_len or 512))
    if name == "long_context":
        ctx = np.asarray(lens) if lens is not None else np.array([32768] * 6 + [65536, 131072])
        return _build(name, seed, dtype or "bf16", len(ctx), num_q_heads or 32, num_kv_heads or 8,
                      head_dim or 128, block_size or 16, ctx, 1.1,
                      partition_size if partition_size is not None else 512, rng, gen)
    if name == "llama3_70b_cb":
        B = batch or 256
        if lens is not None:
            ctx = np.asarray(lens)
        else:
            ctx = np.clip(np.round(rng.lognormal(mean=math.log(1024), sigma=1.0, size=B)),
                          1, max_len or 16384).astype(np.int64)
        return _build(name, seed, dtype or "fp16", len(ctx), num_q_heads or 64, num_kv_heads or 8,
                      head_dim or 128, block_size or 32, ctx, 1.2,
                      partition_size if partition_size is not None else 2048, rng, gen,
                      table_len=max_len or 16384)
    raise KeyError(f"unknown workload {name!r}; known: {NAMES}")


@dataclasses.dataclass
class PrefillWorkload(Workload):
    """A chunked-prefill batch: sequence i appends q_lens[i] new tokens, which
    end its context (positions ctx_i - q_len_i .. ctx_i - 1).  query, key,
    value are [total_q, heads, d] packed by sequence; query_start [B+1] gives
    each sequence's first row; slot_mapping [total_q] each new token's slot.
    Every chunk slot holds the poison value until the scatter writes it."""
    query_start: torch.Tensor = None   # int32 [B + 1]
    q_lens: torch.Tensor = None        # int32 [B]

    @property
    def total_q(self) -> int:
        return int(self.query_start[-1].item())

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max().item()) if self.num_seqs else 0


def make_prefill(name: str, seed: int = 0, *, chunk: int = 512,
                 q_lens: Optional[Sequence[int]] = None, **kw) -> PrefillWorkload:
    """A decode workload turned into a chunked-prefill batch: sequence i's
    last min(chunk, ctx_i) tokens (or q_lens[i]) are the new chunk."""
    w = make(name, seed, **kw)
    ctx = w.context_lens.numpy().astype(np.int64)
    ql = (np.minimum(ctx, chunk) if q_lens is None else np.asarray(q_lens, np.int64))
    ql = np.minimum(ql, ctx)
    qs = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    total = int(qs[-1])
    bs = w.block_size
    bt = w.block_tables.numpy()
    slots = np.empty(total, np.int64)
    for i in range(w.num_seqs):
        for t in range(int(ql[i])):
            pos = int(ctx[i] - ql[i] + t)
            slots[qs[i] + t] = int(bt[i, pos // bs]) * bs + pos % bs
    # the chunk's slots are poisoned until the scatter writes them
    if total:
        blk = torch.from_numpy(slots // bs)
        off = torch.from_numpy(slots % bs)
        for cache in (w.k_cache, w.v_cache):
            v = cache[blk, :, off, :]
            _poison(v, w.dtype)
            cache[blk, :, off, :] = v
    check_distinct_slots(slots)
    gen = torch.Generator().manual_seed(seed + 7919)
    return PrefillWorkload(
        **{f.name: getattr(w, f.name) for f in dataclasses.fields(Workload)
           if f.name not in ("query", "key", "value", "slot_mapping")},
        query=_randn((total, w.num_q_heads, w.head_dim), gen, w.dtype),
        key=_randn((total, w.num_kv_heads, w.head_dim), gen, w.dtype),
        value=_randn((total, w.num_kv_heads, w.head_dim), gen, w.dtype),
        slot_mapping=torch.from_numpy(slots),
        query_start=torch.from_numpy(qs), q_lens=torch.from_numpy(ql.astype(np.int32)))

