"""CPU model of the in-place FP8 widening in the tcgen05 attention kernel.

The kernel copies a step's E4M3 codes (64 rows of head_dim bytes, in the pool
map's swizzle) into the upper half of the step's fp16 stage and widens them
there, pass by pass, into the fp16 tile the MMAs read.  This test replays the
kernel's index arithmetic (f8_stage_to_f16 and its callers: 1 KB passes,
groups of four passes read before they are written, at head_dim 128 the
producer and a helper warp taking the two halves of the passes at the same
time) byte by byte, and checks that

  * every fp16 unit ends up holding exactly the code unit it should,
  * no byte of codes is overwritten before every warp that needs it has read
    it (the warps of a split run in any interleaving of their groups),
  * each 8-lane phase of every 16-byte store touches eight different bank
    groups (no shared-memory bank conflict).

The layouts are the hardware's swizzles as the kernel states them: 16-byte
unit c of 128-byte row r at c ^ (r & 7), of 64-byte row r at
c ^ ((r >> 1) & 3); fp16 tiles are 64-row atoms of 128-byte rows.
"""
import itertools

import pytest

KEYS = 64          # rows of a step
ATOM = 64 * 128    # bytes of one fp16 atom (64 rows x 128 bytes)
GROUP = 4          # passes read before the writes


def code_addr(D, r, c):
    """Byte offset, inside the stage, of 16-byte code unit c of row r."""
    base = (D // 64) * ATOM // 2
    sw = (r & 7) if D == 128 else ((r >> 1) & 3)
    return base + r * D + ((c ^ sw) << 4)


def half_addr(r, k, atom):
    """Byte offset of 16-byte fp16 unit k (8 dims) of row r in the given atom."""
    return atom * ATOM + r * 128 + ((k ^ (r & 7)) << 4)


def lane_plan(D, lane, j):
    """What one lane does in pass j: (row, [code units read], [(fp16 atom,
    unit, source code unit, half)] written), as the kernel computes it."""
    rows = 1024 // D
    per_row = 32 // rows
    r = j * rows + lane // per_row
    c0 = 2 * (lane % per_row)
    flip = D == 128 and bool(lane & 2)
    xa, xb = (c0 + 1, c0) if flip else (c0, c0 + 1)       # h0 from xa, h1 from xb
    ka = 2 * (c0 & 3) + (2 if flip else 0)
    kb = 2 * (c0 & 3) + (0 if flip else 2)
    atom = c0 >> 2
    writes = [(atom, ka, xa, 0), (atom, ka + 1, xa, 1), (atom, kb, xb, 0), (atom, kb + 1, xb, 1)]
    return r, [c0, c0 + 1], writes


def warp_groups(D, helpers):
    passes = KEYS // (1024 // D)
    if helpers:
        return [list(range(0, passes // 2)), list(range(passes // 2, passes))]
    return [list(range(passes))]


@pytest.mark.parametrize("D,helpers", [(128, False), (128, True), (64, False)])
def test_every_unit_lands_where_the_mma_reads_it(D, helpers):
    expected = {}
    for r in range(KEYS):
        for c in range(D // 16):             # code unit c: dims 16c .. 16c + 15
            for half in (0, 1):              # fp16 unit: dims 16c + 8 half ..
                expected[(r, c >> 2, 2 * (c & 3) + half)] = (r, c, half)
    got = {}
    for passes in warp_groups(D, helpers):
        for j in passes:
            for lane in range(32):
                r, _, writes = lane_plan(D, lane, j)
                for atom, k, src, half in writes:
                    key = (r, atom, k)
                    assert key not in got, f"fp16 unit {key} written twice"
                    got[key] = (r, src, half)
    assert got == expected


def _schedule_ok(D, warp_passes, order):
    """Replay one interleaving of the warps' groups: each group reads all its
    lanes' code units, then writes all its fp16 units.  A byte read after it
    was overwritten, or overwritten before its reader ran, fails."""
    live = {}                                # byte -> (row, code unit) still to be read
    for r in range(KEYS):
        for c in range(D // 16):
            a = code_addr(D, r, c)
            for b in range(16):
                live[a + b] = (r, c)
    pending = {w: [ps[i:i + GROUP] for i in range(0, len(ps), GROUP)]
               for w, ps in enumerate(warp_passes)}
    for w in order:
        group = pending[w].pop(0)
        reads, writes = [], []
        for j in group:
            for lane in range(32):
                r, units, wr = lane_plan(D, lane, j)
                reads += [(r, c) for c in units]
                writes += [half_addr(r, k, atom) for atom, k, _, _ in wr]
        for r, c in reads:
            a = code_addr(D, r, c)
            for b in range(16):
                if live.get(a + b) != (r, c):
                    return False                  # already overwritten
                del live[a + b]
        for a in writes:
            for b in range(16):
                if a + b in live:
                    return False                  # clobbers codes not yet read
    return not live


@pytest.mark.parametrize("D,helpers", [(128, False), (128, True), (64, False)])
def test_no_code_is_overwritten_before_it_is_read(D, helpers):
    warp_passes = warp_groups(D, helpers)
    groups = [len(ps) // GROUP for ps in warp_passes]
    # every interleaving of the warps' group sequences
    seq = [w for w, n in enumerate(groups) for _ in range(n)]
    orders = set(itertools.permutations(seq))
    assert orders
    for order in orders:
        assert _schedule_ok(D, warp_passes, order), (D, helpers, order)


def test_the_model_sees_a_hazard_when_there_is_one():
    """At head_dim 64 the four passes are one group; reading them two at a time
    would let the second half's writes clobber codes the first half has
    already read -- fine -- but splitting them over two warps in either order
    overwrites codes the other warp has not read yet."""
    D = 64
    bad = [[0, 1], [2, 3]]
    global GROUP
    saved, GROUP = GROUP, 2
    try:
        assert not _schedule_ok(D, bad, (1, 0))
    finally:
        GROUP = saved


@pytest.mark.parametrize("D", [128, 64])
def test_store_phases_hit_distinct_bank_groups(D):
    rows = 1024 // D
    for j in range(KEYS // rows):
        for inst in range(4):                    # the four 16-byte stores of a pass
            for phase in range(4):               # eight lanes per phase
                groups = []
                for lane in range(8 * phase, 8 * phase + 8):
                    r, _, writes = lane_plan(D, lane, j)
                    atom, k, _, _ = writes[inst]
                    groups.append((half_addr(r, k, atom) // 16) % 8)
                assert len(set(groups)) == 8, (D, j, inst, phase, groups)
