"""Host-side checks of the tensor-core linears' work decomposition, through
the library's own schedule query (tp_linear_schedule, no GPU needed).

For every workload shape and degree, and prompt sizes across the range,
with the scratch size the library asks for:
  * the scratch the launch touches fits in it (the split-tile counters and
    partial sums never leave the buffer);
  * the decomposition the header documents -- with S split items, item
    i < S is part i % parts of tile whole + i / parts, item S + t is the
    whole tile t, unit u takes items u, u + units, ... -- covers every
    (tile, k-block) exactly once, with at most 16 parts of at least 4
    k-blocks each;
  * the split tiles' counters and flags fit the 16 KB counter block;
  * the waits cannot deadlock when every unit is resident: a discrete
    simulation of the units' epilogues (partials published as reached, the
    parts reduced at the end of the unit's work once every part of their
    tile is published) runs to completion.
"""
import itertools

import pytest

from tensor_transformer_layer_03_b300 import inputs as I

SMS, PAIRS = 148, 74
FLAG_BYTES = 16384
PART_BLOCK = 128 * 256 * 4   # one 128 x 256 fp32 partial block per split item and rank


def _items(s):
    """Per-unit item lists [(kind, tile, k0, k1, key)] under the documented
    decomposition; kind is "full" or "part"."""
    units = [[] for _ in range(s.units)]
    kbt = s.k_blocks_per_tile
    n_split = s.items - s.whole_tiles
    for w in range(s.items):
        if w >= n_split:
            units[w % s.units].append(("full", w - n_split, 0, kbt, None))
        else:
            part = w % s.parts
            tile = s.whole_tiles + w // s.parts
            units[w % s.units].append(("part", tile, kbt * part // s.parts, kbt * (part + 1) // s.parts, w))
    return units


def _coverage(units):
    seen = {}
    for items in units:
        for (_, tile, k0, k1, _) in items:
            for kb in range(k0, k1):
                seen[(tile, kb)] = seen.get((tile, kb), 0) + 1
    return seen


def _simulate(units):
    """True when every unit's epilogue gets through its work.  A part is
    published when the unit reaches it (its partial write waits for
    nothing); at the end of its items the unit reduces its parts, each of
    which needs every part of its tile published."""
    parts_of = {}
    for items in units:
        for (kind, tile, _, _, key) in items:
            if kind == "part":
                parts_of.setdefault(tile, set()).add(key)
    published = set()
    for items in units:  # reaching an item depends on nothing else
        published |= {key for (kind, _, _, _, key) in items if kind == "part"}
    return all(parts_of[tile] <= published for items in units for (kind, tile, _, _, _) in items if kind == "part")


SHAPES = [(I.LLAMA7B, (1, 2, 4, 8)), (I.LLAMA13B, (1, 2, 4, 8)), (I.BlockShape(512, 8, 1536, "swiglu"), (1, 2, 4, 8)),
          (I.BlockShape(1024, 8, 2816, "swiglu"), (2, 4, 8)), (I.BlockShape(256, 4, 1024, "gelu"), (1, 2))]
MS = [9, 16, 64, 100, 128, 129, 200, 256, 300, 512, 640, 1000, 1024, 2048, 4096, 8192]


@pytest.mark.parametrize("shape,degs", SHAPES, ids=lambda v: getattr(v, "d_model", None) or str(v))
def test_schedule_bounds_and_coverage(tp, shape, degs):
    n_split = 0
    llama = shape.d_model >= 4096
    for deg, M, (row, which) in itertools.product(degs, MS, ((0, 0), (0, 1), (1, 0), (1, 1))):
        plan = tp.Plan(shape.d_model, shape.n_heads, shape.d_ffn, deg, act=shape.act)
        nscr = plan.linear_scratch_bytes(M)
        s = plan.linear_schedule(row, which, M, nscr, SMS, PAIRS)
        if s.kernel != 0:
            assert M <= 32 or nscr == 0  # the weight streams take up to 32 rows
            continue
        what = f"d={shape.d_model} tp{deg} M={M} row={row} which={which}"
        ranks = 2 if s.paired else 1
        assert s.units <= (PAIRS if s.paired else SMS), what
        assert s.scratch_bytes_touched <= nscr, what
        if s.parts == 1:
            assert s.items == s.tiles == s.whole_tiles and s.scratch_bytes_touched == 0, what
            continue
        n_split += 1
        units = _items(s)
        seen = _coverage(units)
        assert len(seen) == s.tiles * s.k_blocks_per_tile and set(seen.values()) == {1}, what
        assert sum(len(x) for x in units) == s.items, what
        assert _simulate(units), what
        split_tiles = s.tiles - s.whole_tiles
        assert 2 <= s.parts <= 16 and s.whole_tiles % s.units == 0 and 0 < split_tiles < s.units, what
        assert s.items == s.whole_tiles + split_tiles * s.parts, what
        assert s.k_blocks_per_tile // s.parts >= 4, what
        assert s.items - s.whole_tiles <= 4 * s.units, what
        # a part's rows of a warp's block and the residual rows, 512 bytes
        # each, fit the warp's 24 KB share of the ring at the end
        assert (s.parts + 1) * -(-32 // s.parts) * 512 <= 24 * 1024, what
        assert split_tiles * ranks * 8 * 2 * 4 <= FLAG_BYTES, what  # 8 epilogue warps, 2 counters each
        assert s.scratch_bytes_touched == FLAG_BYTES + (s.items - s.whole_tiles) * ranks * PART_BLOCK, what
    assert n_split > 0 or not llama  # the LLaMA shapes do exercise split tiles


def test_schedule_headline_prompt(tp):
    """The 7B block at tp 4.  The 2048-token prompt runs whole tiles in every
    linear: QKV's ragged last round is 14 of 384 tiles, and cutting the 54
    tiles of the row-parallel linears' second round would move more
    partial-sum traffic than the round it saves.  A 128-token prompt (16
    row-parallel tiles for 148 SMs) cuts every row-parallel tile; a
    4096-token prompt cuts the ragged last round of FFN-up and FFN-down.
    No scratch means whole tiles only."""
    plan = tp.Plan(4096, 32, 11008, 4)
    n = plan.linear_scratch_bytes(2048)
    for row, which in ((0, 0), (1, 0), (0, 1), (1, 1)):
        s = plan.linear_schedule(row, which, 2048, n, SMS, PAIRS)
        assert s.kernel == 0 and s.paired and s.parts == 1 and s.whole_tiles == s.tiles
    n = plan.linear_scratch_bytes(128)
    for which in (0, 1):
        s = plan.linear_schedule(1, which, 128, n, SMS, PAIRS)
        assert (s.kernel, s.paired, s.tiles, s.whole_tiles) == (0, 0, 16, 0) and s.parts >= 2
        assert s.items == 16 * s.parts
    n = plan.linear_scratch_bytes(4096)
    s = plan.linear_schedule(1, 1, 4096, n, SMS, PAIRS)
    assert (s.tiles, s.whole_tiles) == (256, 222) and s.parts >= 2
    s0 = plan.linear_schedule(1, 1, 4096, 0, SMS, PAIRS)
    assert (s0.parts, s0.items, s0.units) == (1, 256, 74)
    # the weight-streaming kernels for a handful of rows
    assert plan.linear_schedule(0, 0, 1, n, SMS, PAIRS).kernel == 2
    assert plan.linear_schedule(0, 0, 4, n, SMS, PAIRS).kernel == 1


def test_schedule_query_argument_checks(tp):
    import ctypes
    plan = tp.Plan(512, 8, 1536, 2)
    out = tp.LinearSchedule()
    ptr = ctypes.cast(ctypes.byref(out), ctypes.c_void_p)
    assert tp.tp_linear_schedule(None, 0, 0, 64, 0, SMS, PAIRS, ptr) == 1
    assert tp.tp_linear_schedule(plan.handle, 0, 0, 64, 0, SMS, PAIRS, None) == 1
    assert tp.tp_linear_schedule(plan.handle, 0, 0, 0, 0, SMS, PAIRS, ptr) == 2
    assert tp.tp_linear_schedule(plan.handle, 2, 0, 64, 0, SMS, PAIRS, ptr) == 2
    assert tp.tp_linear_schedule(plan.handle, 0, 0, 64, 0, 0, PAIRS, ptr) == 2


def test_schedule_few_rows(tp):
    """Batched decode (7B block, tp 2): up to 32 token rows the linears run
    the tensor-core weight stream (kernel 1); above, the tensor-core GEMM on
    128-row tiles.  A 48-row tile holds 3/8 of a full tile's rows, so its
    partials are 3/8 as large and cutting the 48 QKV tiles into parts that
    fill the SMs pays; at 128 rows (a full tile) the same 48 tiles stay
    whole."""
    plan = tp.Plan(4096, 32, 11008, 2)
    for M in (2, 9, 16, 24, 32):
        n = plan.linear_scratch_bytes(M)
        assert {plan.linear_schedule(r, w, M, n, SMS, PAIRS).kernel for r in (0, 1) for w in (0, 1)} == {1}, M
    n48 = plan.linear_scratch_bytes(48)
    s = plan.linear_schedule(0, tp.TP_QKV, 48, n48, SMS, PAIRS)
    assert (s.kernel, s.paired, s.tiles) == (0, 0, 48) and s.parts >= 2 and s.items <= SMS
    assert s.whole_tiles == 0 and s.items == 48 * s.parts
    n128 = plan.linear_scratch_bytes(128)
    s = plan.linear_schedule(0, tp.TP_QKV, 128, n128, SMS, PAIRS)
    assert (s.tiles, s.parts, s.whole_tiles) == (48, 1, 48)
