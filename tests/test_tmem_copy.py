"""The tcgen05.cp copy primitive without a GPU: the form parser, the planner's
inference and rejections, and the oracle pinned to the page's lane table.

Page: "TVM Blackwell tcgen05.cp 全解析" — sections 形状选择 (forms and their
multicast), 形状 → 行/复制模式映射表 (lanes and replicas), 调度算法四步 (one
descriptor, a patched start address per instruction), 负向校验 (rejections) and
测试矩阵 (instruction counts of the compile-level tests).
"""
import os
import re

import numpy as np
import pytest

import tile_primitive_tensor_gb300 as tp
from tile_primitive_tensor_gb300 import build as tpbuild
from oracle import tmem_cp as ocp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tcgen05_cp_lane_table.txt")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tpbuild.build()


def plan(**kw):
    rows, bits = kw.pop("rows"), kw.pop("row_bits")
    st, text = tp.tpgemm_cp_plan(tp.cp_desc(rows, bits, **kw))
    return st, text


def instrs(text):
    return [tuple(int(x) for x in m) for m in re.findall(r"smem=(\d+) lane=(\d+) col=(\d+)", text)]


# ------------------------------------------------------------------ parser
@pytest.mark.parametrize("name,code", [
    ("128x256b", tp.TPGEMM_CP_128x256b), ("4x256b", tp.TPGEMM_CP_4x256b),
    ("128x128b", tp.TPGEMM_CP_128x128b),
    ("64x128b.warpx2::02_13", tp.TPGEMM_CP_64x128b_WARPX2_02_13),
    ("64x128b.warpx2::01_23", tp.TPGEMM_CP_64x128b_WARPX2_01_23),
    ("32x128b.warpx4", tp.TPGEMM_CP_32x128b_WARPX4), ("32x128b", tp.TPGEMM_CP_32x128b_WARPX4),
])
def test_parse_legal_forms(name, code):
    assert tp.tpgemm_cp_parse_shape(name) == (tp.TPGEMM_OK, code)


@pytest.mark.parametrize("name,frag", [
    ("64x128b", "requires an explicit multicast"),
    ("128x256b.warpx4", "illegal multicast"),
    ("64x128b.warpx4", "illegal multicast"),
    ("32x128b.warpx2::02_13", "illegal multicast"),
    ("96x128b", "unknown tcgen05.cp shape"),
])
def test_parse_rejections(name, frag):
    st, _ = tp.tpgemm_cp_parse_shape(name)
    assert st == tp.TPGEMM_ERR_SHAPE and frag in tp.tpgemm_last_error_detail()


# --------------------------------------------------------------- inference
def test_wider_256b_atom_inferred_for_rows():
    # A region 128x128b could copy is copied by the wider 128x256b atom: half
    # the instructions (the page's test_cp_128x128b_layout_infers_wider_256b_atom).
    st, text = plan(rows=128, row_bits=256, lbo=2048, sbo=128)
    assert st == 0 and text.startswith("form=128x256b instructions=1 "), text
    st, text = plan(rows=128, row_bits=256, lbo=2048, sbo=128, shape=tp.TPGEMM_CP_128x128b)
    assert st == 0 and text.startswith("form=128x128b instructions=2 "), text
    st, text = plan(rows=128, row_bits=384, lbo=2048, sbo=128)
    assert st == 0 and text.startswith("form=128x128b instructions=3 "), text


@pytest.mark.parametrize("lanes,rows,bits,form", [
    (tp.TPGEMM_CP_LANES_QUADRANTS, 4, 256, "4x256b"),
    (tp.TPGEMM_CP_LANES_PAIRS_02_13, 64, 128, "64x128b.warpx2::02_13"),
    (tp.TPGEMM_CP_LANES_PAIRS_01_23, 64, 128, "64x128b.warpx2::01_23"),
    (tp.TPGEMM_CP_LANES_ALL_QUADS, 32, 128, "32x128b.warpx4"),
])
def test_lane_pattern_selects_its_form(lanes, rows, bits, form):
    st, text = plan(rows=rows, row_bits=bits, lanes=lanes, lbo=1024, sbo=128)
    assert st == 0 and text.startswith(f"form={form} instructions=1 "), text


def test_four_256b_steps_one_descriptor():
    # 128 rows x 1024 bits, 128-byte swizzle: four 128x256b instructions 32 bytes
    # apart in shared memory and 8 columns apart in tensor memory; one template.
    st, text = plan(rows=128, row_bits=1024, swizzle=tp.TPGEMM_CP_SWIZZLE_128B, sbo=1024)
    assert st == 0, text
    assert text.count("desc=") == 1
    assert instrs(text) == [(0, 0, 0), (32, 0, 8), (64, 0, 16), (96, 0, 24)]


def test_4x256b_two_middle_steps():
    st, text = plan(rows=4, row_bits=512, lanes=tp.TPGEMM_CP_LANES_QUADRANTS, lbo=128, sbo=0)
    assert st == 0 and "form=4x256b instructions=2 " in text, text
    assert instrs(text) == [(0, 0, 0), (256, 0, 8)]


def test_4x256b_lane_tiled_scatter():
    # 64 rows in quadrant order: 16 instructions, each on its own lane (0..15)
    # of every quadrant (the page's Layout-F scatter test).
    st, text = plan(rows=64, row_bits=256, lanes=tp.TPGEMM_CP_LANES_QUADRANTS, lbo=1024, sbo=128)
    assert st == 0 and "instructions=16 " in text, text
    ins = instrs(text)
    assert [i[1] for i in ins] == list(range(16))
    assert [i[0] for i in ins] == [(4 * i // 8) * 128 + (4 * i % 8) * 16 for i in range(16)]


def test_4x256b_partial_window_lane_offset():
    # Rows 16..47 of such a region: the lane offset folds into the address so
    # the rows land on lanes 32q + 4..11.
    st, text = plan(rows=32, row_bits=256, lanes=tp.TPGEMM_CP_LANES_QUADRANTS, lbo=1024,
                    sbo=128, lane_offset=4)
    assert st == 0, text
    assert [i[1] for i in instrs(text)] == list(range(4, 12))


# -------------------------------------------------------------- rejections
@pytest.mark.parametrize("kw,frag", [
    (dict(rows=64, row_bits=128, lanes=tp.TPGEMM_CP_LANES_PAIRS_01_23,
          shape=tp.TPGEMM_CP_64x128b_WARPX2_02_13, lbo=1024, sbo=128), "replica mismatch"),
    (dict(rows=64, row_bits=128, lanes=tp.TPGEMM_CP_LANES_PAIRS_02_13,
          shape=tp.TPGEMM_CP_64x128b_WARPX2_01_23, lbo=1024, sbo=128), "replica mismatch"),
    (dict(rows=128, row_bits=256, lanes=tp.TPGEMM_CP_LANES_ROWS,
          shape=tp.TPGEMM_CP_32x128b_WARPX4, lbo=2048, sbo=128), "replica mismatch"),
    (dict(rows=128, row_bits=256, lbo=2048, sbo=128, tmem_col=2), "not 128b-aligned"),
    (dict(rows=128, row_bits=256, lbo=2048, sbo=128, lane_offset=32), "overflows the 128-lane"),
    (dict(rows=64, row_bits=256, lanes=tp.TPGEMM_CP_LANES_QUADRANTS, lbo=1024, sbo=128,
          lane_offset=20), "overflow the 128-lane"),
    (dict(rows=128, row_bits=256, lbo=2048, sbo=120), "not 16B-aligned"),
    (dict(rows=128, row_bits=200, lbo=2048, sbo=128), "multiple of 128"),
    (dict(rows=96, row_bits=256, lbo=2048, sbo=128), "copies exactly 128 rows"),
    (dict(rows=128, row_bits=256, lbo=0, sbo=128), "two 16-byte units"),
    (dict(rows=32, row_bits=256, swizzle=tp.TPGEMM_CP_SWIZZLE_128B, sbo=1024, smem_offset=512,
          lanes=tp.TPGEMM_CP_LANES_QUADRANTS), "swizzle atom"),
    (dict(rows=32, row_bits=512, swizzle=tp.TPGEMM_CP_SWIZZLE_32B, sbo=256, lbo=100,
          lanes=tp.TPGEMM_CP_LANES_QUADRANTS), "16B-aligned"),
    (dict(rows=32, row_bits=512, swizzle=tp.TPGEMM_CP_SWIZZLE_32B, sbo=256, lbo=272,
          lanes=tp.TPGEMM_CP_LANES_QUADRANTS), "multiple of the 256-byte swizzle atom"),
    (dict(rows=128, row_bits=256, lbo=2048, sbo=128, cta_group=3), "cta_group"),
])
def test_plan_rejections(kw, frag):
    st, text = plan(**kw)
    assert st == tp.TPGEMM_ERR_SHAPE, text
    assert frag in text and frag in tp.tpgemm_last_error_detail(), text


def test_roundtrip_argument_checks_need_no_gpu():
    d = tp.cp_desc(128, 256, lbo=2048, sbo=128)
    base = 0x7F0000000000
    assert tp.tpgemm_cp_roundtrip(None, base, 4096, d, 0, 32, 0) == tp.TPGEMM_ERR_NULL
    assert tp.tpgemm_cp_roundtrip(base + 4, base, 4096, d, 0, 32, 0) == tp.TPGEMM_ERR_ALIGN
    assert tp.tpgemm_cp_roundtrip(base, base, 4000, d, 0, 32, 0) == tp.TPGEMM_ERR_SHAPE
    assert tp.tpgemm_cp_roundtrip(base, base, 4096, d, 0, 48, 0) == tp.TPGEMM_ERR_SHAPE
    # the region (16 groups of 128 bytes, second units 2048 bytes on) ends at 4096
    assert tp.tpgemm_cp_roundtrip(base, base, 2048, d, 0, 32, 0) == tp.TPGEMM_ERR_SHAPE
    assert "reads up to byte 4096" in tp.tpgemm_last_error_detail()
    # columns beyond the read-back window
    d = tp.cp_desc(128, 256, lbo=2048, sbo=128, tmem_col=28)
    assert tp.tpgemm_cp_roundtrip(base, base, 4096, d, 0, 32, 0) == tp.TPGEMM_ERR_SHAPE
    assert "writes up to column 36" in tp.tpgemm_last_error_detail()


# ------------------------------------------------------- oracle pins (page)
def read_table():
    forms, prose = {}, []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("@"):
            form, rows, warps = [x.strip() for x in line[1:].split("|")]
            lo, hi = (int(x) for x in rows.split("-"))
            prose.append((form, lo, hi, {int(w) for w in warps.split(",")}))
            continue
        form, rows, bits, pat, rep = [x.strip() for x in line.split("|")]
        modes = [tuple(int(v) for v in m.split(",")) for m in re.findall(r"\((\d+,\d+)\)", pat)]
        if ":" in pat:  # (e0,e1):(s0,s1) -- extents then strides
            (e0, e1), (s0, s1) = modes
            modes = [(e0, s0), (e1, s1)]
        replica = None if rep == "-" else tuple(int(v) for v in rep.strip("()").split(","))
        forms[form] = (int(rows), int(bits), modes, replica)
    return forms, prose


def page_lanes(entry, r):
    """Evaluate the page's notation directly: last mode fastest."""
    rows, _bits, modes, replica = entry
    coords, rem = [], r
    for extent, _stride in reversed(modes):
        coords.append(rem % extent)
        rem //= extent
    base = sum(c * s for c, (_e, s) in zip(coords, reversed(modes)))
    return sorted(base + k * replica[1] for k in range(replica[0])) if replica else [base]


def test_oracle_lane_table_matches_page():
    forms, prose = read_table()
    assert set(forms) == set(ocp.LANE_TABLE)
    for name, entry in forms.items():
        assert ocp.LANE_TABLE[name][:2] == entry[:2], name
        lanes = set()
        for r in range(entry[0]):
            got = sorted(ocp.form_lanes(name, r))
            assert got == page_lanes(entry, r), (name, r)
            lanes.update(got)
        # every form writes each lane at most once per instruction
        copies = 1 if entry[3] is None else entry[3][0]
        assert len(lanes) == entry[0] * copies, name
    for form, lo, hi, warps in prose:
        for r in range(lo, hi + 1):
            assert {lane // 32 for lane in ocp.form_lanes(form, r)} == warps, (form, r)
            if form == "32x128b.warpx4":
                assert sorted(ocp.form_lanes(form, r)) == [r, r + 32, r + 64, r + 96]


def test_oracle_quadrant_region_scatter():
    # A 4x256b region of 64 rows fills lanes 32q + 0..15 (the page's Layout-F
    # scatter), each lane once.
    lanes = [ocp.dest_lanes(ocp.LANES_QUADRANTS, r)[0] for r in range(64)]
    assert sorted(lanes) == sorted(32 * q + i for q in range(4) for i in range(16))
    assert ocp.dest_lanes(ocp.LANES_QUADRANTS, 5, 4) == [32 + 4 + 1]


@pytest.mark.parametrize("swz", [ocp.SWIZZLE_32B, ocp.SWIZZLE_64B, ocp.SWIZZLE_128B])
def test_oracle_swizzle_is_a_permutation_of_each_atom(swz):
    # The XOR only moves 16-byte units inside their own row's atom: within
    # every (8 rows x atom row) block the swizzled addresses are exactly the
    # unswizzled ones, permuted; row 0 of the atom is never moved.
    s = ocp.ROW_BYTES[swz]
    units = s // 16
    for r0 in (0, 8, 16):
        plain = sorted(r0 // 8 * 8 * s + (r % 8) * s + 16 * u for r in range(r0, r0 + 8)
                       for u in range(units))
        swz_addr = sorted(ocp.unit_address(r, u, swz, 0, 8 * s, 0) for r in range(r0, r0 + 8)
                          for u in range(units))
        assert plain == swz_addr
        assert [ocp.unit_address(r0, u, swz, 0, 8 * s, 0) for u in range(units)] == \
            [r0 // 8 * 8 * s + 16 * u for u in range(units)]
    # 128-byte swizzle: unit u of row r sits at unit u ^ (r % 8) of its row
    if swz == ocp.SWIZZLE_128B:
        for r in range(8):
            for u in range(8):
                assert ocp.unit_address(r, u, swz, 0, 1024, 0) == r * 128 + 16 * (u ^ r)


def read_swizzle_cells():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "smem_swizzle_cells.txt")
    rows = []
    with open(path) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(tuple(int(v) for v in line.split()))
    return rows


SWIZZLE_OF_BYTES = {32: ocp.SWIZZLE_32B, 64: ocp.SWIZZLE_64B, 128: ocp.SWIZZLE_128B}


def test_oracle_swizzle_matches_golden_cells():
    # Byte offsets of single units read off the PTX ISA's swizzle figures: a
    # wrong XOR field (other bits, another width) moves at least one of them.
    cells = read_swizzle_cells()
    assert {c[0] for c in cells} == {32, 64, 128}
    for s, r, u, want in cells:
        got = ocp.unit_address(r, u, SWIZZLE_OF_BYTES[s], 0, 8 * s, 0)
        assert got == want, (s, r, u, got, want)


@pytest.mark.parametrize("bad", ["phase_bits_6", "phase_mod_4"])
def test_planted_swizzle_mistakes_fail_the_golden_cells(bad, monkeypatch):
    # Two plausible slips, planted in the oracle: the row phase read from
    # address bits starting at 6 instead of 7, and the 128-byte phase taken
    # modulo 4. Both still permute each atom, and both fail the golden cells.
    def planted(r, u, swizzle, lbo, sbo, offset):
        s = ocp.ROW_BYTES[swizzle]
        per_row = s // 16
        a = offset + (u // per_row) * lbo + (r // 8) * sbo + (r % 8) * s + 16 * (u % per_row)
        if bad == "phase_bits_6":
            return a ^ (((a >> 6) & (per_row - 1)) << 4)
        return a ^ (((a >> 7) & min(per_row - 1, 3)) << 4)
    monkeypatch.setattr(ocp, "unit_address", planted)
    with pytest.raises(AssertionError):
        test_oracle_swizzle_matches_golden_cells()


def test_oracle_tmem_image_fill_and_replicas():
    words = np.arange(32 * 4, dtype=np.uint32).reshape(32, 4)
    out = ocp.tmem_image(words, ocp.LANES_ALL_QUADS, 0, 8, 32, 7)
    for q in range(4):
        assert np.array_equal(out[32 * q: 32 * q + 32, 8:12], words)
    assert out[5, 0] == 7 + 5 * 65536 and out[127, 31] == 7 + 127 * 65536 + 31


# ------------------------------------------- tensor memory <-> registers maps
from oracle import tmem_frag as ofr  # noqa: E402

LDST_CASES = [(s, c) for s in range(4) for c in (2, 4, 8, 16)
              if c >= {0: 1, 1: 2, 2: 4, 3: 8}[s]]


@pytest.mark.parametrize("shape,cols", [c for c in LDST_CASES if c[0] != ofr.S16x64b])
def test_ldst_map_is_a_bijection_onto_the_footprint(shape, cols):
    cells = {ofr.cell(shape, cols, t, j) for t in range(32) for j in range(cols)}
    assert cells == {(lane, c) for lane in range(32) for c in range(cols)}


def read_thread_maps():
    """The golden table: shape name -> {(lane, column): (thread, register)}."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "tcgen05_ldst_thread_maps.txt")
    maps, cur = {}, None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("shape "):
                cur = maps.setdefault(line.split()[1], {})
                continue
            head, cells = line.split(":")
            lane = int(head.split()[1])
            for col, e in enumerate(cells.split()):
                t, r = e.split(".")
                cur[(lane, col)] = (int(t[1:]), int(r[1:]))
    return maps


def test_ldst_16x64b_map_is_declared_unpinned():
    with pytest.raises(ValueError):
        ofr.cell(ofr.S16x64b, 2, 0, 0)


@pytest.mark.parametrize("shape", [ofr.S16x128b, ofr.S16x256b], ids=lambda s: ofr.NAMES[s])
def test_ldst_map_matches_the_golden_figure_table(shape):
    # One .x1 issue (the first 16 lanes of a warp): every cell of the table
    # names the (thread, register) the oracle places there, and the table
    # covers the shape's 16 x w block exactly once.
    table = read_thread_maps()[ofr.NAMES[shape]]
    w, regs = ofr.REPEAT_COLS[shape], ofr.REPEAT_REGS[shape]
    assert set(table) == {(lane, c) for lane in range(16) for c in range(w)}
    assert sorted(table.values()) == sorted((t, r) for t in range(32) for r in range(regs))
    for (lane, col), (t, r) in table.items():
        assert ofr.cell(shape, 2 * regs, t, r) == (lane, col), (lane, col, t, r)


def test_ldst_planted_16x128b_mistake_fails_the_table(monkeypatch):
    # A plausible slip, planted in the oracle: .16x128b with two threads per
    # lane (lane t/2, column 2 (t%2) + h) instead of four; it fails the table.
    real = ofr.cell

    def planted(shape, cols, t, j):
        if shape == ofr.S16x128b:
            half = cols // 2
            slab, k = divmod(j, half)
            rep, h = divmod(k, 2)
            return 16 * slab + t // 2, 4 * rep + 2 * (t % 2) + h
        return real(shape, cols, t, j)
    monkeypatch.setattr(ofr, "cell", planted)
    with pytest.raises(AssertionError):
        test_ldst_map_matches_the_golden_figure_table(ofr.S16x128b)


def test_ldst_16x256b_is_the_mma_accumulator_fragment():
    # The synchronous gemm page, section 三: thread `lane` holds D registers
    # c_id = 2 rM + rN at M = lane // 4 + 8 rM, N = 2 (lane % 4) + rN.
    for lane in range(32):
        for rM in range(2):
            for rN in range(2):
                assert ofr.cell(ofr.S16x256b, 8, lane, 2 * rM + rN) == \
                    (lane // 4 + 8 * rM, 2 * (lane % 4) + rN)
    # the second issue of a warp covers its lanes 16..31 with registers 4..7
    assert ofr.cell(ofr.S16x256b, 8, 5, 6) == (16 + 1 + 8, 2 * 1)


def test_ldst_32x32b_is_the_page_3_demo_layout():
    # 128 x 8 fp16 (4 x 32-bit columns): element (row, col) in thread `row`,
    # register `col`, lane `row`, column `col`.
    for t in range(32):
        for j in range(4):
            assert ofr.cell(ofr.S32x32b, 4, t, j) == (t, j)


def test_ldst_roundtrip_rejections():
    base = 0x7F0000000000
    def f(*a):
        return tp.tpgemm_tmem_ldst_roundtrip(*a, 0)
    assert f(None, base, base, 0, 0, 8, 0, 0) == tp.TPGEMM_ERR_NULL
    assert f(base + 4, base, base, 0, 0, 8, 0, 0) == tp.TPGEMM_ERR_ALIGN
    assert f(base, base, base, 3, 0, 4, 0, 0) == tp.TPGEMM_ERR_SHAPE
    assert "16x256b moves at least 8 columns" in tp.tpgemm_last_error_detail()
    assert f(base, base, base, 0, 0, 6, 0, 0) == tp.TPGEMM_ERR_SHAPE
    assert f(base, base, base, 0, 0, 16, 24, 0) == tp.TPGEMM_ERR_SHAPE
    assert f(base, base, base, 0, 0, 8, 4, 0) == tp.TPGEMM_ERR_SHAPE
    assert f(base, base, base, 5, 0, 8, 0, 0) == tp.TPGEMM_ERR_SHAPE
