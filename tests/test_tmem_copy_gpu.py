"""tcgen05.cp round trips on the GPU, bit for bit against the oracle.

The matrix follows the page "TVM Blackwell tcgen05.cp 全解析", section 测试矩阵:
every (shape, multicast) form x swizzle {none, 32B, 64B, 128B} x element width
{16, 32} bits x {1, 4} instructions along the row; sub-region offsets (shared
memory, tensor-memory column, lane); inferred vs explicit forms; cta_group 2
pair copies. A host image goes to shared memory in the described layout, the
planned copy runs, every warp reads its 32-lane slab back, and the expected
tensor memory is rebuilt on the host from the destination layout alone.
"""
import numpy as np
import pytest
import torch

import tile_primitive_tensor_gb300 as tp
from oracle import tmem_cp as ocp

pytestmark = pytest.mark.gpu

FORMS = [  # (shape code, lane pattern, rows of one instruction, bits of a row)
    (tp.TPGEMM_CP_128x256b, tp.TPGEMM_CP_LANES_ROWS, 128, 256),
    (tp.TPGEMM_CP_4x256b, tp.TPGEMM_CP_LANES_QUADRANTS, 4, 256),
    (tp.TPGEMM_CP_128x128b, tp.TPGEMM_CP_LANES_ROWS, 128, 128),
    (tp.TPGEMM_CP_64x128b_WARPX2_02_13, tp.TPGEMM_CP_LANES_PAIRS_02_13, 64, 128),
    (tp.TPGEMM_CP_64x128b_WARPX2_01_23, tp.TPGEMM_CP_LANES_PAIRS_01_23, 64, 128),
    (tp.TPGEMM_CP_32x128b_WARPX4, tp.TPGEMM_CP_LANES_ALL_QUADS, 32, 128),
]
FORM_IDS = ["128x256b", "4x256b", "128x128b", "64x128b_02_13", "64x128b_01_23",
            "32x128b_warpx4"]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    tp.library()


def layout(swz, rows, units, variant=0):
    """(lbo, sbo) of a compact canonical layout for rows x units 16-byte units."""
    groups = (rows + 7) // 8
    if swz == ocp.SWIZZLE_NONE:
        if variant == 0:  # a row group's core matrices side by side along the row
            return 128, 128 * units
        return 128 * groups, 128  # all row groups of one unit column first
    s = ocp.ROW_BYTES[swz]
    return groups * 8 * s, 8 * s  # swizzle atoms along the row after all row groups


def image_size(words_shape, swz, lbo, sbo, off):
    rows, nw = words_shape
    hi = max(ocp.unit_address(r, u, swz, lbo, sbo, off) for r in range(rows)
             for u in range(nw // 4)) + 16
    return (hi + 1023) // 1024 * 1024


def roundtrip(words, *, swz, lanes, shape=tp.TPGEMM_CP_AUTO, variant=0, smem_offset=0,
              tmem_col=0, lane_offset=0, cta_group=1, seed=0, words2=None):
    rows, nw = words.shape
    lbo, sbo = layout(swz, rows, nw // 4, variant)
    nbytes = image_size(words.shape, swz, lbo, sbo, smem_offset)
    rng = np.random.default_rng(seed + 7)
    imgs = []
    for w in ([words] if cta_group == 1 else [words, words2]):
        bg = rng.integers(0, 256, nbytes, dtype=np.uint8)
        imgs.append(ocp.smem_image(w, swz, lbo, sbo, smem_offset, nbytes, bg))
    image = torch.from_numpy(np.concatenate(imgs)).cuda()
    ncols = max(32, (tmem_col + nw + 31) // 32 * 32)
    out = torch.empty(cta_group * 128 * ncols, dtype=torch.int32, device="cuda")
    fill = int(rng.integers(0, 2 ** 32))
    d = tp.cp_desc(rows, nw * 32, swizzle=swz, lbo=lbo, sbo=sbo, smem_offset=smem_offset,
                   tmem_col=tmem_col, lane_offset=lane_offset, lanes=lanes, shape=shape,
                   cta_group=cta_group)
    st = tp.tpgemm_cp_roundtrip(out, image, nbytes, d, fill, ncols)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK
    got = out.cpu().numpy().view(np.uint32).reshape(cta_group, 128, ncols)
    for k, w in enumerate([words] if cta_group == 1 else [words, words2]):
        exp = ocp.tmem_image(w, lanes, lane_offset, tmem_col, ncols, fill)
        bad = np.argwhere(got[k] != exp)
        assert bad.size == 0, (f"CTA {k}: {len(bad)} cells differ, first (lane, col) "
                               f"{bad[:4].tolist()}: got {got[k][tuple(bad[0])]:#x} "
                               f"expected {exp[tuple(bad[0])]:#x}")
    return got


def random_words(rows, nw, seed):
    return np.random.default_rng(seed).integers(0, 2 ** 32, (rows, nw), dtype=np.uint64).astype(
        np.uint32)


@pytest.mark.parametrize("middle", [1, 4])
@pytest.mark.parametrize("elem_bits", [16, 32], ids=["bf16", "f32"])
@pytest.mark.parametrize("swz", [ocp.SWIZZLE_NONE, ocp.SWIZZLE_32B, ocp.SWIZZLE_64B,
                                 ocp.SWIZZLE_128B], ids=["none", "sw32", "sw64", "sw128"])
@pytest.mark.parametrize("form", range(6), ids=FORM_IDS)
def test_cp_roundtrip_matrix(form, swz, elem_bits, middle):
    shape, lanes, rows, bits = FORMS[form]
    row_bits = bits * middle * (elem_bits // 16)
    words = random_words(rows, row_bits // 32, seed=100 * form + 10 * swz + middle + elem_bits)
    roundtrip(words, swz=swz, lanes=lanes, shape=shape, seed=form)


@pytest.mark.parametrize("form", range(6), ids=FORM_IDS)
def test_cp_inferred_matches_explicit(form):
    shape, lanes, rows, bits = FORMS[form]
    words = random_words(rows, 2 * bits // 32, seed=900 + form)
    a = roundtrip(words, swz=ocp.SWIZZLE_128B, lanes=lanes, shape=shape, seed=5)
    b = roundtrip(words, swz=ocp.SWIZZLE_128B, lanes=lanes, shape=tp.TPGEMM_CP_AUTO, seed=5)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("form", [0, 2, 5], ids=[FORM_IDS[0], FORM_IDS[2], FORM_IDS[5]])
def test_cp_unswizzled_other_lbo(form):
    # Unit columns of all row groups first: a non-trivial LBO between a row's
    # units, with 256-bit rows and several instructions along the row.
    shape, lanes, rows, bits = FORMS[form]
    words = random_words(rows, 4 * bits // 32, seed=950 + form)
    roundtrip(words, swz=ocp.SWIZZLE_NONE, lanes=lanes, shape=shape, variant=1)


@pytest.mark.parametrize("swz", [ocp.SWIZZLE_NONE, ocp.SWIZZLE_128B], ids=["none", "sw128"])
@pytest.mark.parametrize("form", [0, 3, 5], ids=[FORM_IDS[0], FORM_IDS[3], FORM_IDS[5]])
def test_cp_offsets(form, swz):
    # Region inside the staging buffer and a tensor-memory column offset.
    shape, lanes, rows, bits = FORMS[form]
    words = random_words(rows, 2 * bits // 32, seed=970 + form + swz)
    roundtrip(words, swz=swz, lanes=lanes, shape=shape, smem_offset=3072, tmem_col=36)


@pytest.mark.parametrize("swz", [ocp.SWIZZLE_NONE, ocp.SWIZZLE_64B], ids=["none", "sw64"])
def test_cp_4x256b_lane_tiled(swz):
    # 64 rows in quadrant order (16 instructions, lanes 32q + 0..15), then a
    # 32-row window landing on lanes 32q + 4..11.
    words = random_words(64, 16, seed=990)
    roundtrip(words, swz=swz, lanes=tp.TPGEMM_CP_LANES_QUADRANTS)
    words = random_words(32, 8, seed=991)
    roundtrip(words, swz=swz, lanes=tp.TPGEMM_CP_LANES_QUADRANTS, lane_offset=4)


@pytest.mark.parametrize("form", [0, 3], ids=[FORM_IDS[0], FORM_IDS[3]])
def test_cp_cta_group_2_pair(form):
    # The even CTA issues tcgen05.cp.cta_group::2 and a multicast commit; each
    # CTA's tensor memory receives its own shared memory's rows.
    shape, lanes, rows, bits = FORMS[form]
    w0 = random_words(rows, 2 * bits // 32, seed=995 + form)
    w1 = random_words(rows, 2 * bits // 32, seed=996 + form)
    roundtrip(w0, words2=w1, swz=ocp.SWIZZLE_128B, lanes=lanes, shape=shape, cta_group=2)


@pytest.mark.parametrize("issuers", [1, 2, 4, 8])
@pytest.mark.parametrize("form,cta_group", [(0, 1), (5, 1), (0, 2), (4, 2)],
                         ids=["128x256b", "32x128b_warpx4", "pair_128x256b", "pair_64x128b_01_23"])
def test_cp_repeat_many_ctas(form, cta_group, issuers):
    # Several CTAs (pairs) at once, each issuing its copy three times: every
    # CTA ends with the image of one copy.
    shape, lanes, rows, bits = FORMS[form]
    swz = ocp.SWIZZLE_128B
    words = [random_words(rows, 4 * bits // 32, seed=1000 + form + k) for k in range(cta_group)]
    nw = words[0].shape[1]
    lbo, sbo = layout(swz, rows, nw // 4)
    nbytes = image_size(words[0].shape, swz, lbo, sbo, 0)
    rng = np.random.default_rng(form)
    imgs = [ocp.smem_image(w, swz, lbo, sbo, 0, nbytes, rng.integers(0, 256, nbytes, dtype=np.uint8))
            for w in words]
    image = torch.from_numpy(np.concatenate(imgs)).cuda()
    ctas, ncols = 6 if cta_group == 2 else 5, 32 * ((nw + 31) // 32)
    out = torch.empty(ctas * 128 * ncols, dtype=torch.int32, device="cuda")
    d = tp.cp_desc(rows, nw * 32, swizzle=swz, lbo=lbo, sbo=sbo, lanes=lanes, shape=shape,
                   cta_group=cta_group)
    st = tp.tpgemm_cp_roundtrip_repeat(out, image, nbytes, d, 11, ncols, 3, ctas, issuers)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    assert tp.tpgemm_last_device_error() == tp.TPGEMM_OK
    got = out.cpu().numpy().view(np.uint32).reshape(ctas, 128, ncols)
    for k in range(ctas):
        exp = ocp.tmem_image(words[k % cta_group], lanes, 0, 0, ncols, 11)
        assert np.array_equal(got[k], exp), f"CTA {k}"


# ------------------------------------------- tensor memory <-> registers
from oracle import tmem_frag as ofr  # noqa: E402

LDST = [(a, b, c) for a in range(4) for b in range(4) for c in (2, 4, 8, 16)
        if c >= max({0: 1, 1: 2, 2: 4, 3: 8}[a], {0: 1, 1: 2, 2: 4, 3: 8}[b])]


@pytest.mark.parametrize("st,ld,cols", LDST,
                         ids=[f"st{ofr.NAMES[a]}-ld{ofr.NAMES[b]}-c{c}" for a, b, c in LDST])
def test_tmem_ldst_roundtrip(st, ld, cols):
    tmem_col = 8 if cols <= 16 and cols + 8 <= 32 else 0
    rng = np.random.default_rng(31 * st + 7 * ld + cols)
    regs = rng.integers(0, 2 ** 32, (128, cols), dtype=np.uint64).astype(np.uint32)
    fill = int(rng.integers(0, 2 ** 32))
    regs_d = torch.from_numpy(regs.view(np.int32)).cuda()
    regs_out = torch.empty(128 * cols, dtype=torch.int32, device="cuda")
    tmem_out = torch.empty(128 * 32, dtype=torch.int32, device="cuda")
    s = tp.tpgemm_tmem_ldst_roundtrip(regs_out, tmem_out, regs_d, st, ld, cols, tmem_col, fill)
    assert s == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    got_tmem = tmem_out.cpu().numpy().view(np.uint32).reshape(128, 32)
    got_regs = regs_out.cpu().numpy().view(np.uint32).reshape(128, cols)
    fill_img = ofr.fill_pattern(fill)
    # .32x32b, .16x128b and .16x256b: the oracle's map, pinned to the page's
    # demo and to the PTX ISA figure table, cell by cell.
    if st != ofr.S16x64b:
        exp_tmem = ofr.store(fill_img, regs, st, cols, tmem_col)
        bad = np.argwhere(got_tmem != exp_tmem)
        assert bad.size == 0, f"{len(bad)} cells differ, first {bad[:4].tolist()}"
    else:
        # .16x64b (thread map unpinned): outside the footprint nothing changes,
        # and each warp's 16-lane block holds exactly what the warp stored there.
        outside = np.ones((128, 32), bool)
        outside[:, tmem_col: tmem_col + cols] = False
        assert np.array_equal(got_tmem[outside], fill_img[outside])
        for w in range(4):
            for slab in range(2):
                lanes, _ = ofr.slab_cells(st, cols, slab)
                block = got_tmem[32 * w + lanes.start: 32 * w + lanes.stop,
                                 tmem_col: tmem_col + cols]
                r = ofr.slab_regs(st, cols, slab)
                stored = regs[32 * w: 32 * w + 32, r.start: r.stop]
                assert np.array_equal(np.sort(block, axis=None), np.sort(stored, axis=None))
    if ld != ofr.S16x64b:
        assert np.array_equal(got_regs, ofr.load(got_tmem, ld, cols, tmem_col))
    else:
        # each warp's registers of one issue are its 16-lane block, permuted
        for w in range(4):
            for slab in range(2):
                lanes, _ = ofr.slab_cells(ld, cols, slab)
                block = got_tmem[32 * w + lanes.start: 32 * w + lanes.stop,
                                 tmem_col: tmem_col + cols]
                r = ofr.slab_regs(ld, cols, slab)
                loaded = got_regs[32 * w: 32 * w + 32, r.start: r.stop]
                assert np.array_equal(np.sort(block, axis=None), np.sort(loaded, axis=None))
    if st == ld:
        assert np.array_equal(got_regs, regs)


def test_tmem_ldst_page_demo_128x8_fp16():
    # The page's demonstration: a warpgroup round-trips a 128 x 8 fp16 tile
    # through tensor memory with .32x32b.x4 both ways and gets it back exactly;
    # row r of the tile is lane r, fp16 pair c is column c.
    tile = torch.randn(128, 8).half()
    words = tile.view(torch.int32).contiguous()  # 128 x 4 words
    regs_out = torch.empty(128 * 4, dtype=torch.int32, device="cuda")
    tmem_out = torch.empty(128 * 32, dtype=torch.int32, device="cuda")
    s = tp.tpgemm_tmem_ldst_roundtrip(regs_out, tmem_out, words.cuda(), 0, 0, 4, 0, 0)
    assert s == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    back = regs_out.cpu().view(128, 4).view(torch.float16)
    assert torch.equal(back, tile)
    assert torch.equal(tmem_out.cpu().view(128, 32)[:, :4].contiguous().view(torch.float16), tile)
