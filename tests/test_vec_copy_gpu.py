"""The vectorised global <-> shared copy on the GPU: round trips (the page's TASKS
table: warp, warpgroup and CTA scopes x 1/2/4/8-byte elements), padded strides,
unaligned offsets (narrowed vectors), swizzled shared buffers, several CTAs;
the destination and the shared image compared byte for byte with the oracle."""
import numpy as np
import pytest
import torch

import tile_primitive_tensor_gb300 as tp
from oracle import vec_copy as ovc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    tp.library()


def run(rows, cols, eb, *, threads, g_row_stride=None, g_offset=0, s_row_stride=None,
        s_offset=0, swizzle=0, ctas=1, cta_stride=0, seed=0):
    gs = cols if g_row_stride is None else g_row_stride
    ss = cols if s_row_stride is None else s_row_stride
    d = tp.vcopy_desc(rows, cols, eb, g_row_stride=gs, g_offset=g_offset, s_row_stride=ss,
                      s_offset=s_offset, s_swizzle=swizzle, threads=threads)
    st, text = tp.tpgemm_vcopy_plan(d)
    assert st == tp.TPGEMM_OK, text
    smem_bytes = int(text.split("smem=")[1])
    span = (ctas - 1) * cta_stride + g_offset + (rows - 1) * gs + cols
    nbytes = (span * eb + 15) // 16 * 16
    rng = np.random.default_rng(seed)
    src = rng.integers(0, 256, nbytes, dtype=np.uint8)
    dst0 = rng.integers(0, 256, nbytes, dtype=np.uint8)
    src_d = torch.from_numpy(src).cuda()
    dst_d = torch.from_numpy(dst0).cuda()
    smem_d = torch.empty(ctas * smem_bytes, dtype=torch.uint8, device="cuda")
    st = tp.tpgemm_vcopy_roundtrip(dst_d, src_d, nbytes, d, ctas, cta_stride, smem_d)
    assert st == tp.TPGEMM_OK, tp.tpgemm_last_error_detail()
    torch.cuda.synchronize()
    dd = {"rows": rows, "cols": cols, "elem_bytes": eb, "g_row_stride": gs, "g_offset": g_offset,
          "s_row_stride": ss, "s_offset": s_offset, "s_swizzle": swizzle}
    assert np.array_equal(dst_d.cpu().numpy(), ovc.expected_dst(src, dst0, dd, ctas, cta_stride))
    sm = smem_d.cpu().numpy().reshape(ctas, smem_bytes)
    for k in range(ctas):
        assert np.array_equal(sm[k], ovc.expected_smem(src, dd, smem_bytes, k, cta_stride)), k
    return text


@pytest.mark.parametrize("threads", [1, 32, 128, 256])
@pytest.mark.parametrize("eb", [1, 2, 4, 8])
def test_vcopy_tasks_dense(threads, eb):
    text = run(32, 64, eb, threads=threads)
    # 128-bit transfers whenever each thread owns at least 16 bytes
    per_thread_bytes = 32 * 64 // threads * eb
    assert f"vec_bytes={min(16, per_thread_bytes)}" in text


@pytest.mark.parametrize("eb", [1, 2, 4])
@pytest.mark.parametrize("layout", ["padded", "offset", "odd", "col3"])
def test_vcopy_unaligned_layouts(eb, layout):
    kw = {"padded": dict(g_row_stride=72, s_row_stride=80),
          "offset": dict(g_row_stride=96, g_offset=8, s_offset=4),
          "odd": dict(g_row_stride=66, g_offset=2, s_row_stride=65),
          "col3": dict(g_row_stride=80, g_offset=3)}[layout]
    run(32, 64, eb, threads=128, **kw)


@pytest.mark.parametrize("swizzle", [1, 2, 3], ids=["sw32", "sw64", "sw128"])
@pytest.mark.parametrize("eb", [1, 2, 4])
def test_vcopy_swizzled_shared(swizzle, eb):
    run(32, 128 // eb * 2, eb, threads=128, swizzle=swizzle)


@pytest.mark.parametrize("eb", [2, 8])
def test_vcopy_cta_of_1024_threads(eb):
    run(64, 128, eb, threads=1024)


def test_vcopy_many_ctas():
    run(16, 64, 2, threads=128, ctas=5, cta_stride=16 * 80, g_row_stride=80)
