"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit for bit.

Every kernel path is forced in turn on seeded random layouts that span several
tiles and end in ragged tails, for every element width.  Destination buffers
carry canary bytes around and between the permuted elements: the oracle writes
into an identical canary buffer, so a byte written outside the image (or a byte
of the image left unwritten) fails the comparison.  Outputs are compared as raw
bytes, so NaN payloads count.
"""
import os

import numpy as np
import pytest

import movement_tl_permute_gb300 as tl
import oracle
from movement_tl_permute_gb300 import workloads
from oracle import layout_ref as L

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

MARGIN = 256          # canary bytes before the destination (keeps 256-byte alignment)
CANARY = 0xA5
NTHREADS = max(1, len(os.sched_getaffinity(0)))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from movement_tl_permute_gb300 import build
    build.build()
    oracle.build()
    tl.load()
    torch.cuda.init()


def _span(shape, strides):
    return sum((e - 1) * s for e, s in zip(shape, strides)) if all(e > 0 for e in shape) else -1


def run_case(shape, ss, ds, eb, path="auto", seed=0, src_off=0, dst_off=0, **opts):
    """Permute on the GPU and with the oracle; return (got, want) byte arrays."""
    n_src = (src_off + _span(shape, ss) + 1) * eb
    n_dst = MARGIN + (dst_off + _span(shape, ds) + 1) * eb + MARGIN
    src = workloads.random_bits(max(16, n_src), seed)
    want = np.full(n_dst, CANARY, dtype=np.uint8)
    oracle.permute(src, want, shape, ss, ds, eb, src_offset=src_off,
                   dst_offset=MARGIN // eb + dst_off, nthreads=NTHREADS)
    s_gpu = torch.from_numpy(src).cuda()
    d_gpu = torch.full((n_dst,), CANARY, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    tl.tl_permute_ex(s_gpu.data_ptr() + src_off * eb, d_gpu.data_ptr() + MARGIN + dst_off * eb,
                     shape, ss, ds, eb, stream, path=path, **opts)
    torch.cuda.synchronize()
    return d_gpu.cpu().numpy(), want


def check(shape, ss, ds, eb, path="auto", **kw):
    got, want = run_case(shape, ss, ds, eb, path, **kw)
    if not np.array_equal(got, want):
        bad = np.nonzero(got != want)[0]
        raise AssertionError("%d bytes differ (first at %d) for shape=%s ss=%s ds=%s eb=%d path=%s"
                             % (bad.size, bad[0], shape, ss, ds, eb, path))


def perm_layouts(shape, perm, pad=None):
    ss = L.row_major_strides(shape)
    pshape = tuple(shape[p] for p in perm)
    pst = L.row_major_strides(pshape)
    ds = [0] * len(shape)
    for i, p in enumerate(perm):
        ds[p] = pst[i]
    return ss, tuple(ds)


WIDTHS = [1, 2, 4, 8, 16]


# ---------------------------------------------------------------------------
# per-path parity on random small layouts
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("eb", WIDTHS)
def test_generic_path(eb):
    rng = np.random.default_rng(100 + eb)
    for i in range(12):
        nd = int(rng.integers(1, 6))
        shape = tuple(int(x) for x in rng.integers(1, 9, size=nd))
        perm = tuple(int(p) for p in rng.permutation(nd))
        ss, ds = perm_layouts(shape, perm)
        if i % 3 == 1:                          # padded source, offset views
            ss = tuple(s * 2 + (1 if j == 0 else 0) for j, s in enumerate(ss))
        check(shape, ss, ds, eb, "generic", seed=i, src_off=i % 3, dst_off=i % 2)


@pytest.mark.parametrize("eb", WIDTHS)
def test_generic_path_strided_views(eb):
    # strided views on one side, contiguous innermost on the other: the generic
    # kernel moves 16 bytes per step (gather into dst, or scatter from src) when the
    # contiguous side is 16-byte aligned, one element per step otherwise
    v = max(1, 16 // eb)
    for i, (shape, ss, ds) in enumerate((
            ((37, 8 * v), (2 * 8 * v * 2, 2), (8 * v, 1)),          # x[::2, ::2] -> contiguous
            ((37, 8 * v), (8 * v, 1), (2 * 8 * v, 2)),              # contiguous -> y[:, ::2]
            ((5, 3, 4 * v), (0, 4 * v * 3, 3), (12 * v, 4 * v, 1)),  # broadcast, stride-3 gather
            ((9, 2 * v), (1, 9 * 3), (2 * v, 1)))):                  # column gather, stride 27
        check(shape, ss, ds, eb, "generic", seed=110 + i)
        check(shape, ss, ds, eb, "generic", seed=120 + i, src_off=1, dst_off=1)


@pytest.mark.parametrize("eb", WIDTHS)
def test_chunk_path(eb):
    rng = np.random.default_rng(200 + eb)
    for i in range(10):
        inner = int(rng.choice([2, 3, 8, 16, 24, 64, 200]))
        outer = tuple(int(x) for x in rng.integers(1, 7, size=int(rng.integers(1, 4))))
        shape = outer + (inner,)
        perm = tuple(int(p) for p in rng.permutation(len(outer))) + (len(outer),)
        ss, ds = perm_layouts(shape, perm)
        check(shape, ss, ds, eb, "chunk", seed=i, src_off=i % 2)
    # one long contiguous run (a memcpy) and a large row count
    check((100003,), (1,), (1,), eb, "chunk", seed=11)
    check((37, 300, 16), (300 * 16, 16, 1), (16, 37 * 16, 1), eb, "chunk", seed=12)


def _tile_shapes(eb):
    out = []
    for rows, cols in ((300, 256), (128, 256), (1000, 64), (33, 1024), (257, 384)):
        c = max(16 // eb, cols // eb) if eb > 1 else cols
        c = (c + (16 // eb) - 1) // (16 // eb) * (16 // eb)      # src rows 16-byte aligned
        out.append(((rows, c), (c, 1), (1, rows)))
    # batched tiles and tiles inside a bigger batch structure
    a = max(16 // eb, 64 // eb)
    out.append(((5, 130, a), (130 * a, a, 1), (130 * a, 1, 130)))
    out.append(((3, 2, 70, 2 * a), (2 * 70 * 2 * a, 70 * 2 * a, 2 * a, 1),
                (2 * 70 * 2 * a, 70 * 2 * a, 1, 70)))
    return out


@pytest.mark.parametrize("eb", WIDTHS)
@pytest.mark.parametrize("path", ["tile", "cluster"])
def test_tile_and_cluster_paths(eb, path):
    for i, (shape, ss, ds) in enumerate(_tile_shapes(eb)):
        check(shape, ss, ds, eb, path, seed=i)


@pytest.mark.parametrize("eb", WIDTHS)
@pytest.mark.parametrize("stages", [2, 6])
def test_tile_path_256_row_tiles(eb, stages):
    # the taller tile variant: ragged bottom tiles whose second 128-row block is
    # partly or wholly outside the plane, batched planes, element-wise edges
    for i, (shape, ss, ds) in enumerate(_tile_shapes(eb)):
        check(shape, ss, ds, eb, "tile", seed=20 + i, tile_rows=256, tile_stages=stages)
    c = max(1, 256 // eb)
    check((33, c), (c, 1), (1, 33), eb, "tile", seed=5, dst_off=1, tile_rows=256)


@pytest.mark.parametrize("eb", WIDTHS)
@pytest.mark.parametrize("group", [1, 3])
def test_tile_path_visit_groups(eb, group):
    # tile rows visited in groups smaller than the b extent, the last one ragged
    for i, (shape, ss, ds) in enumerate(_tile_shapes(eb)):
        check(shape, ss, ds, eb, "tile", seed=40 + i, tile_group=group)
        check(shape, ss, ds, eb, "cluster", seed=50 + i, tile_group=group)


@pytest.mark.parametrize("eb", WIDTHS)
def test_tile_walk_across_grid_sizes(eb):
    # Each CTA walks its tiles by adding the grid size to the tile coordinates digit
    # by digit (tb, ta, three batch axes).  Grids of 1 .. more than the 72 tiles make
    # every digit carry, several digits at once, and the walk leave the range.
    a = 272 // eb                       # 3 tiles along a (the last one 16 bytes wide)
    shape = (3, 2, 2, 200, a)           # 2 tiles along b (the last 72 rows)
    ss, ds = perm_layouts(shape, (2, 1, 0, 4, 3))   # batch axes reversed: none merge
    for i, ctas in enumerate((1, 5, 7, 11, 24, 71, 72, 200)):
        check(shape, ss, ds, eb, "tile", seed=300 + i, max_ctas=ctas)
        check(shape, ss, ds, eb, "cluster", seed=310 + i, max_ctas=2 * ctas)
    # a batch axis between the plane's two axes in dst, and odd batch extents
    shape = (5, 3, 130, a)
    ss, ds = perm_layouts(shape, (1, 3, 0, 2))
    for i, ctas in enumerate((3, 13, 64)):
        check(shape, ss, ds, eb, "tile", seed=320 + i, max_ctas=ctas)


@pytest.mark.parametrize("eb", WIDTHS)
@pytest.mark.parametrize("staging,receive,warps", [(1, 1, 8), (3, 1, 8), (1, 3, 8), (4, 2, 8),
                                                   (8, 4, 8), (2, 1, 4), (2, 2, 4), (1, 3, 4)])
def test_cluster_ring_depths(eb, staging, receive, warps):
    # staging and receive rings of unequal depth (slot indices of the two sides
    # cycle with different periods), and four consumer warps taking two shares each
    for i, (shape, ss, ds) in enumerate(_tile_shapes(eb)):
        check(shape, ss, ds, eb, "cluster", seed=60 + i, tile_stages=staging,
              cluster_recv_stages=receive, cluster_consumer_warps=warps)


@pytest.mark.parametrize("eb", WIDTHS)
def test_tile_path_unaligned_dst_runs(eb):
    # dst columns of 33 rows: 16-byte runs straddle, the kernel stores element-wise
    c = max(1, 256 // eb)
    check((33, c), (c, 1), (1, 33), eb, "tile", seed=3)
    check((33, c), (c, 1), (1, 33), eb, "tile", seed=4, dst_off=1)


def _panel_cases(eb):
    out = []
    # odd row pitches with ragged tiles on both sides
    for rows, cols in ((300, 517), (33, 1001), (1001, 33), (129, 65), (2, 700), (700, 2)):
        out.append(((rows, cols), (cols, 1), (1, rows)))
    # interleaved channels <-> planes, 2..16 channels (even counts take rotated
    # word stores for 1- and 2-byte elements)
    for c in (2, 3, 4, 5, 16):
        out.append(((70, 90, c), (90 * c, c, 1), (90, 1, 70 * 90)))        # HWC -> CHW
        out.append(((c, 70, 90), (70 * 90, 90, 1), (1, 90 * c, c)))        # CHW -> HWC
    # more than three batch axes, with padded source strides
    shape = (3, 2, 4, 2, 40, 36)
    ss, ds = perm_layouts(shape, (5, 3, 1, 4, 2, 0))
    out.append((shape, ss, ds))
    ss2 = tuple(x * 2 for x in ss[:-1]) + (1,)
    out.append((shape, ss2, ds))
    # a short dst-contiguous axis walked together with the next dst axis; tile rows
    # cross the boundary between the two (7 and 5 do not divide the tile)
    for shape, perm in (((7, 5, 300), (2, 1, 0)), ((4,) * 7, (6, 5, 4, 3, 2, 1, 0)),
                        ((3, 9, 11, 130), (3, 2, 1, 0))):
        ss, ds = perm_layouts(shape, perm)
        out.append((shape, ss, ds))
    return out


@pytest.mark.parametrize("eb", WIDTHS)
@pytest.mark.parametrize("kib", [0, 4, 32])
def test_panel_path(eb, kib):
    for i, (shape, ss, ds) in enumerate(_panel_cases(eb)):
        check(shape, ss, ds, eb, "panel", seed=70 + i, panel_tile_kib=kib)
        check(shape, ss, ds, eb, "panel", seed=80 + i, src_off=1, dst_off=3, panel_tile_kib=kib)


def _panel_vec_cases(eb):
    v = 16 // eb
    out = []
    # odd src row pitch (rows misaligned in the stage), dst rows on 16-byte boundaries
    out.append(((272, 517), (517, 1), (1, 272)))
    # padded dst rows whose extent is no multiple of 16 bytes: the last block of each
    # dst row of a tile is partial
    out.append(((261, 517), (517, 1), (1, 272)))
    out.append(((40 * v + 3, 300), (300, 1), (1, 48 * v)))
    # more than three batch axes, aligned src rows, the short b merged with the next
    # dst axis (tile rows cross the merge boundary for 2-byte elements)
    shape = (min(4 * v, 32), 2, 4, 2, 40, 16 * v)
    ss, ds = perm_layouts(shape, (5, 3, 1, 4, 2, 0))
    out.append((shape, ss, ds))
    # packed src rows (interleaved channels -> planes; 1-byte rows keep word stores)
    c = {1: 3, 2: 6, 4: 3, 8: 3}[eb]
    out.append(((70, 96, c), (96 * c, c, 1), (96, 1, 70 * 96)))
    return out


@pytest.mark.parametrize("eb", [1, 2, 4, 8])
@pytest.mark.parametrize("kib", [0, 4])
def test_panel_vector_stores(eb, kib):
    """Tiles whose dst rows start on 16-byte boundaries are stored as 16-byte runs
    (read down a skewed stage); the same layouts with element stores, and with an
    unaligned dst, give the same bytes.  4-byte elements with src rows off the
    16-byte grid, and packed 1-byte rows, keep their element and word stores (the
    faster choice there)."""
    for i, (shape, ss, ds) in enumerate(_panel_vec_cases(eb)):
        plan = tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, eb, path="panel",
                          panel_tile_kib=kib)
        odd_rows = plan["panel_mode"] in (0, 2, 3) and any((x * eb) % 16 for x in ss if x != 1)
        keep = (eb == 4 and odd_rows) or (eb == 1 and plan["panel_mode"] == 1)
        assert plan["panel_vec"] == (0 if keep else 1), (shape, plan)
        off = tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, eb, path="panel",
                         panel_tile_kib=kib, flags=tl.TL_FLAG_PANEL_ELEMENT_STORES)
        assert off["panel_vec"] == 0
        check(shape, ss, ds, eb, "panel", seed=300 + i, panel_tile_kib=kib)
        check(shape, ss, ds, eb, "panel", seed=310 + i, src_off=1, panel_tile_kib=kib)
        check(shape, ss, ds, eb, "panel", seed=320 + i, panel_tile_kib=kib,
              flags=tl.TL_FLAG_PANEL_ELEMENT_STORES)
        check(shape, ss, ds, eb, "panel", seed=330 + i, dst_off=1, panel_tile_kib=kib)


def _skew_cases():
    """1-byte plane transposes whose dst rows sit at an odd pitch: every pitch residue
    modulo 16, ragged tiles on both sides, planes of exactly whole tiles and of the
    smallest size the walk takes, padded src rows, and batch items whose dst bases
    differ modulo 16 (a different column phase per item)."""
    out = []
    for i, delta in enumerate(range(1, 16, 2)):
        B, A = 300 + 37 * i, 270 + 53 * i             # b: dst-contiguous, a: src-contiguous
        Pd = B + ((-B - delta) % 16)                    # dst row pitch, -Pd = delta mod 16
        Ps = A + (i % 3) * 5
        out.append(((B, A), (Ps, 1), (1, Pd)))
    out.append(((512, 512), (512, 1), (1, 513)))
    out.append(((64, 64), (65, 1), (1, 67)))
    out.append(((1000, 700), (707, 1), (1, 1003)))
    out.append(((3, 130, 200), (200 * 131 + 7, 200, 1), (200 * 131 + 5, 1, 131)))
    return out


@pytest.mark.parametrize("kib", [0, 32])
@pytest.mark.parametrize("stages", [0, 1, 2])
def test_panel_skew_walk(kib, stages):
    """The skew walk (16-byte pieces of dst rows at an odd pitch, 256- and 128-column
    tiles, one or two stages per CTA) against the oracle, with aligned and unaligned
    bases; the same layouts with element stores forced take the word walk."""
    for i, (shape, ss, ds) in enumerate(_skew_cases()):
        for so, do in ((0, 0), (1, 0), (0, 7), (13, 5)):
            plan = tl.tl_plan((1 << 20) + so, (1 << 36) + do, shape, ss, ds, 1, path="panel",
                              panel_tile_kib=kib)
            assert plan["panel_vec"] == 4 and plan["tile_cols"] == (128 if kib else 256), plan
            check(shape, ss, ds, 1, "panel", seed=900 + 10 * i + so + do, src_off=so,
                  dst_off=do, panel_tile_kib=kib, tile_stages=stages)
        off = tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, 1, path="panel",
                         flags=tl.TL_FLAG_PANEL_ELEMENT_STORES)
        assert off["panel_vec"] != 4


@pytest.mark.parametrize("eb", [2, 4, 8])
def test_panel_tma_phase_maps(eb):
    """Block rows whose pitch is off the 16-byte grid, loaded by TMA phase maps (rows
    b = j mod phi as tensors of pitch phi * P, bases aligned down): ragged tiles on
    both sides, an unaligned base, a batch axis on the 16-byte grid; the same bytes as
    the oracle and as the cp.async copy (forced with the element-store flag)."""
    # dst rows off the 16-byte grid too (padded to an odd pitch), so that the tiles
    # store element by element, the store mode the phase layout serves
    cases = [((300, 517), (517, 1), (1, 301)),
             ((4, 150, 303), (45456, 303, 1), (45753, 1, 151)),
             ((150, 1001), (1001, 1), (1, 151))]
    for i, (shape, ss, ds) in enumerate(cases):
        for so in (0, 1):
            plan = tl.tl_plan((1 << 20) + so * eb, 1 << 36, shape, ss, ds, eb, path="panel")
            # (4- and 8-byte elements fill the same phase-major stage by cp.async: mode 3)
            assert plan["panel_mode"] == (2 if eb == 2 else 3), (shape, so, plan)
            off = tl.tl_plan((1 << 20) + so * eb, 1 << 36, shape, ss, ds, eb, path="panel",
                             flags=tl.TL_FLAG_PANEL_ELEMENT_STORES)
            assert off["panel_mode"] == 0
            check(shape, ss, ds, eb, "panel", seed=700 + 10 * i + so, src_off=so)
            check(shape, ss, ds, eb, "panel", seed=750 + 10 * i + so, src_off=so, dst_off=1)
            check(shape, ss, ds, eb, "panel", seed=780 + 10 * i + so, src_off=so,
                  flags=tl.TL_FLAG_PANEL_ELEMENT_STORES)


def _merged_a_cases():
    # high-rank permutes of short axes: the src-contiguous axis a (under 64 elements)
    # is merged with the next src axis, and the tile columns cross the boundary
    # between the two (7, 5, 9 and 6 do not divide the tile); the last case's src is
    # padded past the merged pair, which stays dense
    out = []
    for shape, perm in (((6,) * 7, (6, 5, 4, 3, 2, 1, 0)),
                        ((8,) * 6, (5, 4, 3, 2, 1, 0)),
                        ((5, 7, 9, 11, 13), (4, 3, 2, 1, 0)),
                        ((16, 3, 40, 7, 9), (1, 3, 0, 4, 2)),
                        ((3, 4, 5, 6, 7, 8), (5, 2, 4, 1, 3, 0))):
        ss, ds = perm_layouts(shape, perm)
        out.append((shape, ss, ds))
    shape = (9, 33, 5, 6)
    ss, ds = perm_layouts(shape, (3, 2, 1, 0))
    out.append((shape, (ss[0] * 2, ss[1] * 2, ss[2], ss[3]), ds))
    return out


@pytest.mark.parametrize("eb", WIDTHS)
def test_panel_merged_a(eb):
    """A short src-contiguous axis merged with the next src axis where the a x b
    plane is under 16 KiB: each tile row's dst offset splits a into its two axes.
    Vector, word and element stores, unaligned bases and small tiles give the
    oracle's bytes; planes past the bound stay unmerged and give the same bytes."""
    for i, (shape, ss, ds) in enumerate(_merged_a_cases()):
        plan = tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, eb, path="panel")
        a1 = shape[list(ss).index(1)]
        assert plan["path"] == "panel", (shape, plan)
        assert plan["panel_a1"] == a1 or (eb == 16 and plan["panel_a1"] == 0), (shape, plan)
        check(shape, ss, ds, eb, "panel", seed=900 + i)
        check(shape, ss, ds, eb, "panel", seed=910 + i, src_off=1, dst_off=3)
        check(shape, ss, ds, eb, "panel", seed=920 + i, panel_tile_kib=4)
        check(shape, ss, ds, eb, "panel", seed=930 + i,
              flags=tl.TL_FLAG_PANEL_ELEMENT_STORES)


@pytest.mark.parametrize("eb", [1, 2, 4])
def test_panel_run_stores(eb):
    """Planes -> interleaved channels: a tile's dst is one run, stored as 16-byte
    pieces (store mode 2) with single elements before the first and after the last
    16-byte boundary; the element and word stores give the same bytes."""
    for i, c in enumerate((2, 3, 4, 7, 16)):
        shape, ss, ds = (c, 70, 90), (70 * 90, 90, 1), (1, 90 * c, c)
        plan = tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, eb, path="panel")
        # (16-byte runs along the tile rows take precedence where they apply)
        want = 1 if (c * eb) % 128 == 0 else 2
        assert plan["panel_vec"] == want and plan["vec_bytes"] == 16, (c, plan)
        off = tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, eb, path="panel",
                         flags=tl.TL_FLAG_PANEL_ELEMENT_STORES)
        assert off["panel_vec"] == 0
        for j, (so, do) in enumerate(((0, 0), (1, 0), (0, 1), (3, 5))):
            check(shape, ss, ds, eb, "panel", seed=400 + 10 * i + j, src_off=so, dst_off=do)
        check(shape, ss, ds, eb, "panel", seed=450 + i, flags=tl.TL_FLAG_PANEL_ELEMENT_STORES)
        check(shape, ss, ds, eb, "panel", seed=460 + i, panel_tile_kib=4)


@pytest.mark.parametrize("eb", WIDTHS)
def test_auto_takes_panel_for_untiled_planes(eb):
    # 3-channel interleaves go to the panel kernel (or to the rows / cols register
    # transposes where whole 16-byte pieces allow)
    for shape, ss, ds in ((( 64, 96, 3), (96 * 3, 3, 1), (96, 1, 64 * 96)),
                          ((3, 64, 96), (64 * 96, 96, 1), (1, 96 * 3, 3))):
        assert tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, eb)["path"] in ("panel", "rows", "cols")
        check(shape, ss, ds, eb, "auto", seed=90)


@pytest.mark.parametrize("eb", [1, 2, 4, 8])
def test_cols_path(eb):
    """Interleaved channels -> planes with whole 16-byte plane pieces: the cols kernel
    (pixel loads, register transpose, one store per plane), with batch axes, padded
    planes and offset views; a plane extent off the 16-byte grid goes to the panel
    kernel instead."""
    n = 16 // eb
    for i, c in enumerate(range(2, min(16, 24 // eb) + 1)):
        H, W = 3, 5 * n
        for j, (shape, ss, ds) in enumerate((
                ((H, W, c), (W * c, c, 1), (W, 1, H * W)),                      # HWC -> CHW
                ((2, H, W, c), (H * W * c, W * c, c, 1), (c * H * W, W, 1, H * W)),  # NHWC -> NCHW
                ((H, W, c), (W * c, c, 1), (W, 1, H * W + 2 * n)))):            # padded planes
            assert tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, eb)["path"] == "cols", (shape, c)
            check(shape, ss, ds, eb, "auto", seed=600 + 10 * i + j)
            check(shape, ss, ds, eb, "cols", seed=650 + 10 * i + j, src_off=n, dst_off=2 * n)
        # a plane extent that is not a whole number of pieces
        shape, ss, ds = (H, W + 1, c), ((W + 1) * c, c, 1), (W + 1, 1, H * (W + 1))
        assert tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, eb)["path"] != "cols"
        check(shape, ss, ds, eb, "auto", seed=690 + i)


@pytest.mark.parametrize("eb,R", [(1, 2), (1, 3), (1, 4), (1, 5), (1, 6), (1, 7), (1, 8), (1, 9),
                                  (1, 10), (1, 11), (1, 12), (1, 13), (1, 14), (1, 15), (1, 16),
                                  (2, 2), (2, 3), (2, 4), (2, 5), (2, 6), (2, 7), (2, 8),
                                  (4, 2), (4, 3), (4, 4), (8, 2)])
def test_rows_path(eb, R):
    A = 3 * 16 // eb * 2            # whole 16-byte pieces per row, several units
    for i, batch in enumerate([(1,), (7,), (3, 5)]):
        shape = batch + (R, A)
        ss = L.row_major_strides(shape)
        dss = L.row_major_strides(batch + (A, R))
        ds = dss[:len(batch)] + (1, R)
        check(shape, ss, ds, eb, "rows", seed=i)


WARP_CASES = [((4, 32), (32, 1), (1, 4)), ((8, 16), (16, 1), (1, 8)), ((2, 64), (64, 1), (1, 2)),
              ((4, 8, 4), (32, 4, 1), (1, 16, 4)), ((32,), (1,), (1,)), ((16, 16), (16, 1), (1, 16))]


@pytest.mark.parametrize("eb", WIDTHS)
def test_warp_path(eb):
    ran = 0
    for i, (ext, ss, ds) in enumerate(WARP_CASES):
        for batch in (1, 5):
            n = int(np.prod(ext))
            shape = (batch,) + ext
            try:
                tl.tl_plan(1 << 20, 1 << 30, shape, (n,) + ss, (n,) + ds, eb, path="warp")
            except tl.TLError as e:
                assert e.name == "TL_ERR_PATH"
                continue
            check(shape, (n,) + ss, (n,) + ds, eb, "warp", seed=i)
            ran += 1
    assert ran > 0


def test_auto_paths_on_random_layouts():
    rng = np.random.default_rng(7)
    seen = set()
    for i in range(40):
        eb = int(rng.choice(WIDTHS))
        nd = int(rng.integers(1, 5))
        shape = tuple(int(x) for x in rng.integers(1, 40, size=nd))
        perm = tuple(int(p) for p in rng.permutation(nd))
        ss, ds = perm_layouts(shape, perm)
        seen.add(tl.tl_plan(1 << 20, 1 << 34, shape, ss, ds, eb)["path"])
        check(shape, ss, ds, eb, "auto", seed=i)
    assert {"chunk", "panel"} <= seen, seen


# ---------------------------------------------------------------------------
# block path: high-rank permutes of short axes
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("eb", WIDTHS)
def test_block_path_random_high_rank_permutes(eb):
    """The block tile (up to four axes, a few long runs on both sides) forced on
    random permutes of 3-7 short axes: chunked axes with ragged last chunks, batch
    axes outside the tile, unaligned src and dst bases."""
    rng = np.random.default_rng(400 + eb)
    done = 0
    for i in range(40):
        nd = int(rng.integers(3, 8))
        shape = tuple(int(x) for x in rng.integers(2, 10, size=nd))
        if int(np.prod(shape)) * eb > (64 << 20):
            continue
        perm = tuple(int(p) for p in rng.permutation(nd))
        ss, ds = perm_layouts(shape, perm)
        try:
            tl.tl_plan(1 << 32, 1 << 44, shape, ss, ds, eb, path="block")
        except tl.TLError:
            continue                                  # no block tile for this layout
        check(shape, ss, ds, eb, "block", seed=400 + i, src_off=i % 3, dst_off=(i // 3) % 2)
        done += 1
    assert done >= 20


@pytest.mark.parametrize("eb", WIDTHS)
def test_block_path_named_layouts(eb):
    """Permutes the planner gives the block tile: the interleaved order of 12^k and a
    permute of 9^k whose src and dst share two middle axes, at sizes of a few MiB."""
    for i, (shape, perm) in enumerate((((12,) * 5, (4, 2, 0, 1, 3)),
                                       ((9,) * 6, (1, 4, 2, 3, 5, 0)),
                                       ((7, 9, 5, 11, 6), (3, 0, 4, 2, 1)))):
        ss, ds = perm_layouts(shape, perm)
        check(shape, ss, ds, eb, "block", seed=450 + i)
        check(shape, ss, ds, eb, "auto", seed=460 + i, src_off=1, dst_off=1)


@pytest.mark.parametrize("eb", WIDTHS)
def test_block_store_walks(eb):
    """Both store walks of the block kernel -- consecutive pieces in dst order, and
    groups of pieces across 2-32 dst runs -- with pieces of several elements stored as
    one vector (aligned dst) and of one element (dst one element off), on layouts whose
    bank costs pick each."""
    layouts = (((12,) * 5, (4, 2, 0, 1, 3)), ((12,) * 6, (5, 3, 1, 0, 2, 4)),
               ((8,) * 6, (5, 4, 3, 2, 1, 0)), ((16,) * 5, (4, 3, 2, 1, 0)),
               ((7, 9, 5, 11, 6), (3, 0, 4, 2, 1)))
    runs, vecs = set(), set()
    for i, (shape, perm) in enumerate(layouts):
        ss, ds = perm_layouts(shape, perm)
        plan = tl.tl_plan(1 << 32, 1 << 44, shape, ss, ds, eb, path="block")
        runs.add(plan["block_runs"])
        vecs.add(plan["vec_bytes"])
        check(shape, ss, ds, eb, "block", seed=470 + i)
        check(shape, ss, ds, eb, "block", seed=480 + i, dst_off=1)
    assert 1 in runs and max(runs) > 1, runs
    assert 16 in vecs, vecs


@pytest.mark.parametrize("eb", [1, 4])
def test_block_consumer_warp_counts(eb):
    """The block kernel with 1, 3 and 17 consumer warps, and at one CTA per SM: the same
    bytes as the oracle (the walks' step over the consumer threads changes with the
    count)."""
    for i, (shape, perm) in enumerate((((12,) * 5, (4, 2, 0, 1, 3)),
                                       ((9,) * 6, (1, 4, 2, 3, 5, 0)))):
        ss, ds = perm_layouts(shape, perm)
        for k, kw in enumerate((dict(cluster_consumer_warps=1), dict(cluster_consumer_warps=3),
                                dict(cluster_consumer_warps=17),
                                dict(tile_ctas_per_sm=1, cluster_consumer_warps=17))):
            check(shape, ss, ds, eb, "block", seed=490 + 10 * i + k, dst_off=k % 2, **kw)


def test_per_cta_times_are_recorded_without_changing_the_result():
    """The measurement option: the tile, rows, panel and block kernels write each
    CTA's start and finish time, every CTA of the grid tl_plan reports once, and the
    permute is the same."""
    cases = [((300, 520), (520, 1), (1, 300), 4, "tile"),
             ((1024, 2, 4, 32), (256, 128, 32, 1), (256, 128, 1, 4), 1, "rows"),
             ((301, 517), (517, 1), (1, 301), 4, "panel"),
             ((12,) * 5, None, None, 2, "block")]
    for i, (shape, ss, ds, eb, path) in enumerate(cases):
        if ss is None:
            ss, ds = perm_layouts(shape, (4, 2, 0, 1, 3))
        grid = tl.tl_plan(1 << 32, 1 << 44, shape, ss, ds, eb, path=path)["grid"]
        times = torch.zeros(2 * grid, dtype=torch.int64, device="cuda")
        check(shape, ss, ds, eb, path, seed=500 + i, cta_times=times.data_ptr())
        t = times.cpu().numpy().reshape(grid, 2)
        assert (t[:, 0] > 0).all() and (t[:, 1] >= t[:, 0]).all(), path
        assert t[:, 1].max() - t[:, 0].min() < 10**9, path       # within a second


# ---------------------------------------------------------------------------
# fused permute + cast
# ---------------------------------------------------------------------------
CAST_WIDTHS = {"f32_to_bf16": (4, 2), "f32_to_f16": (4, 2), "bf16_to_f32": (2, 4),
               "f16_to_f32": (2, 4)}


def check_cast(shape, ss, ds, cast, path="auto", seed=0, src_off=0, dst_off=0):
    """The converting permute on the GPU against oracle.permute_cast, canaries around
    and between the destination's elements."""
    seb, deb = CAST_WIDTHS[cast]
    n_src = (src_off + _span(shape, ss) + 1) * seb
    n_dst = MARGIN + (dst_off + _span(shape, ds) + 1) * deb + MARGIN
    src = workloads.random_bits(max(16, n_src), seed)
    want = np.full(n_dst, CANARY, dtype=np.uint8)
    oracle.permute_cast(src, want, shape, ss, ds, cast, src_offset=src_off,
                        dst_offset=MARGIN // deb + dst_off)
    s_gpu = torch.from_numpy(src).cuda()
    d_gpu = torch.full((n_dst,), CANARY, dtype=torch.uint8, device="cuda")
    tl.tl_permute_ex(s_gpu.data_ptr() + src_off * seb, d_gpu.data_ptr() + MARGIN + dst_off * deb,
                     shape, ss, ds, seb, torch.cuda.current_stream().cuda_stream, path=path,
                     cast=cast)
    torch.cuda.synchronize()
    got = d_gpu.cpu().numpy()
    if not np.array_equal(got, want):
        bad = np.nonzero(got != want)[0]
        raise AssertionError("%d bytes differ (first at %d) for %s shape=%s path=%s"
                             % (bad.size, bad[0], cast, shape, path))


@pytest.mark.parametrize("cast", sorted(CAST_WIDTHS))
def test_cast_on_the_tile_path(cast):
    """Converting 2-D and batched transposes on the TMA tile kernel: random bits
    (NaN and infinity patterns included), ragged tiles, element-wise edges."""
    seb, _ = CAST_WIDTHS[cast]
    a = 128 // seb
    for i, (shape, ss, ds) in enumerate((((300, 2 * a), (2 * a, 1), (1, 300)),
                                         ((128, 3 * a), (3 * a, 1), (1, 128)),
                                         ((33, a + a // 2 if seb == 4 else 2 * a), None, None),
                                         ((5, 130, a), (130 * a, a, 1), (130 * a, 1, 130)))):
        if ss is None:
            ss, ds = (shape[1], 1), (1, shape[0])
        check_cast(shape, ss, ds, cast, "tile", seed=600 + i)
        check_cast(shape, ss, ds, cast, "auto", seed=610 + i)
    # dst rows off the 16-byte grid: the element-wise stores
    check_cast((37, 2 * a), (2 * a, 1), (1, 37), cast, "tile", seed=620, dst_off=1)


@pytest.mark.parametrize("cast", sorted(CAST_WIDTHS))
def test_cast_on_the_chunk_and_generic_paths(cast):
    """Converting permutes whose innermost axis is contiguous on both sides (chunk
    kernel, vectors of 4, 2 and 1 elements) and strided layouts (generic kernel)."""
    rng = np.random.default_rng(630)
    for i in range(8):
        inner = int(rng.choice([4, 8, 12, 64, 130]))
        outer = tuple(int(x) for x in rng.integers(1, 7, size=int(rng.integers(1, 4))))
        shape = outer + (inner,)
        perm = tuple(int(p) for p in rng.permutation(len(outer))) + (len(outer),)
        ss, ds = perm_layouts(shape, perm)
        off = (0, 1, 2)[i % 3]
        check_cast(shape, ss, ds, cast, "chunk", seed=640 + i, src_off=off, dst_off=(i // 3) % 2)
        check_cast(shape, ss, ds, cast, "generic", seed=650 + i, src_off=off)
    # a strided gather and a broadcast on the generic kernel
    check_cast((9, 14), (2, 37), (14, 1), cast, "generic", seed=660)
    check_cast((4, 6, 5), (0, 5, 1), (30, 5, 1), cast, "generic", seed=661)
    # paths that move bits only decline a cast
    with pytest.raises(tl.TLError) as e:
        check_cast((64, 256), (256, 1), (1, 64), cast, "panel", seed=662)
    assert e.value.name == "TL_ERR_PATH"


@pytest.mark.parametrize("cast", sorted(CAST_WIDTHS))
def test_cast_on_the_block_path(cast):
    """Converting high-rank permutes of short axes on the block kernel: vector and
    single-element dst pieces, both store walks, chunked tiles, unaligned bases, and the
    planner's own choice of the block tile for a layout no other converting kernel
    takes as a whole."""
    layouts = (((12,) * 5, (4, 2, 0, 1, 3)), ((9,) * 6, (1, 4, 2, 3, 5, 0)),
               ((7, 9, 5, 11, 6), (3, 0, 4, 2, 1)), ((8,) * 6, (5, 4, 3, 2, 1, 0)))
    for i, (shape, perm) in enumerate(layouts):
        ss, ds = perm_layouts(shape, perm)
        check_cast(shape, ss, ds, cast, "block", seed=670 + i)
        check_cast(shape, ss, ds, cast, "block", seed=680 + i, src_off=1, dst_off=(i % 2))
    shape, perm = (9,) * 6, (1, 4, 2, 3, 5, 0)
    ss, ds = perm_layouts(shape, perm)
    seb, _ = CAST_WIDTHS[cast]
    assert tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, seb, cast=cast)["path"] == "block"
    check_cast(shape, ss, ds, cast, "auto", seed=690)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------
def test_tensor_level_permute_matches_torch():
    """An attention-style (B, H, S, D) -> (B, S, H, D) bfloat16 permute at a small
    size, through tl.permute on torch CUDA tensors, equals torch's own
    transpose, and the planner names the chunk path; an fp32 2-D transpose into a
    transposed view equals .t()."""
    x = torch.randn(2, 8, 256, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(2, 256, 8, 128, dtype=torch.bfloat16, device="cuda")
    ds = (y.stride(0), y.stride(2), y.stride(1), y.stride(3))
    tl.permute(x, y, x.shape, x.stride(), ds)
    torch.cuda.synchronize()
    assert torch.equal(y, x.transpose(1, 2))
    assert tl.tl_plan(x.data_ptr(), y.data_ptr(), x.shape, x.stride(), ds, 2)["path"] == "chunk"
    a = torch.randn(300, 520, device="cuda")
    b = torch.empty(520, 300, device="cuda")
    tl.permute(a, b, a.shape, a.stride(), (1, 300))
    torch.cuda.synchronize()
    assert torch.equal(b, a.t())


@pytest.mark.parametrize("eb", [1, 4, 16])
def test_checked_run(eb):
    """TL_FLAG_DEBUG_CHECKS: a valid layout gives the oracle's bytes and a clean
    status; with the host check skipped and dst declared half its real size, the
    device check skips every element past the declared bytes (which stay canary),
    writes the rest exactly, and records TL_ERR_BOUNDS.  The real buffer covers the
    whole layout, so no access could leave the allocation even if a check failed."""
    shape, ss, ds = (64, 48), (48, 1), (1, 64)
    check(shape, ss, ds, eb, "auto", seed=7, flags=tl.TL_FLAG_DEBUG_CHECKS,
          src_bytes=64 * 48 * eb, dst_bytes=64 * 48 * eb)
    src = workloads.random_bits(64 * 48 * eb, 8)
    want = np.full(64 * 48 * eb, CANARY, dtype=np.uint8)
    oracle.permute(src, want, shape, ss, ds, eb)
    declared = 64 * 48 * eb // 2
    want[declared:] = CANARY                           # skipped by the device check
    s_gpu = torch.from_numpy(src).cuda()
    d_gpu = torch.full((64 * 48 * eb,), CANARY, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tl.tl_permute_ex(s_gpu.data_ptr(), d_gpu.data_ptr(), shape, ss, ds, eb,
                     torch.cuda.current_stream().cuda_stream,
                     flags=tl.TL_FLAG_DEBUG_CHECKS | tl.TL_FLAG_TEST_SKIP_HOST_BOUNDS,
                     dev_status=status.data_ptr(), src_bytes=64 * 48 * eb, dst_bytes=declared)
    torch.cuda.synchronize()
    assert int(status.item()) == {v: k for k, v in tl.STATUS.items()}["TL_ERR_BOUNDS"]
    assert np.array_equal(d_gpu.cpu().numpy(), want)


def test_edge_cases():
    check((), (), (), 4)                                         # one element
    check((1, 1, 1), (7, 3, 1), (1, 1, 1), 16)
    check((2,) * 8, L.row_major_strides((2,) * 8),
          tuple(reversed(L.row_major_strides((2,) * 8))), 2)    # 8 dims, full reversal
    check((5, 7), (0, 1), (7, 1), 4, "generic")                  # broadcast source rows
    check((5, 7), (0, 1), (7, 1), 4)
    check((3, 4, 5), (1, 3, 12), (20, 5, 1), 1, seed=5)          # column-major -> row-major
    check((64, 96), (96, 1), (1, 64 + 3), 8, "auto")            # padded destination columns
    check((17, 3), (3, 1), (1, 17), 1, "generic", src_off=1, dst_off=3)   # odd byte offsets
    # empty shapes are no-ops (no launch)
    before = tl.tl_launch_count()
    d = torch.full((64,), CANARY, dtype=torch.uint8, device="cuda")
    tl.tl_permute(d.data_ptr(), d.data_ptr() + 32, (0, 4), (4, 1), (1, 0), 1)
    assert tl.tl_launch_count() == before
    assert bool((d == CANARY).all())


def test_in_place_warp_permute():
    w = workloads.get("sf_transpose")
    src = workloads.make_input(w)
    want = np.zeros_like(src)
    oracle.permute(src, want, w.shape, w.src_strides, w.dst_strides, 4)
    buf = torch.from_numpy(src.copy()).cuda()
    tl.tl_permute(buf.data_ptr(), buf.data_ptr(), w.shape, w.src_strides, w.dst_strides, 4,
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(buf.cpu().numpy(), want)


def test_errors_launch_nothing():
    a = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    before = tl.tl_launch_count()
    with pytest.raises(tl.TLError) as e:
        tl.tl_permute(a.data_ptr(), a.data_ptr() + 64, (16, 16), (16, 1), (1, 16), 4)
    assert e.value.name == "TL_ERR_ALIAS"
    with pytest.raises(tl.TLError) as e:
        tl.permute(a[:1024], a[3072:], (16, 16), (16, 1), (1, 16), elem_bytes=8)
    assert e.value.name == "TL_ERR_BOUNDS"
    assert tl.tl_launch_count() == before


def test_cluster_handoff_timeout_is_reported_and_context_survives():
    shape, ss, ds = (16, 128, 64), (8192, 64, 1), (8192, 1, 128)
    src = torch.zeros(16 * 8192, dtype=torch.float16, device="cuda")
    dst = torch.zeros_like(src)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tl.permute(src, dst, shape, ss, ds, path="cluster", flags=tl.TL_FLAG_TEST_DROP_HANDOFF,
               dev_status=status.data_ptr())
    torch.cuda.synchronize()
    assert int(status.item()) == -12          # TL_ERR_TIMEOUT
    # the context is still usable and the same call without the hook is correct
    check(shape, ss, ds, 2, "cluster", seed=9)
    status.zero_()
    check(shape, ss, ds, 2, "tile", seed=9, dev_status=status.data_ptr())
    assert int(status.item()) == 0


def test_panel_tma_timeout_is_reported_and_context_survives():
    """A panel tile loaded by TMA phase maps whose load never lands (the test hook
    skips one phase load): every thread's bounded wait expires together, the status
    word reads TL_ERR_TIMEOUT, and the context still runs the same permute correctly."""
    R, C, ds_a = 300, 517, 301
    shape, ss, ds = (R, C), (C, 1), (1, ds_a)
    assert tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, 2, path="panel")["panel_mode"] == 2
    src = torch.zeros(R * C, dtype=torch.int16, device="cuda")
    dst = torch.zeros(C * ds_a, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tl.permute(src, dst, shape, ss, ds, path="panel", flags=tl.TL_FLAG_TEST_DROP_HANDOFF,
               dev_status=status.data_ptr())
    torch.cuda.synchronize()
    assert int(status.item()) == -12          # TL_ERR_TIMEOUT
    status.zero_()
    check(shape, ss, ds, 2, "panel", seed=19, dev_status=status.data_ptr())
    assert int(status.item()) == 0


def test_block_copy_timeout_is_reported_and_context_survives():
    """A block tile whose src-run copy never lands (the test hook skips the first
    copy of each CTA's first tile): the consumers' bounded waits expire, the status
    word reads TL_ERR_TIMEOUT, and the context still runs the same permute correctly."""
    # one pipeline per CTA (12^5 u16), and two in one CTA (9^6 fp32, 576 threads)
    for shape, perm, dtype, eb in (((12,) * 5, (4, 2, 0, 1, 3), torch.int16, 2),
                                   ((9,) * 6, (1, 4, 2, 3, 5, 0), torch.int32, 4)):
        ss, ds = perm_layouts(shape, perm)
        plan = tl.tl_plan(1 << 20, 1 << 36, shape, ss, ds, eb, path="block")
        assert plan["path"] == "block"
        n = int(np.prod(shape))
        src = torch.zeros(n, dtype=dtype, device="cuda")
        dst = torch.zeros(n, dtype=dtype, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        tl.permute(src, dst, shape, ss, ds, path="block", flags=tl.TL_FLAG_TEST_DROP_HANDOFF,
                   dev_status=status.data_ptr())
        torch.cuda.synchronize()
        assert int(status.item()) == -12          # TL_ERR_TIMEOUT
        status.zero_()
        check(shape, ss, ds, eb, "block", seed=23, dev_status=status.data_ptr())
        assert int(status.item()) == 0


# ---------------------------------------------------------------------------
# every bench workload at full size, in the launch configuration the bench times
# ---------------------------------------------------------------------------
FULL = ["sf_transpose", "tile_transpose", "mx_sf", "attention", "t2d_u8", "t2d_f16", "t2d_f32",
        "t2d_f64", "t2d_v16", "t2d_odd_f32", "t2d_odd_u8", "hwc_chw_u8", "nd6_f32", "nd8_f32", "nd8_u16"]


def _full(name, path="auto"):
    w = workloads.get(name)
    src = workloads.make_input(w)
    want = np.empty(w.dst_elems * w.elem_bytes, dtype=np.uint8)
    oracle.permute(src, want, w.shape, w.src_strides, w.dst_strides, w.elem_bytes,
                   nthreads=NTHREADS)
    s_gpu = torch.from_numpy(src).cuda()
    del src
    d_gpu = torch.empty(w.dst_elems * w.elem_bytes, dtype=torch.uint8, device="cuda")
    tl.tl_permute_ex(s_gpu.data_ptr(), d_gpu.data_ptr(), w.shape, w.src_strides,
                     w.dst_strides, w.elem_bytes, torch.cuda.current_stream().cuda_stream,
                     path=path)
    torch.cuda.synchronize()
    got = d_gpu.cpu().numpy()
    del s_gpu, d_gpu
    assert np.array_equal(got, want), name


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    _full(name)


def test_full_size_tile_transpose_through_the_cluster_handoff():
    _full("tile_transpose", "cluster")
