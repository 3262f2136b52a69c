"""Host-side logic of the C ABI, on CPU: no kernel is launched here.

The library must load on a machine without a GPU, export every function that
include/tl_permute.h declares, and its host entry points (canonicalisation, the
bank simulator and XOR chooser, validation and planning) must agree with the
oracle's independent Python references.
"""
import os
import re

import numpy as np
import pytest

import movement_tl_permute_gb300 as tl
from movement_tl_permute_gb300 import workloads
from oracle import layout_ref as L
from tests.conftest import ROOT

SRC = 0x10000000      # fake, 4 KiB-aligned device addresses: tl_plan never dereferences
DST = 0x90000000


@pytest.fixture(scope="module", autouse=True)
def _built():
    from movement_tl_permute_gb300 import build
    build.build()
    tl.load()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "tl_permute.h")) as f:
        text = f.read()
    return re.findall(r"TL_API\s+[\w\s\*]+?\b(tl_\w+)\s*\(", text)


def test_library_loads_and_exports_every_declared_symbol():
    names = _declared_functions()
    assert set(names) >= {"tl_layout_canon", "tl_choose_xor_k", "tl_permute", "tl_permute_ex",
                          "tl_plan", "tl_status_string", "tl_launch_count", "tl_version",
                          "tl_bank_conflicts"}
    lib = tl.load()
    for n in names:
        assert hasattr(lib, n), n
    assert tl.tl_version() == 2
    assert tl.tl_status_string(0) == "ok"
    assert "alias" in tl.tl_status_string(-7) or "overlap" in tl.tl_status_string(-7)


def test_plain_c_client(tmp_path):
    """A C99 program that includes only the public header and links only the
    library (tests/c/abi_client.c) runs the host entry points on the pages'
    worked examples."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    libdir = os.path.dirname(os.path.abspath(tl.load()._name))
    exe = str(tmp_path / "abi_client")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(root, "include"), os.path.join(here, "c", "abi_client.c"),
                    "-L", libdir, "-ltl_permute", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failure(s)" in r.stdout


# ---------------------------------------------------------------------------
# canonicalisation vs the oracle reference
# ---------------------------------------------------------------------------
def _rand_layout_pair(rng):
    nd = int(rng.integers(1, 6))
    shape = tuple(int(x) for x in rng.integers(1, 5, size=nd))
    perm = list(rng.permutation(nd))
    ss = L.row_major_strides(shape)
    pst = L.row_major_strides(tuple(shape[p] for p in perm))
    ds = [0] * nd
    for i, p in enumerate(perm):
        ds[p] = pst[i]
    if rng.random() < 0.3:          # padded strides break some merges
        ss = tuple(s * int(rng.integers(1, 3)) for s in ss)
    return shape, tuple(ss), tuple(ds)


def test_canon_matches_reference():
    rng = np.random.default_rng(1)
    for _ in range(400):
        shape, ss, ds = _rand_layout_pair(rng)
        begin = extent = None
        if rng.random() < 0.5:
            begin = tuple(int(rng.integers(0, e)) for e in shape)
            extent = tuple(int(rng.integers(0, e - b + 1)) for e, b in zip(shape, begin))
        so, do = int(rng.integers(0, 9)), int(rng.integers(0, 9))
        got = tl.tl_layout_canon(shape, ss, ds, begin, extent, so, do)
        want = L.canon_ref(shape, ss, ds, begin, extent, so, do)
        assert got == want, (shape, ss, ds, begin, extent)


def test_canon_worked_examples():
    c = tl.tl_layout_canon((2, 1, 4, 32), (128, 128, 32, 1), (128, 128, 1, 4),
                           begin=(1, 0, 0, 0), extent=(1, 1, 4, 32))
    assert c["extent"] == (4, 32) and c["src_str"] == (32, 1) and c["dst_str"] == (1, 4)
    assert c["src_offset"] == 128 and c["chunk_elems"] == 0
    c = tl.tl_layout_canon((128, 64), (64, 1), (64, 1))
    assert c["extent"] == (8192,) and c["chunk_elems"] * 2 == 16384
    with pytest.raises(tl.TLError) as e:
        tl.tl_layout_canon((4, 4), (4, 1), (1, 4), begin=(3, 0), extent=(2, 4))
    assert e.value.name == "TL_ERR_RANGE"


# ---------------------------------------------------------------------------
# bank simulator and chooser vs the oracle reference
# ---------------------------------------------------------------------------
def test_bank_conflicts_match_reference():
    rng = np.random.default_rng(2)
    for _ in range(500):
        eb = int(rng.choice([1, 2, 4, 8, 16]))
        offs = [int(x) for x in rng.integers(0, 400, size=32)]
        if rng.random() < 0.3:
            for i in rng.choice(32, size=5, replace=False):
                offs[int(i)] = None
        for model in ("conservative", "hardware"):
            assert tl.tl_bank_conflicts(offs, eb, model) == \
                L.bank_conflict_degree(offs, eb, model), (eb, model)


def test_choose_xor_k_matches_reference():
    rng = np.random.default_rng(3)
    n = 0
    for _ in range(300):
        P = int(rng.choice([1, 2, 4, 8, 3, 6]))
        total = 32 * P
        nd = int(rng.integers(1, 4))
        # random factorisation of total into nd extents
        ext = [total]
        for _ in range(nd - 1):
            divs = [d for d in range(2, ext[0]) if ext[0] % d == 0]
            if not divs:
                break
            d = int(rng.choice(divs))
            ext = [ext[0] // d, d] + ext[1:]
        perm = list(rng.permutation(len(ext)))
        ss = L.row_major_strides(ext)
        pst = L.row_major_strides(tuple(ext[p] for p in perm))
        ds = [0] * len(ext)
        for i, p in enumerate(perm):
            ds[p] = pst[i]
        eb = int(rng.choice([1, 2, 4, 8, 16]))
        want = L.choose_xor_k_ref(ext, ss, ds, eb)
        if want is None:
            with pytest.raises(tl.TLError) as e:
                tl.tl_choose_xor_k(ext, ss, ds, eb)
            assert e.value.name == "TL_ERR_NO_VALID_K"
        else:
            assert tl.tl_choose_xor_k(ext, ss, ds, eb) == want
            n += 1
    assert n > 50
    assert tl.tl_choose_xor_k((4, 32), (32, 1), (1, 4), 4) == (2, 3, 3)
    with pytest.raises(tl.TLError) as e:
        tl.tl_choose_xor_k((3, 5), (5, 1), (1, 3), 4)
    assert e.value.name == "TL_ERR_EXTENT"


# ---------------------------------------------------------------------------
# the tile kernel's shared-memory reads are conflict-free (model of its lanes)
# ---------------------------------------------------------------------------
def _swz(row, col):
    """Byte offset of byte `col` of tile row `row` under the TMA 128-byte swizzle."""
    return row * 128 + ((((col >> 4) ^ row) & 7) << 4) + (col & 15)


def _tile_read_pattern(eb):
    """Per load instruction: the byte offset each lane reads (mirrors k_tile's lanes)."""
    out = []
    if eb == 4:
        for u in range(32):
            cb, rb = u & 7, u >> 3
            for k in range(4):
                out.append([_swz(rb * 32 + 4 * (l >> 2) + (k ^ ((l >> 3) & 3)), 4 * (4 * cb + (l & 3)))
                            for l in range(32)])
    elif eb == 8:
        for u in range(32):
            cb, rb = u & 7, u >> 3
            for k in range(2):
                out.append([_swz(rb * 32 + 2 * (l >> 1) + (k ^ ((l >> 3) & 1)), 8 * (2 * cb + (l & 1)))
                            for l in range(32)])
    elif eb == 16:
        for u in range(32):
            cb, rb = u & 7, u >> 3
            out.append([_swz(rb * 32 + l, 16 * cb) for l in range(32)])
    elif eb == 2:
        for u in range(16):
            cb, rb = u & 7, u >> 3
            for k in range(8):
                out.append([_swz(rb * 64 + 8 * (l >> 2) + (k ^ (l >> 2)), 4 * (4 * cb + (l & 3)))
                            for l in range(32)])
    else:
        for cb in range(8):
            for k in range(16):
                out.append([_swz(16 * (l >> 2) + (k ^ (l >> 2)), 4 * (4 * cb + (l & 3)))
                            for l in range(32)])
    return out


@pytest.mark.parametrize("eb", [1, 2, 4, 8, 16])
def test_tile_kernel_smem_reads_are_conflict_free(eb):
    access = 4 if eb <= 4 else eb          # widths of the shared loads the kernel issues
    rows_read = set()
    for lanes in _tile_read_pattern(eb):
        assert all(o % access == 0 for o in lanes)
        elems = [o // access for o in lanes]
        assert tl.tl_bank_conflicts(elems, access, "hardware") == 1
        assert L.bank_conflict_degree(elems, access, "hardware") == 1
        rows_read.update(lanes)
    # together the loads cover the whole 16 KiB tile, each 4-byte word once
    words = set()
    for lanes in _tile_read_pattern(eb):
        for o in lanes:
            for b in range(0, access, 4):
                words.add(o + b)
    assert len(words) == 16384 // 4


def _perm_layout(shape, perm):
    ss = L.row_major_strides(shape)
    pst = L.row_major_strides(tuple(shape[p] for p in perm))
    ds = [0] * len(shape)
    for i, p in enumerate(perm):
        ds[p] = pst[i]
    return ss, tuple(ds)


PANEL_LAYOUTS = [
    # odd row pitches (no TMA), every width but 16 (16-byte rows always suit TMA)
    ((16383, 16385), (1, 0), 1), ((16383, 16385), (1, 0), 2), ((16383, 16385), (1, 0), 4),
    ((16383, 16385), (1, 0), 8),
    # interleaved channels <-> planes
    ((1024, 1024, 3), (2, 0, 1), 4), ((3, 1024, 1024), (1, 2, 0), 4),
    ((1024, 1024, 3), (2, 0, 1), 1), ((3, 1024, 1024), (1, 2, 0), 1),
    ((1024, 1024, 6), (2, 0, 1), 2),
    # more than three batch axes
    ((8, 4, 8, 4, 64, 64), (5, 3, 1, 4, 2, 0), 4),
]


def _panel_degrees(ta, tb, eb, pitch, row_off, nblk, aligned, vec):
    """Per-warp bank-conflict degrees (oracle model, hardware mode) of the panel
    kernel's two walks for a block-row layout of byte pitch `pitch`: the copy walk
    (16-byte blocks, nblk per row, row b at b * pitch) and the store walk, row b
    starting (r + row_off(b) * eb) mod 16 bytes into its first block for every base
    residue r (r = 0 only when every row is aligned); row_off(b) is the src element
    offset of row b.  Element stores: a warp takes tile elements f at a = f // tb,
    b = f % tb.  16-byte dst runs: rows are skewed by 16 bytes per V = 16 / eb rows,
    a warp takes 4 dst rows a by 8 blocks q of V elements, and at step k the lane of
    block q reads row q * V + k."""
    q = pitch // 16
    skew = (lambda b: b // (16 // eb)) if vec else (lambda b: 0)
    copy = [L.bank_conflict_degree([(g // nblk) * q + skew(g // nblk) + g % nblk
                                    for g in range(g0, min(nblk * tb, g0 + 32))], 16, "hardware")
            for g0 in range(0, nblk * tb, 32)]
    store = []
    for r in range(0, 1 if aligned else 16, eb):
        off = lambda a, b: (b * pitch + 16 * skew(b) + ((r + row_off(b) * eb) & 15) + a * eb) // eb
        if vec:
            V = 16 // eb
            for a0 in range(0, ta, 4):
                for q0 in range(0, tb // V, 8):
                    for k in range(V):
                        lanes = [(a0 + l // 8, q0 + l % 8) for l in range(32)]
                        offs = [off(a, qq * V + k) for a, qq in lanes if a < ta]
                        store.append(L.bank_conflict_degree(offs, eb, "hardware"))
            continue
        for f0 in range(0, ta * tb, 32):
            offs = [off(f // tb, f % tb) for f in range(f0, min(ta * tb, f0 + 32))]
            store.append(L.bank_conflict_degree(offs, eb, "hardware"))
    return copy, store


def test_interleaved_channel_paths():
    """The planner's kernel for interleaved channels <-> planes (H x W x C, W * H a
    whole number of 16-byte pieces): planes -> interleaved takes the rows register
    transpose for pixels of at most 16 bytes; interleaved -> planes takes the cols
    transpose for 2..16 channels of at most 24 bytes; everything else that is a plane
    goes to the tile or panel kernels."""
    H, W = 64, 96
    for eb in (1, 2, 4, 8):
        for C in range(2, 17):
            hwc = ((H, W, C), (W * C, C, 1), (W, 1, H * W))
            chw = ((C, H, W), (H * W, W, 1), (1, W * C, C))
            got = tl.tl_plan(SRC, DST, *hwc, eb)["path"]
            want_cols = C <= 16 and C * eb <= 24
            assert (got == "cols") == want_cols, ("hwc->chw", C, eb, got)
            if not want_cols:
                assert got in ("panel", "tile"), ("hwc->chw", C, eb, got)
            got = tl.tl_plan(SRC, DST, *chw, eb)["path"]
            want_rows = C * eb <= 16
            assert (got == "rows") == want_rows, ("chw->hwc", C, eb, got)
            if not want_rows:
                assert got in ("panel", "tile"), ("chw->hwc", C, eb, got)


def _permuted(shape, perm):
    ss = L.row_major_strides(shape)
    pst = L.row_major_strides(tuple(shape[p] for p in perm))
    ds = [0] * len(shape)
    for i, p in enumerate(perm):
        ds[p] = pst[i]
    return tuple(ss), tuple(ds)


def test_panel_merges_short_a_with_its_dense_src_neighbour():
    """A short src-contiguous axis a takes in the next src axis only where src is dense
    across the two and the a x b plane is under 16 KiB; merged tiles never take the
    walks that step one dst offset per row (runs, words) or the phase maps."""
    for eb in (1, 2, 4, 8, 16):
        shape = (10,) * 8
        ss, ds = _permuted(shape, tuple(range(7, -1, -1)))
        p = tl.tl_plan(SRC, DST, shape, ss, ds, eb, path="panel")
        # the plane is a (10) x b (10 x 10 merged in dst): 1000 * eb bytes
        assert p["panel_a1"] == (10 if 1000 * eb < 16384 else 0), (eb, p)
        if p["panel_a1"]:
            assert p["panel_vec"] in (0, 1) and p["panel_mode"] in (0, 1), p
            # the merged a spans the tile columns: 100 elements, tiles of at most 100
            assert p["tile_cols"] <= 100
        # src padded past the pair: the merge needs ss of the next axis == ext_a
        ss_pad = tuple(x * 2 if i < 7 else x for i, x in enumerate(ss))
        q = tl.tl_plan(SRC, 1 << 40, shape, ss_pad, ds, eb, path="panel")
        assert q["panel_a1"] == 0, (eb, q)
    # a plane of 16 KiB or more stays unmerged (24^6 fp16: 24 x 576 x 2 bytes)
    shape = (24,) * 6
    ss, ds = _permuted(shape, (5, 0, 4, 1, 3, 2))
    assert tl.tl_plan(SRC, DST, shape, ss, ds, 2, path="panel")["panel_a1"] == 0
    # a of 64 elements or more is never merged
    shape = (4, 4, 64, 64)
    ss, ds = _permuted(shape, (3, 2, 1, 0))
    assert tl.tl_plan(SRC, DST, shape, ss, ds, 1, path="panel")["panel_a1"] == 0


def test_panel_merge_invariants_on_seeded_high_rank_layouts():
    """Seeded high-rank permutes of short axes: wherever the planner merges a, the
    merged axis is the src-contiguous one with its dense src neighbour, the plane was
    under 16 KiB, the merged tiles take neither the run nor the word walk nor a phase
    map, and the stage fits the panel kernel's shared memory."""
    rng = np.random.default_rng(77)
    merged = 0
    for _ in range(300):
        nd = int(rng.integers(4, 9))
        shape = tuple(int(x) for x in rng.integers(2, 13, size=nd))
        perm = tuple(int(x) for x in rng.permutation(nd))
        eb = int(rng.choice([1, 2, 4, 8, 16]))
        ss, ds = _permuted(shape, perm)
        try:
            p = tl.tl_plan(SRC, DST, shape, ss, ds, eb, path="panel")
        except tl.TLError as e:
            assert e.name == "TL_ERR_PATH", e
            continue
        assert p["smem_bytes"] <= 3 * (160 * 1024 // 3) + 128
        if not p["panel_a1"]:
            continue
        merged += 1
        ext, cs, cd = p["extent"], p["src_str"], p["dst_str"]   # canonical layout
        ia = list(cs).index(1)                          # the src-contiguous axis
        a1 = ext[ia]
        assert p["panel_a1"] == a1 < 64, (shape, perm, p)
        nxt = [i for i, x in enumerate(cs) if x == a1]  # its dense src neighbour
        assert nxt and cd[nxt[0]] != cd[ia] * a1, (shape, perm, p)
        assert cd[nxt[0]] != 1                          # a batch axis, not b
        assert p["panel_vec"] in (0, 1) and p["panel_mode"] in (0, 1), p
        assert p["tile_cols"] <= a1 * ext[nxt[0]]
    assert merged >= 20, merged


def test_panel_tile_heights_are_even():
    """The tile count along b is kept and the rows spread evenly in whole 16-byte units
    (b = 100 fp32 rows: 52 + 48, not 96 + 4), unless that loses the 16-byte run walk."""
    shape = (10,) * 8
    ss, ds = _permuted(shape, tuple(range(7, -1, -1)))
    p = tl.tl_plan(SRC, DST, shape, ss, ds, 4, path="panel")
    assert p["tile_rows"] == 52 and p["panel_vec"] == 1, p
    # 1-byte rows: 272 rows at 128 per tile would even out to 96 rows, under the 128
    # bytes the run walk needs, so the tile keeps 128 rows
    p = tl.tl_plan(SRC, DST, (272, 517), (517, 1), (1, 272), 1, path="panel")
    assert p["tile_rows"] == 128 and p["panel_vec"] == 1, p


def test_panel_tma_phase_map_invariants():
    """Every plan that loads rows by TMA phase maps keeps the TMA rules by
    construction, over seeded odd-pitch layouts: the box's x coordinate a0 * eb and its
    row of ta * eb + 16 bytes on the 16-byte grid (an odd number of 16-byte blocks),
    boxes of at most 256 elements a side, tb a multiple of phi, phi * pitch and every
    batch stride multiples of 16 bytes, at most three batch axes, one b axis, and the
    three-stage ring within the shared memory the kernel is set up for."""
    rng = np.random.default_rng(77)
    seen = 0
    for _ in range(400):
        eb = int(rng.choice([1, 2, 4, 8]))
        R, C = (int(x) for x in rng.integers(17, 5000, size=2))
        nb = int(rng.integers(0, 4))
        batch = tuple(int(x) for x in rng.integers(2, 5, size=nb))
        # src rows of pitch C (often odd), batch strides padded to the 16-byte grid
        plane = R * C
        bst, acc = [], -(-plane * eb // 16) * 16 // eb
        for e in reversed(batch):
            bst.insert(0, acc)
            acc *= e
        shape = batch + (R, C)
        ss = tuple(bst) + (C, 1)
        ds_plane = R + int(rng.integers(0, 3))
        dacc, dst_b = ds_plane * C, []
        for e in reversed(batch):
            dst_b.insert(0, dacc)
            dacc *= e
        ds = tuple(dst_b) + (1, ds_plane)
        so = int(rng.integers(0, 3))
        try:
            p = tl.tl_plan(SRC + so * eb, DST, shape, ss, ds, eb, path="panel")
        except tl.TLError:
            continue
        if p["panel_mode"] not in (2, 3):
            continue
        seen += 1
        assert (p["panel_mode"] == 2) == (eb == 2)
        ta, tb, pitch = p["tile_cols"], p["tile_rows"], p["pitch"]
        P = C * eb
        g = 16
        while P % g:
            g //= 2
        phi = 16 // g
        assert eb in (2, 4, 8) and nb <= 3
        assert (ta * eb) % 32 == 0 and pitch == ta * eb + 16 and (pitch // 16) % 2 == 1
        assert ta + 16 // eb <= 256 and tb % phi == 0 and tb // phi <= 256 and R >= phi
        assert (phi * P) % 16 == 0 and all((x * eb) % 16 == 0 for x in bst)
        pb = -(-(tb // phi) * pitch // 128) * 128
        assert p["smem_bytes"] == 3 * phi * pb + (128 if eb == 2 else 0) <= 160 * 1024 + 128
    assert seen > 20, seen


def _word_degrees(ta, tb, eb, pitch, row_off, rs, rm, aligned):
    """Bank-conflict degrees (oracle model, hardware mode) of the panel kernel's word
    walk over block rows: one warp per dst row a (the first four), lane w reading the
    k-th element of its word from row h + V4 w + ((k + rm (w >> rs)) mod V4), V4 = 4 / eb,
    for every head h and every base residue r."""
    V4 = 4 // eb
    out = []
    for r in (range(1) if aligned else range(0, 16, eb)):
        for h in range(V4):
            for a in range(min(ta, 4)):
                for k in range(V4):
                    offs = []
                    for l in range(32):
                        b = h + V4 * l + ((k + rm * (l >> rs)) % V4)
                        if b < tb:
                            offs.append((b * pitch + ((r + row_off(b) * eb) & 15) + a * eb) // eb)
                    out.append(L.bank_conflict_degree(offs, eb, "hardware"))
    return out


def _vec_rows_ok(tb, eb):
    """Tile heights the 16-byte run walk covers: whole 16-byte units, at least 128
    bytes, 8-unit groups at least 3/4 busy."""
    units = tb * eb // 16
    groups = -(-units // 8)
    return (tb * eb) % 16 == 0 and tb * eb >= 128 and 4 * units >= 24 * groups


def _check_skew_layout(p):
    """The skew walk's stage (1-byte elements, odd dst row pitch): tiles of 32 columns
    of a per warp by 256 rows of b, rows of ta + 32 bytes 16 bytes further per 16 rows.
    Lane l of warp w reads, for each of its window rows c = 0..30, the two
    aligned 16-byte words around its 16 columns of stage row 16 (l mod 16) + c (strip
    2w + l // 16): for every src offset u = 0..30 of those columns both reads must be
    conflict-free on the bank model (8 lanes a wavefront), and the copy of a row (16-byte
    blocks, consecutive threads) too."""
    ta, tb, pitch = p["tile_cols"], p["tile_rows"], p["pitch"]
    assert tb == 256 and ta in (128, 256) and pitch == ta + 32
    assert p["panel_vec"] == 4 and p["vec_bytes"] == 16 and p["panel_mode"] == 0
    stage = -(-(271 * pitch + 16 * 17) // 128) * 128
    # one stage per CTA by default (two CTAs an SM); 32 threads per 32 columns
    assert p["smem_bytes"] == stage and p["block"] in (0, ta)
    row = lambda r: r * pitch + 16 * (r // 16)
    assert row(270) + pitch <= stage
    for w in range(ta // 32):
        for c in range(31):
            for u in range(31):
                for half in (0, 16):
                    offs = [(row(16 * (l % 16) + c) + 16 * (2 * w + l // 16) + (u & 16) + half) // 16
                            for l in range(32)]
                    assert L.bank_conflict_degree(offs, 16, "hardware") == 1, (w, c, u)
    nblk = ta // 16 + 2
    for g0 in range(0, 271 * nblk, 32):
        offs = [(row(g // nblk) + 16 * (g % nblk)) // 16 for g in range(g0, min(g0 + 32, 271 * nblk))]
        assert L.bank_conflict_degree(offs, 16, "hardware") <= 2


@pytest.mark.parametrize("shape,perm,eb", PANEL_LAYOUTS)
def test_panel_layout_against_the_bank_model(shape, perm, eb):
    """The shared-memory layout the planner picks for the panel kernel, replayed
    through the oracle's bank model.  Rows copied as 16-byte blocks start on a
    16-byte boundary plus the row's own misalignment, so the column-wise store walk
    cannot be conflict-free in general: the padding the planner picks must give a
    store walk no worse than no padding, keep the copy walk within 2-way and the
    store walk within 4-way; with every row aligned and 16-byte dst runs the store
    walk is conflict-free.  Packed src rows are one run: the store walk stays within 2-way."""
    ss, ds = _perm_layout(shape, perm)
    p = tl.tl_plan(SRC, DST, shape, ss, ds, eb, path="panel")
    assert p["path"] == "panel"
    ta, tb, pitch, mode = p["tile_cols"], p["tile_rows"], p["pitch"], p["panel_mode"]
    ssb = [x for x, d in zip(p["src_str"], p["dst_str"]) if d == 1][0]
    b1 = p["panel_b1"]
    if b1:      # b walks the dst-contiguous axis and the next dst axis (stride b1) as one
        ssb2 = [x for x, d in zip(p["src_str"], p["dst_str"]) if d == b1][0]
        row_off = lambda b: (b % b1) * ssb + (b // b1) * ssb2
    else:
        row_off = lambda b: b * ssb
    n = ta * tb
    if mode in (2, 3):
        # phase-major stage (mode 2: loaded by TMA phase maps, 2- and 8-byte elements;
        # mode 3: by cp.async, 4-byte elements): phi = 16 / gcd(row pitch, 16), row b in
        # block b % phi, at row b // phi of ta * eb + 16 bytes, an odd number of 16-byte
        # blocks; blocks on 128-byte boundaries; the element walk over it reads 4- and
        # 8-byte elements conflict-free, 2-byte ones 2-way
        assert not b1 and (ssb * eb) % 16 != 0
        assert eb in ((2,) if mode == 2 else (4, 8))
        g = 16
        while (ssb * eb) % g:
            g //= 2
        phi = 16 // g
        assert tb % phi == 0 and pitch == ta * eb + 16 and (pitch // 16) % 2 == 1
        assert ta + 16 // eb <= 256 and tb // phi <= 256
        pb = -(-(tb // phi) * pitch // 128) * 128
        assert p["smem_bytes"] == 3 * phi * pb + (128 if mode == 2 else 0)
        assert p["panel_vec"] == 0
        srow = lambda b: (b % phi) * pb + (b // phi) * pitch
        degs = []
        for r in range(0, 16, eb):
            for f0 in range(0, min(n, 4096), 32):
                offs = [(srow(f % tb) + ((r + row_off(f % tb) * eb) & 15) + (f // tb) * eb) // eb
                        for f in range(f0, min(n, f0 + 32))]
                degs.append(L.bank_conflict_degree(offs, eb, "hardware"))
        assert max(degs) == (2 if eb == 2 else 1)
        return
    if mode == 0:
        # every src row on a 16-byte boundary: base, tile step ta and every src
        # stride but a's (1) multiples of 16 bytes
        aligned = SRC % 16 == 0 and (ta * eb) % 16 == 0 and all(
            (x * eb) % 16 == 0 for x in p["src_str"] if x != 1)
        # 16-byte dst runs: 1..8-byte elements, row pieces of whole 16-byte units
        # that keep 3/4 of the walk's lanes busy, every dst stride but b's (1) a
        # multiple of 16 bytes
        vec = eb <= 8 and _vec_rows_ok(tb, eb) and DST % 16 == 0 and all(
            (x * eb) % 16 == 0 for x in p["dst_str"] if x not in (1, b1))
        if b1:
            vec = vec and (ssb * eb) % 16 == 0 and (ssb2 * eb) % 16 == 0
        vec = vec and not (eb == 4 and not aligned)   # measured: element stores win there
        # else 16-byte pieces of one dst run per tile: a short b (the whole extent in
        # one tile) packed in dst next to a
        ext_b = [x for x, d in zip(p["extent"], p["dst_str"]) if d == 1][0]
        ds_a = [d for x, d in zip(p["src_str"], p["dst_str"]) if x == 1][0]
        run = not vec and eb <= 4 and tb <= 16 and tb == ext_b and ds_a == tb and not b1
        # else, 1-byte elements at an odd dst row pitch (planes of 64 x 64 or more):
        # 16-byte dst pieces by the skew walk
        ext_a = [x for x, s_ in zip(p["extent"], p["src_str"]) if s_ == 1][0]
        if not vec and not run and eb == 1 and not b1 and ds_a % 2 == 1 and min(ext_a, ext_b) >= 64:
            _check_skew_layout(p)
            return
        # else 4-byte words per dst row for 1-byte elements (one b axis)
        words = not vec and not run and eb == 1 and not b1
        assert p["panel_vec"] == (1 if vec else 2 if run else 3 if words else 0)
        assert p["vec_bytes"] == (16 if vec or run else 4 if words else eb)
        nblk = ta * eb // 16 if aligned else (ta * eb + 30) // 16
        assert pitch % 16 == 0 and 16 * nblk <= pitch < 16 * (nblk + 8)
        assert p["smem_bytes"] == 3 * (tb * pitch + (16 * (tb * eb // 16) if vec else 0))
        if words:
            # the word walk: lane w packs word w of one dst row from rows h + V4 w + k',
            # k' = (k + m (w >> s)) mod V4 with the planner's (s, m); the rotation must
            # beat or match the unrotated walk and reach 2-way
            rs, rm = p["panel_wrot"]
            store = _word_degrees(ta, tb, eb, pitch, row_off, rs, rm, aligned)
            store0 = _word_degrees(ta, tb, eb, pitch, row_off, 0, 0, aligned)
            assert sum(store) <= sum(store0) and max(store) <= 2
            return
        copy, store = _panel_degrees(ta, tb, eb, pitch, row_off, nblk, aligned, vec)
        copy0, store0 = _panel_degrees(ta, tb, eb, 16 * nblk, row_off, nblk, aligned, vec)
        assert sum(store) <= sum(store0)        # the store walk first ...
        assert max(copy) <= 2 and max(store) <= 4   # ... then a copy walk within 2-way
        if aligned and vec:
            assert max(store) == 1
    else:
        assert mode == 1 and ssb == ta and p["pitch"] == 0      # packed src rows
        assert p["smem_bytes"] == 3 * 16 * ((n * eb + 30) // 16)
        # 16-byte dst runs for 2..8-byte elements where enough of a warp's 4 rows a
        # are busy (the planner's measured rule; 1-byte rows keep word stores)
        busy = 4 * ta >= 3 * 4 * ((ta + 3) // 4)
        ok = {1: False, 2: ta >= 4 and busy, 4: ta != 2, 8: busy}[eb]
        vec = ok and _vec_rows_ok(tb, eb) and DST % 16 == 0 and all(
            (x * eb) % 16 == 0 for x in p["dst_str"] if x not in (1, b1))
        ext_b = [x for x, d in zip(p["extent"], p["dst_str"]) if d == 1][0]
        ds_a = [d for x, d in zip(p["src_str"], p["dst_str"]) if x == 1][0]
        run = not vec and eb <= 4 and tb <= 16 and tb == ext_b and ds_a == tb and not b1
        assert p["panel_vec"] == (1 if vec else 2 if run else 0)
        for f0 in range(0, n, 32):
            offs = [(f % tb) * ta + f // tb for f in range(f0, min(n, f0 + 32))]
            assert L.bank_conflict_degree(offs, eb, "hardware") <= 2


# ---------------------------------------------------------------------------
# planner and validation (tl_plan; no device needed)
# ---------------------------------------------------------------------------
def _plan(w, src=SRC, dst=DST, **kw):
    return tl.tl_plan(src, dst, w.shape, w.src_strides, w.dst_strides, w.elem_bytes, **kw)


def test_plans_of_the_workloads():
    p = _plan(workloads.get("sf_transpose"))
    assert p["path"] == "warp" and (p["k"], p["shift"], p["mask"]) == (2, 3, 3)
    p = _plan(workloads.get("tile_transpose"))
    assert p["path"] == "tile" and p["tiles"] == 65536 and p["vec_bytes"] == 16
    assert (p["tile_rows"], p["tile_cols"]) == (128, 64)
    p = _plan(workloads.get("mx_sf"))
    assert p["path"] == "rows" and p["extent"] == (1 << 21, 32, 4)
    p = _plan(workloads.get("attention"))
    assert p["path"] == "chunk" and p["vec_bytes"] == 16
    for name in ("t2d_u8", "t2d_f16", "t2d_f32", "t2d_f64", "t2d_v16"):
        p = _plan(workloads.get(name))
        assert p["path"] == "tile", name
    p = _plan(workloads.get("tile_transpose"), path="cluster")
    assert p["path"] == "cluster"


def test_tile_height_option():
    w = workloads.get("t2d_f32")                      # 16384 x 16384 float32
    p128 = _plan(w, tile_rows=128)
    p256 = _plan(w, tile_rows=256)
    assert p128["tile_rows"] == 128 and p256["tile_rows"] == 256
    assert p256["tiles"] * 2 == p128["tiles"] == (16384 // 32) * (16384 // 128)
    assert p256["smem_bytes"] == 4 * 256 * 128 + 1024
    # ring depth is capped at 192 KiB of tiles, unknown heights fall back to 128
    assert _plan(w, tile_rows=256, tile_stages=12)["smem_bytes"] == 6 * 256 * 128 + 1024
    assert _plan(w, tile_rows=200)["tile_rows"] == 128
    # the cluster variant keeps 128-row tiles
    assert _plan(w, path="cluster", tile_rows=256)["tile_rows"] == 128


def test_cluster_ring_options():
    w = workloads.get("tile_transpose")
    slot = 128 * 128
    # contiguous 16 KiB tiles: 2 staging + 2 receive slots; strided tiles: 2 + 1
    assert _plan(w, path="cluster")["smem_bytes"] == 4 * slot + 1024
    assert _plan(workloads.get("t2d_f32"), path="cluster")["smem_bytes"] == 3 * slot + 1024
    assert _plan(w, path="cluster", tile_stages=3, cluster_recv_stages=1)["smem_bytes"] == \
        4 * slot + 1024
    assert _plan(w, path="cluster", tile_stages=1, cluster_recv_stages=1)["smem_bytes"] == \
        2 * slot + 1024
    # at most 12 slots: the receive ring gives way
    assert _plan(w, path="cluster", tile_stages=8, cluster_recv_stages=8)["smem_bytes"] == \
        12 * slot + 1024
    assert _plan(w, path="cluster")["block"] == 7 * 32                # 4 consumer warps
    assert _plan(w, path="cluster", cluster_consumer_warps=8)["block"] == 11 * 32
    assert _plan(w, path="cluster", cluster_consumer_warps=5)["block"] == 7 * 32


def test_planner_invariants_on_random_layouts():
    """Every path the planner accepts for a random layout launches within the
    device limits (block <= 1024 threads, dynamic shared memory <= 227 KiB), covers
    the tensor with a positive number of work units, and reports a canonical shape
    with the tensor's element count; refusals are TL_ERR_PATH only."""
    rng = np.random.default_rng(4242)
    seen = set()
    for _ in range(400):
        eb = int(rng.choice([1, 2, 4, 8, 16]))
        nd = int(rng.integers(1, 8))
        hi = 600 if nd <= 2 else (60 if nd <= 4 else 9)
        shape = tuple(int(x) for x in rng.integers(1, hi, size=nd))
        perm = [int(p) for p in rng.permutation(nd)]
        pad = [int(x) for x in rng.integers(0, 3, size=nd)] if rng.random() < 0.4 else [0] * nd
        ss, acc = [], 1
        for e, p_ in zip(reversed(shape), reversed(pad)):
            ss.append(acc)
            acc *= e + p_
        ss = tuple(reversed(ss))
        pst = L.row_major_strides(tuple(shape[p] for p in perm))
        ds = [0] * nd
        for i, p in enumerate(perm):
            ds[p] = pst[i]
        n = int(np.prod(shape))
        so = int(rng.integers(0, 4)) * eb
        for path in tl.PATHS:
            try:
                plan = tl.tl_plan(SRC + so, DST, shape, ss, tuple(ds), eb, path=path)
            except tl.TLError as e:
                assert e.name == "TL_ERR_PATH", (shape, path, e.name)
                continue
            seen.add(plan["path"])
            assert int(np.prod(plan["extent"])) == n
            assert plan["tiles"] > 0 and 0 < plan["block"] <= 1024
            assert 0 <= plan["smem_bytes"] <= 227 * 1024, (shape, ss, ds, eb, path, plan)
            if plan["path"] == "panel":
                # store and copy modes, and the panel ring within its shared memory
                mode, store = plan["panel_mode"], plan["panel_vec"]
                assert mode in (0, 1, 2, 3) and store in (0, 1, 2, 3, 4)
                assert plan["smem_bytes"] <= 160 * 1024 + 128
                assert plan["vec_bytes"] == (16 if store in (1, 2, 4) else 4 if store == 3 else eb)
                if mode in (2, 3):          # phase-major stages: rows off the 16-byte grid
                    assert store == 0 and eb in (2, 4, 8) and (mode == 2) == (eb == 2)
                if store in (3, 4):
                    assert eb == 1 and mode == 0
                seen.add(("panel", mode, store))
            if plan["path"] == "cols":
                A, npx = plan["tile_cols"], plan["tile_rows"]
                assert 2 <= A <= 16 and A * eb <= 24 and npx * eb == 16
    assert {"chunk", "panel", "tile", "generic", "warp", "rows", "cluster", "cols"} <= seen, seen
    assert {("panel", 0, 0), ("panel", 0, 1)} <= seen, seen


def test_checked_run_flags():
    w = workloads.get("t2d_f32")
    dbg = tl.TL_FLAG_DEBUG_CHECKS
    assert _plan(w, flags=dbg)["path"] == "generic"                 # the checked kernel
    assert _plan(w, flags=dbg, path="generic")["path"] == "generic"
    assert _err(SRC, DST, w.shape, w.src_strides, w.dst_strides, 4, flags=dbg,
                path="tile") == "TL_ERR_PATH"
    skip = tl.TL_FLAG_TEST_SKIP_HOST_BOUNDS
    assert _err(SRC, DST, w.shape, w.src_strides, w.dst_strides, 4, flags=skip) == "TL_ERR_ARG"
    small = dict(dst_bytes=1024)
    assert _err(SRC, DST, w.shape, w.src_strides, w.dst_strides, 4, flags=dbg,
                **small) == "TL_ERR_BOUNDS"
    assert _plan(w, flags=dbg | skip, **small)["path"] == "generic"


def test_smoke_cases_take_the_paths_they_name():
    import __graft_entry__ as g
    for name, shape, ss, ds, eb, path in g.SMOKE_CASES:
        assert tl.tl_plan(SRC, DST, shape, ss, ds, eb)["path"] == path, name


def test_forced_paths_that_do_not_apply():
    w = workloads.get("attention")
    for path in ("tile", "rows", "cluster", "panel"):
        with pytest.raises(tl.TLError) as e:
            _plan(w, path=path)
        assert e.value.name == "TL_ERR_PATH"
    assert _plan(w, path="generic")["path"] == "generic"


def _err(*args, **kw):
    with pytest.raises(tl.TLError) as e:
        tl.tl_plan(*args, **kw)
    return e.value.name


def test_validation_errors():
    assert _err(SRC, DST, (4, 4), (4, 1), (1, 4), 3) == "TL_ERR_ELEM_BYTES"
    assert _err(SRC, DST, (4, 4), (4, -1), (1, 4), 4) == "TL_ERR_ARG"
    assert _err(SRC, DST, (4, -4), (4, 1), (1, 4), 4) == "TL_ERR_ARG"
    assert _err(SRC, DST, (4, 4), (4, 1), (1, 2), 4) == "TL_ERR_DST_OVERLAP"
    assert _err(SRC, DST, (4, 4), (4, 1), (0, 4), 4) == "TL_ERR_DST_OVERLAP"
    assert _err(SRC + 2, DST, (4, 4), (4, 1), (1, 4), 4) == "TL_ERR_ALIGN"
    assert _err(SRC, SRC + 32, (4, 4), (4, 1), (1, 4), 4) == "TL_ERR_ALIAS"
    assert _err(SRC, DST, (4, 4), (4, 1), (1, 4), 4, dst_bytes=60) == "TL_ERR_BOUNDS"
    assert _err(SRC, DST, (1 << 40, 1 << 30), (1 << 30, 1), (1, 1 << 40), 1) == "TL_ERR_RANGE"
    assert _err(0, DST, (4,), (1,), (1,), 4) == "TL_ERR_ARG"
    assert _err(SRC, DST, (2,) * 9, (1,) * 9, (1,) * 9, 1) == "TL_ERR_ARG"
    # degenerate calls that are fine
    assert tl.tl_plan(SRC, DST, (0, 5), (5, 1), (1, 0), 4)["path"] == "none"
    assert tl.tl_plan(0, 0, (3, 0), (1, 1), (1, 1), 4)["path"] == "none"
    assert tl.tl_plan(SRC, DST, (), (), (), 16)["path"] == "chunk"
    assert tl.tl_plan(SRC, DST, (4, 4), (4, 1), (1, 4), 4, dst_bytes=64)["path"] != "none"
    # sub-element misalignment is allowed for 1-byte elements
    assert tl.tl_plan(SRC + 1, DST + 3, (64, 64), (64, 1), (1, 64), 1)["path"] == "panel"


def test_in_place_only_on_the_warp_path():
    w = workloads.get("sf_transpose")
    p = tl.tl_plan(SRC, SRC, w.shape, w.src_strides, w.dst_strides, 4)
    assert p["path"] == "warp" and p["in_place"] and p["tiles"] == 2
    # a transpose whose tile does not read exactly what it writes cannot run in place
    assert _err(SRC, SRC, (64, 64), (64, 1), (1, 64), 4) == "TL_ERR_ALIAS"


def test_dst_overlap_check_is_sound():
    """Whatever the planner accepts as a destination is truly non-overlapping."""
    rng = np.random.default_rng(5)
    accepted = 0
    for _ in range(300):
        nd = int(rng.integers(1, 4))
        shape = tuple(int(x) for x in rng.integers(1, 5, size=nd))
        ds = tuple(int(x) for x in rng.integers(0, 20, size=nd))
        ss = L.row_major_strides(shape)
        try:
            tl.tl_plan(SRC, DST, shape, ss, ds, 4)
        except tl.TLError as e:
            assert e.name == "TL_ERR_DST_OVERLAP"
            continue
        accepted += 1
        assert L.offsets_unique(shape, ds), (shape, ds)
    assert accepted > 30


def _stage_chunk(c, R):
    """Physical 16-byte chunk of staged chunk c in the rows kernel's warp stage: an
    XOR swizzle for R a power of two, a single-shift one for R = 12, the plain index
    otherwise."""
    if R & (R - 1) == 0:
        return c ^ (((c >> 3) ^ (c >> 6)) & 7)
    return c ^ ((c >> 3) & 7) if R % 4 == 0 else c


@pytest.mark.parametrize("R", list(range(2, 17)))
def test_rows_kernel_stage_is_conflict_free(R):
    # writes: lane l parks its k-th output vector as chunk l*R + k (2-way for R = 6, 10,
    # 12, 14, which no swizzle of these forms improves further)
    for k in range(R):
        lanes = [_stage_chunk(l * R + k, R) for l in range(32)]
        assert tl.tl_bank_conflicts(lanes, 16, "hardware") == (2 if R in (6, 10, 12, 14) else 1)
    # read-back: lane l takes chunk 32*i + l, so stores are contiguous per instruction
    for i in range(R):
        lanes = [_stage_chunk(32 * i + l, R) for l in range(32)]
        assert tl.tl_bank_conflicts(lanes, 16, "hardware") == 1
    # the swizzle is a permutation of the warp's stage
    assert sorted(_stage_chunk(c, R) for c in range(32 * R)) == list(range(32 * R))


# ---------------------------------------------------------------------------
# plan cache
# ---------------------------------------------------------------------------
def test_plan_cache_hit_costs_under_a_microsecond(tmp_path):
    """A repeated tl_plan (the planning half of every tl_permute) is served from the
    plan cache: timed in C, without binding overhead."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    libdir = os.path.dirname(os.path.abspath(tl.load()._name))
    exe = str(tmp_path / "plan_timing")
    subprocess.run([cc, "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(here, "c", "plan_timing.c"), "-L", libdir, "-ltl_permute",
                    "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    hits = int(r.stdout.split("hits ")[1].split()[0])
    ns = float(r.stdout.split("ns per call ")[1])
    print("\ntl_plan cache hit: %.0f ns per call" % ns)
    assert hits == 500000
    assert ns < 1000.0


def test_plan_cache_keys_on_pointer_offsets_bounds_and_overlap():
    """Cached plans are reused only where they hold: another offset within 16 bytes
    re-plans (vector width), caller-given bounds are checked on every call, and
    buffers whose byte ranges meet are planned afresh (in place or rejected)."""
    shape, ss, ds = (37, 300, 16), (300 * 16, 16, 1), (16, 37 * 16, 1)   # chunk path
    base = 1 << 32
    h0 = tl.tl_plan_cache_hits()
    p0 = tl.tl_plan(base, base + (1 << 30), shape, ss, ds, 2)
    p1 = tl.tl_plan(base + (1 << 20), base + (1 << 30) + (1 << 20), shape, ss, ds, 2)
    assert tl.tl_plan_cache_hits() == h0 + 1 and p1 == p0 and p0["vec_bytes"] == 16
    p2 = tl.tl_plan(base + 2, base + (1 << 30), shape, ss, ds, 2)      # src off by 2 bytes
    assert p2["path"] == "chunk" and p2["vec_bytes"] == 2
    p3 = tl.tl_plan(base + 8, base + (1 << 30) + 8, shape, ss, ds, 2)
    assert p3["vec_bytes"] == 8
    # bounds: the cached plan, then a src buffer one byte too small
    need = ((37 - 1) * 300 * 16 + 299 * 16 + 15 + 1) * 2
    tl.tl_plan(base, base + (1 << 30), shape, ss, ds, 2, src_bytes=need)
    with pytest.raises(tl.TLError) as e:
        tl.tl_plan(base, base + (1 << 30), shape, ss, ds, 2, src_bytes=need - 1)
    assert e.value.name == "TL_ERR_BOUNDS"
    # overlap after a cached disjoint plan: the SF warp tile in place, then aliased
    sf = ((2, 1, 4, 32), (128, 128, 32, 1), (128, 128, 1, 4))
    assert tl.tl_plan(base, base + (1 << 20), *sf, 4)["in_place"] is False
    assert tl.tl_plan(base, base + (1 << 20), *sf, 4)["in_place"] is False
    assert tl.tl_plan(base, base, *sf, 4)["in_place"] is True
    with pytest.raises(tl.TLError) as e:
        tl.tl_plan(base, base + 64, *sf, 4)
    assert e.value.name == "TL_ERR_ALIAS"
    # and a null pointer is still an error on a layout planned before
    with pytest.raises(tl.TLError):
        tl.tl_plan(0, base + (1 << 30), shape, ss, ds, 2)


# ---------------------------------------------------------------------------
# block path planner
# ---------------------------------------------------------------------------
def test_block_planner_invariants_on_random_high_rank_layouts():
    """Whenever the block tile applies: its dst run fits the kernel's position table,
    the copy of a src run (the 16-byte blocks around it, up to 15 bytes past either
    end) fits the distance to the next run, both runs fit the tile's bytes, the
    kernel's shared memory fits the size it is set up for, and the tiles are at least
    the tensor's elements over the tile's."""
    rng = np.random.default_rng(91)
    seen = 0
    for _ in range(600):
        nd = int(rng.integers(2, 9))
        shape = tuple(int(x) for x in rng.integers(2, 13, size=nd))
        perm = tuple(int(p) for p in rng.permutation(nd))
        eb = int(rng.choice([1, 2, 4, 8, 16]))
        ss = L.row_major_strides(shape)
        pst = L.row_major_strides(tuple(shape[p] for p in perm))
        ds = [0] * nd
        for i, p in enumerate(perm):
            ds[p] = pst[i]
        try:
            b = tl.tl_plan(SRC, DST, shape, ss, ds, eb, path="block")
        except tl.TLError as e:
            assert e.name == "TL_ERR_PATH"
            continue
        seen += 1
        Ls, Ld, tiles, pitch = b["tile_cols"], b["tile_rows"], b["tiles"], b["pitch"]
        budget = 12288 if eb <= 2 else 32768
        assert 1 <= Ld <= 2048 and 1 <= Ls
        assert pitch >= Ls * eb + 30
        assert Ls * eb <= budget and Ld * eb <= budget
        assert b["smem_bytes"] <= 226 * 1024
        n = int(np.prod(shape))
        assert tiles * budget >= n * eb
    assert seen > 200


def test_block_path_taken_for_high_rank_short_axes():
    """The planner gives the block tile to the high-rank permutes of short axes whose
    panel tiles move shorter runs (reversed 8^8 fp32 too, whose panel tiles store
    16-byte runs), and keeps the panel where its runs are the longer ones (reversed
    10^8 fp32: block runs of 200 bytes against panel runs of 208) and where it stores
    16-byte runs against a block tile of more than 100 src runs (6-D fp32, 16^7 fp32)."""
    def plan(shape, perm, eb):
        ss = L.row_major_strides(shape)
        pst = L.row_major_strides(tuple(shape[p] for p in perm))
        ds = [0] * len(shape)
        for i, p in enumerate(perm):
            ds[p] = pst[i]
        return tl.tl_plan(1 << 40, 1 << 42, shape, ss, ds, eb)["path"]
    assert plan((12,) * 7, (6, 4, 2, 0, 1, 3, 5), 2) == "block"
    assert plan((12,) * 8, (7, 5, 3, 1, 0, 2, 4, 6), 2) == "block"
    assert plan((9,) * 8, (1, 4, 2, 3, 7, 5, 6, 0), 4) == "block"
    assert plan((12,) * 8, (7, 5, 3, 1, 0, 2, 4, 6), 8) == "block"
    assert plan((8,) * 8, tuple(range(7, -1, -1)), 4) == "block"
    assert plan((10,) * 8, tuple(range(7, -1, -1)), 4) == "panel"
    # panel tiles of 16-byte dst runs against block tiles of more than 100 src runs
    assert plan((16, 16, 16, 16, 64, 64), (5, 3, 1, 4, 2, 0), 4) == "panel"
    assert plan((16,) * 7, tuple(range(6, -1, -1)), 4) == "panel"


def test_every_workload_keeps_its_measured_path():
    """The planner's path for every named workload at full size, as measured fastest
    on GB300 (a rule change that moves one shows here before it costs throughput)."""
    from movement_tl_permute_gb300 import workloads
    want = {"sf_transpose": "warp", "tile_transpose": "tile", "mx_sf": "rows",
            "attention": "chunk", "t2d_u8": "tile", "t2d_f16": "tile", "t2d_f32": "tile",
            "t2d_f64": "tile", "t2d_v16": "tile", "t2d_odd_f32": "panel",
            "t2d_odd_u8": "panel", "hwc_chw_u8": "cols", "nd6_f32": "panel",
            "nd8_f32": "block", "nd8_u16": "block"}
    assert set(want) == set(workloads.WORKLOADS)
    for name, path in want.items():
        w = workloads.get(name)
        got = tl.tl_plan(1 << 40, 1 << 43, w.shape, w.src_strides, w.dst_strides,
                         w.elem_bytes)["path"]
        assert got == path, (name, got)


def test_block_launch_shape_and_tuning():
    """A block pipeline is its consumer warps and one producer warp: 8 consumer warps by
    default (4 for tiles of 48 src runs or more at two rings per SM or more), as many as
    the caller asks (1..17) within 36 warps per SM and 18 per CTA.  Where exactly two
    rings fit an SM, one CTA runs two pipelines (unless the caller sizes the grid by
    CTAs per SM)."""
    def plan(perm, **kw):
        shape = (9,) * 8
        ss = L.row_major_strides(shape)
        pst = L.row_major_strides(tuple(shape[p] for p in perm))
        ds = [0] * 8
        for i, p in enumerate(perm):
            ds[p] = pst[i]
        return tl.tl_plan(1 << 40, 1 << 42, shape, ss, ds, 4, path="block", **kw)
    nd8 = (1, 4, 2, 3, 7, 5, 6, 0)                # 9 src runs a tile, two rings per SM
    many = (6, 7, 2, 1, 4, 5, 3, 0)               # 81 src runs a tile, two rings per SM
    base = plan(nd8)
    assert base["block"] == 2 * 9 * 32            # one CTA, two pipelines of 8 + 1 warps
    assert plan(many)["block"] == 2 * 5 * 32
    assert plan(nd8, cluster_consumer_warps=4)["block"] == 2 * 5 * 32
    assert plan(nd8, cluster_consumer_warps=17)["block"] == 2 * 9 * 32   # 18 warps a CTA
    assert plan(nd8, cluster_consumer_warps=40)["block"] == 2 * 9 * 32   # out of range
    assert plan(nd8, tile_ctas_per_sm=2)["block"] == 9 * 32              # two CTAs of one
    assert plan(nd8, tile_ctas_per_sm=1, cluster_consumer_warps=17)["block"] == 18 * 32
    small = plan(nd8, panel_tile_kib=12)                                 # more rings per SM
    assert small["block"] in (9 * 32, 2 * 9 * 32)
    for b in (base, small):
        assert b["block"] <= 18 * 32 and b["smem_bytes"] <= 226 * 1024


def _random_thread_axis(rng):
    """A valid thread-axis layout: 32 lanes split over 1-2 axes and P registers over
    0-2 axes, each side's strides dense in a random order, the axes shuffled."""
    def split(total, parts):
        ext = []
        for _ in range(parts - 1):
            e = int(rng.choice([d for d in (1, 2, 4, 8) if total % d == 0]))
            ext.append(e)
            total //= e
        return ext + [total]
    lanes = split(32, int(rng.integers(1, 3)))
    regs = split(int(rng.choice([1, 2, 4, 8])), int(rng.integers(0, 3))) if rng.random() < 0.9 else []
    axes = []
    for side, exts in (("lane", lanes), ("reg", regs)):
        order = rng.permutation(len(exts))
        stride = 1
        strides = [0] * len(exts)
        for k in order:
            strides[k] = stride
            stride *= exts[k]
        axes += [(side, e, st) for e, st in zip(exts, strides)]
    axes = [axes[k] for k in rng.permutation(len(axes))][:4]
    shape = tuple(e for _, e, _ in axes)
    lane = [st if side == "lane" else 0 for side, _, st in axes]
    reg = [st if side == "reg" else 0 for side, _, st in axes]
    return shape, lane, reg


def test_thread_axis_check_matches_the_oracle():
    """tl_thread_axis_check against the oracle's enumeration on the page's example
    (8 registers), on seeded valid layouts of 1-4 axes, and on each of them broken
    (a stride doubled, a side swapped)."""
    assert tl.tl_thread_axis_check((32, 8), (1, 0), (0, 1)) == 8
    rng = np.random.default_rng(17)
    valid = 0
    for _ in range(200):
        shape, lane, reg = _random_thread_axis(rng)
        variants = [(lane, reg)]
        k = int(rng.integers(0, len(shape)))
        l2, r2 = list(lane), list(reg)
        if l2[k]:
            l2[k] *= 2
        else:
            r2[k] *= 2
        variants.append((l2, r2))
        variants.append((list(reg), list(lane)))
        for ls, rs in variants:
            want = L.thread_axis_registers(shape, ls, rs)
            try:
                got = tl.tl_thread_axis_check(shape, ls, rs)
            except tl.TLError as e:
                assert e.name == "TL_ERR_EXTENT" and want is None, (shape, ls, rs)
                continue
            assert got == want, (shape, ls, rs)
            valid += 1
    assert valid >= 200
    with pytest.raises(tl.TLError):
        tl.tl_thread_axis_check((32, 8), (1, 1), (0, 1))


def test_no_kernel_spills_registers():
    """ptxas -v on every CUDA source: no kernel or device function spills a register
    (spill stores and loads go through local memory on the hot path)."""
    from movement_tl_permute_gb300 import build
    res = build.kernel_resources()
    assert len(res) > 50 and any("k_panel_skew" in r["name"] for r in res)
    bad = [r for r in res if r["spill_stores"] or r["spill_loads"]]
    assert not bad, bad


def _inv16(d):
    return next(x for x in range(1, 16, 2) if (d * x) % 16 == 1)


@pytest.mark.parametrize("ext_a,ext_b,pd,dmis,ta", [
    (300, 270, 303, 0, 256), (300, 270, 303, 7, 128), (513, 290, 529, 3, 256),
    (64, 64, 67, 15, 256), (290, 513, 521, 9, 128), (600, 260, 601, 12, 256)])
def test_skew_walk_pieces_cover_the_plane(ext_a, ext_b, pd, dmis, ta):
    """The skew walk's ownership, replayed on the host with the kernel's formulas: tiles of
    ta columns (a) by 256 rows (b); strips start e columns into each tile, e = -rho0 / delta
    mod 16 with rho0 the tile's first dst offset to the next 16-byte boundary and delta =
    -pd mod 16; the lane (strip, block) stores at step k the piece of column e + 16 strip +
    (k / delta mod 16) starting at row 16 block + k.  Every full piece must start on a
    16-byte boundary, no two pieces may overlap, and the pieces plus the first row and column
    blocks' element stores must cover every element of the plane."""
    delta = (-pd) % 16
    dinv = _inv16(delta)
    base = 4096 + dmis                       # dst byte address of element (a=0, b=0)
    hits = np.zeros((ext_a, ext_b), dtype=np.int32)
    edge = np.zeros((ext_a, ext_b), dtype=bool)
    for a0 in range(0, ext_a, ta):
        for b0 in range(0, ext_b, 256):
            d = base + a0 * pd + b0
            rho0 = (16 - d % 16) % 16
            e = ((16 - rho0) * dinv) % 16
            xlim, ylim = min(ext_a - a0, ta + 16), min(ext_b - b0, 256 + 16)
            for strip in range(ta // 16):
                x0 = e + 16 * strip
                for blk in range(16):
                    for k in range(16):
                        j = (k * dinv) % 16
                        r0 = 16 * blk + k
                        if x0 + j >= xlim or r0 >= ylim:
                            continue
                        n = min(16, ylim - r0)
                        if n == 16:
                            assert (d + (x0 + j) * pd + r0) % 16 == 0
                        hits[a0 + x0 + j, b0 + r0:b0 + r0 + n] += 1
            if b0 == 0:
                xs = 0 if a0 == 0 else e
                for x in range(xs, min(ta + e, xlim)):
                    edge[a0 + x, 0:min(15, ylim)] = True
            if a0 == 0:
                for x in range(min(e, xlim)):
                    edge[x, b0:b0 + min(256, ylim)] = True
    assert hits.max() <= 1                    # pieces never overlap
    assert ((hits == 1) | edge).all()         # and with the edge stores cover the plane


def test_skew_walk_eligibility():
    """The panel path takes the skew walk for 1-byte planes whose dst rows sit at an odd
    pitch, both extents at least 64, unless element stores are asked for; other widths,
    even pitches and small planes keep the other store modes."""
    def vec(shape, ss, ds, eb=1, **kw):
        return tl.tl_plan(SRC, DST, shape, ss, ds, eb, path="panel", **kw)["panel_vec"]
    assert vec((300, 270), (270, 1), (1, 303)) == 4
    assert vec((64, 64), (65, 1), (1, 65)) == 4
    assert vec((300, 270), (270, 1), (1, 302)) != 4              # even dst pitch
    assert vec((63, 270), (270, 1), (1, 63)) != 4                # b extent under 64
    assert vec((300, 63), (63, 1), (1, 303)) != 4                # a extent under 64
    assert vec((300, 270), (270, 1), (1, 303), eb=2) != 4        # 2-byte elements
    assert vec((300, 270), (270, 1), (1, 303),
               flags=tl.TL_FLAG_PANEL_ELEMENT_STORES) != 4
    assert tl.tl_plan(SRC, DST, (300, 270), (270, 1), (1, 303), 1)["path"] == "panel"
