"""Randomised parity over every kernel path, and concurrent calls from host threads.

Seeded random layouts (rank 1-6, extents 1-70, random axis permutations, padded
source strides, element offsets, every element width) go through the planner's
choice and through every forced path the planner says applies; each result is
compared byte for byte with the CPU oracle (canary bytes around the image).
"""
import threading

import numpy as np
import pytest

import movement_tl_permute_gb300 as tl
import oracle
from movement_tl_permute_gb300 import workloads
from oracle import layout_ref as L

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

PATHS = ["auto", "generic", "chunk", "tile", "rows", "warp", "cluster", "panel", "cols", "block"]
CANARY = 0x3C


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from movement_tl_permute_gb300 import build
    build.build()
    oracle.build()
    tl.load()


def _random_case(rng):
    eb = int(rng.choice([1, 2, 4, 8, 16]))
    nd = int(rng.integers(1, 7))
    shape = tuple(int(x) for x in rng.integers(1, 71 if nd <= 3 else 12, size=nd))
    perm = tuple(int(p) for p in rng.permutation(nd))
    pad = [int(x) for x in rng.integers(0, 3, size=nd)] if rng.random() < 0.3 else [0] * nd
    ss, acc = [], 1
    for e, p in zip(reversed(shape), reversed(pad)):
        ss.append(acc)
        acc *= e + p
    ss = tuple(reversed(ss))
    pst = L.row_major_strides(tuple(shape[p] for p in perm))
    ds = [0] * nd
    for i, p in enumerate(perm):
        ds[p] = pst[i]
    so = int(rng.integers(0, 3)) if rng.random() < 0.3 else 0
    do = int(rng.integers(0, 3)) if rng.random() < 0.3 else 0
    return shape, ss, tuple(ds), eb, so, do


def _run(shape, ss, ds, eb, so, do, path, seed, stream=None, **opts):
    span = lambda st: sum((e - 1) * x for e, x in zip(shape, st)) + 1
    n_src = (so + span(ss)) * eb
    n_dst = 256 + (do + span(ds)) * eb + 256
    src = workloads.random_bits(n_src, seed)
    want = np.full(n_dst, CANARY, dtype=np.uint8)
    oracle.permute(src, want, shape, ss, ds, eb, src_offset=so, dst_offset=256 // eb + do)
    s_gpu = torch.from_numpy(src).cuda()
    d_gpu = torch.full((n_dst,), CANARY, dtype=torch.uint8, device="cuda")
    st = stream if stream is not None else torch.cuda.current_stream()
    with torch.cuda.stream(st):
        tl.tl_permute_ex(s_gpu.data_ptr() + so * eb, d_gpu.data_ptr() + 256 + do * eb, shape,
                         ss, ds, eb, st.cuda_stream, path=path, **opts)
    st.synchronize()
    return d_gpu.cpu().numpy(), want


def test_random_layouts_every_applicable_path():
    rng = np.random.default_rng(2027)
    ran = {p: 0 for p in PATHS}
    for i in range(150):
        shape, ss, ds, eb, so, do = _random_case(rng)
        for path in PATHS:
            try:
                tl.tl_plan((1 << 20) + so * eb, (1 << 36) + 256 + do * eb, shape, ss, ds, eb,
                           path=path)
            except tl.TLError as e:
                assert e.name == "TL_ERR_PATH", e
                continue
            got, want = _run(shape, ss, ds, eb, so, do, path, seed=i)
            assert np.array_equal(got, want), (shape, ss, ds, eb, so, do, path)
            ran[path] += 1
            if path == "tile":                  # the 256-row tile variant as well
                got, want = _run(shape, ss, ds, eb, so, do, path, seed=i, tile_rows=256)
                assert np.array_equal(got, want), (shape, ss, ds, eb, so, do, "tile256")
    assert all(ran[p] > 0 for p in ("auto", "generic", "chunk", "tile", "panel")), ran


def _panel_case(rng):
    """A layout aimed at the panel kernel's store modes: 2-D transposes with odd or
    padded pitches, interleaved channels <-> planes, or 4-5-D permutes of short
    axes; offsets mostly 0 so that aligned dst rows (16-byte runs) occur."""
    eb = int(rng.choice([1, 2, 4, 8, 16]))
    kind = int(rng.integers(0, 3))
    if kind == 0:
        R, C = (int(x) for x in rng.integers(17, 300, size=2))
        ds_a = R + (int(rng.integers(0, 24)) if rng.random() < 0.5 else 0)
        shape, ss, ds = (R, C), (C, 1), (1, ds_a)
    elif kind == 1:
        c, H, W = int(rng.integers(2, 17)), int(rng.integers(2, 40)), int(rng.integers(17, 200))
        if rng.random() < 0.5:          # HWC -> CHW
            shape, ss, ds = (H, W, c), (W * c, c, 1), (W, 1, H * W)
        else:                           # CHW -> HWC
            shape, ss, ds = (c, H, W), (H * W, W, 1), (1, W * c, c)
    else:
        nd = int(rng.integers(4, 6))
        shape = tuple(int(x) for x in rng.integers(2, 12, size=nd))
        shape = shape[:-1] + (int(rng.choice([4, 8, 16, 33])),)
        perm = tuple(int(p) for p in rng.permutation(nd))
        ss = L.row_major_strides(shape)
        pst = L.row_major_strides(tuple(shape[p] for p in perm))
        ds = [0] * nd
        for i, p in enumerate(perm):
            ds[p] = pst[i]
        ds = tuple(ds)
    so = int(rng.integers(1, 4)) if rng.random() < 0.3 else 0
    do = int(rng.integers(1, 4)) if rng.random() < 0.3 else 0
    return shape, tuple(ss), ds, eb, so, do


def test_random_panel_layouts_every_store_mode():
    """The panel kernel's store modes (elements or packed-row words, 16-byte runs
    along tile rows, 16-byte pieces of one dst run, words per dst row of block rows,
    rotated reads) on seeded layouts, with random tile
    sizes and heights, each against the oracle, and again with element stores
    forced; every mode must occur."""
    rng = np.random.default_rng(4242)
    modes = set()
    for i in range(120):
        shape, ss, ds, eb, so, do = _panel_case(rng)
        opts = dict(panel_tile_kib=int(rng.choice([0, 4, 8, 16, 24, 32])),
                    tile_rows=int(rng.choice([0, 0, 16, 32, 64, 128])))
        try:
            plan = tl.tl_plan((1 << 20) + so * eb, (1 << 36) + 256 + do * eb, shape, ss, ds, eb,
                              path="panel", **opts)
        except tl.TLError as e:
            assert e.name == "TL_ERR_PATH", e
            continue
        modes.add(plan["panel_vec"])
        if plan["panel_wrot"][1]:
            modes.add("rotated")
        for flags in (0, tl.TL_FLAG_PANEL_ELEMENT_STORES):
            got, want = _run(shape, ss, ds, eb, so, do, "panel", seed=5000 + i, flags=flags,
                             **opts)
            assert np.array_equal(got, want), (shape, ss, ds, eb, so, do, opts, flags)
    assert {0, 1, 2, 3, "rotated"} <= modes, modes


def test_random_block_layouts_every_walk():
    """The block kernel on seeded high-rank permutes of short axes (3-8 axes of 2-12),
    every width, unaligned bases, random consumer-warp counts and tile sizes, each
    against the oracle; both store walks and both vector and single-element pieces must
    occur."""
    rng = np.random.default_rng(777)
    seen = set()
    done = 0
    for i in range(400):
        nd = int(rng.integers(3, 9))
        shape = tuple(int(x) for x in rng.integers(2, 13, size=nd))
        if int(np.prod(shape)) > (1 << 21):
            continue
        perm = tuple(int(p) for p in rng.permutation(nd))
        ss = L.row_major_strides(shape)
        pst = L.row_major_strides(tuple(shape[p] for p in perm))
        ds = [0] * nd
        for k, p in enumerate(perm):
            ds[p] = pst[k]
        ds = tuple(ds)
        eb = int(rng.choice([1, 2, 4, 8, 16]))
        so = int(rng.integers(0, 3)) if rng.random() < 0.4 else 0
        do = int(rng.integers(0, 3)) if rng.random() < 0.4 else 0
        opts = {}
        if rng.random() < 0.3:
            opts["cluster_consumer_warps"] = int(rng.integers(1, 18))
        if rng.random() < 0.3:
            opts["panel_tile_kib"] = int(rng.choice([4, 8, 16, 24, 32, 48]))
        try:
            plan = tl.tl_plan((1 << 20) + so * eb, (1 << 36) + 256 + do * eb, shape, ss, ds, eb,
                              path="block", **opts)
        except tl.TLError as e:
            assert e.name == "TL_ERR_PATH", e
            continue
        seen.add(("runs", plan["block_runs"] > 1))
        seen.add(("vec", plan["vec_bytes"] > eb))
        got, want = _run(shape, ss, ds, eb, so, do, "block", seed=7000 + i, **opts)
        assert np.array_equal(got, want), (shape, ss, ds, eb, so, do, opts)
        done += 1
    assert done >= 150
    assert {("runs", False), ("runs", True), ("vec", False), ("vec", True)} <= seen, seen


def test_concurrent_calls_from_host_threads():
    """Eight host threads, each on its own stream, permute different layouts at once."""
    rng = np.random.default_rng(99)
    cases = [_random_case(rng) for _ in range(8)]
    results = [None] * len(cases)
    errors = []

    def work(i):
        try:
            shape, ss, ds, eb, so, do = cases[i]
            results[i] = _run(shape, ss, ds, eb, so, do, "auto", seed=1000 + i,
                              stream=torch.cuda.Stream())
        except Exception as e:          # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for got, want in results:
        assert np.array_equal(got, want)
