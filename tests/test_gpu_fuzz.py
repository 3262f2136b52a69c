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

PATHS = ["auto", "generic", "chunk", "tile", "rows", "warp", "cluster", "panel"]
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
