"""Maximum sizes: every kernel path past 2^32 bytes (and the generic and block paths
past 2^32 elements), so that 64-bit offsets are exercised end to end.

The outputs are too large for the whole-tensor oracle loop, so the oracle
evaluates the definition one coordinate at a time (``oracle.sample``) at
seeded random coordinates plus every corner of the shape (the largest offsets),
and the GPU output is read back at exactly those offsets.  Also: a permute
captured into a CUDA graph replays bit-exactly.
"""
import itertools

import numpy as np
import pytest

import movement_tl_permute_gb300 as tl
import oracle
from movement_tl_permute_gb300 import workloads
from oracle import layout_ref as L

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N_SAMPLES = 1 << 18


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from movement_tl_permute_gb300 import build
    build.build()
    tl.load()


def _span(shape, strides):
    return sum((e - 1) * s for e, s in zip(shape, strides))


def _coords(shape, seed):
    rng = np.random.default_rng(seed)
    rand = np.stack([rng.integers(0, e, size=N_SAMPLES) for e in shape], axis=1)
    corners = np.array(list(itertools.product(*[(0, e - 1) for e in shape])))
    return np.concatenate([rand, corners]).astype(np.int64)


def check_sampled(shape, ss, ds, eb, path, seed):
    n_src = (_span(shape, ss) + 1) * eb
    n_dst = (_span(shape, ds) + 1) * eb
    assert max(n_src, n_dst) > (1 << 32) or int(np.prod(shape)) > (1 << 32)
    src = workloads.random_bits(n_src, seed)
    s_gpu = torch.from_numpy(src).cuda()
    d_gpu = torch.zeros(n_dst, dtype=torch.uint8, device="cuda")
    plan = tl.tl_plan(s_gpu.data_ptr(), d_gpu.data_ptr(), shape, ss, ds, eb, path=path)
    assert plan["path"] == path
    tl.tl_permute_ex(s_gpu.data_ptr(), d_gpu.data_ptr(), shape, ss, ds, eb,
                     torch.cuda.current_stream().cuda_stream, path=path)
    torch.cuda.synchronize()
    coords = _coords(shape, seed + 1)
    offs, want = oracle.sample(src, coords, ss, ds, eb)
    idx = torch.from_numpy(offs[:, None] * eb + np.arange(eb)[None, :]).cuda()
    got = d_gpu[idx.reshape(-1)].reshape(-1, eb).cpu().numpy()
    del s_gpu, d_gpu
    torch.cuda.empty_cache()
    bad = np.nonzero((got != want).any(axis=1))[0]
    assert bad.size == 0, "%d of %d sampled elements differ, first at coord %s" % (
        bad.size, len(coords), coords[bad[0]].tolist())


def test_tile_path_past_4gib():
    # u16 40000 x 60032 row-major -> column-major: 4.8 GB each way, 2.4e9 elements
    R, C = 40000, 60032
    check_sampled((R, C), (C, 1), (1, R), 2, "tile", seed=71)


def test_panel_path_past_4gib():
    # u8 65537 x 65539 (odd row pitch, no TMA) row-major -> column-major: 4.3 GB each way
    R, C = 65537, 65539
    check_sampled((R, C), (C, 1), (1, R), 1, "panel", seed=75)


def test_chunk_path_past_4gib():
    # (B, H, S, D) -> (B, S, H, D) with 4.3 GB of bf16: row offsets beyond 2^32 bytes
    shape = (33, 32, 4096, 512)
    ss = L.row_major_strides(shape)
    dss = L.row_major_strides((33, 4096, 32, 512))
    ds = (dss[0], dss[2], dss[1], dss[3])
    check_sampled(shape, ss, ds, 2, "chunk", seed=72)


def test_rows_path_past_4gib():
    # MX scale-factor blocks: (2^25 + 4096, 4, 32) uint8, 4.3 GB
    nb = (1 << 25) + 4096
    check_sampled((nb, 4, 32), (128, 32, 1), (128, 1, 4), 1, "rows", seed=73)


def test_block_path_past_4gib():
    # (126, 12^7) uint8 in the interleaved order (7,5,3,1,0,2,4,6): 4.5 GB each way,
    # 4.5e9 elements; and (18, 12^7) fp64, 5.2 GB each way
    for shape, eb, seed in (((126,) + (12,) * 7, 1, 76), ((18,) + (12,) * 7, 8, 77)):
        perm = (7, 5, 3, 1, 0, 2, 4, 6)
        ss = L.row_major_strides(shape)
        pst = L.row_major_strides(tuple(shape[p] for p in perm))
        ds = [0] * len(shape)
        for i, p in enumerate(perm):
            ds[p] = pst[i]
        check_sampled(shape, ss, tuple(ds), eb, "block", seed=seed)


def test_generic_path_past_2_32_elements():
    # 4.4e9 single bytes, axes fully reversed (no contiguous side): 64-bit flat index
    shape = (1100, 2000, 2000)
    ss = L.row_major_strides(shape)
    rs = L.row_major_strides(tuple(reversed(shape)))
    ds = tuple(reversed(rs))
    check_sampled(shape, ss, ds, 1, "generic", seed=74)


def test_permute_replays_inside_a_cuda_graph():
    w = workloads.scaled(workloads.get("tile_transpose"), 64)
    a = torch.from_numpy(workloads.make_input(w)).cuda()
    want = torch.empty_like(a)
    got = torch.empty_like(a)
    args = (w.shape, w.src_strides, w.dst_strides, w.elem_bytes)
    tl.tl_permute(a.data_ptr(), want.data_ptr(), *args, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tl.tl_permute(a.data_ptr(), got.data_ptr(), *args,
                      torch.cuda.current_stream().cuda_stream)
    for _ in range(3):
        got.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(got, want)
