"""The device-side primitives of include/tl_permute_device.cuh, on the GPU.

Test kernels (tests/cuda/device_primitives.cu, built here with nvcc) call the
header's warp permute on shared memory (in place and out of place), its
register-fragment load + unrotate, its DSMEM region copy between the two CTAs of
a cluster, and its bounded global-word wait between two co-resident blocks.  The
host side uses the product's own tl_choose_xor_k and tl_layout_canon to set them
up; every result is compared byte for byte with the CPU oracle.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import movement_tl_permute_gb300 as tl
import oracle
from movement_tl_permute_gb300 import workloads
from oracle import layout_ref as L
from tests.conftest import ROOT

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CUDA_DIR = os.path.join(ROOT, "tests", "cuda")
LIB = os.path.join(CUDA_DIR, "_build", "libtl_device_tests.so")

_i32, _i64 = ctypes.c_int32, ctypes.c_int64


class TileArgs(ctypes.Structure):
    _fields_ = [("n", _i32), ("ext", _i32 * 4), ("src_str", _i64 * 4), ("dst_str", _i64 * 4),
                ("shift", _i32), ("mask", _i32), ("in_place", _i32), ("items", _i32)]


class ThreadAxisLayout(ctypes.Structure):
    _fields_ = [("n", _i32), ("ext", _i32 * 4), ("lane_str", _i32 * 4), ("reg_str", _i32 * 4),
                ("mem_str", _i64 * 4)]


class ChunkLoop(ctypes.Structure):
    _fields_ = [("chunk_bytes", ctypes.c_uint32), ("outer_n", _i32), ("outer_ext", _i32 * 4),
                ("src_stride", _i64 * 4), ("dst_stride", _i64 * 4)]


class RegionArgs(ctypes.Structure):
    _fields_ = [("loop", ChunkLoop), ("src_bytes", _i32), ("dst_bytes", _i32),
                ("src_off", _i32), ("dst_off", _i32), ("timeout_ns", ctypes.c_uint64)]


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    src = os.path.join(CUDA_DIR, "device_primitives.cu")
    hdr = os.path.join(ROOT, "include", "tl_permute_device.cuh")
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if (not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(src),
                                                               os.path.getmtime(hdr))):
        nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-shared", "-Xcompiler", "-fPIC", "-cudart", "static",
                        "-I", os.path.join(ROOT, "include"), src, "-o", LIB], check=True)
    from movement_tl_permute_gb300 import build
    build.build()
    tl.load()
    h = ctypes.CDLL(LIB)
    vp = ctypes.c_void_p
    h.tdp_warp_smem.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(TileArgs)]
    h.tdp_fragment.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(TileArgs)]
    h.tdp_lanes.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int,
                            ctypes.POINTER(ThreadAxisLayout)]
    h.tdp_dsmem.argtypes = [vp, vp, vp, ctypes.POINTER(RegionArgs)]
    h.tdp_wait.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_uint64]
    h.tdp_wait64.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_uint64]
    h.tdp_dsmem_stream.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint64, vp]
    return h


def _tile_args(ext, ss, ds, shift, mask, in_place=0, items=1):
    a = TileArgs()
    a.n = len(ext)
    for i in range(len(ext)):
        a.ext[i], a.src_str[i], a.dst_str[i] = ext[i], ss[i], ds[i]
    a.shift, a.mask, a.in_place, a.items = shift, mask, in_place, items
    return a


def _transposed(ext):
    """Column-major strides over ext (the reversed axis order is row-major)."""
    rs = L.row_major_strides(tuple(reversed(ext)))
    return tuple(reversed(rs))


def _swizzle(ext, ss, ds, eb):
    """The host chooser's swizzle; where it declines (no conflict-free k, which
    the oracle's simulator must agree with) the primitive still permutes
    correctly without one."""
    try:
        return tl.tl_choose_xor_k(ext, ss, ds, eb)
    except tl.TLError as e:
        assert e.name == "TL_ERR_NO_VALID_K"
        assert L.choose_xor_k_ref(ext, ss, ds, eb) is None
        return 0, 0, 0


CASES = [((4, 32), 4), ((4, 32), 1), ((8, 16), 2), ((2, 64), 4), ((4, 8, 4), 4),
         ((16, 16), 8), ((8, 16), 4), ((4, 32), 16), ((32,), 4), ((16, 32), 4)]


@pytest.mark.parametrize("ext,eb", CASES)
@pytest.mark.parametrize("in_place", [0, 1])
def test_warp_permute_in_shared_memory(lib, ext, eb, in_place):
    n = int(np.prod(ext))
    P = n // 32
    ss = L.row_major_strides(ext)
    ds = _transposed(ext)
    k, shift, mask = _swizzle(ext, ss, ds, eb)
    items = 5
    src = workloads.random_bits(items * n * eb, 500 + n + eb)
    want = np.zeros_like(src)
    for i in range(items):
        oracle.permute(src, want, ext, ss, ds, eb, src_offset=i * n, dst_offset=i * n)
    s_gpu = torch.from_numpy(src).cuda()
    d_gpu = torch.zeros_like(s_gpu)
    a = _tile_args(ext, ss, ds, shift, mask, in_place, items)
    assert lib.tdp_warp_smem(s_gpu.data_ptr(), d_gpu.data_ptr(), eb, P, ctypes.byref(a)) == 0
    torch.cuda.synchronize()
    assert np.array_equal(d_gpu.cpu().numpy(), want)


@pytest.mark.parametrize("ext,eb", CASES)
def test_register_fragment_round_trip(lib, ext, eb):
    n = int(np.prod(ext))
    P = n // 32
    ss = _transposed(ext)             # read the tile column-major ...
    k, shift, mask = _swizzle(ext, ss, L.row_major_strides(ext), eb)
    src = workloads.random_bits(n * eb, 900 + n + eb)
    want = np.zeros_like(src)
    # ... and hold it lane-major: register j of lane l = row-major element l + 32 j
    oracle.permute(src, want, ext, ss, L.row_major_strides(ext), eb)
    s_gpu = torch.from_numpy(src).cuda()
    d_gpu = torch.zeros_like(s_gpu)
    a = _tile_args(ext, ss, ss, shift, mask)
    assert lib.tdp_fragment(s_gpu.data_ptr(), d_gpu.data_ptr(), eb, P, ctypes.byref(a)) == 0
    torch.cuda.synchronize()
    assert np.array_equal(d_gpu.cpu().numpy(), want)


def _region(shape, ss, ds, so, do, eb, src_bytes, dst_bytes, seed):
    """Set the copy up from the two layouts through tl_layout_canon; return the
    GPU result, the oracle's and the two status words."""
    c = tl.tl_layout_canon(shape, ss, ds, src_offset=so, dst_offset=do)
    loop = ChunkLoop()
    loop.chunk_bytes = c["chunk_elems"] * eb
    outer = len(c["extent"]) - 1
    loop.outer_n = outer
    for i in range(outer):
        loop.outer_ext[i] = c["extent"][i]
        loop.src_stride[i] = c["src_str"][i] * eb
        loop.dst_stride[i] = c["dst_str"][i] * eb
    args = RegionArgs()
    args.loop = loop
    args.src_bytes, args.dst_bytes = src_bytes, dst_bytes
    args.src_off, args.dst_off = c["src_offset"] * eb, c["dst_offset"] * eb
    args.timeout_ns = 20_000_000
    src = workloads.random_bits(src_bytes, seed)
    canvas = np.full(dst_bytes, 0x5A, dtype=np.uint8)
    want = canvas.copy()
    oracle.permute(src, want, shape, ss, ds, eb, src_offset=so, dst_offset=do)
    s_gpu = torch.from_numpy(src).cuda()
    d_gpu = torch.from_numpy(canvas).cuda()
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    return s_gpu, d_gpu, status, args, want, canvas


def test_dsmem_copy_of_the_pages_128x64_tile(lib):
    shape, ss = (128, 64), (64, 1)
    c = tl.tl_layout_canon(shape, ss, ss)
    assert c["chunk_elems"] * 2 == 16384           # one bulk copy
    s_gpu, d_gpu, status, args, want, _ = _region(shape, ss, ss, 0, 0, 2, 16384, 16384, 41)
    assert lib.tdp_dsmem(s_gpu.data_ptr(), d_gpu.data_ptr(), status.data_ptr(),
                         ctypes.byref(args)) == 0
    torch.cuda.synchronize()
    assert status.tolist() == [1, 1]
    assert np.array_equal(d_gpu.cpu().numpy(), want)


def test_dsmem_copy_of_a_strided_region(lib):
    # a 64 x 40 float16 block at (3, 8) of a 128 x 64 image, into a 64-row tile of
    # pitch 48: 64 chunks of 80 bytes, strides 128 and 96 bytes
    shape, ss, ds = (64, 40), (64, 1), (48, 1)
    s_gpu, d_gpu, status, args, want, _ = _region(shape, ss, ds, 3 * 64 + 8, 16, 2,
                                                  128 * 64 * 2, 16 * 2 + 64 * 48 * 2 + 64, 42)
    assert args.loop.outer_n == 1 and args.loop.chunk_bytes == 80
    assert lib.tdp_dsmem(s_gpu.data_ptr(), d_gpu.data_ptr(), status.data_ptr(),
                         ctypes.byref(args)) == 0
    torch.cuda.synchronize()
    assert status.tolist() == [1, 1]
    assert np.array_equal(d_gpu.cpu().numpy(), want)


def test_dsmem_copy_declines_chunks_under_16_bytes(lib):
    # 4 float16 = 8 bytes per chunk: the primitive refuses and copies nothing; the
    # receiving CTA's bounded wait expires instead of hanging
    shape, ss, ds = (16, 4), (64, 1), (8, 1)
    s_gpu, d_gpu, status, args, _, canvas = _region(shape, ss, ds, 0, 0, 2, 128 * 16,
                                                    16 * 8 * 2, 43)
    assert args.loop.chunk_bytes == 8
    assert lib.tdp_dsmem(s_gpu.data_ptr(), d_gpu.data_ptr(), status.data_ptr(),
                         ctypes.byref(args)) == 0
    torch.cuda.synchronize()
    assert status.tolist() == [2, 0]
    assert np.array_equal(d_gpu.cpu().numpy(), canvas)


@pytest.mark.parametrize("publish", [1, 0])
def test_wait_until_global(lib, publish):
    n = 4096
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    data = torch.zeros(n, dtype=torch.int32, device="cuda")
    out = torch.zeros(n, dtype=torch.int32, device="cuda")
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    rc = lib.tdp_wait(flag.data_ptr(), data.data_ptr(), out.data_ptr(), status.data_ptr(), n,
                      publish, 20_000_000)
    assert rc == 0
    torch.cuda.synchronize()
    if publish:
        assert status.tolist() == [1, 7]
        assert torch.equal(out, data) and int(data[1].item()) != 0
    else:
        assert int(status[0].item()) == 0          # the bounded wait gave up
        assert not bool(out.any())


@pytest.mark.parametrize("publish", [1, 0])
def test_wait_until_global_64_bit_word_system_scope_with_backoff(lib, publish):
    """The pull request's other parameters ("Other parameters"): a 64-bit word read
    as raw bits, polls at system scope, an opt-in backoff between polls; the
    accepted value is the whole 64-bit word, and the bounded wait still gives up
    when nobody publishes."""
    n = 4096
    flag = torch.zeros(1, dtype=torch.int64, device="cuda")
    data = torch.zeros(n, dtype=torch.int32, device="cuda")
    out = torch.zeros(n, dtype=torch.int32, device="cuda")
    status = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    assert lib.tdp_wait64(flag.data_ptr(), data.data_ptr(), out.data_ptr(), status.data_ptr(),
                          n, publish, 20_000_000) == 0
    torch.cuda.synchronize()
    if publish:
        assert status.tolist() == [1, 1 << 8, 7]
        assert torch.equal(out, data) and int(data[1].item()) != 0
    else:
        assert int(status[0].item()) == 0
        assert not bool(out.any())


def test_dsmem_stream_ceiling(lib):
    """The cluster hand-off pattern with no HBM traffic: 16 KiB pushes into 2-slot
    rings of the peer, released by remote arrives, 3 CTAs per SM.  Prints the
    SM-to-SM throughput this pattern reaches (the cluster path's own ceiling)."""
    grid = 2 * ((torch.cuda.get_device_properties(0).multi_processor_count * 3) // 2)
    iters = 2000
    status = torch.ones(grid, dtype=torch.int32, device="cuda")
    for _ in range(2):                                       # warm-up, then timed
        status.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        assert lib.tdp_dsmem_stream(grid, iters, 2_000_000_000, status.data_ptr()) == 0
        e1.record()
        torch.cuda.synchronize()
    assert bool((status == 1).all())
    gbs = grid * iters * 16384 / (e0.elapsed_time(e1) * 1e-3) / 1e9
    print("\nDSMEM hand-off ceiling: %.0f GB/s pushed (grid %d, %d pushes of 16 KiB per CTA)"
          % (gbs, grid, iters))
    assert gbs > 100


# ---------------------------------------------------------------------------
# thread-axis ("1 @ laneid") layouts: a lane's local registers
# ---------------------------------------------------------------------------
LANE_LAYOUTS = [
    # the page's S[(32, 8) : (1 @ laneid, 1)] over a row-major and a transposed buffer
    ((32, 8), (1, 0), (0, 1), (8, 1)),
    ((32, 8), (1, 0), (0, 1), (1, 32)),
    # lanes over two axes, one register axis
    ((4, 8, 2), (8, 1, 0), (0, 0, 1), (16, 2, 1)),
    # the lane axis in the middle, registers from the outer and inner axes, two orders
    ((2, 32, 4), (0, 1, 0), (4, 0, 1), (128, 4, 1)),
    ((2, 32, 4), (0, 1, 0), (1, 0, 2), (128, 4, 1)),
    # lanes split around a register axis, memory padded
    ((8, 16, 4), (4, 0, 1), (0, 1, 0), (100, 6, 1)),
]


@pytest.mark.parametrize("eb", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("case", range(len(LANE_LAYOUTS)))
def test_thread_axis_load_and_store_match_the_oracle(lib, eb, case):
    """warp_load_lanes puts in lane l's register j the element the oracle places
    there (thread_axis_fragment), for every element width; warp_store_lanes puts it
    back where it came from, leaving the padding untouched."""
    shape, ls, rs, ms = LANE_LAYOUTS[case]
    P = tl.tl_thread_axis_check(shape, ls, rs)
    assert P == L.thread_axis_registers(shape, ls, rs)
    if (eb, P) not in {(1, 1), (1, 2), (1, 8), (2, 2), (2, 8), (4, 1), (4, 2), (4, 4), (4, 8),
                       (4, 16), (8, 4), (8, 8), (16, 2)}:
        pytest.skip("no test kernel for this register count and width")
    span = sum((e - 1) * m for e, m in zip(shape, ms)) + 1
    src = workloads.random_bits(span * eb, 700 + case)
    lay = ThreadAxisLayout()
    lay.n = len(shape)
    for k in range(len(shape)):
        lay.ext[k], lay.lane_str[k], lay.reg_str[k], lay.mem_str[k] = shape[k], ls[k], rs[k], ms[k]
    s_gpu = torch.from_numpy(src).cuda()
    frag = torch.zeros(32 * P * eb, dtype=torch.uint8, device="cuda")
    back = torch.full((span * eb,), 0x3C, dtype=torch.uint8, device="cuda")
    assert lib.tdp_lanes(s_gpu.data_ptr(), frag.data_ptr(), back.data_ptr(), eb, P,
                         ctypes.byref(lay)) == 0
    torch.cuda.synchronize()
    elems = src.reshape(-1, eb)
    want = L.thread_axis_fragment([bytes(e) for e in elems], shape, ms, ls, rs)
    got = frag.cpu().numpy().reshape(32, P, eb)
    for lane in range(32):
        for j in range(P):
            assert bytes(got[lane, j]) == want[lane][j], (lane, j)
    # the store writes exactly the layout's elements back
    expect = np.full(span * eb, 0x3C, dtype=np.uint8).reshape(-1, eb)
    for c in L.thread_axis_places(shape, ls, rs):
        o = L.apply(c, ms)
        expect[o] = elems[o]
    assert np.array_equal(back.cpu().numpy(), expect.reshape(-1))
