"""tl_permute_tile_noalloc: the tile transpose for callers that cannot allocate.

Such callers (plug-ins whose host framework's allocator owns the device memory,
latency-critical code that cannot take cudaMalloc's implicit synchronisation,
fixed-memory deployments) cannot hand the library a status word, so this entry
point keeps it in the library's own static device scratch.  The test calls it
through the C ABI twice in a row, with
different inputs, and requires each result to equal, byte for byte, what the
ordinary tl_permute entry point produces for the same input; it also requires
the status it reports to be 0, and the device's free memory to stay the same
across calls.  This file sorts last so that a run stopping at
its first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import movement_tl_permute_gb300 as tl
from movement_tl_permute_gb300 import workloads

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CASES = [
    # batched 128x64 float16 tiles, row-major -> column-major per tile
    ((96, 128, 64), (8192, 64, 1), (8192, 1, 128), 2),
    # ragged 2-D float32 transpose
    ((300, 520), (520, 1), (1, 300), 4),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "needs a CUDA device"
    from movement_tl_permute_gb300 import build
    build.build()
    tl.load()


@pytest.mark.parametrize("shape,ss,ds,eb", CASES)
def test_noalloc_matches_tl_permute_on_two_calls_in_a_row(shape, ss, ds, eb):
    n = int(np.prod(shape)) * eb
    stream = torch.cuda.current_stream().cuda_stream
    status = ctypes.c_int32(-1)
    for call, seed in enumerate((11, 12)):
        src = torch.from_numpy(workloads.random_bits(n, seed)).cuda()
        ref = torch.full((n,), 0x5A, dtype=torch.uint8, device="cuda")
        out = torch.full((n,), 0xC3, dtype=torch.uint8, device="cuda")
        tl.tl_permute(src.data_ptr(), ref.data_ptr(), shape, ss, ds, eb, stream)
        status.value = -1
        tl.tl_permute_tile_noalloc(src.data_ptr(), out.data_ptr(), shape, ss, ds, eb, stream,
                                   host_status=status)
        torch.cuda.synchronize()
        assert status.value == 0, "call %d reported status %d" % (call, status.value)
        assert torch.equal(out, ref), "call %d differs from tl_permute" % call


def test_noalloc_call_allocates_no_device_memory():
    """Once the first call on the device has looked up the scratch address, a call
    leaves the device's free memory and torch's allocator untouched."""
    shape, ss, ds, eb = CASES[0]
    n = int(np.prod(shape)) * eb
    stream = torch.cuda.current_stream().cuda_stream
    src = torch.from_numpy(workloads.random_bits(n, 13)).cuda()
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    status = ctypes.c_int32(-1)
    tl.tl_permute_tile_noalloc(src.data_ptr(), out.data_ptr(), shape, ss, ds, eb, stream,
                               host_status=status)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        tl.tl_permute_tile_noalloc(src.data_ptr(), out.data_ptr(), shape, ss, ds, eb, stream,
                                   host_status=status)
    torch.cuda.synchronize()
    assert status.value == 0
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0


def test_noalloc_rejects_layouts_without_the_tile_path():
    a = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(tl.TLError) as e:
        tl.tl_permute_tile_noalloc(a.data_ptr(), a.data_ptr() + (1 << 15), (64, 128),
                                   (128, 1), (128, 1), 2)
    assert e.value.name == "TL_ERR_PATH"
