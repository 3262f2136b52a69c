"""GB300-native tensor layout permutation (sm_103a).

A thin ctypes binding over ``libtl_permute.so`` (the C ABI declared in
``include/tl_permute.h``).  Every function here only marshals arguments: the
planning runs in the library's host code and every byte moves in its CUDA
kernels.  There is no Python or CPU fallback: if the library has not been built,
loading it raises.

The names follow the C ABI: ``tl_layout_canon``, ``tl_choose_xor_k``,
``tl_bank_conflicts``, ``tl_permute``, ``tl_permute_ex``, ``tl_plan``,
``tl_status_string``, ``tl_launch_count``, ``tl_plan_cache_hits``, ``tl_version``.  ``permute`` is the
same call for PyTorch tensors (it reads their device pointers, byte bounds and
the current CUDA stream).
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading

__all__ = [
    "TLError", "TL_MAX_DIMS", "PATHS", "PATH_NAMES", "CASTS", "TL_FLAG_TEST_DROP_HANDOFF", "TL_FLAG_NO_PDL",
    "TL_FLAG_DEBUG_CHECKS", "TL_FLAG_TEST_SKIP_HOST_BOUNDS", "TL_FLAG_PANEL_ELEMENT_STORES",
    "load", "library_path", "tl_layout_canon", "tl_choose_xor_k", "tl_bank_conflicts",
    "tl_permute", "tl_permute_ex", "tl_plan", "tl_status_string", "tl_launch_count",
    "tl_plan_cache_hits", "tl_thread_axis_check",
    "tl_version", "permute", "tl_permute_tile_noalloc",
]

TL_MAX_DIMS = 8
PATHS = {"auto": 0, "generic": 1, "chunk": 2, "tile": 3, "warp": 4, "rows": 5, "cluster": 6,
         "panel": 7, "cols": 8, "block": 9}
PATH_NAMES = {v: k for k, v in PATHS.items()}
# fused permute + cast (tl_permute_opts.cast): name -> TL_CAST_*
CASTS = {"none": 0, "f32_to_bf16": 1, "f32_to_f16": 2, "bf16_to_f32": 3, "f16_to_f32": 4}
TL_FLAG_TEST_DROP_HANDOFF = 1 << 8
TL_FLAG_NO_PDL = 1 << 9
TL_FLAG_DEBUG_CHECKS = 1 << 10
TL_FLAG_TEST_SKIP_HOST_BOUNDS = 1 << 11
TL_FLAG_PANEL_ELEMENT_STORES = 1 << 12
STATUS = {0: "TL_OK", -1: "TL_ERR_ARG", -2: "TL_ERR_ELEM_BYTES", -3: "TL_ERR_EXTENT",
          -4: "TL_ERR_NO_VALID_K", -5: "TL_ERR_CHUNK", -6: "TL_ERR_DST_OVERLAP",
          -7: "TL_ERR_ALIAS", -8: "TL_ERR_ALIGN", -9: "TL_ERR_PATH", -10: "TL_ERR_RANGE",
          -11: "TL_ERR_CUDA", -12: "TL_ERR_TIMEOUT", -13: "TL_ERR_BOUNDS"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libtl_permute.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32


class TLError(RuntimeError):
    """A tl_* call returned a negative status."""

    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__("%s: %s (%s)" % (where, tl_status_string(code), self.name))


class TlLayout(ctypes.Structure):
    _fields_ = [("ndim", _i32), ("reserved", _i32), ("shape", _i64 * TL_MAX_DIMS),
                ("stride", _i64 * TL_MAX_DIMS), ("offset", _i64)]


class TlPermuteOpts(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint32), ("max_ctas", _i32), ("dev_status", ctypes.c_void_p),
                ("src_bytes", _i64), ("dst_bytes", _i64), ("tile_group", _i32),
                ("tile_stages", _i32), ("tile_ctas_per_sm", _i32), ("tile_l2_promotion", _i32),
                ("tile_rows", _i32), ("cluster_recv_stages", _i32),
                ("cluster_consumer_warps", _i32), ("panel_tile_kib", _i32),
                ("cast", _i32), ("cta_times", ctypes.c_void_p)]


class TlPlanInfo(ctypes.Structure):
    _fields_ = [("path", _i32), ("ndim", _i32), ("extent", _i64 * TL_MAX_DIMS),
                ("src_str", _i64 * TL_MAX_DIMS), ("dst_str", _i64 * TL_MAX_DIMS),
                ("vec_bytes", _i32), ("in_place", _i32), ("k", _i32), ("shift", _i32),
                ("mask", _i32), ("tile_rows", _i32), ("tile_cols", _i32), ("tiles", _i64),
                ("grid", _i32), ("block", _i32), ("smem_bytes", _i32), ("pitch", _i32),
                ("panel_mode", _i32), ("panel_b1", _i32), ("panel_vec", _i32),
                ("panel_wrot", _i32), ("panel_a1", _i32), ("block_runs", _i32)]


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load the CUDA library; raises if it was not built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                "libtl_permute.so is missing (%s): build it with "
                "`python -m movement_tl_permute_gb300.build` or __graft_entry__.build()"
                % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64p = ctypes.c_void_p, ctypes.POINTER(_i64)
        ip = ctypes.POINTER(ctypes.c_int)
        lib.tl_layout_canon.argtypes = [ctypes.POINTER(TlLayout), ctypes.POINTER(TlLayout), i64p,
                                        i64p, ctypes.POINTER(TlLayout), ctypes.POINTER(TlLayout),
                                        i64p]
        lib.tl_choose_xor_k.argtypes = [ctypes.c_int, i64p, i64p, i64p, ctypes.c_int, ip, ip, ip]
        lib.tl_thread_axis_check.argtypes = [ctypes.c_int, i64p, i64p, i64p, ip]
        lib.tl_bank_conflicts.argtypes = [ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int]
        lib.tl_permute.argtypes = [vp, vp, ctypes.c_int, i64p, i64p, i64p, ctypes.c_int, vp]
        lib.tl_permute_ex.argtypes = [vp, vp, ctypes.c_int, i64p, i64p, i64p, ctypes.c_int, vp,
                                      ctypes.POINTER(TlPermuteOpts)]
        lib.tl_plan.argtypes = [vp, vp, ctypes.c_int, i64p, i64p, i64p, ctypes.c_int,
                                ctypes.POINTER(TlPermuteOpts), ctypes.POINTER(TlPlanInfo)]
        lib.tl_status_string.argtypes = [ctypes.c_int]
        lib.tl_status_string.restype = ctypes.c_char_p
        lib.tl_launch_count.argtypes = []
        lib.tl_launch_count.restype = ctypes.c_uint64
        lib.tl_plan_cache_hits.argtypes = []
        lib.tl_plan_cache_hits.restype = ctypes.c_uint64
        lib.tl_version.argtypes = []
        lib.tl_permute_tile_noalloc.argtypes = [vp, vp, ctypes.c_int, i64p, i64p, i64p,
                                                ctypes.c_int, vp, ctypes.POINTER(_i32)]
        for name in ("tl_layout_canon", "tl_choose_xor_k", "tl_bank_conflicts", "tl_permute",
                     "tl_permute_ex", "tl_plan", "tl_version", "tl_permute_tile_noalloc"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


_ARR_TYPES = [_i64 * n for n in range(TL_MAX_DIMS + 1)]


def _arr(vals):
    n = len(vals)
    if n == 0:
        return _ARR_TYPES[1]()
    if n <= TL_MAX_DIMS:
        return _ARR_TYPES[n](*vals)
    return (_i64 * n)(*vals)


# The launch calls pass the same few shapes, strides and options again and again;
# the C side only reads them, so their ctypes forms are built once and reused.
@functools.lru_cache(maxsize=4096)
def _arr_of(t):
    return _arr(t)


def _carr(vals):
    try:
        return _arr_of(tuple(vals))
    except TypeError:                    # unhashable values: build afresh
        return _arr(vals)


@functools.lru_cache(maxsize=1024)
def _opts_of(items):
    return _opts(**dict(items))


def _check(rc: int, where: str) -> int:
    if rc < 0:
        raise TLError(rc, where)
    return rc


def _layout(shape, strides, offset=0) -> TlLayout:
    L = TlLayout()
    L.ndim = len(shape)
    for i, (e, s) in enumerate(zip(shape, strides)):
        L.shape[i] = int(e)
        L.stride[i] = int(s)
    L.offset = int(offset)
    return L


def tl_status_string(code: int) -> str:
    return load().tl_status_string(int(code)).decode()


def tl_launch_count() -> int:
    return int(load().tl_launch_count())


def tl_plan_cache_hits() -> int:
    return int(load().tl_plan_cache_hits())


def tl_version() -> int:
    return int(load().tl_version())


def tl_layout_canon(shape, src_strides, dst_strides, begin=None, extent=None, src_offset=0,
                    dst_offset=0) -> dict:
    """Slice + canonicalise + regroup a layout pair.  Returns the same keys as
    the oracle's reference: extent, src_str, dst_str, src_offset, dst_offset,
    chunk_elems."""
    lib = load()
    s, d = _layout(shape, src_strides, src_offset), _layout(shape, dst_strides, dst_offset)
    so, do = TlLayout(), TlLayout()
    chunk = _i64(0)
    b = _arr(begin) if begin is not None else None
    e = _arr(extent) if extent is not None else None
    _check(lib.tl_layout_canon(ctypes.byref(s), ctypes.byref(d), b, e, ctypes.byref(so),
                               ctypes.byref(do), ctypes.byref(chunk)), "tl_layout_canon")
    n = so.ndim
    return dict(extent=tuple(so.shape[:n]), src_str=tuple(so.stride[:n]),
                dst_str=tuple(do.stride[:n]), src_offset=so.offset, dst_offset=do.offset,
                chunk_elems=chunk.value)


def tl_thread_axis_check(extent, lane_strides, reg_strides) -> int:
    """Registers per lane of a warp's thread-axis ("1 @ laneid") layout; raises
    TLError if the layout does not place its coordinates on 32 lanes once each."""
    p = ctypes.c_int()
    _check(load().tl_thread_axis_check(len(extent), _arr(extent), _arr(lane_strides),
                                       _arr(reg_strides), ctypes.byref(p)),
           "tl_thread_axis_check")
    return p.value


def tl_choose_xor_k(extent, src_str, dst_str, elem_bytes):
    """(k, shift, mask) of the warp permute's XOR swizzle; raises TLError if none."""
    k, shift, mask = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(load().tl_choose_xor_k(len(extent), _arr(extent), _arr(src_str), _arr(dst_str),
                                  int(elem_bytes), ctypes.byref(k), ctypes.byref(shift),
                                  ctypes.byref(mask)), "tl_choose_xor_k")
    return k.value, shift.value, mask.value


def tl_bank_conflicts(lane_offsets, elem_bytes, model="conservative") -> int:
    offs = [-1 if o is None else int(o) for o in lane_offsets]
    m = {"conservative": 0, "hardware": 1}[model]
    return _check(load().tl_bank_conflicts(len(offs), _arr(offs), int(elem_bytes), m),
                  "tl_bank_conflicts")


def _opts(flags=0, path="auto", dev_status=0, src_bytes=0, dst_bytes=0, max_ctas=0,
          tile_group=0, tile_stages=0, tile_ctas_per_sm=0, tile_l2_promotion=0, tile_rows=0,
          cluster_recv_stages=0, cluster_consumer_warps=0, panel_tile_kib=0, cta_times=0,
          cast="none"):
    o = TlPermuteOpts()
    o.cta_times = int(cta_times) or None
    o.cast = CASTS[cast] if isinstance(cast, str) else int(cast)
    o.panel_tile_kib = int(panel_tile_kib)
    o.cluster_consumer_warps = int(cluster_consumer_warps)
    o.tile_rows = int(tile_rows)
    o.cluster_recv_stages = int(cluster_recv_stages)
    o.tile_group = int(tile_group)
    o.tile_stages = int(tile_stages)
    o.tile_ctas_per_sm = int(tile_ctas_per_sm)
    o.tile_l2_promotion = int(tile_l2_promotion)
    o.flags = (PATHS[path] if isinstance(path, str) else int(path)) | int(flags)
    o.max_ctas = int(max_ctas)
    o.dev_status = int(dev_status) or None
    o.src_bytes = int(src_bytes)
    o.dst_bytes = int(dst_bytes)
    return o


def tl_permute(src_ptr: int, dst_ptr: int, shape, src_strides, dst_strides, elem_bytes: int,
               stream: int = 0) -> None:
    """dst[sum c*dst_strides] = src[sum c*src_strides] on the GPU (device pointers)."""
    n = len(shape)
    _check(load().tl_permute(int(src_ptr) or None, int(dst_ptr) or None, n, _carr(shape),
                             _carr(src_strides), _carr(dst_strides), int(elem_bytes),
                             int(stream) or None), "tl_permute")


def tl_permute_ex(src_ptr: int, dst_ptr: int, shape, src_strides, dst_strides,
                  elem_bytes: int, stream: int = 0, **opts) -> None:
    """tl_permute with options: path=..., flags=..., dev_status=<device ptr>,
    src_bytes=..., dst_bytes=..., max_ctas=..., and the tile tuning fields
    tile_group, tile_stages, tile_ctas_per_sm, tile_l2_promotion, tile_rows,
    cluster_recv_stages, cluster_consumer_warps, panel_tile_kib"""
    try:
        o = _opts_of(tuple(sorted(opts.items())))
    except TypeError:                    # unhashable option values: build afresh
        o = _opts(**opts)
    _check(load().tl_permute_ex(int(src_ptr) or None, int(dst_ptr) or None, len(shape),
                                _carr(shape), _carr(src_strides), _carr(dst_strides),
                                int(elem_bytes), int(stream) or None, ctypes.byref(o)),
           "tl_permute_ex")


def tl_permute_tile_noalloc(src_ptr: int, dst_ptr: int, shape, src_strides, dst_strides,
                            elem_bytes: int, stream: int = 0, host_status=None) -> None:
    """The tile path with its status word in the library's static device scratch
    (for callers that cannot allocate).  ``host_status``: optional ctypes.c_int32
    that receives the status once the stream reaches it."""
    _check(load().tl_permute_tile_noalloc(
        int(src_ptr) or None, int(dst_ptr) or None, len(shape), _arr(shape), _arr(src_strides),
        _arr(dst_strides), int(elem_bytes), int(stream) or None,
        ctypes.byref(host_status) if host_status is not None else None),
        "tl_permute_tile_noalloc")


def tl_plan(src_ptr: int, dst_ptr: int, shape, src_strides, dst_strides, elem_bytes: int,
            **opts) -> dict:
    """What tl_permute_ex would launch (host-only)."""
    o = _opts(**opts)
    info = TlPlanInfo()
    _check(load().tl_plan(int(src_ptr) or None, int(dst_ptr) or None, len(shape), _arr(shape),
                          _arr(src_strides), _arr(dst_strides), int(elem_bytes),
                          ctypes.byref(o), ctypes.byref(info)), "tl_plan")
    n = info.ndim
    return dict(path=PATH_NAMES[info.path] if info.path else "none", ndim=n,
                extent=tuple(info.extent[:n]),
                src_str=tuple(info.src_str[:n]), dst_str=tuple(info.dst_str[:n]),
                vec_bytes=info.vec_bytes, in_place=bool(info.in_place), k=info.k,
                shift=info.shift, mask=info.mask, tile_rows=info.tile_rows,
                tile_cols=info.tile_cols, tiles=info.tiles, grid=info.grid, block=info.block,
                smem_bytes=info.smem_bytes, pitch=info.pitch, panel_mode=info.panel_mode,
                panel_b1=info.panel_b1, panel_vec=info.panel_vec,
                panel_wrot=(info.panel_wrot & 0xFF, info.panel_wrot >> 8),
                panel_a1=info.panel_a1, block_runs=info.block_runs)


def _bytes_after(t) -> int:
    """Bytes addressable from t.data_ptr() to the end of its storage."""
    st = t.untyped_storage()
    return st.nbytes() - (t.data_ptr() - st.data_ptr())


def permute(src, dst, shape, src_strides, dst_strides, elem_bytes=None, stream=None, **opts):
    """Permute between two CUDA tensors used as raw storage.

    ``src``/``dst`` are torch CUDA tensors whose ``data_ptr()`` is coordinate 0;
    strides are in elements of ``elem_bytes`` (default: the tensors' element
    size).  Launches on ``stream`` (default: torch's current stream) and checks
    the layouts against the tensors' storage bounds.
    """
    import torch

    if elem_bytes is None:
        elem_bytes = src.element_size()
    if stream is None:
        stream = torch.cuda.current_stream(src.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    opts.setdefault("src_bytes", _bytes_after(src))
    opts.setdefault("dst_bytes", _bytes_after(dst))
    tl_permute_ex(src.data_ptr(), dst.data_ptr(), shape, src_strides, dst_strides, elem_bytes,
                  stream, **opts)
