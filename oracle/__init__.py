"""CPU oracle for tensor layout permutation -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline
and its ``--impl reference`` arm) may import anything here.  The product path
(the CUDA library and its Python binding) never does, and this package imports
nothing from the product: the two share no code.

Contents
--------
* ``permute`` -- ctypes front of ``permute_ref.c``: the definition
  ``dst[sum c_i*dst_stride_i] = src[sum c_i*src_stride_i]`` for every coordinate
  ``c`` (TVM docs, "Buffers and memory", section "Declaring buffers").
* ``sample`` -- the same definition evaluated at chosen coordinates one by one,
  for outputs too large to permute whole on the host.
* ``permute_cast`` -- the same definition with every element converted on the way
  (``cast_ref``: IEEE 754 binary32 <-> binary16 / bfloat16).
* ``layout_ref`` -- pure-Python references for the host logic: slicing and
  canonicalising a pair of layouts, the shared-memory bank model and the XOR
  swizzle chooser of the warp permute (TVM docs, "permute_layout", section
  "Algorithm"), and a brute-force overlap test.  Small inputs only.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
the pages print, closed forms, library routines (numpy transposes) and brute
force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import cast_ref  # noqa: F401  (re-exported)
from . import layout_ref  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "permute_ref.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_permute.so")
_lock = threading.Lock()
_lib = None

ELEM_BYTES = (1, 2, 4, 8, 16)


def build(force: bool = False) -> str:
    """Compile permute_ref.c into a shared library (gcc, OpenMP when available)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.oracle_permute.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                           i64p, i64p, i64p, ctypes.c_int, ctypes.c_int]
            lib.oracle_permute.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _i64(vals):
    arr = (ctypes.c_int64 * max(1, len(vals)))()
    for i, v in enumerate(vals):
        arr[i] = int(v)
    return arr


def _span(shape, strides):
    """(lowest, highest) element offset a layout reaches, relative to its base."""
    lo = hi = 0
    for e, s in zip(shape, strides):
        if e <= 0:
            return 0, -1
        if s >= 0:
            hi += (e - 1) * s
        else:
            lo += (e - 1) * s
    return lo, hi


def permute(src: np.ndarray, dst: np.ndarray, shape, src_strides, dst_strides,
            elem_bytes: int, src_offset: int = 0, dst_offset: int = 0,
            nthreads: int = 1) -> None:
    """dst[sum c*dst_strides + dst_offset] = src[sum c*src_strides + src_offset].

    ``src`` and ``dst`` are C-contiguous numpy arrays used as raw byte buffers;
    strides and offsets are in elements of ``elem_bytes`` bytes.  Raises on any
    access outside the buffers (checked before the C loop runs).
    """
    shape = [int(x) for x in shape]
    n = len(shape)
    if len(src_strides) != n or len(dst_strides) != n:
        raise ValueError("shape/stride length mismatch")
    if elem_bytes not in ELEM_BYTES:
        raise ValueError("elem_bytes must be one of %s" % (ELEM_BYTES,))
    for buf in (src, dst):
        if not buf.flags["C_CONTIGUOUS"]:
            raise ValueError("oracle buffers must be C-contiguous")
    if any(e == 0 for e in shape):
        return
    for strides, off, buf in ((src_strides, src_offset, src), (dst_strides, dst_offset, dst)):
        lo, hi = _span(shape, strides)
        if off + lo < 0 or (off + hi + 1) * elem_bytes > buf.nbytes:
            raise IndexError("layout reaches outside its buffer")
    if not dst.flags["WRITEABLE"]:
        raise ValueError("dst is read-only")
    rc = _load().oracle_permute(src.ctypes.data + src_offset * elem_bytes,
                                dst.ctypes.data + dst_offset * elem_bytes, n,
                                _i64(shape), _i64(src_strides), _i64(dst_strides),
                                int(elem_bytes), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_permute rejected its arguments (rc=%d)" % rc)


def sample(src: np.ndarray, coords: np.ndarray, src_strides, dst_strides, elem_bytes: int,
           src_offset: int = 0):
    """The definition at chosen coordinates, one by one.

    ``coords`` is an (n, ndim) integer array.  Returns ``(dst_offsets, values)``:
    for each coordinate c, the element offset sum(c * dst_strides) it lands at and
    the elem_bytes bytes found at src[src_offset + sum(c * src_strides)], as an
    (n, elem_bytes) uint8 array.  For checking outputs too large to permute whole.
    """
    coords = np.asarray(coords, dtype=np.int64)
    ss = np.asarray(src_strides, dtype=np.int64)
    ds = np.asarray(dst_strides, dtype=np.int64)
    src_off = src_offset + coords @ ss
    dst_off = coords @ ds
    byte_idx = src_off[:, None] * elem_bytes + np.arange(elem_bytes, dtype=np.int64)[None, :]
    if byte_idx.size and (byte_idx.min() < 0 or byte_idx.max() >= src.nbytes):
        raise IndexError("sampled coordinate outside the source buffer")
    return dst_off, src.reshape(-1).view(np.uint8)[byte_idx]


def permute_cast(src: np.ndarray, dst: np.ndarray, shape, src_strides, dst_strides, cast: str,
                 src_offset: int = 0, dst_offset: int = 0) -> None:
    """dst[sum c*dst_strides + dst_offset] = convert(src[sum c*src_strides + src_offset])
    for every coordinate c, with ``convert`` one of ``cast_ref.CASTS`` (strides and
    offsets in elements of each side's own type).  Small inputs: the coordinates
    are enumerated."""
    src_eb, dst_eb = cast_ref.CASTS[cast]
    shape = [int(x) for x in shape]
    if any(e == 0 for e in shape):
        return
    coords = np.indices(shape).reshape(len(shape), -1).T.astype(np.int64)
    so = src_offset + coords @ np.asarray(src_strides, dtype=np.int64)
    do = dst_offset + coords @ np.asarray(dst_strides, dtype=np.int64)
    sb = so[:, None] * src_eb + np.arange(src_eb)[None, :]
    db = do[:, None] * dst_eb + np.arange(dst_eb)[None, :]
    if sb.min() < 0 or sb.max() >= src.nbytes or db.min() < 0 or db.max() >= dst.nbytes:
        raise IndexError("layout reaches outside its buffer")
    vals = src.reshape(-1).view(np.uint8)[sb]
    out = cast_ref.convert_bytes(vals, cast).reshape(-1, dst_eb)
    dst.reshape(-1).view(np.uint8)[db] = out
