"""Seeded synthetic workloads for the layout permute.

This module only describes inputs: shapes, element strides, element widths,
buffer sizes and seeded value generators.  It holds none of the permute's
arithmetic, so both the CUDA path and the CPU oracle can take their inputs from
it without sharing any method code.

All values come from ``numpy.random.Generator(PCG64(seed))`` on the host, so a
given seed yields the same bytes on x86 and Arm.

The five workloads follow the scale-factor (SF) tile and the 128x64 float16
tile that the TVM pages use as worked examples ("permute_layout",
"Demonstration program"; "copy_async -> dsmem", "Demonstration program"),
grown to sizes that exercise HBM:

=================  =========================================================
``sf_transpose``   float32 (pipe=2, high=1, 4, 32): strides (128,128,32,1) ->
                   (128,128,1,4); one warp's worth of work per stage.
``tile_transpose`` 65536 float16 tiles of 128x64, row-major -> column-major per
                   tile (1 GiB); N(0,1) with 0.1 % NaN / Inf bit patterns.
``mx_sf``          uint8 (2^20, 2, 4, 32): strides (256,128,32,1) ->
                   (256,128,1,4); random bytes (256 MiB).
``attention``      bfloat16 (B=16, H=32, S=4096, D=128) -> (B, S, H, D)
                   contiguous (512 MiB).
``t2d_u8`` ...     2-D row-major -> column-major transposes of ~1 GiB for each
                   element width 1, 2, 4, 8, 16 bytes; random bits.
=================  =========================================================

Three more describe general permutes whose layouts a TMA tensor map cannot take
(the ``B.permute`` case of "Buffers and memory", "Buffer APIs"):

=================  =========================================================
``t2d_odd_f32``    float32 16383 x 16385 row-major -> column-major: row pitches
                   that are not multiples of 16 bytes (1 GiB).
``t2d_odd_u8``     uint8 32767 x 32769 row-major -> column-major: odd row pitches
                   on both sides (1 GiB).
``hwc_chw_u8``     uint8 image 8192 x 8192 x 3 channels (HWC) -> 3 planes (CHW).
``nd6_f32``        float32 (16,16,16,16,64,64) permuted (5,3,1,4,2,0): four
                   batch axes around the transposed plane (1 GiB).
``nd8_f32``        float32 (9,)*8 permuted (1,4,2,3,7,5,6,0): a high-rank permute
                   of short axes whose src- and dst-contiguous axes are 36 bytes
                   long (172 MB).
``nd8_u16``        uint16 (12,)*8 permuted (7,5,3,1,0,2,4,6): the interleaved
                   order of twelve-element axes, runs of 24 bytes (860 MB).
=================  =========================================================
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = ["Workload", "WORKLOADS", "get", "scaled", "make_input", "random_bits"]


@dataclass(frozen=True)
class Workload:
    name: str
    elem_bytes: int
    shape: tuple
    src_strides: tuple
    dst_strides: tuple
    src_elems: int          # size of the source buffer, in elements
    dst_elems: int          # size of the destination buffer, in elements
    seed: int
    values: str             # "uniform_pm1_f32" | "normal_f16_naninf" | "bits" | "normal_bf16"
    description: str = ""
    tags: tuple = field(default_factory=tuple)

    @property
    def n_elems(self) -> int:
        n = 1
        for e in self.shape:
            n *= e
        return n

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes read plus bytes written by one permute: each element once each way."""
        return 2 * self.n_elems * self.elem_bytes


def _t2d(name, eb, rows, cols, seed):
    return Workload(name, eb, (rows, cols), (cols, 1), (1, rows), rows * cols, rows * cols,
                    seed, "bits",
                    "%d-byte %dx%d row-major -> column-major" % (eb, rows, cols), ("t2d",))


def _rm(shape):
    st, acc = [], 1
    for e in reversed(shape):
        st.append(acc)
        acc *= e
    return tuple(reversed(st))


def _perm_dst(shape, perm):
    # dst holds the axes in the order `perm`, row-major: stride of source axis perm[i]
    pst = _rm(tuple(shape[p] for p in perm))
    ds = [0] * len(shape)
    for i, p in enumerate(perm):
        ds[p] = pst[i]
    return tuple(ds)


def _hwc_chw(h, w=8192, c=3):
    # (H, W, C) interleaved -> C planes of H x W
    return Workload("hwc_chw_u8", 1, (h, w, c), (w * c, c, 1), (w, 1, h * w), h * w * c,
                    h * w * c, 56, "bits",
                    "uint8 %dx%dx%d interleaved channels -> %d planes" % (h, w, c, c),
                    ("general",))


def _nd6(lead):
    shape = (lead, 16, 16, 16, 64, 64)
    n = lead * 16 * 16 * 16 * 64 * 64
    return Workload("nd6_f32", 4, shape, _rm(shape), _perm_dst(shape, (5, 3, 1, 4, 2, 0)), n, n,
                    57, "bits", "float32 %s permuted (5,3,1,4,2,0)" % (shape,), ("general",))


def _nd8(lead):
    shape = (lead,) + (9,) * 7
    n = lead * 9 ** 7
    return Workload("nd8_f32", 4, shape, _rm(shape), _perm_dst(shape, (1, 4, 2, 3, 7, 5, 6, 0)),
                    n, n, 58, "bits", "float32 %s permuted (1,4,2,3,7,5,6,0)" % (shape,),
                    ("general",))


def _nd8_u16(lead):
    shape = (lead,) + (12,) * 7
    n = lead * 12 ** 7
    return Workload("nd8_u16", 2, shape, _rm(shape), _perm_dst(shape, (7, 5, 3, 1, 0, 2, 4, 6)),
                    n, n, 59, "bits", "uint16 %s permuted (7,5,3,1,0,2,4,6)" % (shape,),
                    ("general",))


WORKLOADS = {
    w.name: w for w in [
        Workload("sf_transpose", 4, (2, 1, 4, 32), (128, 128, 32, 1), (128, 128, 1, 4),
                 256, 256, 1, "uniform_pm1_f32",
                 "float32 SF-transpose worked example, one warp per pipe stage", ("small",)),
        Workload("tile_transpose", 2, (65536, 128, 64), (8192, 64, 1), (8192, 1, 128),
                 65536 * 8192, 65536 * 8192, 2, "normal_f16_naninf",
                 "65536 float16 tiles of 128x64, row-major -> column-major per tile"),
        Workload("mx_sf", 1, (1 << 20, 2, 4, 32), (256, 128, 32, 1), (256, 128, 1, 4),
                 1 << 28, 1 << 28, 3, "bits",
                 "uint8 MX scale-factor tiles, 4x32 -> 32x4 per 128-byte block"),
        Workload("attention", 2, (16, 32, 4096, 128), (1 << 24, 1 << 19, 128, 1),
                 (1 << 24, 128, 4096, 1), 1 << 28, 1 << 28, 4, "normal_bf16",
                 "bfloat16 (B,H,S,D) -> (B,S,H,D) contiguous"),
        _t2d("t2d_u8", 1, 32768, 32768, 50),
        _t2d("t2d_f16", 2, 16384, 32768, 51),
        _t2d("t2d_f32", 4, 16384, 16384, 52),
        _t2d("t2d_f64", 8, 8192, 16384, 53),
        _t2d("t2d_v16", 16, 8192, 8192, 54),
        _t2d("t2d_odd_f32", 4, 16383, 16385, 55),
        _t2d("t2d_odd_u8", 1, 32767, 32769, 60),
        _hwc_chw(8192),
        _nd6(16),
        _nd8(9),
        _nd8_u16(12),
    ]
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def scaled(w: Workload, leading: int) -> Workload:
    """The same workload with its outermost extent set to ``leading`` (a smaller
    case for profiling).  The 2-D transposes keep their column count and
    recompute their column-major destination strides; the batched workloads keep
    their strides."""
    if leading < 1:
        raise ValueError("leading extent must be positive")
    if "t2d" in w.tags:
        rows, cols = leading, w.shape[1]
        return _t2d(w.name, w.elem_bytes, rows, cols, w.seed)
    if w.name == "hwc_chw_u8":          # dst plane size follows the leading extent
        return _hwc_chw(leading, w.shape[1], w.shape[2])
    if w.name == "nd6_f32":             # the leading axis is innermost in dst
        return _nd6(leading)
    if w.name == "nd8_f32":             # the leading axis is innermost in dst
        return _nd8(leading)
    if w.name == "nd8_u16":             # the leading axis sits inside dst's order
        return _nd8_u16(leading)
    ratio_src = w.src_elems // w.shape[0]
    ratio_dst = w.dst_elems // w.shape[0]
    return Workload(w.name, w.elem_bytes, (leading,) + tuple(w.shape[1:]), w.src_strides,
                    w.dst_strides, leading * ratio_src, leading * ratio_dst, w.seed, w.values,
                    w.description + " (outermost extent %d)" % leading, w.tags)


def random_bits(n_bytes: int, seed: int) -> np.ndarray:
    """``n_bytes`` uniformly random bytes from ``seed``."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.frombuffer(rng.bytes(n_bytes), dtype=np.uint8).copy()


def _normal_f32(n, rng, chunk=1 << 24):
    out = np.empty(n, dtype=np.float32)
    for i in range(0, n, chunk):
        out[i:i + chunk] = rng.standard_normal(min(chunk, n - i), dtype=np.float32)
    return out


def make_values(kind: str, n_elems: int, elem_bytes: int, seed: int) -> np.ndarray:
    """A uint8 buffer of ``n_elems`` elements of ``elem_bytes`` bytes, by value kind.

    * ``bits`` -- uniformly random bytes.
    * ``uniform_pm1_f32`` -- float32 uniform on [-1, 1).
    * ``normal_bf16`` -- N(0,1) float32 truncated to its upper 16 bits (bfloat16).
    * ``normal_f16_naninf`` -- N(0,1) as float16, then 0.1 % of the elements
      replaced by NaN patterns (exponent all ones, random non-zero mantissa,
      random sign) or +/-Inf, half each.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    if kind == "bits":
        return np.frombuffer(rng.bytes(n_elems * elem_bytes), dtype=np.uint8).copy()
    if kind == "uniform_pm1_f32":
        assert elem_bytes == 4
        v = rng.uniform(-1.0, 1.0, size=n_elems).astype(np.float32)
        return v.view(np.uint8).copy()
    if kind == "normal_bf16":
        assert elem_bytes == 2
        v = _normal_f32(n_elems, rng).view(np.uint32)
        return (v >> 16).astype(np.uint16).view(np.uint8).copy()
    if kind == "normal_f16_naninf":
        assert elem_bytes == 2
        v = _normal_f32(n_elems, rng).astype(np.float16).view(np.uint16)
        n_special = max(1, n_elems // 1000)
        idx = rng.choice(n_elems, size=n_special, replace=False) if n_elems < (1 << 22) \
            else rng.integers(0, n_elems, size=n_special)
        sign = rng.integers(0, 2, size=n_special).astype(np.uint16) << 15
        mant = rng.integers(1, 1 << 10, size=n_special).astype(np.uint16)
        is_nan = rng.integers(0, 2, size=n_special).astype(bool)
        special = np.where(is_nan, sign | 0x7C00 | mant, sign | 0x7C00).astype(np.uint16)
        v[idx] = special
        return v.view(np.uint8).copy()
    raise ValueError("unknown value kind %r" % kind)


def make_input(w: Workload, seed: int | None = None) -> np.ndarray:
    """The source buffer of workload ``w`` as raw bytes."""
    return make_values(w.values, w.src_elems, w.elem_bytes, w.seed if seed is None else seed)
