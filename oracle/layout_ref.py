"""Pure-Python references for the host-side layout logic -- TEST INFRASTRUCTURE ONLY.

Small inputs only (every function enumerates coordinates or lanes).  Each
function names the passage it follows.  Where the pages leave a step open, the
reading taken is stated in the docstring; the same readings are listed in the
project's design notes.

Layout convention: a layout is a tuple of per-axis element strides over a shape,
plus an element offset; coordinate ``c`` maps to ``offset + sum(c[i]*stride[i])``
(TVM docs, "Buffers and memory", section "Declaring buffers").
"""
from __future__ import annotations

import itertools

from itertools import product

WARP = 32           # lanes per warp
BANKS = 32          # shared-memory banks
BANK_BYTES = 4      # bytes per bank word


# ---------------------------------------------------------------------------
# Addressing ("Buffers and memory", "Declaring buffers" and "Buffer APIs")
# ---------------------------------------------------------------------------
def apply(coord, strides, offset=0):
    """Element offset of ``coord``: ``offset + sum(coord[i] * strides[i])``."""
    return offset + sum(c * s for c, s in zip(coord, strides))


def row_major_strides(shape):
    """Dense row-major strides (the page's "default" layout)."""
    out, acc = [], 1
    for e in reversed(shape):
        out.append(acc)
        acc *= e
    return tuple(reversed(out))


def view_permute(shape, strides, dims):
    """``B.permute(*dims)``: the same storage with axes reordered (swapped strides)."""
    return tuple(shape[d] for d in dims), tuple(strides[d] for d in dims)


def slice_layout(shape, strides, offset, begin, extent):
    """Restrict a layout to the box ``[begin, begin+extent)``.

    The sliced layout keeps the strides, takes ``extent`` as its shape and moves
    the offset to the box's first element.
    """
    if len(begin) != len(shape) or len(extent) != len(shape):
        raise ValueError("region rank mismatch")
    for b, e, n in zip(begin, extent, shape):
        if b < 0 or e < 0 or b + e > n:
            raise ValueError("region outside the layout")
    return tuple(extent), tuple(strides), apply(begin, strides, offset)


# ---------------------------------------------------------------------------
# Canonicalisation ("permute_layout", "Algorithm" step 1; "copy_async -> dsmem",
# "Algorithm" step 1)
# ---------------------------------------------------------------------------
def canon_ref(shape, src_strides, dst_strides, begin=None, extent=None,
              src_offset=0, dst_offset=0):
    """Slice both layouts to a region, canonicalise them and regroup src to dst.

    Reading taken (the pages give no rules): after slicing, axes of extent 1 are
    dropped, then adjacent axes (outer i, inner i+1) are merged, keeping their
    order, wherever BOTH sides are contiguous across them, i.e.
    ``stride[i] == extent[i+1] * stride[i+1]`` on src and on dst.  The result is
    src expressed in dst's grouping: one shared extent tuple and the two stride
    tuples.  ``chunk_elems`` is the length of the common stride-1 chain at the
    innermost end (the merge has already folded the whole chain into the last
    axis): the last extent when both last strides are 1, otherwise 0 (no chain).
    A region of one element has no axes and a chunk of 1; an empty region has
    shape (0,) and a chunk of 0.

    Returns a dict with keys extent, src_str, dst_str, src_offset, dst_offset,
    chunk_elems.
    """
    n = len(shape)
    if len(src_strides) != n or len(dst_strides) != n:
        raise ValueError("rank mismatch")
    if begin is None:
        begin = (0,) * n
    if extent is None:
        extent = tuple(s - b for s, b in zip(shape, begin))
    ext, s_str, s_off = slice_layout(shape, src_strides, src_offset, begin, extent)
    _, d_str, d_off = slice_layout(shape, dst_strides, dst_offset, begin, extent)
    if any(e == 0 for e in ext):
        return dict(extent=(0,), src_str=(1,), dst_str=(1,), src_offset=s_off,
                    dst_offset=d_off, chunk_elems=0)
    axes = [(e, s, d) for e, s, d in zip(ext, s_str, d_str) if e != 1]
    merged = []
    for e, s, d in axes:
        if merged and merged[-1][1] == e * s and merged[-1][2] == e * d:
            pe, _, _ = merged.pop()
            merged.append((pe * e, s, d))
        else:
            merged.append((e, s, d))
    if not merged:
        chunk = 1
    elif merged[-1][1] == 1 and merged[-1][2] == 1:
        chunk = merged[-1][0]
    else:
        chunk = 0
    return dict(extent=tuple(m[0] for m in merged), src_str=tuple(m[1] for m in merged),
                dst_str=tuple(m[2] for m in merged), src_offset=s_off, dst_offset=d_off,
                chunk_elems=chunk)


def chunk_admits_bulk_copy(chunk_elems, elem_bytes):
    """The bulk-copy rule of the dsmem page ("Algorithm" step 1): the contiguous
    chunk must be at least 16 bytes and a multiple of 16 bytes."""
    nbytes = chunk_elems * elem_bytes
    return nbytes >= 16 and nbytes % 16 == 0


# ---------------------------------------------------------------------------
# Warp permute ("permute_layout", "Algorithm" steps 2 and 3)
# ---------------------------------------------------------------------------
def decompose(i, extent):
    """Row-major coordinates of flat index ``i`` within ``extent``."""
    out = []
    for e in reversed(extent):
        out.append(i % e)
        i //= e
    return tuple(reversed(out))


def warp_phase_offsets(extent, strides, k, shift, offset=0):
    """Element offsets one warp touches in one phase of the register-staged permute.

    Each lane holds P = prod(extent)/32 registers.  In iteration r the lane
    works on iteration index j = r XOR ((lane >> shift) & mask), mask = 2^k - 1,
    whose coordinates are the row-major decomposition of lane + 32*j over the
    extent; the offset is those coordinates applied to ``strides``.
    Returns a list over r of a list over lanes.
    """
    total = 1
    for e in extent:
        total *= e
    if total % WARP:
        raise ValueError("extent does not split into whole warp iterations")
    P = total // WARP
    mask = (1 << k) - 1
    out = []
    for r in range(P):
        row = []
        for lane in range(WARP):
            j = r ^ ((lane >> shift) & mask)
            row.append(apply(decompose(lane + WARP * j, extent), strides, offset))
        out.append(row)
    return out


def lanes_per_wavefront(elem_bytes):
    """Lanes served together by one shared-memory wavefront of 128 bytes.

    Reading taken: 32 lanes for widths up to 4 bytes, 16 for 8-byte and 8 for
    16-byte accesses (the page only says the simulation is "at shard
    granularity").
    """
    return WARP if elem_bytes <= BANK_BYTES else (BANKS * BANK_BYTES) // elem_bytes


def bank_conflict_degree(lane_offsets, elem_bytes, model="conservative"):
    """Worst bank conflict of one warp-wide access, under the 32 x 4-byte bank model.

    ``lane_offsets[l]`` is the element offset lane l touches (None = idle lane).
    A lane covers the 4-byte words floor(o*w/4) .. floor((o*w+w-1)/4); word x sits
    in bank x mod 32.  Within each wavefront:

    * ``conservative`` (the reading of the permute_layout page): the degree of a
      bank is the number of lanes touching it -- lanes that share a word count as
      a conflict, which is why stride-1 sub-4-byte reads can leave no valid k;
    * ``hardware``: the degree of a bank is the number of DISTINCT words touched
      in it (several lanes reading one word are served by one broadcast).

    Returns the maximum degree over banks and wavefronts (1 = conflict-free,
    0 = no lane active).
    """
    per = lanes_per_wavefront(elem_bytes)
    worst = 0
    for base in range(0, len(lane_offsets), per):
        lanes_in_bank = {}
        words_in_bank = {}
        for lane in range(base, min(base + per, len(lane_offsets))):
            o = lane_offsets[lane]
            if o is None:
                continue
            first = (o * elem_bytes) // BANK_BYTES
            last = (o * elem_bytes + elem_bytes - 1) // BANK_BYTES
            for word in range(first, last + 1):
                bank = word % BANKS
                lanes_in_bank.setdefault(bank, set()).add(lane)
                words_in_bank.setdefault(bank, set()).add(word)
        table = lanes_in_bank if model == "conservative" else words_in_bank
        for members in table.values():
            worst = max(worst, len(members))
    return worst


def phase_is_conflict_free(extent, strides, elem_bytes, k, shift, model="conservative"):
    return all(bank_conflict_degree(lanes, elem_bytes, model) <= 1
               for lanes in warp_phase_offsets(extent, strides, k, shift))


def candidate_xor_params(P):
    """(k, shift) pairs in the order they are tried.

    Reading taken: k ascending over 0 .. log2(P) (only k = 0 when P is not a
    power of two, since an XOR could then leave [0, P)); for each k > 0, shift
    ascending over 0 .. 5-k so the XOR bits come from the 5-bit lane index;
    k = 0 has a single candidate with shift 0.
    """
    kmax = P.bit_length() - 1 if P > 0 and (P & (P - 1)) == 0 else 0
    out = [(0, 0)]
    for k in range(1, kmax + 1):
        for shift in range(0, 5 - k + 1):
            out.append((k, shift))
    return out


def choose_xor_k_ref(extent, src_str, dst_str, elem_bytes, model="conservative"):
    """Smallest (k, shift) whose XOR swizzle leaves BOTH phases conflict-free.

    Returns (k, shift, mask) or None when no candidate works (the warp variant
    then declines) or when prod(extent) is not a whole number of warp
    iterations.
    """
    total = 1
    for e in extent:
        total *= e
    if total == 0 or total % WARP:
        return None
    P = total // WARP
    for k, shift in candidate_xor_params(P):
        if (phase_is_conflict_free(extent, src_str, elem_bytes, k, shift, model) and
                phase_is_conflict_free(extent, dst_str, elem_bytes, k, shift, model)):
            return k, shift, (1 << k) - 1
    return None


def warp_permute_ref(buf_src, buf_dst, extent, src_str, dst_str, k, shift,
                     src_offset=0, dst_offset=0):
    """The two register-staged phases on Python lists, in the page's order.

    All 32 lanes read their P elements (phase 1) before any lane writes (phase
    2), so the routine is correct when ``buf_src is buf_dst``.
    """
    reads = warp_phase_offsets(extent, src_str, k, shift, src_offset)
    writes = warp_phase_offsets(extent, dst_str, k, shift, dst_offset)
    regs = [[buf_src[o] for o in lanes] for lanes in reads]          # phase 1
    for r, lanes in enumerate(writes):                                # phase 2
        for lane, o in enumerate(lanes):
            buf_dst[o] = regs[r][lane]


# ---------------------------------------------------------------------------
# Thread-axis layouts ("Buffers and memory", "Buffer APIs", "Registers -- local")
# ---------------------------------------------------------------------------
def thread_axis_places(shape, lane_strides, reg_strides):
    """Where each coordinate of a warp's thread-axis ``local`` layout lives.

    An axis either carries a stride ``s @ laneid`` (``lane_strides[k] = s``,
    ``reg_strides[k] = 0``) or a plain register stride (``reg_strides[k] = s``,
    ``lane_strides[k] = 0``): coordinate c sits in lane sum(c * lane_strides) and in
    that lane's register sum(c * reg_strides), the "local" slice of the page's
    ``S[(32, 8) : (1 @ laneid, 1)]`` example taken one lane at a time.  Returns
    ``{coord: (lane, register)}`` for every coordinate, row-major."""
    out = {}
    for c in itertools.product(*[range(e) for e in shape]):
        lane = sum(ci * s for ci, s in zip(c, lane_strides))
        reg = sum(ci * s for ci, s in zip(c, reg_strides))
        out[c] = (lane, reg)
    return out


def thread_axis_registers(shape, lane_strides, reg_strides):
    """Registers per lane of a valid thread-axis layout, else None.  Valid: every
    axis on exactly one side, and the map coordinate -> (lane, register) a bijection
    onto 32 lanes x P registers (checked by enumerating it)."""
    if any((ls != 0) == (rs != 0) for ls, rs in zip(lane_strides, reg_strides)):
        return None
    if any(ls < 0 or rs < 0 for ls, rs in zip(lane_strides, reg_strides)):
        return None
    n = 1
    for e in shape:
        n *= e
    if n % 32:
        return None
    P = n // 32
    places = thread_axis_places(shape, lane_strides, reg_strides)
    seen = set(places.values())
    if len(seen) != n or seen != {(l, r) for l in range(32) for r in range(P)}:
        return None
    return P


def thread_axis_fragment(buf, shape, mem_strides, lane_strides, reg_strides, offset=0):
    """Lane l's registers of a thread-axis layout loaded from a memory buffer that
    holds the same logical tensor under ``mem_strides``: an array [32, P] whose
    entry (l, j) is buf[offset + sum(c * mem_strides)] for the coordinate c placed
    in lane l, register j."""
    P = thread_axis_registers(shape, lane_strides, reg_strides)
    if P is None:
        raise ValueError("not a thread-axis layout of one warp")
    out = [[None] * P for _ in range(32)]
    for c, (lane, reg) in thread_axis_places(shape, lane_strides, reg_strides).items():
        out[lane][reg] = buf[offset + apply(c, mem_strides)]
    return out


# ---------------------------------------------------------------------------
# Overlap (no passage: the pages only permute dense tiles)
# ---------------------------------------------------------------------------
def offsets_unique(shape, strides):
    """Brute force: does every coordinate map to a distinct offset?"""
    seen = set()
    for c in product(*[range(e) for e in shape]):
        o = apply(c, strides)
        if o in seen:
            return False
        seen.add(o)
    return True
