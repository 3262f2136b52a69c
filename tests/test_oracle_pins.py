"""Pins for the CPU oracle: it is checked against what the pages and mathematics fix.

Nothing here compares the oracle with itself.  The pins are: index expressions
and swizzle parameters the TVM pages print for their worked examples (fixtures in
``tests/golden``), numpy's own transpose machinery (a library routine that a
strided permute reduces to), closed-form invariants (bijection, inverse, memcpy
on identity strides), textbook shared-memory bank facts, and brute force on tiny
layouts.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import layout_ref as L
from tests.conftest import read_golden

NP_BY_WIDTH = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64, 16: np.dtype("V16")}


def _bytes(a):
    return np.ascontiguousarray(a).view(np.uint8).reshape(-1)


def _perm_layouts(shape, perm):
    """src row-major over ``shape``; dst = the row-major array of shape shape[perm]."""
    src = L.row_major_strides(shape)
    pst = L.row_major_strides(tuple(shape[p] for p in perm))
    dst = [0] * len(shape)
    for i, p in enumerate(perm):
        dst[p] = pst[i]
    return src, tuple(dst)


def _eval(expr, **env):
    return eval(expr, {"__builtins__": {}}, env)


# ---------------------------------------------------------------------------
# Addressing: "Buffers and memory", "Declaring buffers" and "Buffer APIs"
# ---------------------------------------------------------------------------
def test_buffer_addressing_4x8_matches_page():
    rows, _ = read_golden("buffer_addressing_4x8.txt")
    assert len(rows) == 4
    a = np.arange(32, dtype=np.uint32)          # A is row-major 4x8: A[i,j] at i*8+j
    for name, strides, off, expr in rows:
        strides = tuple(int(x) for x in strides.split())
        off = int(off)
        for i in range(4):
            for j in range(8):
                assert L.apply((i, j), strides, off) == _eval(expr, i=i, j=j), name
        # B[i, j] = A[i, j] through the oracle permute lands where the page says
        dst = np.zeros(off + 64, dtype=np.uint32)
        oracle.permute(a, dst, (4, 8), (8, 1), strides, 4, dst_offset=off)
        for i in range(4):
            for j in range(8):
                assert dst[_eval(expr, i=i, j=j)] == i * 8 + j, name


def test_view_and_permute_index_forms_match_page():
    rows, _ = read_golden("buffer_view_permute.txt")
    ops = {r[0]: r for r in rows}
    base_shape = (64, 4)
    base = L.row_major_strides(base_shape)
    _, _, _, expr = ops["view_64x4"]
    for tx in range(64):
        for j in range(4):
            assert L.apply((tx, j), base) == _eval(expr, tx=tx, j=j)
    _, _, _, expr = ops["permute_10"]
    pshape, pstr = L.view_permute(base_shape, base, (1, 0))
    assert pshape == (4, 64)
    for i in range(4):
        for j in range(64):
            assert L.apply((i, j), pstr) == _eval(expr, i=i, j=j)


# ---------------------------------------------------------------------------
# Warp permute worked example: "permute_layout" demonstration, Algorithm, IR
# ---------------------------------------------------------------------------
def _sf():
    _, kv = read_golden("sf_transpose_warp.txt")
    ints = lambda k: tuple(int(x) for x in kv[k].split())
    return kv, ints


def test_sf_canon_per_stage_matches_page():
    kv, ints = _sf()
    shape, s_str, d_str = ints("shape"), ints("src_strides"), ints("dst_strides")
    for s in range(shape[0]):
        c = L.canon_ref(shape, s_str, d_str, begin=(s, 0, 0, 0), extent=(1, 1, 4, 32))
        assert c["extent"] == ints("extent")
        assert c["src_str"] == (32, 1) and c["dst_str"] == (1, 4)
        assert c["src_offset"] == 128 * s and c["dst_offset"] == 128 * s
        assert c["chunk_elems"] == 0           # row vs column: no common chain
        P = (4 * 32) // 32
        assert P == int(kv["P"])


def test_sf_choose_xor_k_matches_page():
    kv, ints = _sf()
    want = (2, int(kv["shift"]), int(kv["mask"]))
    assert want == (2, 3, 3)
    for model in ("conservative", "hardware"):
        assert L.choose_xor_k_ref(ints("extent"), (32, 1), (1, 4), 4, model) == want


def test_sf_phase_offsets_match_printed_ir():
    kv, ints = _sf()
    for s in range(2):
        reads = L.warp_phase_offsets(ints("extent"), (32, 1), 2, 3, offset=128 * s)
        writes = L.warp_phase_offsets(ints("extent"), (1, 4), 2, 3, offset=128 * s)
        for r in range(4):
            for tx in range(32):
                assert reads[r][tx] == _eval(kv["phase1_src"], s=s, r=r, tx=tx)
                assert writes[r][tx] == _eval(kv["phase2_dst"], s=s, r=r, tx=tx)


def test_sf_unswizzled_write_is_4way_and_swizzled_is_free():
    # lanes tx, tx+8, tx+16, tx+24 write words 4*tx + r: same bank without the XOR
    writes = L.warp_phase_offsets((4, 32), (1, 4), 0, 0)
    assert max(L.bank_conflict_degree(w, 4) for w in writes) == 4
    writes = L.warp_phase_offsets((4, 32), (1, 4), 2, 3)
    assert max(L.bank_conflict_degree(w, 4) for w in writes) == 1
    # k = 1 cannot work: four lanes share a bank group, an XOR of one bit gives two values
    for shift in range(5):
        writes = L.warp_phase_offsets((4, 32), (1, 4), 1, shift)
        assert max(L.bank_conflict_degree(w, 4) for w in writes) >= 2


def test_sf_oracle_output_is_transposed_block_per_stage():
    kv, ints = _sf()
    from movement_tl_permute_gb300 import workloads
    w = workloads.get("sf_transpose")
    src = workloads.make_input(w)
    dst = np.zeros_like(src)
    oracle.permute(src, dst, ints("shape"), ints("src_strides"), ints("dst_strides"), 4)
    a = src.view(np.float32).reshape(2, 4, 32)
    want = np.ascontiguousarray(a.transpose(0, 2, 1)).reshape(-1)
    assert np.array_equal(dst.view(np.uint32), want.view(np.uint32))


def test_warp_two_phase_in_place_equals_out_of_place():
    rng = np.random.default_rng(7)
    buf = list(rng.integers(0, 2**31, size=256))
    ref = np.array(buf, dtype=np.int64)
    want = np.zeros(256, dtype=np.int64)
    oracle.permute(ref, want, (2, 4, 32), (128, 32, 1), (128, 1, 4), 8)
    for s in range(2):
        L.warp_permute_ref(buf, buf, (4, 32), (32, 1), (1, 4), 2, 3, 128 * s, 128 * s)
    assert buf == list(want)


# ---------------------------------------------------------------------------
# Contiguous chunk: "copy_async -> dsmem", Algorithm step 1 and worked example
# ---------------------------------------------------------------------------
def test_dsmem_chunk_cases_match_page():
    rows, _ = read_golden("dsmem_chunk.txt")
    for name, shape, ss, ds, eb, chunk, cbytes, admitted in rows:
        shape = tuple(int(x) for x in shape.split())
        ss = tuple(int(x) for x in ss.split())
        ds = tuple(int(x) for x in ds.split())
        c = L.canon_ref(shape, ss, ds)
        assert c["chunk_elems"] == int(chunk), name
        assert c["chunk_elems"] * int(eb) == int(cbytes), name
        assert L.chunk_admits_bulk_copy(c["chunk_elems"], int(eb)) == (admitted == "yes"), name


def test_chunk_rule_small_and_unaligned_decline():
    # padded source rows stop the merge; the common chain is one row
    c = L.canon_ref((8, 4), (8, 1), (4, 1))
    assert c["chunk_elems"] == 4
    assert not L.chunk_admits_bulk_copy(4, 2)          # 8 bytes < 16
    c = L.canon_ref((8, 24), (32, 1), (24, 1))
    assert c["chunk_elems"] == 24
    assert not L.chunk_admits_bulk_copy(24, 1)         # 24 bytes, not a multiple of 16
    assert L.chunk_admits_bulk_copy(16, 1) and L.chunk_admits_bulk_copy(8, 2)


def test_canon_of_the_large_workloads():
    # MX scale factors: (2^20, 2, 4, 32) merges the two outer axes on both sides
    c = L.canon_ref((1 << 20, 2, 4, 32), (256, 128, 32, 1), (256, 128, 1, 4))
    assert c["extent"] == (1 << 21, 4, 32)
    assert c["src_str"] == (128, 32, 1) and c["dst_str"] == (128, 1, 4)
    # attention (B,H,S,D) -> (B,S,H,D): nothing merges; the D chain is common
    c = L.canon_ref((16, 32, 4096, 128), (1 << 24, 1 << 19, 128, 1), (1 << 24, 128, 4096, 1))
    assert c["extent"] == (16, 32, 4096, 128) and c["chunk_elems"] == 128
    # identical dense layouts collapse to one axis
    c = L.canon_ref((3, 5, 7), (35, 7, 1), (35, 7, 1))
    assert c["extent"] == (105,) and c["chunk_elems"] == 105
    # a single element and an empty region
    assert L.canon_ref((1, 1), (5, 1), (1, 9))["extent"] == ()
    assert L.canon_ref((1, 1), (5, 1), (1, 9))["chunk_elems"] == 1
    assert L.canon_ref((4, 0), (1, 4), (1, 4))["chunk_elems"] == 0


def test_canon_preserves_the_permutation():
    # Canonicalising must not change which source element lands where.
    rng = np.random.default_rng(3)
    for _ in range(60):
        nd = int(rng.integers(1, 5))
        shape = tuple(int(x) for x in rng.integers(1, 5, size=nd))
        perm = tuple(rng.permutation(nd))
        ss, ds = _perm_layouts(shape, perm)
        c = L.canon_ref(shape, ss, ds)
        n = int(np.prod(shape))
        a = np.arange(n, dtype=np.uint32)
        d1 = np.zeros(n, dtype=np.uint32)
        d2 = np.zeros(n, dtype=np.uint32)
        oracle.permute(a, d1, shape, ss, ds, 4)
        oracle.permute(a, d2, c["extent"], c["src_str"], c["dst_str"], 4)
        assert np.array_equal(d1, d2)


# ---------------------------------------------------------------------------
# The permute itself against numpy's transpose (library routine)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("eb", [1, 2, 4, 8, 16])
def test_permute_equals_numpy_transpose(eb):
    rng = np.random.default_rng(11 + eb)
    dt = NP_BY_WIDTH[eb]
    for _ in range(25):
        nd = int(rng.integers(1, 6))
        shape = tuple(int(x) for x in rng.integers(1, 7, size=nd))
        perm = tuple(int(p) for p in rng.permutation(nd))
        n = int(np.prod(shape))
        raw = np.frombuffer(rng.bytes(n * eb), dtype=np.uint8).copy()
        a = raw.view(dt).reshape(shape)
        want = _bytes(np.transpose(a, perm))
        ss, ds = _perm_layouts(shape, perm)
        got = np.zeros(n * eb, dtype=np.uint8)
        oracle.permute(raw, got, shape, ss, ds, eb)
        assert np.array_equal(got, want), (shape, perm)


@pytest.mark.parametrize("eb", [1, 4, 16])
def test_permute_with_padded_strides_and_offsets_equals_numpy(eb):
    """A strided, offset source view (numpy as_strided) gathered into a dense dst."""
    rng = np.random.default_rng(5 * eb)
    dt = NP_BY_WIDTH[eb]
    for _ in range(20):
        nd = int(rng.integers(1, 5))
        shape = tuple(int(x) for x in rng.integers(1, 6, size=nd))
        # padded row-major source: each axis gets slack
        pad = [int(x) for x in rng.integers(0, 3, size=nd)]
        strides, acc = [], 1
        for e, p in zip(reversed(shape), reversed(pad)):
            strides.append(acc)
            acc *= e + p
        strides = tuple(reversed(strides))
        off = int(rng.integers(0, 5))
        total = off + acc
        raw = np.frombuffer(rng.bytes(total * eb), dtype=np.uint8).copy()
        typed = raw.view(dt)
        view = np.lib.stride_tricks.as_strided(typed[off:], shape=shape,
                                               strides=tuple(s * eb for s in strides))
        perm = tuple(int(p) for p in rng.permutation(nd))
        want = _bytes(np.transpose(view, perm))
        _, ds = _perm_layouts(shape, perm)
        got = np.zeros(int(np.prod(shape)) * eb, dtype=np.uint8)
        oracle.permute(raw, got, shape, strides, ds, eb, src_offset=off)
        assert np.array_equal(got, want)


def test_permute_invariants():
    rng = np.random.default_rng(21)
    for _ in range(30):
        nd = int(rng.integers(2, 6))
        shape = tuple(int(x) for x in rng.integers(1, 6, size=nd))
        perm = tuple(int(p) for p in rng.permutation(nd))
        n = int(np.prod(shape))
        iota = np.arange(n, dtype=np.uint32)
        ss, ds = _perm_layouts(shape, perm)
        out = np.zeros(n, dtype=np.uint32)
        oracle.permute(iota, out, shape, ss, ds, 4)
        assert np.array_equal(np.sort(out), iota)                 # bijection
        # the inverse permutation brings it back
        pshape = tuple(shape[p] for p in perm)
        inv = tuple(int(i) for i in np.argsort(perm))
        ss2, ds2 = _perm_layouts(pshape, inv)
        back = np.zeros(n, dtype=np.uint32)
        oracle.permute(out, back, pshape, ss2, ds2, 4)
        assert np.array_equal(back, iota)
        # identity strides are a memcpy
        same = np.zeros(n, dtype=np.uint32)
        oracle.permute(iota, same, shape, ss, ss, 4)
        assert np.array_equal(same, iota)


def test_transpose_twice_is_identity():
    rng = np.random.default_rng(2)
    for eb in (1, 2, 4, 8, 16):
        r, c = 37, 53
        raw = np.frombuffer(rng.bytes(r * c * eb), dtype=np.uint8).copy()
        t = np.zeros_like(raw)
        tt = np.zeros_like(raw)
        oracle.permute(raw, t, (r, c), (c, 1), (1, r), eb)
        oracle.permute(t, tt, (c, r), (r, 1), (1, c), eb)
        assert np.array_equal(tt, raw)


def test_threads_split_gives_identical_bytes():
    rng = np.random.default_rng(4)
    shape, ss, ds = (64, 33, 17), (33 * 17, 17, 1), (1, 64 * 17, 64)
    n = 64 * 33 * 17
    raw = np.frombuffer(rng.bytes(n * 2), dtype=np.uint8).copy()
    one = np.zeros_like(raw)
    many = np.zeros_like(raw)
    oracle.permute(raw, one, shape, ss, ds, 2, nthreads=1)
    oracle.permute(raw, many, shape, ss, ds, 2, nthreads=4)
    assert np.array_equal(one, many)


def test_oracle_guards():
    a = np.zeros(16, dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle.permute(a, a.copy(), (4,), (1,), (1,), 3)
    with pytest.raises(IndexError):
        oracle.permute(a, a.copy(), (4,), (6,), (1,), 1)
    b = a.copy()
    oracle.permute(a, b, (0, 4), (4, 1), (4, 1), 1)                # empty: no-op
    assert not b.any()


# ---------------------------------------------------------------------------
# Bank model: textbook facts about 32 banks of 4 bytes
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("eb,stride,conservative,hardware", [
    (4, 1, 1, 1),      # consecutive words: conflict-free
    (4, 2, 2, 2),      # every other word: 2-way
    (4, 32, 32, 32),   # one column of a 32-wide array: 32-way
    (4, 33, 1, 1),     # padded column: conflict-free
    (8, 1, 1, 1),      # 16 lanes x 8 B per wavefront
    (8, 2, 2, 2),
    (16, 1, 1, 1),     # 8 lanes x 16 B per wavefront
    (16, 2, 2, 2),
    (2, 1, 2, 1),      # two halves of a word: broadcast in hardware
    (1, 1, 4, 1),      # four bytes of a word
    (1, 4, 1, 1),
    (1, 128, 32, 32),  # every lane in bank 0, distinct words
])
def test_bank_degree_textbook(eb, stride, conservative, hardware):
    lanes = [l * stride for l in range(32)]
    assert L.bank_conflict_degree(lanes, eb, "conservative") == conservative
    assert L.bank_conflict_degree(lanes, eb, "hardware") == hardware


def test_bank_degree_against_byte_level_brute_force():
    """Recount conflicts byte by byte, independently of the word arithmetic."""
    rng = np.random.default_rng(9)
    for _ in range(200):
        eb = int(rng.choice([1, 2, 4, 8, 16]))
        offs = [int(x) for x in rng.integers(0, 300, size=32)]
        per = 32 if eb <= 4 else 128 // eb
        want_c = want_h = 0
        for base in range(0, 32, per):
            owners, words = {}, {}
            for lane in range(base, base + per):
                for byte in range(offs[lane] * eb, offs[lane] * eb + eb):
                    bank = (byte >> 2) & 31
                    owners.setdefault(bank, set()).add(lane)
                    words.setdefault(bank, set()).add(byte >> 2)
            want_c = max([want_c] + [len(v) for v in owners.values()])
            want_h = max([want_h] + [len(v) for v in words.values()])
        assert L.bank_conflict_degree(offs, eb, "conservative") == want_c
        assert L.bank_conflict_degree(offs, eb, "hardware") == want_h


def test_chooser_is_the_first_valid_candidate_by_exhaustion():
    """Try every (k, shift) on tiny layouts; the chooser must return the first that
    leaves both phases conflict-free, and None when none does."""
    cases = [((4, 32), (32, 1), (1, 4), 4), ((2, 64), (64, 1), (1, 2), 4),
             ((8, 16), (16, 1), (1, 8), 4), ((4, 32), (32, 1), (1, 4), 8),
             ((4, 32), (32, 1), (1, 4), 1), ((32,), (1,), (1,), 4),
             ((16, 8), (8, 1), (1, 16), 2), ((4, 8, 4), (32, 4, 1), (1, 16, 4), 4)]
    for extent, ss, ds, eb in cases:
        P = int(np.prod(extent)) // 32
        valid = []
        for k in range(0, 6):
            for shift in range(0, 6):
                if (1 << k) > P or (k == 0 and shift > 0) or shift + k > 5:
                    continue
                ok = all(max(L.bank_conflict_degree(lanes, eb) for lanes in ph) <= 1
                         for ph in (L.warp_phase_offsets(extent, ss, k, shift),
                                    L.warp_phase_offsets(extent, ds, k, shift)))
                if ok:
                    valid.append((k, shift))
        got = L.choose_xor_k_ref(extent, ss, ds, eb)
        if valid:
            k, shift = min(valid)
            assert got == (k, shift, (1 << k) - 1), (extent, eb)
        else:
            assert got is None, (extent, eb)


def test_sub_4_byte_stride_one_reads_can_leave_no_valid_k():
    # the page: stride-1 sub-4-byte reads can pack lanes into one bank and make the
    # variant decline.  With P = 1 there is no XOR to spread them.
    assert L.choose_xor_k_ref((32,), (1,), (1,), 1) is None
    assert L.choose_xor_k_ref((32,), (1,), (1,), 2) is None
    assert L.choose_xor_k_ref((64,), (1,), (1,), 2) == (1, 0, 1)
    # the hardware model lets same-word reads broadcast
    assert L.choose_xor_k_ref((32,), (1,), (1,), 1, "hardware") == (0, 0, 0)
    # with P = 4 the XOR moves the four lanes of a word into four different rows
    assert L.choose_xor_k_ref((4, 32), (32, 1), (1, 4), 1) == (2, 0, 3)
    assert L.choose_xor_k_ref((4, 32), (32, 1), (1, 4), 1, "hardware") == (0, 0, 0)


def test_four_byte_claim_by_brute_force():
    """The page says 4-byte types always admit a valid k.  Brute force over dense
    2-D transposes of power-of-two extents (prod = 32*P, P <= 32) confirms it;
    for 3-D layouts it fails on full axis reversals such as (2, 32, 2) -> (2, 32, 2)
    reversed, where the needed XOR bit does not line up with a contiguous lane
    field.  Both findings are recorded here."""
    count = 0
    for P in (1, 2, 4, 8, 16, 32):
        for e0 in range(1, 11):
            e1 = (32 * P).bit_length() - 1 - e0
            if e1 < 1:
                continue
            extent = (1 << e0, 1 << e1)
            for perm in ((0, 1), (1, 0)):
                ss, ds = _perm_layouts(extent, perm)
                assert L.choose_xor_k_ref(extent, ss, ds, 4) is not None, extent
                count += 1
    assert count == 78
    ss, ds = _perm_layouts((2, 32, 2), (2, 1, 0))
    assert L.choose_xor_k_ref((2, 32, 2), ss, ds, 4) is None
    ss, ds = _perm_layouts((2, 32, 2), (1, 0, 2))
    assert L.choose_xor_k_ref((2, 32, 2), ss, ds, 4) is not None


# ---------------------------------------------------------------------------
# Overlap brute force
# ---------------------------------------------------------------------------
def test_offsets_unique_brute_force():
    assert L.offsets_unique((4, 8), (8, 1))
    assert L.offsets_unique((2, 3), (3, 2))            # interleaved but distinct
    assert not L.offsets_unique((4, 8), (4, 1))
    assert not L.offsets_unique((3,), (0,))
    assert L.offsets_unique((1, 5), (0, 1))


def test_sample_agrees_with_whole_permute():
    """The one-by-one sampler against the whole-tensor loop and numpy."""
    rng = np.random.default_rng(31)
    for eb in (1, 2, 16):
        shape, perm = (5, 7, 3), (2, 0, 1)
        ss, ds = _perm_layouts(shape, perm)
        n = int(np.prod(shape))
        raw = np.frombuffer(rng.bytes(n * eb), dtype=np.uint8).copy()
        whole = np.zeros_like(raw)
        oracle.permute(raw, whole, shape, ss, ds, eb)
        coords = np.array(list(itertools.product(*[range(e) for e in shape])))
        offs, vals = oracle.sample(raw, coords, ss, ds, eb)
        got = whole.reshape(-1, eb)[offs]
        assert np.array_equal(got, vals)
        assert sorted(offs.tolist()) == list(range(n))            # a bijection


@pytest.mark.parametrize("eb", [1, 2, 4, 8, 16])
def test_sample_with_offset_and_padded_strides_equals_numpy(eb):
    """The sampler's src_offset: a padded, offset source view (numpy as_strided) read
    at every coordinate, against numpy's own view of the same bytes and against the
    whole-tensor loop given the same offset ("Buffers and memory", "Declaring
    buffers": the address is data + elem_offset + the layout's offset of c)."""
    rng = np.random.default_rng(7 * eb + 1)
    dt = NP_BY_WIDTH[eb]
    for _ in range(12):
        nd = int(rng.integers(1, 5))
        shape = tuple(int(x) for x in rng.integers(1, 6, size=nd))
        pad = [int(x) for x in rng.integers(0, 3, size=nd)]
        strides, acc = [], 1
        for e, p in zip(reversed(shape), reversed(pad)):
            strides.append(acc)
            acc *= e + p
        strides = tuple(reversed(strides))
        off = int(rng.integers(1, 9))
        raw = np.frombuffer(rng.bytes((off + acc) * eb), dtype=np.uint8).copy()
        view = np.lib.stride_tricks.as_strided(raw.view(dt)[off:], shape=shape,
                                               strides=tuple(s * eb for s in strides))
        perm = tuple(int(p) for p in rng.permutation(nd))
        _, ds = _perm_layouts(shape, perm)
        coords = np.array(list(itertools.product(*[range(e) for e in shape])),
                          dtype=np.int64).reshape(-1, nd)
        offs, vals = oracle.sample(raw, coords, strides, ds, eb, src_offset=off)
        # numpy reads element c of the offset view directly
        want_vals = np.stack([_bytes(view[tuple(c)]) for c in coords])
        assert np.array_equal(vals, want_vals)
        # the dst offsets are those of the transposed dense output
        want = _bytes(np.transpose(view, perm))
        got = np.zeros(int(np.prod(shape)) * eb, dtype=np.uint8)
        got.reshape(-1, eb)[offs] = vals
        assert np.array_equal(got, want)
        # and the sampler agrees with the whole-tensor loop at the same offset
        whole = np.zeros_like(got)
        oracle.permute(raw, whole, shape, strides, ds, eb, src_offset=off)
        assert np.array_equal(whole, got)
        # an offset of zero reads different bytes (the offset is not ignored)
        _, vals0 = oracle.sample(raw, coords, strides, ds, eb, src_offset=0)
        want0 = np.lib.stride_tricks.as_strided(raw.view(dt), shape=shape,
                                                strides=tuple(s * eb for s in strides))
        assert np.array_equal(vals0, np.stack([_bytes(want0[tuple(c)]) for c in coords]))


# ---------------------------------------------------------------------------
# thread-axis ("1 @ laneid") layouts and the lane's local registers
# ---------------------------------------------------------------------------
def test_thread_axis_page_example():
    """The page's S[(32, 8) : (1 @ laneid, 1)] with R.local(8): 8 registers per lane,
    element (l, j) in register j of lane l (tests/golden/thread_axis_local.txt)."""
    rows, kv = read_golden("thread_axis_local.txt")
    shape = tuple(int(x) for x in kv["shape"].split())
    ls = tuple(int(x) for x in kv["lane_strides"].split())
    rs = tuple(int(x) for x in kv["reg_strides"].split())
    assert L.thread_axis_registers(shape, ls, rs) == int(kv["registers"])
    places = L.thread_axis_places(shape, ls, rs)
    for coord, where in rows:
        c = tuple(int(x) for x in coord.split())
        assert places[c] == tuple(int(x) for x in where.split())
    assert all(places[(l, j)] == (l, j) for l in range(32) for j in range(8))
    # loaded from a row-major (32, 8) buffer: lane l's registers are its row
    buf = list(range(256))
    frag = L.thread_axis_fragment(buf, shape, L.row_major_strides(shape), ls, rs)
    assert frag == [[8 * l + j for j in range(8)] for l in range(32)]


def test_thread_axis_fragments_equal_numpy_transposes():
    """Other thread-axis layouts against numpy (library routine) on iota buffers:
    the fragment [lane, register] is the tensor with its lane axes moved first."""
    buf = np.arange(256)
    # lanes over two axes (8 @ laneid, 1 @ laneid), one register axis
    frag = L.thread_axis_fragment(list(range(64)), (4, 8, 2), (16, 2, 1),
                                  (8, 1, 0), (0, 0, 1))
    assert np.array_equal(np.array(frag), np.arange(64).reshape(4, 8, 2).reshape(32, 2))
    # the lane axis in the middle, registers from the outer and inner axes (4 * c0 + c2)
    shape, ls, rs = (2, 32, 4), (0, 1, 0), (4, 0, 1)
    frag = L.thread_axis_fragment(list(buf), shape, L.row_major_strides(shape), ls, rs)
    want = buf.reshape(2, 32, 4).transpose(1, 0, 2).reshape(32, 8)
    assert np.array_equal(np.array(frag), want)
    # the same registers with their two axes swapped (c0 + 2 * c2)
    frag = L.thread_axis_fragment(list(buf), shape, L.row_major_strides(shape), ls, (1, 0, 2))
    want = buf.reshape(2, 32, 4).transpose(1, 2, 0).reshape(32, 8)
    assert np.array_equal(np.array(frag), want)
    # a transposed memory layout of the page's example: element (l, j) at j * 32 + l
    frag = L.thread_axis_fragment(list(buf), (32, 8), (1, 32), (1, 0), (0, 1))
    assert np.array_equal(np.array(frag), buf.reshape(8, 32).T)


def test_thread_axis_layouts_that_are_not_one_warp():
    """Rejected: an axis on both sides or on neither, lanes that do not cover 0..31
    once, registers with holes."""
    assert L.thread_axis_registers((32, 8), (1, 1), (0, 1)) is None     # both sides
    assert L.thread_axis_registers((32, 8), (1, 0), (0, 0)) is None     # neither
    assert L.thread_axis_registers((32, 8), (2, 0), (0, 1)) is None     # lanes 0, 2, ..
    assert L.thread_axis_registers((16, 8), (1, 0), (0, 1)) is None     # 16 lanes
    assert L.thread_axis_registers((32, 8), (1, 0), (0, 2)) is None     # registers 0, 2, ..
    assert L.thread_axis_registers((8, 4, 2), (4, 1, 0), (0, 0, 1)) == 2


# ---------------------------------------------------------------------------
# element conversions of the fused permute + cast (IEEE 754)
# ---------------------------------------------------------------------------
from oracle import cast_ref as C  # noqa: E402


def _f32(vals):
    return np.asarray(vals, dtype=np.float32).view(np.uint32)


def test_f32_to_f16_equals_numpy_on_every_class_of_value():
    """binary32 -> binary16, ties to even, against numpy's astype (library routine):
    random bit patterns, exact ties, the subnormal and overflow boundaries, signed
    zeros, infinities and NaN payloads."""
    rng = np.random.default_rng(61)
    bits = [rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)]
    # ties: halfway between two binary16 neighbours (a 1 just past the kept bits)
    h = rng.integers(0, 0x7BFF, size=5000, dtype=np.uint64).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float32).view(np.uint32)
    hi = (h + 1).view(np.float16).astype(np.float32)
    mid = ((lo.view(np.float32).astype(np.float64) + hi.astype(np.float64)) / 2).astype(np.float32)
    bits.append(mid.view(np.uint32))
    special = [0.0, -0.0, 65504.0, 65519.0, 65520.0, 65536.0, 2.0**-24, 2.0**-25, 3 * 2.0**-26,
               2.0**-14, 2.0**-14 - 2.0**-25, np.inf, -np.inf, 1e-40]
    bits.append(_f32(special))
    bits.append(np.array([0x7FC00000, 0x7F800001, 0xFFC00001, 0x7F802000, 0x7FFFFFFF,
                          0xFF800001], dtype=np.uint32))
    u = np.concatenate(bits)
    want = u.view(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(C.f32_to_f16_bits(u), want)


def test_f16_to_f32_equals_numpy_for_all_65536_patterns():
    u = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    assert np.array_equal(C.f16_to_f32_bits(u), u.view(np.float16).astype(np.float32).view(np.uint32))


def test_f32_to_bf16_is_the_nearest_bf16_with_ties_to_even():
    """binary32 -> bfloat16 by brute force: the result's neighbours on the bfloat16
    grid are never nearer, a tie takes the even one, overflow gives infinity, and
    NaNs stay NaNs of the same sign with their upper payload bits."""
    rng = np.random.default_rng(62)
    u = rng.integers(0, 2**32, size=100000, dtype=np.uint64).astype(np.uint32)
    ties = ((rng.integers(0, 0x7F7F, size=2000, dtype=np.uint64).astype(np.uint32) << 16)
            | np.uint32(0x8000))                       # exactly halfway
    u = np.concatenate([u, ties, _f32([0.0, -0.0, 1.0, np.inf, -np.inf, 3.3895313892515355e38,
                                      3.4e38, 1e-45])])
    got = C.f32_to_bf16_bits(u)
    x = u.view(np.float32).astype(np.float64)
    fin = np.isfinite(x)
    as_f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    v = as_f(got)
    for d in (-1, 1):                                  # the two grid neighbours of v
        nb = got.astype(np.int64) + d
        ok = (nb >= 0) & (nb < 0x10000)
        ok &= ((nb & 0x7F80) != 0x7F80)                # neighbours that are finite
        w = as_f(np.where(ok, nb, 0).astype(np.uint16))
        closer = np.abs(w - x) < np.abs(v - x)
        tie = np.abs(w - x) == np.abs(v - x)
        bad = fin & ok & np.isfinite(v) & (closer | (tie & ((got & 1) == 1)))
        assert not bad.any(), u[bad][:4]
    # overflow and exact values
    assert C.f32_to_bf16_bits(_f32([3.4e38]))[0] == 0x7F80
    assert C.f32_to_bf16_bits(_f32([1.0]))[0] == 0x3F80
    assert C.f32_to_bf16_bits(_f32([-0.0]))[0] == 0x8000
    assert C.f32_to_bf16_bits(np.array([0x3F808000], dtype=np.uint32))[0] == 0x3F80   # tie -> even
    assert C.f32_to_bf16_bits(np.array([0x3F818000], dtype=np.uint32))[0] == 0x3F82   # tie -> even
    nan = np.array([0x7FC00000, 0x7F800001, 0xFF812345], dtype=np.uint32)
    assert C.f32_to_bf16_bits(nan).tolist() == [0x7FC0, 0x7F81, 0xFF81]


def test_bf16_round_trips_through_f32():
    """bfloat16 -> binary32 is exact: back to bfloat16 gives every pattern again
    (NaN payloads included)."""
    u = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    assert np.array_equal(C.f32_to_bf16_bits(C.bf16_to_f32_bits(u)), u)
    f = C.bf16_to_f32_bits(u).view(np.float32)
    fin = (u & 0x7F80) != 0x7F80
    assert np.array_equal(f[fin].view(np.uint32) >> 16, u[fin])


def test_permute_cast_equals_numpy_transpose_and_astype():
    """The fused permute + cast against numpy: a transpose, then astype (binary16) or
    the bfloat16 view of the rounded values."""
    rng = np.random.default_rng(63)
    shape, perm = (5, 7, 9), (2, 0, 1)
    ss, ds = _perm_layouts(shape, perm)
    x = rng.standard_normal(int(np.prod(shape))).astype(np.float32)
    dst = np.zeros(int(np.prod(shape)) * 2, dtype=np.uint8)
    oracle.permute_cast(x.view(np.uint8), dst, shape, ss, ds, "f32_to_f16")
    want = np.transpose(x.reshape(shape), perm).astype(np.float16)
    assert np.array_equal(dst.view(np.float16), want.reshape(-1))
    h = want.reshape(-1).view(np.uint16)
    back = np.zeros(int(np.prod(shape)) * 4, dtype=np.uint8)
    ss2, ds2 = _perm_layouts(tuple(shape[p] for p in perm), (1, 2, 0))
    oracle.permute_cast(h.view(np.uint8), back, tuple(shape[p] for p in perm), ss2, ds2,
                        "f16_to_f32")
    assert np.array_equal(back.view(np.float32),
                          x.reshape(shape).astype(np.float16).astype(np.float32).reshape(-1))
