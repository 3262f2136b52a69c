"""Host-side pieces of bench.py that need no GPU: the sampled parity check."""
import numpy as np

import bench
import oracle
from movement_tl_permute_gb300 import workloads


def test_sampled_parity_compares_exactly_the_sampled_image():
    """The check compares the bytes the oracle's leading-m sample writes and no
    others: a wrong byte inside that image fails it, one outside does not."""
    w = workloads.scaled(workloads.get("t2d_f32"), 48)          # 48 x 16384 fp32
    src = workloads.make_input(w)
    full = np.zeros(w.dst_elems * w.elem_bytes, dtype=np.uint8)
    oracle.permute(src, full, w.shape, w.src_strides, w.dst_strides, w.elem_bytes)
    m = 5                                                       # rows 0..4 of src
    ok, n = bench.sampled_parity(w, src, full.copy(), m, 1)
    assert ok and n == m * w.shape[1] * w.elem_bytes
    # dst is column-major: src row r lands at elements r, r + 48, r + 96, ...
    bad = full.copy()
    bad[(2 + 48 * 7) * 4 + 1] ^= 0x10                           # row 2, column 7: sampled
    assert bench.sampled_parity(w, src, bad, m, 1) == (False, n)
    bad = full.copy()
    bad[(20 + 48 * 7) * 4] ^= 0x10                              # row 20: outside the sample
    assert bench.sampled_parity(w, src, bad, m, 1) == (True, n)


def test_config_runs_name_every_configuration():
    """Every configuration of the metric, plus the two high-rank block-path workloads and
    the odd-pitch u8 transpose (inputs larger than L2, like the rest)."""
    names = {wname for _, wname, _ in bench.CONFIG_RUNS}
    assert names == {"tile_transpose", "mx_sf", "attention", "t2d_u8", "t2d_f16", "t2d_f32",
                     "t2d_f64", "t2d_v16", "nd8_f32", "nd8_u16", "t2d_odd_u8"}
    for name in names:
        w = workloads.get(name)
        assert w.src_elems * w.elem_bytes > bench.L2_BYTES, name
    assert ("tile_transpose_cluster", "tile_transpose", "cluster") in bench.CONFIG_RUNS
