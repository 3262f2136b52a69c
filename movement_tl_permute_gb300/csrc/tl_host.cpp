// tl_host.cpp -- host-side layout logic of the permute library: validation,
// canonicalisation, the shared-memory bank simulator with its XOR-swizzle search,
// and the planner that picks a kernel path.  No CUDA calls in this file.
//
// A layout maps coordinate c to offset + sum c[i]*stride[i] (TVM docs, "Buffers
// and memory", section "Declaring buffers").  The warp path follows the TVM
// "permute_layout" page, section "Algorithm": align the two layouts, pick the
// XOR swizzle that keeps both phases bank-conflict-free, stage through registers.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "tl_internal.h"

namespace tl {
namespace {

bool valid_eb(int eb) { return eb == 1 || eb == 2 || eb == 4 || eb == 8 || eb == 16; }

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

// Highest offset a layout reaches (all strides >= 0); false on overflow.
bool layout_span(int n, const int64_t* ext, const int64_t* str, int64_t* span) {
    int64_t acc = 0;
    for (int i = 0; i < n; ++i) {
        if (ext[i] == 0) { *span = -1; return true; }
        int64_t t;
        if (!mul_ok(ext[i] - 1, str[i], &t) || !add_ok(acc, t, &acc)) return false;
    }
    *span = acc;
    return true;
}

// Merge adjacent axes (outer i, inner i+1) where both sides are contiguous across
// them, after dropping extent-1 axes.  Order is kept.
void drop_and_merge(const Axes& in, Axes* out) {
    Axes r;
    for (int i = 0; i < in.n; ++i) {
        if (in.ext[i] == 1) continue;
        if (r.n > 0 && r.ss[r.n - 1] == in.ext[i] * in.ss[i] &&
            r.ds[r.n - 1] == in.ext[i] * in.ds[i]) {
            r.ext[r.n - 1] *= in.ext[i];
            r.ss[r.n - 1] = in.ss[i];
            r.ds[r.n - 1] = in.ds[i];
        } else {
            r.ext[r.n] = in.ext[i];
            r.ss[r.n] = in.ss[i];
            r.ds[r.n] = in.ds[i];
            ++r.n;
        }
    }
    *out = r;
}

// Sufficient test that a layout never maps two coordinates onto one element:
// with axes sorted by stride, each stride exceeds everything the smaller axes reach.
bool non_overlapping(int n, const int64_t* ext, const int64_t* str) {
    int idx[kMaxDims];
    int m = 0;
    for (int i = 0; i < n; ++i)
        if (ext[i] > 1) idx[m++] = i;
    std::sort(idx, idx + m, [&](int a, int b) { return str[a] < str[b]; });
    int64_t reach = 0;
    for (int t = 0; t < m; ++t) {
        int i = idx[t];
        if (str[i] <= reach) return false;
        int64_t step;
        if (!mul_ok(ext[i] - 1, str[i], &step) || !add_ok(reach, step, &reach)) return false;
    }
    return true;
}

// Row-major coordinates of flat index f within ext[0..n).
void decompose(int64_t f, int n, const int64_t* ext, int64_t* coord) {
    for (int i = n - 1; i >= 0; --i) {
        coord[i] = f % ext[i];
        f /= ext[i];
    }
}

int64_t dot(int n, const int64_t* c, const int64_t* s) {
    int64_t o = 0;
    for (int i = 0; i < n; ++i) o += c[i] * s[i];
    return o;
}

// Offsets of one phase, iteration r, for all 32 lanes.
void phase_offsets(int n, const int64_t* ext, const int64_t* str, int r, int shift, int mask,
                   int64_t* out) {
    int64_t coord[kMaxDims];
    for (int lane = 0; lane < 32; ++lane) {
        int j = r ^ ((lane >> shift) & mask);
        decompose(lane + 32LL * j, n, ext, coord);
        out[lane] = dot(n, coord, str);
    }
}

bool phase_free(int n, const int64_t* ext, const int64_t* str, int P, int eb, int shift,
                int mask) {
    int64_t offs[32];
    for (int r = 0; r < P; ++r) {
        phase_offsets(n, ext, str, r, shift, mask, offs);
        if (bank_degree(32, offs, eb, false) > 1) return false;
    }
    return true;
}

}  // namespace

int bank_degree(int n_lanes, const int64_t* lane_offsets, int eb, bool hardware) {
    const int per = eb <= 4 ? 32 : 128 / eb;   // lanes per 128-byte wavefront
    int worst = 0;
    for (int base = 0; base < n_lanes; base += per) {
        // per bank: the lanes (conservative) or words (hardware) that touch it
        int64_t members[32][32];
        int count[32] = {0};
        for (int lane = base; lane < std::min(n_lanes, base + per); ++lane) {
            int64_t o = lane_offsets[lane];
            if (o < 0) continue;
            int64_t w0 = (o * eb) >> 2, w1 = (o * eb + eb - 1) >> 2;
            for (int64_t w = w0; w <= w1; ++w) {
                int bank = (int)(w & 31);
                int64_t key = hardware ? w : lane;
                bool seen = false;
                for (int q = 0; q < count[bank]; ++q) seen |= members[bank][q] == key;
                if (!seen) members[bank][count[bank]++] = key;
            }
        }
        for (int b = 0; b < 32; ++b) worst = std::max(worst, count[b]);
    }
    return worst;
}

int choose_xor(int n, const int64_t* ext, const int64_t* ss, const int64_t* ds, int eb, int* k,
               int* shift, int* mask) {
    if (n < 1 || n > kMaxDims) return TL_ERR_ARG;
    if (!valid_eb(eb)) return TL_ERR_ELEM_BYTES;
    int64_t total = 1;
    for (int i = 0; i < n; ++i) {
        if (ext[i] < 0) return TL_ERR_ARG;
        if (!mul_ok(total, ext[i], &total)) return TL_ERR_EXTENT;
    }
    if (total == 0 || total % 32 != 0 || total / 32 > 1024) return TL_ERR_EXTENT;
    const int P = (int)(total / 32);
    const bool pow2 = (P & (P - 1)) == 0;
    int kmax = 0;
    if (pow2)
        while ((1 << (kmax + 1)) <= P) ++kmax;
    for (int kk = 0; kk <= kmax; ++kk) {
        const int m = (1 << kk) - 1;
        for (int sh = 0; sh <= (kk == 0 ? 0 : 5 - kk); ++sh) {
            if (phase_free(n, ext, ss, P, eb, sh, m) && phase_free(n, ext, ds, P, eb, sh, m)) {
                *k = kk;
                *shift = sh;
                *mask = m;
                return TL_OK;
            }
        }
    }
    return TL_ERR_NO_VALID_K;
}

// ---------------------------------------------------------------------------
// Planner
// ---------------------------------------------------------------------------
namespace {

int64_t abs_addr(const void* p) { return (int64_t)(uintptr_t)p; }

bool aligned(int64_t v, int64_t a) { return a <= 1 || v % a == 0; }

// Memo of warp-tile searches: the swizzle search simulates every candidate, and
// small permutes tend to repeat the same layouts call after call.
struct WarpMemo {
    Axes kept;
    int eb;
    bool found;
    int start, P, k, shift, mask;
};
std::mutex g_warp_memo_mu;
std::vector<WarpMemo> g_warp_memo;
constexpr size_t kWarpMemoMax = 64;

bool same_axes(const Axes& a, const Axes& b) {
    if (a.n != b.n) return false;
    for (int i = 0; i < a.n; ++i)
        if (a.ext[i] != b.ext[i] || a.ss[i] != b.ss[i] || a.ds[i] != b.ds[i]) return false;
    return true;
}

bool plan_warp_search(Plan* p);

void apply_warp(Plan* p, int start, int P, int k, int sh, int m) {
    const Axes& kept = p->kept;
    Axes t, b;
    for (int i = start; i < kept.n; ++i) {
        t.ext[t.n] = kept.ext[i]; t.ss[t.n] = kept.ss[i]; t.ds[t.n] = kept.ds[i]; ++t.n;
    }
    for (int i = 0; i < start; ++i) {
        b.ext[b.n] = kept.ext[i]; b.ss[b.n] = kept.ss[i]; b.ds[b.n] = kept.ds[i]; ++b.n;
    }
    p->wtile = t;
    p->wbatch = b;
    p->P = P;
    p->k = k;
    p->shift = sh;
    p->mask = m;
}

bool plan_warp(Plan* p) {
    {
        std::lock_guard<std::mutex> lk(g_warp_memo_mu);
        for (const WarpMemo& e : g_warp_memo)
            if (e.eb == p->eb && same_axes(e.kept, p->kept)) {
                if (e.found) apply_warp(p, e.start, e.P, e.k, e.shift, e.mask);
                return e.found;
            }
    }
    const bool found = plan_warp_search(p);
    WarpMemo e{p->kept, p->eb, found, p->kept.n - p->wtile.n, p->P, p->k, p->shift, p->mask};
    std::lock_guard<std::mutex> lk(g_warp_memo_mu);
    if (g_warp_memo.size() >= kWarpMemoMax) g_warp_memo.erase(g_warp_memo.begin());
    g_warp_memo.push_back(e);
    return found;
}

// Order-kept canonical pair and its warp tile: the smallest innermost suffix that
// holds a whole number of warp iterations and admits a swizzle.
bool plan_warp_search(Plan* p) {
    const Axes& kept = p->kept;
    if (kept.n == 0) return false;
    int64_t prod = 1;
    for (int start = kept.n - 1; start >= 0; --start) {
        prod *= kept.ext[start];
        if (prod > 32LL * 32) break;
        int tdims = kept.n - start;
        if (tdims > kMaxWarpTileDims) break;
        if (prod % 32 != 0) continue;
        int P = (int)(prod / 32);
        if (P * p->eb > kWarpMaxRegBytes || (P & (P - 1)) != 0) continue;
        int k, sh, m;
        if (choose_xor(tdims, kept.ext + start, kept.ss + start, kept.ds + start, p->eb, &k, &sh,
                       &m) != TL_OK)
            continue;
        apply_warp(p, start, P, k, sh, m);
        return true;
    }
    return false;
}

// In place is only safe on the warp path, with identical pointers, identical
// batch strides and each tile reading exactly the elements it writes.
bool warp_in_place_ok(const Plan& p) {
    for (int i = 0; i < p.wbatch.n; ++i)
        if (p.wbatch.ss[i] != p.wbatch.ds[i]) return false;
    const Axes& t = p.wtile;
    int64_t total = 32LL * p.P;
    std::vector<int64_t> a(total), b(total);
    int64_t coord[kMaxDims];
    for (int64_t f = 0; f < total; ++f) {
        decompose(f, t.n, t.ext, coord);
        a[f] = dot(t.n, coord, t.ss);
        b[f] = dot(t.n, coord, t.ds);
    }
    std::sort(a.begin(), a.end());
    std::sort(b.begin(), b.end());
    return a == b;
}

// Plane of the transpose paths: b = dst-innermost axis (dst stride 1), a = the
// src-contiguous axis (src stride 1), everything else batch.
bool plan_plane(Plan* p) {
    const Axes& s = p->sorted;
    if (s.n < 2) return false;
    const int b = s.n - 1;
    if (s.ds[b] != 1 || s.ss[b] == 1) return false;
    int a = -1;
    for (int i = 0; i < s.n - 1; ++i)
        if (s.ss[i] == 1) { a = i; break; }
    if (a < 0 || s.n - 2 > kMaxBatch) return false;
    p->ext_a = s.ext[a];
    p->ext_b = s.ext[b];
    p->ss_b = s.ss[b];
    p->ds_a = s.ds[a];
    Axes bt;
    int64_t bt_total = 1;
    for (int i = 0; i < s.n - 1; ++i) {
        if (i == a) continue;
        bt.ext[bt.n] = s.ext[i]; bt.ss[bt.n] = s.ss[i]; bt.ds[bt.n] = s.ds[i]; ++bt.n;
        bt_total *= s.ext[i];
    }
    p->batch = bt;
    p->batch_total = bt_total;
    return true;
}

bool rows_ok(const Plan& p, int64_t src, int64_t dst) {
    const int eb = p.eb;
    const int64_t R = p.ext_b;
    const int64_t rw = R * eb;
    // any R whose run fits 16 bytes (planes -> 2..16 interleaved channels)
    if (R < 2 || rw > 16) return false;
    if (p.ds_a != R) return false;                       // dense plane in dst
    if ((p.ext_a * eb) % 16 != 0) return false;          // whole 16-byte row pieces
    if ((p.ss_b * eb) % 16 != 0 || src % 16 || dst % 16) return false;
    for (int i = 0; i < p.batch.n; ++i)
        if ((p.batch.ss[i] * eb) % 16 || (p.batch.ds[i] * eb) % 16) return false;
    return true;
}

// Short src runs: pixels of A = ext_a elements (2..16, at most 24 bytes) packed back
// to back along b, one dst plane per a; whole 16-byte pieces of every plane (ext_b a
// multiple of 16 / eb) and every piece, pixel run and plane on the 16-byte grid.
// Measured on GB300 (interleaved -> planes): 1.0-1.6x the panel kernel up to 24-byte
// pixels (u8 4..8 channels 4.3 -> 6.1 TB/s), 0.87x at 32 bytes (8 fp32 channels).
bool cols_ok(const Plan& p, int64_t src, int64_t dst) {
    const int eb = p.eb;
    const int64_t A = p.ext_a;
    if (eb > 8 || A < 2 || A > 16 || A * eb > 24) return false;
    if (p.ss_b != A || p.ext_b % (16 / eb) != 0) return false;
    if (src % 16 || dst % 16 || (p.ds_a * eb) % 16) return false;
    for (int i = 0; i < p.batch.n; ++i)
        if ((p.batch.ss[i] * eb) % 16 || (p.batch.ds[i] * eb) % 16) return false;
    return true;
}

bool tile_ok(const Plan& p, int64_t src) {
    const int eb = p.eb;
    if (p.batch.n > kMaxTmaBatch) return false;
    if (src % 16 != 0) return false;
    if ((p.ss_b * eb) % 16 != 0) return false;
    const int64_t lim_coord = (1LL << 31) - 1, lim_stride = 1LL << 40;
    if (p.ext_a * eb > lim_coord || p.ext_b > lim_coord) return false;
    if (p.ss_b * eb >= lim_stride) return false;
    for (int i = 0; i < p.batch.n; ++i) {
        if ((p.batch.ss[i] * eb) % 16 != 0 || p.batch.ss[i] * eb >= lim_stride) return false;
        if (p.batch.ext[i] > lim_coord) return false;
    }
    return true;
}

// Tile-path fit: 64 rows of b and whole 128-byte rows of a.  Measured on GB300:
// transposes with 64-byte rows of a run at 3.7-5.1 TB/s on half-empty TMA tiles and
// 6.0-6.1 on the panel kernel, 96-byte rows about even (4.9-6.1 against 5.9-6.0),
// 128-byte rows faster on tiles (6.2-6.8 against 5.7-6.0).
bool tile_fits(const Plan& p) { return p.ext_b >= 64 && p.ext_a * p.eb >= 128; }

// Extent of b once a short b takes in the next dst axis (see panel_merge_b).
int64_t panel_b_extent(const Plan& p) {
    if (p.ext_b >= 64) return p.ext_b;
    for (int i = 0; i < p.batch.n; ++i)
        if (p.batch.ds[i] == p.ext_b && p.ext_b * p.batch.ext[i] < (1LL << 31))
            return p.ext_b * p.batch.ext[i];
    return p.ext_b;
}

// Panel path: the plane needs one extent of at least 16 elements (else the
// batch is the long dimension and the generic kernel walks it as well).
bool panel_ok(const Plan& p) { return p.ext_a >= 16 || panel_b_extent(p) >= 16; }

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Panel pitch: the byte pitch (a multiple of 16) of the rows of the shared-memory
// tile, chosen by simulating both walks' warp accesses on the banks (hardware
// model).  The copy walk takes item g, a 16-byte block, at (b = g / nblk,
// k = g % nblk), a warp covering 32 consecutive items.  In the store walk a row b
// starts (r + b * (ss_b * eb mod 16)) mod 16 bytes into its first block, simulated
// for every residue r of the tile's base address (r = 0 only when every row is
// aligned).  Element stores: a warp takes 32 consecutive tile elements f at
// (a = f / tb, b = f % tb).  16-byte dst runs (vec): rows are skewed (row b at
// b * pitch + 16 * (b / V), V = 16 / eb) and a warp takes 4 rows a by 8 blocks q;
// at step k lane (a, q) reads row b = qV + k, the reads of the panel kernel's
// drain_vec.  Among the pitches with the lowest summed degree of the store walk the
// narrowest whose copy walk stays within 2-way wins (stage capacity decides the
// bytes in flight, which bound this kernel, more than conflicts among the copy
// walk's asynchronous writes), else the one with the lowest copy-walk degree.
struct PanelMemo {
    int ta, tb, eb, pitch;
    int64_t ssb, b1, ssb2;
    int nblk, aligned, walk, rot_s, rot_m;
};
std::mutex g_panel_memo_mu;
std::vector<PanelMemo> g_panel_memo;

int panel_blocks_per_row(int64_t ta, int eb) { return (int)((ta * eb + 30) / 16); }

// src byte offset of b modulo 16: b is one axis (stride ss_b) or, when b1 > 0, two
// merged axes (b % b1 with stride ss_b, b / b1 with stride ss_b2)
int64_t b_mis16(int64_t b, int eb, int64_t ssb, int64_t b1, int64_t ssb2) {
    const int64_t off = b1 > 0 ? (b % b1) * ssb + (b / b1) * ssb2 : b * ssb;
    return (off * eb) & 15;
}

// Store walks the pitch search models (the panel kernel's drains).
enum PanelWalk { kWalkElems = 0, kWalkRuns = 1, kWalkWords = 2 };

int panel_pitch(int ta, int tb, int eb, int64_t ssb, int64_t b1, int64_t ssb2, int nblk,
                bool aligned, int walk, int* rot_s, int* rot_m) {
    const bool vec = walk == kWalkRuns;
    *rot_s = *rot_m = 0;
    // the row misalignments repeat with a period of 16 rows (one axis) or are
    // sampled over the tile's rows (merged axes); normalise the memo key
    const int64_t ssb_k = b1 > 0 ? ssb : (ssb * eb) & 15;
    {
        std::lock_guard<std::mutex> lk(g_panel_memo_mu);
        for (const PanelMemo& e : g_panel_memo)
            if (e.ta == ta && e.tb == tb && e.eb == eb && e.ssb == ssb_k && e.b1 == b1 &&
                e.ssb2 == ssb2 && e.nblk == nblk && e.aligned == (int)aligned &&
                e.walk == walk) {
                *rot_s = e.rot_s;
                *rot_m = e.rot_m;
                return e.pitch;
            }
    }
    const int64_t n_copy = (int64_t)nblk * tb, n_store = (int64_t)ta * tb;
    const int64_t samples = 32 * 64;
    const int V = 16 / eb;
    const int64_t qb8 = vec ? ((int64_t)tb * eb + 127) / 128 : 1;
    auto skew = [&](int64_t b) { return vec ? b / V : 0; };          // 16-byte units
    const int64_t units = vec ? (int64_t)((ta + 3) / 4) * qb8 : 0;
    struct Cand {
        int pitch;
        int64_t store, copy;
        int copy_max;
        int rs, rm;
    };
    std::vector<Cand> cands;
    for (int64_t q = nblk; q < nblk + 8; ++q) {
        const int64_t pitch = 16 * q;
        int64_t copy = 0, store = 0, ideal_copy = 0, ideal_store = 0;
        int copy_max = 0, best_rs = 0, best_rm = 0;
        for (int64_t g0 = 0; g0 < std::min(n_copy, samples); g0 += 32, ++ideal_copy) {
            int64_t o[32];
            int m = 0;
            for (int64_t g = g0; g < g0 + 32 && g < n_copy; ++g, ++m)
                o[m] = (g / nblk) * q + skew(g / nblk) + g % nblk;   // 16-byte units
            const int d = bank_degree(m, o, 16, true);
            copy += d;
            copy_max = std::max(copy_max, d);
        }
        if (walk == kWalkWords) {
            // one warp per dst row: lane w packs word w from rows h + V4 w + k', k' the
            // rotated step; sampled over the row's head h, two columns and four base
            // residues; the best rotation for this pitch is kept
            const int V4 = 4 / eb;
            int64_t best = -1, ideal = 0;
            for (int m = 0; m < V4; ++m)
                for (int sh = 0; sh <= 4; ++sh) {
                    if (m == 0 && sh > 0) break;
                    int64_t cost = 0, cnt = 0;
                    for (int r = 0; r < (aligned ? 1 : 16); r += aligned ? 1 : 4)
                        for (int h = 0; h < V4; ++h)
                            for (int a = 0; a < std::min(ta, 2); ++a)
                                for (int k = 0; k < V4; ++k, ++cnt) {
                                    int64_t o[32];
                                    for (int l = 0; l < 32; ++l) {
                                        const int64_t b =
                                            h + (int64_t)V4 * l + ((k + m * (l >> sh)) & (V4 - 1));
                                        o[l] = b < tb ? (b * pitch +
                                                         ((r + b_mis16(b, eb, ssb, b1, ssb2)) & 15) +
                                                         a * eb) / eb
                                                      : -1;
                                    }
                                    cost += bank_degree(32, o, eb, true);
                                }
                    if (best < 0 || cost < best) {
                        best = cost;
                        best_rs = sh;
                        best_rm = m;
                        ideal = cnt;
                    }
                }
            store = best;
            ideal_store = ideal;
        }
        for (int r = 0; r < (aligned ? 1 : 16) && walk != kWalkWords; r += eb) {
            auto off = [&](int64_t a, int64_t b) {
                return (b * pitch + 16 * skew(b) + ((r + b_mis16(b, eb, ssb, b1, ssb2)) & 15) +
                        a * eb) / eb;
            };
            if (vec) {
                for (int64_t u = 0; u < std::min(units, samples / 32); ++u) {
                    const int64_t g4 = u / qb8, qg = u % qb8;
                    for (int k = 0; k < V; ++k, ++ideal_store) {
                        int64_t o[32];
                        for (int l = 0; l < 32; ++l) {
                            const int64_t a = 4 * g4 + l / 8, qq = 8 * qg + l % 8;
                            const int64_t b = qq * V + k;
                            o[l] = a < ta && b < tb ? off(a, b) : -1;
                        }
                        store += bank_degree(32, o, eb, true);
                    }
                }
                continue;
            }
            for (int64_t f0 = 0; f0 < std::min(n_store, samples); f0 += 32, ++ideal_store) {
                int64_t o[32];
                int m = 0;
                for (int64_t f = f0; f < f0 + 32 && f < n_store; ++f, ++m)
                    o[m] = off(f / tb, f % tb);
                store += bank_degree(m, o, eb, true);
            }
        }
        cands.push_back({(int)pitch, store, copy, copy_max, best_rs, best_rm});
        if (store == ideal_store && copy == ideal_copy) break;   // degree 1 everywhere
    }
    int64_t min_store = cands[0].store;
    for (const Cand& c : cands) min_store = std::min(min_store, c.store);
    const Cand* pick = nullptr;
    int64_t best_copy = -1;
    for (const Cand& c : cands) {
        if (c.store != min_store) continue;
        if (c.copy_max <= 2) {
            pick = &c;
            break;
        }
        if (best_copy < 0 || c.copy < best_copy) {
            best_copy = c.copy;
            pick = &c;
        }
    }
    const int best = pick->pitch;
    *rot_s = pick->rs;
    *rot_m = pick->rm;
    std::lock_guard<std::mutex> lk(g_panel_memo_mu);
    if (g_panel_memo.size() >= 64) g_panel_memo.erase(g_panel_memo.begin());
    g_panel_memo.push_back({ta, tb, eb, best, ssb_k, b1, ssb2, nblk, (int)aligned, walk, *rot_s,
                            *rot_m});
    return best;
}

// Word-store rotation for packed rows of 1- and 2-byte elements (the panel
// kernel's word walk): lane l of a warp packs word w = l of a dst row, reading its
// k-th element from stage element ((w * V + k') * ta + e), V = 4 / eb,
// k' = (k + m * (l >> s)) mod V.  Every (s, m) is simulated on the bank model
// (hardware mode) for the tile's ta, every dst row e of the first four, every step k
// and every start of the run within a 4-byte word; the lowest summed degree wins, the
// unrotated walk (m = 0) on ties.
// Worst bank-conflict degree of the 16-byte run walk over packed rows (stage
// element (b * ta + e), a warp taking 4 rows e by 8 blocks q, lane (e, q) reading
// b = qV + k at step k), over every start of the run within a 16-byte block.
int panel_packed_vec_degree(int ta, int eb) {
    const int V = 16 / eb;
    int worst = 0;
    for (int r = 0; r < V; ++r)
        for (int k = 0; k < V; ++k) {
            int64_t o[32];
            for (int l = 0; l < 32; ++l) {
                const int e = l / 8, q = l % 8;
                o[l] = e < ta ? (int64_t)(q * V + k) * ta + e + r : -1;
            }
            worst = std::max(worst, bank_degree(32, o, eb, true));
        }
    return worst;
}

// 16-byte runs over packed rows (a short a axis of ta elements): a warp's 32 lanes
// take 4 rows a by 8 blocks, so rows beyond ta leave lanes idle.  Measured on GB300
// (interleaved channels -> planes, 2..7 channels): 1-byte rows keep the word
// stores; 2-byte rows take the runs with at least 4 rows, 3 of 4 lanes busy and
// reads within 2-way conflicts (word stores are faster otherwise: 6.0 against 3.3
// TB/s at 2 channels); 4-byte rows take them but for 2 channels; 8-byte rows with 3
// of 4 lanes busy.
bool panel_packed_vec_ok(int ta, int eb) {
    const bool busy = 4 * ta >= 3 * (4 * ((ta + 3) / 4));
    switch (eb) {
    case 1: return false;
    case 2: return ta >= 4 && busy && panel_packed_vec_degree(ta, eb) <= 2;
    case 4: return ta != 2;
    default: return busy;
    }
}

struct RotMemo {
    int ta, eb, rs, rm;
};
std::mutex g_rot_memo_mu;
std::vector<RotMemo> g_rot_memo;

void panel_word_rotation(int ta, int eb, int* rs, int* rm) {
    {
        std::lock_guard<std::mutex> lk(g_rot_memo_mu);
        for (const RotMemo& e : g_rot_memo)
            if (e.ta == ta && e.eb == eb) {
                *rs = e.rs;
                *rm = e.rm;
                return;
            }
    }
    const int V = 4 / eb;
    int64_t best = -1;
    *rs = 0;
    *rm = 0;
    for (int m = 0; m < V; ++m) {
        for (int sh = 0; sh <= 4; ++sh) {
            if (m == 0 && sh > 0) break;
            int64_t cost = 0;
            for (int r = 0; r < V; ++r)
                for (int e = 0; e < std::min(ta, 4); ++e)
                    for (int k = 0; k < V; ++k) {
                        int64_t o[32];
                        for (int l = 0; l < 32; ++l) {
                            const int kk = (k + m * (l >> sh)) & (V - 1);
                            o[l] = (int64_t)(l * V + kk) * ta + e + r;
                        }
                        cost += bank_degree(32, o, eb, true);
                    }
            if (best < 0 || cost < best) {
                best = cost;
                *rs = sh;
                *rm = m;
            }
        }
    }
    std::lock_guard<std::mutex> lk(g_rot_memo_mu);
    if (g_rot_memo.size() >= 64) g_rot_memo.erase(g_rot_memo.begin());
    g_rot_memo.push_back({ta, eb, *rs, *rm});
}

// Panel tile of about tile_bytes: a tiny extent is taken whole and the other one
// fills the tile; otherwise 128 (eb = 1), 64 (eb = 2, 4) or 32 rows of b by the rest
// of a (whole 128-byte dst runs for 1- and 2-byte elements), or more
// rows when a runs out; no tile side exceeds its extent.  64 rows of 4-byte
// elements (256 dst bytes per tile row) measured 6.0 against 4.5 TB/s for 32 rows on
// fp32 transposes whose dst rows are not 16-byte aligned (half as many tile edges
// inside a dst row).  Src rows packed back to back are copied as one run.
}  // namespace

// A short b axis (under 64 elements) takes in the next dst axis when dst is dense
// across the two (that axis's dst stride equals the b extent): the tile's dst runs
// and its row count grow, its src rows stay contiguous.
void panel_merge_b(Plan* p) {
    if (p->ext_b >= 64) return;
    for (int i = 0; i < p->batch.n; ++i) {
        if (p->batch.ds[i] != p->ext_b) continue;
        const int64_t merged = p->ext_b * p->batch.ext[i];
        if (merged >= (1LL << 31)) return;     // same rule as panel_b_extent
        p->panel_b1 = p->ext_b;
        p->panel_ss_b2 = p->batch.ss[i];
        p->ext_b = merged;
        p->batch_total /= p->batch.ext[i];
        for (int j = i; j + 1 < p->batch.n; ++j) {
            p->batch.ext[j] = p->batch.ext[j + 1];
            p->batch.ss[j] = p->batch.ss[j + 1];
            p->batch.ds[j] = p->batch.ds[j + 1];
        }
        --p->batch.n;
        return;
    }
}

namespace {

// Every src row of every tile starts on a 16-byte boundary: the base, the tile
// column step ta, the row strides and the batch strides are all multiples of 16 bytes.
bool panel_src_aligned(const Plan& p, int64_t ta) {
    const int eb = p.eb;
    bool ok = p.src_mis16 == 0 && (ta * eb) % 16 == 0 && (p.ss_b * eb) % 16 == 0 &&
              (p.panel_b1 == 0 || (p.panel_ss_b2 * eb) % 16 == 0);
    for (int i = 0; i < p.batch.n; ++i) ok = ok && (p.batch.ss[i] * eb) % 16 == 0;
    return ok;
}

// 16-byte dst runs: 1-, 2-, 4- or 8-byte elements, tb * eb a multiple of 128 (whole
// 8-block groups), every dst row of every tile on a 16-byte boundary, and a row
// misalignment in the stage that follows b linearly (packed rows, one b axis, or
// merged axes whose src strides are multiples of 16 bytes).  Measured on GB300:
// 4-byte elements whose src rows are not 16-byte aligned store faster element by
// element (6.2 against 5.7 TB/s on odd-pitch fp32 transposes); the other block-row
// layouts gain from the runs (by up to 30 % on 2-byte elements, 64 % on 1-byte
// transposes).  Packed rows are decided by panel_packed_vec_ok as well.
// Tile heights whose dst row pieces the 16-byte run walk covers: whole 16-byte units,
// at least one 128-byte group of them, and at least 3/4 of the lanes of the 8-unit
// groups busy (a height of 100 4-byte elements: 25 units in 4 groups).
bool panel_vec_rows_ok(int64_t tb, int eb) {
    const int64_t bytes = tb * eb, units = bytes / 16, groups = (units + 7) / 8;
    return bytes % 16 == 0 && bytes >= 128 && 4 * units >= 3 * 8 * groups;
}

bool panel_dst_vec(const Plan& p, int64_t tb, bool packed, bool aligned) {
    const int eb = p.eb;
    if (p.panel_elem_stores || eb > 8 || !panel_vec_rows_ok(tb, eb)) return false;
    if (eb == 4 && !packed && !aligned) return false;
    bool ok = p.dst_mis16 == 0 && (p.ds_a * eb) % 16 == 0 &&
              (p.panel_a1 == 0 || (p.panel_ds_a2 * eb) % 16 == 0);
    for (int i = 0; i < p.batch.n; ++i) ok = ok && (p.batch.ds[i] * eb) % 16 == 0;
    if (p.panel_b1 > 0 && !packed)
        ok = ok && (p.ss_b * eb) % 16 == 0 && (p.panel_ss_b2 * eb) % 16 == 0;
    return ok;
}

// A short b axis packed in dst (planes -> interleaved channels): each tile's dst is
// one run of ta * tb elements, stored in 16-byte pieces (unless 16-byte runs along
// the tile rows apply, or the caller declined vector stores).  Measured on GB300
// (3..8 planes -> interleaved): 1.2-1.4x the element and word stores for 1-, 2- and
// 4-byte elements (fp32, 3 planes: 5.7 against 4.0 TB/s); 8-byte elements store as
// fast element by element, and keep doing so.
bool panel_dst_run(const Plan& p, int64_t tb) {
    return !p.panel_vec && !p.panel_elem_stores && p.eb <= 4 && tb <= 16 && tb == p.ext_b &&
           p.ds_a == tb && p.panel_b1 == 0 && p.panel_a1 == 0;
}

// Phase-major stage for block rows (TMA phase maps, k_panel_tma, or cp.async into
// the same arrangement): one b axis, at most three batch axes on the 16-byte grid,
// element stores (the drain that takes the phase layout), a row pitch P whose phase
// count phi = 16 / gcd(P, 16) divides the tile height, and boxes within the TMA
// limits (at most 256 elements a side).  Returns phi, or 0 when the tile cannot take
// the arrangement.
int panel_tma_phases(const Plan& p, int64_t ta, int64_t tb) {
    const int eb = p.eb;
    // (1-byte tiles keep the block-row stage: their word walk's rotation is searched
    // for it)
    if (eb == 1 || eb > 8 || p.panel_b1 != 0 || p.panel_a1 != 0 || p.batch.n > 3 ||
        p.panel_vec || p.panel_run)
        return 0;
    // rows of ta * eb + 16 bytes, an odd number of 16-byte blocks: the phase blocks'
    // rows then fall in distinct bank groups
    if (tb <= 16 || (ta * eb) % 32 != 0 || ta + 16 / eb > 256) return 0;
    for (int i = 0; i < p.batch.n; ++i)
        if ((p.batch.ss[i] * eb) % 16 != 0 || p.batch.ss[i] * eb >= (1LL << 40)) return 0;
    const int64_t P = p.ss_b * eb;
    int64_t g = 16;
    while (P % g != 0) g >>= 1;
    const int phi = (int)(16 / g);
    if (phi == 1 && p.src_mis16 == 0) return 0;       // the tile path takes aligned pitches
    if (tb % phi != 0 || tb / phi > 256 || p.ext_b < phi || phi * P >= (1LL << 40)) return 0;
    return phi;
}

}  // namespace

// A short a axis (under 64 elements) takes in the next src axis when src is dense
// across the two (that axis's src stride equals the a extent): the tile's src rows
// stay contiguous and grow, and each tile row's dst offset splits a into its two
// axes (the panel kernel's drow_off).  Only where the whole a x b plane is under
// 16 KiB: high-rank permutes of short axes otherwise get tiles of a few KiB.
// Measured on GB300 (one box, merged against unmerged): 10^8 reversed fp32 3.98
// against 0.95 TB/s and fp64 3.54 against 2.58, 16^7 reversed fp16 4.89 against
// 2.35; planes of 27 KiB and more stay faster unmerged (24^6 fp16 4.47 against 4.05,
// a 6-D fp32 with a = 28 4.71 against 4.10).
void panel_merge_a(Plan* p) {
    if (p->ext_a >= 64 || p->ext_a * p->ext_b * p->eb >= 16384) return;
    for (int i = 0; i < p->batch.n; ++i) {
        if (p->batch.ss[i] != p->ext_a) continue;
        const int64_t merged = p->ext_a * p->batch.ext[i];
        if (merged >= (1LL << 31)) return;
        p->panel_a1 = p->ext_a;
        p->panel_ds_a2 = p->batch.ds[i];
        p->ext_a = merged;
        p->batch_total /= p->batch.ext[i];
        for (int j = i; j + 1 < p->batch.n; ++j) {
            p->batch.ext[j] = p->batch.ext[j + 1];
            p->batch.ss[j] = p->batch.ss[j + 1];
            p->batch.ds[j] = p->batch.ds[j + 1];
        }
        --p->batch.n;
        return;
    }
}

// The skew walk (1-byte elements whose dst rows sit at an odd pitch, one a and one b
// axis): no tile row's dst run is on the 16-byte grid, so the word walk would pack
// every element from a 1-byte shared load; the skew walk stores 16-byte pieces of the
// dst rows instead.  Planes of at least 64 x 64.
static bool panel_skew_ok(const Plan& p) {
    return p.eb == 1 && p.cast == TL_CAST_NONE && !p.panel_elem_stores && p.panel_b1 == 0 &&
           p.panel_a1 == 0 && p.ds_a > 0 && (p.ds_a & 1) == 1 && p.ss_b > 0 && p.ext_a >= 64 &&
           p.ext_b >= 64;
}

void plan_panel(Plan* p, int tile_bytes, int rows) {
    const int eb = p->eb;
    p->panel_skew = false;
    if (panel_skew_ok(*p)) {
        // tiles of 256 x 256 (8 warps) or, asked for tiles of 32 KiB or less, 128 x 256
        const int warps = tile_bytes > 0 && tile_bytes <= 32768 ? 4 : 8;
        p->panel_skew = true;
        p->panel_skew_warps = warps;
        p->tile_cols = 32 * warps;
        p->tile_rows = kSkewRows;
        p->panel_mode = 0;
        p->panel_aligned = p->panel_vec = p->panel_run = p->panel_words = false;
        p->panel_tma = p->panel_phase = false;
        p->panel_wrot_s = p->panel_wrot_m = 0;
        p->pitch = skew_pitch(p->tile_cols);
        p->panel_nblk = p->tile_cols / 16 + 2;
        p->panel_stage = skew_stage_bytes(p->tile_cols);
        const int64_t na = (p->ext_a + p->tile_cols - 1) / p->tile_cols;
        const int64_t nb = (p->ext_b + kSkewRows - 1) / kSkewRows;
        p->tiles = na * nb * p->batch_total;
        p->vec_bytes = 16;
        return;
    }
    const bool tiny = p->ext_a <= 16 || p->ext_b <= 16;
    if (tile_bytes <= 0) tile_bytes = tiny ? 24576 : 32768;
    const int64_t E = tile_bytes / eb;
    const int64_t ru = std::max(32, 128 / eb);   // rows of b: whole 128-byte dst runs
    int64_t ta, tb;
    if (p->ext_b <= 16) {
        tb = p->ext_b;
        ta = std::min(round_up((E + tb - 1) / tb, 32), p->ext_a);
    } else if (p->ext_a <= 16) {
        ta = p->ext_a;
        tb = std::min(round_up((E + ta - 1) / ta, ru), p->ext_b);
    } else {
        tb = std::min<int64_t>(rows > 0 ? rows : eb == 1 ? 128 : eb <= 4 ? 64 : 32, p->ext_b);
        ta = std::max<int64_t>(1, std::min(E / tb, p->ext_a));
        // rows off the 16-byte grid (widths that take a phase-major stage): a TMA
        // phase box holds at most 256 elements (ta + 16 / eb of them), and a row of
        // ta * eb + 16 bytes spans an odd number of 16-byte blocks (ta * eb a multiple
        // of 32); the tile keeps its height
        const bool capped = eb >= 2 && eb <= 8 && (p->ss_b * eb) % 16 != 0 && ta + 16 / eb > 256;
        if (capped) ta = (256 - 16 / eb) / (32 / eb) * (32 / eb);
        if (ta * tb < E && !capped)   // a short a extent: the tile grows along b instead
            tb = std::min(round_up((E + ta - 1) / ta, ru), p->ext_b);
        // the same number of tiles along b, evened out (whole 16-byte dst pieces): b =
        // 100 4-byte elements takes 52 + 48 rows instead of 96 + 4 (measured on 10^8
        // reversed fp32 with a merged a: the 4-row tiles cost 30 %)
        if (tb < p->ext_b) {
            const int64_t nb = (p->ext_b + tb - 1) / tb;
            const int64_t even = round_up((p->ext_b + nb - 1) / nb, std::max(1, 16 / eb));
            if (even < tb && (panel_vec_rows_ok(even, eb) || !panel_vec_rows_ok(tb, eb)))
                tb = even;
        }
    }
    int64_t stage;
    for (;;) {
        p->tile_cols = (int)ta;
        p->tile_rows = (int)tb;
        // src rows packed back to back over the whole b range (merged axes too);
        // packed rows that are whole 16-byte blocks on the 16-byte grid are staged
        // as block rows instead, whose skewed layout the 16-byte run walk reads
        // without bank conflicts
        // (rows of whole blocks leave no lane idle when 4 rows a fill a warp's rows)
        const bool packed_rows = ta == p->ext_a && p->ss_b == ta &&
                                 (p->panel_b1 == 0 || p->panel_ss_b2 == p->panel_b1 * ta);
        const bool packed_vec = packed_rows && panel_packed_vec_ok((int)ta, eb);
        const bool packed = packed_rows &&
                            !((ta * eb) % 16 == 0 && ta % 4 == 0 && panel_src_aligned(*p, ta) &&
                              panel_dst_vec(*p, tb, false, true));
        p->panel_aligned = false;
        p->panel_vec = false;
        p->panel_wrot_s = p->panel_wrot_m = 0;
        p->panel_run = false;
        p->panel_words = false;
        p->panel_tma = false;
        p->panel_phase = false;
        if (packed) {
            p->panel_mode = 1;
            p->pitch = 0;
            p->panel_nblk = 0;
            p->panel_vec = packed_vec && panel_dst_vec(*p, tb, true, false);
            p->panel_run = !p->panel_vec && panel_dst_run(*p, tb);
            if (eb < 4 && !p->panel_vec)
                panel_word_rotation((int)ta, eb, &p->panel_wrot_s, &p->panel_wrot_m);
            stage = 16 * ((ta * tb * eb + 30) / 16);
        } else {
            p->panel_mode = 0;
            p->panel_aligned = panel_src_aligned(*p, ta);
            p->panel_vec = panel_dst_vec(*p, tb, false, p->panel_aligned);
            p->panel_run = panel_dst_run(*p, tb);
            // 1-byte elements whose dst rows take neither run mode: 4-byte words per dst
            // row (measured on odd-pitch transposes: u8 3.2 -> 3.6 TB/s; 2-byte elements
            // stay faster element by element, 4.4 against 3.4)
            p->panel_words = !p->panel_vec && !p->panel_run && !p->panel_elem_stores &&
                             eb == 1 && p->panel_b1 == 0 && p->panel_a1 == 0;
            p->panel_nblk = p->panel_aligned ? (int)(ta * eb / 16) : panel_blocks_per_row(ta, eb);
            // skewed rows for 16-byte dst runs: 16 more bytes per 16 / eb rows; the
            // pitch search runs when at least its narrowest pitch fits
            const int64_t skew = p->panel_vec ? 16 * (tb / (16 / eb)) : 0;
            stage = tb * 16 * p->panel_nblk + skew;
            const int phi = p->panel_elem_stores ? 0 : panel_tma_phases(*p, ta, tb);
            if (phi > 0) {
                // phase-major stage: phi blocks of tb / phi rows of ta * eb + 16 bytes,
                // each block on a 128-byte boundary.  Measured on GB300 (odd-pitch
                // transposes, against block rows filled by cp.async, one box per A/B):
                // TMA phase maps fp16 4.18 -> 5.39 TB/s; for fp32 and fp64 the maps
                // measured 0.89x and 0.89-1.03x, while cp.async into the phase-major
                // stage gains 2 % (fp32 5.71 -> 5.82) and 4 % (fp64 6.09 -> 6.36).
                p->panel_phase = true;
                p->panel_tma = eb == 2;
                p->panel_phi_lg = 0;
                while ((1 << p->panel_phi_lg) < phi) ++p->panel_phi_lg;
                p->pitch = (int)(ta * eb + 16);
                p->panel_phase_bytes = (int)round_up((tb / phi) * p->pitch, 128);
                p->panel_nblk = panel_blocks_per_row(ta, eb);   // for the cp.async fallback
                p->panel_aligned = false;
                stage = phi * p->panel_phase_bytes;
            } else if (kPanelStages * stage <= kPanelMaxSmem) {
                const int walk = p->panel_vec ? kWalkRuns : p->panel_words ? kWalkWords : kWalkElems;
                p->pitch = panel_pitch((int)ta, (int)tb, eb, p->ss_b, p->panel_b1, p->panel_ss_b2,
                                       p->panel_nblk, p->panel_aligned, walk, &p->panel_wrot_s,
                                       &p->panel_wrot_m);
                stage = tb * p->pitch + skew;
            }
        }
        if (kPanelStages * stage <= kPanelMaxSmem || (ta <= 1 && tb <= 1)) break;
        if (tb >= ta) tb = (tb + 1) / 2; else ta = (ta + 1) / 2;   // halve the longer side
    }
    p->panel_stage = (int)stage;
    const int64_t na = (p->ext_a + ta - 1) / ta, nb = (p->ext_b + tb - 1) / tb;
    p->tiles = na * nb * p->batch_total;
    p->vec_bytes = p->panel_vec || p->panel_run ? 16 : p->panel_words ? 4 : eb;
}

// ---------------------------------------------------------------- block path
// A tile of up to four axes that is a few long contiguous runs on both sides: the
// dense chain of axes from src stride 1 (S) and from dst stride 1 (D); T is a prefix
// of S joined with a prefix of D.  Every (S prefix, D prefix) pair with at most four
// axes is tried, with at most one axis split into chunks so the tile fits its bytes
// (the last axis of each run it belongs to, so both runs stay dense); the tile whose
// shorter run (capped at 512 bytes) is longest wins, then the bigger tile.  The
// shared-memory strides of the src-run index axes are chosen by replaying the store
// walk's warp reads on the bank model (hardware mode).
namespace {

// mixed-radix digits of x over `n` extents (innermost first)
void digits(int64_t x, int n, const int64_t* ext, int64_t* d) {
    for (int k = 0; k < n; ++k) {
        d[k] = x % ext[k];
        x /= ext[k];
    }
}

// Stage layout of a block tile (byte strides b.sq, stage bytes b.stage): the src-run
// axes at their src byte strides; the src-run index axes, innermost first, each at
// the smallest stride that is at least the span of the runs inside it and congruent
// to its src byte stride modulo 16, plus 16 * extra[k].  A run's copy covers the
// aligned 16-byte blocks around it, up to 15 bytes past either end, so one run spans
// Ls * eb + 30 bytes; a 16-byte lead holds the tile origin's offset inside its block.
// An element thus sits at the same offset modulo 16 in the stage as in src.
int64_t block_layout(BlockPlan& b, int eb, const int* extra) {
    for (int k = 0; k < b.ns; ++k) b.sq[b.sax[k]] = b.ss[b.sax[k]] * eb;
    int64_t span = b.Ls * eb + 30;
    for (int k = 0; k < b.nr; ++k) {
        const int q = b.rax[k];
        const int64_t want = (b.ss[q] * eb) & 15;
        const int64_t P = span + ((want - span) & 15) + 16 * (extra ? extra[k] : 0);
        b.sq[q] = P;
        span += (b.tile[q] - 1) * P;
    }
    b.stage = (16 + span + 15) & ~int64_t(15);
    b.pitch = (int)(b.nr > 0 ? b.sq[b.rax[0]] : b.stage);
    return b.stage;
}

// Cost of the store walk under the layout in b, in L1 wavefronts per element: the
// stage reads (each warp-wide read takes as many wavefronts as its worst bank
// conflict, replayed on the bank model in hardware mode over the first warp-steps)
// plus the 128-byte lines each warp-wide store touches.  r_lg == 0: a warp takes 32
// consecutive pieces (b.vec dst elements each) in dst order, on into the next dst run;
// r_lg > 0: 32 >> r_lg consecutive pieces in each of 1 << r_lg consecutive dst runs,
// lanes without a piece counted as work lost.
double block_drain_cost(const BlockPlan& b, int eb, int deb) {
    int64_t ta[kBlockMaxLd], tb[kBlockMaxRuns];
    auto fill = [&](int64_t* t, int64_t n, int na, const int* ax) {
        for (int64_t x = 0; x < n; ++x) {
            int64_t r = x, o = 0;
            for (int k = 0; k < na; ++k) {
                const int64_t e = b.tile[ax[k]];
                o += (r % e) * b.sq[ax[k]];
                r /= e;
            }
            t[x] = o;
        }
    };
    fill(ta, b.Ld, b.nd, b.dax);
    fill(tb, b.Rd, b.nj, b.jax);
    const int64_t V = b.vec, W = b.Ld / V, R = int64_t(1) << b.r_lg, PW = 32 / R;
    const bool flat = b.r_lg == 0;
    const int64_t GW = flat ? 1 : (W + PW - 1) / PW, GR = flat ? 1 : (b.Rd + R - 1) / R;
    const int64_t units = flat ? (W * b.Rd + 31) / 32 : GW * GR;
    const int64_t steps = std::min<int64_t>(units, std::max<int64_t>(1, 64 / V));
    int64_t waves = 0;
    for (int64_t g = 0; g < steps; ++g)
        for (int64_t k = 0; k < V; ++k) {
            int64_t o[32];
            for (int l = 0; l < 32; ++l) {
                int64_t v, j;
                if (flat) {
                    v = (32 * g + l) % W;
                    j = (32 * g + l) / W;
                } else {
                    v = (g % GW) * PW + l % PW;
                    j = (g / GW) * R + l / PW;
                }
                o[l] = v < W && j < b.Rd ? (ta[v * V + k] + tb[j]) / eb : -1;
            }
            waves += bank_degree(32, o, eb, true);
        }
    const int64_t seg = (flat ? 32 : PW) * V * deb;          // bytes of a run segment
    const double lines = (double)(flat ? 1 : R) * (double)((seg + 127) / 128);
    const double lanes = flat ? 1.0 : (double)(W * b.Rd) / (double)(GW * PW * GR * R);
    return ((double)waves / (double)steps + lines) / (32.0 * (double)V * lanes);
}

// The store walk and stage layout the cost above finds cheapest: runs per warp-step
// 1 .. 32 and extra 16-byte steps for the two innermost src-run index axes (stages of
// at most 48 KiB); the fewest runs per warp-step (the longest stores) within 3 % of
// the best.
void block_search(BlockPlan& b, int eb, int deb) {
    int best_r = 0, best_e[6][2] = {};
    double best_c[6];
    const int n0 = b.nr > 0 ? 8 : 1, n1 = b.nr > 1 ? 8 : 1;
    for (int r = 0; r <= 5; ++r) {
        best_c[r] = -1;
        b.r_lg = r;
        for (int e0 = 0; e0 < n0; ++e0)
            for (int e1 = 0; e1 < n1; ++e1) {
                const int extra[kBlockAxes] = {e0, e1, 0, 0};
                if (block_layout(b, eb, extra) > 48 * 1024) continue;
                const double c = block_drain_cost(b, eb, deb);
                if (best_c[r] < 0 || c < best_c[r]) {
                    best_c[r] = c;
                    best_e[r][0] = e0;
                    best_e[r][1] = e1;
                }
            }
    }
    double lo = -1;
    for (int r = 0; r <= 5; ++r)
        if (best_c[r] >= 0 && (lo < 0 || best_c[r] < lo)) lo = best_c[r];
    for (int r = 5; r >= 0; --r)
        if (best_c[r] >= 0 && best_c[r] <= 1.03 * lo) best_r = r;
    b.r_lg = best_r;
    const int extra[kBlockAxes] = {best_e[best_r][0], best_e[best_r][1], 0, 0};
    block_layout(b, eb, extra);
}

}  // namespace

int64_t plan_block(Plan* p, int64_t tile_bytes) {
    const Axes& s = p->sorted;
    const int n = s.n, eb = p->eb, deb = p->deb > 0 ? p->deb : p->eb;   // (dst element bytes)
    // measured on GB300 (12^7 and 12^8 permutes, 9^8 permutes): 12 KiB tiles for 1- and
    // 2-byte elements (12^8 u16 5.6 TB/s against 4.3 at 32 KiB, u8 3.6 against 2.4),
    // 32 KiB for wider ones (9^8 fp32 5.7 TB/s against 4.3 at 12 KiB)
    if (tile_bytes <= 0) tile_bytes = eb <= 2 ? 12288 : 32768;
    if (n < 2) return 0;
    // the dense chains from src stride 1 and from dst stride 1
    auto chain = [&](const int64_t* str, int* out) {
        int m = 0;
        int64_t prod = 1;
        bool used[kMaxDims] = {};
        for (;;) {
            int next = -1;
            for (int i = 0; i < n; ++i)
                if (!used[i] && str[i] == prod) { next = i; break; }
            if (next < 0 || m == kMaxDims) break;
            used[next] = true;
            out[m++] = next;
            prod *= s.ext[next];
        }
        return m;
    };
    int S[kMaxDims], D[kMaxDims];
    const int nS = chain(s.ss, S), nD = chain(s.ds, D);
    if (nS == 0 || nD == 0 || S[0] == D[0]) return 0;
    BlockPlan best;
    int64_t best_score = -1, best_run = 0;
    for (int i = 1; i <= nS; ++i) {
        for (int j = 1; j <= nD; ++j) {
            int T[kMaxDims], nt = 0;
            auto add = [&](int ax) {
                for (int q = 0; q < nt; ++q)
                    if (T[q] == ax) return;
                T[nt++] = ax;
            };
            for (int q = 0; q < i; ++q) add(S[q]);
            for (int q = 0; q < j; ++q) add(D[q]);
            if (nt > kBlockAxes) continue;
            auto in_t = [&](int ax) {
                for (int q = 0; q < nt; ++q)
                    if (T[q] == ax) return q;
                return -1;
            };
            // the runs: the longest prefixes of S and D inside T
            int sr = 0, dr0 = 0;
            while (sr < nS && in_t(S[sr]) >= 0) ++sr;
            while (dr0 < nD && in_t(D[dr0]) >= 0) ++dr0;
            int64_t full = 1;
            for (int q = 0; q < nt; ++q) full *= s.ext[T[q]];
            // candidates for the chunked axis: none, or an axis that is the last of
            // each run it belongs to; a dst run longer than the kernel's position
            // table is cut to a shorter prefix of D (the cut-off axes index dst runs
            // that lie back to back)
            for (int c = -1; c < nt; ++c) {
                int64_t tile[kBlockAxes];
                for (int q = 0; q < nt; ++q) tile[q] = s.ext[T[q]];
                int dr = dr0;
                auto ld_of = [&](int m) {
                    int64_t v = 1;
                    for (int q = 0; q < m; ++q) v *= tile[in_t(D[q])];
                    return v;
                };
                if (c < 0) {
                    if (full * eb > tile_bytes) continue;
                    while (dr > 1 && ld_of(dr) > kBlockMaxLd) --dr;
                } else {
                    const int ax = T[c];
                    if (full * eb <= tile_bytes) continue;
                    const int64_t rest = full / s.ext[ax];
                    int64_t k = tile_bytes / (rest * eb);
                    if (k < 1) continue;
                    const int64_t nc = (s.ext[ax] + k - 1) / k;
                    tile[c] = (s.ext[ax] + nc - 1) / nc;           // chunks evened out
                    while (dr > 1 && ld_of(dr) > kBlockMaxLd) --dr;
                    bool ok = true;
                    for (int q = 0; q < sr - 1; ++q) ok = ok && S[q] != ax;
                    for (int q = 0; q < dr - 1; ++q) ok = ok && D[q] != ax;
                    if (!ok) continue;
                }
                BlockPlan b;
                b.nt = nt;
                b.chunk = c;
                for (int q = 0; q < nt; ++q) {
                    b.idx[q] = T[q];
                    b.ext[q] = s.ext[T[q]];
                    b.ss[q] = s.ss[T[q]];
                    b.ds[q] = s.ds[T[q]];
                    b.tile[q] = tile[q];
                }
                b.Ls = b.Ld = 1;
                for (int q = 0; q < sr; ++q) {
                    b.sax[b.ns++] = in_t(S[q]);
                    b.Ls *= tile[in_t(S[q])];
                }
                for (int q = 0; q < dr; ++q) {
                    b.dax[b.nd++] = in_t(D[q]);
                    b.Ld *= tile[in_t(D[q])];
                }
                int64_t tot = 1;
                for (int q = 0; q < nt; ++q) {
                    tot *= tile[q];
                    bool in_s = false, in_d = false;
                    for (int u = 0; u < b.ns; ++u) in_s = in_s || b.sax[u] == q;
                    for (int u = 0; u < b.nd; ++u) in_d = in_d || b.dax[u] == q;
                    if (!in_s) b.rax[b.nr++] = q;
                    if (!in_d) b.jax[b.nj++] = q;
                }
                b.Rs = tot / b.Ls;
                b.Rd = tot / b.Ld;
                if (b.Ld > kBlockMaxLd || b.Rd > kBlockMaxRuns || b.Rs > kBlockMaxRuns) continue;
                if (b.Ls >= (1 << 24) || block_layout(b, eb, nullptr) > 48 * 1024) continue;
                const int64_t run = std::min(b.Ls, b.Ld) * eb;
                const int64_t score = std::min<int64_t>(run, 512) * (int64_t(1) << 32) + tot;
                if (score > best_score) {
                    best_score = score;
                    best_run = run;
                    best = b;
                }
            }
        }
    }
    if (best_score < 0) return 0;
    // the axes outside T: the batch (dst order, outermost first)
    Axes bt;
    for (int q = 0; q < n; ++q) {
        bool in = false;
        for (int u = 0; u < best.nt; ++u) in = in || best.idx[u] == q;
        if (in) continue;
        bt.ext[bt.n] = s.ext[q]; bt.ss[bt.n] = s.ss[q]; bt.ds[bt.n] = s.ds[q]; ++bt.n;
    }
    best.batch = bt;
    // pieces of vec dst elements stored as one vector: whole pieces in every dst run
    // (and in its part inside a chunk), each piece aligned in dst
    auto in_dst_run = [&](int q) {
        for (int k = 0; k < best.nd; ++k)
            if (best.dax[k] == q) return true;
        return false;
    };
    auto vec_ok = [&](int64_t v) {
        if (best.Ld % v != 0 || p->dst_mis16 % (v * deb) != 0) return false;
        if (best.chunk >= 0) {
            const int c = best.chunk;
            if (in_dst_run(c) && (best.Ld / best.tile[c]) % v != 0) return false;
            if ((best.tile[c] * best.ds[c]) % v != 0) return false;
        }
        for (int k = 0; k < best.nj; ++k)
            if (best.ds[best.jax[k]] % v != 0) return false;
        for (int q = 0; q < bt.n; ++q)
            if (bt.ds[q] % v != 0) return false;
        return true;
    };
    int v = deb >= 16 ? 1 : 16 / deb;
    while (v > 1 && !vec_ok(v)) v >>= 1;
    best.vec = v;
    block_search(best, eb, deb);
    int64_t tiles = 1;
    for (int q = 0; q < best.nt; ++q) tiles *= (best.ext[q] + best.tile[q] - 1) / best.tile[q];
    for (int q = 0; q < bt.n; ++q) tiles *= bt.ext[q];
    p->blk = best;
    p->tiles = tiles;
    return best_run;
}

int make_plan(const void* src, const void* dst, int ndim, const int64_t* shape,
              const int64_t* src_strides, const int64_t* dst_strides, int eb, uint32_t flags,
              int64_t src_bytes, int64_t dst_bytes, Plan* plan, int cast) {
    Plan p;
    if (!valid_eb(eb)) return TL_ERR_ELEM_BYTES;
    // a cast fixes both element sizes: elem_bytes must be its source's
    int deb = eb;
    if (cast != TL_CAST_NONE) {
        if (cast < TL_CAST_NONE || cast > TL_CAST_F16_TO_F32) return TL_ERR_ARG;
        const bool narrow = cast == TL_CAST_F32_TO_BF16 || cast == TL_CAST_F32_TO_F16;
        if (eb != (narrow ? 4 : 2)) return TL_ERR_ELEM_BYTES;
        deb = narrow ? 2 : 4;
    }
    p.cast = cast;
    p.deb = deb;
    if (ndim < 0 || ndim > kMaxDims) return TL_ERR_ARG;
    if (ndim > 0 && (!shape || !src_strides || !dst_strides)) return TL_ERR_ARG;
    uint32_t forced = flags & TL_PATH_MASK;
    if (forced > TL_PATH_BLOCK) return TL_ERR_ARG;
    const bool checked = (flags & TL_FLAG_DEBUG_CHECKS) != 0;
    if ((flags & TL_FLAG_TEST_SKIP_HOST_BOUNDS) && !checked) return TL_ERR_ARG;
    if (checked && cast != TL_CAST_NONE) return TL_ERR_ARG;   // the checked run moves bits
    if (checked) {                 // the checked run is the generic kernel
        if (forced != TL_PATH_AUTO && forced != TL_PATH_GENERIC) return TL_ERR_PATH;
        forced = TL_PATH_GENERIC;
    }
    p.eb = eb;
    int64_t total = 1;
    for (int i = 0; i < ndim; ++i) {
        if (shape[i] < 0 || src_strides[i] < 0 || dst_strides[i] < 0) return TL_ERR_ARG;
        if (!mul_ok(total, shape[i], &total)) return TL_ERR_RANGE;
    }
    p.total = total;
    if (total == 0) {           // nothing to move
        *plan = p;
        return TL_OK;
    }
    if (!src || !dst) return TL_ERR_ARG;
    const int align = eb < 16 ? eb : 16, dalign = deb < 16 ? deb : 16;
    if (!aligned(abs_addr(src), align) || !aligned(abs_addr(dst), dalign)) return TL_ERR_ALIGN;

    int64_t sspan, dspan;
    if (!layout_span(ndim, shape, src_strides, &sspan) ||
        !layout_span(ndim, shape, dst_strides, &dspan))
        return TL_ERR_RANGE;
    int64_t sbytes, dbytes;
    if (!mul_ok(sspan + 1, eb, &sbytes) || !mul_ok(dspan + 1, deb, &dbytes)) return TL_ERR_RANGE;
    p.sbytes = sbytes;
    p.dbytes = dbytes;
    if (((src_bytes > 0 && sbytes > src_bytes) || (dst_bytes > 0 && dbytes > dst_bytes)) &&
        !(flags & TL_FLAG_TEST_SKIP_HOST_BOUNDS))
        return TL_ERR_BOUNDS;
    if (!non_overlapping(ndim, shape, dst_strides)) return TL_ERR_DST_OVERLAP;

    // canonical forms
    Axes raw;
    raw.n = ndim;
    for (int i = 0; i < ndim; ++i) {
        raw.ext[i] = shape[i]; raw.ss[i] = src_strides[i]; raw.ds[i] = dst_strides[i];
    }
    drop_and_merge(raw, &p.kept);
    Axes srt;
    {
        int idx[kMaxDims], m = 0;
        for (int i = 0; i < ndim; ++i)
            if (shape[i] != 1) idx[m++] = i;
        std::stable_sort(idx, idx + m, [&](int a, int b) {
            if (dst_strides[a] != dst_strides[b]) return dst_strides[a] > dst_strides[b];
            return src_strides[a] > src_strides[b];
        });
        Axes t;
        t.n = m;
        for (int q = 0; q < m; ++q) {
            t.ext[q] = shape[idx[q]]; t.ss[q] = src_strides[idx[q]]; t.ds[q] = dst_strides[idx[q]];
        }
        drop_and_merge(t, &srt);
    }
    p.sorted = srt;

    const int64_t s0 = abs_addr(src), d0 = abs_addr(dst);
    const bool ranges_meet = s0 < d0 + dbytes && d0 < s0 + sbytes;

    // eligibility of every path
    // The warp path's swizzle search simulates every candidate; run it only when
    // the warp path can be chosen (aliased buffers, forced, or a tiny tensor).
    const bool warp_wanted = ranges_meet || forced == TL_PATH_WARP ||
                             (forced == TL_PATH_AUTO && total <= kWarpAutoMaxElems);
    // (under a cast only the chunk, tile and generic kernels convert)
    const bool casting = cast != TL_CAST_NONE;
    const bool warp_ok = !casting && warp_wanted && plan_warp(&p);
    bool chunk_ok = false;
    if (srt.n == 0 || (srt.ds[srt.n - 1] == 1 && srt.ss[srt.n - 1] == 1)) chunk_ok = true;
    const bool plane = plan_plane(&p);
    const bool rows = !casting && plane && rows_ok(p, s0, d0);
    const bool cols = !casting && plane && cols_ok(p, s0, d0);
    const bool tile = plane && tile_ok(p, s0);
    const bool panel = !casting && plane && panel_ok(p);

    int path = 0;
    if (ranges_meet) {
        if (casting || !(s0 == d0 && warp_ok && warp_in_place_ok(p))) return TL_ERR_ALIAS;
        if (forced != TL_PATH_AUTO && forced != TL_PATH_WARP) return TL_ERR_PATH;
        p.in_place = true;
        path = TL_PATH_WARP;
    } else switch (forced) {
    case TL_PATH_AUTO:
        if (chunk_ok) path = TL_PATH_CHUNK;
        else if (warp_ok) path = TL_PATH_WARP;
        else if (rows) path = TL_PATH_ROWS;
        else if (cols) path = TL_PATH_COLS;
        else if (tile && tile_fits(p)) path = TL_PATH_TILE;
        else if (panel) path = TL_PATH_PANEL;
        else if (tile) path = TL_PATH_TILE;
        else path = TL_PATH_GENERIC;
        break;
    case TL_PATH_GENERIC: path = TL_PATH_GENERIC; break;
    case TL_PATH_CHUNK: path = chunk_ok ? TL_PATH_CHUNK : 0; break;
    case TL_PATH_WARP: path = warp_ok ? TL_PATH_WARP : 0; break;
    case TL_PATH_ROWS: path = rows ? TL_PATH_ROWS : 0; break;
    case TL_PATH_TILE: path = tile ? TL_PATH_TILE : 0; break;
    case TL_PATH_CLUSTER: path = tile && !casting ? TL_PATH_CLUSTER : 0; break;
    case TL_PATH_PANEL: path = panel ? TL_PATH_PANEL : 0; break;
    case TL_PATH_COLS: path = cols ? TL_PATH_COLS : 0; break;
    case TL_PATH_BLOCK: {
        Plan q = p;
        path = plan_block(&q) > 0 ? TL_PATH_BLOCK : 0;
        break;
    }
    }
    if (path == 0) return TL_ERR_PATH;
    p.src_mis16 = s0 & 15;
    p.dst_mis16 = d0 & 15;
    // The panel tile of the plane: merged short axes, tile shape, stage layout.
    auto setup_panel = [&](Plan& q) {
        q.panel_elem_stores = (flags & TL_FLAG_PANEL_ELEMENT_STORES) != 0;
        panel_merge_b(&q);
        panel_merge_a(&q);
        plan_panel(&q, 0);
    };
    // The block tile takes layouts of canonical rank 3 or more whose panel tile would
    // move short runs on one side (high-rank permutes of short axes) when its own
    // shorter run is 128 bytes or more and at least as long.
    if (forced == TL_PATH_AUTO && !ranges_meet && srt.n >= 3 &&
        (path == TL_PATH_PANEL || path == TL_PATH_GENERIC)) {
        Plan q = p;
        const int64_t brun = plan_block(&q);
        if (brun >= 128) {
            int64_t prun = 0;
            bool pvec = false;                 // the panel tile stores 16-byte dst runs
            if (path == TL_PATH_PANEL) {
                Plan r = p;
                setup_panel(r);
                const int64_t ta = r.tile_cols, tb = r.tile_rows;
                // src rows back to back (one run per tile) or one run per tile row
                const bool packed = ta == r.ext_a && r.ss_b == ta &&
                                    (r.panel_b1 == 0 || r.panel_ss_b2 == r.panel_b1 * ta);
                const int64_t srun = packed ? ta * tb * eb : ta * eb;
                const int64_t drun = r.panel_run ? ta * tb * eb : tb * eb;
                prun = std::min(srun, drun);
                pvec = r.panel_vec || r.panel_run;
            }
            // Against a panel tile stored as 16-byte dst runs the block tile needs few
            // src runs: measured on GB300, reversed 8^8 fp32 (64 runs a tile) 1.19x as
            // blocks and 12^8 fp64 in the interleaved order (24) 1.48x, but `nd6_f32`
            // (128 runs of 256 bytes) 0.38x and reversed 16^7 fp32 (256 runs) 0.33x:
            // their stages hold one CTA per SM.
            if (brun >= prun && !(pvec && q.blk.Rs > 100)) path = TL_PATH_BLOCK;
        }
    }
    p.path = path;

    if (path == TL_PATH_CHUNK) {
        Axes o;
        int64_t row = 1;
        if (srt.n > 0) {
            row = srt.ext[srt.n - 1];
            for (int i = 0; i < srt.n - 1; ++i) {
                o.ext[o.n] = srt.ext[i]; o.ss[o.n] = srt.ss[i]; o.ds[o.n] = srt.ds[i]; ++o.n;
            }
        }
        p.row_elems = row;
        p.outer = o;
        p.rows = total / row;
        p.tiles = p.rows;                  // work units: rows
        if (!casting) {
            int vb = 16;
            auto fits = [&](int64_t v) { return v % vb == 0; };
            while (vb > 1) {
                bool ok = fits(row * eb) && fits(s0) && fits(d0);
                for (int i = 0; i < o.n && ok; ++i)
                    ok = ok && fits(o.ss[i] * eb) && fits(o.ds[i] * eb);
                if (ok) break;
                vb >>= 1;
            }
            p.vec_bytes = vb;
        } else {
            // vectors of 4, 2 or 1 elements, aligned on both sides (vec_bytes: the
            // source side's vector)
            int ve = 4;
            while (ve > 1) {
                const int64_t sv = (int64_t)ve * eb, dv = (int64_t)ve * deb;
                bool ok = row % ve == 0 && s0 % sv == 0 && d0 % dv == 0;
                for (int i = 0; i < o.n && ok; ++i)
                    ok = (o.ss[i] * eb) % sv == 0 && (o.ds[i] * deb) % dv == 0;
                if (ok) break;
                ve >>= 1;
            }
            p.vec_bytes = ve * eb;
        }
    } else if (path == TL_PATH_TILE || path == TL_PATH_CLUSTER) {
        p.tile_cols = 128 / eb;
        p.tile_rows = 128;
        bool vs = (d0 % 16 == 0) && (p.ds_a * deb) % 16 == 0;
        for (int i = 0; i < p.batch.n; ++i) vs = vs && (p.batch.ds[i] * deb) % 16 == 0;
        p.vec_store = vs;
        p.vec_bytes = vs ? 16 : eb;
        const int64_t ta = (p.ext_a + p.tile_cols - 1) / p.tile_cols;
        const int64_t tb = (p.ext_b + p.tile_rows - 1) / p.tile_rows;
        p.tiles = ta * tb * p.batch_total;
    } else if (path == TL_PATH_PANEL) {
        setup_panel(p);
    } else if (path == TL_PATH_BLOCK) {
        plan_block(&p);
        p.vec_bytes = p.blk.vec * deb;
    } else if (path == TL_PATH_COLS) {
        p.vec_bytes = 16;
        p.tile_cols = (int)p.ext_a;          // elements per pixel
        p.tile_rows = 16 / eb;               // pixels per 16-byte piece
        p.tiles = p.batch_total * (p.ext_b / p.tile_rows);
    } else if (path == TL_PATH_ROWS) {
        p.vec_bytes = 16;
        p.tiles = p.batch_total * (p.ext_a * eb / 16);
    } else if (path == TL_PATH_WARP) {
        p.vec_bytes = eb;
        int64_t nb = 1;
        for (int i = 0; i < p.wbatch.n; ++i) nb *= p.wbatch.ext[i];
        p.tiles = nb;
    } else {
        p.vec_bytes = eb;
        p.tiles = total;
    }
    *plan = p;
    return TL_OK;
}

}  // namespace tl

// ---------------------------------------------------------------------------
// C ABI: host-only entry points
// ---------------------------------------------------------------------------
extern "C" {

int tl_layout_canon(const tl_layout* src, const tl_layout* dst, const int64_t* begin,
                    const int64_t* extent, tl_layout* src_out, tl_layout* dst_out,
                    int64_t* chunk_elems) {
    using namespace tl;
    if (!src || !dst || !src_out || !dst_out) return TL_ERR_ARG;
    const int n = src->ndim;
    if (n < 0 || n > kMaxDims || dst->ndim != n) return TL_ERR_ARG;
    Axes sl;
    sl.n = n;
    int64_t so = src->offset, dof = dst->offset;
    bool empty = false;
    for (int i = 0; i < n; ++i) {
        if (src->shape[i] != dst->shape[i] || src->shape[i] < 0) return TL_ERR_ARG;
        const int64_t b = begin ? begin[i] : 0;
        const int64_t e = extent ? extent[i] : src->shape[i] - b;
        if (b < 0 || e < 0 || b + e > src->shape[i]) return TL_ERR_RANGE;
        sl.ext[i] = e;
        sl.ss[i] = src->stride[i];
        sl.ds[i] = dst->stride[i];
        int64_t t;
        if (!mul_ok(b, src->stride[i], &t) || !add_ok(so, t, &so)) return TL_ERR_RANGE;
        if (!mul_ok(b, dst->stride[i], &t) || !add_ok(dof, t, &dof)) return TL_ERR_RANGE;
        empty |= e == 0;
    }
    tl_layout s{}, d{};
    s.offset = so;
    d.offset = dof;
    int64_t chunk;
    if (empty) {
        s.ndim = d.ndim = 1;
        s.shape[0] = d.shape[0] = 0;
        s.stride[0] = d.stride[0] = 1;
        chunk = 0;
    } else {
        Axes c;
        drop_and_merge(sl, &c);
        s.ndim = d.ndim = c.n;
        for (int i = 0; i < c.n; ++i) {
            s.shape[i] = d.shape[i] = c.ext[i];
            s.stride[i] = c.ss[i];
            d.stride[i] = c.ds[i];
        }
        if (c.n == 0) chunk = 1;
        else if (c.ss[c.n - 1] == 1 && c.ds[c.n - 1] == 1) chunk = c.ext[c.n - 1];
        else chunk = 0;
    }
    *src_out = s;
    *dst_out = d;
    if (chunk_elems) *chunk_elems = chunk;
    return TL_OK;
}

int tl_thread_axis_check(int ndim, const int64_t* extent, const int64_t* lane_str,
                         const int64_t* reg_str, int* registers) {
    if (ndim < 1 || ndim > 4 || !extent || !lane_str || !reg_str || !registers)
        return TL_ERR_ARG;
    int64_t total = 1;
    for (int k = 0; k < ndim; ++k) {
        if (extent[k] < 1 || lane_str[k] < 0 || reg_str[k] < 0) return TL_ERR_EXTENT;
        if ((lane_str[k] > 0) == (reg_str[k] > 0)) return TL_ERR_EXTENT;   // one side each
        total *= extent[k];
        if (total > 32 * 256) return TL_ERR_EXTENT;        // at most 256 registers a lane
    }
    if (total % 32 != 0) return TL_ERR_EXTENT;
    const int64_t P = total / 32;
    // every coordinate once on (lane, register), enumerated
    std::vector<char> seen((size_t)total, 0);
    for (int64_t f = 0; f < total; ++f) {
        int64_t x = f, lane = 0, reg = 0;
        for (int k = ndim - 1; k >= 0; --k) {
            const int64_t c = x % extent[k];
            x /= extent[k];
            lane += c * lane_str[k];
            reg += c * reg_str[k];
        }
        if (lane >= 32 || reg >= P) return TL_ERR_EXTENT;
        char& s = seen[(size_t)(lane * P + reg)];
        if (s) return TL_ERR_EXTENT;
        s = 1;
    }
    *registers = (int)P;
    return TL_OK;
}

int tl_choose_xor_k(int ndim, const int64_t* extent, const int64_t* src_str,
                    const int64_t* dst_str, int elem_bytes, int* k, int* shift, int* mask) {
    if (!extent || !src_str || !dst_str || !k || !shift || !mask) return TL_ERR_ARG;
    return tl::choose_xor(ndim, extent, src_str, dst_str, elem_bytes, k, shift, mask);
}

int tl_bank_conflicts(int n_lanes, const int64_t* lane_offsets, int elem_bytes, int model) {
    if (!lane_offsets || n_lanes < 0 || n_lanes > 32 || (model != 0 && model != 1))
        return TL_ERR_ARG;
    if (!tl::valid_eb(elem_bytes)) return TL_ERR_ELEM_BYTES;
    return tl::bank_degree(n_lanes, lane_offsets, elem_bytes, model == 1);
}

const char* tl_status_string(int status) {
    switch (status) {
    case TL_OK: return "ok";
    case TL_ERR_ARG: return "invalid argument";
    case TL_ERR_ELEM_BYTES: return "element width must be 1, 2, 4, 8 or 16 bytes";
    case TL_ERR_EXTENT: return "extent is not a whole number of warp iterations";
    case TL_ERR_NO_VALID_K: return "no XOR swizzle makes both phases bank-conflict-free";
    case TL_ERR_CHUNK: return "contiguous chunk is under 16 bytes or not a multiple of 16";
    case TL_ERR_DST_OVERLAP: return "destination layout may map two coordinates to one element";
    case TL_ERR_ALIAS: return "source and destination memory overlap";
    case TL_ERR_ALIGN: return "pointer not aligned to the element width";
    case TL_ERR_PATH: return "the requested kernel path does not apply to this layout";
    case TL_ERR_RANGE: return "offset overflow or region outside the layout";
    case TL_ERR_CUDA: return "CUDA call failed";
    case TL_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case TL_ERR_BOUNDS: return "layout reaches outside the given buffer size";
    default: return "unknown status";
    }
}

int tl_version(void) { return TL_VERSION; }

}  // extern "C"
