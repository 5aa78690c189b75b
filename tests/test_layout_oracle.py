"""Pins for the layout-algebra oracle against the pages' worked examples.

Each golden fixture under tests/golden states its source; these tests check
that the plain definitions in oracle/layout.py reproduce the printed values.
"""
import ast

from conftest import read_golden
from oracle import layout as L


def parse_tuple(s):
    return ast.literal_eval(s)


def test_rowmajor_4x8_crd2idx():
    g = read_golden("layout_rowmajor_4x8.txt")
    shape = tuple(int(v) for v in g[0][1:])
    stride = tuple(int(v) for v in g[1][1:])
    for r, c, idx in g[2:]:
        assert L.crd2idx((int(r), int(c)), shape, stride) == int(idx)
    # and as a function of the colexicographic flat index (column-major walk)
    assert L.table(shape, stride)[:4] == [0, 8, 16, 24]
    assert L.is_bijective_onto(shape, stride, 32)


def test_logical_divide_1024_by_128():
    g = read_golden("logical_divide_1024_128.txt")
    shape, stride = int(g[0][1]), int(g[0][2])
    ts, td = int(g[1][1]), int(g[1][2])
    sizes = [int(v) for v in g[2][1:]]
    dom, tab = L.logical_divide_table(shape, stride, ts, td)
    assert [L.size(m) for m in dom] == sizes
    for i, t, off in g[3:]:
        flat = int(i) + sizes[0] * int(t)
        assert tab[flat] == int(off)
    assert L.complement(ts, td, shape) == ((8,), (128,))


def test_ldmatrix_x1_tv_layout():
    """(lane, value) -> 8x8 row-major offset: lane = l0 + 4 l1, value v.
    row = l1, col = 2 l0 + v, i.e. ((4, 8), 2) : ((2, 8), 1)."""
    shape, stride = ((4, 8), 2), ((2, 8), 1)
    for lane, r0, c0, r1, c1 in read_golden("ldmatrix_x1.txt"):
        lane = int(lane)
        o0 = L.crd2idx((lane, 0), shape, stride)
        o1 = L.crd2idx((lane, 1), shape, stride)
        assert divmod(o0, 8) == (int(r0), int(c0))
        assert divmod(o1, 8) == (int(r1), int(c1))
    assert L.is_bijective_onto(shape, stride, 64)


def test_ldmatrix_x4_tables_match_alayout():
    """Part 2's x4 table and Part 3's ALayout describe the same fragment."""
    g = read_golden("ldmatrix_x4.txt")
    shape, stride = ((4, 8), (2, 2, 2)), ((32, 1), (16, 8, 128))
    reg_of_mat = {}
    for row in g:
        if row[0] == "mat":
            _, m, t0, t1, r0, r1, k0, k1, reg = row
            reg_of_mat[int(m)] = (int(r0), int(r1), int(k0), int(k1), reg)
    for row in g:
        if row[0] == "t5":
            reg, r, c = row[1], int(row[2]), int(row[3])
            d = int(reg[1])
            # register d holds values 2d, 2d+1 of the thread
            for v in (2 * d, 2 * d + 1):
                idx = L.crd2idx((5, v), shape, stride)
                m, k = idx % 16, idx // 16
                assert (m, k) == (r, c + (v - 2 * d))
                r0, r1, k0, k1, regname = reg_of_mat[d]
                assert r0 <= m <= r1 and k0 <= k <= k1 and regname == reg


def test_sm80_alayout():
    g = read_golden("sm80_alayout.txt")
    shape = parse_tuple(g[0][1])
    stride = parse_tuple(g[1][1])
    assert shape == ((4, 8), (2, 2, 2)) and stride == ((32, 1), (16, 8, 128))
    modes = [r for r in g if r[0] == "mode"]
    flat_s, flat_d = L.flatten(shape), L.flatten(stride)
    assert [int(r[2]) for r in modes] == flat_s
    assert [int(r[3]) for r in modes] == flat_d
    for tag in ("t0", "t5"):
        row = next(r for r in g if r[0] == tag)
        t = int(tag[1:])
        coords = [(int(row[1 + 2 * v]), int(row[2 + 2 * v])) for v in range(8)]
        got = []
        for v in range(8):
            idx = L.crd2idx((t, v), shape, stride)
            got.append((idx % 16, idx // 16))
        assert got == coords
    assert L.is_bijective_onto(shape, stride, 256)


def test_stripmined_map_64x64():
    g = {r[0]: r[1:] for r in read_golden("stripmined_64x64.txt") if not r[0].isdigit()}
    rows = [r for r in read_golden("stripmined_64x64.txt") if r[0].isdigit()]
    R, C = int(g["tile"][0]), int(g["tile"][1])
    T, V, I = int(g["threads"][0]), int(g["vec"][0]), int(g["iterations"][0])
    assert R * C // T // V == I
    for r in rows:
        tid, cg, c0, c1, ra = (int(v) for v in r[:5])
        want_rows = [int(v) for v in r[5:]]
        for it in range(I):
            row, col = L.stripmined_coords(R, C, T, V, tid, it)
            assert row == want_rows[it] and col == c0 and c0 + V - 1 == c1
            assert col // V == cg and row % int(g["row_stride"][0]) == ra
    # the same map as a layout (thread, vec, iter) -> row-major tile offset
    shape = ((16, 8), 4, 8)
    stride = ((4, 64), 1, 512)
    for tid in range(T):
        for it in range(I):
            row, col = L.stripmined_coords(R, C, T, V, tid, it)
            for v in range(V):
                assert L.crd2idx((tid, v, it), shape, stride) == row * C + col + v
    assert L.is_bijective_onto(shape, stride, R * C)


def test_predicate_m63_reading():
    g = {r[0]: r[1:] for r in read_golden("predicate_m63.txt")}
    er, ec = (int(v) for v in g["extent"])
    masked = [(t, it) for t in range(128) for it in range(8)
              if not L.stripmined_predicate(64, 64, 128, 4, er, ec, t, it)]
    lo, hi = (int(v) for v in g["masked_tids"])
    it = int(g["masked_iteration"][0])
    assert masked == [(t, it) for t in range(lo, hi + 1)]
    assert len(masked) * 4 == int(g["masked_elements"][0])
    # a stride re-derived from the ragged extent skips rows
    fs = int(g["floor_stride"][0])
    visited = {ra + k * fs for ra in range(8) for k in range(8)}
    u0, u1 = (int(v) for v in g["unvisited_rows"])
    assert all(r not in visited for r in range(u0, u1 + 1))


def test_transpose_partition():
    rows = read_golden("transpose_partition.txt")
    thr_shape, thr_stride = (8, 32), (32, 1)  # row-major (8, 32) thread grid
    for r in rows[2:]:
        t = int(r[0])
        want = [int(v) for v in r[1:5]]
        col = int(r[5])
        # invert the thread layout: the coordinate whose index is t
        crd = next((i, j) for i in range(8) for j in range(32)
                   if L.crd2idx((i, j), thr_shape, thr_stride) == t)
        owned = [(crd[0] + 8 * j, crd[1]) for j in range(4)]
        assert [o[0] for o in owned] == want and all(o[1] == col for o in owned)


def test_composition_is_function_composition():
    # (4,8):(8,1) o (8,4):(4,1) transposes the walk order
    a = ((4, 8), (8, 1))
    b = ((8, 4), (4, 1))
    tab = L.compose_table(a[0], a[1], b[0], b[1])
    for i in range(32):
        assert tab[i] == L.evaluate(a[0], a[1], L.evaluate(b[0], b[1], i))


def test_zipped_divide_matches_transpose_closed_form():
    """"4.21 What is CuTe?", transpose kernel: a tensor divided into 32 x 32
    blocks and indexed as ((i, j), bx, by) holds element (bx*32 + i, by*32 + j)
    of the undivided tensor.  For a row-major M x N tensor that element sits at
    (bx*32 + i)*N + by*32 + j; for the kernel's column-major output view at
    (bx*32 + i) + (by*32 + j)*M.  The divided domain is ((32, 32), (M/32, N/32)),
    walked colexicographically, so the flat index of ((i, j), (bx, by)) is
    i + 32 j + 1024 (bx + (M/32) by)."""
    for M, N in [(32, 32), (64, 64), (96, 64), (64, 160), (128, 96)]:
        nbx, nby = M // 32, N // 32
        for stride, closed in [((N, 1), lambda r, c: r * N + c), ((1, M), lambda r, c: r + c * M)]:
            dom, tab = L.zipped_divide_table((M, N), stride, (32, 32))
            assert dom == ((32, 32), (nbx, nby))
            assert len(tab) == M * N
            for bx in range(nbx):
                for by in range(nby):
                    for i in range(32):
                        for j in range(32):
                            flat = i + 32 * j + 1024 * (bx + nbx * by)
                            assert tab[flat] == closed(bx * 32 + i, by * 32 + j), (M, N, stride, bx, by, i, j)
            # every element of the tensor appears exactly once
            assert sorted(tab) == sorted(closed(r, c) for r in range(M) for c in range(N))


def test_complement_multi_mode_hand_worked():
    """complement(L, m), worked by hand from its definition: take L's modes in
    order of stride; each gap between the range covered so far (the previous
    extent x stride) and the next stride becomes a mode of the complement
    (extent = stride / covered, stride = covered); a last mode repeats the
    covered range up to m."""
    # (2,2):(1,4) in 16.  Sorted: 2:1 covers [0,2); 4 / 2 = 2 -> mode 2:2; 2:4
    # covers up to 8; 16 / 8 = 2 -> mode 2:8.  Image {0,1,4,5} + {0,2,8,10} = [0,16).
    assert L.complement((2, 2), (1, 4), 16) == ((2, 2), (2, 8))
    # 4:2 in 64.  The stride 2 leaves a gap of 2 -> mode 2:1; 4:2 covers up to 8;
    # 64 / 8 = 8 -> mode 8:8.  Image {0,2,4,6} + {0,1} + {0,8,..,56} = [0,64).
    assert L.complement(4, 2, 64) == ((2, 8), (1, 8))
    # (4,2):(1,16) in 128.  4:1 covers [0,4); 16 / 4 = 4 -> mode 4:4; 2:16 covers
    # up to 32; 128 / 32 = 4 -> mode 4:32.
    assert L.complement((4, 2), (1, 16), 128) == ((4, 4), (4, 32))
    # modes listed out of stride order give the same complement: (2,4):(8,1) in 64.
    # 4:1 covers [0,4); 8 / 4 = 2 -> mode 2:4; 2:8 covers up to 16; 64 / 16 = 4 -> 4:16.
    assert L.complement((2, 4), (8, 1), 64) == ((2, 4), (4, 16))
    # a stride-0 (broadcast) mode and an extent-1 mode take no part
    assert L.complement((3, 1, 4), (0, 7, 1), 8) == ((2,), (4,))
    # defining property, for each case: L followed by its complement is a
    # bijection onto [0, m)
    for shape, stride, m in [((2, 2), (1, 4), 16), (4, 2, 64), ((4, 2), (1, 16), 128), ((2, 4), (8, 1), 64)]:
        cs, cd = L.complement(shape, stride, m)
        both_s = (shape, cs) if isinstance(shape, tuple) else ((shape,), cs)
        both_d = (stride, cd) if isinstance(stride, tuple) else ((stride,), cd)
        assert L.is_bijective_onto(both_s, both_d, m), (shape, stride, m)


def test_logical_divide_by_strided_tiler_hand_worked():
    """logical_divide(16:1, 4:2) = 16:1 o (4:2, complement(4:2, 16)).
    complement(4:2, 16) = (2,2):(1,8) (the gap 2:1, then the repeat 2:8), so the
    divided layout maps (i, (a, b)) to 2 i + a + 8 b: tile 0 = {0,2,4,6},
    tile 1 = {1,3,5,7}, tile 2 = {8,..,14}, tile 3 = {9,..,15}."""
    assert L.complement(4, 2, 16) == ((2, 2), (1, 8))
    dom, tab = L.logical_divide_table(16, 1, 4, 2)
    assert [L.size(m) for m in dom] == [4, 4]
    tiles = [tab[4 * t:4 * t + 4] for t in range(4)]
    assert tiles == [[0, 2, 4, 6], [1, 3, 5, 7], [8, 10, 12, 14], [9, 11, 13, 15]]
