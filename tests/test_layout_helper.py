"""The product's layout helper (include/ttc_layout.hpp) against the pages'
worked examples (tests/golden) and the layout oracle's definitions."""
import ast
import itertools
import os
import random
import subprocess

import pytest

from conftest import ROOT, read_golden
from oracle import layout as L

DRIVER_SRC = os.path.join(ROOT, "tests", "cpp", "layout_driver.cpp")


@pytest.fixture(scope="module")
def helper(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("layout") / "layout_driver")
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"), DRIVER_SRC, "-o", exe],
                   check=True)

    def run(cmds):
        out = subprocess.run([exe], input="\n".join(cmds) + "\n", capture_output=True, text=True, check=True)
        return out.stdout.splitlines()
    return run


def tstr(t):
    return str(t).replace(" ", "")


def split_result(line):
    assert not line.startswith("error"), line
    lay, vals = line.split(" | ")
    return lay, [int(v) for v in vals.split()]


def test_golden_layouts_through_helper(helper):
    # 4x8 row-major
    g = read_golden("layout_rowmajor_4x8.txt")
    cmds = [f"crd (4,8) (8,1) ({r},{c})" for r, c, _ in g[2:]]
    assert [int(x) for x in helper(cmds)] == [int(r[2]) for r in g[2:]]
    # SM80 A layout: thread 0 and thread 5
    sa = read_golden("sm80_alayout.txt")
    shape, stride = ast.literal_eval(sa[0][1]), ast.literal_eval(sa[1][1])
    for tag in ("t0", "t5"):
        row = next(r for r in sa if r[0] == tag)
        t = int(tag[1:])
        cmds = [f"crd {tstr(shape)} {tstr(stride)} ({t},{v})" for v in range(8)]
        idx = [int(x) for x in helper(cmds)]
        got = [(i % 16, i // 16) for i in idx]
        want = [(int(row[1 + 2 * v]), int(row[2 + 2 * v])) for v in range(8)]
        assert got == want
    # ldmatrix x1
    rows = read_golden("ldmatrix_x1.txt")
    cmds = [f"crd ((4,8),2) ((2,8),1) ({r[0]},{v})" for r in rows for v in (0, 1)]
    out = [int(x) for x in helper(cmds)]
    for k, r in enumerate(rows):
        assert divmod(out[2 * k], 8) == (int(r[1]), int(r[2]))
        assert divmod(out[2 * k + 1], 8) == (int(r[3]), int(r[4]))


def test_logical_divide_golden(helper):
    g = read_golden("logical_divide_1024_128.txt")
    lay, vals = split_result(helper(["divide 1024 1 128 1"])[0])
    assert lay == "(128,8):(1,128)"
    for i, t, off in g[3:]:
        assert vals[int(i) + 128 * int(t)] == int(off)
    assert helper(["complement 128 1 1024"]) == ["8:128"]


def test_stripmined_golden(helper):
    lay, vals = split_result(helper(["stripmined 64 64 128 4"])[0])
    assert lay == "((16,8),4,8):((4,64),1,512)"
    rows = [r for r in read_golden("stripmined_64x64.txt") if r[0].isdigit()]
    for r in rows:
        tid, c0 = int(r[0]), int(r[2])
        want_rows = [int(v) for v in r[5:]]
        for it in range(8):
            # flat index of (tid, vec 0, it) in the colexicographic domain (128, 4, 8)
            off = vals[tid + 128 * 4 * it]
            assert divmod(off, 64) == (want_rows[it], c0)
    assert sorted(vals) == list(range(4096))
    assert helper(["stripmined 64 64 120 4"])[0].startswith("error")


def random_layout(rng, max_modes=3):
    n = rng.randint(1, max_modes)
    shape = tuple(rng.choice([1, 2, 3, 4, 8]) for _ in range(n))
    stride = tuple(rng.choice([0, 1, 2, 4, 8, 16, 32]) for _ in range(n))
    if rng.random() < 0.3 and n >= 2:
        shape, stride = ((shape[0], shape[1]),) + shape[2:], ((stride[0], stride[1]),) + stride[2:]
    return shape, stride


def test_eval_matches_oracle_on_random_layouts(helper):
    rng = random.Random(5)
    cases = [random_layout(rng) for _ in range(200)]
    out = helper([f"eval {tstr(s)} {tstr(d)}" for s, d in cases])
    for (s, d), line in zip(cases, out):
        assert [int(v) for v in line.split()] == L.table(s, d)


def test_composition_matches_function_composition(helper):
    # compact left operands and tiling right operands: the cases composition is defined for
    cases = []
    for a_shape in [(4, 8), (8, 4), (2, 3, 4), (16,), ((4, 2), 8)]:
        size = L.size(a_shape)
        a_stride = []
        acc = 1
        for x in L.flatten(a_shape):
            a_stride.append(acc)
            acc *= x
        # column-major compact stride, re-nested like the shape
        it = iter(a_stride)
        def nest(s):
            return tuple(nest(e) for e in s) if isinstance(s, tuple) else next(it)
        a_st = nest(a_shape)
        for b in [((size,), (1,)), ((2, size // 2), (size // 2, 1)), ((size // 2,), (2,)),
                  ((2, 2), (1, size // 2))]:
            if L.size(b[0]) * 1 <= size and all(x > 0 for x in L.flatten(b[0])):
                cases.append((a_shape, a_st, b[0], b[1]))
    out = helper([f"compose {tstr(a)} {tstr(ad)} {tstr(b)} {tstr(bd)}" for a, ad, b, bd in cases])
    checked = 0
    for (a, ad, b, bd), line in zip(cases, out):
        if line.startswith("error"):
            continue
        _, vals = split_result(line)
        assert vals == L.compose_table(a, ad, b, bd), (a, ad, b, bd)
        checked += 1
    assert checked >= 12


def test_logical_divide_matches_oracle(helper):
    cases = [(1024, 1, 128, 1), (64, 1, 8, 1), (96, 1, 32, 1), (64, 1, 4, 2)]
    out = helper([f"divide {a} {b} {c} {d}" for a, b, c, d in cases])
    for (ls, ld, ts, td), line in zip(cases, out):
        _, vals = split_result(line)
        _, want = L.logical_divide_table(ls, ld, ts, td)
        assert vals == want


def test_logical_product_replicates(helper):
    # (4:1) x (3:1): three copies of a 4-element run, placed 4 apart
    lay, vals = split_result(helper(["product 4 1 3 1"])[0])
    assert vals == list(range(12))
    lay, vals = split_result(helper(["product (2,2) (1,4) 2 1"])[0])
    # A covers {0,1,4,5}; its complement fills {2,3} and repeats: copies at +0 and +2
    assert vals == [0, 1, 4, 5, 2, 3, 6, 7]


def test_swizzle_128_equals_element_swizzle_333_and_avoids_bank_conflicts(helper):
    # byte Swizzle<3,4,3> on 2-byte elements == element Swizzle<3,3,3>:
    # element bits [3,6) ^= bits [6,9)
    offs = list(range(0, 8192, 2))
    out = [int(x) for x in helper([f"swizzle 3 {o}" for o in offs])]
    for o, y in zip(offs, out):
        e = o // 2
        e_sw = e ^ ((e >> 6 & 7) << 3)
        assert y == 2 * e_sw
    # [T] Part 4: eight rows read at the same logical 16-byte chunk land in
    # eight different chunks (hence different banks) of the 128-byte row
    for chunk in range(8):
        phys = [int(x) for x in helper([f"swizzle 3 {row * 128 + chunk * 16}" for row in range(8)])]
        assert sorted((p % 128) // 16 for p in phys) == list(range(8))


def test_local_partition_matches_transpose_golden(helper):
    """Thread t of a row-major (8, 32) thread grid over a 32 x 32 row-major tile
    owns rows t/32 + 8j of column t mod 32 (reading T4 of the transpose kernel)."""
    rows = read_golden("transpose_partition.txt")
    for r in rows[2:]:
        t = int(r[0])
        want = [int(v) * 32 + int(r[5]) for v in r[1:5]]
        out = helper([f"partition (32,32) (32,1) (8,32) (32,1) {t}"])[0]
        off, vals = out.split(" | ")
        assert [int(v) for v in vals.split()] == want
        assert L.local_partition_offsets((32, 32), (32, 1), (8, 32), (32, 1), t) == want


def test_local_partition_random(helper):
    rng = random.Random(3)
    cases = []
    for _ in range(40):
        tm, tn = rng.choice([1, 2, 4, 8]), rng.choice([1, 2, 4, 8])
        M, N = tm * rng.choice([1, 2, 3, 4]), tn * rng.choice([1, 2, 3])
        tile = ((M, N), rng.choice([(N, 1), (1, M), (N + 3, 1)]))
        thr = ((tm, tn), rng.choice([(tn, 1), (1, tm)]))
        idx = rng.randrange(tm * tn)
        cases.append((tile, thr, idx))
    out = helper([f"partition {tstr(tl[0])} {tstr(tl[1])} {tstr(th[0])} {tstr(th[1])} {i}" for tl, th, i in cases])
    for (tl, th, i), line in zip(cases, out):
        vals = [int(v) for v in line.split(" | ")[1].split()]
        assert vals == L.local_partition_offsets(tl[0], tl[1], th[0], th[1], i), (tl, th, i)


def test_zipped_and_tiled_divide(helper):
    rng = random.Random(4)
    for _ in range(30):
        t0, t1 = rng.choice([1, 2, 4, 8]), rng.choice([1, 2, 4])
        M, N = t0 * rng.choice([1, 2, 3]), t1 * rng.choice([1, 2, 4])
        stride = rng.choice([(N, 1), (1, M), (N + 5, 1)])
        dom, tab = L.zipped_divide_table((M, N), stride, (t0, t1))
        z = helper([f"zdivide ({M},{N}) {tstr(stride)} {t0} {t1}"])[0]
        lay, vals = split_result(z)
        assert vals == tab
        t = helper([f"tdivide ({M},{N}) {tstr(stride)} {t0} {t1}"])[0]
        lay_t, vals_t = split_result(t)
        assert vals_t == tab  # same function, rest modes flattened
        assert lay_t.count("(") >= 2
