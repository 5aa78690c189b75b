"""The kernels' index maps, derived on the host from Shape/Stride layouts
(logical_divide / zipped_divide of the operand and output layouts,
local_partition of the TMEM accumulator layout; "Advanced CUTLASS Architecture
and Kernel Optimization", Advanced Layout Operations, and the transpose kernel
of "4.21 What is CuTe?"), must equal the maps the kernels were written for:
tile origins, each CTA's share of a pair tile, the TMA boxes of every
majorness, and the epilogue's thread -> (row, column) and TMEM maps.  Every
tile width of both GEMM kernels and all four A/B majorness combinations."""
import os
import subprocess

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "tests", "cpp", "index_maps_driver.cpp")


@pytest.fixture(scope="module")
def derive(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("maps") / "index_maps_driver")
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(ROOT, "tiled_tensor_core_02_gb300", "csrc"), SRC, "-o", exe], check=True)

    def run(keys):
        inp = "\n".join(" ".join(str(int(v)) for v in k) for k in keys) + "\n"
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout.splitlines()
        res = []
        for line in out:
            assert not line.startswith("error"), line
            v = [int(x) for x in line.split()]
            box = lambda i: dict(zip(("k_inner", "inner", "outer", "boxes", "step", "smem"), v[i:i + 6]))
            res.append({"tile": (v[0], v[1]), "cta": (v[2], v[3]), "a": box(4), "b": box(10),
                        "half": (v[16], v[17]), "b_half": box(18), "epi": (v[24], v[25], v[26])})
        return res
    return run


def boxes_swizzled(k_major, rows, esize=2):
    """A k-block tile of `rows` rows x 64 k as the kernels load it: K-major, one
    box of 64 k x rows; MN-major, slabs of 64 rows x 64 k, 8 KB apart (at
    least one slab)."""
    if k_major:
        return {"k_inner": 1, "inner": 64, "outer": rows, "boxes": 1, "step": 64, "smem": 64 * rows * esize}
    n = max(1, (rows + 63) // 64)
    return {"k_inner": 0, "inner": 64, "outer": 64, "boxes": n, "step": 64, "smem": 64 * 64 * esize}


MAJORNESS = [(a, b) for a in (0, 1) for b in (0, 1)]  # a_mn, b_mn


@pytest.mark.parametrize("a_mn,b_mn", MAJORNESS)
def test_single_cta_maps(derive, a_mn, b_mn):
    keys, want = [], []
    for bn in (256, 128, 64, 32):
        if b_mn and bn < 64:
            continue  # an MN-major B needs whole 64-column slabs
        for a_rows in (128, 72, 64, 16, 8):
            keys.append((128, bn, 1, a_rows, a_mn, b_mn, 2, 1, 0))
            want.append((bn, a_rows))
    for got, (bn, a_rows) in zip(derive(keys), want):
        assert got["tile"] == (128, bn)          # tile (mb, nb) at (128 mb, bn nb)
        assert got["cta"] == (0, 0)              # one CTA per tile
        assert got["a"] == boxes_swizzled(not a_mn, a_rows)
        assert got["b"] == boxes_swizzled(not b_mn, bn)
        assert got["epi"] == (1, 1 << 16, 32)    # thread t: row t, TMEM lane t; 32-column chunks


@pytest.mark.parametrize("a_mn,b_mn", MAJORNESS)
def test_pair_maps(derive, a_mn, b_mn):
    keys, want = [], []
    for pbn in (256, 224, 192, 128):
        if b_mn and pbn in (224, 192):
            continue  # a CTA's 112 or 96 columns are not whole MN-major slabs
        keys.append((256, pbn, 2, 128, a_mn, b_mn, 2, 1, pbn // 2 if pbn == 256 else 0))
        want.append(pbn)
    for got, pbn in zip(derive(keys), want):
        assert got["tile"] == (256, pbn)
        assert got["cta"] == (128, pbn // 2)    # CTA r: A rows from 128 r, B columns from r pbn / 2
        assert got["a"] == boxes_swizzled(not a_mn, 128)
        assert got["b"] == boxes_swizzled(not b_mn, pbn // 2)
        if pbn == 256:
            assert got["half"] == (128, 64)      # half h from column 128 h; CTA r from 64 r
            assert got["b_half"] == boxes_swizzled(not b_mn, 64)
        assert got["epi"] == (1, 1 << 16, 32)


@pytest.mark.parametrize("a_mn,b_mn", MAJORNESS)
def test_int8_staging_maps(derive, a_mn, b_mn):
    """Raw int8 tiles, unswizzled: K-major boxes of 64 k x rows, MN-major boxes
    of rows x 64 k, one box each."""
    for bn in (128, 64, 32):
        got = derive([(128, bn, 1, 128, a_mn, b_mn, 1, 0, 0)])[0]
        for rows, mn, g in ((128, a_mn, got["a"]), (bn, b_mn, got["b"])):
            want = ({"k_inner": 0, "inner": rows, "outer": 64} if mn else {"k_inner": 1, "inner": 64, "outer": rows})
            assert {k: g[k] for k in ("k_inner", "inner", "outer")} == want
            assert g["boxes"] == 1 and g["smem"] == rows * 64


def test_maps_do_not_depend_on_problem_extents(derive):
    """The derivation takes only the tile configuration: the same key gives the
    same maps however often it is asked (the planner caches them by key)."""
    k = (256, 256, 2, 128, 1, 0, 2, 1, 128)
    a, b = derive([k, k])
    assert a == b
