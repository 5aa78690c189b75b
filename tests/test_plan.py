"""The planner on the CPU (ttc_gemm_plan: no GPU touched): which kernels the
benchmark configurations get, and over 10,000 seeded random problems
(sizes from 1 to 10000, every majorness, padded and odd pitches, base
pointers off alignment, batches, workspaces, beta) that no valid call is
refused and that every plan keeps the rules its kernels rely on: TMA only
on 16-byte aligned bases, pitches and batch strides, vector loads only where
every group start is aligned, the CTA-pair kernel only untransposed and
unsplit, and one recorded launch per counted launch."""
import re

import numpy as np
import pytest

import tiled_tensor_core_02_gb300 as ttc
from tiled_tensor_core_02_gb300 import _build

R, COL = ttc.ROW_MAJOR, ttc.COL_MAJOR
BASE = 1 << 36  # fake, widely spaced device addresses: only their alignment matters
SMS = 152


@pytest.fixture(autouse=True, scope="module")
def built():
    _build.build()  # nvcc cross-compiles here; nothing below touches a GPU
    ttc.load()


def plan(M, N, K, dtype="bf16", la="row", lb="col", lda=None, ldb=None, ldc=None, ldd=None, beta=0.0,
         workspace=None, offs=(0, 0, 0, 0), batch=1, strides=(0, 0, 0, 0), sm_count=SMS):
    """(status, items, addresses) for one call; workspace: None, "repack" or "staged"."""
    es, oes = (1, 4) if dtype == "i8" else (2, 2)
    lda = lda if lda is not None else (K if la == "row" else M)
    ldb = ldb if ldb is not None else (N if lb == "row" else K)
    ldc = ldc if ldc is not None else N
    ldd = ldd if ldd is not None else N
    A, B = BASE + offs[0] * es, 2 * BASE + offs[1] * es
    C, D = 3 * BASE + offs[2] * oes, 4 * BASE + offs[3] * oes
    lay = {"row": R, "col": COL}
    dt = ttc.DTYPE[dtype]
    ws, wsb = None, 0
    if workspace == "repack":
        wsb = ttc.ttc_gemm_workspace_size(M, N, K, A, lda, lay[la], B, ldb, lay[lb], dt)
    elif workspace == "staged":
        wsb = ttc.ttc_gemm_workspace_size_staged(M, N, K, A, lda, lay[la], B, ldb, lay[lb], D, ldd, dt)
    if wsb:
        ws = 5 * BASE
    n0 = ttc.ttc_launch_count()
    st, text = ttc.ttc_gemm_plan(batch, M, N, K, A, lda, strides[0], lay[la], B, ldb, strides[1], lay[lb],
                                 C if beta else None, ldc, strides[2], D, ldd, strides[3], 1.0, beta, None, 0, dt, ws,
                                 wsb, sm_count)
    items = [dict([("kernel", it.split()[0])] + [kv.split("=") for kv in it.split()[1:]])
             for it in text.split("; ") if it]
    assert ttc.ttc_launch_count() - n0 == (len(items) if st == 0 else ttc.ttc_launch_count() - n0)
    return st, items, dict(A=A, B=B, C=C, D=D, lda=lda, ldb=ldb, ldc=ldc, ldd=ldd)


def kernels(items):
    return [it["kernel"] for it in items]


# ------------------------------------------------------------------ the benchmark configurations

def test_benchmark_configurations_take_the_intended_kernels():
    st, it, _ = plan(8192, 8192, 8192)
    assert st == 0 and kernels(it) == ["pair"] and it[0]["bn"] == "256" and it[0]["d_tma"] == "1"
    assert it[0]["clusters"] == "76" and it[0]["tiles"] == "1024"
    st, it, _ = plan(4096, 4096, 4096, beta=0.5)
    assert kernels(it) == ["pair"] and it[0]["bn"] == "224" and it[0]["tiles"] == "304"
    st, it, _ = plan(8192, 14336, 4096)
    assert kernels(it) == ["pair"] and it[0]["bn"] == "256" and it[0]["tiles"] == "1792"
    # int8: with the staged workspace the fp16 copies and the pair kernel, else the single-CTA kernel
    st, it, _ = plan(8192, 8192, 8192, dtype="i8", workspace="staged")
    assert kernels(it) == ["widen_i8", "pair_i8"]
    st, it, _ = plan(8192, 8192, 8192, dtype="i8")
    assert kernels(it) == ["single"] and it[0]["mode"] == "tma_i8_tmem_a"
    # ragged, tight odd pitches: one repack launch, then twelve epilogue warps writing D's rows
    st, it, _ = plan(4099, 3001, 1023, beta=1.0, workspace="staged")
    assert kernels(it) == ["repack", "pair"] and it[0]["a"] == "1" and it[0]["b"] == "1"
    assert it[1]["ew"] == "12" and it[1]["d_tma"] == "0" and it[1]["tiles"] == "204"
    # skinny: the long operand on the MMA's 128-row side, K split over a cluster
    st, it, _ = plan(16, 8192, 8192, beta=1.0)
    assert kernels(it) == ["single"] and it[0]["swap"] == "1" and it[0]["ksplit"] == "2" and it[0]["bn"] == "32"
    st, it, _ = plan(8192, 24, 4096, beta=1.0)
    assert kernels(it) == ["single"] and it[0]["swap"] == "0" and it[0]["ksplit"] == "2"
    # matrix-vector: the reduction, or the outputs, contiguous in the matrix
    assert kernels(plan(1, 4096, 4096)[1]) == ["gemv_rows"]
    assert kernels(plan(1, 4096, 4096, lb="row")[1]) == ["gemv_cols"]
    st, it, _ = plan(256, 256, 256, dtype="f16")
    assert kernels(it) == ["single"] and it[0]["mode"] == "tma_f16"


def test_planning_needs_a_sensible_device_and_a_buffer():
    A, B, D = BASE, 2 * BASE, 4 * BASE
    args = (1, 64, 64, 64, A, 64, 0, R, B, 64, 0, COL, None, 64, 0, D, 64, 0, 1.0, 0.0, None, 0, ttc.DTYPE["bf16"],
            None, 0)
    assert ttc.ttc_gemm_plan(*args, 1)[0] == 1
    assert ttc.ttc_gemm_plan(*args, 5000)[0] == 1
    assert ttc.load().ttc_gemm_plan(*args, 152, None, 16) == 1
    assert ttc.load().ttc_gemm_plan(*args, 152, None, 0) == 0
    # argument errors come back as from the real call
    bad = list(args)
    bad[5] = 10  # lda below K
    assert ttc.ttc_gemm_plan(*bad, 152)[0] == 1


def test_small_mn_major_b_problems_are_not_refused():
    """A column-major A and a row-major B with M and N below 33 once found no
    tile width (an MN-major B needs whole 64-column slabs)."""
    for (M, N, K) in [(7, 2, 200), (2, 2, 1025), (7, 7, 8), (1, 1, 64), (33, 5, 100)]:
        st, it, _ = plan(M, N, K, la="col", lb="row")
        assert st == 0 and len(it) == 1, (M, N, K, it)


@pytest.mark.parametrize("sm_count", [152, 148, 132, 16, 2])
def test_other_device_sizes_plan_every_benchmark_shape(sm_count):
    for shape in [(8192, 8192, 8192), (4096, 4096, 4096), (4099, 3001, 1023), (16, 8192, 8192), (1, 4096, 4096)]:
        st, it, _ = plan(*shape, beta=1.0, sm_count=sm_count)
        assert st == 0 and it, (shape, it)
        for x in it:
            if "clusters" in x:
                assert int(x["clusters"]) <= sm_count // 2
            if x["kernel"] == "single":
                assert int(x["grid"]) <= sm_count


# ------------------------------------------------------------------ random problems

def _aligned(addr, ld, stride, esize, batch, need=16, lines=2):
    """Every line of an operand (and every batch) starts aligned; with one
    line the pitch never enters an address."""
    return (addr % need == 0 and (lines <= 1 or (ld * esize) % need == 0) and
            (batch <= 1 or stride == 0 or (stride * esize) % need == 0))


def _lines(q, op):
    """Lines (rows as stored) of operand A or B.  A one-element-wide operand
    with a pitch of 1 is one contiguous line read the other way (M = 1 or
    K = 1 for A, K = 1 or N = 1 for B)."""
    if op == "A":
        if q["lda"] == 1 and ((q["M"] == 1 and q["la"] == "col") or (q["K"] == 1 and q["la"] == "row")):
            return 1
        return q["M"] if q["la"] == "row" else q["K"]
    if q["ldb"] == 1 and ((q["N"] == 1 and q["lb"] == "row") or (q["K"] == 1 and q["lb"] == "col")):
        return 1
    return q["K"] if q["lb"] == "row" else q["N"]


def _random_problem(rng):
    dtype = str(rng.choice(["bf16", "f16", "i8"]))
    M, N, K = (int(np.round(np.exp(rng.uniform(0, np.log(10000))))) for _ in range(3))
    if rng.integers(0, 4) == 0:
        M = int(rng.choice([1, 2, 16, 24]))
    la, lb = str(rng.choice(["row", "col"])), str(rng.choice(["row", "col"]))
    pads = [int(rng.choice([0, 0, 1, 3, 8, 16])) for _ in range(4)]
    offs = [int(rng.choice([0, 0, 0, 1, 4, 8])) for _ in range(4)]
    batch = int(rng.choice([1, 1, 1, 2, 5]))
    beta = float(rng.choice([0.0, 1.0]))
    workspace = rng.choice([None, "repack", "staged"]) if batch == 1 else None
    lda = (K if la == "row" else M) + pads[0]
    ldb = (N if lb == "row" else K) + pads[1]
    ldc, ldd = N + pads[2], N + pads[3]
    a_size = (M * lda if la == "row" else K * lda)
    b_size = (K * ldb if lb == "row" else N * ldb)
    gaps = [int(rng.choice([0, 0, 3, 16])) for _ in range(4)]
    strides = (a_size + gaps[0], 0 if rng.integers(0, 4) == 0 else b_size + gaps[1], M * ldc + gaps[2],
               M * ldd + gaps[3]) if batch > 1 else (0, 0, 0, 0)
    if rng.integers(0, 25) == 0:
        # a large int8 problem with the staged workspace (the CTA-pair int8 path when TMA can read it)
        dtype, M, N, workspace, batch, strides = "i8", int(rng.integers(2048, 9000)), int(rng.integers(2048, 9000)), \
            "staged", 1, (0, 0, 0, 0)
        up16 = lambda x: -(-x // 16) * 16
        lda, ldb = up16(K if la == "row" else M) + 16 * pads[0], up16(N if lb == "row" else K) + 16 * pads[1]
        ldc, ldd = N + pads[2], -(-N // 4) * 4 + 4 * pads[3]
        offs = [0, 0, offs[2], 0]
    return dict(M=M, N=N, K=K, dtype=dtype, la=la, lb=lb, lda=lda, ldb=ldb, ldc=ldc, ldd=ldd, beta=beta,
                workspace=workspace, offs=tuple(offs), batch=batch, strides=strides)


def test_random_problems_are_planned_and_keep_the_kernels_rules():
    rng = np.random.default_rng(20261207)
    counts = {}
    for _ in range(10000):
        q = _random_problem(rng)
        st, items, ad = plan(**q)
        assert st == 0, (q, st)
        assert items, q
        es, oes = (1, 4) if q["dtype"] == "i8" else (2, 2)
        names = kernels(items)
        repacked = "repack" in names or "widen_i8" in names
        staged = "stage_c" in names or "unstage_d" in names
        for it in items:
            counts[it["kernel"]] = counts.get(it["kernel"], 0) + 1
            if it["kernel"] == "pair":
                assert q["batch"] >= 1
                if not repacked:
                    # TMA reads A and B where they are
                    assert _aligned(ad["A"], ad["lda"], q["strides"][0], es, q["batch"], lines=_lines(q, "A")), (q, it)
                    assert _aligned(ad["B"], ad["ldb"], q["strides"][1], es, q["batch"], lines=_lines(q, "B")), (q, it)
            if it.get("d_tma") == "1" and not staged and it["kernel"] in ("pair", "pair_i8") + ("single",):
                if it.get("swap", "0") == "0":
                    ok_pitch = (ad["ldd"] * oes) % 16 == 0 or q["M"] == 1
                    assert ad["D"] % 16 == 0 and ok_pitch, (q, it)
                    assert q["batch"] == 1 or (q["strides"][3] * oes) % 16 == 0, (q, it)
            if it["kernel"] in ("pair", "pair_i8"):
                assert int(it["clusters"]) <= SMS // 2 and int(it["units"]) >= int(it["tiles"]), (q, it)
            if it.get("d_tma") == "1":
                # TMA stores whole 16-byte granules only: a row needs at least one
                assert q["N"] * oes >= 16, (q, it)
            if it["kernel"] == "single":
                assert int(it["grid"]) <= SMS and it["ksplit"] in ("1", "2", "4", "8"), (q, it)
                assert it["ksplit"] == "1" or int(it["bn"]) <= 128, (q, it)
                swap = it["swap"] == "1"
                assert not (swap and it.get("d_tma") == "1"), (q, it)
                if it["mode"].startswith("tma") and not repacked:
                    for op in ("A", "B"):
                        ld = ad["lda"] if op == "A" else ad["ldb"]
                        sidx = 0 if op == "A" else 1
                        assert _aligned(ad[op], ld, q["strides"][sidx], es, q["batch"], lines=_lines(q, op)), (q, it)
                if it["mode"].startswith("plain") and not repacked:
                    # the kernel's A is B after the swap
                    ka, kb = (("B", "A") if swap else ("A", "B"))
                    for flag, op in (("a_vec", ka), ("b_vec", kb)):
                        if it[flag] == "1":
                            ld = ad["lda"] if op == "A" else ad["ldb"]
                            sidx = 0 if op == "A" else 1
                            assert _aligned(ad[op], ld, q["strides"][sidx], es, q["batch"], need=8 * es,
                                            lines=_lines(q, op)), (q, it)
        if q["workspace"] is None:
            assert not repacked and not staged, (q, items)
        if staged:
            assert q["dtype"] == "i8" and q["workspace"] == "staged", (q, items)  # only int32 D is staged
        if names[0].startswith("gemv"):
            assert q["dtype"] != "i8" and q["batch"] == 1 and (q["M"] == 1 or q["N"] == 1), (q, items)
            assert len(items) == 1, (q, items)  # no workspace copies for matrix-vector problems
        if "pair" in names or "pair_i8" in names:
            assert q["M"] >= 256 and q["N"] >= 256, (q, items)
    # the sweep reaches every kind of launch
    for k in ("pair", "single", "repack", "gemv_rows", "gemv_cols", "stage_c", "unstage_d", "widen_i8", "pair_i8"):
        assert counts.get(k, 0) > 0, (k, counts)


# ------------------------------------------------------------------ knobs and workspaces

@pytest.fixture
def knob():
    set_ = []

    def f(name, value):
        ttc.ttc_set_knob(name, value)
        set_.append(name)
    yield f
    for name in set_:
        ttc.ttc_set_knob(name, 0)


def test_knobs_steer_the_plan(knob):
    knob("pair", 2)
    assert kernels(plan(8192, 8192, 8192)[1]) == ["single"]
    knob("pair", 1)
    assert kernels(plan(300, 300, 64)[1]) == ["pair"]
    knob("pair", 0)
    knob("pair_tile_n", 128)
    assert plan(8192, 8192, 8192)[1][0]["bn"] == "128"
    knob("pair_tile_n", 0)
    knob("swap_ab", 1)
    it = plan(300, 500, 64)[1]
    assert it[0]["kernel"] == "single" and it[0]["swap"] == "1"
    knob("swap_ab", 0)
    knob("split_k", 4)
    it = plan(256, 256, 4096)[1]
    assert it[0]["ksplit"] == "4" and it[0]["grid"] == str(4 * int(it[0]["tiles"]))
    knob("split_k", 0)
    knob("gemv", 1)
    assert kernels(plan(1, 4096, 4096)[1]) == ["single"]
    knob("gemv", 0)
    knob("force_generic_load", 1)
    assert plan(1024, 1024, 1024)[1][0]["mode"] == "plain_bf16"
    knob("force_generic_load", 0)
    knob("force_generic_store", 1)
    it = plan(1024, 1024, 1024)[1]
    assert all(x.get("d_tma", "0") == "0" for x in it)
    knob("force_generic_store", 0)
    knob("pair_epi_warps", 8)
    it = plan(4099, 3001, 1023, beta=1.0, workspace="staged")[1]
    assert it[-1]["kernel"] == "pair" and it[-1]["ew"] == "8"


def test_workspaces_decide_the_copies():
    # odd pitches: nothing copied without a workspace, both operands with one
    q = dict(M=2000, N=1500, K=300, lda=301, ldb=303, beta=1.0, ldc=1501, ldd=1503)
    it = plan(**q)[1]
    assert kernels(it) == ["single"] and it[0]["mode"] == "plain_bf16"  # the plain-load producer
    it = plan(**q, workspace="repack")[1]
    assert kernels(it) == ["repack", "pair"] and it[1]["d_tma"] == "0"  # TMA on the copies; D rows written directly
    # int8 with an unaligned D: staged through an aligned copy (C copied in, D copied out)
    q8 = dict(M=300, N=200, K=72, dtype="i8", lda=73, ldb=75, beta=1.0, ldd=203)
    assert kernels(plan(**q8, workspace="staged")[1]) == ["repack", "stage_c", "single", "unstage_d"]
    assert kernels(plan(**q8, workspace="repack")[1]) == ["repack", "single"]
    # a 16-bit D is never staged: its rows are written at any alignment
    assert "unstage_d" not in kernels(plan(**q, workspace="staged")[1])
    # matrix-vector problems need no workspace at all
    assert kernels(plan(1, 4096, 4096, ldb=4097, workspace="staged")[1]) == ["gemv_rows"]


def test_sizes_near_two_to_the_31_are_refused_before_any_loop_could_wrap():
    """The kernels count rows, columns and k in 32-bit integers and step past
    the end by up to a grid's stride before testing a loop bound, so sizes
    within 2^24 of 2^31 are refused; just below the limit a matrix-vector
    problem (the kernel whose loops stride furthest) is planned."""
    lim = (1 << 31) - (1 << 24)
    for kw in (dict(M=1, N=lim + 1, K=16), dict(M=1, N=4096, K=lim + 1, lb="col"), dict(M=lim + 1, N=1, K=16),
               dict(M=64, N=64, K=64, lda=lim + 1)):
        assert plan(**kw)[0] == 2, kw
    st, it, _ = plan(M=1, N=lim, K=16, lb="row")
    assert st == 0 and kernels(it) == ["gemv_cols"]
    st, it, _ = plan(M=1, N=4096, K=lim, lb="col")
    assert st == 0 and kernels(it) == ["gemv_rows"]


def test_reported_workspace_sizes_are_enough_and_needed():
    """For random problems whose operands TMA cannot read: with exactly the
    size ttc_gemm_workspace_size reports the plan repacks them, with one byte
    less it does not (the plain-load producer reads them in place); the
    staged size adds D's aligned copy for int32 outputs alike."""
    rng = np.random.default_rng(20261208)
    checked = staged_checked = 0
    lay = {"row": R, "col": COL}
    for _ in range(400):
        dtype = str(rng.choice(["bf16", "i8"]))
        M, N, K = (int(rng.integers(2, 3000)) for _ in range(3))
        la, lb = str(rng.choice(["row", "col"])), str(rng.choice(["row", "col"]))
        lda = (K if la == "row" else M) + int(rng.choice([1, 3]))
        ldb = (N if lb == "row" else K) + int(rng.choice([0, 1]))
        ldd = N + int(rng.choice([0, 1, 3]))
        es, oes = (1, 4) if dtype == "i8" else (2, 2)
        A, B, D = BASE, 2 * BASE, 4 * BASE
        dt = ttc.DTYPE[dtype]
        need = ttc.ttc_gemm_workspace_size(M, N, K, A, lda, lay[la], B, ldb, lay[lb], dt)
        need_st = ttc.ttc_gemm_workspace_size_staged(M, N, K, A, lda, lay[la], B, ldb, lay[lb], D, ldd, dt)
        assert need_st >= need

        def names(ws):
            st, text = ttc.ttc_gemm_plan(1, M, N, K, A, lda, 0, lay[la], B, ldb, 0, lay[lb], None, N, 0, D, ldd, 0,
                                         1.0, 0.0, None, 0, dt, 5 * BASE if ws else None, ws, SMS)
            assert st == 0
            return [it.split()[0] for it in text.split("; ") if it]
        if need == 0:
            continue  # a matrix-vector problem, or nothing to repack
        checked += 1
        with_ws = names(need)
        if "widen_i8" not in with_ws:
            assert with_ws[0] == "repack", (dtype, M, N, K, la, lb, lda, ldb, with_ws)
        assert "repack" not in names(need - 1)
        if need_st > need and "widen_i8" not in names(need_st):
            staged_checked += 1
            assert "unstage_d" in names(need_st) and "unstage_d" not in names(need_st - 1)
    assert checked > 300 and staged_checked > 50, (checked, staged_checked)
