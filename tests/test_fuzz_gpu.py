"""Seeded random problems through every planner branch, checked in full
against the oracle.  GEMM: sizes around the tile, k-block and chunk boundaries
(1 to 513 rows and columns, K from 1 to 1025), all four A/B majorness
combinations, tight and padded pitches, fp16/bf16 with every epilogue
(alpha, beta with C, bias, ReLU, tanh-GELU) and int8 with and without C,
through ttc_gemm and ttc_gemm_ws (with the workspace for the operand repack
only, or for its fastest path), with the int8 CTA-pair path forced on some
int8 calls.  The planner picks the kernel (CTA pair or single CTA, tile
width, orientation, split K, matrix-vector kernels) from each shape.  Then
random strided batches (gaps between batches, a shared B), random
convolutions (filter sizes, padding, strides, dilations, channel counts on
and off the 64-channel blocks, an unaligned input, a padded output pitch),
larger random convolutions on the CTA-pair paths (halo tiles for unit
strides, im2col loads otherwise), random transposes (every element size,
tight, odd and 16-byte pitches), and
GEMMs whose A, B, C and D start at element offsets off every alignment,
through each entry point including the static-scratch one (nothing outside
D's elements written).  The pitch padding of A, B and C, and the elements
just before and after them, hold NaN (int8: 127), which no kernel may read."""
import numpy as np
import pytest

import oracle
import synth
import tiled_tensor_core_02_gb300 as ttc
from gpu_util import run
from test_gemm_gpu import _poison_padding

pytestmark = pytest.mark.gpu

SIZES_MN = [1, 2, 7, 16, 33, 64, 100, 128, 129, 255, 256, 257, 300, 513]
SIZES_K = [1, 8, 16, 63, 64, 65, 100, 127, 128, 200, 300, 1024, 1025]
ACTS = ["none", "relu", "gelu_tanh"]


def _cases(n=240, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = rng.choice(["bf16", "bf16", "f16", "i8"])
        M, N, K = (int(rng.choice(SIZES_MN)), int(rng.choice(SIZES_MN)), int(rng.choice(SIZES_K)))
        la, lb = rng.choice(["row", "col"]), rng.choice(["row", "col"])
        pad = [int(rng.choice([0, 0, 1, 3, 8, 9])) for _ in range(3)]
        entry = rng.choice(["plain", "ws_repack", "ws_staged"])
        if dtype == "i8":
            alpha, beta, act, bias = 1.0, float(rng.choice([0.0, 1.0])), "none", False
        else:
            alpha = float(rng.choice([1.0, 0.5, -2.0]))
            beta = float(rng.choice([0.0, 1.0, 0.25]))
            act = str(rng.choice(ACTS))
            bias = bool(rng.integers(0, 2))
        wide = dtype == "i8" and entry == "ws_staged" and bool(rng.integers(0, 2))
        out.append((i, str(dtype), M, N, K, str(la), str(lb), pad, str(entry), alpha, beta, act, bias, wide))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}x{c[3]}x{c[4]}-{c[5]}{c[6]}-{c[8]}")
def test_random_problem_matches_oracle(case):
    i, dtype, M, N, K, la, lb, pad, entry, alpha, beta, act, bias, wide = case
    lda = (K if la == "row" else M) + pad[0]
    ldb = (N if lb == "row" else K) + pad[1]
    ldc = N + pad[2]
    dist = "int8" if dtype == "i8" else "uniform"
    p = synth.Problem(M, N, K, dtype=dtype, layoutA=la, layoutB=lb, seed=1000 + i, distA=dist, distB=dist,
                      distC=("int8" if dtype == "i8" else "uniform") if beta != 0.0 else None,
                      dist_bias="normal:0.5" if bias else None, lda=lda, ldb=ldb, ldc=ldc)
    _poison_padding(p)
    ws = {"plain": None, "ws_repack": -1, "ws_staged": -2}[entry]
    ttc.ttc_set_knob("i8_wide", 1 if wide else 0)
    try:
        d = run(p, alpha, beta, act, use_bias=bias, workspace=ws)
    finally:
        ttc.ttc_set_knob("i8_wide", 0)
    r, sabs = oracle.gemm_full(p, alpha=alpha, beta=beta, act=act, use_bias=bias)
    if dtype == "i8":
        assert np.array_equal(d.astype(np.int64), r.astype(np.int64))
        return
    ok, worst, w = oracle.check_float(oracle.decode(d.ravel(), dtype), r.ravel(), sabs.ravel(), dtype)
    assert ok, f"worst error ratio {worst:.3f} at {divmod(w, p.N)}"


# ---------------------------------------------------------------- strided batched
def _batched_cases(n=80, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = str(rng.choice(["bf16", "f16", "i8"]))
        nb = int(rng.choice([1, 2, 3, 5]))
        M, N, K = (int(rng.choice(SIZES_MN)), int(rng.choice(SIZES_MN)), int(rng.choice(SIZES_K)))
        la, lb = str(rng.choice(["row", "col"])), str(rng.choice(["row", "col"]))
        pads = [int(rng.choice([0, 0, 1, 8])) for _ in range(3)]
        # extra elements between consecutive batches (odd ones break 16-byte alignment)
        gaps = [int(rng.choice([0, 0, 3, 64])) for _ in range(4)]
        share_b = bool(rng.integers(0, 4) == 0)
        if dtype == "i8":
            alpha, beta, act, bias = 1.0, float(rng.choice([0.0, 1.0])), "none", False
        else:
            alpha, beta = float(rng.choice([1.0, -0.5])), float(rng.choice([0.0, 1.0]))
            act, bias = str(rng.choice(ACTS)), bool(rng.integers(0, 2))
        out.append((i, dtype, nb, M, N, K, la, lb, pads, gaps, share_b, alpha, beta, act, bias))
    return out


@pytest.mark.parametrize("case", _batched_cases(),
                         ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}x{c[3]}x{c[4]}x{c[5]}-{c[6]}{c[7]}")
def test_random_batched_problem_matches_oracle(case):
    from gpu_util import run_batched
    i, dtype, nb, M, N, K, la, lb, pads, gaps, share_b, alpha, beta, act, bias = case
    lda = (K if la == "row" else M) + pads[0]
    ldb = (N if lb == "row" else K) + pads[1]
    ldc = N + pads[2]
    dist = "int8" if dtype == "i8" else "uniform"
    probs = [synth.Problem(M, N, K, dtype=dtype, layoutA=la, layoutB=lb, seed=5000 + 8 * i + b, distA=dist,
                           distB=dist, distC=dist if beta != 0.0 else None,
                           dist_bias="normal:0.5" if bias else None, lda=lda, ldb=ldb, ldc=ldc)
             for b in range(nb)]
    for q in probs[1:]:
        q.bias = probs[0].bias  # one bias for every batch
        if share_b:
            q.B = probs[0].B
    p0 = probs[0]
    strides = {"A": p0.A.size + gaps[0], "B": 0 if share_b else p0.B.size + gaps[1],
               "C": (p0.C.size + gaps[2]) if p0.C is not None else 0, "D": M * N + gaps[3]}
    outs = run_batched(probs, strides, alpha, beta, act, share_b=share_b)
    for q, d in zip(probs, outs):
        r, sabs = oracle.gemm_full(q, alpha=alpha, beta=beta, act=act, use_bias=bias)
        if dtype == "i8":
            assert np.array_equal(d.astype(np.int64), r.astype(np.int64))
            continue
        ok, worst, w = oracle.check_float(oracle.decode(np.ascontiguousarray(d).ravel(), dtype), r.ravel(),
                                          sabs.ravel(), dtype)
        assert ok, f"worst error ratio {worst:.3f} at {divmod(w, N)}"


# ---------------------------------------------------------------- convolution
def _conv_cases(n=80, seed=20261204):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        N = int(rng.choice([1, 2]))
        H, W = int(rng.integers(1, 17)), int(rng.integers(1, 17))
        C = int(rng.choice([1, 3, 8, 16, 24, 64, 72, 128]))
        K = int(rng.choice([1, 8, 24, 32, 40, 64, 96, 136, 256]))
        R, S = int(rng.choice([1, 2, 3, 5])), int(rng.choice([1, 2, 3, 5]))
        pad = (int(rng.integers(0, 3)), int(rng.integers(0, 3)))
        stride = (int(rng.choice([1, 1, 2, 3])), int(rng.choice([1, 1, 2, 3])))
        dil = (int(rng.choice([1, 1, 2])), int(rng.choice([1, 1, 2])))
        if H + 2 * pad[0] - dil[0] * (R - 1) - 1 < 0 or W + 2 * pad[1] - dil[1] * (S - 1) - 1 < 0:
            continue  # the filter does not fit the padded input (an argument error, tested elsewhere)
        dtype = str(rng.choice(["bf16", "f16"]))
        alpha, beta = float(rng.choice([1.0, 0.75])), float(rng.choice([0.0, 0.0, 1.0]))
        act, bias = str(rng.choice(ACTS)), bool(rng.integers(0, 2))
        ldd_pad = int(rng.choice([0, 0, 1, 8]))
        x_off = int(rng.choice([0, 0, 0, 1]))
        out.append((len(out), N, H, W, C, K, R, S, pad, stride, dil, dtype, alpha, beta, act, bias, ldd_pad, x_off))
    return out


@pytest.mark.parametrize("case", _conv_cases(),
                         ids=lambda c: f"{c[0]}-{c[11]}-n{c[1]}h{c[2]}w{c[3]}c{c[4]}k{c[5]}r{c[6]}s{c[7]}")
def test_random_convolution_matches_oracle(case):
    from test_conv_gpu import run_conv
    i, N, H, W, C, K, R, S, pad, stride, dil, dtype, alpha, beta, act, bias, ldd_pad, x_off = case
    cp = synth.ConvProblem(N, H, W, C, K, R, S, pad, stride, dil, dtype=dtype, seed=7000 + i,
                           with_c=beta != 0.0, dist_bias="uniform" if bias else None)
    ldd = K + ldd_pad
    out = run_conv(cp, alpha=alpha, beta=beta, act=act, use_bias=bias, ldd=ldd, x_offset=x_off)
    r, sabs = oracle.conv_full(cp, alpha=alpha, beta=beta, act=act, use_bias=bias)
    d = oracle.decode(out.reshape(-1)[:cp.M * ldd].reshape(cp.M, ldd)[:, :K], dtype)
    ok, worst, w = oracle.check_float(d.ravel(), r.ravel(), sabs.ravel(), dtype)
    assert ok, f"worst error ratio {worst:.3f} at {divmod(w, K)}"
    if ldd_pad:
        assert (out.reshape(-1)[:cp.M * ldd].reshape(cp.M, ldd)[:, K:] == 0xFFFF).all()


# ---------------------------------------------------------------- transpose
def _transpose_cases(n=60, seed=20261205):
    rng = np.random.default_rng(seed)
    sizes = [1, 2, 7, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 300, 513]
    return [(i, int(rng.choice(sizes)), int(rng.choice(sizes)), int(rng.choice([1, 2, 4, 8])),
             str(rng.choice(["tight", "odd", "aligned"])), str(rng.choice(["tight", "odd", "aligned"])))
            for i in range(n)]


@pytest.mark.parametrize("case", _transpose_cases(), ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}-e{c[3]}-{c[4]}-{c[5]}")
def test_random_transpose_matches_oracle(case):
    from test_transpose_gpu import pitch, run
    i, rows, cols, eb, ms, md = case
    lds = cols if ms == "tight" else pitch(cols, eb, ms)
    ldd = rows if md == "tight" else pitch(rows, eb, md)
    src = synth.transpose_input(rows, cols, eb, seed=9000 + i, lds=lds)
    got = run(src, rows, cols, lds, ldd, eb).reshape(cols, ldd)
    want = oracle.transpose(src, rows, cols, lds, ldd).reshape(cols, ldd)
    assert np.array_equal(got[:, :rows], want[:, :rows])
    assert (got[:, rows:] == np.iinfo(synth.ELEM_DTYPE[eb]).max).all()  # the pitch padding is not written


# ---------------------------------------------------------------- base pointers at any element offset
def _offset_cases(n=200, seed=20261206):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = str(rng.choice(["bf16", "bf16", "f16", "i8"]))
        M, N, K = (int(rng.choice(SIZES_MN)), int(rng.choice(SIZES_MN)), int(rng.choice(SIZES_K)))
        la, lb = str(rng.choice(["row", "col"])), str(rng.choice(["row", "col"]))
        pad = [int(rng.choice([0, 0, 1, 8])) for _ in range(4)]
        offs = [int(rng.choice([0, 0, 1, 3, 8])) for _ in range(4)]  # elements before A, B, C, D
        if rng.integers(0, 3) == 0:
            # D's pitch rounded up to 16 bytes (TMA can store its rows) and its
            # start kept aligned: the rows end inside a 16-byte granule
            per16 = 4 if dtype == "i8" else 8
            pad[3] = -N % per16
            offs[3] = 0
        entry = str(rng.choice(["plain", "ws_repack", "ws_staged", "static"]))
        if dtype == "i8":
            alpha, beta, act, bias = 1.0, float(rng.choice([0.0, 1.0])), "none", False
        else:
            alpha, beta = float(rng.choice([1.0, 0.5])), float(rng.choice([0.0, 1.0, 0.25]))
            act, bias = str(rng.choice(ACTS)), bool(rng.integers(0, 2))
        out.append((i, dtype, M, N, K, la, lb, pad, offs, entry, alpha, beta, act, bias))
    return out


def _at_offset(host, off, fill=0):
    """A device copy of `host` that starts `off` elements into its allocation
    (with `fill` before it and in 8 elements after it), and its address."""
    from gpu_util import to_dev
    edge = np.full(off, fill, host.dtype), np.full(8, fill, host.dtype)
    buf = to_dev(np.concatenate([edge[0], host, edge[1]]))
    return buf, buf.data_ptr() + off * host.dtype.itemsize


@pytest.mark.parametrize("case", _offset_cases(),
                         ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}x{c[3]}x{c[4]}-{c[5]}{c[6]}-{c[9]}")
def test_random_offsets_match_oracle(case):
    import torch
    from gpu_util import LAY
    i, dtype, M, N, K, la, lb, pad, offs, entry, alpha, beta, act, bias = case
    lda = (K if la == "row" else M) + pad[0]
    ldb = (N if lb == "row" else K) + pad[1]
    ldc, ldd = N + pad[2], N + pad[3]
    dist = "int8" if dtype == "i8" else "uniform"
    p = synth.Problem(M, N, K, dtype=dtype, layoutA=la, layoutB=lb, seed=11000 + i, distA=dist, distB=dist,
                      distC=dist if beta != 0.0 else None, dist_bias="normal:0.5" if bias else None,
                      lda=lda, ldb=ldb, ldc=ldc)
    _poison_padding(p)
    nan = {"i8": 127, "bf16": 0x7FC0, "f16": 0x7E00}[dtype]
    A, a_ptr = _at_offset(p.A, offs[0], nan)
    B, b_ptr = _at_offset(p.B, offs[1], nan)
    c_ptr = None
    if p.C is not None:
        C, c_ptr = _at_offset(p.C, offs[2], 1 << 30 if dtype == "i8" else nan)
    out_t = torch.int32 if dtype == "i8" else torch.int16
    out_size = 4 if dtype == "i8" else 2
    D = torch.full((offs[3] + M * ldd + 8,), -1, dtype=out_t, device="cuda")
    d_ptr = D.data_ptr() + offs[3] * out_size
    bias_dev = torch.from_numpy(p.bias).cuda() if bias else None
    s = torch.cuda.current_stream().cuda_stream
    args = (M, N, K, a_ptr, lda, LAY[la], b_ptr, ldb, LAY[lb], c_ptr if beta != 0.0 else None, ldc, d_ptr, ldd,
            alpha, beta, bias_dev.data_ptr() if bias else None, ttc.ACT[act], ttc.DTYPE[dtype])
    if entry == "plain":
        st = ttc.ttc_gemm(*args, s)
    elif entry == "static":
        st = ttc.ttc_gemm_static_scratch(*args, s)
    else:
        if entry == "ws_staged":
            need = ttc.ttc_gemm_workspace_size_staged(M, N, K, a_ptr, lda, LAY[la], b_ptr, ldb, LAY[lb], d_ptr,
                                                      ldd, ttc.DTYPE[dtype])
        else:
            need = ttc.ttc_gemm_workspace_size(M, N, K, a_ptr, lda, LAY[la], b_ptr, ldb, LAY[lb], ttc.DTYPE[dtype])
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        st = ttc.ttc_gemm_ws(*args, ws.data_ptr() if need else None, need, s)
    if entry == "static" and st == 5:
        return  # more scratch than the static array holds: refused before any work
    assert st == 0, ttc.STATUS.get(st, st)
    assert ttc.ttc_get_device_error(s) == 0
    full = D.cpu().numpy()
    if dtype != "i8":
        full = full.view(np.uint16)
    none = np.int32(-1) if dtype == "i8" else np.uint16(0xFFFF)
    assert np.all(full[:offs[3]] == none) and np.all(full[offs[3] + M * ldd:] == none)
    rows = full[offs[3]:offs[3] + M * ldd].reshape(M, ldd)
    assert np.all(rows[:, N:] == none)  # the pitch padding is not written
    d = rows[:, :N]
    r, sabs = oracle.gemm_full(p, alpha=alpha, beta=beta, act=act, use_bias=bias)
    if dtype == "i8":
        assert np.array_equal(d.astype(np.int64), r.astype(np.int64))
        return
    ok, worst, w = oracle.check_float(oracle.decode(np.ascontiguousarray(d).ravel(), dtype), r.ravel(),
                                      sabs.ravel(), dtype)
    assert ok, f"worst error ratio {worst:.3f} at {divmod(w, N)}"


# ---------------------------------------------------------------- larger convolutions (the CTA-pair paths)
def _large_conv_cases(n=30, seed=77):
    """Whole 64-channel blocks and at least 128 filters on outputs of a few
    hundred pixels: unit strides take the halo kernel, other strides the
    im2col loads on the CTA-pair kernel."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        N = int(rng.integers(1, 5))
        H, W = int(rng.integers(8, 41)), int(rng.integers(8, 41))
        C = int(rng.choice([64, 128, 192]))
        K = int(rng.choice([128, 160, 256, 320]))
        R, S = int(rng.choice([1, 3, 5])), int(rng.choice([1, 3, 5]))
        pad = (int(rng.integers(0, 3)), int(rng.integers(0, 3)))
        stride = (int(rng.choice([1, 1, 2, 3])), int(rng.choice([1, 1, 2, 3])))
        dil = (int(rng.choice([1, 1, 2])), int(rng.choice([1, 1, 2])))
        if H + 2 * pad[0] - dil[0] * (R - 1) - 1 < 0 or W + 2 * pad[1] - dil[1] * (S - 1) - 1 < 0:
            continue
        dtype = str(rng.choice(["bf16", "f16"]))
        beta = float(rng.choice([0.0, 1.0]))
        act = str(rng.choice(["none", "relu", "gelu_tanh"]))
        out.append((len(out), N, H, W, C, K, R, S, pad, stride, dil, dtype, beta, act))
    return out


@pytest.mark.parametrize("case", _large_conv_cases(),
                         ids=lambda c: f"{c[0]}-{c[11]}-n{c[1]}h{c[2]}w{c[3]}c{c[4]}k{c[5]}r{c[6]}s{c[7]}")
def test_random_larger_convolution_matches_oracle(case):
    from test_conv_gpu import run_conv
    i, N, H, W, C, K, R, S, pad, stride, dil, dtype, beta, act = case
    cp = synth.ConvProblem(N, H, W, C, K, R, S, pad, stride, dil, dtype=dtype, seed=500 + i, with_c=beta != 0.0,
                           dist_bias="uniform")
    out = run_conv(cp, alpha=1.0, beta=beta, act=act)
    r, sabs = oracle.conv_full(cp, alpha=1.0, beta=beta, act=act)
    d = oracle.decode(out.reshape(-1)[:cp.M * K].reshape(cp.M, K), dtype)
    ok, worst, w = oracle.check_float(d.ravel(), r.ravel(), sabs.ravel(), dtype)
    assert ok, f"worst error ratio {worst:.3f} at {divmod(w, K)}"
