"""Pins for the CPU GEMM oracle: brute force, closed forms, library routines.

None of these re-derive the oracle's own formula; each compares it with
something independent (an integer loop in another order, a closed form, a
library conversion, erf-based GELU), so a dropped term, a wrong sign or index
or a transposed operand fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import synth

DT = ["f16", "bf16", "i8"]
COMBOS = synth.MAJORNESS


def small_int_problem(M, N, K, dtype, la, lb, rng, with_c=True, pad=0):
    """Integer-valued operands in [-4, 4]: exact in fp16, bf16 and int8."""
    a = rng.integers(-4, 5, size=(M, K))
    b = rng.integers(-4, 5, size=(K, N))
    c = rng.integers(-4, 5, size=(M, N))
    store = (lambda v: v.astype(np.int8)) if dtype == "i8" else (lambda v: synth.store(v.astype(np.float64), dtype))
    cst = c.astype(np.int32) if dtype == "i8" else synth.store(c.astype(np.float64), dtype)
    lda = (K if la == "row" else M) + pad
    ldb = (N if lb == "row" else K) + pad
    p = synth.Problem.from_logical(store(a), store(b), cst if with_c else None, dtype=dtype,
                                   layoutA=la, layoutB=lb, lda=lda, ldb=ldb, ldc=N + pad)
    return p, a, b, c


def int_loop(a, b):
    """Independent integer GEMM, k-outermost accumulation into the whole matrix."""
    M, K = a.shape
    N = b.shape[1]
    out = [[0] * N for _ in range(M)]
    for k in range(K):
        for i in range(M):
            aik = int(a[i, k])
            for j in range(N):
                out[i][j] += aik * int(b[k, j])
    return np.array(out, dtype=np.int64).reshape(M, N)


@pytest.mark.parametrize("dtype", DT)
def test_bruteforce_tiny_all_shapes_and_layouts(dtype):
    rng = np.random.default_rng(7)
    for M, N, K in itertools.product(range(1, 6), repeat=3):
        for la, lb in COMBOS:
            pad = (M + N + K) % 3
            p, a, b, c = small_int_problem(M, N, K, dtype, la, lb, rng, pad=pad)
            if dtype == "i8":
                alpha, beta = 1.0, 1.0
            else:
                alpha, beta = 2.0, -1.0
            r, sabs = oracle.gemm_full(p, alpha=alpha, beta=beta)
            ref = int_loop(a, b)
            want = alpha * ref + beta * c
            assert np.array_equal(r, want.astype(np.float64)), (M, N, K, la, lb)
            # S_abs is the sum of |products|
            sref = int_loop(np.abs(a), np.abs(b))
            assert np.array_equal(sabs, sref.astype(np.float64))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_closed_form_all_ones(dtype):
    M, N, K = 37, 29, 300
    one = synth.store(np.ones(1), dtype)[0]
    st = synth.Stream(11)
    c = synth.store(st.uniform(M * N), dtype).reshape(M, N)
    for la, lb in COMBOS:
        p = synth.Problem.from_logical(np.full((M, K), one, dtype=np.uint16),
                                       np.full((K, N), one, dtype=np.uint16), c, dtype=dtype,
                                       layoutA=la, layoutB=lb)
        r, sabs = oracle.gemm_full(p, alpha=1.5, beta=0.5)
        cval = oracle.decode(c, dtype)
        assert np.array_equal(r, 1.5 * K + 0.5 * cval)
        assert np.all(sabs == K)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_closed_form_identity_b(dtype):
    M, K = 41, 64
    st = synth.Stream(12)
    a = synth.store(st.uniform(M * K), dtype).reshape(M, K)
    c = synth.store(st.uniform(M * K), dtype).reshape(M, K)
    eye = synth.store(np.eye(K), dtype)
    for la, lb in COMBOS:
        p = synth.Problem.from_logical(a, eye, c, dtype=dtype, layoutA=la, layoutB=lb)
        r, _ = oracle.gemm_full(p, alpha=-2.0, beta=0.25)
        want = -2.0 * oracle.decode(a, dtype) + 0.25 * oracle.decode(c, dtype)
        assert np.array_equal(r, want)


def test_closed_form_int8_all_ones_and_extremes():
    M, N, K = 5, 6, 8192
    for v in (1, -128, 127):
        p = synth.Problem.from_logical(np.full((M, K), v, np.int8), np.full((K, N), -128, np.int8),
                                       dtype="i8")
        r, _ = oracle.gemm_full(p)
        assert np.all(r == float(v * -128 * K))


@pytest.mark.parametrize("la,lb", COMBOS)
def test_transpose_identity_via_layout_swap(la, lb):
    """(A B)^T = B^T A^T: B's buffer read with the other layout flag is B^T."""
    M, N, K = 23, 31, 57
    p = synth.Problem(M, N, K, dtype="bf16", layoutA=la, layoutB=lb, seed=5)
    r, _ = oracle.gemm_full(p)
    flip = {"row": "col", "col": "row"}
    q = synth.Problem.from_logical(np.zeros((N, K), np.uint16), np.zeros((K, M), np.uint16),
                                   dtype="bf16", layoutA=flip[lb], layoutB=flip[la])
    q.A, q.lda = p.B, p.ldb
    q.B, q.ldb = p.A, p.lda
    rt, _ = oracle.gemm_full(q)
    assert np.array_equal(rt, r.T)


def test_epilogue_terms_with_k_zero():
    """K = 0: the product vanishes and D = act(beta C + bias) (cuBLAS semantics)."""
    M, N = 4, 7
    st = synth.Stream(3)
    c = synth.store(st.uniform(M * N), "bf16").reshape(M, N)
    bias = np.linspace(-1, 1, N).astype(np.float32)
    p = synth.Problem.from_logical(np.zeros((M, 0), np.uint16), np.zeros((0, N), np.uint16), c,
                                   bias=bias, dtype="bf16")
    r, sabs = oracle.gemm_full(p, alpha=3.0, beta=-0.5, act="relu")
    want = np.maximum(-0.5 * oracle.decode(c, "bf16") + bias.astype(np.float64), 0.0)
    assert np.array_equal(r, want) and np.all(sabs == 0)


@pytest.mark.parametrize("act", ["none", "relu", "gelu_tanh"])
def test_epilogue_order_all_terms(act):
    """All epilogue terms at once, K > 0, all-ones A and B: D = act(alpha K +
    beta C + bias), the order of the epilogue box in the CUTLASS tutorial's
    section 1 (alpha/beta, then bias, then the activation).  A bias scaled by
    alpha, an activation applied before the bias, or beta applied to the bias
    each give a different value here."""
    M, N, K = 6, 9, 40
    one = synth.store(np.ones(1), "bf16")[0]
    st = synth.Stream(5)
    c = synth.store(st.uniform(M * N), "bf16").reshape(M, N)
    bias = np.linspace(-50.0, 30.0, N).astype(np.float32)
    p = synth.Problem.from_logical(np.full((M, K), one, np.uint16), np.full((K, N), one, np.uint16), c,
                                   bias=bias, dtype="bf16")
    r, sabs = oracle.gemm_full(p, alpha=0.75, beta=-2.0, act=act)
    pre = 0.75 * K - 2.0 * oracle.decode(c, "bf16") + bias.astype(np.float64)
    tol = 1e-12
    if act == "relu":
        want = np.maximum(pre, 0.0)
    elif act == "gelu_tanh":
        # x Phi(x) (the erf form), which the tanh form stays within 5e-4 of
        want = np.array([0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0))) for x in pre.ravel()]).reshape(pre.shape)
        tol = 5e-4
    else:
        want = pre
    assert np.allclose(r, want, rtol=0.0, atol=tol) and np.all(sabs == K)
    # the alternatives differ from it (so the test can tell them apart)
    assert not np.allclose(want, 0.75 * (K + bias.astype(np.float64)) - 2.0 * oracle.decode(c, "bf16"))
    if act == "relu":
        assert not np.allclose(want, np.maximum(pre - bias, 0.0) + bias)


def test_beta_zero_does_not_read_c():
    M, N, K = 3, 3, 2
    one = synth.store(np.ones(1), "bf16")[0]
    c = np.full((M, N), 0x7FC0, dtype=np.uint16)  # NaN everywhere
    p = synth.Problem.from_logical(np.full((M, K), one, np.uint16), np.full((K, N), one, np.uint16),
                                   c, dtype="bf16")
    r, _ = oracle.gemm_full(p, alpha=1.0, beta=0.0)
    assert np.all(r == 2.0)
    r2, _ = oracle.gemm_full(p, alpha=1.0, beta=1.0)
    assert np.all(np.isnan(r2))


def test_bias_is_per_column():
    M, N, K = 3, 5, 1
    one = synth.store(np.ones(1), "bf16")[0]
    bias = np.arange(N, dtype=np.float32) * 0.5
    p = synth.Problem.from_logical(np.full((M, K), one, np.uint16), np.full((K, N), one, np.uint16),
                                   bias=bias, dtype="bf16")
    r, _ = oracle.gemm_full(p)
    assert np.array_equal(r, np.tile(1.0 + bias.astype(np.float64), (M, 1)))


def test_activations_against_independent_forms():
    assert oracle.act("relu", -1.0) == 0.0 and oracle.act("relu", 2.5) == 2.5
    assert oracle.act("gelu_tanh", 0.0) == 0.0
    xs = np.linspace(-12, 12, 4801)
    for x in xs:
        g = oracle.act("gelu_tanh", x)
        exact = 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))  # x * Phi(x)
        # the tanh form is within 5e-4 of x * Phi(x) everywhere
        assert abs(g - exact) <= 5e-4, x
        # gelu(x) - gelu(-x) = x because tanh is odd
        assert abs(g - oracle.act("gelu_tanh", -x) - x) <= 1e-12 * max(1.0, abs(x))
    assert abs(oracle.act("gelu_tanh", 20.0) - 20.0) < 1e-12
    assert abs(oracle.act("gelu_tanh", -20.0)) < 1e-12


def test_gelu_tanh_matches_float64_library_evaluation():
    """The tanh-form GELU (constants sqrt(2/pi) and 0.044715) against torch's
    own float64 evaluation of the same form, gelu(x, approximate='tanh').  Both
    evaluate 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) in double; only the
    rounding order differs, so they agree to ~1e-15.  A slip in the 4th digit
    of either constant moves the result by > 1e-8 somewhere on the grid."""
    xs = np.linspace(-12, 12, 9601)
    ref = torch.nn.functional.gelu(torch.from_numpy(xs), approximate="tanh").numpy()
    got = np.array([oracle.act("gelu_tanh", float(x)) for x in xs])
    err = np.abs(got - ref)
    assert err.max() <= 1e-12, (xs[err.argmax()], err.max())


def test_f16_decode_matches_library_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(b) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_decode_matches_torch_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_double(b) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_synth_bf16_rounding_matches_torch():
    x = synth.Stream(9).normal(100000, 3.0).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16_bits(x), ref)


def test_half_ulp_matches_format_facts():
    # bf16 keeps 8 significant bits, fp16 keeps 11
    assert oracle.half_ulp(1.0, "bf16") == 2.0**-8
    assert oracle.half_ulp(1.5, "bf16") == 2.0**-8
    assert oracle.half_ulp(32.0, "bf16") == 2.0**-3
    assert oracle.half_ulp(1.0, "f16") == 2.0**-11
    assert oracle.half_ulp(1000.0, "f16") == 2.0**-2
    # nextafter in the format, via the library: the gap above 3.0 in fp16
    gap = float(np.nextafter(np.float16(3.0), np.float16(10)) - np.float16(3.0))
    assert oracle.half_ulp(3.0, "f16") == gap / 2


def test_checker_accepts_rounded_oracle_and_rejects_one_ulp_plus():
    p = synth.Problem(64, 48, 512, dtype="bf16", seed=21, distC="uniform")
    r, sabs = oracle.gemm_full(p, alpha=1.5, beta=0.5)
    d = oracle.decode(synth.store(r.ravel(), "bf16"), "bf16")
    ok, worst, _ = oracle.check_float(d, r.ravel(), sabs.ravel(), "bf16")
    assert ok
    d2 = d.copy()
    d2[100] = r.ravel()[100] + 4 * oracle.half_ulp(r.ravel()[100], "bf16") + 0.01 * sabs.ravel()[100]
    ok2, _, w = oracle.check_float(d2, r.ravel(), sabs.ravel(), "bf16")
    assert not ok2 and w == 100


def test_freivalds_int8_detects_single_error():
    p = synth.Problem(40, 33, 70, dtype="i8", distA="int8", distB="int8", seed=3)
    r, _ = oracle.gemm_full(p)
    x = oracle.freivalds_vector(p.N, 3)
    bx = oracle.matvec(p.K, p.N, p.B, p.ldb, p.layoutB, "i8", x)
    abx = oracle.matvec(p.M, p.K, p.A, p.lda, p.layoutA, "i8", bx)
    assert np.array_equal(r @ x, abx)
    r[7, 5] += 1
    assert not np.array_equal(r @ x, abx)


def test_sample_indices_cover_first_and_last():
    ii, jj = oracle.sample_indices(8192, 14336, 2)
    assert ii.min() == 0 and ii.max() == 8191 and jj.min() == 0 and jj.max() == 14335
    rows = set(ii[:8 * 14336].tolist())
    assert 0 in rows and 8191 in rows and len(rows) == 8
    assert np.array_equal(jj[:14336], np.arange(14336))


def test_synth_layouts_hold_same_logical_matrix():
    ps = [synth.Problem(13, 9, 11, dtype="bf16", layoutA=la, layoutB=lb, seed=4) for la, lb in COMBOS]
    for p in ps[1:]:
        assert np.array_equal(p.A_log, ps[0].A_log) and np.array_equal(p.B_log, ps[0].B_log)
        assert np.array_equal(synth.from_layout(p.A, 13, 11, p.layoutA, p.lda), p.A_log)
        assert np.array_equal(synth.from_layout(p.B, 11, 9, p.layoutB, p.ldb), p.B_log)


# ---------------------------------------------------------------- transpose

def test_transpose_worked_example():
    # 2 x 3 source with pitch 4 (the 4th column is padding) -> 3 x 2 with pitch 3
    src = np.array([1, 2, 3, 99,
                    4, 5, 6, 99], dtype=np.uint32)
    dst = oracle.transpose(src, 2, 3, lds=4, ldd=3)
    assert dst.tolist() == [1, 4, 0,
                            2, 5, 0,
                            3, 6, 0]


@pytest.mark.parametrize("rows,cols,eb", [(1, 1, 1), (7, 3, 2), (33, 65, 4), (64, 1, 8), (1, 70, 2)])
def test_transpose_matches_numpy_and_is_an_involution(rows, cols, eb):
    src = synth.transpose_input(rows, cols, eb, seed=rows * 131 + cols, lds=cols + 3)
    dst = oracle.transpose(src, rows, cols, lds=cols + 3, ldd=rows + 1)
    logical = src.reshape(rows, cols + 3)[:, :cols]
    assert np.array_equal(dst.reshape(cols, rows + 1)[:, :rows], logical.T)
    assert not dst.reshape(cols, rows + 1)[:, rows:].any()
    back = oracle.transpose(dst, cols, rows, lds=rows + 1, ldd=cols)
    assert np.array_equal(back.reshape(rows, cols), logical)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "i8"])
@pytest.mark.parametrize("layout", ["row", "col"])
def test_matvec_matches_numpy(dtype, layout):
    rows, cols = 37, 53
    st = synth.Stream(17)
    vals = synth.draw(st, rows * cols, "int8" if dtype == "i8" else "uniform")
    X = synth.store(vals, dtype).reshape(rows, cols)
    buf, ld = synth.to_layout(X, layout, (cols if layout == "row" else rows) + 3)
    x = synth.Stream(18).uniform(cols)
    logical = X.astype(np.float64) if dtype == "i8" else oracle.decode(X, dtype)
    y = oracle.matvec(rows, cols, buf, ld, layout, dtype, x)
    assert np.allclose(y, logical @ x, rtol=1e-13, atol=1e-12)
