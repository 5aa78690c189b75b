"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Floating outputs must lie within the oracle's per-element tolerance (see
oracle/__init__.py); int8 -> int32 must be bit-exact.  Sizes the oracle can
finish in seconds are compared element by element; the full-size workloads
are compared on sampled rows, columns and elements (and with a Freivalds
check where the epilogue is linear).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_tensor_core_02_gb300 as ttc
from gpu_util import run, run_batched, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_tensor_core_02_gb300 import _build
    _build.build()
    ttc.load()
    for k in ("inject_stall", "force_generic_load", "force_generic_store", "tile_n", "pair", "swap_ab",
              "split_k", "pair_tile_n", "pair_tail", "conv_halo", "pair_epi_warps"):
        ttc.ttc_set_knob(k, 0)
    yield


def check_full(p, d, alpha, beta, act="none", use_bias=True):
    r, sabs = oracle.gemm_full(p, alpha=alpha, beta=beta, act=act, use_bias=use_bias)
    if p.dtype == "i8":
        assert np.array_equal(d.astype(np.int64), r.astype(np.int64))
        return 0.0
    ok, worst, w = oracle.check_float(oracle.decode(d.ravel(), p.dtype), r.ravel(), sabs.ravel(), p.dtype)
    assert ok, f"worst error ratio {worst:.3f} at {divmod(w, p.N)}: got {oracle.decode(d.ravel()[w:w+1], p.dtype)} want {r.ravel()[w]}"
    return worst


def check_sampled(p, d, alpha, beta, act="none", seed=0):
    ii, jj = oracle.sample_indices(p.M, p.N, seed)
    r, sabs, _ = oracle.gemm_elements(p, ii, jj, alpha=alpha, beta=beta, act=act)
    got = d[ii, jj]
    if p.dtype == "i8":
        assert np.array_equal(got.astype(np.int64), r.astype(np.int64))
        return
    ok, worst, w = oracle.check_float(oracle.decode(got, p.dtype), r, sabs, p.dtype)
    assert ok, f"worst ratio {worst:.3f} at ({ii[w]},{jj[w]})"


def freivalds(p, d, alpha, beta, seed):
    """D x == alpha A (B x) + beta C x within the summed per-element tolerance."""
    x = oracle.freivalds_vector(p.N, seed)
    bx = oracle.matvec(p.K, p.N, p.B, p.ldb, p.layoutB, p.dtype, x)
    want = alpha * oracle.matvec(p.M, p.K, p.A, p.lda, p.layoutA, p.dtype, bx)
    if beta != 0.0:
        want += beta * (oracle.decode(p.C, p.dtype).reshape(p.M, p.ldc)[:, :p.N] @ x)
    dv = oracle.decode(d, p.dtype) if p.dtype != "i8" else d.astype(np.float64)
    got = dv @ x
    if p.dtype == "i8":
        assert np.array_equal(got, want)
        return
    # per-row bound: the sum of per-element tolerances, with S_abs bounded by K*max|a|*max|b|
    amax = np.abs(oracle.decode(p.A, p.dtype)).max()
    bmax = np.abs(oracle.decode(p.B, p.dtype)).max()
    tol = p.N * (1e-2 * p.K * amax * bmax * 2.0**-7 + 1e-3) + np.abs(dv).sum(axis=1) * 2.0**-8
    assert np.all(np.abs(got - want) <= tol)


# ------------------------------------------------------------------ small, full checks

def test_fp16_256_cube():
    p, a, b, act = synth.make(synth.WORKLOADS["fp16_256"])
    d = run(p, a, b, act)
    check_full(p, d, a, b, act)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_majorness_ragged_tiles(dtype, la, lb):
    # several tiles plus ragged tails in M, N and K; leading dims keep TMA legal
    M, N, K = 300, 520, 200
    p = synth.Problem(M, N, K, dtype=dtype, layoutA=la, layoutB=lb, seed=10, distC="uniform",
                      dist_bias="normal:0.5",
                      lda=(208 if la == "row" else 304), ldb=(520 if lb == "row" else 200))
    d = run(p, 1.25, -0.75, "none")
    check_full(p, d, 1.25, -0.75)


@pytest.mark.parametrize("act", ["none", "relu", "gelu_tanh"])
def test_epilogue_bias_activation(act):
    p = synth.Problem(256, 384, 192, dtype="bf16", seed=11, distA="normal:1.0",
                      distB="normal:0.1", dist_bias="normal:0.5")
    d = run(p, 1.0, 0.0, act)
    check_full(p, d, 1.0, 0.0, act)


@pytest.mark.parametrize("tile_n", [256, 128, 64, 32])
def test_every_tile_width(tile_n):
    ttc.ttc_set_knob("tile_n", tile_n)
    try:
        p = synth.Problem(200, 136, 136, dtype="bf16", seed=12, distC="uniform")
        d = run(p, 0.5, 2.0)
        check_full(p, d, 0.5, 2.0)
    finally:
        ttc.ttc_set_knob("tile_n", 0)


def test_generic_store_path():
    ttc.ttc_set_knob("force_generic_store", 1)
    try:
        p = synth.Problem(130, 70, 64, dtype="bf16", seed=13, distC="uniform")
        d = run(p, 1.0, 1.0, ldd=77)
        check_full(p, d, 1.0, 1.0)
    finally:
        ttc.ttc_set_knob("force_generic_store", 0)


def test_k_zero_is_epilogue_only():
    p = synth.Problem(64, 48, 0, dtype="bf16", seed=14, distC="uniform", dist_bias="uniform",
                      lda=1, ldb=1)
    d = run(p, 3.0, 0.5, "relu")
    check_full(p, d, 3.0, 0.5, "relu")


def test_beta_zero_ignores_nan_c():
    p = synth.Problem(128, 64, 64, dtype="bf16", seed=15, distC="uniform")
    p.C[:] = 0x7FC0
    d = run(p, 1.0, 0.0)
    check_full(p, d, 1.0, 0.0)


def test_in_place_c_equals_d():
    p = synth.Problem(192, 256, 128, dtype="bf16", seed=16, distC="uniform")
    Cd = to_dev(p.C)
    d = run(p, 1.0, 1.0, C_dev=Cd, D=Cd)
    check_full(p, d, 1.0, 1.0)


@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (7, 8, 16), (1, 1, 1), (129, 33, 65), (16, 512, 1024)])
def test_small_and_degenerate(M, N, K):
    p = synth.Problem(M, N, K, dtype="bf16", seed=17, distC="uniform",
                      lda=((K + 7) // 8) * 8, ldb=((K + 7) // 8) * 8)
    d = run(p, 1.0, 1.0, ldd=((N + 7) // 8) * 8)
    check_full(p, d, 1.0, 1.0)


def test_two_streams_and_repeat():
    p = synth.Problem(256, 256, 256, dtype="bf16", seed=18)
    s2 = torch.cuda.Stream()
    d1 = run(p, 1.0, 0.0)
    d2 = run(p, 1.0, 0.0, stream=s2.cuda_stream)
    assert np.array_equal(d1, d2)
    check_full(p, d1, 1.0, 0.0)


# ------------------------------------------------------------------ the suite's workloads

def test_bf16_4096_alpha_beta_full():
    p, a, b, act = synth.make(synth.WORKLOADS["bf16_4096"])
    d = run(p, a, b, act)
    check_full(p, d, a, b, act)


def test_bf16_mlp_gelu_sampled():
    p, a, b, act = synth.make(synth.WORKLOADS["bf16_mlp_8192x14336x4096"])
    d = run(p, a, b, act)
    check_sampled(p, d, a, b, act, seed=2)


def test_bf16_8192_sampled_and_freivalds():
    p, a, b, act = synth.make(synth.WORKLOADS["bf16_8192"])
    d = run(p, a, b, act)
    check_sampled(p, d, a, b, act, seed=1)
    freivalds(p, d, a, b, seed=1)


# ------------------------------------------------------------------ failure detection

@pytest.mark.parametrize("pair", [1, 2], ids=["pair", "single"])
def test_stalled_pipeline_times_out_and_context_survives(pair):
    """A tensor-core issuer that waits on a barrier nothing arrives at must end
    the kernel with TTC_ERR_TIMEOUT within the wait budget, and the context
    must stay usable."""
    p = synth.Problem(256, 512, 512, dtype="bf16", seed=19)
    ttc.ttc_set_knob("pair", pair)
    ttc.ttc_set_knob("timeout_ns", 200_000_000)
    ttc.ttc_set_knob("inject_stall", 1)
    try:
        A, B = to_dev(p.A), to_dev(p.B)
        D = torch.zeros(p.M * p.N, dtype=torch.int16, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        st = ttc.ttc_gemm(p.M, p.N, p.K, A.data_ptr(), p.lda, 0, B.data_ptr(), p.ldb, 1, None, p.N,
                          D.data_ptr(), p.N, 1.0, 0.0, None, 0, ttc.DTYPE["bf16"], s)
        assert st == 0
        assert ttc.ttc_get_device_error(s) == 4
    finally:
        ttc.ttc_set_knob("inject_stall", 0)
        ttc.ttc_set_knob("timeout_ns", 0)
    assert ttc.ttc_get_device_error(None) == 0
    try:
        d = run(p, 1.0, 0.0)
        check_full(p, d, 1.0, 0.0)
    finally:
        ttc.ttc_set_knob("pair", 0)


def test_int8_pair_path_stall_times_out_and_context_survives():
    """The same on the int8 CTA-pair path (widening copy, then the pair kernel
    with 1024-deep partials): its issuer stalls, every wait gives up within
    the budget, and the next call on the path is exact."""
    p = synth.Problem(256, 512, 2048, dtype="i8", seed=36, distA="int8", distB="int8")
    ttc.ttc_set_knob("i8_wide", 1)
    ttc.ttc_set_knob("timeout_ns", 200_000_000)
    ttc.ttc_set_knob("inject_stall", 1)
    try:
        A, B = to_dev(p.A), to_dev(p.B)
        D = torch.zeros(p.M * p.N, dtype=torch.int32, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        need = ttc.ttc_gemm_workspace_size_staged(p.M, p.N, p.K, A.data_ptr(), p.lda, 0, B.data_ptr(), p.ldb, 1,
                                                  D.data_ptr(), p.N, ttc.DTYPE["i8"])
        assert need > 0
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        n0 = ttc.ttc_launch_count()
        st = ttc.ttc_gemm_ws(p.M, p.N, p.K, A.data_ptr(), p.lda, 0, B.data_ptr(), p.ldb, 1, None, p.N,
                             D.data_ptr(), p.N, 1.0, 0.0, None, 0, ttc.DTYPE["i8"], ws.data_ptr(), need, s)
        assert st == 0 and ttc.ttc_launch_count() - n0 == 2
        assert ttc.ttc_get_device_error(s) == 4
    finally:
        ttc.ttc_set_knob("inject_stall", 0)
        ttc.ttc_set_knob("timeout_ns", 0)
    try:
        assert ttc.ttc_get_device_error(None) == 0
        d = run(p, 1.0, 0.0, workspace=-2)
        check_full(p, d, 1.0, 0.0)
    finally:
        ttc.ttc_set_knob("i8_wide", 0)


# ------------------------------------------------------------------ operands TMA cannot describe

@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_generic_producer_forced(dtype, la, lb):
    ttc.ttc_set_knob("force_generic_load", 1)
    try:
        p = synth.Problem(300, 520, 200, dtype=dtype, layoutA=la, layoutB=lb, seed=20, distC="uniform",
                          dist_bias="normal:0.5")
        d = run(p, 1.0, 1.0, "relu")
        check_full(p, d, 1.0, 1.0, "relu")
    finally:
        ttc.ttc_set_knob("force_generic_load", 0)


@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_odd_leading_dimensions(la, lb):
    # odd pitches: no TMA for any operand, no vector loads, predicated stores
    M, N, K = 257, 131, 97
    p = synth.Problem(M, N, K, dtype="bf16", layoutA=la, layoutB=lb, seed=21, distC="uniform",
                      lda=(K if la == "row" else M) + 1, ldb=(N if lb == "row" else K) + 3, ldc=N + 5)
    d = run(p, 1.0, 1.0, ldd=N + 7)
    check_full(p, d, 1.0, 1.0)


@pytest.mark.parametrize("shape", synth.RAGGED_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_ragged_sweep(shape, la, lb):
    """The ragged / skinny sweep with tight leading dimensions, checked in full."""
    p, a, b, act = synth.make(synth.ragged_workload(*shape, la, lb))
    d = run(p, a, b, act)
    check_full(p, d, a, b, act)


# ------------------------------------------------------------------ int8 -> int32, exact

@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_int8_small_all_layouts(la, lb):
    p = synth.Problem(200, 150, 300, dtype="i8", layoutA=la, layoutB=lb, seed=22, distA="int8",
                      distB="int8")
    d = run(p, 1.0, 0.0)
    check_full(p, d, 1.0, 0.0)


@pytest.mark.parametrize("tile_n", [128, 64, 32])
@pytest.mark.parametrize("K", [32, 64, 192, 960, 1088])
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_int8_k_tails(la, lb, K, tile_n):
    """int8 K tails on every tile width: the two converter groups take
    alternate k-blocks, so an odd count leaves one group a k-block short; K
    below one k-block leaves most of the raw tile zero-filled.  Both majorness
    of B (the MN-major one from 64 columns up)."""
    if lb == "row" and tile_n < 64:
        pytest.skip("an MN-major B needs whole 64-column slabs")
    ttc.ttc_set_knob("tile_n", tile_n)
    try:
        p = synth.Problem(136, 200, K, dtype="i8", layoutA=la, layoutB=lb, seed=29, distA="int8", distB="int8")
        d = run(p, 1.0, 0.0)
        check_full(p, d, 1.0, 0.0)
    finally:
        ttc.ttc_set_knob("tile_n", 0)


def _run_i8_wide(p, beta=0.0, force=True):
    """Runs p through ttc_gemm_ws with the workspace for fp16 copies of the
    operands; returns the output and the number of kernels launched."""
    ttc.ttc_set_knob("i8_wide", 1 if force else 0)
    try:
        n0 = ttc.ttc_launch_count()
        d = run(p, 1.0, beta, workspace=-2)
        return d, ttc.ttc_launch_count() - n0
    finally:
        ttc.ttc_set_knob("i8_wide", 0)


@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (300, 520, 1000), (520, 600, 2112), (257, 300, 1088)])
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_int8_pair_path_exact(la, lb, M, N, K):
    """int8 on the CTA-pair kernel (fp16 copies of the operands, 1024-deep
    partial sums added as int32): bit-exact, with ragged tiles, K tails of an
    odd number of k-blocks, and more than one partial per tile.  Two launches:
    the widening copy and the pair kernel."""
    p = synth.Problem(M, N, K, dtype="i8", layoutA=la, layoutB=lb, seed=33, distA="int8", distB="int8")
    d, launches = _run_i8_wide(p)
    assert launches == 2
    check_full(p, d, 1.0, 0.0)


def test_int8_pair_path_adds_c_and_stays_exact():
    """beta = 1 adds an int32 C; -128 * -128 over K = 8192 reaches K * 2^14 =
    2^27, eight 1024-deep partials of 2^24 each."""
    M, N, K = 256, 512, 8192
    p = synth.Problem.from_logical(np.full((M, K), -128, np.int8), np.full((K, N), -128, np.int8), dtype="i8")
    d, launches = _run_i8_wide(p)
    assert launches == 2 and np.all(d == K * 16384)
    q = synth.Problem(300, 600, 1500, dtype="i8", seed=34, distA="int8", distB="int8")
    rng = np.random.default_rng(1)
    c = rng.integers(-2**20, 2**20, size=(q.M, q.N)).astype(np.int32)
    q.C_log = c
    q.C, q.ldc = synth.to_layout(c, "row")
    d, launches = _run_i8_wide(q, beta=1.0)
    assert launches == 2
    check_full(q, d, 1.0, 1.0)


def test_int8_pair_path_half_tile_tail():
    """81 pair tiles on the resident pairs: the last partial wave runs as half
    tiles (N = 128 units); the planner takes the pair path by itself."""
    p = synth.Problem(2304, 2304, 192, dtype="i8", layoutA="row", layoutB="col", seed=35, distA="int8",
                      distB="int8")
    d, launches = _run_i8_wide(p, force=False)
    assert launches == 2
    check_full(p, d, 1.0, 0.0)


def test_int8_8192_pair_path_sampled_and_freivalds():
    p, a, b, act = synth.make(synth.WORKLOADS["i8_8192"])
    d, launches = _run_i8_wide(p, force=False)
    assert launches == 2
    check_sampled(p, d, a, b, act, seed=5)
    freivalds(p, d, a, b, seed=5)


def test_int8_beta_one_adds_c():
    p = synth.Problem(130, 70, 64, dtype="i8", seed=23, distA="int8", distB="int8")
    rng = np.random.default_rng(0)
    c = rng.integers(-2**20, 2**20, size=(p.M, p.N)).astype(np.int32)
    p.C_log = c
    p.C, p.ldc = synth.to_layout(c, "row")
    d = run(p, 1.0, 1.0)
    check_full(p, d, 1.0, 1.0)


@pytest.mark.parametrize("K", [1024, 1025, 8192])
def test_int8_extreme_values_stay_exact(K):
    """-128 * -128 everywhere: each 1024-deep partial sum reaches 2^24, the
    largest integer an fp32 accumulator holds exactly; the int32 result is
    K * 2^14."""
    M, N = 128, 64
    p = synth.Problem.from_logical(np.full((M, K), -128, np.int8), np.full((K, N), -128, np.int8), dtype="i8")
    d = run(p, 1.0, 0.0)
    assert np.all(d == K * 16384)
    # mixed signs that cancel only in exact arithmetic
    a = np.full((M, K), 127, np.int8)
    a[:, 1::2] = -128
    b = np.full((K, N), 127, np.int8)
    q = synth.Problem.from_logical(a, b, dtype="i8")
    d = run(q, 1.0, 0.0)
    check_full(q, d, 1.0, 0.0)


def test_int8_8192_sampled_and_freivalds():
    p, a, b, act = synth.make(synth.WORKLOADS["i8_8192"])
    d = run(p, a, b, act)
    check_sampled(p, d, a, b, act, seed=3)
    freivalds(p, d, a, b, seed=3)


# ------------------------------------------------------------------ single-CTA vs CTA-pair kernels

@pytest.mark.parametrize("pair", [1, 2, 3], ids=["pair", "single", "pair-whole-tiles"])
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_pair_and_single_kernels(pair, la, lb):
    """9 pair tiles: on the pair kernel as 18 half tiles (the default for a
    problem of at most half a wave) or as whole tiles."""
    ttc.ttc_set_knob("pair", 1 if pair == 3 else pair)
    ttc.ttc_set_knob("pair_tail", 1 if pair == 3 else 0)
    try:
        p = synth.Problem(520, 600, 264, dtype="bf16", layoutA=la, layoutB=lb, seed=24, distC="uniform",
                          dist_bias="normal:0.5")
        d = run(p, 0.75, 1.5, "gelu_tanh")
        check_full(p, d, 0.75, 1.5, "gelu_tanh")
    finally:
        ttc.ttc_set_knob("pair_tail", 0)
        ttc.ttc_set_knob("pair", 0)


@pytest.mark.parametrize("tail", [0, 1], ids=["halves", "whole"])
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_pair_kernel_last_wave_halves(tail, la, lb):
    """80 pair tiles (10 x 8, ragged in M and N): on 76 resident pairs the
    last 4 run as 8 half tiles (tail = 0) or whole (tail = 1); the second half
    of the last tile column lies partly past N."""
    ttc.ttc_set_knob("pair", 1)
    ttc.ttc_set_knob("pair_tail", tail)
    try:
        p = synth.Problem(2500, 2000, 192, dtype="bf16", layoutA=la, layoutB=lb, seed=26, distC="uniform",
                          dist_bias="normal:0.5")
        d = run(p, 1.25, 0.5, "gelu_tanh")
        check_full(p, d, 1.25, 0.5, "gelu_tanh")
    finally:
        ttc.ttc_set_knob("pair_tail", 0)
        ttc.ttc_set_knob("pair", 0)


@pytest.mark.parametrize("M,N,K", [(130, 70, 64), (1, 300, 128), (257, 9, 100), (600, 40, 0)])
def test_pair_kernel_on_small_and_ragged(M, N, K):
    ttc.ttc_set_knob("pair", 1)
    try:
        p = synth.Problem(M, N, K, dtype="f16", seed=25, distC="uniform", lda=max(8, (K + 7) // 8 * 8),
                          ldb=max(8, (K + 7) // 8 * 8))
        d = run(p, 1.0, 1.0, ldd=(N + 7) // 8 * 8)
        check_full(p, d, 1.0, 1.0)
    finally:
        ttc.ttc_set_knob("pair", 0)


# ------------------------------------------------------------------ D^T = B^T A^T (skinny problems)

@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
@pytest.mark.parametrize("act", ["none", "gelu_tanh"])
def test_swap_ab_forced(la, lb, act):
    ttc.ttc_set_knob("swap_ab", 1)
    try:
        p = synth.Problem(150, 300, 136, dtype="bf16", layoutA=la, layoutB=lb, seed=26, distC="uniform",
                          dist_bias="normal:0.5")
        d = run(p, 1.25, 0.5, act, ldd=304)
        check_full(p, d, 1.25, 0.5, act)
    finally:
        ttc.ttc_set_knob("swap_ab", 0)


def test_swap_ab_int8_with_c():
    ttc.ttc_set_knob("swap_ab", 1)
    try:
        p = synth.Problem(70, 200, 300, dtype="i8", seed=27, distA="int8", distB="int8")
        rng = np.random.default_rng(1)
        c = rng.integers(-2**20, 2**20, size=(p.M, p.N)).astype(np.int32)
        p.C_log = c
        p.C, p.ldc = synth.to_layout(c, "row")
        d = run(p, 1.0, 1.0)
        check_full(p, d, 1.0, 1.0)
    finally:
        ttc.ttc_set_knob("swap_ab", 0)


@pytest.mark.parametrize("swap", [1, 2], ids=["swap", "noswap"])
def test_skinny_orientation_both_ways(swap):
    ttc.ttc_set_knob("swap_ab", swap)
    try:
        p, a, b, act = synth.make(synth.ragged_workload(8192, 24, 4096, "row", "col"))
        d = run(p, a, b, act)
        check_full(p, d, a, b, act)
    finally:
        ttc.ttc_set_knob("swap_ab", 0)


# ------------------------------------------------------------------ split-K across a cluster

@pytest.mark.parametrize("split", [2, 3, 4, 8])
@pytest.mark.parametrize("la,lb", [("row", "col"), ("col", "row")])
def test_split_k_forced(split, la, lb):
    # K = 1000 gives 16 k-blocks: uneven splits, and for 8 splits two blocks each
    ttc.ttc_set_knob("split_k", split)
    try:
        p = synth.Problem(200, 200, 1000, dtype="bf16", layoutA=la, layoutB=lb, seed=28, distC="uniform",
                          dist_bias="normal:0.5")
        d = run(p, 1.0, 0.5, "relu")
        check_full(p, d, 1.0, 0.5, "relu")
    finally:
        ttc.ttc_set_knob("split_k", 0)


def test_split_k_more_splits_than_k_blocks():
    # 2 k-blocks over 8 CTAs: six CTAs hold empty (zero) partial sums
    ttc.ttc_set_knob("split_k", 8)
    try:
        p = synth.Problem(130, 90, 100, dtype="f16", seed=29, distC="uniform")
        d = run(p, 1.0, 1.0)
        check_full(p, d, 1.0, 1.0)
    finally:
        ttc.ttc_set_knob("split_k", 0)


def test_split_k_generic_producer_and_swap():
    ttc.ttc_set_knob("split_k", 4)
    ttc.ttc_set_knob("swap_ab", 1)
    try:
        p = synth.Problem(40, 300, 777, dtype="bf16", seed=30, distC="uniform", lda=779, ldb=781)
        d = run(p, 1.0, 1.0, ldd=303)
        check_full(p, d, 1.0, 1.0)
    finally:
        ttc.ttc_set_knob("split_k", 0)
        ttc.ttc_set_knob("swap_ab", 0)


# ------------------------------------------------------------------ ttc_gemm_ws: repacked operands

@pytest.mark.parametrize("ws", [-1, -2], ids=["repack", "repack+D"])
@pytest.mark.parametrize("shape", synth.RAGGED_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_ragged_sweep_with_workspace(shape, la, lb, ws):
    p, a, b, act = synth.make(synth.ragged_workload(*shape, la, lb))
    d = run(p, a, b, act, workspace=ws)
    check_full(p, d, a, b, act)


@pytest.mark.parametrize("ws", [-1, -2], ids=["repack", "repack+D"])
def test_workspace_int8_odd_pitch(ws):
    """Odd operand pitches; with the staged size the int32 D (pitch 203, rows
    not 16-byte aligned) and C are staged through an aligned copy too."""
    p = synth.Problem(300, 200, 72, dtype="i8", layoutA="row", layoutB="col", seed=31, distA="int8",
                      distB="int8", lda=73, ldb=75, distC="int8")
    d = run(p, 1.0, 1.0, workspace=ws, ldd=203)
    check_full(p, d, 1.0, 1.0)


@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_workspace_staged_d_in_place_and_padding(beta):
    """The staged workspace size with a bf16 D at an odd pitch (written
    directly, no copy of D): C == D in place, and the pitch padding of D left
    untouched."""
    p = synth.Problem(260, 301, 96, dtype="bf16", layoutA="col", layoutB="row", seed=34, distC="uniform",
                      lda=261, ldb=303, ldc=305)
    D = to_dev(p.C.copy())  # C and D share storage, pitch 305
    d = run(p, 1.5, beta, "relu", D=D, C_dev=D, ldd=305, workspace=-2)
    check_full(p, d, 1.5, beta, "relu")
    full = D.cpu().numpy().view(np.uint16).reshape(-1)
    rows = full[: p.M * 305].reshape(p.M, 305)
    assert np.array_equal(rows[:, p.N:], p.C.reshape(-1)[: p.M * 305].reshape(p.M, 305)[:, p.N:])


@pytest.mark.parametrize("pair,N,ew", [(1, 300, 12), (1, 300, 8), (2, 77, 0), (1, 320, 12), (1, 320, 8), (2, 96, 0),
                                       (1, 600, 12), (1, 600, 0)])
@pytest.mark.parametrize("c_off,d_off", [(1, 3), (2, 5), (3, 7), (4, 6), (7, 1), (0, 2)])
def test_unaligned_c_and_d_rows(pair, N, ew, c_off, d_off):
    """C and D rows at every 2-byte phase of a 16-byte block (odd pitches and
    element offsets of the base pointers): the epilogue moves each row segment
    as the aligned 16-byte blocks that cover it, and the block two chunks of a
    row share is stored once with the second.  N = 300 and 77 end inside a
    32-column chunk; N = 320 and 96 end at a chunk boundary inside a tile, so
    the tile's last chunks hold no columns.  Nothing outside D's M x N
    elements is written.  On the CTA-pair kernel, 256-wide tiles of such
    outputs take twelve epilogue warps (ew = 12, the planner's choice; a
    third of a tile's chunks each, one or two of a half tile's), eight when
    forced (ew = 8); ew = 0 leaves the tile width to the planner too."""
    M, K = 300, 128
    ldc, ldd = N + 3, N + 5
    p = synth.Problem(M, N, K, dtype="bf16", seed=50 + c_off, distC="uniform", dist_bias="normal:0.5", ldc=ldc)
    ttc.ttc_set_knob("pair", pair)
    ttc.ttc_set_knob("pair_epi_warps", ew)
    ttc.ttc_set_knob("pair_tile_n", 256 if ew else 0)
    try:
        cbig = np.concatenate([np.zeros(c_off, np.uint16), p.C, np.zeros(8, np.uint16)])
        C_dev = to_dev(cbig)[c_off:]
        Dbig = torch.full((M * ldd + d_off + 8,), -1, dtype=torch.int16, device="cuda")
        d = run(p, 1.0, 0.75, "gelu_tanh", C_dev=C_dev, D=Dbig[d_off:], ldd=ldd)
        check_full(p, d, 1.0, 0.75, "gelu_tanh")
        full = Dbig.cpu().numpy().view(np.uint16)
        assert np.all(full[:d_off] == 0xFFFF) and np.all(full[d_off + M * ldd:] == 0xFFFF)
        rows = full[d_off:d_off + M * ldd].reshape(M, ldd)
        assert np.all(rows[:, N:] == 0xFFFF)
    finally:
        ttc.ttc_set_knob("pair", 0)
        ttc.ttc_set_knob("pair_epi_warps", 0)
        ttc.ttc_set_knob("pair_tile_n", 0)


@pytest.mark.parametrize("dtype,M,N,K,ldd,pair,ws", [
    ("bf16", 300, 300, 64, 304, 0, None), ("bf16", 300, 297, 64, 304, 0, None),
    ("bf16", 600, 601, 128, 608, 1, None), ("bf16", 600, 601, 128, 608, 2, None),
    ("f16", 40, 300, 64, 304, 0, None), ("bf16", 300, 12, 64, 16, 2, None),
    ("i8", 300, 255, 64, 256, 0, None), ("i8", 300, 254, 64, 256, 0, None), ("i8", 1, 255, 16, 255, 0, None),
    ("i8", 2048, 2049, 64, 2052, 0, -2)])
def test_tma_stored_rows_leave_the_pitch_padding(dtype, M, N, K, ldd, pair, ws):
    """D rows TMA can store (16-byte aligned pitch) whose length is not a
    whole number of 16-byte granules: a TMA store clips at the row's end only
    to the granule, so the tensor map stops at the last whole granule and the
    epilogue writes the rest; nothing in the pitch padding is written.  The
    last case runs int8 on the CTA-pair path (fp16 copies in the workspace);
    M = 1 lets the planner pick its own pitch for D's single row."""
    dist = "int8" if dtype == "i8" else "uniform"
    p = synth.Problem(M, N, K, dtype=dtype, seed=71, distA=dist, distB=dist, distC=dist)
    beta = 1.0
    out_t = torch.int32 if dtype == "i8" else torch.int16
    D = torch.full((M * ldd + 16,), -1, dtype=out_t, device="cuda")
    ttc.ttc_set_knob("pair", pair)
    try:
        d = run(p, 1.0, beta, D=D, ldd=ldd, workspace=ws)
    finally:
        ttc.ttc_set_knob("pair", 0)
    check_full(p, d, 1.0, beta)
    full = D.cpu().numpy()
    rows = full[:M * ldd].reshape(M, ldd)
    assert np.all(rows[:, N:] == -1) and np.all(full[M * ldd:] == -1)


def _poison_padding(p):
    """Fills the pitch padding of A, B and C with NaN (int8: 127, int32 C:
    2^30), which the oracle never reads: a kernel that read it would show."""
    val = np.int8(127) if p.dtype == "i8" else np.uint16(0x7FC0 if p.dtype == "bf16" else 0x7E00)
    for buf, rows, cols, ld, lay in ((p.A, p.M, p.K, p.lda, p.layoutA), (p.B, p.K, p.N, p.ldb, p.layoutB)):
        if lay == "row":
            buf.reshape(rows, ld)[:, cols:] = val
        else:
            buf.reshape(cols, ld)[:, rows:] = val
    if p.C is not None:
        p.C.reshape(p.M, p.ldc)[:, p.N:] = np.int32(1 << 30) if p.dtype == "i8" else val


@pytest.mark.parametrize("ws", [None, -2], ids=["plain", "staged"])
@pytest.mark.parametrize("M,N,K", [(300, 300, 100), (40, 300, 1000), (2048, 2049, 100)])
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
@pytest.mark.parametrize("dtype", ["bf16", "i8"])
def test_operand_and_c_pitch_padding_is_never_read(dtype, la, lb, M, N, K, ws):
    """Pitches padded past rows that end inside a 16-byte granule (TMA can
    still read them), with NaN in every padding element: TMA loads fill past
    a row's end with zeros element by element, and no other path reads the
    padding either."""
    per = 16 if dtype == "i8" else 8
    ra, rb = (K if la == "row" else M), (N if lb == "row" else K)
    lda, ldb = -(-ra // per) * per + (per if ra % per == 0 else 0), -(-rb // per) * per + (per if rb % per == 0 else 0)
    dist = "int8" if dtype == "i8" else "uniform"
    p = synth.Problem(M, N, K, dtype=dtype, layoutA=la, layoutB=lb, seed=73, distA=dist, distB=dist, distC=dist,
                      lda=lda, ldb=ldb, ldc=-(-N // 8) * 8 + 8)
    _poison_padding(p)
    d = run(p, 1.0, 1.0, workspace=ws)
    check_full(p, d, 1.0, 1.0)


def test_batched_and_conv_tma_rows_leave_the_pitch_padding():
    probs = batch_problems(3, 300, 300, 64, distC="uniform")
    p0 = probs[0]
    sD = 300 * 304 + 8
    full = []
    outs = run_batched(probs, {"A": p0.A.size, "B": p0.B.size, "C": p0.C.size, "D": sD}, 1.0, 1.0, ldd=304,
                       full=full)
    check_batches(probs, outs, 1.0, 1.0)
    written = np.zeros(full[0].size, dtype=bool)
    for b in range(3):
        rows = np.arange(b * sD, b * sD + 300 * 304).reshape(300, 304)[:, :300]
        written[rows.ravel()] = True
    assert np.all(full[0][~written] == -1)  # pitch padding and the gaps between batches
    from test_conv_gpu import run_conv
    cp = synth.ConvProblem(2, 10, 10, 16, 70, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=72)
    out = run_conv(cp, ldd=72).reshape(-1)[:cp.M * 72].reshape(cp.M, 72)
    r, sabs = oracle.conv_full(cp)
    ok, worst, w = oracle.check_float(oracle.decode(out[:, :70], "bf16").ravel(), r.ravel(), sabs.ravel(), "bf16")
    assert ok, worst
    assert np.all(out[:, 70:] == 0xFFFF)


def test_workspace_too_small_falls_back():
    p = synth.Problem(257, 131, 97, dtype="bf16", seed=32, distC="uniform", lda=98, ldb=99)
    d = run(p, 1.0, 1.0, workspace=64)
    check_full(p, d, 1.0, 1.0)


@pytest.mark.parametrize("width", [224, 192, 128])
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_pair_tile_widths(width, la, lb):
    if width in (224, 192) and lb == "row":
        pytest.skip("224- and 192-wide pair tiles take a column-major B only")
    ttc.ttc_set_knob("pair", 1)
    ttc.ttc_set_knob("pair_tile_n", width)
    try:
        p = synth.Problem(520, 700, 200, dtype="bf16", layoutA=la, layoutB=lb, seed=33, distC="uniform",
                          dist_bias="normal:0.5")
        d = run(p, 1.0, 0.5, "gelu_tanh")
        check_full(p, d, 1.0, 0.5, "gelu_tanh")
    finally:
        ttc.ttc_set_knob("pair_tile_n", 0)
        ttc.ttc_set_knob("pair", 0)


# ------------------------------------------------------------------ strided batched GEMM

def batch_problems(nb, M, N, K, dtype="bf16", la="row", lb="col", seed=50, share_b=False, **kw):
    probs = [synth.Problem(M, N, K, dtype=dtype, layoutA=la, layoutB=lb, seed=seed + i, **kw) for i in range(nb)]
    if share_b:
        for q in probs[1:]:
            q.B, q.B_log = probs[0].B, probs[0].B_log
    # one shared bias for every batch
    for q in probs[1:]:
        q.bias = probs[0].bias
    return probs


def check_batches(probs, outs, alpha, beta, act="none"):
    for q, d in zip(probs, outs):
        check_full(q, d, alpha, beta, act)


@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_batched_all_layouts(la, lb):
    probs = batch_problems(3, 200, 300, 150, la=la, lb=lb, distC="uniform", dist_bias="normal:0.5")
    p0 = probs[0]
    strides = {"A": p0.A.size + 64, "B": p0.B.size + 128, "C": p0.C.size + 8, "D": 200 * 300 + 64}
    outs = run_batched(probs, strides, 1.0, 0.5, "gelu_tanh")
    check_batches(probs, outs, 1.0, 0.5, "gelu_tanh")


def test_batched_shared_b():
    probs = batch_problems(4, 256, 192, 128, share_b=True)
    p0 = probs[0]
    strides = {"A": p0.A.size, "B": 0, "C": 0, "D": 256 * 192}
    outs = run_batched(probs, strides, 1.0, 0.0, share_b=True)
    check_batches(probs, outs, 1.0, 0.0)


def test_batched_odd_strides_use_plain_loads():
    probs = batch_problems(3, 130, 70, 90, distC="uniform")
    p0 = probs[0]
    strides = {"A": p0.A.size + 3, "B": p0.B.size + 5, "C": p0.C.size + 7, "D": 130 * 70 + 9}
    outs = run_batched(probs, strides, 1.0, 1.0)
    check_batches(probs, outs, 1.0, 1.0)


@pytest.mark.parametrize("pair", [1, 2], ids=["pair", "single"])
def test_batched_large_tiles(pair):
    ttc.ttc_set_knob("pair", pair)
    try:
        probs = batch_problems(2, 520, 600, 200, distC="uniform", dist_bias="normal:0.5")
        p0 = probs[0]
        strides = {"A": p0.A.size, "B": p0.B.size, "C": p0.C.size, "D": 520 * 600}
        outs = run_batched(probs, strides, 1.0, 1.0, "relu")
        check_batches(probs, outs, 1.0, 1.0, "relu")
    finally:
        ttc.ttc_set_knob("pair", 0)


def test_batched_int8():
    probs = batch_problems(3, 150, 130, 300, dtype="i8", distA="int8", distB="int8")
    p0 = probs[0]
    strides = {"A": p0.A.size + 16, "B": p0.B.size + 32, "C": 0, "D": 150 * 130 + 4}
    outs = run_batched(probs, strides, 1.0, 0.0)
    check_batches(probs, outs, 1.0, 0.0)


@pytest.mark.parametrize("dtype", ["bf16", "i8"])
def test_batched_aligned_rows_but_odd_batch_strides(dtype):
    """Rows whose pitch allows vector loads, but a batch stride that moves
    every other batch off the vector boundary (and a row-major B whose pitch
    TMA cannot describe, so the plain-load producers run): each batch's
    start decides the vector loads too."""
    dist = "int8" if dtype == "i8" else "uniform"
    probs = batch_problems(5, 256, 129, 128, dtype=dtype, la="row", lb="row", distA=dist, distB=dist, distC=dist,
                           ldc=130)
    p0 = probs[0]
    strides = {"A": p0.A.size + 3, "B": p0.B.size + 1, "C": p0.C.size, "D": 256 * 129}
    outs = run_batched(probs, strides, 1.0, 1.0)
    check_batches(probs, outs, 1.0, 1.0)


@pytest.mark.parametrize("M,N,K", [(16, 1024, 2048), (1024, 24, 1024)])
def test_batched_skinny_split_and_transpose(M, N, K):
    probs = batch_problems(3, M, N, K, distC="uniform")
    p0 = probs[0]
    strides = {"A": p0.A.size, "B": p0.B.size, "C": p0.C.size, "D": M * N}
    outs = run_batched(probs, strides, 1.0, 1.0)
    check_batches(probs, outs, 1.0, 1.0)
