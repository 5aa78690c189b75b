"""GPU parity of the matrix-vector path (M == 1 or N == 1) against the oracle,
and of the same problems on the tensor-core kernels (gemv knob = 1)."""
import numpy as np
import pytest

import oracle
import synth
import tiled_tensor_core_02_gb300 as ttc
from gpu_util import run

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _knobs():
    ttc.load()
    ttc.ttc_set_knob("gemv", 0)
    yield
    ttc.ttc_set_knob("gemv", 0)


def check(p, d, alpha, beta, act="none"):
    r, sabs = oracle.gemm_full(p, alpha=alpha, beta=beta, act=act)
    ok, worst, w = oracle.check_float(oracle.decode(d.ravel(), p.dtype), r.ravel(), sabs.ravel(), p.dtype)
    assert ok, f"worst error ratio {worst:.3f} at {divmod(w, p.N)}"


SHAPES = [(1, 4096, 4096), (1, 300, 1000), (1, 7, 5), (1, 64, 4099), (1, 1, 777), (1, 5000, 20000),
          (4096, 1, 4096), (1000, 1, 300), (5, 1, 7), (4099, 1, 64), (5000, 1, 20000)]


@pytest.mark.parametrize("gemv_off", [0, 1])
@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_matrix_vector_all_layouts(shape, la, lb, gemv_off):
    M, N, K = shape
    p = synth.Problem(M, N, K, dtype="bf16", layoutA=la, layoutB=lb, seed=M + 3 * N + 7 * K, distC="uniform",
                      dist_bias="uniform")
    ttc.ttc_set_knob("gemv", gemv_off)
    check(p, run(p, 1.0, 1.0), 1.0, 1.0)


@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
@pytest.mark.parametrize("shape", [(1, 520, 2000), (2000, 1, 520)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_matrix_vector_epilogue_and_dtypes(shape, dtype, act):
    M, N, K = shape
    for la, lb in synth.MAJORNESS:
        p = synth.Problem(M, N, K, dtype=dtype, layoutA=la, layoutB=lb, seed=11, distC="uniform",
                          dist_bias="uniform")
        check(p, run(p, 0.5, -1.5, act), 0.5, -1.5, act)


@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_matrix_vector_odd_pitches(la, lb):
    # pitches that break 16-byte alignment: the per-element loads
    for M, N, K in [(1, 333, 515), (515, 1, 333)]:
        p = synth.Problem(M, N, K, dtype="bf16", layoutA=la, layoutB=lb, seed=13, distC="uniform",
                          lda=(K if la == "row" else M) + 3, ldb=(N if lb == "row" else K) + 5, ldc=N + 1)
        check(p, run(p, 1.0, 1.0, ldd=N + 3), 1.0, 1.0)


@pytest.mark.parametrize("la,lb", synth.MAJORNESS)
def test_matrix_vector_is_one_launch(la, lb):
    """Either matrix-vector kernel (the reduction or the outputs contiguous in
    B) is one launch, with no workspace."""
    p = synth.Problem(1, 4096, 4096, dtype="bf16", layoutA=la, layoutB=lb, seed=2)
    n0 = ttc.ttc_launch_count()
    run(p, 1.0, 0.0)
    assert ttc.ttc_launch_count() == n0 + 1
