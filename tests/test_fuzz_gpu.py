"""Seeded random problems through every planner branch, checked in full
against the oracle: sizes around the tile, k-block and chunk boundaries
(1 to 513 rows and columns, K from 1 to 1025), all four A/B majorness
combinations, tight and padded pitches, fp16/bf16 with every epilogue
(alpha, beta with C, bias, ReLU, tanh-GELU) and int8 with and without C,
through ttc_gemm and ttc_gemm_ws (with the workspace for the operand repack
only, or for its fastest path), with the int8 CTA-pair path forced on some
int8 calls.  The planner picks the kernel (CTA pair or single CTA, tile
width, orientation, split K, matrix-vector kernels) from each shape."""
import numpy as np
import pytest

import oracle
import synth
import tiled_tensor_core_02_gb300 as ttc
from gpu_util import run

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
