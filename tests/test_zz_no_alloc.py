"""ttc_gemm_static_scratch: the GEMM for callers that cannot allocate device memory.

Some callers may not call cudaMalloc (a plugin inside an application that owns
the device's memory pool, or a path that cannot afford cudaMalloc's implicit
synchronisation), so they cannot pass ttc_gemm_ws a workspace.  This entry
point uses the library's fixed device scratch array instead.  The test runs it
through the C ABI twice in a row, on two different problems whose operands
need scratch (odd pitches), and compares each result with the existing
workspace entry point's, within the parity tolerance; the second call also
shows that stale scratch left by the first does not matter.

Collected last (file name) so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_tensor_core_02_gb300 as ttc
from gpu_util import LAY, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_tensor_core_02_gb300 import _build
    _build.build()
    ttc.load()
    for k in ("inject_stall", "force_generic_load", "force_generic_store", "tile_n", "pair", "swap_ab",
              "split_k"):
        ttc.ttc_set_knob(k, 0)
    yield


def _call(p, entry, alpha, beta, act):
    A, B = to_dev(p.A), to_dev(p.B)
    C = to_dev(p.C) if p.C is not None else None
    bias = to_dev(p.bias) if p.bias is not None else None
    D = torch.full((p.M * p.N,), -1, dtype=torch.int16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    args = (p.M, p.N, p.K, A.data_ptr(), p.lda, LAY[p.layoutA], B.data_ptr(), p.ldb, LAY[p.layoutB],
            C.data_ptr() if C is not None else None, p.ldc, D.data_ptr(), p.N, alpha, beta,
            bias.data_ptr() if bias is not None else None, ttc.ACT[act], ttc.DTYPE[p.dtype])
    if entry == "static":
        before = ttc.ttc_launch_count()
        st = ttc.ttc_gemm_static_scratch(*args, s)
    else:
        # the workspace entry point given room for its fastest path (operand
        # repack and the aligned copy of D), as the static array provides
        need = ttc.ttc_gemm_workspace_size_staged(p.M, p.N, p.K, A.data_ptr(), p.lda, LAY[p.layoutA],
                                                  B.data_ptr(), p.ldb, LAY[p.layoutB], D.data_ptr(), p.N,
                                                  ttc.DTYPE[p.dtype])
        assert need <= ttc.STATIC_SCRATCH_BYTES
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        before = ttc.ttc_launch_count()
        st = ttc.ttc_gemm_ws(*args, ws.data_ptr(), need, s)
    launches = ttc.ttc_launch_count() - before
    assert st == 0, ttc.STATUS.get(st, st)
    assert ttc.ttc_get_device_error(s) == 0
    return D.cpu().numpy().view(np.uint16).reshape(p.M, p.N), launches


def _expected_launches(p, beta):
    """Kernels a call launches when the scratch is used: one repack (of every
    operand whose pitch is not a 16-byte multiple), then the GEMM, which
    writes fp16/bf16 rows at any alignment itself."""
    rep = int((p.lda * 2) % 16 != 0 or (p.ldb * 2) % 16 != 0)
    return rep + 1


def test_static_scratch_matches_workspace_entry_twice():
    problems = [
        (synth.Problem(300, 260, 197, dtype="bf16", layoutA="row", layoutB="col", seed=40,
                       distC="uniform", lda=199, ldb=201), 1.0, 1.0, "none"),
        (synth.Problem(517, 390, 333, dtype="f16", layoutA="col", layoutB="row", seed=41,
                       distC="uniform", dist_bias="normal:0.5", lda=519, ldb=391), 0.5, -1.0, "gelu_tanh"),
    ]
    for p, alpha, beta, act in problems:
        A, B = to_dev(p.A), to_dev(p.B)
        need = ttc.ttc_gemm_workspace_size(p.M, p.N, p.K, A.data_ptr(), p.lda, LAY[p.layoutA],
                                           B.data_ptr(), p.ldb, LAY[p.layoutB], ttc.DTYPE[p.dtype])
        assert 0 < need <= ttc.STATIC_SCRATCH_BYTES  # the case that needs scratch
        d_static, n_static = _call(p, "static", alpha, beta, act)
        d_ws, n_ws = _call(p, "ws", alpha, beta, act)
        # the static call really ran on its scratch: the same repack and D-staging
        # kernels as the workspace call (a call that found no usable scratch would
        # launch the GEMM alone, reading the operands with plain loads)
        assert n_static == n_ws == _expected_launches(p, beta), (n_static, n_ws)
        r, sabs = oracle.gemm_full(p, alpha=alpha, beta=beta, act=act)
        # the two entry points agree within the parity tolerance (both against the
        # oracle's S_abs-based bound, and with each other)
        tol = oracle.tolerance(oracle.decode(d_static.ravel(), p.dtype), r.ravel(), sabs.ravel(), p.dtype)
        diff = np.abs(oracle.decode(d_static.ravel(), p.dtype) - oracle.decode(d_ws.ravel(), p.dtype))
        assert np.all(diff <= tol)
        ok, worst, _ = oracle.check_float(oracle.decode(d_static.ravel(), p.dtype), r.ravel(), sabs.ravel(),
                                          p.dtype)
        assert ok, worst


def test_static_scratch_runs_int8_on_the_pair_path():
    """An int8 problem of 64 pair tiles whose fp16 operand copies (8 MiB) fit
    the static array: the call widens them there and runs the CTA-pair kernel
    (two launches), exact against the oracle."""
    p = synth.Problem(2048, 2048, 1024, dtype="i8", layoutA="row", layoutB="col", seed=44, distA="int8",
                      distB="int8")
    A, B = to_dev(p.A), to_dev(p.B)
    D = torch.full((p.M * p.N,), -1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    before = ttc.ttc_launch_count()
    st = ttc.ttc_gemm_static_scratch(p.M, p.N, p.K, A.data_ptr(), p.lda, LAY[p.layoutA], B.data_ptr(), p.ldb,
                                     LAY[p.layoutB], None, p.N, D.data_ptr(), p.N, 1.0, 0.0, None, 0,
                                     ttc.DTYPE["i8"], s)
    assert st == 0, ttc.STATUS.get(st, st)
    assert ttc.ttc_get_device_error(s) == 0
    assert ttc.ttc_launch_count() - before == 2
    r, _ = oracle.gemm_full(p, alpha=1.0, beta=0.0)
    assert np.array_equal(D.cpu().numpy().reshape(p.M, p.N).astype(np.int64), r.astype(np.int64))
