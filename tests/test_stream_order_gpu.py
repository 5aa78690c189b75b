"""Dependent calls back to back on one stream, and replayed from a CUDA graph.

The GEMM, convolution and matrix-vector kernels are launched with
programmatic dependent launch: a kernel may begin its prologue while the
kernel before it on the stream is finishing, and touches global memory only
once that kernel has completed.  These tests chain calls whose operands
depend on one another (read after write, write after read, write after
write) with no synchronisation between them, with programmatic launch on and
off, and replay the same chain from a CUDA graph.  Each result must equal,
bit for bit, what the same call gives when run alone (the plans and kernels
are deterministic; split-K partial sums are added in a fixed order), and two
of them are also checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_tensor_core_02_gb300 as ttc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_tensor_core_02_gb300 import _build
    _build.build()
    ttc.load()
    yield
    ttc.ttc_set_knob("pdl", 0)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _operands(seed):
    """bf16 operands of the chain, drawn with the shared generator."""
    st = synth.Stream(seed)

    def mat(rows, cols, col_major=False):
        v = synth.store(synth.draw(st, rows * cols, "uniform"), "bf16").reshape(rows, cols)
        t = torch.from_numpy(v.view(np.int16).copy()).cuda().view(torch.bfloat16)
        # a column-major rows x cols matrix is the transposed view of a row-major cols x rows one
        return t.t().contiguous().t() if col_major else t

    return dict(X=mat(2048, 128), W1=mat(128, 2048, True), W2=mat(2048, 64, True),
                Y=mat(2048, 128), W3=mat(128, 2048, True), x=mat(2048, 1, True), W5=mat(64, 256, True))


def _chain(o, H, E, v, F):
    """Five calls, no synchronisation between them:
    H = X W1 (CTA-pair kernel); E = H W2 (split-K over a cluster, reads H);
    H = Y W3 (pair kernel, overwrites the H that E's call read); v = H x
    (matrix-vector kernel, reads the new H); F = E W5 (single-CTA kernel,
    reads E)."""
    H.fill_(float("nan"))
    E.fill_(float("nan"))
    ttc.gemm(o["X"], o["W1"], out=H)
    ttc.gemm(H, o["W2"], out=E)
    ttc.gemm(o["Y"], o["W3"], out=H)
    ttc.gemm(H, o["x"], out=v)
    ttc.gemm(E, o["W5"], out=F)


def _alone(o):
    """The same calls one at a time, synchronising after each."""
    out = {}

    def one(a, b):
        d = torch.empty(a.shape[0], b.shape[1], dtype=torch.bfloat16, device="cuda")
        ttc.gemm(a, b, out=d)
        torch.cuda.synchronize()
        return d

    H1 = one(o["X"], o["W1"])
    out["E"] = one(H1, o["W2"])
    out["H"] = one(o["Y"], o["W3"])
    out["v"] = one(out["H"], o["x"])
    out["F"] = one(out["E"], o["W5"])
    out["H1"] = H1
    return out


def _buffers():
    mk = lambda r, c: torch.empty(r, c, dtype=torch.bfloat16, device="cuda")
    return mk(2048, 2048), mk(2048, 64), mk(2048, 1), mk(2048, 256)


def _same(got, ref, name):
    g, r = _bits(got), _bits(ref)
    assert np.array_equal(g, r), f"{name}: {np.count_nonzero(g != r)} of {g.size} elements differ"


def _oracle_check(a, b, d):
    """d = a b within the oracle's tolerance (a row-major, b column-major, bf16)."""
    A = _bits(a.contiguous())
    B = _bits(b.t().contiguous()).T
    p = synth.Problem.from_logical(A, B, dtype="bf16", layoutA="row", layoutB="col")
    r, sabs = oracle.gemm_full(p, alpha=1.0, beta=0.0, act="none", use_bias=False)
    ok, worst, w = oracle.check_float(oracle.decode(_bits(d).ravel(), "bf16"), r.ravel(), sabs.ravel(), "bf16")
    assert ok, f"worst error ratio {worst:.3f} at flat index {w}"


@pytest.mark.parametrize("pdl_off", [0, 1])
def test_dependent_calls_back_to_back(pdl_off):
    assert ttc.ttc_set_knob("pdl", pdl_off) == 0
    try:
        o = _operands(41)
        ref = _alone(o)
        H, E, v, F = _buffers()
        for _ in range(3):
            _chain(o, H, E, v, F)
        assert ttc.ttc_get_device_error() == 0
        _same(E, ref["E"], "E (read after write)")
        _same(H, ref["H"], "H (write after read and write)")
        _same(v, ref["v"], "v (matrix-vector, read after write)")
        _same(F, ref["F"], "F (read after write)")
        if pdl_off == 0:
            _oracle_check(ref["H1"], o["W2"], ref["E"])
            _oracle_check(ref["H"], o["x"], ref["v"])
    finally:
        ttc.ttc_set_knob("pdl", 0)


def test_chain_replayed_from_cuda_graph():
    o = _operands(42)
    ref = _alone(o)
    H, E, v, F = _buffers()
    _chain(o, H, E, v, F)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _chain(o, H, E, v, F)
    for _ in range(2):
        H.zero_()
        v.zero_()
        g.replay()
        torch.cuda.synchronize()
        _same(E, ref["E"], "E")
        _same(H, ref["H"], "H")
        _same(v, ref["v"], "v")
        _same(F, ref["F"], "F")
    # new operand values in the same buffers: the replay computes with them
    o2 = _operands(43)
    for k in ("X", "Y"):
        o[k].copy_(o2[k])
    ref2 = _alone(dict(o))
    g.replay()
    torch.cuda.synchronize()
    _same(E, ref2["E"], "E after new inputs")
    _same(v, ref2["v"], "v after new inputs")
    assert ttc.ttc_get_device_error() == 0
