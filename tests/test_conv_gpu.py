"""GPU parity of ttc_conv2d_fprop (implicit-GEMM convolution) against the
oracle's per-element convolution, with the GEMM's float tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_tensor_core_02_gb300 as ttc
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


def run_conv(cp, alpha=1.0, beta=0.0, act="none", use_bias=True, ldd=None, x_offset=0, in_place=False, expect=0):
    ldd = cp.K if ldd is None else ldd
    X = to_dev(np.concatenate([np.zeros(x_offset, np.uint16), cp.X]))
    Wt = to_dev(cp.Wt)
    bias = to_dev(cp.bias) if (use_bias and cp.bias is not None) else None
    if in_place:
        D = to_dev(cp.Cm)
        Cm = D
    else:
        D = torch.full((max(cp.M * ldd, 1),), -1, dtype=torch.int16, device="cuda")
        Cm = to_dev(cp.Cm) if (beta != 0.0 and cp.Cm is not None) else None
    st = ttc.ttc_conv2d_fprop(*cp.dims(), X.data_ptr() + 2 * x_offset, Wt.data_ptr(),
                              Cm.data_ptr() if Cm is not None else None, cp.ldc if Cm is not None else cp.K,
                              D.data_ptr(), ldd, alpha, beta, bias.data_ptr() if bias is not None else None,
                              ttc.ACT[act], ttc.DTYPE[cp.dtype], torch.cuda.current_stream().cuda_stream)
    assert st == expect, ttc.ttc_status_string(st)
    torch.cuda.synchronize()
    assert ttc.ttc_get_device_error(None) == 0
    return D.cpu().numpy().view(np.uint16)


def check_full(cp, out, ldd=None, **kw):
    ldd = cp.K if ldd is None else ldd
    r, sabs = oracle.conv_full(cp, **kw)
    d = oracle.decode(out.reshape(-1)[:cp.M * ldd].reshape(cp.M, ldd)[:, :cp.K], cp.dtype)
    ok, worst, w = oracle.check_float(d.ravel(), r.ravel(), sabs.ravel(), cp.dtype)
    assert ok, f"worst error {worst:.3f} x tolerance at {np.unravel_index(w, d.shape)}"


SHAPES = [
    # N, H, W, C, K, R, S, pad, stride, dil
    (2, 9, 9, 64, 96, 3, 3, (1, 1), (1, 1), (1, 1)),       # vector path, ragged K
    (1, 14, 14, 128, 256, 3, 3, (1, 1), (2, 2), (1, 1)),   # strided
    (2, 8, 8, 256, 64, 1, 1, (0, 0), (1, 1), (1, 1)),      # 1 x 1
    (1, 32, 32, 3, 64, 7, 7, (3, 3), (2, 2), (1, 1)),      # first-layer shape, C = 3 (per-element path)
    (1, 17, 13, 16, 40, 3, 3, (2, 2), (1, 1), (2, 2)),     # dilated
    (3, 7, 11, 24, 70, 2, 3, (1, 0), (1, 2), (1, 1)),      # rectangular filter, asymmetric stride/pad
    (1, 5, 5, 8, 8, 5, 5, (0, 0), (1, 1), (1, 1)),         # one output pixel per image
    (4, 12, 12, 72, 136, 3, 3, (1, 1), (1, 1), (1, 1)),    # M, K and R S C all ragged vs the tiles
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_conv_matches_oracle(shape, dtype):
    N, H, W, C, K, R, S, pad, stride, dil = shape
    cp = synth.ConvProblem(N, H, W, C, K, R, S, pad, stride, dil, dtype=dtype, seed=sum(shape[:7]))
    check_full(cp, run_conv(cp))


@pytest.mark.parametrize("act", ["none", "relu", "gelu_tanh"])
def test_conv_epilogue(act):
    cp = synth.ConvProblem(2, 10, 10, 32, 48, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=7, with_c=True,
                           dist_bias="uniform")
    check_full(cp, run_conv(cp, alpha=0.75, beta=0.5, act=act), alpha=0.75, beta=0.5, act=act)


def test_conv_in_place_c_and_padded_output_pitch():
    cp = synth.ConvProblem(1, 9, 9, 16, 24, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=8, with_c=True)
    check_full(cp, run_conv(cp, beta=1.0, in_place=True, use_bias=False), beta=1.0, use_bias=False)
    out = run_conv(cp, ldd=40).reshape(cp.M, 40)
    check_full(cp, out.ravel(), ldd=40)
    assert (out[:, cp.K:] == 0xFFFF).all()  # the pitch padding is not written


def test_conv_unaligned_input_takes_the_per_element_path():
    cp = synth.ConvProblem(2, 6, 6, 16, 32, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=9)
    check_full(cp, run_conv(cp, x_offset=1))


def test_conv_empty_and_degenerate():
    cp = synth.ConvProblem(1, 4, 4, 8, 8, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=10, with_c=True,
                           dist_bias="uniform")
    # C = 0 channels: a zero sum, the epilogue alone
    cp0 = synth.ConvProblem(1, 4, 4, 0, 8, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=10, with_c=True,
                            dist_bias="uniform")
    cp0.Cm, cp0.bias = cp.Cm, cp.bias
    check_full(cp0, run_conv(cp0, beta=1.0), beta=1.0)
    # N = 0 and K = 0 are no-ops
    assert ttc.ttc_conv2d_fprop(0, 4, 4, 8, 8, 3, 3, 1, 1, 1, 1, 1, 1, None, None, None, 8, None, 8, 1.0, 0.0,
                                None, 0, ttc.DTYPE["bf16"], None) == 0
    assert ttc.ttc_conv2d_fprop(1, 4, 4, 8, 0, 3, 3, 1, 1, 1, 1, 1, 1, None, None, None, 1, None, 1, 1.0, 0.0,
                                None, 0, ttc.DTYPE["bf16"], None) == 0


@pytest.mark.parametrize("halo", [0, 2])
@pytest.mark.parametrize("name", sorted(synth.CONV_WORKLOADS))
def test_conv_full_size_sampled(name, halo):
    """The benchmark's convolution in its launch configuration (halo = 0: the
    planner's choice, the halo kernel; 2: im2col loads): sampled rows, columns
    and elements against the oracle."""
    spec = dict(synth.CONV_WORKLOADS[name])
    cp = synth.ConvProblem(**spec)
    ttc.ttc_set_knob("conv_halo", halo)
    try:
        out = run_conv(cp).reshape(cp.M, cp.K)
    finally:
        ttc.ttc_set_knob("conv_halo", 0)
    mm, kk = oracle.sample_indices(cp.M, cp.K, seed=spec["seed"], n_lines=4, n_elems=16384)
    r, sabs, _ = oracle.conv_elements(cp, mm, kk)
    d = oracle.decode(out[mm, kk], cp.dtype)
    ok, worst, w = oracle.check_float(d, r, sabs, cp.dtype)
    assert ok, f"worst error {worst:.3f} x tolerance at (m={mm[w]}, k={kk[w]})"


# Shapes the im2col-TMA CTA-pair path takes (C a multiple of 64): forced onto
# it (pair = 1) and onto the plain-load kernel (pair = 2), both against the oracle.
PAIR_SHAPES = [
    (2, 20, 20, 64, 128, 3, 3, (1, 1), (1, 1), (1, 1)),    # 800 pixels: ragged against 256-pixel tiles
    (3, 30, 28, 128, 256, 3, 3, (1, 1), (2, 2), (1, 1)),   # strided; tiles cross image boundaries
    (2, 17, 19, 64, 192, 5, 5, (2, 2), (1, 1), (2, 2)),    # dilated 5 x 5
    (3, 9, 31, 128, 320, 1, 3, (0, 1), (1, 2), (1, 1)),    # rectangular filter, ragged K
    (2, 7, 7, 256, 256, 3, 3, (0, 0), (1, 1), (1, 1)),     # no padding, 50 pixels: the odd CTA's rows all past M
    (4, 16, 16, 64, 128, 1, 1, (0, 0), (2, 2), (1, 1)),    # 1 x 1, stride 2
]


@pytest.fixture
def pair_knob():
    yield lambda v: ttc.ttc_set_knob("pair", v)
    ttc.ttc_set_knob("pair", 0)


@pytest.fixture
def halo_knob():
    yield lambda v: ttc.ttc_set_knob("conv_halo", v)
    ttc.ttc_set_knob("conv_halo", 0)


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("shape", PAIR_SHAPES)
def test_conv_im2col_pair_path_matches_oracle(shape, pair, pair_knob, halo_knob):
    N, H, W, C, K, R, S, pad, stride, dil = shape
    cp = synth.ConvProblem(N, H, W, C, K, R, S, pad, stride, dil, dtype="bf16", seed=sum(shape[:7]) + 100,
                           with_c=True, dist_bias="uniform")
    pair_knob(pair)
    halo_knob(2)
    check_full(cp, run_conv(cp, alpha=1.25, beta=0.5, act="relu"), alpha=1.25, beta=0.5, act="relu")


def test_conv_im2col_pair_path_f16(halo_knob):
    halo_knob(2)
    cp = synth.ConvProblem(2, 12, 12, 128, 256, 3, 3, (1, 1), (1, 1), (1, 1), dtype="f16", seed=77)
    check_full(cp, run_conv(cp))


# Unit-stride shapes the halo kernel takes (C a multiple of 64, K of 32): one
# box of padded input rows per 64-channel block feeds every filter tap.
HALO_SHAPES = [
    (2, 20, 20, 64, 128, 3, 3, (1, 1), (1, 1), (1, 1)),    # 4 position tiles per image, the last ragged
    (3, 9, 11, 64, 96, 3, 3, (1, 1), (1, 1), (1, 1)),      # odd N: the last pair's second image is absent
    (2, 17, 19, 128, 192, 5, 5, (2, 2), (1, 1), (2, 2)),   # dilated 5 x 5, a partial 256-wide channel block
    (1, 9, 31, 64, 320, 1, 3, (0, 1), (1, 1), (1, 1)),     # rectangular filter, one image, 3 channel blocks of 128
    (2, 7, 7, 256, 256, 3, 3, (0, 0), (1, 1), (1, 1)),     # no padding: 5 x 5 outputs
    (4, 16, 16, 64, 128, 1, 1, (0, 0), (1, 1), (1, 1)),    # 1 x 1: no dropped positions
    (2, 14, 14, 128, 384, 7, 7, (3, 3), (1, 1), (1, 1)),   # 7 x 7, 3 blocks of 128 output channels
    (5, 6, 40, 64, 64, 3, 1, (2, 0), (1, 1), (3, 1)),      # tall dilation, pad > 1, tiles spanning 4 rows
]


@pytest.mark.parametrize("shape", HALO_SHAPES)
def test_conv_halo_path_matches_oracle(shape, halo_knob):
    N, H, W, C, K, R, S, pad, stride, dil = shape
    cp = synth.ConvProblem(N, H, W, C, K, R, S, pad, stride, dil, dtype="bf16", seed=sum(shape[:7]) + 200,
                           with_c=True, dist_bias="uniform")
    halo_knob(1)
    check_full(cp, run_conv(cp, alpha=1.25, beta=0.5, act="relu"), alpha=1.25, beta=0.5, act="relu")


@pytest.mark.parametrize("tail", [0, 1], ids=["halves", "whole"])
@pytest.mark.parametrize("K", [256, 192])
def test_conv_halo_path_half_and_whole_tiles(K, tail, halo_knob):
    """Few tiles on many pairs: the default walk splits every tile into two
    halves of 128 output channels (K = 192: the second half only 64 wide);
    tail = 1 keeps whole tiles."""
    halo_knob(1)
    ttc.ttc_set_knob("pair_tail", tail)
    try:
        cp = synth.ConvProblem(3, 14, 15, 64, K, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=80 + K,
                               with_c=True, dist_bias="uniform")
        check_full(cp, run_conv(cp, alpha=0.5, beta=1.0, act="relu"), alpha=0.5, beta=1.0, act="relu")
    finally:
        ttc.ttc_set_knob("pair_tail", 0)


@pytest.mark.parametrize("act", ["none", "gelu_tanh"])
def test_conv_halo_path_f16_and_epilogue(act, halo_knob):
    halo_knob(1)
    cp = synth.ConvProblem(3, 12, 12, 128, 256, 3, 3, (1, 1), (1, 1), (1, 1), dtype="f16", seed=78)
    check_full(cp, run_conv(cp, act=act), act=act)


def test_conv_halo_path_in_place_c_and_padded_pitch(halo_knob):
    halo_knob(1)
    cp = synth.ConvProblem(3, 10, 10, 64, 96, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=79, with_c=True)
    check_full(cp, run_conv(cp, beta=1.0, in_place=True, use_bias=False), beta=1.0, use_bias=False)
    out = run_conv(cp, ldd=136).reshape(cp.M, 136)
    check_full(cp, out.ravel(), ldd=136)
    assert (out[:, cp.K:] == 0xFFFF).all()  # the pitch padding is not written


def test_conv_halo_declines_what_it_cannot_run(halo_knob):
    """Forced, the halo kernel still leaves strided, unaligned and too-wide
    problems to the other paths; the results stay right."""
    halo_knob(1)
    for shape, kw in [((1, 14, 14, 128, 256, 3, 3, (1, 1), (2, 2), (1, 1)), {}),     # stride 2
                      ((2, 6, 6, 64, 96, 3, 3, (1, 1), (1, 1), (1, 1)), dict(ldd=100)),  # ldd not a multiple of 8
                      ((1, 3, 300, 64, 64, 3, 3, (1, 1), (1, 1), (1, 1)), {}),       # padded row over 256 pixels
                      ((1, 8, 8, 64, 80, 3, 3, (1, 1), (1, 1), (1, 1)), {})]:        # K not a multiple of 32
        N, H, W, C, K, R, S, pad, stride, dil = shape
        cp = synth.ConvProblem(N, H, W, C, K, R, S, pad, stride, dil, dtype="bf16", seed=sum(shape[:7]))
        ldd = kw.get("ldd", K)
        check_full(cp, run_conv(cp, ldd=ldd), ldd=ldd)


def test_conv_halo_stalled_pipeline_times_out_and_context_survives(halo_knob):
    """The halo kernel's tensor-core issuer waits on a barrier nothing arrives
    at: the launch ends with TTC_ERR_TIMEOUT within the wait budget (the
    producers drain their halo and filter loads), and the context stays
    usable."""
    cp = synth.ConvProblem(2, 10, 10, 64, 128, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=81)
    halo_knob(1)
    ttc.ttc_set_knob("timeout_ns", 200_000_000)
    ttc.ttc_set_knob("inject_stall", 1)
    try:
        X, Wt = to_dev(cp.X), to_dev(cp.Wt)
        D = torch.zeros(cp.M * cp.K, dtype=torch.int16, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        st = ttc.ttc_conv2d_fprop(*cp.dims(), X.data_ptr(), Wt.data_ptr(), None, cp.K, D.data_ptr(), cp.K, 1.0,
                                  0.0, None, 0, ttc.DTYPE["bf16"], s)
        assert st == 0
        assert ttc.ttc_get_device_error(s) == 4
    finally:
        ttc.ttc_set_knob("inject_stall", 0)
        ttc.ttc_set_knob("timeout_ns", 0)
    assert ttc.ttc_get_device_error(None) == 0
    check_full(cp, run_conv(cp))
