"""Pins of the convolution oracle (CPU): a library convolution in float64, the
1 x 1 case as a matrix product, an all-ones closed form, the epilogue terms and
the output extents."""
import numpy as np
import pytest
import torch

import oracle
import synth

CASES = [
    # N, H, W, C, K, R, S, pad, stride, dil
    (1, 5, 5, 3, 4, 3, 3, (1, 1), (1, 1), (1, 1)),
    (2, 7, 6, 5, 3, 3, 3, (1, 1), (2, 2), (1, 1)),
    (1, 9, 8, 4, 2, 3, 3, (2, 2), (1, 1), (2, 2)),
    (2, 6, 7, 3, 5, 2, 3, (1, 0), (1, 2), (1, 1)),
    (1, 4, 4, 2, 3, 4, 4, (0, 0), (1, 1), (1, 1)),
    (1, 3, 5, 8, 2, 1, 3, (0, 2), (3, 1), (1, 2)),
]


def logical(cp):
    x = oracle.decode(cp.X, cp.dtype).reshape(cp.N, cp.H, cp.W, cp.C)
    w = oracle.decode(cp.Wt, cp.dtype).reshape(cp.K, cp.R, cp.S, cp.C)
    return x, w


def torch_conv(cp):
    x, w = logical(cp)
    y = torch.nn.functional.conv2d(torch.from_numpy(x).permute(0, 3, 1, 2), torch.from_numpy(w).permute(0, 3, 1, 2),
                                   stride=cp.stride, padding=cp.pad, dilation=cp.dil)
    return y.permute(0, 2, 3, 1).reshape(-1, cp.K).numpy()


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_conv_matches_library_conv2d_in_float64(case, dtype):
    N, H, W, C, K, R, S, pad, stride, dil = case
    cp = synth.ConvProblem(N, H, W, C, K, R, S, pad, stride, dil, dtype=dtype, seed=sum(case[:7]))
    r, sabs = oracle.conv_full(cp)
    want = torch_conv(cp)
    assert r.shape == want.shape
    assert np.allclose(r, want, rtol=1e-12, atol=1e-12)
    assert (sabs >= np.abs(r) - 1e-12).all()


def test_conv_1x1_is_a_matrix_product():
    cp = synth.ConvProblem(2, 6, 5, 16, 7, 1, 1, dtype="bf16", seed=9)
    x, w = logical(cp)
    r, _ = oracle.conv_full(cp)
    assert np.allclose(r, x.reshape(-1, cp.C) @ w.reshape(cp.K, cp.C).T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("case", CASES)
def test_conv_all_ones_counts_the_taps_inside_the_input(case):
    N, H, W, C, K, R, S, pad, stride, dil = case
    cp = synth.ConvProblem(N, H, W, C, K, R, S, pad, stride, dil, dtype="bf16", seed=1)
    cp.X = synth.store(np.ones(cp.X.size), "bf16")
    cp.Wt = synth.store(np.ones(cp.Wt.size), "bf16")
    r, sabs = oracle.conv_full(cp)
    for m in range(cp.M):
        p, q = (m // cp.Q) % cp.P, m % cp.Q
        rows = sum(1 for i in range(R) if 0 <= p * stride[0] - pad[0] + i * dil[0] < H)
        cols = sum(1 for j in range(S) if 0 <= q * stride[1] - pad[1] + j * dil[1] < W)
        assert (r[m] == C * rows * cols).all() and (sabs[m] == C * rows * cols).all()


def test_conv_epilogue_terms():
    cp = synth.ConvProblem(2, 5, 6, 4, 6, 3, 3, (1, 1), (1, 1), (1, 1), dtype="bf16", seed=4, with_c=True,
                           dist_bias="uniform")
    base, _ = oracle.conv_full(cp, use_bias=False)
    c = oracle.decode(cp.Cm, "bf16").reshape(cp.M, cp.K)
    r, _ = oracle.conv_full(cp, alpha=0.5, beta=2.0, act="relu")
    want = np.maximum(0.5 * base + 2.0 * c + cp.bias.astype(np.float64)[None, :], 0.0)
    assert np.allclose(r, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n,pad,dil,taps,stride", [(56, 1, 1, 3, 1), (56, 1, 1, 3, 2), (7, 0, 1, 7, 1),
                                                   (9, 2, 2, 3, 1), (5, 0, 3, 3, 2), (4, 0, 1, 5, 1)])
def test_conv_output_extent_matches_library_shapes(n, pad, dil, taps, stride):
    got = oracle.conv_out_extent(n, pad, dil, taps, stride)
    if n + 2 * pad < dil * (taps - 1) + 1:
        assert got == 0
        return
    y = torch.nn.functional.conv2d(torch.zeros(1, 1, n, 1), torch.zeros(1, 1, taps, 1), stride=(stride, 1),
                                   padding=(pad, 0), dilation=(dil, 1))
    assert got == y.shape[2] == synth.conv_out_extent(n, pad, dil, taps, stride)
