"""GPU parity of ttc_transpose against the oracle's element-by-element
definition (bit-exact: the kernel moves bit patterns)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_tensor_core_02_gb300 as ttc

pytestmark = pytest.mark.gpu

TORCH_OF = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}
SIGNED_OF = {1: np.uint8, 2: np.int16, 4: np.int32, 8: np.int64}


def upload(a, eb):
    return torch.from_numpy(np.ascontiguousarray(a).view(SIGNED_OF[eb])).cuda()


def run(src_np, rows, cols, lds, ldd, eb):
    """Destination starts as all-ones bit patterns, so unwritten padding shows."""
    src = upload(src_np, eb)
    ones = np.full(max(cols * ldd, 1), np.iinfo(synth.ELEM_DTYPE[eb]).max, dtype=synth.ELEM_DTYPE[eb])
    dst = upload(ones, eb)
    st = ttc.ttc_transpose(rows, cols, src.data_ptr(), lds, dst.data_ptr(), ldd, eb,
                           torch.cuda.current_stream().cuda_stream)
    assert st == 0, ttc.ttc_status_string(st)
    assert ttc.ttc_get_device_error(None) == 0
    return dst.cpu().numpy().view(synth.ELEM_DTYPE[eb])


SHAPES = [(1, 1), (64, 64), (63, 65), (65, 63), (130, 1), (1, 300), (257, 131), (512, 384), (1000, 777)]


def pitch(n, eb, mode):
    """'odd': pitches that break 16-byte alignment (per-element path);
    'aligned': rounded up to 16 bytes plus one more 16-byte step (vector path)."""
    if mode == "odd":
        return n + (n % 3) + 1
    v = 16 // eb
    return -(-n // v) * v + v


@pytest.mark.parametrize("mode", ["odd", "aligned"])
@pytest.mark.parametrize("eb", [1, 2, 4, 8])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_transpose_matches_oracle(rows, cols, eb, mode):
    lds, ldd = pitch(cols, eb, mode), pitch(rows, eb, mode)
    src = synth.transpose_input(rows, cols, eb, seed=rows * 7919 + cols * 31 + eb, lds=lds)
    got = run(src, rows, cols, lds, ldd, eb).reshape(cols, ldd)
    want = oracle.transpose(src, rows, cols, lds, ldd).reshape(cols, ldd)
    assert np.array_equal(got[:, :rows], want[:, :rows])
    # the pitch padding of the destination is not written
    pad = got[:, rows:]
    assert (pad == np.iinfo(synth.ELEM_DTYPE[eb]).max).all()


@pytest.mark.parametrize("name", sorted(synth.TRANSPOSE_WORKLOADS))
def test_transpose_full_size_sampled_windows(name):
    """Bench-sized problem in the bench's launch configuration: compare 64 x 64
    source windows (random ones, plus the four corners) with the oracle's
    transpose of the same window."""
    w = synth.TRANSPOSE_WORKLOADS[name]
    rows, cols, eb = w["rows"], w["cols"], w["elem_bytes"]
    src = synth.transpose_input(rows, cols, eb, seed=w["seed"])
    got = run(src, rows, cols, cols, rows, eb).reshape(cols, rows)
    s2 = src.reshape(rows, cols)
    rng = np.random.default_rng(5)
    corners = [(0, 0), (0, cols - 64), (rows - 64, 0), (rows - 64, cols - 64)]
    picks = corners + [(int(rng.integers(0, rows - 64)), int(rng.integers(0, cols - 64))) for _ in range(12)]
    for r0, c0 in picks:
        win = np.ascontiguousarray(s2[r0:r0 + 64, c0:c0 + 64]).ravel()
        want = oracle.transpose(win, 64, 64, 64, 64).reshape(64, 64)
        assert np.array_equal(got[c0:c0 + 64, r0:r0 + 64], want), (r0, c0)
    # every element, by a property: transposing back gives the source
    back = torch.empty(rows * cols, dtype=TORCH_OF[eb], device="cuda")
    g = upload(got.ravel(), eb)
    assert ttc.ttc_transpose(cols, rows, g.data_ptr(), rows, back.data_ptr(), cols, eb, None) == 0
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy().view(synth.ELEM_DTYPE[eb]), src)


def test_transpose_launch_is_counted():
    n0 = ttc.ttc_launch_count()
    src = synth.transpose_input(96, 80, 2, seed=3)
    run(src, 96, 80, 80, 96, 2)
    assert ttc.ttc_launch_count() == n0 + 1
