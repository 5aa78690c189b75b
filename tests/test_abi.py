"""CPU-side checks of the C ABI: the library builds and loads, exports every
symbol include/ttc.h declares, and rejects bad arguments before touching a GPU."""
import os
import re

import pytest

import tiled_tensor_core_02_gb300 as ttc
from tiled_tensor_core_02_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ttc.load()


def declared_symbols():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(ttc_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert names, "no declarations found"
    assert names == set(ttc.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in ttc.STATUS.items():
        assert ttc.ttc_status_string(code) == name


def test_knobs_validate(lib):
    assert ttc.ttc_set_knob("tile_n", 128) == 0
    assert ttc.ttc_set_knob("tile_n", 100) == 1
    assert ttc.ttc_set_knob("tile_n", 0) == 0
    assert ttc.ttc_set_knob("inject_stall", 2) == 1
    assert ttc.ttc_set_knob(99, 0) == 1
    assert ttc.ttc_set_knob("gemv", 1) == 0 and ttc.ttc_set_knob("gemv", 2) == 1
    assert ttc.ttc_set_knob("gemv", 0) == 0
    assert ttc.ttc_set_knob("conv_halo", 2) == 0 and ttc.ttc_set_knob("conv_halo", 3) == 1
    assert ttc.ttc_set_knob("conv_halo", 0) == 0
    assert ttc.ttc_set_knob("pair_tail", 1) == 0 and ttc.ttc_set_knob("pair_tail", 2) == 1
    assert ttc.ttc_set_knob("pair_tail", 0) == 0
    assert ttc.ttc_set_knob("pdl", 1) == 0 and ttc.ttc_set_knob("pdl", 2) == 1
    assert ttc.ttc_set_knob("pdl", 0) == 0


BF16 = ttc.DTYPE["bf16"]
I8 = ttc.DTYPE["i8"]
R, C = ttc.ROW_MAJOR, ttc.COL_MAJOR
P = 1 << 20  # a fake, never-dereferenced address: these calls must fail before any GPU work


def call(M=64, N=64, K=64, A=P, lda=None, la=R, B=P, ldb=None, lb=C, Cp=None, ldc=None, D=P * 2,
         ldd=None, alpha=1.0, beta=0.0, bias=None, act=0, dtype=BF16):
    lda = (K if la == R else M) if lda is None else lda
    ldb = (N if lb == R else K) if ldb is None else ldb
    ldc = N if ldc is None else ldc
    ldd = N if ldd is None else ldd
    return ttc.ttc_gemm(M, N, K, A, lda, la, B, ldb, lb, Cp, ldc, D, ldd, alpha, beta, bias, act,
                        dtype, None)


@pytest.mark.parametrize("kw", [
    dict(M=-1), dict(N=-2), dict(K=-3),
    dict(la=5), dict(lb=7), dict(act=9), dict(dtype=9),
    dict(lda=63), dict(la=C, lda=63), dict(ldb=63), dict(lb=R, ldb=63), dict(ldd=63),
    dict(A=None), dict(B=None), dict(D=None),
    dict(beta=1.0, Cp=None), dict(beta=1.0, Cp=P * 4, ldc=63),
    dict(beta=1.0, Cp=P * 2 + 2, D=P * 2),       # partial overlap of C and D
    dict(beta=1.0, Cp=P * 2, ldc=96, D=P * 2),    # same base, different pitch
])
def test_invalid_arguments(lib, kw):
    assert call(**kw) == 1


@pytest.mark.parametrize("kw", [
    dict(dtype=I8, bias=P), dict(dtype=I8, act=1), dict(dtype=I8, alpha=2.0),
    dict(dtype=I8, beta=0.5, Cp=P * 4),
    dict(M=1 << 31),
])
def test_unsupported_combinations(lib, kw):
    assert call(**kw) == 2


def test_empty_problems_are_noops(lib):
    assert call(M=0) == 0
    assert call(N=0) == 0
    assert call(M=0, A=None, B=None, D=None) == 0


def test_workspace_size_query(lib):
    # aligned operands need nothing; an odd pitch needs one padded copy
    assert ttc.ttc_gemm_workspace_size(64, 64, 64, P, 64, R, P, 64, C, BF16) == 0
    # A row-major 4099 x 1023 and B column-major 1023 x 3001, tight pitches of
    # 2046 bytes: copies of 4099 and 3001 rows of 1024 elements
    n = ttc.ttc_gemm_workspace_size(4099, 3001, 1023, P, 1023, R, P, 1023, C, BF16)
    r256 = lambda b: (b + 255) // 256 * 256
    assert n == r256(4099 * 1024 * 2) + r256(3001 * 1024 * 2)
    # int8: pitch must be a 16-byte multiple
    assert ttc.ttc_gemm_workspace_size(64, 64, 64, P, 64, R, P, 64, C, I8) == 0
    assert ttc.ttc_gemm_workspace_size(64, 64, 72, P, 72, R, P, 72, C, I8) == 2 * r256(64 * 80)
    # misaligned base
    assert ttc.ttc_gemm_workspace_size(64, 64, 64, P + 2, 64, R, P, 64, C, BF16) > 0
    # empty or invalid problems
    assert ttc.ttc_gemm_workspace_size(0, 64, 64, P, 63, R, P, 64, C, BF16) == 0
    assert ttc.ttc_gemm_workspace_size(64, 64, 64, P, 63, 9, P, 64, C, BF16) == 0


def test_staged_workspace_size_query(lib):
    """The staged size adds an aligned copy of an int32 D (pitch rounded to 16
    bytes, size to 256) after the operand repack, only when D's rows cannot
    take TMA stores; 16-bit outputs, matrix-vector shapes and invalid
    arguments need nothing beyond the repack."""
    r256 = lambda b: (b + 255) // 256 * 256
    ab = ttc.ttc_gemm_workspace_size(4099, 3001, 1023, P, 1023, R, P, 1023, C, BF16)
    staged = ttc.ttc_gemm_workspace_size_staged
    # bf16 D at a pitch of 3001 elements: the epilogue writes such rows itself
    assert staged(4099, 3001, 1023, P, 1023, R, P, 1023, C, P, 3001, BF16) == ab
    assert staged(4099, 3001, 1023, P, 1023, R, P, 1023, C, P, 3008, BF16) == ab
    assert staged(64, 64, 64, P, 64, R, P, 64, C, P + 2, 64, BF16) == 0
    # int8: int32 D with a pitch of 203 elements (812 bytes); the copy's pitch
    # is N rounded to 16 bytes (200)
    assert staged(300, 200, 64, P, 64, R, P, 64, C, P, 203, I8) == r256(300 * 200 * 4)
    # matrix-vector shapes run without a workspace
    assert staged(1, 4096, 4096, P, 4096, R, P, 4096, C, P, 4096, BF16) == 0
    assert staged(4096, 1, 4096, P, 4096, R, P, 4096, C, P, 1, BF16) == 0
    # empty or invalid problems
    assert staged(0, 64, 64, P, 64, R, P, 64, C, P, 64, BF16) == 0
    assert staged(64, 64, 64, P, 64, R, P, 64, C, P, 63, BF16) == 0
    assert staged(64, 64, 64, P, 64, 9, P, 64, C, P, 64, BF16) == 0


def test_int8_pair_path_workspace_size(lib):
    """int8 problems of at least 64 tiles of 256 x 256 whose operands TMA can
    read and whose int32 D it can write ask for fp16 copies of A and B (rows
    padded to 16 elements, each copy rounded to 256 bytes); smaller ones, and
    any with the knob at 2, need only what the single-CTA path needs."""
    r256 = lambda b: (b + 255) // 256 * 256
    staged = ttc.ttc_gemm_workspace_size_staged
    # 8192^3, A row-major, B column-major: two 8192 x 8192 fp16 copies
    assert staged(8192, 8192, 8192, P, 8192, R, P, 8192, C, P, 8192, I8) == 2 * 8192 * 8192 * 2
    # K = 1000 pads each row to 1008 elements; B row-major: K rows of N
    assert staged(2048, 3000, 1000, P, 1008, R, P, 3008, R, P, 3000, I8) == \
        r256(2048 * 1008 * 2) + r256(1000 * 3008 * 2)
    # 36 tiles: below the threshold, and the pitch-only query never changes
    assert staged(1536, 1536, 4096, P, 4096, R, P, 4096, C, P, 1536, I8) == 0
    assert ttc.ttc_gemm_workspace_size(8192, 8192, 8192, P, 8192, R, P, 8192, C, I8) == 0
    # an int32 D that TMA cannot write keeps the single-CTA path (and its aligned
    # copy of D, whose pitch is N rounded to 16 bytes)
    assert staged(8192, 8192, 8192, P, 8192, R, P, 8192, C, P, 8194, I8) == r256(8192 * 8192 * 4)
    try:
        assert ttc.ttc_set_knob("i8_wide", 1) == 0
        assert staged(1536, 1536, 4096, P, 4096, R, P, 4096, C, P, 1536, I8) == 2 * r256(1536 * 4096 * 2)
        assert ttc.ttc_set_knob("i8_wide", 2) == 0
        assert staged(8192, 8192, 8192, P, 8192, R, P, 8192, C, P, 8192, I8) == 0
        assert ttc.ttc_set_knob("i8_wide", 3) == 1
    finally:
        ttc.ttc_set_knob("i8_wide", 0)


def test_static_scratch_rejects_oversized_problems(lib):
    # 4099 x 8192 bf16 with an odd pitch needs ~64 MiB of repacked A: beyond the
    # fixed 16 MiB, refused before any device work
    st = ttc.ttc_gemm_static_scratch(4099, 64, 8191, P, 8191, R, P, 8191, C, None, 64, P * 2, 64, 1.0, 0.0,
                                     None, 0, BF16, None)
    assert st == 5 and ttc.ttc_status_string(st) == "TTC_ERR_SCRATCH_TOO_SMALL"


def test_matrix_vector_problems_need_no_scratch(lib):
    """A matrix-vector problem takes a kernel that reads its operands with plain
    loads, whatever their pitch: the workspace query reports 0 for it and the
    no-allocation entry point does not refuse it, however large its B.
    M = 1, B column-major 4097 x 4096 with an odd pitch (33.6 MB of bf16)."""
    assert ttc.ttc_gemm_workspace_size(1, 4096, 4097, P, 4097, R, P, 4097, C, BF16) == 0
    assert ttc.ttc_gemm_workspace_size(1, 4096, 4097, P, 1, C, P, 4097, C, BF16) == 0  # 1 x K, lda free
    assert ttc.ttc_gemm_workspace_size(4096, 1, 4097, P, 4097, R, P, 4097, C, BF16) == 0
    # the same with B row-major (the outputs contiguous in B): the other
    # matrix-vector kernel, no scratch either
    assert ttc.ttc_gemm_workspace_size(1, 4095, 4097, P, 4097, R, P, 4095, R, BF16) == 0
    assert ttc.ttc_gemm_workspace_size(4095, 1, 4097, P, 4095, C, P, 4097, C, BF16) == 0
    # two output rows are a GEMM for the tensor-core kernels: repacked
    assert ttc.ttc_gemm_workspace_size(2, 4095, 4097, P, 4097, R, P, 4095, R, BF16) > 16 << 20
    st = ttc.ttc_gemm_static_scratch(1, 4096, 4097, P, 4097, R, P, 4097, C, None, 4096, P * 2, 4096, 1.0, 0.0,
                                     None, 0, BF16, None)
    assert st != 5  # not refused (without a GPU the call then stops at the CUDA device query)


def test_batched_validation(lib):
    sb = ttc.ttc_gemm_strided_batched
    # negative batch or stride; overlapping D batches; in-place C needs equal strides
    assert sb(-1, 64, 64, 64, P, 64, 0, R, P, 64, 0, C, None, 64, 0, P * 2, 64, 4096, 1.0, 0.0, None, 0, BF16, None) == 1
    assert sb(2, 64, 64, 64, P, 64, -5, R, P, 64, 0, C, None, 64, 0, P * 2, 64, 4096, 1.0, 0.0, None, 0, BF16, None) == 1
    assert sb(2, 64, 64, 64, P, 64, 0, R, P, 64, 0, C, None, 64, 0, P * 2, 64, 4000, 1.0, 0.0, None, 0, BF16, None) == 1
    assert sb(2, 64, 64, 64, P, 64, 0, R, P, 64, 0, C, P * 2, 64, 0, P * 2, 64, 4096, 1.0, 1.0, None, 0, BF16, None) == 1
    # empty batch is a no-op
    assert sb(0, 64, 64, 64, P, 64, 0, R, P, 64, 0, C, None, 64, 0, P * 2, 64, 4096, 1.0, 0.0, None, 0, BF16, None) == 0
    assert sb(70000, 64, 64, 64, P, 64, 0, R, P, 64, 0, C, None, 64, 0, P * 2, 64, 4096, 1.0, 0.0, None, 0, BF16, None) == 2


def test_transpose_validation(lib):
    t = ttc.ttc_transpose
    assert t(-1, 4, P, 4, P * 2, 4, 4, None) == 1
    assert t(4, 4, P, 4, P * 2, 4, 3, None) == 1            # element size
    assert t(4, 4, None, 4, P * 2, 4, 4, None) == 1         # null source
    assert t(4, 8, P, 7, P * 2, 4, 4, None) == 1            # lds < cols
    assert t(8, 4, P, 4, P * 2, 7, 4, None) == 1            # ldd < rows
    assert t(4, 4, P + 2, 4, P * 2, 4, 4, None) == 1        # misaligned for 4-byte elements
    assert t(64, 64, P, 64, P + 1024, 64, 4, None) == 1     # overlapping ranges
    assert t(0, 64, None, 64, None, 0, 4, None) == 0        # empty is a no-op
    assert t(64, 0, None, 0, None, 64, 2, None) == 0


def test_conv_validation(lib):
    cv = ttc.ttc_conv2d_fprop
    base = [2, 8, 8, 16, 32, 3, 3, 1, 1, 1, 1, 1, 1]
    ok_args = lambda dims: dims + [P, P * 4, None, 32, P * 8, 32, 1.0, 0.0, None, 0, BF16, None]
    a = list(base); a[7] = -1
    assert cv(*ok_args(a)) == 1                   # negative padding
    a = list(base); a[9] = 0
    assert cv(*ok_args(a)) == 1                   # zero stride
    a = list(base); a[5] = 11
    assert cv(*ok_args(a)) == 1                   # filter larger than the padded input
    assert cv(*(base + [P, P * 4, None, 32, P * 8, 31, 1.0, 0.0, None, 0, BF16, None])) == 1   # ldd < K
    assert cv(*(base + [P, P * 4, None, 32, None, 32, 1.0, 0.0, None, 0, BF16, None])) == 1     # no output
    assert cv(*(base + [P, P * 4, None, 32, P * 8, 32, 1.0, 1.0, None, 0, BF16, None])) == 1    # beta without C
    assert cv(*(base + [P + 1, P * 4, None, 32, P * 8, 32, 1.0, 0.0, None, 0, BF16, None])) == 1  # misaligned X
    assert cv(*(base + [P, P * 4, None, 32, P, 32, 1.0, 0.0, None, 0, BF16, None])) == 1        # D overlaps X
    assert cv(*(base + [P, P * 4, None, 32, P * 8, 32, 1.0, 0.0, None, 0, 2, None])) == 2       # int8
    a = list(base); a[0] = 0
    assert cv(*ok_args(a)) == 0                   # N = 0: no-op
