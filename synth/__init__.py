"""Seeded synthetic inputs for the tiled GEMM D = act(alpha*A*B + beta*C + bias).

This module is the one piece of code that both the CPU oracle's tests and the
CUDA path's tests/benchmark use.  It holds no GEMM arithmetic: it only draws
numbers and stores them in the requested element type and memory layout.

Generator
---------
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) used as a counter-based generator: draw number
``i`` (0-based) of a stream with seed ``s`` is ``mix64(s + (i + 1) * GAMMA)``
with GAMMA = 0x9E3779B97F4A7C15 and mix64 the published finaliser
(xor-shift 30 / multiply / xor-shift 27 / multiply / xor-shift 31).

One stream per problem, seeded with the problem's seed.  The operands are drawn
in the order A, B, C, bias, each in *logical row-major order* (A is M x K, B is
K x N, C is M x N, bias has N entries) whatever its storage layout, so the four
row/column-major combinations of one shape see the same logical matrices.

Value mappings (per draw ``x``):
  * uniform[-1, 1):   2 * ((x >> 40) * 2**-24) - 1
  * normal(0, sigma): Box-Muller over two consecutive draws x1, x2:
        u1 = ((x1 >> 11) + 1) * 2**-53   (in (0, 1])
        u2 = (x2 >> 11) * 2**-53         (in [0, 1))
        z  = sigma * sqrt(-2 ln u1) * cos(2 pi u2)
    (sigma is the standard deviation); a normal element consumes two draws.
  * int8 uniform over [-128, 127]: the top byte of x read as a signed byte.

Floating values are rounded to float32 (round-to-nearest-even), then to the
storage type (fp16 by numpy's RNE cast, bf16 by RNE on the float32 bits).
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

DTYPES = ("f16", "bf16", "i8", "f32", "i32")


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the SplitMix64 stream ``seed`` (uint64)."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * GAMMA
        z = (x ^ (x >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


class Stream:
    """Sequential reader over one SplitMix64 stream."""

    def __init__(self, seed: int):
        self.seed = int(seed)
        self.pos = 0

    def raw(self, count: int) -> np.ndarray:
        out = np.empty(count, dtype=np.uint64)
        for lo in range(0, count, _CHUNK):
            n = min(_CHUNK, count - lo)
            out[lo:lo + n] = splitmix64(self.seed, self.pos + lo, n)
        self.pos += count
        return out

    def uniform(self, count: int) -> np.ndarray:
        """float64 values in [-1, 1)."""
        out = np.empty(count, dtype=np.float64)
        for lo in range(0, count, _CHUNK):
            n = min(_CHUNK, count - lo)
            x = splitmix64(self.seed, self.pos + lo, n)
            out[lo:lo + n] = 2.0 * ((x >> np.uint64(40)).astype(np.float64) * 2.0**-24) - 1.0
        self.pos += count
        return out

    def normal(self, count: int, sigma: float) -> np.ndarray:
        """float64 values ~ N(0, sigma^2); two draws per value."""
        out = np.empty(count, dtype=np.float64)
        for lo in range(0, count, _CHUNK):
            n = min(_CHUNK, count - lo)
            x = splitmix64(self.seed, self.pos + 2 * lo, 2 * n)
            x1 = x[0::2]
            x2 = x[1::2]
            u1 = ((x1 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53
            u2 = (x2 >> np.uint64(11)).astype(np.float64) * 2.0**-53
            out[lo:lo + n] = sigma * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        self.pos += 2 * count
        return out

    def int8(self, count: int) -> np.ndarray:
        out = np.empty(count, dtype=np.int8)
        for lo in range(0, count, _CHUNK):
            n = min(_CHUNK, count - lo)
            x = splitmix64(self.seed, self.pos + lo, n)
            out[lo:lo + n] = (x >> np.uint64(56)).astype(np.uint8).view(np.int8)
        self.pos += count
        return out


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round-to-nearest-even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    nan = np.isnan(x32)
    r = r.astype(np.uint16)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def store(values: np.ndarray, dtype: str) -> np.ndarray:
    """Round logical float64 (or int8) values to the storage type.

    Returns uint16 bit patterns for f16/bf16, int8 for i8, float32 for f32."""
    if dtype == "i8":
        return np.asarray(values, dtype=np.int8)
    if dtype == "i32":
        return np.asarray(values, dtype=np.int32)
    x32 = np.asarray(values, dtype=np.float32)
    if dtype == "f32":
        return x32
    if dtype == "f16":
        return x32.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(dtype)


def to_layout(logical: np.ndarray, layout: str, ld: int | None = None) -> tuple[np.ndarray, int]:
    """Place a logical rows x cols matrix in memory.

    layout 'row': element (i, j) at i*ld + j (ld >= cols);
    layout 'col': element (i, j) at i + j*ld (ld >= rows).
    Padding elements are zero.  Returns (flat buffer, ld)."""
    rows, cols = logical.shape
    if layout == "row":
        ld = cols if ld is None else ld
        assert ld >= cols
        buf = np.zeros(max(rows * ld, 0) if rows else 0, dtype=logical.dtype)
        if rows and cols:
            buf.reshape(rows, ld)[:, :cols] = logical
        return buf, ld
    if layout == "col":
        ld = rows if ld is None else ld
        assert ld >= rows
        buf = np.zeros(max(cols * ld, 0) if cols else 0, dtype=logical.dtype)
        if rows and cols:
            buf.reshape(cols, ld)[:, :rows] = logical.T
        return buf, ld
    raise ValueError(layout)


def from_layout(buf: np.ndarray, rows: int, cols: int, layout: str, ld: int) -> np.ndarray:
    """Inverse of to_layout: the logical rows x cols view (a copy)."""
    if rows == 0 or cols == 0:
        return np.zeros((rows, cols), dtype=buf.dtype)
    if layout == "row":
        return np.array(buf[: rows * ld].reshape(rows, ld)[:, :cols])
    return np.array(buf[: cols * ld].reshape(cols, ld)[:, :rows].T)


def draw(stream: Stream, count: int, dist: str) -> np.ndarray:
    """dist: 'uniform', 'normal:<sigma>' or 'int8'."""
    if dist == "uniform":
        return stream.uniform(count)
    if dist.startswith("normal:"):
        return stream.normal(count, float(dist.split(":", 1)[1]))
    if dist == "int8":
        return stream.int8(count)
    raise ValueError(dist)


class Problem:
    """One synthetic GEMM problem: logical operands, stored in their layouts.

    Attributes (numpy):
      A, B, C: flat storage buffers (bit patterns for f16/bf16), with lda/ldb/ldc;
      bias: float32[N] or None; the logical views A_log (M x K), B_log (K x N),
      C_log (M x N) as storage-typed arrays.
    """

    def __init__(self, M, N, K, dtype="bf16", layoutA="row", layoutB="col",
                 seed=0, distA="uniform", distB="uniform", distC=None,
                 dist_bias=None, lda=None, ldb=None, ldc=None):
        self.M, self.N, self.K = int(M), int(N), int(K)
        self.dtype = dtype
        self.layoutA, self.layoutB = layoutA, layoutB
        self.seed = seed
        st = Stream(seed)
        if dtype == "i8":
            cdtype = "i32"
        else:
            cdtype = dtype
        self.cdtype = cdtype
        a = store(draw(st, self.M * self.K, distA), dtype).reshape(self.M, self.K)
        b = store(draw(st, self.K * self.N, distB), dtype).reshape(self.K, self.N)
        self.A_log, self.B_log = a, b
        self.A, self.lda = to_layout(a, layoutA, lda)
        self.B, self.ldb = to_layout(b, layoutB, ldb)
        if distC is not None:
            if cdtype == "i32":
                c = draw(st, self.M * self.N, distC).astype(np.int32)
            else:
                c = store(draw(st, self.M * self.N, distC), cdtype)
            c = c.reshape(self.M, self.N)
            self.C_log = c
            self.C, self.ldc = to_layout(c, "row", ldc)
        else:
            self.C_log, self.C, self.ldc = None, None, (self.N if ldc is None else ldc)
        if dist_bias is not None:
            self.bias = draw(st, self.N, dist_bias).astype(np.float32)
        else:
            self.bias = None

    @classmethod
    def from_logical(cls, A_log, B_log, C_log=None, bias=None, dtype="bf16",
                     layoutA="row", layoutB="col", lda=None, ldb=None, ldc=None):
        """A problem from given storage-typed logical operands (no drawing)."""
        p = cls.__new__(cls)
        p.M, p.K = A_log.shape
        p.N = B_log.shape[1]
        assert B_log.shape[0] == p.K
        p.dtype = dtype
        p.cdtype = "i32" if dtype == "i8" else dtype
        p.layoutA, p.layoutB = layoutA, layoutB
        p.seed = None
        p.A_log, p.B_log = A_log, B_log
        p.A, p.lda = to_layout(A_log, layoutA, lda)
        p.B, p.ldb = to_layout(B_log, layoutB, ldb)
        if C_log is not None:
            p.C_log = C_log
            p.C, p.ldc = to_layout(C_log, "row", ldc)
        else:
            p.C_log, p.C, p.ldc = None, None, (p.N if ldc is None else ldc)
        p.bias = None if bias is None else np.asarray(bias, dtype=np.float32)
        return p


# The five workloads of the benchmark suite, by name.
WORKLOADS = {
    # fp16 256^3, A row-major, B column-major, alpha=1 beta=0, uniform[-1,1], seed 0
    "fp16_256": dict(M=256, N=256, K=256, dtype="f16", layoutA="row", layoutB="col", seed=0,
                     distA="uniform", distB="uniform", alpha=1.0, beta=0.0, act="none"),
    # bf16 4096^3, C bf16, alpha=1.5 beta=0.5, uniform[-1,1], seed 1
    "bf16_4096": dict(M=4096, N=4096, K=4096, dtype="bf16", layoutA="row", layoutB="col", seed=1,
                      distA="uniform", distB="uniform", distC="uniform", alpha=1.5, beta=0.5,
                      act="none"),
    # bf16 MLP projection 8192 x 14336 x 4096, A~N(0,1), B~N(0,0.02), bias~N(0,0.02), GELU(tanh)
    "bf16_mlp_8192x14336x4096": dict(M=8192, N=14336, K=4096, dtype="bf16", layoutA="row",
                                     layoutB="col", seed=2, distA="normal:1.0",
                                     distB="normal:0.02", dist_bias="normal:0.02", alpha=1.0,
                                     beta=0.0, act="gelu_tanh"),
    # int8 x int8 -> int32 8192^3, uniform integers in [-128, 127], seed 3
    "i8_8192": dict(M=8192, N=8192, K=8192, dtype="i8", layoutA="row", layoutB="col", seed=3,
                    distA="int8", distB="int8", alpha=1.0, beta=0.0, act="none"),
    # strided batched bf16: 32 independent 1024^3 GEMMs in one call, uniform[-1,1], seeds 5..36
    "bf16_batched_32x1024": dict(M=1024, N=1024, K=1024, dtype="bf16", layoutA="row", layoutB="col",
                                 seed=5, distA="uniform", distB="uniform", alpha=1.0, beta=0.0,
                                 act="none", batch=32),
    # int8 4096^3: a smaller case of the int8 recipe, for profiling
    "i8_4096": dict(M=4096, N=4096, K=4096, dtype="i8", layoutA="row", layoutB="col", seed=3,
                    distA="int8", distB="int8", alpha=1.0, beta=0.0, act="none"),
    # bf16 8192^3 (the headline throughput shape), same recipe as bf16_4096 but alpha=1 beta=0
    "bf16_8192": dict(M=8192, N=8192, K=8192, dtype="bf16", layoutA="row", layoutB="col", seed=1,
                      distA="uniform", distB="uniform", alpha=1.0, beta=0.0, act="none"),
}

# The ragged / skinny sweep: 4 shapes x 4 majorness combinations, alpha=beta=1, seed 4.
RAGGED_SHAPES = [(4099, 3001, 1023), (16, 8192, 8192), (8192, 24, 4096), (1, 4096, 4096)]
MAJORNESS = [("row", "row"), ("row", "col"), ("col", "row"), ("col", "col")]


def ragged_workload(M, N, K, la, lb):
    return dict(M=M, N=N, K=K, dtype="bf16", layoutA=la, layoutB=lb, seed=4, distA="uniform",
                distB="uniform", distC="uniform", alpha=1.0, beta=1.0, act="none")


def workload(name):
    """Workload dict by name: a WORKLOADS key, or ragged_<M>x<N>x<K>_<a><b> with
    a, b in {r, c} (row/column-major A and B) for the ragged sweep."""
    if name in WORKLOADS:
        return dict(WORKLOADS[name])
    if name.startswith("ragged_"):
        dims, lay = name[len("ragged_"):].split("_")
        M, N, K = (int(v) for v in dims.split("x"))
        full = {"r": "row", "c": "col"}
        return ragged_workload(M, N, K, full[lay[0]], full[lay[1]])
    raise KeyError(name)


def all_workload_names():
    names = list(WORKLOADS)
    for (M, N, K) in RAGGED_SHAPES:
        for la, lb in MAJORNESS:
            names.append(f"ragged_{M}x{N}x{K}_{la[0]}{lb[0]}")
    return names


def make(spec, **override):
    """Build the synth.Problem for a workload dict; returns (problem, alpha, beta, act).
    A batched workload returns the problem of batch 0 (see make_batch)."""
    s = dict(spec)
    s.update(override)
    s.pop("batch", None)
    alpha, beta, act = s.pop("alpha"), s.pop("beta"), s.pop("act")
    return Problem(**s), alpha, beta, act


def make_batch(spec):
    """The problems of a batched workload: batch b drawn from seed + b."""
    n = spec.get("batch", 1)
    return [make(spec, seed=spec["seed"] + b)[0] for b in range(n)]


# ---------------------------------------------------------------- transpose inputs

ELEM_DTYPE = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}

# Out-of-place transpose workloads: rows x cols source, element size in bytes.
# The CuTe transpose page runs its kernel on a float matrix and names no size;
# 16384 x 16384 fp32 (1 GiB each way) is well beyond the 129 MB L2.
TRANSPOSE_WORKLOADS = {
    "transpose_f32_16384": dict(rows=16384, cols=16384, elem_bytes=4, seed=21),
    "transpose_bf16_16384": dict(rows=16384, cols=16384, elem_bytes=2, seed=22),
    # the small case profiled with the full ncu section set (256 MiB each way)
    "transpose_f32_8192": dict(rows=8192, cols=8192, elem_bytes=4, seed=23),
}


def transpose_input(rows: int, cols: int, elem_bytes: int, seed: int, lds: int | None = None) -> np.ndarray:
    """rows x cols source of random bit patterns, row-major with pitch lds,
    as a flat unsigned array (padding filled with random bits too)."""
    lds = cols if lds is None else lds
    n = rows * lds if rows else 0
    raw = Stream(seed).raw(n)
    return raw.astype(ELEM_DTYPE[elem_bytes]) if elem_bytes < 8 else raw


# ---------------------------------------------------------------- convolution inputs

def conv_out_extent(n, pad, dil, taps, stride):
    """Output extent of one spatial mode (for sizing C only)."""
    span = n + 2 * pad - dil * (taps - 1) - 1
    return span // stride + 1 if span >= 0 else 0


class ConvProblem:
    """Inputs of one 2-D convolution: X (N, H, W, C) NHWC and Wt (K, R, S, C)
    KRSC, tightly packed, stored as fp16/bf16 bit patterns; optional C
    ((N P Q) x K row-major) and fp32 bias[K].  Draw order X, Wt, C, bias."""

    def __init__(self, N, H, W, C, K, R, S, pad=(0, 0), stride=(1, 1), dil=(1, 1), dtype="bf16", seed=0,
                 dist_x="uniform", dist_w="uniform", with_c=False, dist_bias=None):
        self.N, self.H, self.W, self.C, self.K, self.R, self.S = N, H, W, C, K, R, S
        self.pad, self.stride, self.dil = tuple(pad), tuple(stride), tuple(dil)
        self.dtype = dtype
        self.P = conv_out_extent(H, pad[0], dil[0], R, stride[0])
        self.Q = conv_out_extent(W, pad[1], dil[1], S, stride[1])
        self.M = N * self.P * self.Q
        st = Stream(seed)
        self.X = store(draw(st, N * H * W * C, dist_x), dtype)
        self.Wt = store(draw(st, K * R * S * C, dist_w), dtype)
        self.Cm = store(draw(st, self.M * K, "uniform"), dtype) if with_c else None
        self.ldc = K
        self.bias = draw(st, K, dist_bias).astype(np.float32) if dist_bias else None

    def dims(self):
        return (self.N, self.H, self.W, self.C, self.K, self.R, self.S) + self.pad + self.stride + self.dil


# 3 x 3, stride 1, pad 1 over a 56 x 56 feature map with 256 channels in and
# out, batch 32 (a mid-network layer of a residual image network; the pages
# name implicit-GEMM convolution without a workload).
CONV_WORKLOADS = {
    "conv3x3_bf16_32x56x56x256": dict(N=32, H=56, W=56, C=256, K=256, R=3, S=3, pad=(1, 1), stride=(1, 1),
                                      dil=(1, 1), dtype="bf16", seed=31),
}
