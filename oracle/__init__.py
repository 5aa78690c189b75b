"""CPU oracle for the tiled GEMM, the implicit-GEMM convolution, the transpose
and the layout algebra.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product (the CUDA
library ``tiled_tensor_core_02_gb300`` and its C ABI) never imports, links or
calls anything here, and nothing here imports the product.

Contents
  * ``gemm_oracle.c`` (built into ``liboracle.so`` with gcc): the plain
    per-element GEMM definition, fp64 (fp16/bf16) / int64 (int8) accumulation,
    fp64 epilogue; and the plain per-element 2-D convolution (NHWC x KRSC,
    stride / padding / dilation, zero taps outside the input) with the same
    epilogue.  Bound through ctypes below.
  * ``layout.py``: the layout-algebra definitions (crd2idx, composition,
    complement, logical_divide) in plain Python.
  * the parity checker: the float tolerance, the sampling rule for large
    outputs and the Freivalds check.

Float tolerance (per element), against the unrounded fp64 oracle value r:
    |D - r| <= 1e-2 * S_abs * 2**-7 + 1e-3 + ulp_out(max(|D|, |r|)) / 2
S_abs = sum_k |a_ik b_kj|.  The first two terms are the stated bound on the
fp32 accumulation; the half-ulp term admits the final round-to-nearest of the
fp32 result into the fp16/bf16 output, which the stated bound alone is tighter
than once |D| exceeds roughly 2**-7 S_abs.  int8 -> int32 must be bit-exact.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPE = {"f16": 0, "bf16": 1, "i8": 2}
LAYOUT = {"row": 0, "col": 1}
ACT = {"none": 0, "relu": 1, "gelu_tanh": 2}

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C, IEEE semantics, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-std=c11", "-D_GNU_SOURCE", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-pthread", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, vp, f, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        L.oracle_gemm_elements.argtypes = [i64, i64, i64, vp, i64, i, vp, i64, i, vp, i64,
                                           f, f, vp, i, i, i64, vp, vp, vp, vp, i]
        L.oracle_gemm_elements.restype = i
        L.oracle_matvec.argtypes = [i64, i64, vp, i64, i, i, vp, vp]
        L.oracle_matvec.restype = None
        L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_gelu_tanh.argtypes = [ctypes.c_double]
        L.oracle_gelu_tanh.restype = ctypes.c_double
        L.oracle_act.argtypes = [ctypes.c_int, ctypes.c_double]
        L.oracle_act.restype = ctypes.c_double
        L.oracle_num_cpus.restype = ctypes.c_int
        L.oracle_conv2d_elements.argtypes = [i64] * 13 + [vp, vp, vp, i64, f, f, vp, i, i, i64, vp, vp, vp, vp, i]
        L.oracle_conv2d_elements.restype = i
        L.oracle_conv_out_extent.argtypes = [i64] * 5
        L.oracle_conv_out_extent.restype = i64
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def gemm_elements(p, ii, jj, alpha=1.0, beta=0.0, act="none", use_bias=True, nthreads=0):
    """r and S_abs (float64 arrays) for output elements (ii[e], jj[e]) of synth.Problem p.

    Returns (r, sabs, threads_used)."""
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    n = ii.size
    r = np.empty(n, dtype=np.float64)
    sabs = np.empty(n, dtype=np.float64)
    A = np.ascontiguousarray(p.A)
    B = np.ascontiguousarray(p.B)
    C = None if (beta == 0.0 or p.C is None) else np.ascontiguousarray(p.C)
    bias = p.bias if (use_bias and p.bias is not None) else None
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
    if beta != 0.0 and C is None:
        raise ValueError("beta != 0 needs C")
    used = lib().oracle_gemm_elements(p.M, p.N, p.K, _ptr(A), p.lda, LAYOUT[p.layoutA],
                                      _ptr(B), p.ldb, LAYOUT[p.layoutB], _ptr(C), p.ldc,
                                      float(alpha), float(beta), _ptr(bias), ACT[act], DTYPE[p.dtype],
                                      n, _ptr(ii), _ptr(jj), _ptr(r), _ptr(sabs), int(nthreads))
    return r, sabs, used


def gemm_full(p, **kw):
    """The whole M x N result (r, sabs), each as an M x N float64 array."""
    M, N = p.M, p.N
    ii, jj = np.meshgrid(np.arange(M, dtype=np.int64), np.arange(N, dtype=np.int64), indexing="ij")
    r, s, _ = gemm_elements(p, ii.ravel(), jj.ravel(), **kw)
    return r.reshape(M, N), s.reshape(M, N)


def matvec(rows, cols, X, ld, layout, dtype, x):
    """y = X x in fp64 for a stored rows x cols matrix X."""
    X = np.ascontiguousarray(X)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(rows, dtype=np.float64)
    lib().oracle_matvec(rows, cols, _ptr(X), ld, LAYOUT[layout], DTYPE[dtype], _ptr(x), _ptr(y))
    return y


def f16_to_double(h):
    return lib().oracle_f16_to_double(int(h))


def bf16_to_double(h):
    return lib().oracle_bf16_to_double(int(h))


def act(name, v):
    return lib().oracle_act(ACT[name], float(v))


# ---------------------------------------------------------------- checking

def decode(bits, dtype):
    """Stored output (uint16 bit patterns / int32) -> float64 values."""
    if dtype == "f16":
        return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)
    if dtype == "bf16":
        b = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
        return b.astype(np.float64)
    return np.asarray(bits, dtype=np.float64)


def half_ulp(x, dtype):
    """Half a unit in the last place of |x| in the output format (fp16 or bf16)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    mant, emin = (10, -14) if dtype == "f16" else (7, -126)
    e = np.floor(np.log2(np.maximum(x, 2.0**emin)))
    e = np.maximum(e, emin)
    return 0.5 * 2.0 ** (e - mant)


def tolerance(d, r, sabs, dtype):
    return 1e-2 * sabs * 2.0**-7 + 1e-3 + half_ulp(np.maximum(np.abs(d), np.abs(r)), dtype)


def check_float(d, r, sabs, dtype):
    """Returns (ok, worst_ratio, index of worst) for decoded outputs d vs oracle r."""
    d = np.asarray(d, dtype=np.float64)
    if not np.all(np.isfinite(d)):
        bad = np.flatnonzero(~np.isfinite(d))
        return False, float("inf"), int(bad[0])
    tol = tolerance(d, r, sabs, dtype)
    ratio = np.abs(d - r) / tol
    w = int(np.argmax(ratio)) if ratio.size else 0
    worst = float(ratio[w]) if ratio.size else 0.0
    return worst <= 1.0, worst, w


def sample_indices(M, N, seed, n_lines=8, n_elems=65536):
    """Elements checked on outputs larger than 4096^2: 8 full rows and 8 full
    columns (SplitMix64 stream seed+1000, always including the first and the
    last) and n_elems single elements (stream seed+2000).  Returns (ii, jj)."""
    from synth import splitmix64
    x = splitmix64(seed + 1000, 0, 2 * (n_lines - 2))
    rows = sorted(set([0, M - 1] + [int(v % M) for v in x[:n_lines - 2]]))
    cols = sorted(set([0, N - 1] + [int(v % N) for v in x[n_lines - 2:]]))
    ii = [np.full(N, r, dtype=np.int64) for r in rows] + [np.arange(M, dtype=np.int64) for _ in cols]
    jj = [np.arange(N, dtype=np.int64) for _ in rows] + [np.full(M, c, dtype=np.int64) for c in cols]
    y = splitmix64(seed + 2000, 0, 2 * n_elems)
    ii.append((y[:n_elems] % np.uint64(M)).astype(np.int64))
    jj.append((y[n_elems:] % np.uint64(N)).astype(np.int64))
    return np.concatenate(ii), np.concatenate(jj)


def freivalds_vector(N, seed):
    """x in {-1, +1}^N from SplitMix64 stream seed+3000."""
    from synth import splitmix64
    x = splitmix64(seed + 3000, 0, N)
    return np.where((x >> np.uint64(63)) == 1, -1.0, 1.0)


# ---------------------------------------------------------------- transpose

def transpose(src, rows, cols, lds, ldd):
    """dst[j * ldd + i] = src[i * lds + j]: the definition, element by element.
    src is a flat array of any element type; returns a flat dst of
    cols * ldd elements (padding left zero)."""
    dst = np.zeros(max(cols * ldd, 0), dtype=src.dtype)
    for i in range(rows):
        row = src[i * lds:i * lds + cols]
        for j in range(cols):
            dst[j * ldd + i] = row[j]
    return dst


# ---------------------------------------------------------------- convolution

def conv_out_extent(n, pad, dil, taps, stride):
    return lib().oracle_conv_out_extent(n, pad, dil, taps, stride)


def conv_elements(cp, mm, kk, alpha=1.0, beta=0.0, act="none", use_bias=True, nthreads=0):
    """r and S_abs for output elements (mm[e], kk[e]) of synth.ConvProblem cp
    (row m = (n P + p) Q + q, column k = output channel).  Returns (r, sabs, threads)."""
    mm = np.ascontiguousarray(mm, dtype=np.int64)
    kk = np.ascontiguousarray(kk, dtype=np.int64)
    n = mm.size
    r = np.empty(n, dtype=np.float64)
    sabs = np.empty(n, dtype=np.float64)
    X = np.ascontiguousarray(cp.X)
    Wt = np.ascontiguousarray(cp.Wt)
    C = None if (beta == 0.0 or cp.Cm is None) else np.ascontiguousarray(cp.Cm)
    if beta != 0.0 and C is None:
        raise ValueError("beta != 0 needs C")
    bias = cp.bias if (use_bias and cp.bias is not None) else None
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
    used = lib().oracle_conv2d_elements(*cp.dims(), _ptr(X), _ptr(Wt), _ptr(C), cp.ldc, float(alpha),
                                        float(beta), _ptr(bias), ACT[act], DTYPE[cp.dtype], n, _ptr(mm),
                                        _ptr(kk), _ptr(r), _ptr(sabs), int(nthreads))
    if used < 0:
        raise ValueError("empty convolution output")
    return r, sabs, used


def conv_full(cp, **kw):
    """The whole (N P Q) x K result (r, sabs) as float64 arrays."""
    M, K = cp.M, cp.K
    mm, kk = np.meshgrid(np.arange(M, dtype=np.int64), np.arange(K, dtype=np.int64), indexing="ij")
    r, s, _ = conv_elements(cp, mm.ravel(), kk.ravel(), **kw)
    return r.reshape(M, K), s.reshape(M, K)
