"""Python binding of the ttc C ABI (libttc.so): argument marshalling only.

Every step of the GEMM runs in the library's CUDA kernels.  There is no CPU
or PyTorch fallback: if libttc.so is missing or cannot be loaded, importing
the binding's entry points raises.

Names follow the C header include/ttc.h:
  ttc_gemm(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd,
           alpha, beta, bias, act, dtype, stream) -> status (int)
  ttc_get_device_error(stream) -> status
  ttc_status_string(status) -> str
  ttc_set_knob(knob, value) -> status
  ttc_launch_count() -> int
plus `gemm(...)`, a convenience wrapper on torch tensors that reads the
layouts and leading dimensions off the tensors' strides.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

ROW_MAJOR, COL_MAJOR = 0, 1
ACT = {"none": 0, "relu": 1, "gelu_tanh": 2}
DTYPE = {"f16": 0, "bf16": 1, "i8": 2}
STATUS = {0: "TTC_OK", 1: "TTC_ERR_INVALID_ARG", 2: "TTC_ERR_UNSUPPORTED", 3: "TTC_ERR_CUDA",
          4: "TTC_ERR_TIMEOUT", 5: "TTC_ERR_SCRATCH_TOO_SMALL"}
STATIC_SCRATCH_BYTES = 16 * 1024 * 1024
KNOB = {"timeout_ns": 0, "inject_stall": 1, "force_generic_load": 2, "force_generic_store": 3,
        "tile_n": 4, "pair": 5, "swap_ab": 6, "split_k": 7, "pair_tile_n": 8,
        "group_m": 9, "gemv": 10, "conv_halo": 11, "pair_tail": 12, "pdl": 13, "i8_wide": 14, "pair_epi_warps": 15}

# Every symbol the C header declares (checked by the test suite).
EXPORTS = ("ttc_gemm", "ttc_gemm_strided_batched", "ttc_gemm_ws", "ttc_gemm_workspace_size",
           "ttc_gemm_workspace_size_staged",
           "ttc_gemm_static_scratch", "ttc_transpose", "ttc_conv2d_fprop",
           "ttc_get_device_error", "ttc_status_string", "ttc_set_knob", "ttc_launch_count", "ttc_gemm_plan")

_lib = None


class TTCError(RuntimeError):
    def __init__(self, status: int, what: str = "ttc_gemm"):
        self.status = status
        super().__init__(f"{what} failed: {STATUS.get(status, status)}")


def library_path() -> str:
    return _build.LIB


def load():
    """Load libttc.so (it must have been built: __graft_entry__.build() or _build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libttc.so is not built ({_build.LIB}); run tiled_tensor_core_02_gb300._build.build()")
    L = ctypes.CDLL(_build.LIB)
    i64, vp, f, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    L.ttc_gemm.argtypes = [i64, i64, i64, vp, i64, i, vp, i64, i, vp, i64, vp, i64, f, f, vp, i, i, vp]
    L.ttc_gemm.restype = i
    L.ttc_gemm_strided_batched.argtypes = [i64, i64, i64, i64, vp, i64, i64, i, vp, i64, i64, i, vp, i64, i64,
                                           vp, i64, i64, f, f, vp, i, i, vp]
    L.ttc_gemm_strided_batched.restype = i
    L.ttc_conv2d_fprop.argtypes = [i64] * 13 + [vp, vp, vp, i64, vp, i64, f, f, vp, i, i, vp]
    L.ttc_conv2d_fprop.restype = i
    L.ttc_transpose.argtypes = [i64, i64, vp, i64, vp, i64, i, vp]
    L.ttc_transpose.restype = i
    L.ttc_gemm_ws.argtypes = [i64, i64, i64, vp, i64, i, vp, i64, i, vp, i64, vp, i64, f, f, vp, i, i, vp,
                              ctypes.c_size_t, vp]
    L.ttc_gemm_ws.restype = i
    L.ttc_gemm_static_scratch.argtypes = [i64, i64, i64, vp, i64, i, vp, i64, i, vp, i64, vp, i64, f, f,
                                          vp, i, i, vp]
    L.ttc_gemm_static_scratch.restype = i
    L.ttc_gemm_workspace_size.argtypes = [i64, i64, i64, vp, i64, i, vp, i64, i, i]
    L.ttc_gemm_workspace_size.restype = ctypes.c_size_t
    L.ttc_gemm_workspace_size_staged.argtypes = [i64, i64, i64, vp, i64, i, vp, i64, i, vp, i64, i]
    L.ttc_gemm_workspace_size_staged.restype = ctypes.c_size_t
    L.ttc_get_device_error.argtypes = [vp]
    L.ttc_get_device_error.restype = i
    L.ttc_status_string.argtypes = [i]
    L.ttc_status_string.restype = ctypes.c_char_p
    L.ttc_set_knob.argtypes = [i, i64]
    L.ttc_set_knob.restype = i
    L.ttc_launch_count.argtypes = []
    L.ttc_launch_count.restype = i64
    L.ttc_gemm_plan.argtypes = [i64, i64, i64, i64, vp, i64, i64, i, vp, i64, i64, i, vp, i64, i64, vp, i64, i64,
                                f, f, vp, i, i, vp, ctypes.c_size_t, i, ctypes.c_char_p, ctypes.c_size_t]
    L.ttc_gemm_plan.restype = i
    _lib = L
    return L


# ------------------------------------------------------------------ raw C-ABI names

def ttc_gemm(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta, bias, act,
             dtype, stream) -> int:
    """Pointers are ints (device addresses) or None; stream is a cudaStream_t as int or None."""
    return load().ttc_gemm(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta,
                           bias, act, dtype, stream)


def ttc_gemm_strided_batched(batch, M, N, K, A, lda, strideA, layoutA, B, ldb, strideB, layoutB, C, ldc,
                             strideC, D, ldd, strideD, alpha, beta, bias, act, dtype, stream) -> int:
    return load().ttc_gemm_strided_batched(batch, M, N, K, A, lda, strideA, layoutA, B, ldb, strideB,
                                           layoutB, C, ldc, strideC, D, ldd, strideD, alpha, beta, bias,
                                           act, dtype, stream)


def ttc_conv2d_fprop(N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w, X, Wt, Cm, ldc, D,
                     ldd, alpha, beta, bias, act, dtype, stream) -> int:
    return load().ttc_conv2d_fprop(N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w, dil_h, dil_w, X, Wt, Cm,
                                   ldc, D, ldd, alpha, beta, bias, act, dtype, stream)


def ttc_transpose(rows, cols, src, lds, dst, ldd, elem_bytes, stream) -> int:
    return load().ttc_transpose(rows, cols, src, lds, dst, ldd, elem_bytes, stream)


def ttc_gemm_ws(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta, bias, act,
                dtype, workspace, workspace_bytes, stream) -> int:
    return load().ttc_gemm_ws(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta,
                              bias, act, dtype, workspace, workspace_bytes, stream)


def ttc_gemm_static_scratch(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd, alpha, beta,
                            bias, act, dtype, stream) -> int:
    """ttc_gemm_ws with the library's fixed device scratch array: for callers
    that cannot allocate device memory (see include/ttc.h)."""
    return load().ttc_gemm_static_scratch(M, N, K, A, lda, layoutA, B, ldb, layoutB, C, ldc, D, ldd,
                                          alpha, beta, bias, act, dtype, stream)


def ttc_gemm_plan(batch, M, N, K, A, lda, strideA, layoutA, B, ldb, strideB, layoutB, C, ldc, strideC, D, ldd,
                  strideD, alpha, beta, bias, act, dtype, workspace, workspace_bytes, sm_count):
    """(status, plan): the launches the call would make on a device with
    sm_count SMs, planned on the host without a GPU (see include/ttc.h)."""
    buf = ctypes.create_string_buffer(4096)
    st = load().ttc_gemm_plan(batch, M, N, K, A, lda, strideA, layoutA, B, ldb, strideB, layoutB, C, ldc, strideC,
                              D, ldd, strideD, alpha, beta, bias, act, dtype, workspace, workspace_bytes, sm_count,
                              buf, len(buf))
    return st, buf.value.decode()


def ttc_gemm_workspace_size(M, N, K, A, lda, layoutA, B, ldb, layoutB, dtype) -> int:
    return load().ttc_gemm_workspace_size(M, N, K, A, lda, layoutA, B, ldb, layoutB, dtype)


def ttc_gemm_workspace_size_staged(M, N, K, A, lda, layoutA, B, ldb, layoutB, D, ldd, dtype) -> int:
    return load().ttc_gemm_workspace_size_staged(M, N, K, A, lda, layoutA, B, ldb, layoutB, D, ldd, dtype)


def ttc_get_device_error(stream=None) -> int:
    return load().ttc_get_device_error(stream)


def ttc_status_string(status: int) -> str:
    return load().ttc_status_string(status).decode()


def ttc_set_knob(knob, value: int) -> int:
    k = KNOB[knob] if isinstance(knob, str) else int(knob)
    return load().ttc_set_knob(k, int(value))


def ttc_launch_count() -> int:
    return load().ttc_launch_count()


# ------------------------------------------------------------------ torch convenience

def _matrix_layout(t, rows, cols):
    """(layout, ld) of a 2-D tensor viewed as a rows x cols matrix."""
    s0, s1 = t.stride()
    if cols == 1 and rows >= 1 and s0 == 1:
        return COL_MAJOR, max(s1, rows)
    if s1 == 1 or cols == 1:
        return ROW_MAJOR, max(s0, cols, 1)
    if s0 == 1 or rows == 1:
        return COL_MAJOR, max(s1, rows, 1)
    raise ValueError("operand must be row- or column-major (one unit stride)")


def gemm(a, b, c=None, out=None, *, alpha=1.0, beta=0.0, bias=None, act="none", stream=None,
         check=True):
    """D = act(alpha * a @ b + beta * c + bias) through the C ABI.

    a: M x K, b: K x N (torch CUDA tensors, fp16/bf16/int8, row- or column-major);
    c, out: M x N row-major (input dtype, int32 for int8).  Returns out."""
    import torch

    M, K = a.shape
    K2, N = b.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    dt = {torch.float16: "f16", torch.bfloat16: "bf16", torch.int8: "i8"}[a.dtype]
    odt = torch.int32 if dt == "i8" else a.dtype
    if out is None:
        out = torch.empty((M, N), dtype=odt, device=a.device)
    la, lda = _matrix_layout(a, M, K)
    lb, ldb = _matrix_layout(b, K, N)
    if out.stride(1) != 1 and N > 1:
        raise ValueError("out must be row-major")
    ldd = max(out.stride(0), N)
    if c is not None:
        if c.stride(1) != 1 and N > 1:
            raise ValueError("c must be row-major")
        ldc = max(c.stride(0), N)
        cptr = c.data_ptr()
    else:
        ldc, cptr = N, None
    bptr = bias.data_ptr() if bias is not None else None
    if stream is None:
        stream = torch.cuda.current_stream(a.device).cuda_stream
    st = ttc_gemm(M, N, K, a.data_ptr(), lda, la, b.data_ptr(), ldb, lb, cptr, ldc, out.data_ptr(),
                  ldd, float(alpha), float(beta), bptr, ACT[act], DTYPE[dt], stream)
    if check and st != 0:
        raise TTCError(st)
    return out
