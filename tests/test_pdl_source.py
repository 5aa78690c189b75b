"""Source checks for programmatic dependent launch (no GPU).

A kernel launched with programmatic stream serialization may start while the
previous grid on the stream is still running, so it must execute
`grid_dependency_wait()` before its first global load or store.  These tests
read the CUDA sources: every launcher that adds the attribute launches a
kernel whose body calls `grid_dependency_wait()`, and in each such body the
call comes before the kernel's first global access helper (TMA loads,
plain global loads, error-word reads).
"""
import os
import re

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tiled_tensor_core_02_gb300",
                    "csrc")


def _sources():
    out = {}
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(CSRC, name)) as f:
                out[name] = f.read()
    return out


def _kernel_body(src, kernel):
    """Text of the body of `__global__ ... kernel(...) {...}` (brace-matched)."""
    m = re.search(r"__global__[^;{]*?\b" + re.escape(kernel) + r"\s*\(", src)
    if m is None:
        return None
    i = src.index("{", m.end())
    depth = 0
    for j in range(i, len(src)):
        if src[j] == "{":
            depth += 1
        elif src[j] == "}":
            depth -= 1
            if depth == 0:
                return src[i:j + 1]
    raise AssertionError(f"unbalanced braces in {kernel}")


def _pdl_launched_kernels(srcs):
    """Kernel names passed to cudaLaunchKernelEx in a function that also calls add_pdl_attribute."""
    names = set()
    for text in srcs.values():
        # the launches that closely follow each add_pdl_attribute call
        for m in re.finditer(r"add_pdl_attribute\s*\(", text):
            window = text[m.end():m.end() + 600]
            for k in re.finditer(r"cudaLaunchKernelEx\s*\(\s*&\w+\s*,\s*(\w+)", window):
                names.add(k.group(1))
    return names


def test_pdl_launches_found():
    names = _pdl_launched_kernels(_sources())
    assert {"gemm_kernel", "gemm_pair_kernel", "conv_halo_kernel", "gemv_rows_kernel", "repack_rows_kernel"} <= names, names


@pytest.mark.parametrize("kernel", ["gemm_kernel", "gemm_pair_kernel", "conv_halo_kernel", "gemv_rows_kernel",
                                    "repack_rows_kernel"])
def test_kernel_waits_before_global_access(kernel):
    srcs = _sources()
    body = None
    for text in srcs.values():
        body = _kernel_body(text, kernel)
        if body is not None:
            break
    assert body is not None, kernel
    w = body.find("grid_dependency_wait()")
    assert w >= 0, f"{kernel} never waits for the previous grid"
    # global-memory helpers that must not run before the wait
    first = [body.find(tok) for tok in ("tma_load", "__ldg(", "__ldcs(", "c_fetch16(", "error_raised(",
                                        "mbar_wait(", "mbar_wait_cluster(", "repack_load(")]
    first = [x for x in first if x >= 0]
    assert first and w < min(first), f"{kernel}: a global access precedes grid_dependency_wait()"


def test_launches_without_the_attribute_do_not_signal():
    """Kernels launched in plain stream order (unpack, transpose) do not
    signal dependents, so a kernel after them waits for their completion."""
    srcs = _sources()
    assert "grid_dependents_launch" not in srcs["transpose.cu"]
    assert "add_pdl_attribute" not in srcs["transpose.cu"]
    body = _kernel_body(srcs["repack.cu"], "unpack_rows_kernel")
    assert body is not None and "grid_dependents_launch" not in body and "griddepcontrol" not in body
    assert "cudaLaunchKernelEx" not in srcs["repack.cu"].split("launch_unpack(")[-1]
