"""Helpers shared by the GPU tests: upload a synth.Problem, run the C ABI, read back."""
import numpy as np
import torch

import tiled_tensor_core_02_gb300 as ttc

LAY = {"row": ttc.ROW_MAJOR, "col": ttc.COL_MAJOR}


def to_dev(buf):
    if buf is None:
        return None
    a = np.ascontiguousarray(buf)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    if a.size == 0:
        a = np.zeros(1, dtype=a.dtype)
    return torch.from_numpy(a).cuda()


def run(p, alpha=1.0, beta=0.0, act="none", use_bias=True, ldd=None, D=None, C_dev=None,
        expect=0, stream=None, workspace=None):
    """Runs ttc_gemm on problem p; returns the M x N output (storage type) as numpy."""
    out_np = np.int32 if p.dtype == "i8" else np.int16
    ldd = p.N if ldd is None else ldd
    A = to_dev(p.A)
    B = to_dev(p.B)
    C = C_dev if C_dev is not None else (to_dev(p.C) if p.C is not None else None)
    bias = to_dev(p.bias) if (use_bias and p.bias is not None) else None
    if D is None:
        D = torch.full((max(p.M * ldd, 1),), -1, dtype=torch.int32 if out_np == np.int32 else torch.int16,
                       device="cuda")
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    args = (p.M, p.N, p.K, A.data_ptr(), p.lda, LAY[p.layoutA], B.data_ptr(), p.ldb,
            LAY[p.layoutB], C.data_ptr() if (C is not None and beta != 0.0) else None,
            p.ldc, D.data_ptr(), ldd, alpha, beta,
            bias.data_ptr() if bias is not None else None, ttc.ACT[act], ttc.DTYPE[p.dtype])
    if workspace is None:
        st = ttc.ttc_gemm(*args, s)
    else:
        # workspace: bytes to allocate (-1: what the library asks for the
        # operand repack; -2: for the repack and an aligned copy of D)
        if workspace == -2:
            need = ttc.ttc_gemm_workspace_size_staged(p.M, p.N, p.K, A.data_ptr(), p.lda, LAY[p.layoutA],
                                                      B.data_ptr(), p.ldb, LAY[p.layoutB], D.data_ptr(), ldd,
                                                      ttc.DTYPE[p.dtype])
        else:
            need = ttc.ttc_gemm_workspace_size(p.M, p.N, p.K, A.data_ptr(), p.lda, LAY[p.layoutA],
                                               B.data_ptr(), p.ldb, LAY[p.layoutB], ttc.DTYPE[p.dtype])
        nbytes = need if workspace < 0 else workspace
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
        st = ttc.ttc_gemm_ws(*args, ws.data_ptr() if nbytes else None, nbytes, s)
    assert st == expect, ttc.STATUS.get(st, st)
    if st != 0:
        return None
    err = ttc.ttc_get_device_error(s)
    assert err == 0, ttc.STATUS.get(err, err)
    d = D.cpu().numpy()
    if out_np == np.int16:
        d = d.view(np.uint16)
    return d[: p.M * ldd].reshape(p.M, ldd)[:, : p.N] if p.M else d[:0].reshape(0, p.N)


def run_batched(probs, strides, alpha=1.0, beta=0.0, act="none", share_b=False, ldd=None, full=None):
    """Packs a list of same-shaped problems into strided buffers (stride in
    elements per operand: dict with keys A, B, C, D; B's stride 0 when
    share_b), runs ttc_gemm_strided_batched, and returns one output per batch
    (and appends the whole D buffer, -1 where nothing was written, to the list
    `full` when one is given)."""
    p0 = probs[0]
    nb = len(probs)
    out_np = np.int32 if p0.dtype == "i8" else np.int16
    ldd = p0.N if ldd is None else ldd

    def pack(bufs, stride, dtype):
        n = max((len(bufs) - 1) * stride + max(b.size for b in bufs), 1)
        big = np.zeros(n, dtype=dtype)
        for i, b in enumerate(bufs):
            big[i * stride:i * stride + b.size] = b
        return big

    A = to_dev(pack([q.A for q in probs], strides["A"], probs[0].A.dtype))
    sB = 0 if share_b else strides["B"]
    B = to_dev(pack([q.B for q in (probs[:1] if share_b else probs)], sB, probs[0].B.dtype))
    C = to_dev(pack([q.C for q in probs], strides["C"], probs[0].C.dtype)) if p0.C is not None else None
    bias = to_dev(p0.bias) if p0.bias is not None else None
    sD = strides["D"]
    D = torch.full((max((nb - 1) * sD + p0.M * ldd, 1),), -1,
                   dtype=torch.int32 if out_np == np.int32 else torch.int16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = ttc.ttc_gemm_strided_batched(nb, p0.M, p0.N, p0.K, A.data_ptr(), p0.lda, strides["A"], LAY[p0.layoutA],
                                      B.data_ptr(), p0.ldb, sB, LAY[p0.layoutB],
                                      C.data_ptr() if (C is not None and beta != 0.0) else None, p0.ldc,
                                      strides["C"], D.data_ptr(), ldd, sD, alpha, beta,
                                      bias.data_ptr() if bias is not None else None, ttc.ACT[act],
                                      ttc.DTYPE[p0.dtype], s)
    assert st == 0, ttc.STATUS.get(st, st)
    assert ttc.ttc_get_device_error(s) == 0
    d = D.cpu().numpy()
    if full is not None:
        full.append(d.copy())
    if out_np == np.int16:
        d = d.view(np.uint16)
    return [d[i * sD:i * sD + p0.M * ldd].reshape(p0.M, ldd)[:, :p0.N] for i in range(nb)]
