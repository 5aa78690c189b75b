"""Run as a child process by test_threads_gpu.py: several host threads, each
on its own CUDA stream, call the library at once from a cold start (no
kernel variant used before, so the first-use set-up of tensor-map encoders,
shared-memory attributes, occupancy and index-map caches races too), and
every result is checked against the oracle.  Prints one line per thread and
exits non-zero on any mismatch."""
import sys
import threading

import numpy as np
import torch

import oracle
import synth
import tiled_tensor_core_02_gb300 as ttc
from gpu_util import run

PROBLEMS = [
    # (M, N, K, dtype, layoutA, layoutB, kwargs, alpha, beta, act, workspace)
    (300, 300, 100, "bf16", "row", "col", {}, 1.0, 0.0, "none", None),
    (600, 700, 256, "bf16", "col", "row", {"distC": "uniform"}, 1.5, 0.5, "gelu_tanh", None),
    (300, 200, 72, "i8", "row", "col", {"distA": "int8", "distB": "int8", "distC": "int8", "lda": 73,
                                        "ldb": 75}, 1.0, 1.0, "none", -2),
    (1, 4096, 512, "f16", "row", "col", {}, 1.0, 0.0, "relu", None),
    (16, 2048, 2048, "bf16", "row", "col", {}, 1.0, 0.0, "none", None),
    (257, 131, 97, "f16", "col", "col", {"distC": "uniform", "lda": 259, "ldb": 99}, 1.0, 1.0, "none", -1),
    (520, 600, 200, "bf16", "row", "row", {"dist_bias": "normal:0.5"}, 1.0, 0.0, "relu", None),
]


def main(threads=6, reps=3):
    ttc.load()
    probs, want = [], []
    for i, (M, N, K, dt, la, lb, kw, a, b, act, ws) in enumerate(PROBLEMS):
        p = synth.Problem(M, N, K, dtype=dt, layoutA=la, layoutB=lb, seed=900 + i, **kw)
        probs.append(p)
        want.append(oracle.gemm_full(p, alpha=a, beta=b, act=act))
    errors = []

    def worker(t):
        stream = torch.cuda.Stream()
        bad = 0
        with torch.cuda.stream(stream):
            for rep in range(reps):
                for j in range(len(PROBLEMS)):
                    k = (j + t) % len(PROBLEMS)  # every thread starts on a different problem
                    M, N, K, dt, la, lb, kw, a, b, act, ws = PROBLEMS[k]
                    p = probs[k]
                    try:
                        d = run(p, a, b, act, workspace=ws)
                        r, sabs = want[k]
                        if dt == "i8":
                            ok = np.array_equal(d.astype(np.int64), r.astype(np.int64))
                        else:
                            ok = oracle.check_float(oracle.decode(np.ascontiguousarray(d).ravel(), dt), r.ravel(),
                                                    sabs.ravel(), dt)[0]
                    except Exception as e:  # a failed status or a device error
                        ok = False
                        errors.append(f"thread {t} problem {k}: {e}")
                    bad += 0 if ok else 1
        print(f"thread {t}: {reps * len(PROBLEMS)} calls, {bad} wrong", flush=True)
        if bad:
            errors.append(f"thread {t}: {bad} wrong")

    ts = [threading.Thread(target=worker, args=(t,)) for t in range(threads)]
    for th in ts:
        th.start()
    for th in ts:
        th.join()
    for e in errors:
        print(e)
    return 1 if errors else 0


if __name__ == "__main__":
    sys.exit(main())
