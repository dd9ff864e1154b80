"""Comparison rules shared by the GPU parity tests.

* logits / hidden rows: per row, max|gpu - oracle| / max|oracle| <= tol, with
  tol = 1e-4 for fp32 models and 2e-2 for bf16 / Q4_0 models;
* tokens: bit-exact wherever the oracle's top-1 minus top-2 logit margin
  exceeds 0.05; at a smaller margin a mismatch is an allowed flip (batched
  arithmetic can reorder near ties) and a free-running comparison stops there.
"""
import numpy as np

MARGIN = 0.05
TOL = {"f32": 1e-4, "bf16": 2e-2, "q4_0": 2e-2}


def rel_rows(gpu, ref):
    gpu = np.asarray(gpu, np.float64).reshape(len(ref), -1)
    ref = np.asarray(ref, np.float64).reshape(len(ref), -1)
    return np.abs(gpu - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)


def assert_rows_close(gpu, ref, tol, what=""):
    r = rel_rows(gpu, ref)
    assert np.all(r <= tol), "%s: worst row relative error %.3e > %.1e" % (what, r.max(), tol)
    return r.max()


def compare_tokens(gpu, ref, margins):
    """Number of leading positions that were compared and agreed; raises on a
    mismatch at a position whose oracle margin exceeds MARGIN."""
    n = min(len(gpu), len(ref))
    for i in range(n):
        if int(gpu[i]) != int(ref[i]):
            assert margins[i] <= MARGIN, "token %d: gpu %d vs oracle %d at margin %.4f" % (
                i, gpu[i], ref[i], margins[i])
            return i
    return n
