"""Shared helpers for the GPU parity tests: moving synthetic inputs to the
device and checking results against the oracle."""
import numpy as np
import torch

TOL_REL = 2e-3   # |y - y_ref| <= TOL_REL * sum_k |w'_k x_k| + TOL_ABS
TOL_ABS = 1e-6


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def weights_dev(q: np.ndarray, s: np.ndarray):
    return dev(q), dev(s.view(np.int16), torch.float16)


def x_dev(x_bits: np.ndarray):
    return dev(x_bits.view(np.int16), torch.bfloat16)


def check_tol(y_gpu: np.ndarray, y_ref: np.ndarray, B: np.ndarray, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        err = np.abs(y_gpu - y_ref)
    lim = TOL_REL * B + TOL_ABS
    # a NaN where the reference is a number fails (a comparison with NaN is
    # false either way); the same NaN or infinity on both sides passes
    same_special = (np.isnan(y_gpu) & np.isnan(y_ref)) | (np.isinf(y_ref) & (y_gpu == y_ref))
    bad = ~(err <= lim) & ~same_special
    err = np.where(same_special, 0.0, err)
    ratio = float(np.max(err / np.maximum(B, 1e-30))) if err.size else 0.0
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outputs outside tolerance; "
                           f"worst err {err.max():.3e}, max err/B {ratio:.3e}")
    return ratio
