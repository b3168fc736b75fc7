"""Comparison helpers shared by the GPU parity tests (no method arithmetic).

Tolerances (stated once, used everywhere):
* Q codes: |Q_gpu - Q_oracle| <= 1 everywhere; mismatches on at most 1e-4 of
  the elements; and only where the oracle's fp64 pre-rounding code v lies
  within 1e-6 of a rounding boundary relative to the row's full scale of 127
  codes (|v - (k + 1/2)| <= 1.27e-4).
* scales: relative error <= 1e-6; an all-zero row has scale exactly 0.
* int32 accumulators: bit-exact when fed the oracle's codes.
* Y fed with the oracle's codes: within one bf16 ulp of the oracle's fp64 Y
  plus 1e-6 of the magnitudes that entered the fp32 epilogue.
* Y end to end from X: max|Y_gpu - Y_oracle| <= 1e-2 * max|Y_oracle|.
"""
import numpy as np
import torch

import oracle as O

CODE_BOUNDARY_TOL = 1e-6 * 127
CODE_MISMATCH_FRAC = 1e-4
SCALE_RTOL = 1e-6
Y_E2E_RTOL = 1e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def check_codes(q_gpu, q_or, v, label=""):
    q_gpu = np.asarray(q_gpu).astype(np.int64)
    q_or = np.asarray(q_or).astype(np.int64)
    d = q_gpu - q_or
    bad = d != 0
    n_bad = int(bad.sum())
    assert np.abs(d).max(initial=0) <= 1, f"{label}: code differs by more than 1 LSB"
    assert n_bad <= CODE_MISMATCH_FRAC * d.size, f"{label}: {n_bad} mismatches of {d.size}"
    if n_bad:
        dist = O.boundary_distance(np.asarray(v)[bad])
        assert dist.max() <= CODE_BOUNDARY_TOL, \
            f"{label}: mismatch {dist.max():.3g} from a rounding boundary"
    return n_bad


def check_scales(s_gpu, s_or, label=""):
    s_gpu = np.asarray(s_gpu, dtype=np.float64)
    s_or = np.asarray(s_or, dtype=np.float64)
    zero = s_or == 0
    assert np.all(s_gpu[zero] == 0), f"{label}: zero rows must get scale 0"
    nz = ~zero
    if nz.any():
        rel = np.abs(s_gpu[nz] - s_or[nz]) / s_or[nz]
        assert rel.max() <= SCALE_RTOL, f"{label}: scale rel err {rel.max():.3g}"


def bf16_ulp(y):
    y = np.abs(np.asarray(y, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(y, 1e-30)))
    return np.exp2(e - 7)


def check_y_same_codes(y_gpu, A, sx, sw, bias, label=""):
    """Y computed by the GPU from codes identical to the oracle's."""
    y64 = O.reconstruct(A, sx, sw, bias)
    mag = np.abs(np.asarray(A, np.float64) * np.asarray(sx, np.float64)[:, None]
                 * np.asarray(sw, np.float64)[None, :])
    if bias is not None:
        mag = mag + np.abs(np.asarray(bias, np.float64))[None, :]
    tol = bf16_ulp(y64) + 1e-6 * mag + 1e-30
    err = np.abs(np.asarray(y_gpu, np.float64) - y64)
    worst = (err / tol).max(initial=0)
    assert worst <= 1.0, f"{label}: Y off by {worst:.3g} x tolerance"


def check_y_e2e(y_gpu, y_or, label=""):
    y_gpu = np.asarray(y_gpu, np.float64)
    y_or = np.asarray(y_or, np.float64)
    err = np.abs(y_gpu - y_or).max()
    assert err <= Y_E2E_RTOL * np.abs(y_or).max(), f"{label}: Y error {err:.3g}"
    return err / np.abs(y_or).max()


def tensor_core_takes(K, G, transform="h4"):
    """Whether the library's tensor-core rotate+quantize kernel takes rows of
    K with this group (it then runs where the caller does not ask for a
    kernel): the regular Hadamard, K a multiple of 256 (1024 for G = 1024),
    or for G <= 64 a multiple of 64 from 256 up whose tiles of 2 or 4 rows
    (a whole number of 4-line superblocks) fit the 48 KB stage."""
    if transform != "h4" or G not in (4, 16, 64, 256, 1024) or K % 64 != 0:
        return False
    lines = K // 64
    if K % max(256, G) == 0:
        return lines <= 256 or (lines % ((lines + 255) // 256) == 0 and (lines // ((lines + 255) // 256)) % 8 == 0)
    r0 = 2 if lines % 2 == 0 else 4
    return G <= 64 and K >= 256 and lines <= 256 and r0 * K * 2 <= 48 * 1024

