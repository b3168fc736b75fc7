"""Plain fp64 CPU oracle of the INT8 ConvRot W8A8 linear layer.

TEST INFRASTRUCTURE ONLY. This module is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the
product path never imports, calls or links it, and it shares no code, table
or helper with the CUDA library. It is written to be checked against the
pages by eye: each step is the textbook definition, with a library matmul
as the only building block, no blocking, no fusion and no reordering.

Sources (page title, section):

* "INT8 Convrot Safetensors" (stable-diffusion.cpp docs), sections
  "How INT8 convrot works", "Weight quantization" and
  "Runtime activation quantization": the rotation R (normalized Kronecker
  power of the printed H4, block-diagonal over contiguous groups of G input
  features), the per-row absmax/127 scale, round-and-clamp to [-127, 127],
  the int32 GEMM and the reconstruction Y = A * s_x[r] * s_w[o] + b[o].
* "Add experimental W8A8 MatMul with optional QuaRot-style rotation"
  (gemma.cpp issue), sections "Quantization method" and "Rotation method":
  the block randomized Hadamard variant (Rademacher signs, then a
  Walsh-Hadamard transform, then 1/sqrt(B), applied to activation and weight
  rows alike) and the naive variant without rotation.

Readings where the pages are silent:

* round() is round-half-to-even (``numpy.rint``).
* An all-zero row has s = 0 and Q = 0 (the pages divide by s without saying
  what happens at s = 0).
* Scales are stored as fp32 (the sglang digest stores the weight scale as
  float32); the divide uses the unrounded fp64 scale.
* The Walsh-Hadamard matrix is in natural (Sylvester) order, and the block
  transform acts on each row as on the vector it holds (R x, written as the
  row x R^T), as "(Ra)^T (Rb)" in "Rotation method" has it.
* Y is reconstructed in fp64 from the stored fp32 scales and rounded once to
  bf16, round-to-nearest-even.
* 4-bit ConvRot ("feat: load ConvRot int4 and per-channel int8 safetensors",
  sections "Solution" and "The rotation"): codes in [-7, 7] with one fp32
  scale per output channel, adjacent pairs packed in a byte. The pages do not
  say which nibble holds the first element nor how the 4-bit activations are
  scaled: element 2j goes to the low nibble as a two's-complement nibble, and
  activations use the int8 recipe with 7 in place of 127 (s = max|x_rot|/7,
  q = clamp(round(x_rot/s), -7, 7)).

Every function is pinned by ``tests/test_oracle_pins.py`` against what the
pages and the mathematics fix: the printed H4, closed forms of R, basis
vectors, orthogonality and dot-product preservation, hand-built quantizer
rows, brute-force integer dot products and library routines.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "H4", "TRANSFORMS", "log4", "check_group", "regular_hadamard",
    "sylvester_hadamard", "rht_block", "row_operator", "rotate_rows",
    "quantize_rows", "prepare_weights", "quantize_act", "int_gemm",
    "reconstruct", "round_to_bf16", "linear", "float_linear",
    "boundary_distance", "QMAX", "QMAX4", "pack_int4", "unpack_int4",
    "row_absmax", "quantize_rows_given",
]

# "INT8 Convrot Safetensors", "How INT8 convrot works": the printed matrix,
# divided by 2.
H4 = np.array([[1.0, 1.0, 1.0, -1.0],
               [1.0, 1.0, -1.0, 1.0],
               [1.0, -1.0, 1.0, 1.0],
               [-1.0, 1.0, 1.0, 1.0]], dtype=np.float64) / 2.0

TRANSFORMS = ("h4", "rht", "none")

QMAX = 127  # "clamp(round(...), -127, 127)" in both quantization sections
QMAX4 = 7   # 4-bit ConvRot: "int4 values occupy [-7,7]"


def log4(G: int) -> int:
    """n with 4**n == G, or -1 if G is not a power of four."""
    n, v = 0, 1
    while v < G:
        v *= 4
        n += 1
    return n if v == G else -1


def check_group(K: int, G: int, transform: str) -> None:
    """Validity rules for the group size.

    "INT8 Convrot Safetensors", "Checkpoint format": the convrot group size
    must be a power of four and must divide the input feature dimension.
    gemma.cpp issue, "Rotation method": the block transform is used only when
    K is divisible by the block size (128 there; any power of two here).
    """
    if transform == "none":
        return
    if G <= 0 or K % G != 0:
        raise ValueError(f"group {G} must divide K={K}")
    if transform == "h4":
        if G < 4 or log4(G) < 0:
            raise ValueError(f"group {G} is not a power of four")
    elif transform == "rht":
        if G < 2 or (G & (G - 1)) != 0:
            raise ValueError(f"block {G} is not a power of two")
    else:
        raise ValueError(f"unknown transform {transform!r}")


def regular_hadamard(G: int) -> np.ndarray:
    """R_G: the normalized Kronecker power H4 (x) ... (x) H4 (n factors, G = 4**n).

    "INT8 Convrot Safetensors", "How INT8 convrot works". Each factor already
    carries its 1/2, so the product carries 2**-n = 1/sqrt(G).
    """
    n = log4(G)
    if n < 1:
        raise ValueError(f"group {G} is not a power of four >= 4")
    R = np.ones((1, 1), dtype=np.float64)
    for _ in range(n):
        R = np.kron(R, H4)
    return R


def sylvester_hadamard(B: int) -> np.ndarray:
    """Unnormalized Walsh-Hadamard matrix of order B in natural order."""
    if B < 1 or (B & (B - 1)) != 0:
        raise ValueError(f"order {B} is not a power of two")
    H2 = np.array([[1.0, 1.0], [1.0, -1.0]])
    H = np.ones((1, 1), dtype=np.float64)
    while H.shape[0] < B:
        H = np.kron(H, H2)
    return H


def rht_block(B: int, signs) -> np.ndarray:
    """Column-vector operator of the block randomized Hadamard transform.

    gemma.cpp issue, "Rotation method": a fixed +-1 Rademacher diagonal D,
    then a Walsh-Hadamard transform H, then 1/sqrt(B); so v -> H (D v) / sqrt(B).
    """
    s = np.asarray(signs, dtype=np.float64).reshape(-1)
    if s.shape[0] != B or not np.all(np.abs(s) == 1.0):
        raise ValueError("signs must be B values of +-1")
    return sylvester_hadamard(B) @ np.diag(s) / np.sqrt(B)


def row_operator(G: int, transform: str, signs=None) -> np.ndarray:
    """T with x_rot = x @ T for one row-major group x of length G.

    h4:  X_rot = X R ("How INT8 convrot works"), so T = R_G.
    rht: the page rotates each row vector v as R v, so for a row x the
         rotated row is x R^T.
    """
    if transform == "h4":
        return regular_hadamard(G)
    if transform == "rht":
        return rht_block(G, signs).T
    raise ValueError(f"no group operator for transform {transform!r}")


def rotate_rows(X, G: int, transform: str = "h4", signs=None) -> np.ndarray:
    """Apply the block-diagonal rotation to every row of X, in fp64.

    Every contiguous group of G input features is multiplied by the same
    G x G operator (a dense product, O(K*G) per row).
    """
    X = np.asarray(X, dtype=np.float64)
    rows, K = X.shape
    if transform == "none":
        return X.copy()
    check_group(K, G, transform)
    T = row_operator(G, transform, signs)
    return (X.reshape(rows, K // G, G) @ T).reshape(rows, K)


def quantize_rows(Xrot, qmax: int = QMAX):
    """Per-row symmetric quantization of an already rotated matrix.

    "Weight quantization" / "Runtime activation quantization":
        s[r]    = max_i |X_rot[r, i]| / 127
        Q[r, i] = clamp(round(X_rot[r, i] / s[r]), -127, 127)
    and the same with 7 for the 4-bit codes (qmax = QMAX4).

    Returns (Q int8, s float32 as stored, v = X_rot / s in fp64 before
    rounding, s in fp64). A zero row gets s = 0 and Q = 0.
    """
    Xrot = np.asarray(Xrot, dtype=np.float64)
    amax = np.abs(Xrot).max(axis=1) if Xrot.shape[1] else np.zeros(Xrot.shape[0])
    s64 = amax / qmax
    safe = np.where(s64 > 0, s64, 1.0)
    v = np.where(s64[:, None] > 0, Xrot / safe[:, None], 0.0)
    Q = np.clip(np.rint(v), -qmax, qmax).astype(np.int8)
    return Q, s64.astype(np.float32), v, s64


def row_absmax(Xrot) -> np.ndarray:
    """max_i |X_rot[r, i]| for every row, in fp64: the numerator of the row
    scale of "Runtime activation quantization"."""
    Xrot = np.asarray(Xrot, dtype=np.float64)
    return np.abs(Xrot).max(axis=1) if Xrot.shape[1] else np.zeros(Xrot.shape[0])


def quantize_rows_given(Xrot, amax, qmax: int = QMAX):
    """Per-row quantization with each row's maximum supplied instead of
    taken over the given columns:

        s[r]    = amax[r] / 127
        Q[r, i] = clamp(round(X_rot[r, i] / s[r]), -127, 127)

    This is the step a row-parallel linear needs (sglang digest, "风险与影响",
    on tensor parallelism splitting the rotated input dimension over ranks,
    each with whole groups): the scale belongs to the whole row, so its
    maximum is the largest of the slices' maxima, and every slice is
    quantized with it. With amax = row_absmax(Xrot) this is quantize_rows.
    Returns (Q int8, s float32 as stored, v = X_rot / s in fp64, s in fp64).
    """
    Xrot = np.asarray(Xrot, dtype=np.float64)
    s64 = np.asarray(amax, dtype=np.float64) / qmax
    safe = np.where(s64 > 0, s64, 1.0)
    v = np.where(s64[:, None] > 0, Xrot / safe[:, None], 0.0)
    Q = np.clip(np.rint(v), -qmax, qmax).astype(np.int8)
    return Q, s64.astype(np.float32), v, s64


def prepare_weights(W, G: int, transform: str = "h4", signs=None, qmax: int = QMAX):
    """Offline weight path: W_rot = W R per K-group, then per-output-row codes.

    "How INT8 convrot works" (W_rot = W R) and "Weight quantization".
    Returns (Q_w int8 [N,K], s_w float32 [N], v fp64 [N,K]).
    """
    Q, s, v, _ = quantize_rows(rotate_rows(W, G, transform, signs), qmax)
    return Q, s, v


def quantize_act(X, G: int, transform: str = "h4", signs=None, qmax: int = QMAX):
    """Runtime activation path: X_rot = X R, then one dynamic scale per row.

    "Runtime activation quantization". The packed activation is the pair
    (Q_x, s_x). Returns (Q_x int8 [M,K], s_x float32 [M], v fp64 [M,K]).
    """
    Q, s, v, _ = quantize_rows(rotate_rows(X, G, transform, signs), qmax)
    return Q, s, v


def pack_int4(Q) -> np.ndarray:
    """4-bit codes in [-7, 7], two per byte: element 2j in the low nibble,
    2j + 1 in the high nibble, each as a two's-complement nibble."""
    Q = np.asarray(Q)
    if Q.shape[-1] % 2 or np.abs(Q.astype(np.int64)).max(initial=0) > QMAX4:
        raise ValueError("need an even row length and codes in [-7, 7]")
    lo = Q[..., 0::2].astype(np.int64) & 0xF
    hi = Q[..., 1::2].astype(np.int64) & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_int4(P) -> np.ndarray:
    """Inverse of pack_int4: bytes -> int8 codes, sign-extended nibbles."""
    P = np.asarray(P, dtype=np.uint8).astype(np.int64)
    lo, hi = P & 0xF, (P >> 4) & 0xF
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(P.shape[:-1] + (2 * P.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def int_gemm(Qx, Qw) -> np.ndarray:
    """A[r, o] = sum_i Q_x[r, i] * Q_w[o, i] ("Runtime activation quantization").

    Computed with one fp64 matrix product. This is exact: every product and
    every partial sum is an integer of magnitude at most 127 * 127 * K, far
    below 2**53, so each one is representable in fp64 and the result does not
    depend on the order of summation. The result is returned as int64 and
    checked to fit the int32 accumulator the page names.
    """
    Qx = np.asarray(Qx)
    Qw = np.asarray(Qw)
    K = Qx.shape[1]
    if 127 * 127 * K >= 2 ** 53:
        raise ValueError("K too large for an exact fp64 product")
    A = (Qx.astype(np.float64) @ Qw.astype(np.float64).T).astype(np.int64)
    if A.size and np.abs(A).max() >= 2 ** 31:
        raise OverflowError("accumulator exceeds int32")
    return A


def reconstruct(A, sx, sw, bias=None) -> np.ndarray:
    """Y[r, o] = A[r, o] * s_x[r] * s_w[o] + b[o], in fp64 from the stored scales."""
    Y = np.asarray(A, dtype=np.float64) * np.asarray(sx, np.float64)[:, None] \
        * np.asarray(sw, np.float64)[None, :]
    if bias is not None:
        Y = Y + np.asarray(bias, dtype=np.float64)[None, :]
    return Y


def round_to_bf16(Y) -> np.ndarray:
    """Round fp64 values once to bf16 (8 significant bits), ties to even.

    Written out on the frexp decomposition y = m * 2**e, 0.5 <= |m| < 1:
    the bf16 value is rint(m * 256) / 256 * 2**e. Values are returned as
    fp64 holding bf16 numbers. (Normal range only; the outputs here are far
    from the bf16 subnormal range.)
    """
    Y = np.asarray(Y, dtype=np.float64)
    m, e = np.frexp(Y)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def linear(X, Qw, sw, bias, G: int, transform: str = "h4", signs=None, qmax: int = QMAX):
    """The whole runtime path for one linear: rotate, quantize, GEMM, reconstruct.

    Returns a dict with Qx, sx, v (pre-rounding activation codes), A (int64),
    Y64 (fp64) and Y (bf16 values as fp64).
    """
    Qx, sx, v = quantize_act(X, G, transform, signs, qmax)
    A = int_gemm(Qx, Qw)
    Y64 = reconstruct(A, sx, sw, bias)
    return {"Qx": Qx, "sx": sx, "v": v, "A": A, "Y64": Y64, "Y": round_to_bf16(Y64)}


def float_linear(X, W, bias=None) -> np.ndarray:
    """Unquantized reference Y = X W^T + b in fp64 (quality side output only)."""
    Y = np.asarray(X, np.float64) @ np.asarray(W, np.float64).T
    if bias is not None:
        Y = Y + np.asarray(bias, np.float64)[None, :]
    return Y


def boundary_distance(v) -> np.ndarray:
    """Distance of each pre-rounding code v to the nearest rounding boundary k + 1/2."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    return np.abs(a - (np.floor(a) + 0.5))
