"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a matrix
printed on the pages, a closed form derived independently of the oracle's
construction, a basis-vector case, an invariant (orthogonality, dot-product
preservation), hand-worked quantizer rows, brute-force integer dot products,
or a library routine (scipy's Hadamard matrix, torch's fp32->bf16 rounding).

The last group plants mistakes in a copy of the oracle (on the CPU) and
checks that the pins catch them.
"""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fixtures --

def load_printed_h4():
    rows, div = [], None
    with open(os.path.join(GOLDEN, "h4_printed.txt")) as f:
        for line in f:
            line = line.strip()
            if line.startswith("# divisor"):
                div = float(line.split()[-1])
            elif line and not line.startswith("#"):
                rows.append([float(t) for t in line.split()])
    return np.array(rows) / div


def load_quantizer_rows():
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, "quantizer_rows.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *vals = line.split()
            if tag == "row4":  # a 4-bit row: codes in [-7, 7]
                tag, cur["qmax"] = "row", 7
            cur[tag] = [float(v) for v in vals]
            if tag == "s":
                cases.append(cur)
                cur = {}
    return cases


def load_rht_basis_rows():
    """[(B, signs, rows)] from the hand-worked RHT basis rows: rows[j] is
    sqrt(B) times the rotated form of the basis row e_j."""
    blocks = []
    with open(os.path.join(GOLDEN, "rht_basis_rows.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *vals = line.split()
            if tag == "block":
                blocks.append({"B": int(vals[0]), "rows": []})
            elif tag == "signs":
                blocks[-1]["signs"] = [float(v) for v in vals]
            elif tag == "rows":
                blocks[-1]["rows"].append([float(v) for v in vals])
    return [(b["B"], np.array(b["signs"]), np.array(b["rows"])) for b in blocks]


def load_given_max_rows():
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, "quantizer_given_max.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *vals = line.split()
            cur[tag] = [float(v) for v in vals]
            if tag == "s":
                cases.append(cur)
                cur = {}
    return cases


# --------------------------------------------------------- pin predicates --
# Written as predicates so the planted-mistake tests can reuse them.

def closed_form_R(G):
    """R_G[i, j] = 2**-n * prod_k (-1)**[i_k + j_k == 3] over base-4 digits.

    H4[a, b] is -1/2 exactly where a + b == 3 and +1/2 elsewhere (read off
    the printed matrix), and a Kronecker power multiplies the factors digit
    by digit.
    """
    n = O.log4(G)
    idx = np.arange(G)
    sign = np.ones((G, G))
    for k in range(n):
        di = (idx // 4 ** k) % 4
        sign *= np.where((di[:, None] + di[None, :]) == 3, -1.0, 1.0)
    return sign / 2 ** n


def pin_orthogonal_symmetric(R, tol=1e-12):
    G = R.shape[0]
    return (np.abs(R - R.T).max() <= tol
            and np.abs(R @ R.T - np.eye(G)).max() <= tol)


def pin_quantizer_rows(quantize_rows):
    for case in load_quantizer_rows():
        if "qmax" in case:
            Q, s, v, _ = quantize_rows(np.array([case["row"]]), case["qmax"])
        else:
            Q, s, v, _ = quantize_rows(np.array([case["row"]]))
        if not (np.array_equal(Q[0].astype(np.int64), np.array(case["q"], dtype=np.int64))
                and float(s[0]) == case["s"][0]):
            return False
    return True


def pin_rht_basis(rht_block, B=16, seed=3):
    """x -> H (D x) / sqrt(B): e_0 maps to s_0 * (1, ..., 1) / sqrt(B), and
    e_j to s_j times column j of the Walsh-Hadamard matrix over sqrt(B)."""
    rng = np.random.default_rng(seed)
    signs = rng.choice([-1.0, 1.0], size=B)
    T = rht_block(B, signs)
    H = O.sylvester_hadamard(B)
    for j in range(B):
        e = np.zeros(B)
        e[j] = 1.0
        if np.abs(T @ e - signs[j] * H[:, j] / np.sqrt(B)).max() > 1e-15:
            return False
    return True


def pin_rht_row_orientation(rotate_rows):
    """Rows rotated by the block randomized Hadamard transform hold the
    numbers of R x with R = H D / sqrt(B) (gemma.cpp issue, "Rotation
    method", where R acts on the vectors a and b): the hand-worked rows of
    tests/golden/rht_basis_rows.txt for every basis row e_j."""
    for B, signs, rows in load_rht_basis_rows():
        if rows.shape != (B, B):
            return False
        for j in range(B):
            e = np.zeros((1, B))
            e[0, j] = 1.0
            got = rotate_rows(e, B, "rht", signs)[0] * np.sqrt(B)
            if np.abs(got - rows[j]).max() > 1e-12:
                return False
    return True


# -------------------------------------------------------------- H4 and R --

def test_h4_is_the_printed_matrix():
    assert np.array_equal(O.H4, load_printed_h4())


def test_h4_orthogonal_symmetric():
    assert pin_orthogonal_symmetric(O.H4, tol=0.0)


@pytest.mark.parametrize("G", [4, 16, 64, 256, 1024])
def test_regular_hadamard_matches_digit_closed_form(G):
    assert np.array_equal(O.regular_hadamard(G), closed_form_R(G))


@pytest.mark.parametrize("G", [4, 16, 64, 256, 1024, 4096])
def test_regular_hadamard_orthogonal_symmetric(G):
    R = O.regular_hadamard(G)
    assert pin_orthogonal_symmetric(R)
    assert np.all(np.abs(R) == 1.0 / np.sqrt(G))


@pytest.mark.parametrize("G", [4, 16, 64, 256, 1024])
def test_regular_hadamard_invariants(G):
    R = O.regular_hadamard(G)
    # every row of H4 sums to (1 + 1 + 1 - 1) / 2 = 1, so R fixes the all-ones vector
    assert np.abs(R @ np.ones(G) - np.ones(G)).max() < 1e-12
    # trace(H4) = 2, trace of a Kronecker power = product of traces = 2**n = sqrt(G)
    assert abs(np.trace(R) - np.sqrt(G)) < 1e-9
    # symmetric involution: eigenvalues +-1, (G + trace) / 2 of them equal to +1
    ev = np.linalg.eigvalsh(R)
    assert np.abs(np.abs(ev) - 1).max() < 1e-9
    assert int(np.sum(ev > 0)) == (G + int(round(np.sqrt(G)))) // 2


def test_group_validation():
    with pytest.raises(ValueError):
        O.check_group(256, 8, "h4")       # not a power of four
    with pytest.raises(ValueError):
        O.check_group(2688, 256, "h4")    # does not divide K
    with pytest.raises(ValueError):
        O.check_group(1152, 96, "rht")    # not a power of two
    O.check_group(2688, 64, "h4")
    O.check_group(1152, 128, "rht")
    O.check_group(100, 0, "none")


# -------------------------------------------------------------- rotation --

@pytest.mark.parametrize("G", [16, 64, 256])
def test_basis_vector_quantizes_to_pm127(G):
    """X = e_j: X_rot is row j of R (all +-1/sqrt(G)) inside its group, so
    s = (1/sqrt(G))/127 and every code of that group is +-127 with the sign
    pattern of the closed form; every other group stays 0."""
    K = 4 * G
    for j in [0, 1, G - 1, G + 5, 3 * G + G // 2]:
        X = np.zeros((1, K))
        X[0, j] = 1.0
        Q, s, v = O.quantize_act(X, G)
        g0 = (j // G) * G
        expect = np.zeros(K, dtype=np.int64)
        expect[g0:g0 + G] = np.sign(closed_form_R(G)[j - g0]).astype(np.int64) * 127
        assert np.array_equal(Q[0].astype(np.int64), expect)
        assert s[0] == np.float32((1.0 / np.sqrt(G)) / 127.0)


def test_constant_group_is_unchanged():
    """R fixes the all-ones vector, so a row constant within each group is
    returned unchanged by the rotation."""
    X = np.repeat(np.array([[3.0, -1.0, 0.5, 7.0]]), 256, axis=1)
    assert np.abs(O.rotate_rows(X, 256) - X).max() < 1e-12


@pytest.mark.parametrize("transform,G", [("h4", 16), ("h4", 256), ("h4", 1024), ("rht", 128)])
def test_rotation_preserves_products(transform, G):
    """X_rot W_rot^T = X R R^T W^T = X W^T ("How INT8 convrot works";
    gemma.cpp "Rotation method"), in fp64 to 1e-12 relative."""
    rng = np.random.default_rng(0)
    K = 2 * G if G >= 256 else 8 * G
    X = rng.standard_normal((7, K))
    W = rng.standard_normal((5, K))
    signs = rng.choice([-1, 1], size=G) if transform == "rht" else None
    lhs = O.rotate_rows(X, G, transform, signs) @ O.rotate_rows(W, G, transform, signs).T
    rhs = X @ W.T
    assert np.abs(lhs - rhs).max() <= 1e-12 * np.abs(rhs).max()


def test_rotation_acts_on_each_group_independently():
    rng = np.random.default_rng(1)
    X = rng.standard_normal((3, 3 * 64))
    full = O.rotate_rows(X, 64)
    for g in range(3):
        part = O.rotate_rows(X[:, g * 64:(g + 1) * 64], 64)
        assert np.abs(full[:, g * 64:(g + 1) * 64] - part).max() <= 1e-14


def test_sylvester_matches_scipy():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    for B in [2, 8, 128, 512]:
        assert np.array_equal(O.sylvester_hadamard(B), scipy_linalg.hadamard(B).astype(float))


def test_rht_step_order_and_orthogonality():
    assert pin_rht_basis(O.rht_block)
    rng = np.random.default_rng(2)
    signs = rng.choice([-1, 1], size=128)
    T = O.rht_block(128, signs)
    assert np.abs(T @ T.T - np.eye(128)).max() < 1e-12


def test_rht_row_orientation_hand_rows():
    """The orientation of the rotation on row-major rows: e_j becomes
    s_j H[:, j] / sqrt(B), worked out by hand for B = 4 and 8. Both
    orientations are orthogonal, so only such a pin tells them apart."""
    assert len(load_rht_basis_rows()) == 2
    assert pin_rht_row_orientation(O.rotate_rows)


def test_none_transform_is_identity():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((4, 96))
    assert np.array_equal(O.rotate_rows(X, 0, "none"), X)


# ------------------------------------------------------------- quantizer --

def test_quantizer_hand_rows():
    assert pin_quantizer_rows(O.quantize_rows)


def test_quantizer_extremes():
    rng = np.random.default_rng(4)
    X = rng.standard_normal((50, 300)) * np.exp(rng.standard_normal((50, 1)) * 3)
    Q, s, v, s64 = O.quantize_rows(X)
    assert Q.min() >= -127 and Q.max() <= 127
    # the row maximum maps to exactly +-127
    i = np.abs(X).argmax(axis=1)
    assert np.all(np.abs(Q[np.arange(50), i]) == 127)
    assert np.all(s == s64.astype(np.float32))
    # |Q - v| <= 1/2 everywhere (round to nearest)
    assert np.abs(Q - v).max() <= 0.5


# ----------------------------------------------------------- integer GEMM --

def test_int_gemm_brute_force():
    rng = np.random.default_rng(5)
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (4, 3, 64), (2, 2, 300)]:
        Qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
        Qw = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
        A = O.int_gemm(Qx, Qw)
        for r, o in itertools.product(range(M), range(N)):
            acc = 0
            for i in range(K):
                acc += int(Qx[r, i]) * int(Qw[o, i])
            assert A[r, o] == acc


def test_int_gemm_all_127_closed_form():
    for K in [1024, 1040, 6144]:
        Qx = np.full((2, K), 127, dtype=np.int8)
        Qw = np.full((3, K), 127, dtype=np.int8)
        Qw[1] = -127
        A = O.int_gemm(Qx, Qw)
        assert np.all(A[:, 0] == 16129 * K)
        assert np.all(A[:, 1] == -16129 * K)


# -------------------------------------------------------- reconstruction --

def test_reconstruct_hand_values():
    A = np.array([[100, -3], [0, 16129]])
    sx = np.array([0.5, 2.0], dtype=np.float32)
    sw = np.array([0.25, 4.0], dtype=np.float32)
    b = np.array([1.0, -1.0])
    Y = O.reconstruct(A, sx, sw, b)
    assert np.array_equal(Y, np.array([[100 * 0.125 + 1, -3 * 2.0 - 1], [1.0, 16129 * 8.0 - 1]]))


def test_round_to_bf16_matches_torch_on_fp32_values():
    """For values that are exactly fp32, rounding fp32 -> bf16 is a single
    rounding, so torch's conversion is a valid library reference."""
    g = torch.Generator().manual_seed(6)
    x = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 4)
    # add exact ties: low 16 bits == 0x8000
    bits = x[:2000].view(torch.int32) & ~0xFFFF | 0x8000
    x = torch.cat([x, bits.view(torch.float32)])
    ours = O.round_to_bf16(x.double().numpy())
    ref = x.to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------ properties --

def test_linear_row_split_is_bit_identical():
    rng = np.random.default_rng(7)
    X = rng.standard_normal((37, 256))
    W = rng.standard_normal((19, 256))
    Qw, sw, _ = O.prepare_weights(W, 64)
    whole = O.linear(X, Qw, sw, None, 64)["Y"]
    parts = np.concatenate([O.linear(X[a:a + 10], Qw, sw, None, 64)["Y"] for a in range(0, 37, 10)])
    assert np.array_equal(whole, parts)


def _rel_err(Y, ref):
    return np.abs(Y - ref).max() / np.abs(ref).max()


def test_rotation_reduces_error_on_outlier_rows():
    """Direction only ("How INT8 convrot works": the rotation spreads isolated
    large values; gemma.cpp: rotated W8A8 is closer to the control)."""
    rng = np.random.default_rng(8)
    M, K, N = 64, 1024, 128
    X = rng.standard_normal((M, K))
    X[:, rng.choice(K, 4, replace=False)] *= 50
    W = rng.standard_normal((N, K)) * 0.02
    ref = O.float_linear(X, W)
    errs = {}
    for t, G in [("h4", 256), ("rht", 128), ("none", 0)]:
        signs = rng.choice([-1, 1], size=G) if t == "rht" else None
        Qw, sw, _ = O.prepare_weights(W, G, t, signs)
        errs[t] = _rel_err(O.linear(X, Qw, sw, None, G, t, signs)["Y64"], ref)
    assert errs["h4"] < errs["none"] / 2
    assert errs["rht"] < errs["none"] / 2


def test_missing_rotation_gives_noise():
    """Un-rotated dequantized weights correlate with W; used as-is they do
    not (the stable-diffusion.cpp PR, "Verification": 0.06 as-is vs
    0.954-0.993 after un-rotation; synthetic data here, direction only)."""
    rng = np.random.default_rng(9)
    W = rng.standard_normal((64, 512)) * 0.02
    Qw, sw, _ = O.prepare_weights(W, 256)
    deq = Qw.astype(np.float64) * sw[:, None]
    unrot = O.rotate_rows(deq, 256)  # R is symmetric and orthogonal: R^-1 = R
    c_asis = np.corrcoef(deq.ravel(), W.ravel())[0, 1]
    c_unrot = np.corrcoef(unrot.ravel(), W.ravel())[0, 1]
    assert abs(c_asis) < 0.2 and c_unrot > 0.99


def test_boundary_distance():
    d = O.boundary_distance(np.array([0.5, 1.0, -2.5, 2.499, -0.75]))
    assert np.allclose(d, [0.0, 0.5, 0.0, 0.001, 0.25])


# ----------------------------------------------------- row-parallel split --
# sglang digest, "风险与影响": tensor parallelism splits the rotated input
# dimension over ranks, each slice a whole number of groups.

def pin_given_max_rows(quantize_rows_given):
    for case in load_given_max_rows():
        Q, s, v, _ = quantize_rows_given(np.array([case["row"]]), np.array(case["amax"]))
        if not (np.array_equal(Q[0].astype(np.int64), np.array(case["q"], dtype=np.int64))
                and float(s[0]) == case["s"][0]):
            return False
    return True


def sharded_linear(X, Qw, sw, bias, G, shards, combine_max=True):
    """The row-parallel evaluation of the layer, step by step: every slice is
    rotated alone, the row maxima are combined by max (the all-reduce), every
    slice is quantized with them, the int32 partial products are summed (the
    all-reduce) and the output is reconstructed once."""
    K = X.shape[1]
    w = K // shards
    sl = [slice(i * w, (i + 1) * w) for i in range(shards)]
    rot = [O.rotate_rows(X[:, c], G, "h4") for c in sl]
    maxima = [O.row_absmax(r) for r in rot]
    parts = []
    for r, c, m in zip(rot, sl, maxima):
        amax = np.maximum.reduce(maxima) if combine_max else m
        Q, sx, _, _ = O.quantize_rows_given(r, amax)
        parts.append((Q, sx, O.int_gemm(Q, Qw[:, c])))
    A = sum(p[2] for p in parts)
    return np.concatenate([p[0] for p in parts], axis=1), parts[0][1], A, O.reconstruct(A, parts[0][1], sw, bias)


def test_row_absmax_and_given_max_hand_rows():
    assert len(load_given_max_rows()) == 3
    assert pin_given_max_rows(O.quantize_rows_given)
    assert np.array_equal(O.row_absmax(np.array([[1.0, -3.0, 2.0], [0.0, 0.0, 0.0]])), [3.0, 0.0])


def test_given_max_of_the_row_itself_is_the_plain_quantizer():
    rng = np.random.default_rng(21)
    X = rng.standard_t(3, size=(50, 256)) * np.where(rng.random(256) < 0.01, 50.0, 1.0)
    X[3] = 0.0
    a, b = O.quantize_rows_given(X, O.row_absmax(X)), O.quantize_rows(X)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("shards,G", [(2, 256), (4, 64), (3, 16)])
def test_row_parallel_split_reproduces_the_whole_row(shards, G):
    """Whole groups per slice: rotating a slice alone gives that slice of the
    whole row's rotation (R is block-diagonal), so with the combined maximum
    the codes, the scales, the int32 accumulators and Y are exactly those of
    the layer on the whole row."""
    rng = np.random.default_rng(shards * G)
    K = 1536
    X = rng.standard_t(3, size=(20, K)) * np.where(rng.random(K) < 0.01, 50.0, 1.0)
    W = rng.normal(0, 0.02, size=(40, K))
    b = rng.normal(0, 0.01, size=40)
    Qw, sw, _ = O.prepare_weights(W, G, "h4")
    whole = O.linear(X, Qw, sw, b, G, "h4")
    Q, sx, A, Y = sharded_linear(X, Qw, sw, b, G, shards)
    assert np.array_equal(Q, whole["Qx"]) and np.array_equal(sx, whole["sx"])
    assert np.array_equal(A, whole["A"]) and np.array_equal(Y, whole["Y64"])
    w = K // shards
    assert np.array_equal(O.rotate_rows(X[:, w:2 * w], G, "h4"), O.rotate_rows(X, G, "h4")[:, w:2 * w])


def test_row_parallel_slice_must_hold_whole_groups():
    # a slice of 384 values cuts a group of 256 (the constraint the digest names)
    with pytest.raises(ValueError):
        O.rotate_rows(np.zeros((2, 384)), 256, "h4")


def test_planted_slice_local_maximum_is_caught():
    # quantizing every slice with its own maximum (no all-reduce) changes the
    # codes and the output: the whole-row comparison rejects it
    rng = np.random.default_rng(5)
    X = rng.standard_t(3, size=(20, 512))
    X[:, 7] *= 50.0  # one large channel in the first slice only
    W = rng.normal(0, 0.02, size=(16, 512))
    Qw, sw, _ = O.prepare_weights(W, 256, "h4")
    whole = O.linear(X, Qw, sw, None, 256, "h4")
    Q, _, A, _ = sharded_linear(X, Qw, sw, None, 256, 2, combine_max=False)
    assert not np.array_equal(Q, whole["Qx"]) and not np.array_equal(A, whole["A"])
    wrong = lambda Xr, amax: O.quantize_rows(Xr)  # ignores the given maximum
    assert not pin_given_max_rows(wrong)


# ----------------------------------------------------- planted mistakes --
# Mutated copies of oracle parts; each pin above must reject them.

def test_planted_sign_error_in_h4_is_caught():
    bad = O.H4.copy()
    bad[1, 2] = -bad[1, 2]
    assert not pin_orthogonal_symmetric(bad)
    assert not np.array_equal(bad, load_printed_h4())


def test_planted_wrong_digit_rule_is_caught():
    R = O.regular_hadamard(16)
    wrong = closed_form_R(16).copy()
    wrong[3, 3] = -wrong[3, 3]
    assert not np.array_equal(R, wrong)


def test_planted_transposed_rht_is_caught():
    # D H / sqrt(B) instead of H D / sqrt(B): still orthogonal, but the basis pin rejects it
    def rht_swapped(B, signs):
        return np.diag(np.asarray(signs, float)) @ O.sylvester_hadamard(B) / np.sqrt(B)
    assert not pin_rht_basis(rht_swapped)


def test_planted_rht_row_orientation_is_caught():
    # rows multiplied by R instead of R^T (x R in place of R x): orthogonal
    # too, and every other pin passes; the hand-worked rows reject it
    def rotate_wrong(X, G, transform, signs=None):
        X = np.asarray(X, dtype=np.float64)
        rows, K = X.shape
        return (X.reshape(rows, K // G, G) @ O.rht_block(G, signs)).reshape(rows, K)
    assert pin_rht_row_orientation(O.rotate_rows)
    assert not pin_rht_row_orientation(rotate_wrong)


def test_planted_rounding_errors_are_caught():
    def q_floor(X):
        X = np.asarray(X, float)
        s64 = np.abs(X).max(axis=1) / 127
        safe = np.where(s64 > 0, s64, 1)
        v = X / safe[:, None]
        return np.clip(np.floor(v + 0.5), -127, 127).astype(np.int8), s64.astype(np.float32), v, s64

    def q_scale_128(X):
        X = np.asarray(X, float)
        s64 = np.abs(X).max(axis=1) / 128
        safe = np.where(s64 > 0, s64, 1)
        v = X / safe[:, None]
        return np.clip(np.rint(v), -127, 127).astype(np.int8), s64.astype(np.float32), v, s64

    assert not pin_quantizer_rows(q_floor)       # half-up instead of half-even
    assert not pin_quantizer_rows(q_scale_128)   # wrong denominator


def test_planted_dropped_term_in_gemm_is_caught():
    rng = np.random.default_rng(10)
    Qx = rng.integers(-127, 128, size=(3, 40)).astype(np.int8)
    Qw = rng.integers(-127, 128, size=(2, 40)).astype(np.int8)
    bad = (Qx[:, :-1].astype(np.int64) @ Qw[:, :-1].astype(np.int64).T)
    good = O.int_gemm(Qx, Qw)
    brute = np.array([[sum(int(Qx[r, i]) * int(Qw[o, i]) for i in range(40)) for o in range(2)]
                      for r in range(3)])
    assert np.array_equal(good, brute) and not np.array_equal(bad, brute)


# ------------------------------------------------------------ 4-bit codes --
# "feat: load ConvRot int4 and per-channel int8 safetensors", "Solution":
# int4 values occupy [-7, 7], adjacent pairs packed in a byte (nibble order
# and two's-complement nibbles are a reading of that section, pinned here).

def pin_int4_bytes(pack):
    # codes (1, -1) -> low nibble 0x1, high nibble 0xF; (7, -7) -> 0x7, 0x9;
    # (0, 3) -> 0x0, 0x3; (-4, 5) -> 0xC, 0x5
    got = pack(np.array([[1, -1, 7, -7, 0, 3, -4, 5]], dtype=np.int8))
    return np.array_equal(got, np.array([[0xF1, 0x97, 0x30, 0x5C]], dtype=np.uint8))


def test_int4_packing_hand_bytes():
    assert pin_int4_bytes(O.pack_int4)


def test_int4_pack_round_trip_and_range():
    rng = np.random.default_rng(4)
    Q = rng.integers(-7, 8, size=(5, 64)).astype(np.int8)
    P = O.pack_int4(Q)
    assert P.shape == (5, 32) and P.dtype == np.uint8
    assert np.array_equal(O.unpack_int4(P), Q)
    with pytest.raises(ValueError):
        O.pack_int4(np.array([[8, 0]], dtype=np.int8))
    with pytest.raises(ValueError):
        O.pack_int4(np.array([[1, 2, 3]], dtype=np.int8))


def test_4bit_quantizer_range_and_scale():
    """Every 4-bit code is within [-7, 7]; the largest |x_rot| of a row maps to
    exactly +-7; a basis vector in a G = 256 group maps to +-7 everywhere."""
    rng = np.random.default_rng(5)
    X = rng.standard_t(3, size=(9, 1024))
    Q, s, v = O.quantize_act(X, 256, "h4", qmax=O.QMAX4)
    assert np.abs(Q).max() == 7 and np.all(np.abs(Q).max(axis=1) == 7)
    Xr = O.rotate_rows(X, 256, "h4")
    assert np.allclose(s, np.abs(Xr).max(axis=1) / 7, rtol=1e-7)
    e = np.zeros((1, 256))
    e[0, 17] = 3.0
    Qe, _, _ = O.quantize_act(e, 256, "h4", qmax=O.QMAX4)
    assert np.all(np.abs(Qe) == 7)


def test_planted_int4_nibble_swap_is_caught():
    def swapped(Q):
        Q = np.asarray(Q)
        return ((Q[..., 1::2].astype(np.int64) & 0xF) | ((Q[..., 0::2].astype(np.int64) & 0xF) << 4)).astype(np.uint8)
    assert not pin_int4_bytes(swapped)


def test_planted_int4_offset_binary_is_caught():
    def biased(Q):  # +8 offset nibbles instead of two's complement
        Q = np.asarray(Q).astype(np.int64) + 8
        return (Q[..., 0::2] | (Q[..., 1::2] << 4)).astype(np.uint8)
    assert not pin_int4_bytes(biased)
