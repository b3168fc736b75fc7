"""Parity of the int8 GEMM + fused epilogue with the CPU oracle.

The accumulators must be bit-exact when the GPU is fed the oracle's codes;
Y from those codes must match the oracle's fp64 reconstruction within one
bf16 ulp; end to end from X, Y must be within 1e-2 of max|Y|. Every check
runs on both GEMM paths: the tensor-core path (fp16 operand copies given)
and the int8 warp-MMA path (no copies)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import check_codes, check_y_e2e, check_y_same_codes, to_np

pytestmark = pytest.mark.gpu

PATHS = ["tc", "mma"]


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def packed_from_codes(cr, Q, s, G, transform, f16, kind):
    q = torch.from_numpy(np.ascontiguousarray(Q)).cuda()
    sc = torch.from_numpy(np.ascontiguousarray(s.astype(np.float32))).cuda()
    q16 = q.to(torch.float16) if f16 else None
    t = cr.TRANSFORMS[transform]
    cls = cr.PackedAct if kind == "act" else cr.PackedWeight
    return cls(q, sc, q16, G, t)


def oracle_case(wl, i=0):
    sg = None if wl.signs is None else wl.signs.numpy()
    X64 = wl.X.float().numpy().astype(np.float64)
    W64 = wl.weights[i].numpy().astype(np.float64)
    Qw, sw, _ = O.prepare_weights(W64, wl.group, wl.transform, sg)
    Qx, sx, v = O.quantize_act(X64, wl.group, wl.transform, sg)
    return Qx, sx, v, Qw, sw


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,N,K", [(64, 256, 256), (200, 384, 1024), (129, 300, 3072), (16, 1000, 1152),
                                   (1, 64, 256), (300, 128, 6144), (257, 136, 2688), (3, 40, 80),
                                   (33, 100, 1040), (48, 13824, 1152), (16, 96, 6144)])
def test_gemm_s32_bit_exact_on_oracle_codes(cr, path, M, N, K):
    rng = np.random.default_rng(M + N + K)
    Qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    Qw = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    a = packed_from_codes(cr, Qx, np.ones(M), 0, "none", path == "tc", "act")
    w = packed_from_codes(cr, Qw, np.ones(N), 0, "none", path == "tc", "w")
    A = to_np(cr.convrot_gemm_s32(a, w, int8_mma=path == "mma"))
    assert np.array_equal(A.astype(np.int64), O.int_gemm(Qx, Qw))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("K", [1024, 1040, 3072, 6144])
def test_gemm_s32_adversarial_magnitudes(cr, path, K):
    """All-127 rows give |A| = 16129 K, far above 2^24 for K = 6144: any
    accumulation that is not exact over the whole K shows up here. Mixed
    rows put large and small partial sums next to each other."""
    M, N = 130, 136
    Qx = np.full((M, K), 127, dtype=np.int8)
    Qx[1::2] = -127
    Qx[2::5, ::3] = 1
    Qw = np.full((N, K), 127, dtype=np.int8)
    Qw[3::4] = -127
    Qw[5::7, 1::2] = -1
    a = packed_from_codes(cr, Qx, np.ones(M), 0, "none", path == "tc", "act")
    w = packed_from_codes(cr, Qw, np.ones(N), 0, "none", path == "tc", "w")
    A = to_np(cr.convrot_gemm_s32(a, w, int8_mma=path == "mma")).astype(np.int64)
    ref = O.int_gemm(Qx, Qw)
    assert np.array_equal(A, ref)
    assert np.abs(ref).max() == 16129 * K


@pytest.mark.parametrize("M,K,path", [(300, 32768, "tc"), (300, 32768, "mma"), (40, 32768, "tc"), (8, 32768, "tc"),
                                      (40, 8192, "tc")])
def test_gemm_s32_at_the_largest_k(cr, M, K, path):
    """K up to the largest the library accepts (CONVROT_MAX_K = 32768): all-127
    rows give |A| = 16129 K = 5.3e8, exact in int32 on every route (the
    large-M tensor-core GEMM with 32 exact fp32 chunks per tile, the small-M
    weight stream, the small-M tensor-core kernel at K = 8192, and the int8
    warp MMA), with random rows between them."""
    N = 136
    rng = np.random.default_rng(M + K)
    Qx = np.full((M, K), 127, dtype=np.int8)
    Qx[1::2] = -127
    Qx[2::5, ::3] = 1
    Qx[3::7] = rng.integers(-127, 128, size=Qx[3::7].shape, dtype=np.int8)
    Qw = np.full((N, K), 127, dtype=np.int8)
    Qw[3::4] = -127
    Qw[5::7, 1::2] = -1
    Qw[6::9] = rng.integers(-127, 128, size=Qw[6::9].shape, dtype=np.int8)
    a = packed_from_codes(cr, Qx, np.ones(M), 0, "none", path == "tc", "act")
    w = packed_from_codes(cr, Qw, np.ones(N), 0, "none", path == "tc", "w")
    A = to_np(cr.convrot_gemm_s32(a, w, int8_mma=path == "mma")).astype(np.int64)
    ref = O.int_gemm(Qx, Qw)
    assert np.abs(ref).max() == 16129 * K
    assert np.array_equal(A, ref)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", ["tiny", "dit", "ffn_rht", "g64_2688"])
def test_linear_on_oracle_codes(cr, path, case):
    wl = {"tiny": lambda: WL.tiny(),
          "dit": lambda: WL.dit6144(M=96),
          "ffn_rht": lambda: WL.ffn_pair(),
          "g64_2688": lambda: WL.k2688(M=70)}[case]()
    Qx, sx, v, Qw, sw = oracle_case(wl)
    a = packed_from_codes(cr, Qx, sx, wl.group, wl.transform, path == "tc", "act")
    w = packed_from_codes(cr, Qw, sw, wl.group, wl.transform, path == "tc", "w")
    bias = wl.biases[0]
    Y = cr.convrot_linear(a, w, bias.cuda(), int8_mma=path == "mma")
    A = O.int_gemm(Qx, Qw)
    assert np.array_equal(to_np(cr.convrot_gemm_s32(a, w, int8_mma=path == "mma")).astype(np.int64), A)
    check_y_same_codes(to_np(Y.float()), A, sx, sw, bias.numpy(), f"{case}/{path}")
    Y0 = cr.convrot_linear(a, w, None, int8_mma=path == "mma")
    check_y_same_codes(to_np(Y0.float()), A, sx, sw, None, f"{case}/{path}/nobias")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", ["tiny", "dit", "ffn_rht", "g16", "g1024"])
def test_linear_end_to_end(cr, path, case):
    wl = {"tiny": lambda: WL.tiny(),
          "dit": lambda: WL.dit6144(M=200),
          "ffn_rht": lambda: WL.ffn_pair(),
          "g16": lambda: WL.gsweep(16, M=130),
          "g1024": lambda: WL.gsweep(1024, M=130)}[case]()
    f16 = path == "tc"
    sg = None if wl.signs is None else wl.signs.cuda()
    pw = cr.convrot_prepare_weights(wl.weights[0].cuda(), wl.group, wl.transform, sg, with_f16=f16)
    a = cr.convrot_quantize_act(wl.X.cuda(), wl.group, wl.transform, sg, with_f16=f16)
    Y = cr.convrot_linear(a, pw, wl.biases[0].cuda(), int8_mma=path == "mma")
    Qx, sx, v, Qw, sw = oracle_case(wl)
    ref = O.reconstruct(O.int_gemm(Qx, Qw), sx, sw, wl.biases[0].numpy())
    check_codes(to_np(a.q), Qx, v, case)
    check_y_e2e(to_np(Y.float()), ref, case)


@pytest.mark.parametrize("path", PATHS)
def test_linear_multi_equals_separate_calls_and_concatenation(cr, path):
    wl = WL.qkv32700(M=300)
    f16 = path == "tc"
    a = cr.convrot_quantize_act(wl.X.cuda(), 256, "h4", with_f16=f16)
    ws = [cr.convrot_prepare_weights(W.cuda(), 256, "h4", with_f16=f16) for W in wl.weights]
    bs = [b.cuda() for b in wl.biases]
    Ys = cr.convrot_linear_multi(a, ws, bs, int8_mma=path == "mma")
    for Y, w, b in zip(Ys, ws, bs):
        assert torch.equal(Y, cr.convrot_linear(a, w, b, int8_mma=path == "mma"))
    cat = cr.PackedWeight(torch.cat([w.q for w in ws]), torch.cat([w.scale for w in ws]),
                          torch.cat([w.q_f16 for w in ws]) if f16 else None, 256, 0)
    Ycat = cr.convrot_linear(a, cat, torch.cat(bs), int8_mma=path == "mma")
    assert torch.equal(Ycat, torch.cat(Ys, dim=1))


@pytest.mark.parametrize("path", PATHS)
def test_row_split_is_bit_identical(cr, path):
    """Every row's arithmetic is the same however the rows are split (the
    sglang digest's row split of large-M calls)."""
    wl = WL.dit6144(M=300)
    f16 = path == "tc"
    pw = cr.convrot_prepare_weights(wl.weights[0][:512].cuda(), 256, "h4", with_f16=f16)
    X = wl.X.cuda()
    full = cr.convrot_linear(cr.convrot_quantize_act(X, 256, "h4", with_f16=f16), pw, int8_mma=path == "mma")
    parts = [cr.convrot_linear(cr.convrot_quantize_act(X[r:r + 100], 256, "h4", with_f16=f16), pw, int8_mma=path == "mma")
             for r in range(0, 300, 100)]
    assert torch.equal(full, torch.cat(parts))


def test_paths_agree(cr):
    wl = WL.dit6144(M=257)
    pw = cr.convrot_prepare_weights(wl.weights[0][:640].cuda(), 256, "h4", with_f16=True)
    a = cr.convrot_quantize_act(wl.X.cuda(), 256, "h4", with_f16=True)
    a_int8 = cr.PackedAct(a.q, a.scale, None, a.group, a.transform)
    assert torch.equal(cr.convrot_gemm_s32(a, pw), cr.convrot_gemm_s32(a_int8, pw, int8_mma=True))
    assert torch.equal(cr.convrot_linear(a, pw), cr.convrot_linear(a_int8, pw, int8_mma=True))
    # without the activation's fp16 copy the tensor-core path is not silently replaced
    with pytest.raises(cr.ConvRotError, match="fp16 operand copies"):
        cr.convrot_linear(a_int8, pw)


def test_output_stride_and_empty(cr):
    wl = WL.dit6144(M=40)
    pw = cr.convrot_prepare_weights(wl.weights[0][:200].cuda(), 256, "h4")
    a = cr.convrot_quantize_act(wl.X.cuda(), 256, "h4")
    big = torch.full((40, 264), 7.0, dtype=torch.bfloat16, device="cuda")
    Y = cr.convrot_linear(a, pw, out=big[:, :200])
    assert torch.equal(Y, cr.convrot_linear(a, pw))
    assert torch.all(big[:, 200:] == 7.0)
    e = cr.convrot_quantize_act(torch.empty((0, 6144), dtype=torch.bfloat16, device="cuda"), 256, "h4")
    assert cr.convrot_linear(e, pw).shape == (0, 200)


def test_convrot_linear_module_flattens_leading_dims(cr):
    wl = WL.dit6144(M=64)
    lin = cr.ConvRotLinear.from_float(wl.weights[0][:256].cuda(), wl.biases[0][:256], 256)
    x = wl.X.cuda().reshape(4, 16, 6144)
    y = lin(x)
    assert y.shape == (4, 16, 256)
    assert torch.equal(y.reshape(64, 256), lin(wl.X.cuda()))
    with pytest.raises(TypeError):
        cr.ConvRotLinear.from_float(torch.zeros((4, 256), dtype=torch.int8), None, 256)


@pytest.mark.parametrize("name", ["dit6144", "qkv32700"])
def test_full_size_sampled_outputs(cr, name):
    """Full-size workloads in the bench's launch configuration; the oracle
    checks a seeded sample of (row, column) outputs from the GPU's own codes
    (bit-exact accumulators) and from X (end-to-end bound)."""
    wl = WL.dit6144() if name == "dit6144" else WL.qkv32700()
    a = cr.convrot_quantize_act(wl.X.cuda(), wl.group, "h4")
    ws = [cr.convrot_prepare_weights(W.cuda(), wl.group, "h4") for W in wl.weights]
    Ys = cr.convrot_linear_multi(a, ws, [b.cuda() for b in wl.biases])
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([rng.choice(wl.M, 256, replace=False), np.arange(wl.M - 40, wl.M)]))
    qx = to_np(a.q)[rows].astype(np.int8)
    sx = to_np(a.scale)[rows]
    X64 = wl.X[torch.from_numpy(rows)].float().numpy().astype(np.float64)
    Qx_or, sx_or, v = O.quantize_act(X64, wl.group, "h4")
    check_codes(qx, Qx_or, v, name)
    for i, (W, b, Y) in enumerate(zip(wl.weights, wl.biases, Ys)):
        cols = np.unique(np.concatenate([rng.choice(W.shape[0], 256, replace=False),
                                         np.arange(W.shape[0] - 8, W.shape[0])]))
        qw = to_np(ws[i].q)[cols].astype(np.int8)
        sw = to_np(ws[i].scale)[cols]
        A = O.int_gemm(qx, qw)
        Ys_np = to_np(Y.float())[np.ix_(rows, cols)]
        check_y_same_codes(Ys_np, A, sx, sw, b.numpy()[cols], f"{name}[{i}]")
        W64 = W.numpy().astype(np.float64)[cols]
        Qw_or, sw_or, _ = O.prepare_weights(W64, wl.group, "h4")
        ref = O.reconstruct(O.int_gemm(Qx_or, Qw_or), sx_or, sw_or, b.numpy()[cols])
        check_y_e2e(Ys_np, ref, f"{name}[{i}] e2e")


@pytest.mark.parametrize("M,N", [(1024, 4608), (4096, 4096), (300, 2688)])
def test_every_column_tile_width_is_exact(cr, M, N):
    """Shapes on which the library's tile chooser picks each of its column
    widths on the pair (2-SM) path (256, 224 and 192 columns respectively);
    the raw accumulators must be bit-exact against the oracle."""
    rng = np.random.default_rng(M + N)
    K = 1024
    Qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    Qw = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    a = packed_from_codes(cr, Qx, np.ones(M), 0, "none", True, "act")
    w = packed_from_codes(cr, Qw, np.ones(N), 0, "none", True, "w")
    A = to_np(cr.convrot_gemm_s32(a, w)).astype(np.int64)
    assert np.array_equal(A, O.int_gemm(Qx, Qw))


def test_small_m_multi_equals_separate_calls(cr):
    """The gated-FFN pair at M = 16 (weight-stream path): one launch for both
    linears gives exactly what two separate linears give."""
    wl = WL.ffn_pair()
    sg = wl.signs.cuda()
    a = cr.convrot_quantize_act(wl.X.cuda(), wl.group, wl.transform, sg, with_f16=False)
    ws = [cr.convrot_prepare_weights(W.cuda(), wl.group, wl.transform, sg, with_f16=False) for W in wl.weights]
    bs = [b.cuda() for b in wl.biases]
    Ys = cr.convrot_linear_multi(a, ws, bs)
    for Y, w, b in zip(Ys, ws, bs):
        assert torch.equal(Y, cr.convrot_linear(a, w, b))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("N,ld", [(1000, None), (24, None), (8, None), (200, 264), (1000, 1008)])
def test_epilogue_ragged_columns_and_row_pitch(cr, path, N, ld):
    """Large-M outputs whose width is not a multiple of the tile or of the
    16-column store piece (or narrower than one piece), written densely or
    into a wider buffer. Columns past N stay untouched."""
    M, K = 333, 1024
    rng = np.random.default_rng(N + (ld or 0))
    Qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    Qw = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    sx = rng.uniform(0.5, 2.0, M) / 127.0
    sw = rng.uniform(0.5, 2.0, N) / 127.0
    bias = rng.normal(0, 0.5, N).astype(np.float32)
    a = packed_from_codes(cr, Qx, sx, 0, "none", path == "tc", "act")
    w = packed_from_codes(cr, Qw, sw, 0, "none", path == "tc", "w")
    A = O.int_gemm(Qx, Qw)
    if ld is None:
        Y = cr.convrot_linear(a, w, torch.from_numpy(bias).cuda(), int8_mma=path == "mma")
    else:
        big = torch.full((M, ld), 7.0, dtype=torch.bfloat16, device="cuda")
        Y = cr.convrot_linear(a, w, torch.from_numpy(bias).cuda(), out=big[:, :N], int8_mma=path == "mma")
        assert torch.all(big[:, N:] == 7.0)
    check_y_same_codes(to_np(Y.float()), A, sx.astype(np.float32), sw.astype(np.float32), bias, f"{path}/{N}/{ld}")


def test_row_pitch_not_multiple_of_8_is_rejected(cr):
    M, K, N = 96, 1024, 200
    a = packed_from_codes(cr, np.ones((M, K), np.int8), np.ones(M), 0, "none", True, "act")
    w = packed_from_codes(cr, np.ones((N, K), np.int8), np.ones(N), 0, "none", True, "w")
    big = torch.zeros((M, 203), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cr.ConvRotError, match="ALIGNMENT"):
        cr.convrot_linear(a, w, out=big[:, :N])
    assert torch.all(big == 0)


@pytest.mark.parametrize("M,N", [(300, 1000), (1024, 5120), (129, 1000), (100, 1000)])
def test_split_last_round_is_bit_exact(cr, M, N):
    """With a workspace the tensor-core GEMM splits a mostly idle last round
    of tiles along K (on these shapes for every column width it may pick, on
    the pair path and, for M = 100, the single-CTA path). The accumulators
    must equal the oracle's and the unsplit run's, twice in a row on the same
    workspace, and the workspace must be left all zero."""
    K = 1024
    rng = np.random.default_rng(7 * M + N)
    Qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    Qw = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    a = packed_from_codes(cr, Qx, np.ones(M), 0, "none", True, "act")
    w = packed_from_codes(cr, Qw, np.ones(N), 0, "none", True, "w")
    ws = cr.gemm_workspace()
    A1 = cr.convrot_gemm_s32(a, w, workspace=ws)
    A2 = cr.convrot_gemm_s32(a, w, workspace=ws)
    A0 = cr.convrot_gemm_s32(a, w)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    assert torch.equal(A1, A0) and torch.equal(A2, A0)
    assert np.array_equal(to_np(A1).astype(np.int64), O.int_gemm(Qx, Qw))


def test_split_adversarial_magnitudes(cr):
    """All-127 codes with K = 6144 (the largest partial sums) through split
    pieces: still exact."""
    M, N, K = 300, 1000, 6144
    Qx = np.full((M, K), 127, np.int8)
    Qw = np.full((N, K), 127, np.int8)
    Qw[::2] = -127
    a = packed_from_codes(cr, Qx, np.ones(M), 0, "none", True, "act")
    w = packed_from_codes(cr, Qw, np.ones(N), 0, "none", True, "w")
    ws = cr.gemm_workspace()
    A = to_np(cr.convrot_gemm_s32(a, w, workspace=ws)).astype(np.int64)
    assert np.array_equal(A, O.int_gemm(Qx, Qw))
    assert int(ws.count_nonzero()) == 0


def test_split_linear_multi_matches_unsplit(cr):
    """The bf16 linear through split tiles (three linears sharing one packed
    activation, ragged M): bit-identical to the unsplit run and within one
    bf16 ulp of the oracle's reconstruction."""
    wl = WL.qkv32700(M=129)
    a = cr.convrot_quantize_act(wl.X.cuda(), 256, "h4")
    wts = [cr.convrot_prepare_weights(W.cuda(), 256, "h4") for W in wl.weights]
    bs = [b.cuda() for b in wl.biases]
    ws = cr.gemm_workspace()
    Y1 = cr.convrot_linear_multi(a, wts, bs, workspace=ws)
    Y0 = cr.convrot_linear_multi(a, wts, bs)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    qx, sx = to_np(a.q).astype(np.int8), to_np(a.scale)
    for y1, y0, w, b in zip(Y1, Y0, wts, wl.biases):
        assert torch.equal(y1, y0)
        A = O.int_gemm(qx, to_np(w.q).astype(np.int8))
        check_y_same_codes(to_np(y1.float()), A, sx, to_np(w.scale), b.numpy(), "split multi")


def test_split_full_size_dit_matches_unsplit(cr):
    """The DiT linear at full size (4096 x 6144 x 6144), as the bench runs it
    with a workspace: bit-identical to the unsplit launch."""
    wl = WL.dit6144()
    a = cr.convrot_quantize_act(wl.X.cuda(), 256, "h4")
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), 256, "h4")
    b = wl.biases[0].cuda()
    ws = cr.gemm_workspace()
    Y1 = cr.convrot_linear(a, w, b, workspace=ws)
    Y0 = cr.convrot_linear(a, w, b)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    assert torch.equal(Y1, Y0)


@pytest.mark.parametrize("M,N,K", [(17, 296, 128), (24, 1000, 1152), (32, 13824, 1152), (33, 264, 4096),
                                   (48, 136, 2048), (64, 4096, 4096)])
def test_small_m_tensor_core_path_bit_exact(cr, M, N, K):
    """17..64 rows with K a multiple of 128 take the small-M tensor-core
    kernel (int8 tiles widened to fp16 on chip, swapped operands, one TMEM
    region per exact 1024-long chunk): accumulators bit-exact, and Y within
    one bf16 ulp of the oracle's reconstruction from the same codes."""
    rng = np.random.default_rng(3 * M + N + K)
    Qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    Qw = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    sx = (rng.uniform(0.5, 2.0, M) / 127.0).astype(np.float32)
    sw = (rng.uniform(0.5, 2.0, N) / 127.0).astype(np.float32)
    bias = rng.normal(0, 0.5, N).astype(np.float32)
    a = packed_from_codes(cr, Qx, sx, 0, "none", False, "act")
    w = packed_from_codes(cr, Qw, sw, 0, "none", False, "w")
    A = O.int_gemm(Qx, Qw)
    assert np.array_equal(to_np(cr.convrot_gemm_s32(a, w)).astype(np.int64), A)
    Y = cr.convrot_linear(a, w, torch.from_numpy(bias).cuda())
    check_y_same_codes(to_np(Y.float()), A, sx, sw, bias, f"small tc {M}x{N}x{K}")


def test_small_m_tensor_core_adversarial_and_multi(cr):
    """All +-127 codes at K = 4096 (four exact chunks summed in int32), and two
    linears in one launch equal to two launches."""
    M, K = 40, 4096
    Qx = np.full((M, K), 127, np.int8)
    Qw = np.full((200, K), 127, np.int8)
    Qw[::3] = -127
    a = packed_from_codes(cr, Qx, np.ones(M), 0, "none", False, "act")
    w = packed_from_codes(cr, Qw, np.ones(200), 0, "none", False, "w")
    assert np.array_equal(to_np(cr.convrot_gemm_s32(a, w)).astype(np.int64), O.int_gemm(Qx, Qw))
    rng = np.random.default_rng(9)
    Qw2 = rng.integers(-127, 128, size=(296, K)).astype(np.int8)
    w2 = packed_from_codes(cr, Qw2, np.ones(296) / 127.0, 0, "none", False, "w")
    ys = cr.convrot_linear_multi(a, [w, w2], [None, None])
    assert torch.equal(ys[0], cr.convrot_linear(a, w)) and torch.equal(ys[1], cr.convrot_linear(a, w2))
