"""Parity of the 4-bit ConvRot path (codes in [-7, 7], "feat: load ConvRot
int4 and per-channel int8 safetensors", "Solution") with the CPU oracle:
packed codes, scales and e4m3 copies from both rotate+quantize kernels, exact
int32 accumulators from the kind::f8f6f4 tensor-core GEMM, and Y."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import check_codes, check_scales, check_y_e2e, check_y_same_codes, tensor_core_takes, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def _codes4(a):
    """(codes from the nibbles, codes from the e4m3 copy) of a packed 4-bit tensor."""
    q = O.unpack_int4(to_np(a.q4))
    f = None if a.q_f8 is None else to_np(a.q_f8.view(torch.float8_e4m3fn).float()).astype(np.int64)
    return q, f


def _oracle4(X_bf16, G, transform, signs=None):
    X64 = X_bf16.float().numpy().astype(np.float64)
    Q, _, v, s64 = O.quantize_rows(O.rotate_rows(X64, G, transform, None if signs is None else signs.numpy()),
                                   O.QMAX4)
    return Q, s64, v


@pytest.mark.parametrize("M,K,G,transform", [
    (37, 6144, 256, "h4"), (33, 4096, 16, "h4"), (33, 4096, 64, "h4"), (33, 4096, 1024, "h4"),
    (16, 1152, 128, "rht"), (21, 2048, 128, "rht"), (21, 2048, 256, "rht"), (9, 1152, 0, "none"), (1, 128, 4, "h4"),
    (300, 3072, 256, "h4"), (45, 2688, 64, "h4"), (13, 2688, 16, "h4"),
])
def test_quantize_act4_matches_oracle_on_both_kernels(cr, M, K, G, transform):
    wl = WL.make_case(M, K, [], dist="t3", outlier_frac=0.002, outlier_scale=40.0, group=max(G, 2),
                      transform=transform, seed=M + K + G)
    X = wl.X.cuda()
    sg = None if wl.signs is None else wl.signs.cuda()
    fast = cr.convrot_quantize_act4(X, G, transform, sg)
    # outputs 16 but not 32 bytes aligned: the generic kernel
    qb = torch.empty(M * K // 2 + 16, dtype=torch.uint8, device="cuda")
    fb = torch.empty(M * K + 16, dtype=torch.uint8, device="cuda")
    out = cr.PackedAct4(qb[16:].view(M, K // 2), torch.empty(M, dtype=torch.float32, device="cuda"),
                        fb[16:].view(M, K), G, cr.TRANSFORMS[transform])
    gen = cr.convrot_quantize_act4(X, G, transform, sg, out=out)
    torch.cuda.synchronize()
    Q, s, v = _oracle4(wl.X, G, transform, wl.signs)
    q_fast, f_fast = _codes4(fast)
    check_codes(q_fast, Q, v, f"w4 {transform} G{G}")
    check_scales(to_np(fast.scale), s, f"w4 {transform} G{G}")
    assert np.abs(q_fast).max() <= 7
    assert np.array_equal(f_fast, q_fast.astype(np.int64))
    q_gen, f_gen = _codes4(gen)
    check_codes(q_gen, Q, v, f"w4 generic {transform} G{G}")
    assert np.array_equal(f_gen, q_gen.astype(np.int64))
    if tensor_core_takes(K, G, transform):
        # the tensor-core kernel: its 16-point stage sums in the tensor core's
        # order, so a code may differ by one from the generic kernel's where
        # the value lies within a few fp32 ulps of a rounding boundary
        d = np.abs(q_fast.astype(np.int64) - q_gen)
        assert d.max() <= 1 and (d > 0).sum() <= max(1, int(1e-4 * d.size))
    else:
        assert torch.equal(fast.q4, gen.q4) and torch.equal(fast.scale, gen.scale) and torch.equal(fast.q_f8, gen.q_f8)


def test_prepare_weights4_matches_oracle(cr):
    wl = WL.make_case(8, 2048, [300], group=256, seed=21)
    W = wl.weights[0]
    w = cr.convrot_prepare_weights4(W.cuda(), 256, "h4")
    torch.cuda.synchronize()
    Q, s, v, s64 = O.quantize_rows(O.rotate_rows(W.numpy().astype(np.float64), 256, "h4"), O.QMAX4)
    q, f = _codes4(w)
    check_codes(q, Q, v, "w4 weights")
    check_scales(to_np(w.scale), s64, "w4 weights")
    assert np.array_equal(f, q.astype(np.int64))


def _packed4(cr, Q, s, kind):
    q4 = torch.from_numpy(O.pack_int4(Q)).cuda()
    f8 = torch.from_numpy(Q.astype(np.float32)).cuda().to(torch.float8_e4m3fn).view(torch.uint8)
    sc = torch.from_numpy(np.ascontiguousarray(s.astype(np.float32))).cuda()
    cls = cr.PackedAct4 if kind == "act" else cr.PackedWeight4
    return cls(q4, sc, f8, 0, cr.TRANSFORMS["none"])


@pytest.mark.parametrize("M,N,K,ws", [(1, 64, 128, False), (100, 300, 1024, False), (129, 1000, 2048, False),
                                      (300, 1000, 1024, True), (1024, 5120, 1024, True), (257, 136, 2688 + 128, False)])
def test_gemm4_s32_bit_exact(cr, M, N, K, ws):
    rng = np.random.default_rng(M + N + K)
    Qx = rng.integers(-7, 8, size=(M, K)).astype(np.int8)
    Qw = rng.integers(-7, 8, size=(N, K)).astype(np.int8)
    a = _packed4(cr, Qx, np.ones(M), "act")
    w = _packed4(cr, Qw, np.ones(N), "w")
    wsp = cr.gemm_workspace() if ws else None
    A = to_np(cr.convrot_gemm4_s32(a, w, workspace=wsp)).astype(np.int64)
    assert np.array_equal(A, O.int_gemm(Qx, Qw))
    if ws:
        assert torch.equal(cr.convrot_gemm4_s32(a, w, workspace=wsp), cr.convrot_gemm4_s32(a, w))
        torch.cuda.synchronize()
        assert int(wsp.count_nonzero()) == 0


def test_gemm4_adversarial_magnitudes(cr):
    """All +-7 codes with K = 8192: the largest partial sums, still exact."""
    M, N, K = 200, 300, 8192
    Qx = np.full((M, K), 7, np.int8)
    Qw = np.full((N, K), 7, np.int8)
    Qw[1::2] = -7
    A = to_np(cr.convrot_gemm4_s32(_packed4(cr, Qx, np.ones(M), "act"), _packed4(cr, Qw, np.ones(N), "w")))
    assert np.array_equal(A.astype(np.int64), O.int_gemm(Qx, Qw))


def test_linear4_end_to_end_and_multi(cr):
    """The DiT-shaped linear at 4 bits, from X: codes against the oracle, Y
    within one bf16 ulp of the reconstruction from the GPU's codes and within
    1e-2 of max|Y| of the oracle's 4-bit linear; two linears in one launch
    equal two separate launches."""
    wl = WL.make_case(200, 6144, [1024, 512], group=256, seed=23)
    a = cr.convrot_quantize_act4(wl.X.cuda(), 256, "h4")
    ws = [cr.convrot_prepare_weights4(W.cuda(), 256, "h4") for W in wl.weights]
    bs = [b.cuda() for b in wl.biases]
    Ys = cr.convrot_linear4_multi(a, ws, bs, workspace=cr.gemm_workspace())
    for Y, w, b in zip(Ys, ws, bs):
        assert torch.equal(Y, cr.convrot_linear4(a, w, b))
    qx, _ = _codes4(a)
    X64 = wl.X.float().numpy().astype(np.float64)
    Qx_or, sx_or, v = O.quantize_act(X64, 256, "h4", qmax=O.QMAX4)
    check_codes(qx, Qx_or, v, "w4 act")
    for Y, w, W, b in zip(Ys, ws, wl.weights, wl.biases):
        qw, _ = _codes4(w)
        check_y_same_codes(to_np(Y.float()), O.int_gemm(qx, qw), to_np(a.scale), to_np(w.scale), b.numpy(), "w4")
        Qw_or, sw_or, _ = O.prepare_weights(W.numpy().astype(np.float64), 256, "h4", qmax=O.QMAX4)
        ref = O.reconstruct(O.int_gemm(Qx_or, Qw_or), sx_or, sw_or, b.numpy())
        check_y_e2e(to_np(Y.float()), ref, "w4 e2e")


def test_linear4_rejections(cr):
    X = torch.zeros((4, 192), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cr.ConvRotError, match="ALIGNMENT"):
        cr.convrot_quantize_act4(X, 64, "h4")  # K not a multiple of 128
    a = cr.convrot_quantize_act4(torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda"), 64, "h4", with_f8=False)
    w = cr.convrot_prepare_weights4(torch.zeros((8, 256), device="cuda"), 64, "h4")
    with pytest.raises(cr.ConvRotError, match="INVALID_ARG"):
        cr.convrot_linear4(a, w)  # no e4m3 copy of the activation
