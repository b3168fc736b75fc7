"""Parity of the rotate + quantize kernels (activations and weights) with the
CPU oracle, on seeded inputs of the pages' shapes. Runs through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import check_codes, check_scales, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def _oracle_act(X_bf16, G, transform, signs=None):
    """(Q, s as fp64 before rounding to fp32, v) from the oracle."""
    X64 = X_bf16.float().numpy().astype(np.float64)
    Q, _, v, s64 = O.quantize_rows(O.rotate_rows(X64, G, transform, None if signs is None else signs.numpy()))
    return Q, s64, v


def _run_act(cr, X_bf16, G, transform, signs=None, with_f16=True):
    Xd = X_bf16.cuda()
    sd = None if signs is None else signs.cuda()
    a = cr.convrot_quantize_act(Xd, G, transform, sd, with_f16=with_f16)
    torch.cuda.synchronize()
    return a


@pytest.mark.parametrize("M,K,G", [
    (64, 256, 256),     # the tiny workload
    (37, 6144, 256),    # DiT width, ragged rows
    (50, 3072, 256),    # qkv width
    (33, 4096, 16), (33, 4096, 64), (33, 4096, 256), (33, 4096, 1024),  # group sweep
    (45, 2688, 64),     # AdaLN width
    (7, 64, 4), (3, 4096, 4096), (1, 1024, 1024),
])
def test_quantize_act_h4_matches_oracle(cr, M, K, G):
    wl = WL.make_case(M, K, [], dist="t3", outlier_frac=0.001, outlier_scale=50.0, group=G, seed=M * 7 + G)
    a = _run_act(cr, wl.X, G, "h4")
    Q, s, v = _oracle_act(wl.X, G, "h4")
    check_codes(to_np(a.q), Q, v, f"M{M} K{K} G{G}")
    check_scales(to_np(a.scale), s, f"M{M} K{K} G{G}")
    # the fp16 operand copy holds exactly the int8 codes
    assert torch.equal(a.q_f16.float(), a.q.float())


def test_tiny_workload_spikes_spread(cr):
    wl = WL.tiny()
    a = _run_act(cr, wl.X, 256, "h4")
    Q, s, v = _oracle_act(wl.X, 256, "h4")
    check_codes(to_np(a.q), Q, v, "tiny")
    # +-40 spikes in a N(0,1) row: after the rotation the spike spreads over
    # the group, so the codes use a wide range instead of saturating one slot
    assert np.mean(np.abs(to_np(a.q)) > 10) > 0.5


def test_misaligned_outputs_take_the_generic_kernel(cr):
    """Outputs at a 16- but not 32-byte aligned address make the library take
    the generic kernel: bit-identical to the butterfly kernel asked for by
    name (both run the same fp32 operations in the same order)."""
    for G in (16, 64, 256, 1024):
        wl = WL.make_case(40, 4096, [], seed=11 + G, group=G)
        X = wl.X.cuda()
        M, K = X.shape
        fast = cr.convrot_quantize_act_kernel(X, G, "h4", kernel="butterfly")
        qbuf = torch.empty(M * K + 16, dtype=torch.int8, device="cuda")
        hbuf = torch.empty(M * K + 8, dtype=torch.float16, device="cuda")
        q_un = qbuf[16:].view(M, K)
        h_un = hbuf[8:].view(M, K)
        assert q_un.data_ptr() % 32 == 16 and h_un.data_ptr() % 32 == 16
        out = cr.PackedAct(q_un, torch.empty(M, dtype=torch.float32, device="cuda"), h_un, G, 0)
        gen = cr.convrot_quantize_act(X, G, "h4", out=out)
        torch.cuda.synchronize()
        assert torch.equal(gen.q, fast.q), G
        assert torch.equal(gen.scale, fast.scale), G
        assert torch.equal(gen.q_f16, fast.q_f16), G


@pytest.mark.parametrize("M,K,G", [(37, 6144, 256), (130, 3072, 256), (33, 4096, 16), (33, 4096, 64),
                                   (33, 4096, 1024), (7, 1024, 4), (37, 5376, 256), (37, 5376, 64),
                                   (3, 21504, 256), (2, 24576, 1024), (1, 256, 16), (300, 1024, 1024),
                                   # K not a multiple of 256: superblocks across rows
                                   (45, 2688, 64), (41, 2688, 16), (13, 2688, 4), (9, 320, 64), (33, 1088, 64),
                                   (7, 1088, 16), (300, 2688, 64), (1, 2688, 64), (5, 4032, 64)])
def test_tensor_core_kernel_matches_oracle(cr, M, K, G):
    """The 16-point stage on the tensor cores (mma.sync bf16 -> fp32 from the
    staged tile), the higher digits on fp32 registers: codes and scales
    against the oracle; against the all-fp32 butterfly kernel at most one
    code apart, on at most 1e-4 of the elements (the tensor core sums its 16
    exact products in its own order)."""
    wl = WL.make_case(M, K, [], dist="t3", outlier_frac=0.001, outlier_scale=50.0, group=G, seed=M + K + 3 * G)
    X = wl.X.cuda()
    tc = cr.convrot_quantize_act_kernel(X, G, "h4", kernel="tensor_core")
    auto = cr.convrot_quantize_act(X, G, "h4")
    bf = cr.convrot_quantize_act_kernel(X, G, "h4", kernel="butterfly")
    torch.cuda.synchronize()
    Q, s, v = _oracle_act(wl.X, G, "h4")
    check_codes(to_np(tc.q), Q, v, f"tc M{M} K{K} G{G}")
    check_scales(to_np(tc.scale), s, f"tc M{M} K{K} G{G}")
    assert torch.equal(tc.q_f16.float(), tc.q.float())
    # the library's choice for this shape is the tensor-core kernel
    assert torch.equal(auto.q, tc.q) and torch.equal(auto.scale, tc.scale) and torch.equal(auto.q_f16, tc.q_f16)
    d = (tc.q.int() - bf.q.int()).abs()
    assert int(d.max()) <= 1 and int((d > 0).sum()) <= max(1, int(1e-4 * d.numel()))


def test_tensor_core_kernel_concurrent_launches(cr):
    """The kernel hands out its tiles through a counter slot per launch:
    launches in flight together on four streams, and 300 launches in a row
    (more than the slots, so every slot is reused), each give the result of
    a lone launch."""
    wl = WL.make_case(300, 3072, [], seed=77, group=256)
    X = wl.X.cuda()
    ref = cr.convrot_quantize_act(X, 256, "h4")
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(4)]
    outs = []
    for i in range(40):
        s = streams[i % 4]
        with torch.cuda.stream(s):
            outs.append(cr.convrot_quantize_act(X, 256, "h4", stream=s))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.q, ref.q) and torch.equal(o.scale, ref.scale) and torch.equal(o.q_f16, ref.q_f16)
    a = cr.convrot_quantize_act(X, 256, "h4")
    for _ in range(300):
        cr.convrot_quantize_act(X, 256, "h4", out=a)
    torch.cuda.synchronize()
    assert torch.equal(a.q, ref.q) and torch.equal(a.scale, ref.scale)
    assert cr.convrot_get_device_status() == 0


def test_tensor_core_kernel_refuses_other_shapes(cr):
    for K in (192, 2720):   # fewer than 256 columns; not a multiple of 64
        X = torch.zeros((4, K), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(cr.ConvRotError, match="does not take"):
            cr.convrot_quantize_act_kernel(X, 16, "h4", kernel="tensor_core")
    X = torch.zeros((4, 2688), dtype=torch.bfloat16, device="cuda")   # G = 256 does not divide K
    with pytest.raises(cr.ConvRotError):
        cr.convrot_quantize_act_kernel(X, 256, "h4", kernel="tensor_core")
    Y = torch.zeros((4, 1536), dtype=torch.bfloat16, device="cuda")   # G = 1024 needs K % 1024 == 0
    with pytest.raises(cr.ConvRotError):
        cr.convrot_quantize_act_kernel(Y, 1024, "h4", kernel="tensor_core")
    Z = torch.zeros((4, 1024), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(128, dtype=torch.int8, device="cuda")
    with pytest.raises(cr.ConvRotError):                               # RHT stays on the butterfly
        cr.convrot_quantize_act_kernel(Z, 128, "rht", g, kernel="tensor_core")


def test_tensor_core_kernel_takes_exactly_the_documented_shapes(cr):
    """The routing rule of the header (and of the parity helper): asked for
    by name, the tensor-core kernel runs on exactly the widths and groups the
    rule names and refuses the rest without launching."""
    from parity import tensor_core_takes
    for K in (192, 256, 320, 1088, 2688, 4032, 5376, 6144, 6208, 12288, 12416, 21504, 24576):
        X = torch.zeros((3, K), dtype=torch.bfloat16, device="cuda")
        for G in (4, 16, 64, 256, 1024):
            if K % G:
                continue
            if tensor_core_takes(K, G):
                a = cr.convrot_quantize_act_kernel(X, G, "h4", kernel="tensor_core")
                assert int(a.q.abs().max()) == 0 and float(a.scale.abs().max()) == 0.0
            else:
                with pytest.raises(cr.ConvRotError, match="does not take"):
                    cr.convrot_quantize_act_kernel(X, G, "h4", kernel="tensor_core")
    torch.cuda.synchronize()
    assert cr.convrot_get_device_status() == 0


@pytest.mark.parametrize("G", [256, 1024])
def test_quantize_act_at_the_largest_k(cr, G):
    """Rows of K = 32768 (CONVROT_MAX_K), wider than any tile of the fast
    kernels: codes and scales against the oracle."""
    wl = WL.make_case(3, 32768, [], dist="t3", outlier_frac=0.001, outlier_scale=50.0, group=G, seed=G + 1)
    a = _run_act(cr, wl.X, G, "h4")
    Q, s, v = _oracle_act(wl.X, G, "h4")
    check_codes(to_np(a.q), Q, v, f"K32768 G{G}")
    check_scales(to_np(a.scale), s, f"K32768 G{G}")
    assert torch.equal(a.q_f16.float(), a.q.float())


def test_without_f16_copy(cr):
    wl = WL.make_case(20, 3072, [], seed=12)
    a = _run_act(cr, wl.X, 256, "h4", with_f16=False)
    b = _run_act(cr, wl.X, 256, "h4", with_f16=True)
    assert a.q_f16 is None and torch.equal(a.q, b.q) and torch.equal(a.scale, b.scale)


def test_zero_rows_and_basis_rows(cr):
    K, G = 1024, 256
    X = torch.zeros((6, K), dtype=torch.bfloat16)
    X[1, 5] = 1.0                # basis vector: whole group +-127
    X[3, 300] = -2.0
    X[5, :] = 3.0                # constant row: R fixes the all-ones vector
    a = _run_act(cr, X, G, "h4")
    Q, s, v = _oracle_act(X, G, "h4")
    assert np.array_equal(to_np(a.q), Q)
    check_scales(to_np(a.scale), s)
    assert float(a.scale[0]) == 0.0 and float(a.scale[2]) == 0.0
    assert np.all(np.abs(to_np(a.q)[1, :256]) == 127) and np.all(to_np(a.q)[1, 256:] == 0)
    assert np.all(to_np(a.q)[5] == 127)


def test_single_row_and_empty(cr):
    wl = WL.make_case(1, 6144, [], seed=13)
    a = _run_act(cr, wl.X, 256, "h4")
    Q, s, v = _oracle_act(wl.X, 256, "h4")
    check_codes(to_np(a.q), Q, v, "M=1")
    e = cr.convrot_quantize_act(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"), 256, "h4")
    assert e.q.shape == (0, 256)


@pytest.mark.parametrize("M,K,B", [(16, 1152, 128), (9, 256, 16), (5, 4096, 1024)])
def test_quantize_act_rht_matches_oracle(cr, M, K, B):
    wl = WL.make_case(M, K, [], dist="normal", outlier_frac=0.005, outlier_scale=30.0, group=B,
                      transform="rht", seed=B + M)
    a = _run_act(cr, wl.X, B, "rht", wl.signs)
    Q, s, v = _oracle_act(wl.X, B, "rht", wl.signs)
    check_codes(to_np(a.q), Q, v, f"rht B{B}")
    check_scales(to_np(a.scale), s, f"rht B{B}")


def _fast_and_generic(cr, X, G, transform, signs=None):
    """The register butterfly kernel and the generic kernel, each asked for
    by name, on the same input (the generic kernel twice where the register
    kernel does not take the shape, e.g. a row of 264 lines, which does not
    split into TMA boxes that start on whole 1 KB swizzle atoms)."""
    try:
        fast = cr.convrot_quantize_act_kernel(X, G, transform, signs, kernel="butterfly")
    except cr.ConvRotError as e:
        assert "does not take" in str(e)
        fast = cr.convrot_quantize_act_kernel(X, G, transform, signs, kernel="generic")
    gen = cr.convrot_quantize_act_kernel(X, G, transform, signs, kernel="generic")
    torch.cuda.synchronize()
    return fast, gen


def _check_auto(cr, X, G, transform, signs, Q, s, v, label):
    """What convrot_quantize_act picks for the shape, against the oracle."""
    a = cr.convrot_quantize_act(X, G, transform, signs)
    torch.cuda.synchronize()
    check_codes(to_np(a.q), Q, v, label + " auto")
    check_scales(to_np(a.scale), s, label + " auto")
    assert torch.equal(a.q_f16.float(), a.q.float())


@pytest.mark.parametrize("M,K,B", [(37, 1152, 2), (37, 1152, 8), (37, 1152, 32), (37, 1152, 64),
                                   (37, 1152, 128), (37, 2048, 128), (300, 4096, 128), (37, 2048, 256),
                                   (300, 4096, 256), (1, 256, 256), (3, 21504, 128)])
def test_quantize_act_rht_register_kernel(cr, M, K, B):
    """Block randomized Hadamard on the register kernel (signs applied to the
    bf16 bits, radix-2 stages in registers and across lanes): codes and
    scales against the oracle, and bit-identical to the generic kernel."""
    wl = WL.make_case(M, K, [], dist="t3", outlier_frac=0.002, outlier_scale=40.0, group=B,
                      transform="rht", seed=3 * B + M)
    X, sg = wl.X.cuda(), wl.signs.cuda()
    fast, gen = _fast_and_generic(cr, X, B, "rht", sg)
    Q, s, v = _oracle_act(wl.X, B, "rht", wl.signs)
    check_codes(to_np(fast.q), Q, v, f"rht B{B}")
    check_scales(to_np(fast.scale), s, f"rht B{B}")
    assert torch.equal(fast.q, gen.q) and torch.equal(fast.scale, gen.scale) and torch.equal(fast.q_f16, gen.q_f16)
    assert torch.equal(fast.q_f16.float(), fast.q.float())


@pytest.mark.parametrize("M,K", [(21, 1152), (300, 6144), (5, 64)])
def test_quantize_act_none_register_kernel(cr, M, K):
    """The naive variant (no rotation) on the register kernel: against the
    oracle and bit-identical to the generic kernel."""
    wl = WL.make_case(M, K, [], seed=M + K)
    fast, gen = _fast_and_generic(cr, wl.X.cuda(), 0, "none")
    Q, s, v = _oracle_act(wl.X, 0, "none")
    check_codes(to_np(fast.q), Q, v, "none")
    check_scales(to_np(fast.scale), s, "none")
    assert torch.equal(fast.q, gen.q) and torch.equal(fast.scale, gen.scale) and torch.equal(fast.q_f16, gen.q_f16)


@pytest.mark.parametrize("M,K,G,transform", [(9, 21504, 256, "h4"), (9, 24576, 1024, "h4"), (7, 21504, 16, "h4"),
                                               (9, 21504, 256, "rht"), (5, 21504, 0, "none"), (3, 16896, 256, "h4")])
def test_wide_rows_register_kernel(cr, M, K, G, transform):
    """Rows wider than one TMA box (256 lines of 64 values: an MLP width
    such as 4 x 5376) arrive in two equal copies; codes and scales against
    the oracle, and bit-identical to the generic kernel."""
    wl = WL.make_case(M, K, [], dist="t3", outlier_frac=0.001, outlier_scale=50.0, group=max(G, 2),
                      transform=transform, seed=K + G + M)
    sg = None if wl.signs is None else wl.signs.cuda()
    fast, gen = _fast_and_generic(cr, wl.X.cuda(), G, transform, sg)
    Q, s, v = _oracle_act(wl.X, G, transform, wl.signs)
    check_codes(to_np(fast.q), Q, v, f"{transform} G{G} K{K}")
    check_scales(to_np(fast.scale), s, f"{transform} G{G} K{K}")
    assert torch.equal(fast.q, gen.q) and torch.equal(fast.scale, gen.scale) and torch.equal(fast.q_f16, gen.q_f16)
    _check_auto(cr, wl.X.cuda(), G, transform, sg, Q, s, v, f"{transform} G{G} K{K}")


@pytest.mark.parametrize("M,K,G,transform", [(37, 5376, 256, "h4"), (37, 5376, 128, "rht"), (37, 5376, 64, "h4"),
                                               (29, 2304, 256, "rht"), (41, 2688, 16, "h4"), (11, 1664, 4, "h4")])
def test_tiles_with_padding_threads(cr, M, K, G, transform):
    """Widths whose tile is not a whole number of warps (K = 5376, the DiT
    block width: 3 rows of 84 lines, 252 threads in blocks of 256): the
    padding threads own no line and must neither change a row maximum nor
    write. Ragged M leaves a partial last tile. Codes and scales against the
    oracle, bit-identical to the generic kernel."""
    wl = WL.make_case(M, K, [], dist="t3", outlier_frac=0.001, outlier_scale=50.0, group=G,
                      transform=transform, seed=M + K + G)
    sg = None if wl.signs is None else wl.signs.cuda()
    fast, gen = _fast_and_generic(cr, wl.X.cuda(), G, transform, sg)
    Q, s, v = _oracle_act(wl.X, G, transform, wl.signs)
    check_codes(to_np(fast.q), Q, v, f"{transform} G{G} K{K}")
    check_scales(to_np(fast.scale), s, f"{transform} G{G} K{K}")
    assert torch.equal(fast.q, gen.q) and torch.equal(fast.scale, gen.scale) and torch.equal(fast.q_f16, gen.q_f16)
    _check_auto(cr, wl.X.cuda(), G, transform, sg, Q, s, v, f"{transform} G{G} K{K}")


def test_quantize_act_none_matches_oracle(cr):
    wl = WL.make_case(21, 1152, [], seed=14)
    a = _run_act(cr, wl.X, 0, "none")
    Q, s, v = _oracle_act(wl.X, 0, "none")
    check_codes(to_np(a.q), Q, v, "none")


@pytest.mark.parametrize("N,K,G,transform,dtype", [
    (256, 256, 256, "h4", torch.float32),
    (300, 6144, 256, "h4", torch.float32),
    (129, 4096, 1024, "h4", torch.float32),
    (77, 2688, 64, "h4", torch.float32),
    (200, 1152, 128, "rht", torch.float32),
    (64, 3072, 256, "h4", torch.bfloat16),
])
def test_prepare_weights_matches_oracle(cr, N, K, G, transform, dtype):
    g = torch.Generator().manual_seed(N + K)
    W = torch.randn((N, K), generator=g) * 0.02
    W = W.to(dtype)
    signs = WL.draw_signs(g, G) if transform == "rht" else None
    pw = cr.convrot_prepare_weights(W.cuda(), G, transform, None if signs is None else signs.cuda())
    torch.cuda.synchronize()
    W64 = W.float().numpy().astype(np.float64)
    sg = None if signs is None else signs.numpy()
    Q, s, v = O.prepare_weights(W64, G, transform, sg)
    check_codes(to_np(pw.q), Q, v, f"W {N}x{K}")
    check_scales(to_np(pw.scale), O.quantize_rows(O.rotate_rows(W64, G, transform, sg))[3])
    assert torch.equal(pw.q_f16.float(), pw.q.float())


@pytest.mark.parametrize("name", ["dit6144", "qkv32700", "gsweep1024", "k2688"])
def test_full_size_sampled_rows(cr, name):
    """Full-size workloads in the launch configuration the bench times;
    the oracle checks a seeded sample of rows (rows are independent)."""
    wl = {"dit6144": lambda: WL.dit6144(), "qkv32700": lambda: WL.qkv32700(),
          "gsweep1024": lambda: WL.gsweep(1024), "k2688": lambda: WL.k2688()}[name]()
    a = _run_act(cr, wl.X, wl.group, "h4")
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(wl.M, 512, replace=False), np.arange(wl.M - 70, wl.M)]))
    Xs = wl.X[torch.from_numpy(rows)]
    Q, s, v = _oracle_act(Xs, wl.group, "h4")
    check_codes(to_np(a.q)[rows], Q, v, name)
    check_scales(to_np(a.scale)[rows], s, name)


@pytest.mark.parametrize("M,K,G", [(64, 256, 256), (37, 6144, 256), (130, 3072, 256), (33, 4096, 64),
                                   (45, 2688, 64), (20, 2048, 16), (3, 64, 16)])
def test_hmatmul_variant_matches_oracle(cr, M, K, G):
    """The rotation applied as a dense tensor-core matmul gives the same
    codes as the oracle (within the code tolerance) and the same scales."""
    wl = WL.make_case(M, K, [], dist="t3", outlier_frac=0.001, outlier_scale=50.0, group=G, seed=M + K + G)
    X = wl.X.cuda()
    a = cr.convrot_quantize_act_hmatmul(X, G)
    torch.cuda.synchronize()
    Q, s, v = _oracle_act(wl.X, G, "h4")
    check_codes(to_np(a.q), Q, v, f"hmatmul M{M} K{K} G{G}")
    check_scales(to_np(a.scale), s, f"hmatmul M{M} K{K} G{G}")
    assert torch.equal(a.q_f16.float(), a.q.float())
    # against the butterfly kernel: at most one code apart, rarely
    b = cr.convrot_quantize_act(X, G, "h4")
    d = (a.q.int() - b.q.int()).abs()
    assert int(d.max()) <= 1 and int((d > 0).sum()) <= max(1, int(1e-4 * d.numel()))


def test_hmatmul_zero_rows_and_rejections(cr):
    X = torch.zeros((5, 1024), dtype=torch.bfloat16, device="cuda")
    X[2, 7] = 3.0
    a = cr.convrot_quantize_act_hmatmul(X, 256)
    torch.cuda.synchronize()
    assert float(a.scale[0]) == 0.0 and torch.all(a.q[0] == 0)
    assert torch.all(a.q[2, :256].abs() == 127)
    with pytest.raises(cr.ConvRotError):
        cr.convrot_quantize_act_hmatmul(X, 1024)            # G outside {16, 64, 256}
    with pytest.raises(cr.ConvRotError):
        big = torch.zeros((2, 16 * 1024 + 64 * 0), dtype=torch.bfloat16, device="cuda")
        cr.convrot_quantize_act_hmatmul(big, 64)            # K / 64 > 128
