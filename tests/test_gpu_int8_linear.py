"""The linear from the activation in one call (convrot_int8_linear): the
sglang digest's single fused op, rotation -> per-row quantization -> int8
GEMM -> dequant epilogue -> bias, for linears sharing one input.

It must equal, bit for bit, the two-call path (convrot_quantize_act, then
convrot_linear_multi_ws) on every GEMM route (weight stream M <= 16, small-M
tensor cores 17..64, 2-SM tensor cores above, with and without a split of the
last round), and match the oracle end to end."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import check_codes, check_y_e2e, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def _scratch_codes(scratch, M, K):
    """The codes the GEMM read: the int8 region, or with the 2-SM tensor-core
    path (M > 64, K a multiple of 64) the fp16 copy."""
    up = lambda v: (v + 255) // 256 * 256
    if M > 64 and K % 64 == 0:
        off16 = up(M * K) + up(4 * M)
        return scratch[off16: off16 + 2 * M * K].view(torch.float16).view(M, K).to(torch.int8)
    return scratch[: M * K].view(torch.int8).view(M, K)


CASES = [
    # M, K, Ns, transform, group
    (1, 256, [256], WL.TRANSFORM_H4, 256),
    (16, 1152, [512, 384], WL.TRANSFORM_RHT, 128),
    (5, 1152, [256, 96], WL.TRANSFORM_RHT, 64),
    (1, 128, [64], WL.TRANSFORM_RHT, 128),
    (16, 1024, [512], WL.TRANSFORM_H4, 64),
    (3, 640, [296], WL.TRANSFORM_H4, 16),
    (16, 1536, [256], WL.TRANSFORM_H4, 4),
    (12, 1280, [256], WL.TRANSFORM_NONE, 256),
    (16, 1280, [512], WL.TRANSFORM_RHT, 256),
    (16, 1664, [256], WL.TRANSFORM_H4, 64),
    (48, 1152, [256, 136], WL.TRANSFORM_RHT, 128),
    # large M with K not a multiple of 256: the tensor-core rotate+quantize's
    # tiles of whole superblocks across rows, writing only the fp16 copy
    (300, 2688, [256, 136], WL.TRANSFORM_H4, 64),
    (130, 1088, [200], WL.TRANSFORM_H4, 16),
    (300, 512, [512, 272], WL.TRANSFORM_H4, 64),
    (1000, 1024, [768], WL.TRANSFORM_NONE, 256),
    (4096, 2048, [2048, 1024, 512], WL.TRANSFORM_H4, 256),
]


@pytest.mark.parametrize("M,K,Ns,transform,group", CASES)
@pytest.mark.parametrize("use_ws", [False, True])
def test_one_call_equals_two_calls(cr, M, K, Ns, transform, group, use_ws):
    wl = WL.make_case(M, K, Ns, transform=transform, group=group, seed=11, name="one_call")
    sg = None if wl.signs is None else wl.signs.cuda()
    ws = [cr.convrot_prepare_weights(W.cuda(), group, transform, sg) for W in wl.weights]
    bs = [b.cuda() for b in wl.biases]
    X = wl.X.cuda()
    gws = cr.gemm_workspace() if use_ws else None
    Y1 = cr.convrot_int8_linear(X, ws, bs, signs=sg, workspace=gws)
    a = cr.convrot_quantize_act(X, group, transform, sg, with_f16=True)
    Y2 = cr.convrot_linear_multi(a, ws, bs, workspace=gws)
    torch.cuda.synchronize()
    assert cr.convrot_get_device_status() == 0
    for y1, y2 in zip(Y1, Y2):
        assert torch.equal(y1, y2)
    if gws is not None:
        assert int(gws.count_nonzero()) == 0  # the workspace is left clear


def test_scratch_layout_and_reuse(cr):
    """The scratch holds the packed activation: codes, scales, and the fp16
    copy when the 2-SM tensor-core path runs (which then needs no codes);
    one scratch serves successive calls on a stream."""
    K = 512
    for M, f16 in [(16, False), (64, False), (65, True), (300, True)]:
        up = lambda v: (v + 255) // 256 * 256
        want = up(M * K) + up(4 * M) + (up(2 * M * K) if f16 else 0)
        assert cr.lib.convrot_int8_linear_scratch_bytes(M, K) == want
    wl = WL.make_case(300, K, [256], group=64, seed=12, name="scratch")
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), 64, "h4")
    scratch = cr.int8_linear_scratch(300, K)
    X = wl.X.cuda()
    a = cr.convrot_quantize_act(X, 64, "h4")
    Y = cr.convrot_int8_linear(X, [w], scratch=scratch)[0]
    # the scratch now holds the same scales and fp16 copy (the tensor-core GEMM
    # reads only the fp16 copy, so the int8 codes are not written)
    off = (300 * K + 255) // 256 * 256
    assert torch.equal(scratch[off: off + 4 * 300].view(torch.float32), a.scale)
    off16 = off + (4 * 300 + 255) // 256 * 256
    assert torch.equal(scratch[off16: off16 + 2 * 300 * K].view(torch.float16).view(300, K), a.q_f16)
    X2 = X.flip(0).contiguous()
    Y2 = cr.convrot_int8_linear(X2, [w], scratch=scratch)[0]
    assert torch.equal(Y2, cr.convrot_int8_linear(X2, [w])[0])
    assert torch.equal(Y, cr.convrot_linear(a, w))


@pytest.mark.parametrize("M,K,G,transform", [(16, 1152, 128, "rht"), (7, 1024, 64, "h4"), (2, 512, 0, "none")])
def test_small_m_writes_the_packed_activation(cr, M, K, G, transform):
    """With a handful of rows the scratch receives the packed activation too
    (codes and scales, no fp16 copy), equal to convrot_quantize_act's."""
    wl = WL.make_case(M, K, [128], transform=transform, group=max(G, 2), seed=13, name="small_m")
    sg = None if wl.signs is None else wl.signs.cuda()
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), G, transform, sg)
    X = wl.X.cuda()
    scratch = cr.int8_linear_scratch(M, K)
    cr.convrot_int8_linear(X, [w], signs=sg, scratch=scratch)
    a = cr.convrot_quantize_act(X, G, transform, sg, with_f16=False)
    torch.cuda.synchronize()
    assert torch.equal(scratch[: M * K].view(torch.int8).view(M, K), a.q)
    off = (M * K + 255) // 256 * 256
    assert torch.equal(scratch[off: off + 4 * M].view(torch.float32), a.scale)


@pytest.mark.parametrize("case", ["dit", "ffn_rht", "g16"])
def test_one_call_end_to_end(cr, case):
    wl = {"dit": lambda: WL.dit6144(M=200),
          "ffn_rht": lambda: WL.ffn_pair(),
          "g16": lambda: WL.gsweep(16, M=130)}[case]()
    sg = None if wl.signs is None else wl.signs.cuda()
    ws = [cr.convrot_prepare_weights(W.cuda(), wl.group, wl.transform, sg) for W in wl.weights]
    bs = [b.cuda() for b in wl.biases]
    scratch = cr.int8_linear_scratch(wl.M, wl.K)
    Ys = cr.convrot_int8_linear(wl.X.cuda(), ws, bs, signs=sg, scratch=scratch)
    torch.cuda.synchronize()
    sgn = None if wl.signs is None else wl.signs.numpy()
    X64 = wl.X.float().numpy().astype(np.float64)
    Qx, sx, v = O.quantize_act(X64, wl.group, wl.transform, sgn)
    check_codes(to_np(_scratch_codes(scratch, wl.M, wl.K)), Qx, v, case)
    for i, Y in enumerate(Ys):
        Qw, sw, _ = O.prepare_weights(wl.weights[i].numpy().astype(np.float64), wl.group, wl.transform, sgn)
        ref = O.reconstruct(O.int_gemm(Qx, Qw), sx, sw, wl.biases[i].numpy())
        check_y_e2e(to_np(Y.float()), ref, f"{case}[{i}]")


def test_layer_forward_uses_the_one_call_path(cr):
    wl = WL.dit6144(M=96)
    layer = cr.ConvRotLinear.from_float(wl.weights[0][:512].cuda(), wl.biases[0][:512].cuda(), 256)
    x = wl.X.cuda().view(2, 48, -1)
    y = layer(x)
    a = cr.convrot_quantize_act(wl.X.cuda(), 256)
    ref = cr.convrot_linear(a, layer.weight, layer.bias)
    assert y.shape == (2, 48, 512)
    assert torch.equal(y.reshape(96, 512), ref)


def test_one_call_strided_input_and_empty_batch(cr):
    """X given as a column slice of a wider buffer (row stride > K), and an
    empty batch, through the one-call linear."""
    wl = WL.make_case(130, 1024, [256], group=64, seed=14, name="strided")
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), 64, "h4")
    wide = torch.zeros(130, 1024 + 64, dtype=torch.bfloat16, device="cuda")
    wide[:, 32:32 + 1024] = wl.X.cuda()
    Xs = wide[:, 32:32 + 1024]
    assert Xs.stride(0) == 1088
    Y = cr.convrot_int8_linear(Xs, [w])[0]
    a = cr.convrot_quantize_act(wl.X.cuda(), 64, "h4")
    assert torch.equal(Y, cr.convrot_linear(a, w))
    E = cr.convrot_int8_linear(torch.empty(0, 1024, dtype=torch.bfloat16, device="cuda"), [w])[0]
    assert E.shape == (0, 256)


def test_one_call_wide_rows(cr):
    """An MLP-width input (K = 21504, wider than one TMA box of the
    rotate+quantize kernel) through the one-call linear on the tensor cores."""
    wl = WL.make_case(300, 21504, [256], group=256, seed=15, name="wide")
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), 256, "h4")
    X = wl.X.cuda()
    Y = cr.convrot_int8_linear(X, [w], workspace=cr.gemm_workspace())[0]
    a = cr.convrot_quantize_act(X, 256, "h4")
    assert torch.equal(Y, cr.convrot_linear(a, w))
    sgn = None
    Qx, sx, v = O.quantize_act(wl.X.float().numpy().astype(np.float64), 256, "h4", sgn)
    check_codes(to_np(a.q), Qx, v, "wide")
