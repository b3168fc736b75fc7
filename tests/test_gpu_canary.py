"""Guard bytes around the outputs: every kernel writes exactly its outputs.

Outputs are views into larger buffers filled with a sentinel; after the call
the bytes outside the views must still hold it. Shapes leave partial tiles
(rows past the last whole tile of the rotate+quantize kernel, a last row
block and a last column tile of the GEMM) and use the two-box rows of the
register rotate+quantize kernel."""
import pytest
import torch

import workloads as WL

pytestmark = pytest.mark.gpu

SENT8 = 0x5A


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def _guarded(shape, dtype, pad_rows=3, pad_cols=16):
    """A view of `shape` inside a sentinel-filled buffer with extra rows and columns."""
    rows, cols = shape
    buf = torch.empty((rows + pad_rows, cols + pad_cols), dtype=dtype, device="cuda")
    buf.view(torch.uint8).fill_(SENT8)
    return buf, buf[:rows, :cols]


def _outside_untouched(buf, rows, cols):
    u8 = buf.view(torch.uint8)
    esz = buf.element_size()
    inner = torch.zeros_like(u8, dtype=torch.bool)
    inner[:rows, : cols * esz] = True
    return bool((u8[~inner] == SENT8).all())


@pytest.mark.parametrize("M,K,G,transform", [(37, 1152, 64, "h4"), (37, 1152, 128, "rht"), (3, 21504, 256, "h4"),
                                             (9, 4096, 256, "rht"), (13, 640, 0, "none"), (37, 5376, 256, "h4")])
def test_rotate_quantize_writes_only_its_outputs(cr, M, K, G, transform):
    wl = WL.make_case(M, K, [], transform=transform, group=max(G, 2), seed=M + K, name="canary")
    sg = None if wl.signs is None else wl.signs.cuda()
    qbuf, _ = _guarded((M, K), torch.int8, pad_cols=32)
    hbuf, _ = _guarded((M, K), torch.float16, pad_cols=32)
    sbuf = torch.empty(M + 64, dtype=torch.float32, device="cuda")
    sbuf.view(torch.uint8).fill_(SENT8)
    # the kernels write dense [M, K] outputs: dense storage at the start of the
    # guarded buffers, the rest of each buffer must keep the sentinel
    qd = qbuf.view(-1)[: M * K].view(M, K)
    hd = hbuf.view(-1)[: M * K].view(M, K)
    out = cr.PackedAct(qd, sbuf[:M], hd, G, cr.TRANSFORMS[transform])
    cr.convrot_quantize_act(wl.X.cuda(), G, transform, sg, out=out)
    torch.cuda.synchronize()
    assert bool((qbuf.view(torch.uint8).view(-1)[M * K:] == SENT8).all())
    assert bool((hbuf.view(torch.uint8).view(-1)[2 * M * K:] == SENT8).all())
    assert bool((sbuf.view(torch.uint8)[4 * M:] == SENT8).all())
    ref = cr.convrot_quantize_act(wl.X.cuda(), G, transform, sg)
    assert torch.equal(qd, ref.q) and torch.equal(sbuf[:M], ref.scale) and torch.equal(hd, ref.q_f16)


@pytest.mark.parametrize("M,N,K,path", [(300, 520, 1024, "tc"), (300, 520, 1024, "mma"), (48, 520, 1152, "small"),
                                        (9, 136, 1152, "small"), (4100, 6144, 1024, "tc")])
def test_gemm_writes_only_its_outputs(cr, M, N, K, path):
    wl = WL.make_case(M, K, [N], group=64, seed=M + N, name="canary_gemm")
    f16 = path == "tc"
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), 64, "h4", with_f16=f16)
    a = cr.convrot_quantize_act(wl.X.cuda(), 64, "h4", with_f16=f16)
    ybuf, y = _guarded((M, N), torch.bfloat16, pad_rows=5, pad_cols=24)
    if path == "mma":
        cr.convrot_linear(a, w, wl.biases[0].cuda(), out=y, int8_mma=True)
    else:
        cr.convrot_linear(a, w, wl.biases[0].cuda(), out=y, workspace=cr.gemm_workspace())
    torch.cuda.synchronize()
    assert cr.convrot_get_device_status() == 0
    assert _outside_untouched(ybuf, M, N)
    assert torch.equal(y, cr.convrot_linear(a, w, wl.biases[0].cuda(), int8_mma=path == "mma"))


def test_w4_gemm_writes_only_its_outputs(cr):
    M, N, K = 300, 520, 1024
    wl = WL.make_case(M, K, [N], group=64, seed=21, name="canary_w4")
    w = cr.convrot_prepare_weights4(wl.weights[0].cuda(), 64, "h4")
    a = cr.convrot_quantize_act4(wl.X.cuda(), 64, "h4")
    ybuf, y = _guarded((M, N), torch.bfloat16, pad_rows=5, pad_cols=24)
    cr.convrot_linear4_multi(a, [w], [wl.biases[0].cuda()], outs=[y], workspace=cr.gemm_workspace())
    torch.cuda.synchronize()
    assert _outside_untouched(ybuf, M, N)
