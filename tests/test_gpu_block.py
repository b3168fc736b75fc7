"""The linears of one DiT block chained on the GPU (qkv on one packed
activation, out_proj, fc1 on out_proj's output, fc2 on fc1's), each group one
convrot_int8_linear call from its bf16 input: the packed-activation reuse and
the single fused op of "INT8 Convrot Safetensors" ("Runtime activation
quantization") and the sglang digest ("关键源码片段", int8_linear).

Every layer is checked against the oracle run on that layer's own input,
which for out_proj's successors is the previous layer's GPU output: codes and
scales of the layer's packed activation, and sampled output channels both
from the GPU's codes (one bf16 ulp) and end to end from the input (1e-2 of
max|Y|). Width 5376 (21 groups of 256 per row, a tile that is not a whole
number of warps on the rotate+quantize kernels), MLP width 21504 (rows wider
than one TMA box), 200 rows (a ragged last tile)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import check_codes, check_scales, check_y_e2e, check_y_same_codes, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def _check_layer(cr, name, x, ws, pws, bs, ys, G, rng, n_cols=192):
    """x: the layer's bf16 input on the GPU; ws: host fp32 weights; pws: the
    GPU's prepared weights; ys: the GPU outputs of the call."""
    X64 = x.float().cpu().numpy().astype(np.float64)
    a = cr.convrot_quantize_act(x, G, "h4")
    torch.cuda.synchronize()
    Qx, sx, v = O.quantize_act(X64, G, "h4")
    check_codes(to_np(a.q), Qx, v, f"{name} codes")
    check_scales(to_np(a.scale), O.quantize_rows(O.rotate_rows(X64, G, "h4"))[3], f"{name} scales")
    qx = to_np(a.q).astype(np.int8)
    sxg = to_np(a.scale)
    for i, (W, pw, b, Y) in enumerate(zip(ws, pws, bs, ys)):
        N = W.shape[0]
        cols = np.unique(np.concatenate([rng.choice(N, n_cols, replace=False), np.arange(N - 8, N)]))
        Yg = to_np(Y.float())[:, cols]
        bc = b.numpy()[cols]
        # from the GPU's own codes (activation and weight): one bf16 ulp
        qw, swg = to_np(pw.q)[cols].astype(np.int8), to_np(pw.scale)[cols]
        check_y_same_codes(Yg, O.int_gemm(qx, qw), sxg, swg, bc, f"{name}[{i}] same codes")
        # end to end from the layer's input: 1e-2 of max|Y|
        Qw, sw, _ = O.prepare_weights(W.numpy()[cols].astype(np.float64), G, "h4")
        check_y_e2e(Yg, O.reconstruct(O.int_gemm(Qx, Qw), sx, sw, bc), f"{name}[{i}] end to end")


def test_dit_block_chain_matches_oracle_layer_by_layer(cr):
    blk = WL.dit_block(M=200)
    G = blk.group
    dev = torch.device("cuda")
    prep = lambda W: cr.convrot_prepare_weights(W.to(dev), G, "h4")
    qkv_w = [prep(W) for W in blk.qkv]
    out_w, fc1_w, fc2_w = prep(blk.out), prep(blk.fc1), prep(blk.fc2)
    X, A = blk.X.to(dev), blk.A.to(dev)
    gws = cr.gemm_workspace(dev)
    # the chain, as the block bench runs it: one call per linear group
    Yqkv = cr.convrot_int8_linear(X, qkv_w, [b.to(dev) for b in blk.qkv_b], workspace=gws)
    Yo = cr.convrot_int8_linear(A, [out_w], [blk.out_b.to(dev)], workspace=gws)[0]
    Yh = cr.convrot_int8_linear(Yo, [fc1_w], [blk.fc1_b.to(dev)], workspace=gws)[0]
    Y2 = cr.convrot_int8_linear(Yh, [fc2_w], [blk.fc2_b.to(dev)], workspace=gws)[0]
    torch.cuda.synchronize()
    assert cr.convrot_get_device_status() == 0
    assert Yh.shape == (200, 21504) and Y2.shape == (200, 5376)
    rng = np.random.default_rng(5)
    _check_layer(cr, "qkv", X, blk.qkv, qkv_w, blk.qkv_b, Yqkv, G, rng)
    _check_layer(cr, "out_proj", A, [blk.out], [out_w], [blk.out_b], [Yo], G, rng)
    _check_layer(cr, "fc1", Yo, [blk.fc1], [fc1_w], [blk.fc1_b], [Yh], G, rng)
    _check_layer(cr, "fc2", Yh, [blk.fc2], [fc2_w], [blk.fc2_b], [Y2], G, rng)
