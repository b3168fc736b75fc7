"""The row-parallel (K-sharded) steps of the library on one GPU: ranks are
emulated one after another on the same device (nothing waits on another
launch); the two all-reduces are done with torch between the calls. Codes,
scales, int32 accumulators and Y must be bit-identical to the one-device
path on the whole row, and within the oracle's bounds (sglang digest,
"风险与影响": each rank's slice of the input features a whole number of
groups)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import check_codes, check_scales, check_y_e2e, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def _slice_weight(cr, w, cols):
    return cr.PackedWeight(w.q[:, cols].contiguous(), w.scale, w.q_f16[:, cols].contiguous(), w.group, w.transform)


@pytest.mark.parametrize("M,K,N,G,ranks", [(300, 6144, 520, 256, 2), (130, 6144, 256, 256, 4),
                                           (77, 4096, 136, 1024, 2), (40, 3072, 264, 64, 3)])
def test_row_parallel_steps_match_the_whole_row(cr, M, K, N, G, ranks):
    wl = WL.make_case(M, K, [N], group=G, seed=M + K + ranks, name="row_parallel")
    wl.X[3] = 0.0      # a zero row: every rank's maximum is 0, so scale 0 and codes 0
    X = wl.X.cuda()
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), G, "h4")  # offline, on the whole K
    b = wl.biases[0].cuda()
    width = K // ranks
    cols = [slice(r * width, (r + 1) * width) for r in range(ranks)]
    # step 1 on every rank, then the all-reduce (max)
    amax = torch.stack([cr.convrot_rotate_absmax(X[:, c], G) for c in cols]).amax(dim=0)
    # steps 3 and 4 on every rank, then the all-reduce (sum)
    acts = [cr.convrot_quantize_act_given_max(X[:, c], amax, G) for c in cols]
    A = sum(cr.convrot_gemm_s32(a, _slice_weight(cr, w, c)) for a, c in zip(acts, cols))
    Y = cr.convrot_dequant(A, acts[0].scale, w.scale, b)
    # the one-device path on the whole row
    full = cr.convrot_quantize_act(X, G, "h4")
    A_full = cr.convrot_gemm_s32(full, w)
    Y_full = cr.convrot_linear(full, w, b)
    torch.cuda.synchronize()
    assert cr.convrot_get_device_status() == 0
    assert torch.equal(torch.cat([a.q for a in acts], dim=1), full.q)
    assert torch.equal(torch.cat([a.q_f16 for a in acts], dim=1), full.q_f16)
    for a in acts:
        assert torch.equal(a.scale, full.scale)
        assert float(a.scale[3]) == 0.0 and not bool(a.q[3].any())
    assert torch.equal(A, A_full)
    assert torch.equal(Y, Y_full)
    # and against the oracle
    X64 = wl.X.float().numpy().astype(np.float64)
    Qx, sx, v = O.quantize_act(X64, G, "h4")
    check_codes(to_np(full.q), Qx, v, "row-parallel codes")
    check_scales(to_np(full.scale), O.quantize_rows(O.rotate_rows(X64, G, "h4"))[3], "row-parallel scales")
    assert np.allclose(to_np(amax), O.row_absmax(O.rotate_rows(X64, G, "h4")), rtol=1e-6, atol=0)
    Qw, sw, _ = O.prepare_weights(wl.weights[0].numpy().astype(np.float64), G, "h4")
    check_y_e2e(to_np(Y.float()), O.reconstruct(O.int_gemm(Qx, Qw), sx, sw, wl.biases[0].numpy()), "row-parallel Y")


def test_dequant_matches_the_fused_epilogue(cr):
    """convrot_dequant against the GEMM's fused epilogue on the same
    accumulators, with a ragged N, a wider output pitch and no bias."""
    wl = WL.make_case(70, 1024, [1003], group=256, seed=3, name="dequant")
    a = cr.convrot_quantize_act(wl.X.cuda(), 256, "h4")
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), 256, "h4")
    # int32 rows need a pitch that is a multiple of 4
    A = cr.convrot_gemm_s32(a, w, out=torch.empty((70, 1008), dtype=torch.int32, device="cuda")[:, :1003])
    for bias in (wl.biases[0].cuda(), None):
        big = torch.full((70, 1016), 7.0, dtype=torch.bfloat16, device="cuda")
        Y = cr.convrot_dequant(A, a.scale, w.scale, bias, out=big[:, :1003])
        torch.cuda.synchronize()
        ref = cr.convrot_linear(a, w, bias, out=torch.empty((70, 1008), dtype=torch.bfloat16, device="cuda")[:, :1003])
        assert torch.equal(Y, ref)
        assert torch.all(big[:, 1003:] == 7.0)


def test_row_parallel_rejections(cr):
    X = torch.zeros((4, 2688), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cr.ConvRotError):           # slice not a multiple of 256
        cr.convrot_rotate_absmax(X, 64)
    Y = torch.zeros((4, 1024), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cr.ConvRotError):           # randomized Hadamard: not on these steps
        cr.convrot_rotate_absmax(Y, 128, "rht")
