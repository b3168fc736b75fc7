"""The static-scratch GEMM entry point (convrot_linear_multi_static): the
split-K GEMM with its workspace in a static device array of the library, so
the call allocates nothing. Collected last on purpose: it is the only test
that leaves library-owned device state (the located scratch) behind."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import check_y_same_codes, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def _codes(cr, M, N, K, seed, nlin=1):
    rng = np.random.default_rng(seed)
    Qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    sx = (rng.uniform(0.5, 2.0, M) / 127.0).astype(np.float32)
    a = cr.PackedAct(torch.from_numpy(Qx).cuda(), torch.from_numpy(sx).cuda(),
                     torch.from_numpy(Qx).cuda().to(torch.float16), 0, 2)
    ws, host = [], []
    for _ in range(nlin):
        Qw = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
        sw = (rng.uniform(0.5, 2.0, N) / 127.0).astype(np.float32)
        b = rng.normal(0, 0.5, N).astype(np.float32)
        ws.append(cr.PackedWeight(torch.from_numpy(Qw).cuda(), torch.from_numpy(sw).cuda(),
                                  torch.from_numpy(Qw).cuda().to(torch.float16), 0, 2))
        host.append((Qw, sw, b))
    return a, ws, Qx, sx, host


@pytest.mark.parametrize("M,N,nlin", [(300, 1000, 2), (1024, 5120, 1), (100, 1000, 1)])
def test_static_scratch_matches_oracle_and_caller_workspace(cr, M, N, nlin):
    """Shapes whose last round is split: the static-scratch call equals the
    unsplit call and the caller-workspace call bit for bit, and the oracle's
    reconstruction within one bf16 ulp, on repeated calls."""
    a, ws, Qx, sx, host = _codes(cr, M, N, 1024, M + N)
    bs = [torch.from_numpy(b).cuda() for _, _, b in host]
    y_plain = cr.convrot_linear_multi(a, ws, bs)
    y_ws = cr.convrot_linear_multi(a, ws, bs, workspace=cr.gemm_workspace())
    for _ in range(3):
        y_static = cr.convrot_linear_multi_static(a, ws, bs)
        for ys, yp, yw in zip(y_static, y_plain, y_ws):
            assert torch.equal(ys, yp) and torch.equal(ys, yw)
    for ys, (Qw, sw, b) in zip(y_static, host):
        check_y_same_codes(to_np(ys.float()), O.int_gemm(Qx, Qw), sx, sw, b, f"static {M}x{N}")


def test_static_scratch_full_size_dit(cr):
    """The DiT linear at full size (4096 x 6144 x 6144, a split last round):
    bit-identical to the unsplit launch, twice in a row."""
    wl = WL.dit6144()
    a = cr.convrot_quantize_act(wl.X.cuda(), 256, "h4")
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), 256, "h4")
    b = wl.biases[0].cuda()
    y0 = cr.convrot_linear(a, w, b)
    for _ in range(2):
        y = cr.convrot_linear_multi_static(a, [w], [b])[0]
        assert torch.equal(y, y0)


def test_static_scratch_allocates_nothing(cr):
    """After the first call has located the scratch, calls change neither the
    device's free memory nor PyTorch's allocations (outputs preallocated)."""
    a, ws, _, _, host = _codes(cr, 300, 1000, 1024, 5)
    bs = [torch.from_numpy(b).cuda() for _, _, b in host]
    outs = [torch.empty((300, 1000), dtype=torch.bfloat16, device="cuda")]
    cr.convrot_linear_multi_static(a, ws, bs, outs=outs)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(5):
        cr.convrot_linear_multi_static(a, ws, bs, outs=outs)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert cr.convrot_get_device_status() == 0


def test_static_scratch_is_cleared_after_a_timeout(cr):
    """A kernel that gives up a bounded wait records a timeout; reading the
    device status then clears the static scratch, where an aborted split
    could have left partial sums. The recovery runs here because an earlier
    static call has located the scratch; the next static call still equals
    the unsplit call bit for bit."""
    a, ws, _, _, host = _codes(cr, 300, 1000, 1024, 9)
    bs = [torch.from_numpy(b).cuda() for _, _, b in host]
    y0 = cr.convrot_linear_multi(a, ws, bs)[0]
    assert torch.equal(cr.convrot_linear_multi_static(a, ws, bs)[0], y0)
    assert cr.convrot_get_device_status() == 0
    cr.convrot_selftest_wait_timeout(2000)
    assert cr.convrot_get_device_status() == 5   # CONVROT_ERR_TIMEOUT, scratch cleared
    assert cr.convrot_get_device_status() == 0
    for _ in range(2):
        assert torch.equal(cr.convrot_linear_multi_static(a, ws, bs)[0], y0)
    assert cr.convrot_get_device_status() == 0
