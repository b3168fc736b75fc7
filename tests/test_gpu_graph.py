"""Library calls captured into CUDA graphs and replayed. Every kernel launch
is a stream operation with its arguments fixed at capture, so a replay on
new input written into the captured buffers equals the eager call on that
input bit for bit: the one-call linear (rotate+quantize, then the GEMM as its
programmatic dependent) on the large-M path with and without a split last
round, the small-M weight stream, and the 4-bit path. The tensor-core
rotate+quantize keeps the tile hand-out slot it was given at capture; a
graph replayed more often than there are slots, and two graphs replayed in
turn, still give the eager result."""
import pytest
import torch

import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def _capture(fn):
    """One warm-up call on a side stream (kernel attributes and the library's
    per-device queries happen outside the capture), then the capture."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _new_inputs(shape, seed, reps):
    rng = torch.Generator().manual_seed(seed)
    return [(torch.randn(shape, generator=rng) * (0.5 + rep)).to(torch.bfloat16) for rep in range(reps)]


@pytest.mark.parametrize("M,K,Ns,split", [(300, 3072, [3072, 3072, 1000], False), (300, 1024, [1000, 1000], True)])
def test_one_call_linear_graph_equals_eager(cr, M, K, Ns, split):
    wl = WL.make_case(M, K, Ns, seed=M + K, group=256)
    ws = [cr.convrot_prepare_weights(W.cuda(), 256, "h4") for W in wl.weights]
    bs = [b.cuda() for b in wl.biases]
    if split:  # the shape's last round is split along K through the workspace
        assert cr.gemm_tc_plan(M, K, Ns)["split_tiles"] > 0
    Xs = wl.X.cuda().clone()
    outs = [torch.empty((M, w.N), dtype=torch.bfloat16, device="cuda") for w in ws]
    scratch = cr.int8_linear_scratch(M, K)
    wsp = cr.gemm_workspace()
    g = _capture(lambda: cr.convrot_int8_linear(Xs, ws, bs, outs=outs, scratch=scratch, workspace=wsp))
    for X in _new_inputs((M, K), 7, 3):
        Xs.copy_(X.cuda())
        g.replay()
        ref = cr.convrot_int8_linear(X.cuda(), ws, bs, workspace=cr.gemm_workspace())
        torch.cuda.synchronize()
        for y, r in zip(outs, ref):
            assert torch.equal(y, r)
    assert cr.convrot_get_device_status() == 0


def test_small_m_pair_graph_equals_eager(cr):
    """The gated-FFN pair: 16 rows, block-128 randomized Hadamard, the weight
    stream kernel."""
    wl = WL.ffn_pair()
    sg = wl.signs.cuda()
    ws = [cr.convrot_prepare_weights(W.cuda(), wl.group, wl.transform, sg) for W in wl.weights]
    bs = [b.cuda() for b in wl.biases]
    M, K = wl.X.shape
    Xs = wl.X.cuda().clone()
    outs = [torch.empty((M, w.N), dtype=torch.bfloat16, device="cuda") for w in ws]
    scratch = cr.int8_linear_scratch(M, K)
    g = _capture(lambda: cr.convrot_int8_linear(Xs, ws, bs, signs=sg, outs=outs, scratch=scratch))
    for X in _new_inputs((M, K), 8, 3):
        Xs.copy_(X.cuda())
        g.replay()
        ref = cr.convrot_int8_linear(X.cuda(), ws, bs, signs=sg)
        torch.cuda.synchronize()
        for y, r in zip(outs, ref):
            assert torch.equal(y, r)
    assert cr.convrot_get_device_status() == 0


def test_four_bit_path_graph_equals_eager(cr):
    wl = WL.make_case(300, 2048, [1000, 512], seed=41, group=256)
    ws = [cr.convrot_prepare_weights4(W.cuda(), 256, "h4") for W in wl.weights]
    bs = [b.cuda() for b in wl.biases]
    Xs = wl.X.cuda().clone()
    a = cr.convrot_quantize_act4(Xs, 256, "h4")
    outs = [torch.empty((300, w.N), dtype=torch.bfloat16, device="cuda") for w in ws]

    def step():
        cr.convrot_quantize_act4(Xs, 256, "h4", out=a)
        cr.convrot_linear4_multi(a, ws, bs, outs=outs)

    g = _capture(step)
    for X in _new_inputs((300, 2048), 9, 3):
        Xs.copy_(X.cuda())
        g.replay()
        ref = cr.convrot_linear4_multi(cr.convrot_quantize_act4(X.cuda(), 256, "h4"), ws, bs)
        torch.cuda.synchronize()
        for y, r in zip(outs, ref):
            assert torch.equal(y, r)
    assert cr.convrot_get_device_status() == 0


def test_rotate_quantize_graphs_keep_their_slots(cr):
    """Two captured tensor-core rotate+quantize launches (two hand-out slots),
    replayed in turn and one of them 300 times in a row (more replays than
    slots): each replay gives the eager result."""
    wl = WL.make_case(500, 3072, [], seed=43, group=256)
    X1 = wl.X.cuda().clone()
    X2 = (wl.X * 3).to(torch.bfloat16).cuda()
    a1 = cr.convrot_quantize_act(X1, 256, "h4")
    a2 = cr.convrot_quantize_act(X2, 256, "h4")
    ref1 = cr.convrot_quantize_act(X1, 256, "h4")
    ref2 = cr.convrot_quantize_act(X2, 256, "h4")
    g1 = _capture(lambda: cr.convrot_quantize_act(X1, 256, "h4", out=a1))
    g2 = _capture(lambda: cr.convrot_quantize_act(X2, 256, "h4", out=a2))
    for _ in range(10):
        a1.q.zero_()
        a2.q.zero_()
        g1.replay()
        g2.replay()
        torch.cuda.synchronize()
        assert torch.equal(a1.q, ref1.q) and torch.equal(a1.scale, ref1.scale) and torch.equal(a1.q_f16, ref1.q_f16)
        assert torch.equal(a2.q, ref2.q) and torch.equal(a2.scale, ref2.scale) and torch.equal(a2.q_f16, ref2.q_f16)
    a1.q.zero_()
    for _ in range(300):
        g1.replay()
    torch.cuda.synchronize()
    assert torch.equal(a1.q, ref1.q) and torch.equal(a1.scale, ref1.scale)
    assert cr.convrot_get_device_status() == 0
