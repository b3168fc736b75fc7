"""The synthetic inputs: each named workload has the shapes, seed and
structure its description states (Student-t(3) or normal activations, a
seeded set of round(frac * K) outlier channels, row spikes, weight and bias
scales, +-1 block signs), and a (workload, seed) pair always gives the same
tensors. CPU only; reduced M where the workload takes one."""
import torch

import workloads as WL


def _outlier_channels(X: torch.Tensor, threshold: float = 10.0) -> int:
    """Channels whose median |x| stands far above the rest (a x30 or x50
    channel of a unit-scale distribution has a median of |x| near 20-40)."""
    med = X.float().abs().median(dim=0).values
    return int((med > threshold).sum())


def test_same_seed_same_tensors_other_seed_differs():
    a, b, c = WL.dit6144(M=16), WL.dit6144(M=16), WL.dit6144(seed=11, M=16)
    assert torch.equal(a.X, b.X) and torch.equal(a.weights[0], b.weights[0])
    assert torch.equal(a.biases[0], b.biases[0])
    assert not torch.equal(a.X, c.X)


def test_named_shapes_groups_and_dtypes():
    cases = [
        (WL.tiny(), 64, 256, [256], 256, "h4", 0),
        (WL.dit6144(M=32), 32, 6144, [6144], 256, "h4", 1),
        (WL.qkv32700(M=32), 32, 3072, [3072] * 3, 256, "h4", 2),
        (WL.ffn_pair(), 16, 1152, [6912, 6912], 128, "rht", 3),
        (WL.gsweep(64, M=32), 32, 4096, [4096], 64, "h4", 4),
        (WL.k2688(M=32), 32, 2688, [2688], 64, "h4", 5),
    ]
    for wl, M, K, Ns, G, T, seed in cases:
        assert tuple(wl.X.shape) == (M, K) and wl.X.dtype == torch.bfloat16, wl.name
        assert [tuple(W.shape) for W in wl.weights] == [(n, K) for n in Ns], wl.name
        assert all(W.dtype == torch.float32 for W in wl.weights)
        assert [tuple(b.shape) for b in wl.biases] == [(n,) for n in Ns]
        assert wl.group == G and wl.transform == T and wl.seed == seed, wl.name
        assert (wl.signs is not None) == (T == "rht")


def test_outlier_channel_counts():
    """round(frac * K) scaled channels: 6 of 6144, 3 of 3072, 4 of 4096,
    3 of 2688 at 0.1 %; 6 of 1152 at 0.5 % (the FFN pair, normal draws);
    none in the tiny workload."""
    assert _outlier_channels(WL.dit6144(M=256).X) == 6
    assert _outlier_channels(WL.qkv32700(M=256).X) == 3
    assert _outlier_channels(WL.gsweep(256, M=256).X) == 4
    assert _outlier_channels(WL.k2688(M=256).X) == 3
    assert _outlier_channels(WL.make_case(256, 1152, [], dist="normal", outlier_frac=0.005,
                                          outlier_scale=30.0, seed=3).X) == 6
    assert _outlier_channels(WL.tiny().X) == 0


def test_tiny_row_spikes():
    """Two entries of every row set to +-40 over N(0, 1) draws."""
    X = WL.tiny().X.float()
    spikes = (X.abs() == 40.0)
    assert torch.all(spikes.sum(dim=1) == 2)
    assert float(X[~spikes].abs().max()) < 10.0


def test_value_scales_and_signs():
    wl = WL.ffn_pair()
    assert set(wl.signs.tolist()) <= {-1, 1} and wl.signs.numel() == 128 and wl.signs.dtype == torch.int8
    # weights N(0, 0.03^2) for the FFN pair, N(0, 0.02^2) elsewhere; biases N(0, 0.01^2)
    W = torch.cat([w.flatten() for w in wl.weights])
    b = torch.cat(wl.biases)
    assert abs(float(W.std()) - 0.03) < 0.001 and abs(float(W.mean())) < 0.001
    assert abs(float(b.std()) - 0.01) < 0.002
    W2 = WL.k2688(M=8).weights[0]
    assert abs(float(W2.std()) - 0.02) < 0.001
    # Student-t(3) body: heavier tails than a normal, unit scale
    X = WL.make_case(512, 1024, [], dist="t3", outlier_frac=0.0, seed=9).X.float()
    med = float(X.abs().median())
    assert 0.6 < med < 0.9          # median |t3| = 0.765
    assert float((X.abs() > 5).float().mean()) > 10 * 5.7e-7  # normal: P(|z| > 5) = 5.7e-7


def test_dit_block_layers():
    blk = WL.dit_block(M=8, D=256, mlp=4)
    assert blk.layers() == [("qkv", 256, [256, 256, 256]), ("out_proj", 256, [256]),
                            ("fc1", 256, [1024]), ("fc2", 1024, [256])]
    assert tuple(blk.X.shape) == (8, 256) and tuple(blk.A.shape) == (8, 256)
    assert tuple(blk.fc1.shape) == (1024, 256) and tuple(blk.fc2.shape) == (256, 1024)
    assert blk.group == 256 and blk.transform == "h4" and blk.seed == 6


def test_bench_names_the_kernel_the_routing_rule_picks():
    """bench.py labels its rotate+quantize lines with the kernel the library
    routes the shape to; that label follows the same rule as the parity
    tests' helper (the GPU test of the rule itself is in test_gpu_quant)."""
    import types
    import bench
    from parity import tensor_core_takes
    for K in (192, 256, 320, 1088, 1152, 2688, 3072, 4032, 5376, 6144, 6208, 12288, 12416, 21504, 24576):
        for G in (4, 16, 64, 256, 1024):
            if K % G:
                continue
            wl = types.SimpleNamespace(K=K, group=G, transform="h4")
            assert (bench.rq_kernel_name(wl) == "rq_mma_kernel") == tensor_core_takes(K, G), (K, G)
    # the bench workloads' shapes: DiT, qkv, the group sweep, K = 2688
    for K, G in ((6144, 256), (3072, 256), (4096, 16), (4096, 1024), (2688, 64)):
        assert bench.rq_kernel_name(types.SimpleNamespace(K=K, group=G, transform="h4")) == "rq_mma_kernel"
    ffn = types.SimpleNamespace(K=1152, group=128, transform="rht")  # the small-M FFN pair
    assert bench.rq_kernel_name(ffn) == "rq_lane_kernel"
