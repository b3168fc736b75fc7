"""Quantization error of the three rotations on the same outlier-heavy DiT
inputs, end to end on the GPU, against the unquantized fp64 product from the
oracle: the comparison of rotated and naive W8A8 that the gemma.cpp issue
makes ("Results", mean KL of rotated vs naive) and that motivates ConvRot
("INT8 Convrot Safetensors", "How INT8 convrot works": the rotation spreads
outlier channels over the group before the per-row scale is taken)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from parity import to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def _relative_error(cr, wl, rows):
    sg = None if wl.signs is None else wl.signs.cuda()
    w = cr.convrot_prepare_weights(wl.weights[0].cuda(), wl.group, wl.transform, sg)
    a = cr.convrot_quantize_act(wl.X[rows].cuda(), wl.group, wl.transform, sg)
    y = to_np(cr.convrot_linear(a, w, wl.biases[0].cuda()).float()).astype(np.float64)
    ref = O.float_linear(wl.X[rows].float().numpy().astype(np.float64),
                         wl.weights[0].numpy().astype(np.float64), wl.biases[0].numpy())
    return float(np.linalg.norm(y - ref) / np.linalg.norm(ref))


def test_rotation_reduces_quantization_error(cr):
    """Student-t(3) activations with 0.1 % channels x50 (the DiT workload's
    inputs, 256 rows): the regular Hadamard (G = 256) and the randomized
    Hadamard (B = 128, 256) each cut the relative error of Y well below the
    naive W8A8 error."""
    rows = torch.arange(0, 4096, 16)
    err = {}
    for name, wl in [("h4 G256", WL.dit6144(M=4096)), ("rht B128", WL.dit6144_variant("rht", 128)),
                     ("rht B256", WL.dit6144_variant("rht", 256)), ("none", WL.dit6144_variant("none", 0))]:
        err[name] = _relative_error(cr, wl, rows)
    print("relative Frobenius error of Y vs the fp64 product:",
          ", ".join(f"{k} {v:.4g}" for k, v in err.items()))
    for k in ("h4 G256", "rht B128", "rht B256"):
        assert err[k] < 0.5 * err["none"], (k, err)


def _relative_error4(cr, wl, rows):
    sg = None if wl.signs is None else wl.signs.cuda()
    w = cr.convrot_prepare_weights4(wl.weights[0].cuda(), wl.group, wl.transform, sg)
    a = cr.convrot_quantize_act4(wl.X[rows].cuda(), wl.group, wl.transform, sg)
    y = to_np(cr.convrot_linear4(a, w, wl.biases[0].cuda()).float()).astype(np.float64)
    ref = O.float_linear(wl.X[rows].float().numpy().astype(np.float64),
                         wl.weights[0].numpy().astype(np.float64), wl.biases[0].numpy())
    return float(np.linalg.norm(y - ref) / np.linalg.norm(ref))


def test_rotation_reduces_4bit_error(cr):
    """The same comparison at 4 bits (codes in [-7, 7]): rotating before the
    per-row scale still roughly halves the error of the naive path."""
    rows = torch.arange(0, 4096, 16)
    err = {name: _relative_error4(cr, wl, rows) for name, wl in [
        ("h4 G256", WL.dit6144()), ("rht B256", WL.dit6144_variant("rht", 256)),
        ("none", WL.dit6144_variant("none", 0))]}
    print("W4A4 relative Frobenius error of Y vs the fp64 product:",
          ", ".join(f"{k} {v:.4g}" for k, v in err.items()))
    for k in ("h4 G256", "rht B256"):
        assert err[k] < 0.7 * err["none"], (k, err)
