"""Seeded synthetic inputs for the INT8 ConvRot W8A8 linear.

This module only draws random numbers. It holds none of the method's
arithmetic (no rotation, no quantisation, no GEMM), so that both the CUDA
path and the CPU oracle can be fed from it without sharing any of the
computation they are compared on.

Every tensor is drawn on the CPU from a ``torch.Generator`` seeded with the
workload's seed, so a (workload, seed) pair always yields the same values in
one process. Activations are drawn in fp32 and rounded once to bf16;
weights and biases stay fp32.

Distributions (stand-ins for the pages' DiT / Gemma layers, which are not
available as data):

* ``normal``:  X ~ N(0, 1)
* ``t3``:      X ~ Student-t with 3 degrees of freedom, built as
               Z / sqrt(V / 3) with Z ~ N(0,1) and V = sum of three squared
               N(0,1) draws (the textbook construction of Student-t).
* outlier channels: a seeded set of round(frac * K) input channels (the same
  channels for every row) is multiplied by a fixed factor.
* row spikes: a fixed number of seeded positions per row are overwritten
  with +-value (random sign).
* weights W ~ N(0, w_std^2), bias ~ N(0, b_std^2).
* block-RHT signs: seeded +-1 values (one vector, reused by every block).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch

TRANSFORM_H4 = "h4"      # regular Hadamard, Kronecker power of H4
TRANSFORM_RHT = "rht"    # block randomized Hadamard (signs, Walsh-Hadamard, 1/sqrt(B))
TRANSFORM_NONE = "none"  # naive W8A8, no rotation


@dataclasses.dataclass
class Workload:
    name: str
    X: torch.Tensor                 # bf16 [M, K]
    weights: List[torch.Tensor]     # fp32 [N_i, K] each
    biases: List[torch.Tensor]      # fp32 [N_i] each
    group: int
    transform: str
    signs: Optional[torch.Tensor]   # int8 [group] for "rht", else None
    seed: int
    description: str = ""

    @property
    def M(self) -> int:
        return self.X.shape[0]

    @property
    def K(self) -> int:
        return self.X.shape[1]

    @property
    def Ns(self) -> List[int]:
        return [w.shape[0] for w in self.weights]


def _gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def student_t3(g: torch.Generator, shape) -> torch.Tensor:
    z = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.zeros(shape, dtype=torch.float32)
    for _ in range(3):
        e = torch.randn(shape, generator=g, dtype=torch.float32)
        v.add_(e * e)
    return z / torch.sqrt(v / 3.0)


def draw_activations(g: torch.Generator, M: int, K: int, dist: str = "t3",
                     outlier_frac: float = 0.0, outlier_scale: float = 1.0,
                     row_spikes: int = 0, spike_value: float = 0.0) -> torch.Tensor:
    """bf16 [M, K] activations with the requested structure."""
    if dist == "t3":
        X = student_t3(g, (M, K))
    elif dist == "normal":
        X = torch.randn((M, K), generator=g, dtype=torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    n_out = int(round(outlier_frac * K))
    if n_out > 0:
        ch = torch.randperm(K, generator=g)[:n_out]
        X[:, ch] *= outlier_scale
    if row_spikes > 0 and M > 0:
        pos = torch.rand((M, K), generator=g).argsort(dim=1)[:, :row_spikes]
        sign = torch.randint(0, 2, (M, row_spikes), generator=g).float() * 2 - 1
        X.scatter_(1, pos, sign * spike_value)
    return X.to(torch.bfloat16)


def draw_signs(g: torch.Generator, B: int) -> torch.Tensor:
    return (torch.randint(0, 2, (B,), generator=g) * 2 - 1).to(torch.int8)


def make_case(M: int, K: int, Ns: List[int], *, dist: str = "t3",
              outlier_frac: float = 0.001, outlier_scale: float = 50.0,
              row_spikes: int = 0, spike_value: float = 0.0,
              w_std: float = 0.02, b_std: float = 0.01,
              group: int = 256, transform: str = TRANSFORM_H4,
              seed: int = 0, name: str = "case") -> Workload:
    g = _gen(seed)
    X = draw_activations(g, M, K, dist, outlier_frac, outlier_scale,
                         row_spikes, spike_value)
    weights, biases = [], []
    for N in Ns:
        weights.append(torch.randn((N, K), generator=g, dtype=torch.float32) * w_std)
        biases.append(torch.randn((N,), generator=g, dtype=torch.float32) * b_std)
    signs = draw_signs(g, group) if transform == TRANSFORM_RHT else None
    return Workload(name, X, weights, biases, group, transform, signs, seed)


# --- the named workloads ----------------------------------------------------
# Shapes follow the pages' layers: a 6144-wide DiT linear, the MiniMax-H3 qkv
# projection at 32700 tokens, a Gemma 3 1B gated-FFN pair (1152 -> 6912) with
# block-128 randomized Hadamard, and a 4096-wide group-size sweep plus the
# 2688-wide AdaLN projection.

def tiny(seed: int = 0) -> Workload:
    w = make_case(64, 256, [256], dist="normal", outlier_frac=0.0,
                  row_spikes=2, spike_value=40.0, w_std=0.02, b_std=0.01,
                  group=256, seed=seed, name="tiny_64x256x256_G256")
    w.description = ("X bf16 [64,256] ~N(0,1), 2 entries/row set to +-40; "
                     "W fp32 [256,256] ~N(0,0.02^2); bias ~N(0,0.01^2); G=256")
    return w


def dit6144(seed: int = 1, M: int = 4096) -> Workload:
    w = make_case(M, 6144, [6144], dist="t3", outlier_frac=0.001,
                  outlier_scale=50.0, group=256, seed=seed,
                  name=f"dit_linear_{M}x6144x6144_G256")
    w.description = ("X bf16 [M,6144] Student-t(3), 0.1% channels x50; "
                     "W [6144,6144] ~N(0,0.02^2); bias ~N(0,0.01^2); G=256")
    return w


def dit6144_variant(transform: str, group: int, seed: int = 1, M: int = 4096) -> Workload:
    """The DiT linear's inputs (same seed, so the same X, W and bias) under
    another rotation: the block randomized Hadamard or none (naive W8A8)."""
    w = make_case(M, 6144, [6144], dist="t3", outlier_frac=0.001,
                  outlier_scale=50.0, group=group, transform=transform, seed=seed,
                  name=f"dit_linear_{M}x6144x6144_{transform.upper()}{group if transform != 'none' else ''}")
    w.description = ("X bf16 [M,6144] Student-t(3), 0.1% channels x50; "
                     f"W [6144,6144] ~N(0,0.02^2); bias ~N(0,0.01^2); {transform} {group}")
    return w


def qkv32700(seed: int = 2, M: int = 32700) -> Workload:
    w = make_case(M, 3072, [3072, 3072, 3072], dist="t3", outlier_frac=0.001,
                  outlier_scale=50.0, group=256, seed=seed,
                  name=f"qkv_{M}x3072x(3x3072)_G256")
    w.description = ("X bf16 [M,3072] Student-t(3), 0.1% channels x50; three "
                     "W [3072,3072] ~N(0,0.02^2) sharing one packed activation; G=256")
    return w


def ffn_pair(seed: int = 3, M: int = 16) -> Workload:
    w = make_case(M, 1152, [6912, 6912], dist="normal", outlier_frac=0.005,
                  outlier_scale=30.0, w_std=0.03, group=128,
                  transform=TRANSFORM_RHT, seed=seed,
                  name=f"ffn_pair_{M}x1152x(2x6912)_RHT128")
    w.description = ("X bf16 [M,1152] ~N(0,1), 0.5% channels x30; gate/up W "
                     "[6912,1152] ~N(0,0.03^2) sharing one packed activation; "
                     "block-128 randomized Hadamard with seeded signs")
    return w


def gsweep(G: int, seed: int = 4, M: int = 8192) -> Workload:
    w = make_case(M, 4096, [4096], dist="t3", outlier_frac=0.001,
                  outlier_scale=50.0, group=G, seed=seed,
                  name=f"gsweep_{M}x4096x4096_G{G}")
    w.description = f"X bf16 [M,4096] Student-t(3), 0.1% channels x50; W [4096,4096]; G={G}"
    return w


def k2688(seed: int = 5, M: int = 8192) -> Workload:
    w = make_case(M, 2688, [2688], dist="t3", outlier_frac=0.001,
                  outlier_scale=50.0, group=64, seed=seed,
                  name=f"k2688_{M}x2688x2688_G64")
    w.description = "X bf16 [M,2688] Student-t(3), 0.1% channels x50; W [2688,2688]; G=64"
    return w


@dataclasses.dataclass
class BlockWorkload:
    """The linears of one DiT block, chained: qkv (three linears sharing the
    block input X), the output projection on the attention output A, then the
    MLP pair fc1 (D -> mlp*D) and fc2 (mlp*D -> D), fc2 fed with fc1's output
    and fc1 with the output projection's. Every layer uses the same group."""
    name: str
    X: torch.Tensor                 # bf16 [M, D], the block input (qkv)
    A: torch.Tensor                 # bf16 [M, D], stand-in for the attention output
    qkv: List[torch.Tensor]         # 3 x fp32 [D, D]
    qkv_b: List[torch.Tensor]
    out: torch.Tensor               # fp32 [D, D]
    out_b: torch.Tensor
    fc1: torch.Tensor               # fp32 [mlp*D, D]
    fc1_b: torch.Tensor
    fc2: torch.Tensor               # fp32 [D, mlp*D]
    fc2_b: torch.Tensor
    group: int
    transform: str
    seed: int
    description: str = ""

    @property
    def M(self) -> int:
        return self.X.shape[0]

    @property
    def D(self) -> int:
        return self.X.shape[1]

    def layers(self):
        """(name, K, [N...]) of the four linear groups, in block order."""
        D, H = self.D, self.fc1.shape[0]
        return [("qkv", D, [D, D, D]), ("out_proj", D, [D]), ("fc1", D, [H]), ("fc2", H, [D])]


def dit_block(seed: int = 6, M: int = 4096, D: int = 5376, mlp: int = 4) -> BlockWorkload:
    """A MiniMax-H3-style DiT block: hidden width 5376 (the narrow out_proj /
    fc2 output of the sglang digest's row-split note), qkv 3 x 5376, MLP ratio
    4 (the pages give no MLP width: the common DiT ratio), G = 256, inputs as
    for the 6144-wide DiT linear."""
    g = _gen(seed)
    X = draw_activations(g, M, D, "t3", 0.001, 50.0, 0, 0.0)
    A = draw_activations(g, M, D, "t3", 0.001, 50.0, 0, 0.0)

    def lin(n, k):
        return (torch.randn((n, k), generator=g, dtype=torch.float32) * 0.02,
                torch.randn((n,), generator=g, dtype=torch.float32) * 0.01)

    qkv = [lin(D, D) for _ in range(3)]
    out, out_b = lin(D, D)
    fc1, fc1_b = lin(mlp * D, D)
    fc2, fc2_b = lin(D, mlp * D)
    b = BlockWorkload(f"dit_block_{M}x{D}_mlp{mlp}_G256", X, A, [w for w, _ in qkv], [bb for _, bb in qkv],
                      out, out_b, fc1, fc1_b, fc2, fc2_b, 256, TRANSFORM_H4, seed)
    b.description = (f"X, A bf16 [{M},{D}] Student-t(3), 0.1% channels x50; qkv 3x[{D},{D}], out_proj "
                     f"[{D},{D}], fc1 [{mlp * D},{D}], fc2 [{D},{mlp * D}] ~N(0,0.02^2); biases ~N(0,0.01^2); "
                     "G=256; fc1 reads out_proj's output, fc2 reads fc1's")
    return b
