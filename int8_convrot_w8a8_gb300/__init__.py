"""GB300-native INT8 ConvRot W8A8 linear layer.

A thin Python binding over ``libconvrot.so`` (C ABI declared in
``include/convrot.h``). This module only marshals arguments: it allocates
output tensors with PyTorch, passes raw device pointers and the current CUDA
stream to the library, and turns status codes into exceptions. Every step of
the layer (rotation, quantization, GEMM, reconstruction) runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback.

The layer ("INT8 Convrot Safetensors", stable-diffusion.cpp docs, sections
"How INT8 convrot works", "Weight quantization", "Runtime activation
quantization"):

    X_rot = X R, s_x = max|X_rot|/127 per row, Q_x = round(X_rot/s_x)
    A = Q_x Q_w^T (int32),  Y = A * s_x * s_w + b   (bf16)
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import List, Optional, Sequence

import torch

__all__ = [
    "ConvRotError", "PackedAct", "PackedWeight", "ConvRotLinear", "TRANSFORMS",
    "convrot_prepare_weights", "convrot_quantize_act", "convrot_quantize_act_hmatmul",
    "convrot_quantize_act_kernel", "RQ_KERNELS", "convrot_rotate_absmax", "convrot_quantize_act_given_max",
    "convrot_dequant",
    "convrot_linear", "convrot_linear_multi", "convrot_linear_multi_static", "convrot_gemm_s32", "gemm_workspace",
    "GEMM_WORKSPACE_BYTES", "convrot_get_device_status", "convrot_selftest_wait_timeout", "lib", "lib_path",
    "PackedAct4", "PackedWeight4", "convrot_prepare_weights4", "convrot_quantize_act4", "convrot_linear4",
    "convrot_linear4_multi", "convrot_gemm4_s32", "convrot_int8_linear", "int8_linear_scratch",
    "gemm_tc_plan",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_PKG, "libconvrot.so")

TRANSFORMS = {"h4": 0, "rht": 1, "none": 2}
# CONVROT_GEMM_WORKSPACE_BYTES: scratch that lets the GEMM split a mostly idle
# last round of tiles along K
GEMM_WORKSPACE_BYTES = 4096 + 40 * 256 * 1024
_DTYPE_F32, _DTYPE_BF16 = 0, 1
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED_GROUP", 3: "ALIGNMENT", 4: "CUDA", 5: "TIMEOUT"}


class ConvRotError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"convrot {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _load():
    if not os.path.exists(lib_path):
        raise ImportError(
            f"{lib_path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(nvcc, sm_103a). There is no fallback implementation.")
    return ctypes.CDLL(lib_path)


lib = _load()


class _Act(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("q_f16", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("group", ctypes.c_int32),
                ("transform", ctypes.c_int32)]


class _Weight(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("q_f16", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("group", ctypes.c_int32),
                ("transform", ctypes.c_int32)]


class _Act4(ctypes.Structure):
    _fields_ = [("q4", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("q_f8", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("group", ctypes.c_int32),
                ("transform", ctypes.c_int32)]


class _Weight4(ctypes.Structure):
    _fields_ = [("q4", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("q_f8", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("group", ctypes.c_int32),
                ("transform", ctypes.c_int32)]


_P, _I64, _I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
_SIGS = {
    "convrot_prepare_weights": [_P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P],
    "convrot_quantize_act": [_P, _I64, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P],
    "convrot_quantize_act_hmatmul": [_P, _I64, _I64, _I64, _I32, _P, _P, _P, _P],
    "convrot_quantize_act_kernel": [_P, _I64, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _I32, _P],
    "convrot_rotate_absmax": [_P, _I64, _I64, _I64, _I32, _I32, _P, _P],
    "convrot_quantize_act_given_max": [_P, _I64, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P],
    "convrot_dequant": [_P, _I64, _I64, _I64, _P, _P, _P, _P, _I64, _P],
    "convrot_linear": [ctypes.POINTER(_Act), ctypes.POINTER(_Weight), _P, _P, _I64, _P],
    "convrot_linear_multi": [ctypes.POINTER(_Act), _I32, ctypes.POINTER(_Weight), ctypes.POINTER(_P),
                             ctypes.POINTER(_P), ctypes.POINTER(_I64), _P],
    "convrot_linear_multi_ws": [ctypes.POINTER(_Act), _I32, ctypes.POINTER(_Weight), ctypes.POINTER(_P),
                                ctypes.POINTER(_P), ctypes.POINTER(_I64), _P, _I64, _P],
    "convrot_gemm_s32": [ctypes.POINTER(_Act), ctypes.POINTER(_Weight), _P, _I64, _P],
    "convrot_linear_multi_int8mma": [ctypes.POINTER(_Act), _I32, ctypes.POINTER(_Weight), ctypes.POINTER(_P),
                                     ctypes.POINTER(_P), ctypes.POINTER(_I64), _P],
    "convrot_gemm_s32_int8mma": [ctypes.POINTER(_Act), ctypes.POINTER(_Weight), _P, _I64, _P],
    "convrot_gemm_s32_ws": [ctypes.POINTER(_Act), ctypes.POINTER(_Weight), _P, _I64, _P, _I64, _P],
    "convrot_linear_multi_static": [ctypes.POINTER(_Act), _I32, ctypes.POINTER(_Weight), ctypes.POINTER(_P),
                                    ctypes.POINTER(_P), ctypes.POINTER(_I64), _P],
    "convrot_prepare_weights4": [_P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P],
    "convrot_quantize_act4": [_P, _I64, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P],
    "convrot_linear4_multi": [ctypes.POINTER(_Act4), _I32, ctypes.POINTER(_Weight4), ctypes.POINTER(_P),
                              ctypes.POINTER(_P), ctypes.POINTER(_I64), _P, _I64, _P],
    "convrot_gemm4_s32": [ctypes.POINTER(_Act4), ctypes.POINTER(_Weight4), _P, _I64, _P, _I64, _P],
    "convrot_int8_linear_scratch_bytes": [_I64, _I64],
    "convrot_int8_linear": [_P, _I64, _I64, _I64, _I32, _I32, _P, _I32, ctypes.POINTER(_Weight), ctypes.POINTER(_P),
                            ctypes.POINTER(_P), ctypes.POINTER(_I64), _P, _I64, _P, _I64, _P],
    "convrot_gemm_tc_plan": [_I64, _I64, _I32, ctypes.POINTER(_I64), _I32, _I32, _I64, ctypes.POINTER(_I32),
                             ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I32)],
    "convrot_get_device_status": [],
    "convrot_selftest_wait_timeout": [_I64, _P],
    "convrot_status_str": [_I32],
    "convrot_last_error": [],
    "convrot_version": [],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = (ctypes.c_char_p if _name in ("convrot_status_str", "convrot_last_error") else
                  ctypes.c_int64 if _name == "convrot_int8_linear_scratch_bytes" else ctypes.c_int32)

EXPORTED = tuple(_SIGS)


def _check(status: int) -> None:
    if status != 0:
        msg = lib.convrot_last_error().decode(errors="replace")
        raise ConvRotError(status, msg or lib.convrot_status_str(status).decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _transform_id(transform) -> int:
    if isinstance(transform, int):
        return transform
    return TRANSFORMS[transform]


@dataclasses.dataclass
class PackedAct:
    """{int8 rows, fp32 row scales} (+ fp16 operand copy), reusable by every
    linear that shares the input and the group size."""
    q: torch.Tensor
    scale: torch.Tensor
    q_f16: Optional[torch.Tensor]
    group: int
    transform: int

    @property
    def M(self) -> int:
        return self.q.shape[0]

    @property
    def K(self) -> int:
        return self.q.shape[1]

    def _c(self) -> _Act:
        return _Act(_ptr(self.q), _ptr(self.scale), _ptr(self.q_f16), self.M, self.K, self.group, self.transform)


@dataclasses.dataclass
class PackedWeight:
    q: torch.Tensor
    scale: torch.Tensor
    q_f16: Optional[torch.Tensor]
    group: int
    transform: int

    @property
    def N(self) -> int:
        return self.q.shape[0]

    @property
    def K(self) -> int:
        return self.q.shape[1]

    def _c(self) -> _Weight:
        return _Weight(_ptr(self.q), _ptr(self.scale), _ptr(self.q_f16), self.N, self.K, self.group,
                       self.transform)


def convrot_prepare_weights(W: torch.Tensor, group: int, transform="h4", signs: Optional[torch.Tensor] = None,
                            with_f16: bool = True, stream=None) -> PackedWeight:
    """Offline path: W_rot = W R, per-output-row int8 (Q_w, s_w)."""
    if W.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("W must be fp32 or bf16")
    W = W.contiguous()
    N, K = W.shape
    t = _transform_id(transform)
    q = torch.empty((N, K), dtype=torch.int8, device=W.device)
    s = torch.empty((N,), dtype=torch.float32, device=W.device)
    q16 = torch.empty((N, K), dtype=torch.float16, device=W.device) if with_f16 else None
    _check(lib.convrot_prepare_weights(W.data_ptr(), _DTYPE_F32 if W.dtype == torch.float32 else _DTYPE_BF16,
                                       N, K, group, t, _ptr(signs), q.data_ptr(), s.data_ptr(), _ptr(q16),
                                       _stream(stream)))
    return PackedWeight(q, s, q16, group, t)


def convrot_quantize_act(X: torch.Tensor, group: int, transform="h4", signs: Optional[torch.Tensor] = None,
                         with_f16: bool = True, out: Optional[PackedAct] = None, stream=None) -> PackedAct:
    """Runtime path: fused X_rot = X R, per-row absmax scale, int8 codes."""
    if X.dtype != torch.bfloat16 or X.dim() != 2:
        raise TypeError("X must be a 2-D bf16 tensor")
    if X.stride(1) != 1:
        X = X.contiguous()
    M, K = X.shape
    t = _transform_id(transform)
    if out is None:
        q = torch.empty((M, K), dtype=torch.int8, device=X.device)
        s = torch.empty((M,), dtype=torch.float32, device=X.device)
        q16 = torch.empty((M, K), dtype=torch.float16, device=X.device) if with_f16 else None
        out = PackedAct(q, s, q16, group, t)
    _check(lib.convrot_quantize_act(X.data_ptr(), M, K, X.stride(0), group, t, _ptr(signs), out.q.data_ptr(),
                                    out.scale.data_ptr(), _ptr(out.q_f16), _stream(stream)))
    return out


RQ_KERNELS = {"auto": 0, "generic": 1, "butterfly": 2, "tensor_core": 3}


def convrot_quantize_act_kernel(X: torch.Tensor, group: int, transform="h4", signs: Optional[torch.Tensor] = None,
                                kernel: str = "auto", with_f16: bool = True, out: Optional[PackedAct] = None,
                                stream=None) -> PackedAct:
    """convrot_quantize_act with the rotate+quantize kernel chosen by name
    ("auto", "generic", "butterfly", "tensor_core"); raises if that kernel
    does not take the shape."""
    if X.dtype != torch.bfloat16 or X.dim() != 2:
        raise TypeError("X must be a 2-D bf16 tensor")
    if X.stride(1) != 1:
        X = X.contiguous()
    M, K = X.shape
    t = _transform_id(transform)
    if out is None:
        q = torch.empty((M, K), dtype=torch.int8, device=X.device)
        s = torch.empty((M,), dtype=torch.float32, device=X.device)
        q16 = torch.empty((M, K), dtype=torch.float16, device=X.device) if with_f16 else None
        out = PackedAct(q, s, q16, group, t)
    _check(lib.convrot_quantize_act_kernel(X.data_ptr(), M, K, X.stride(0), group, t, _ptr(signs),
                                           out.q.data_ptr(), out.scale.data_ptr(), _ptr(out.q_f16),
                                           RQ_KERNELS[kernel], _stream(stream)))
    return out


def convrot_rotate_absmax(X: torch.Tensor, group: int, transform="h4", out: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """Row-parallel step 1: amax[r] = max |X_rot[r, :]| over X's columns (a
    slice of whole groups of a longer row), fp32 [M]."""
    if X.dtype != torch.bfloat16 or X.dim() != 2 or X.stride(1) != 1:
        raise TypeError("X must be a 2-D bf16 tensor with unit column stride")
    M, K = X.shape
    if out is None:
        out = torch.empty((M,), dtype=torch.float32, device=X.device)
    _check(lib.convrot_rotate_absmax(X.data_ptr(), M, K, X.stride(0), group, _transform_id(transform),
                                     out.data_ptr(), _stream(stream)))
    return out


def convrot_quantize_act_given_max(X: torch.Tensor, amax: torch.Tensor, group: int, transform="h4",
                                   with_f16: bool = True, out: Optional[PackedAct] = None,
                                   stream=None) -> PackedAct:
    """Row-parallel step 3: quantize X's columns with the whole row's maxima
    (amax fp32 [M], the all-reduced step-1 values)."""
    if X.dtype != torch.bfloat16 or X.dim() != 2 or X.stride(1) != 1:
        raise TypeError("X must be a 2-D bf16 tensor with unit column stride")
    M, K = X.shape
    t = _transform_id(transform)
    if out is None:
        q = torch.empty((M, K), dtype=torch.int8, device=X.device)
        s = torch.empty((M,), dtype=torch.float32, device=X.device)
        q16 = torch.empty((M, K), dtype=torch.float16, device=X.device) if with_f16 else None
        out = PackedAct(q, s, q16, group, t)
    _check(lib.convrot_quantize_act_given_max(X.data_ptr(), M, K, X.stride(0), group, t, amax.data_ptr(),
                                              out.q.data_ptr(), out.scale.data_ptr(), _ptr(out.q_f16),
                                              _stream(stream)))
    return out


def convrot_dequant(A: torch.Tensor, sx: torch.Tensor, sw: torch.Tensor, bias: Optional[torch.Tensor] = None,
                    out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Y = A * s_x * s_w + b (bf16) from int32 accumulators (row-parallel
    step 6, after the all-reduce of the partial A)."""
    if A.dtype != torch.int32 or A.dim() != 2:
        raise TypeError("A must be a 2-D int32 tensor")
    M, N = A.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check(lib.convrot_dequant(A.data_ptr(), M, N, A.stride(0), sx.data_ptr(), sw.data_ptr(), _ptr(bias),
                               out.data_ptr(), out.stride(0), _stream(stream)))
    return out


def convrot_quantize_act_hmatmul(X: torch.Tensor, group: int, with_f16: bool = True, stream=None) -> PackedAct:
    """Same result as convrot_quantize_act (regular Hadamard), with the
    rotation applied as a dense G x G matmul on the tensor cores."""
    if X.dtype != torch.bfloat16 or X.dim() != 2:
        raise TypeError("X must be a 2-D bf16 tensor")
    if X.stride(1) != 1:
        X = X.contiguous()
    M, K = X.shape
    q = torch.empty((M, K), dtype=torch.int8, device=X.device)
    s = torch.empty((M,), dtype=torch.float32, device=X.device)
    q16 = torch.empty((M, K), dtype=torch.float16, device=X.device) if with_f16 else None
    _check(lib.convrot_quantize_act_hmatmul(X.data_ptr(), M, K, X.stride(0), group, q.data_ptr(), s.data_ptr(),
                                            _ptr(q16), _stream(stream)))
    return PackedAct(q, s, q16, group, TRANSFORMS["h4"])


def gemm_workspace(device=None) -> torch.Tensor:
    """A zeroed GEMM workspace (caller-owned; calls sharing it must be ordered,
    e.g. on one stream). Every completed call leaves it zeroed again."""
    return torch.zeros(GEMM_WORKSPACE_BYTES, dtype=torch.uint8, device=device or "cuda")


def convrot_linear(a: PackedAct, w: PackedWeight, bias: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None, stream=None,
                   workspace: Optional[torch.Tensor] = None, int8_mma: bool = False) -> torch.Tensor:
    """Y = A * s_x * s_w + b (bf16) for one linear. Above 64 rows the
    tensor-core GEMM needs the fp16 operand copies; ``int8_mma=True`` runs the
    int8 warp-MMA GEMM instead (no copies needed, about 11x slower)."""
    if out is None:
        out = torch.empty((a.M, w.N), dtype=torch.bfloat16, device=a.q.device)
    if workspace is not None or int8_mma:
        return convrot_linear_multi(a, [w], [bias], outs=[out], stream=stream, workspace=workspace,
                                    int8_mma=int8_mma)[0]
    ca, cw = a._c(), w._c()
    _check(lib.convrot_linear(ctypes.byref(ca), ctypes.byref(cw), _ptr(bias), out.data_ptr(), out.stride(0),
                              _stream(stream)))
    return out


def convrot_linear_multi(a: PackedAct, ws: Sequence[PackedWeight], biases: Optional[Sequence] = None,
                         outs: Optional[List[torch.Tensor]] = None, stream=None,
                         workspace: Optional[torch.Tensor] = None, int8_mma: bool = False) -> List[torch.Tensor]:
    """Several linears sharing one packed activation, in one launch
    (``int8_mma``: the int8 warp-MMA GEMM, asked for by name)."""
    n = len(ws)
    if outs is None:
        outs = [torch.empty((a.M, w.N), dtype=torch.bfloat16, device=a.q.device) for w in ws]
    warr = (_Weight * n)(*[w._c() for w in ws])
    barr = (ctypes.c_void_p * n)(*[(_ptr(b) if b is not None else None) for b in (biases or [None] * n)])
    yarr = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    larr = (ctypes.c_int64 * n)(*[o.stride(0) for o in outs])
    ca = a._c()
    if int8_mma:
        if workspace is not None:
            raise ValueError("the int8 warp-MMA GEMM takes no workspace")
        _check(lib.convrot_linear_multi_int8mma(ctypes.byref(ca), n, warr, barr, yarr, larr, _stream(stream)))
    elif workspace is None:
        _check(lib.convrot_linear_multi(ctypes.byref(ca), n, warr, barr, yarr, larr, _stream(stream)))
    else:
        _check(lib.convrot_linear_multi_ws(ctypes.byref(ca), n, warr, barr, yarr, larr, workspace.data_ptr(),
                                           workspace.numel() * workspace.element_size(), _stream(stream)))
    return outs


def convrot_linear_multi_static(a: PackedAct, ws: Sequence[PackedWeight], biases: Optional[Sequence] = None,
                                outs: Optional[List[torch.Tensor]] = None, stream=None) -> List[torch.Tensor]:
    """convrot_linear_multi with the library's static per-device GEMM scratch
    (the library allocates nothing). Calls that may overlap on the GPU race
    on that scratch: keep them on one stream."""
    n = len(ws)
    if outs is None:
        outs = [torch.empty((a.M, w.N), dtype=torch.bfloat16, device=a.q.device) for w in ws]
    warr = (_Weight * n)(*[w._c() for w in ws])
    barr = (ctypes.c_void_p * n)(*[(_ptr(b) if b is not None else None) for b in (biases or [None] * n)])
    yarr = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    larr = (ctypes.c_int64 * n)(*[o.stride(0) for o in outs])
    ca = a._c()
    _check(lib.convrot_linear_multi_static(ctypes.byref(ca), n, warr, barr, yarr, larr, _stream(stream)))
    return outs


def gemm_tc_plan(M: int, K: int, Ns: Sequence[int], bits: int = 8, sms: int = 152,
                 workspace_bytes: int = GEMM_WORKSPACE_BYTES) -> dict:
    """The large-M tensor-core GEMM's schedule for a shape, from the host
    alone: tile width, whole tiles, split tiles and K pieces per split tile."""
    Na = (_I64 * len(Ns))(*[int(n) for n in Ns])
    bn, pieces = _I32(), _I32()
    whole, split = _I64(), _I64()
    _check(lib.convrot_gemm_tc_plan(M, K, len(Ns), Na, bits, sms, workspace_bytes, ctypes.byref(bn),
                                    ctypes.byref(whole), ctypes.byref(split), ctypes.byref(pieces)))
    return {"bn": bn.value, "whole_tiles": whole.value, "split_tiles": split.value, "pieces": pieces.value}


def int8_linear_scratch(M: int, K: int, device=None) -> torch.Tensor:
    """A scratch buffer for convrot_int8_linear with M rows of K."""
    nbytes = int(lib.convrot_int8_linear_scratch_bytes(M, K))
    if nbytes < 0:
        raise ValueError(f"no scratch size for M={M}, K={K}")
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device or "cuda")


def convrot_int8_linear(X: torch.Tensor, ws: Sequence[PackedWeight], biases: Optional[Sequence] = None,
                        signs: Optional[torch.Tensor] = None, outs: Optional[List[torch.Tensor]] = None,
                        scratch: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None) -> List[torch.Tensor]:
    """The linears sharing X, from the bf16 activation in one call: rotate +
    per-row quantize into `scratch`, then the GEMM with the fused epilogue."""
    if X.dtype != torch.bfloat16 or X.dim() != 2:
        raise TypeError("X must be a 2-D bf16 tensor")
    if X.stride(1) != 1:
        X = X.contiguous()
    M, K = X.shape
    n = len(ws)
    if n == 0:
        raise ValueError("at least one weight")
    if outs is None:
        outs = [torch.empty((M, w.N), dtype=torch.bfloat16, device=X.device) for w in ws]
    if scratch is None:
        scratch = int8_linear_scratch(M, K, X.device)
    warr = (_Weight * n)(*[w._c() for w in ws])
    barr = (ctypes.c_void_p * n)(*[(_ptr(b) if b is not None else None) for b in (biases or [None] * n)])
    yarr = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    larr = (ctypes.c_int64 * n)(*[o.stride(0) for o in outs])
    wsp = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.convrot_int8_linear(X.data_ptr(), M, K, X.stride(0), ws[0].group, ws[0].transform, _ptr(signs), n,
                                   warr, barr, yarr, larr, scratch.data_ptr(), scratch.numel(), wsp, wsb,
                                   _stream(stream)))
    return outs


def convrot_gemm_s32(a: PackedAct, w: PackedWeight, out: Optional[torch.Tensor] = None, stream=None,
                     workspace: Optional[torch.Tensor] = None, int8_mma: bool = False) -> torch.Tensor:
    """Raw int32 accumulators A = Q_x Q_w^T through the linear's GEMM main loop
    (``int8_mma``: the int8 warp-MMA GEMM, asked for by name)."""
    if out is None:
        out = torch.empty((a.M, w.N), dtype=torch.int32, device=a.q.device)
    ca, cw = a._c(), w._c()
    if int8_mma:
        if workspace is not None:
            raise ValueError("the int8 warp-MMA GEMM takes no workspace")
        _check(lib.convrot_gemm_s32_int8mma(ctypes.byref(ca), ctypes.byref(cw), out.data_ptr(), out.stride(0),
                                            _stream(stream)))
    elif workspace is None:
        _check(lib.convrot_gemm_s32(ctypes.byref(ca), ctypes.byref(cw), out.data_ptr(), out.stride(0),
                                    _stream(stream)))
    else:
        _check(lib.convrot_gemm_s32_ws(ctypes.byref(ca), ctypes.byref(cw), out.data_ptr(), out.stride(0),
                                       workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                       _stream(stream)))
    return out


# ---------------------------------------------------------------- 4-bit ---
# "feat: load ConvRot int4 and per-channel int8 safetensors", "Solution":
# codes in [-7, 7], adjacent pairs in a byte (element 2j in the low nibble),
# one fp32 scale per row; the GEMM reads the e4m3 copies.

@dataclasses.dataclass
class PackedAct4:
    q4: torch.Tensor                # uint8 [M, K/2]
    scale: torch.Tensor             # fp32 [M]
    q_f8: Optional[torch.Tensor]    # uint8 (e4m3 bits) [M, K]
    group: int
    transform: int

    @property
    def M(self) -> int:
        return self.q4.shape[0]

    @property
    def K(self) -> int:
        return 2 * self.q4.shape[1]

    def _c(self) -> _Act4:
        return _Act4(self.q4.data_ptr(), self.scale.data_ptr(), _ptr(self.q_f8), self.M, self.K, self.group,
                     self.transform)


@dataclasses.dataclass
class PackedWeight4:
    q4: torch.Tensor
    scale: torch.Tensor
    q_f8: Optional[torch.Tensor]
    group: int
    transform: int

    @property
    def N(self) -> int:
        return self.q4.shape[0]

    @property
    def K(self) -> int:
        return 2 * self.q4.shape[1]

    def _c(self) -> _Weight4:
        return _Weight4(self.q4.data_ptr(), self.scale.data_ptr(), _ptr(self.q_f8), self.N, self.K, self.group,
                        self.transform)


def convrot_prepare_weights4(W: torch.Tensor, group: int, transform="h4", signs: Optional[torch.Tensor] = None,
                             with_f8: bool = True, stream=None) -> PackedWeight4:
    """Offline 4-bit weight path: W_rot = W R, per-output-row codes in [-7, 7]."""
    if W.dtype not in (torch.float32, torch.bfloat16) or W.dim() != 2:
        raise TypeError("W must be a 2-D fp32 or bf16 tensor")
    W = W.contiguous()
    N, K = W.shape
    t = _transform_id(transform)
    q4 = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
    s = torch.empty((N,), dtype=torch.float32, device=W.device)
    f8 = torch.empty((N, K), dtype=torch.uint8, device=W.device) if with_f8 else None
    _check(lib.convrot_prepare_weights4(W.data_ptr(), _DTYPE_F32 if W.dtype == torch.float32 else _DTYPE_BF16, N, K,
                                        group, t, _ptr(signs), q4.data_ptr(), s.data_ptr(), _ptr(f8),
                                        _stream(stream)))
    return PackedWeight4(q4, s, f8, group, t)


def convrot_quantize_act4(X: torch.Tensor, group: int, transform="h4", signs: Optional[torch.Tensor] = None,
                          with_f8: bool = True, out: Optional[PackedAct4] = None, stream=None) -> PackedAct4:
    """Runtime 4-bit path: X_rot = X R, per-row scale max/7, codes in [-7, 7]."""
    if X.dtype != torch.bfloat16 or X.dim() != 2:
        raise TypeError("X must be a 2-D bf16 tensor")
    if X.stride(1) != 1:
        X = X.contiguous()
    M, K = X.shape
    t = _transform_id(transform)
    if out is None:
        q4 = torch.empty((M, K // 2), dtype=torch.uint8, device=X.device)
        s = torch.empty((M,), dtype=torch.float32, device=X.device)
        f8 = torch.empty((M, K), dtype=torch.uint8, device=X.device) if with_f8 else None
        out = PackedAct4(q4, s, f8, group, t)
    _check(lib.convrot_quantize_act4(X.data_ptr(), M, K, X.stride(0), group, t, _ptr(signs), out.q4.data_ptr(),
                                     out.scale.data_ptr(), _ptr(out.q_f8), _stream(stream)))
    return out


def convrot_linear4_multi(a: PackedAct4, ws: Sequence[PackedWeight4], biases: Optional[Sequence] = None,
                          outs: Optional[List[torch.Tensor]] = None, stream=None,
                          workspace: Optional[torch.Tensor] = None) -> List[torch.Tensor]:
    """4-bit linears sharing one packed activation, in one launch (e4m3 tensor cores)."""
    n = len(ws)
    if outs is None:
        outs = [torch.empty((a.M, w.N), dtype=torch.bfloat16, device=a.q4.device) for w in ws]
    warr = (_Weight4 * n)(*[w._c() for w in ws])
    barr = (ctypes.c_void_p * n)(*[(_ptr(b) if b is not None else None) for b in (biases or [None] * n)])
    yarr = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    larr = (ctypes.c_int64 * n)(*[o.stride(0) for o in outs])
    ca = a._c()
    wsp = None if workspace is None else workspace.data_ptr()
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.convrot_linear4_multi(ctypes.byref(ca), n, warr, barr, yarr, larr, wsp, wsb, _stream(stream)))
    return outs


def convrot_linear4(a: PackedAct4, w: PackedWeight4, bias: Optional[torch.Tensor] = None,
                    out: Optional[torch.Tensor] = None, stream=None,
                    workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    return convrot_linear4_multi(a, [w], [bias], outs=None if out is None else [out], stream=stream,
                                 workspace=workspace)[0]


def convrot_gemm4_s32(a: PackedAct4, w: PackedWeight4, out: Optional[torch.Tensor] = None, stream=None,
                      workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Raw int32 accumulators of the 4-bit GEMM."""
    if out is None:
        out = torch.empty((a.M, w.N), dtype=torch.int32, device=a.q4.device)
    ca, cw = a._c(), w._c()
    wsp = None if workspace is None else workspace.data_ptr()
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.convrot_gemm4_s32(ctypes.byref(ca), ctypes.byref(cw), out.data_ptr(), out.stride(0), wsp, wsb,
                                 _stream(stream)))
    return out


def convrot_get_device_status() -> int:
    """Synchronizes, then reads and clears the library's device error word."""
    return int(lib.convrot_get_device_status())


def convrot_selftest_wait_timeout(spin_limit: int, stream=None) -> None:
    _check(lib.convrot_selftest_wait_timeout(spin_limit, _stream(stream)))


class ConvRotLinear:
    """A linear layer holding prepared ConvRot weights.

    ``forward`` flattens leading dimensions and runs the linear from the
    activation in one library call (rotate + quantize, then the int8 GEMM with
    the fused epilogue), then restores the shape.
    """

    def __init__(self, packed: PackedWeight, bias: Optional[torch.Tensor], signs: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None):
        self.weight = packed
        self.bias = None if bias is None else bias.to(device=packed.q.device, dtype=torch.float32).contiguous()
        self.signs = signs
        self.workspace = workspace  # optional GEMM workspace (see gemm_workspace)

    @classmethod
    def from_float(cls, W: torch.Tensor, bias: Optional[torch.Tensor], group: int, transform="h4",
                   signs: Optional[torch.Tensor] = None, with_f16: bool = True) -> "ConvRotLinear":
        if W.dtype == torch.int8:
            raise TypeError("weight is already quantized; build ConvRotLinear from a PackedWeight instead")
        return cls(convrot_prepare_weights(W, group, transform, signs, with_f16), bias, signs)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        shape = x.shape
        x2 = x.reshape(-1, shape[-1])
        y = convrot_int8_linear(x2, [self.weight], [self.bias], signs=self.signs, workspace=self.workspace)[0]
        return y.reshape(*shape[:-1], y.shape[-1])

    __call__ = forward
