"""Host-side checks of the C-ABI library: it loads, exports every entry point
declared in include/convrot.h, and rejects bad arguments on the host before
touching the GPU. Needs no GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "convrot.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(convrot_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def cr():
    import int8_convrot_w8a8_gb300 as cr
    return cr


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["convrot_prepare_weights", "convrot_quantize_act", "convrot_linear",
                     "convrot_linear_multi", "convrot_gemm_s32", "convrot_get_device_status"]:
        assert required in names


def test_library_exports_every_declared_symbol(cr):
    raw = ctypes.CDLL(cr.lib_path)
    for name in declared_functions():
        assert hasattr(raw, name), name
    assert set(declared_functions()) == set(cr.EXPORTED)


def test_version_and_status_strings(cr):
    assert cr.lib.convrot_version() == 102
    for code in range(6):
        assert cr.lib.convrot_status_str(code)
    assert cr.lib.convrot_status_str(99) == b"unknown status"


def _qa(cr, M=4, K=256, ldx=256, group=256, transform=0, X=0x1000, Qx=0x2000, sx=0x3000, signs=None):
    return cr.lib.convrot_quantize_act(X, M, K, ldx, group, transform, signs, Qx, sx, None, None)


def test_host_validation_rejects_bad_groups(cr):
    assert _qa(cr, group=8) == 2                    # not a power of four
    assert _qa(cr, K=2688, ldx=2688, group=256) == 2  # does not divide K
    assert _qa(cr, group=8192, K=8192, ldx=8192) == 2  # too large
    assert _qa(cr, transform=1, group=96, K=1152, ldx=1152) == 2  # RHT block not a power of two
    assert b"power of two" in cr.lib.convrot_last_error()
    assert _qa(cr, group=8) == 2
    assert b"power of four" in cr.lib.convrot_last_error()


def test_host_validation_rejects_bad_arguments(cr):
    assert _qa(cr, K=100, ldx=100, group=4) == 3     # K % 16
    assert _qa(cr, X=0x1001) == 3                    # misaligned X
    assert _qa(cr, ldx=100) == 1                     # ldx < K
    assert _qa(cr, X=None) == 1                      # null input
    assert _qa(cr, M=-1) == 1
    assert _qa(cr, transform=7) == 1
    assert _qa(cr, transform=1, group=128, K=1152, ldx=1152, signs=None) == 1  # RHT without signs
    assert _qa(cr, K=40000, ldx=40000, transform=2) == 1  # K above the maximum


def test_empty_batch_is_a_no_op(cr):
    assert _qa(cr, M=0, X=None, Qx=None, sx=None) == 0


def test_linear_validation(cr):
    act = cr._Act(0x1000, 0x2000, None, 4, 256, 256, 0)
    w_ok = cr._Weight(0x4000, 0x5000, None, 16, 256, 256, 0)
    w_k = cr._Weight(0x4000, 0x5000, None, 16, 512, 256, 0)
    w_g = cr._Weight(0x4000, 0x5000, None, 16, 256, 64, 0)
    f = cr.lib.convrot_linear
    assert f(ctypes.byref(act), ctypes.byref(w_k), None, 0x8000, 16, None) == 1   # K mismatch
    assert f(ctypes.byref(act), ctypes.byref(w_g), None, 0x8000, 16, None) == 1   # group mismatch
    assert f(ctypes.byref(act), ctypes.byref(w_ok), None, 0x8000, 8, None) == 1   # ldy < N
    assert f(ctypes.byref(act), ctypes.byref(w_ok), None, 0x8004, 16, None) == 3  # misaligned Y
    assert f(None, ctypes.byref(w_ok), None, 0x8000, 16, None) == 1
    n_bad = cr.lib.convrot_linear_multi(ctypes.byref(act), 9, None, None, None, None, None)
    assert n_bad == 1


def test_large_m_without_fp16_copies_is_refused(cr):
    """Above 64 rows the tensor-core GEMM reads the fp16 operand copies; a
    call without them is refused on the host, never routed to the ~11x
    slower int8 warp-MMA kernel unless that kernel is asked for by name."""
    act = cr._Act(0x1000, 0x2000, None, 300, 256, 256, 0)
    act16 = cr._Act(0x1000, 0x2000, 0x3000, 300, 256, 256, 0)
    w = cr._Weight(0x4000, 0x5000, None, 16, 256, 256, 0)
    f = cr.lib.convrot_linear
    assert f(ctypes.byref(act), ctypes.byref(w), None, 0x8000, 16, None) == 1
    assert b"fp16 operand copies" in cr.lib.convrot_last_error()
    assert f(ctypes.byref(act16), ctypes.byref(w), None, 0x8000, 16, None) == 1  # weight copy missing
    assert cr.lib.convrot_gemm_s32(ctypes.byref(act), ctypes.byref(w), 0x8000, 16, None) == 1
    # the one-call linear refuses before its first launch
    wa = (cr._Weight * 1)(w)
    bias = (ctypes.c_void_p * 1)(None)
    ys = (ctypes.c_void_p * 1)(0x6000)
    ld = (ctypes.c_int64 * 1)(16)
    need = cr.lib.convrot_int8_linear_scratch_bytes(300, 256)
    assert cr.lib.convrot_int8_linear(0x1000, 300, 256, 256, 256, 0, None, 1, wa, bias, ys, ld, 0x10000, need,
                                      None, 0, None) == 1
    assert b"fp16 operand copies" in cr.lib.convrot_last_error()


def test_selftest_argument_check(cr):
    assert cr.lib.convrot_selftest_wait_timeout(0, None) == 1


def test_workspace_constant_matches_header(cr):
    text = open(HEADER).read()
    m = re.search(r"#define CONVROT_GEMM_WORKSPACE_BYTES \(([0-9 +*]+)\)", text)
    assert m, "CONVROT_GEMM_WORKSPACE_BYTES not found"
    assert eval(m.group(1), {"__builtins__": {}}) == cr.GEMM_WORKSPACE_BYTES


def test_workspace_validation(cr):
    act = cr._Act(0x1000, 0x2000, None, 4, 256, 256, 0)
    w = (cr._Weight * 1)(cr._Weight(0x4000, 0x5000, None, 16, 256, 256, 0))
    bias = (ctypes.c_void_p * 1)(None)
    ys = (ctypes.c_void_p * 1)(0x6000)
    ld = (ctypes.c_int64 * 1)(16)
    f = cr.lib.convrot_linear_multi_ws
    assert f(ctypes.byref(act), 1, w, bias, ys, ld, 0x7010, cr.GEMM_WORKSPACE_BYTES, None) == 3  # misaligned
    assert b"256-byte" in cr.lib.convrot_last_error()
    assert f(ctypes.byref(act), 1, w, bias, ys, ld, 0x7000, -1, None) == 1  # negative size
    assert f(ctypes.byref(act), 0, w, bias, ys, ld, None, 0, None) == 1     # n out of range


def test_int8_linear_scratch_size(cr):
    f = cr.lib.convrot_int8_linear_scratch_bytes
    up = lambda v: (v + 255) // 256 * 256
    assert f(4, 256) == up(4 * 256) + up(16)                      # weight-stream path: no fp16 copy
    assert f(128, 256) == up(128 * 256) + up(512) + 2 * 128 * 256  # 2-SM tensor-core path
    assert f(128, 1040) == up(128 * 1040) + up(512)              # K not a multiple of 64: int8 MMA path
    assert f(0, 256) == 0
    assert f(-1, 256) == -1 and f(4, 0) == -1 and f(4, 40000) == -1


def test_int8_linear_validation(cr):
    w = (cr._Weight * 1)(cr._Weight(0x4000, 0x5000, None, 16, 256, 256, 0))
    w64 = (cr._Weight * 1)(cr._Weight(0x4000, 0x5000, None, 16, 256, 64, 0))
    bias = (ctypes.c_void_p * 1)(None)
    ys = (ctypes.c_void_p * 1)(0x6000)
    ld = (ctypes.c_int64 * 1)(16)
    need = cr.lib.convrot_int8_linear_scratch_bytes(4, 256)
    f = cr.lib.convrot_int8_linear

    def call(M=4, group=256, wts=w, scratch=0x10000, nbytes=need, X=0x1000, n=1):
        return f(X, M, 256, 256, group, 0, None, n, wts, bias, ys, ld, scratch, nbytes, None, 0, None)

    assert call(scratch=0x10010) == 3                     # scratch not 256-byte aligned
    assert b"256-byte" in cr.lib.convrot_last_error()
    assert call(nbytes=need - 1) == 1                     # scratch too small
    assert call(scratch=None) == 1
    assert call(wts=w64) == 1                             # weight rotated with another group
    assert call(group=8) == 2                             # not a power of four
    assert call(X=0x1008) == 3                            # misaligned X
    assert call(n=0) == 1
    assert call(M=0, X=None, scratch=None, nbytes=0) == 0  # empty batch: no-op


def test_gemm_plan_documented_schedules(cr):
    """The tensor-core GEMM's schedules on the DiT and qkv shapes: 384
    256-wide tiles are 5 rounds of 76 pairs plus 4 tiles, which are split
    along K into 19 pieces; without a workspace 224-wide tiles (6 rounds)
    cost less; the 4-bit path's tiles are half as long, so the split's fixed
    cost loses to 224-wide tiles there."""
    plan = lambda *a, **k: tuple(cr.gemm_tc_plan(*a, **k).values())
    assert plan(4096, 6144, [6144]) == (256, 380, 4, 19)
    assert plan(4096, 6144, [6144], workspace_bytes=0) == (224, 448, 0, 1)
    assert plan(4096, 6144, [6144], bits=4) == (224, 448, 0, 1)
    assert plan(32700, 3072, [3072] * 3) == (256, 4608, 0, 1)
    assert plan(32700, 3072, [3072] * 3) == plan(32700, 3072, [9216])


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("sms", [152, 148, 132, 8, 2])
def test_gemm_plan_invariants(cr, bits, sms):
    """Over shapes, SM counts and workspace sizes: every tile is run once,
    a split takes only a last round that leaves at least half of the
    clusters idle, its pieces fit the clusters and keep two k blocks each,
    and its partial sums fit the workspace."""
    bke = 64 if bits == 8 else 128
    for M in (65, 129, 300, 4096, 32700):
        for K in (128, 1024, 6144):
            for Ns in ([256], [6144], [3072] * 3, [136, 520]):
                for ws in (0, 4096 + 256 * 1024, cr.GEMM_WORKSPACE_BYTES):
                    p = cr.gemm_tc_plan(M, K, Ns, bits=bits, sms=sms, workspace_bytes=ws)
                    bn = p["bn"]
                    assert bn in (256, 224, 192)
                    cl = 2 if M > 128 else 1
                    clusters = max(1, sms // cl)
                    tiles = -(-(-(-M // 128)) // cl) * sum(-(-n // bn) for n in Ns)
                    assert p["whole_tiles"] + p["split_tiles"] == tiles
                    if p["split_tiles"] == 0:
                        assert p["pieces"] == 1
                        continue
                    assert p["whole_tiles"] % clusters == 0
                    assert p["split_tiles"] == tiles % clusters
                    assert 2 <= p["pieces"] <= (K // bke) // 2
                    assert p["split_tiles"] * p["pieces"] <= clusters
                    assert 4096 + p["split_tiles"] * cl * 128 * bn * 4 <= ws


def test_gemm_plan_validation(cr):
    with pytest.raises(cr.ConvRotError):
        cr.gemm_tc_plan(4096, 6144, [6144], bits=6)
    with pytest.raises(cr.ConvRotError):
        cr.gemm_tc_plan(64, 6144, [6144])              # 8-bit tensor-core path needs M > 64
    with pytest.raises(cr.ConvRotError):
        cr.gemm_tc_plan(4096, 6144 + 64, [6144], bits=4)  # 4-bit needs K a multiple of 128
    with pytest.raises(cr.ConvRotError):
        cr.gemm_tc_plan(4096, 6144, [])
    with pytest.raises(cr.ConvRotError):
        cr.gemm_tc_plan(4096, 6144, [256] * 9)
    with pytest.raises(cr.ConvRotError):
        cr.gemm_tc_plan(4096, 6144, [0])
    with pytest.raises(cr.ConvRotError):
        cr.gemm_tc_plan(4096, 6144, [6144], sms=0)
    with pytest.raises(cr.ConvRotError):
        cr.gemm_tc_plan(4096, 6144, [6144], workspace_bytes=-1)
    with pytest.raises(cr.ConvRotError):
        cr.gemm_tc_plan(1 << 40, 6144, [6144] * 8)     # more tiles than one launch takes
    assert cr.gemm_tc_plan(1, 128, [256], bits=4)["bn"] in (256, 224, 192)
