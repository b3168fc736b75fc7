"""The data layout of the tensor-core rotate+quantize kernel, replayed on the
CPU (no GPU): the TMA stage's 128B swizzle, every lane's ldmatrix row
addresses, the m16n8k16 fragment layouts, the permuted 16-point matrix, the
digits above the chunk on XOR-permuted register slots (and, for G = 1024,
the 4-lane transpose before the superblock digit), and the staging offsets
of the codes, including K not a multiple of 256 (G <= 64), where a
superblock may end in the next row of the tile and the kernel takes each
line's scale from the row it lies in. The replayed
rotation must equal the oracle's (unnormalized by sqrt(G)); every output
position must be written exactly once; the eight rows of every ldmatrix
phase and the 32 lanes of every int8 staging store must fall in distinct
banks."""
import numpy as np
import pytest

import oracle as O


def h16_entry(G, p, k):
    """Entry (p, k) of the unnormalized 16-point stage (2*H4 Kronecker 2*H4,
    or I4 Kronecker 2*H4 for G = 4): -1 where the two digits satisfy b = a ^ 3."""
    lo = -1.0 if ((p & 3) ^ (k & 3)) == 3 else 1.0
    if G == 4:
        return lo if (p >> 2) == (k >> 2) else 0.0
    return (-1.0 if ((p >> 2) ^ (k >> 2)) == 3 else 1.0) * lo


def h4_stage(x0, x1, x2, x3):
    u01, w0, u23, w2 = x0 + x1, x0 - x1, x2 + x3, x2 - x3
    return u01 + w2, u01 - w2, u23 + w0, u23 - w0


def replay(X, G):
    """The kernel's arithmetic on one tile of R = X.shape[0] rows, in fp64."""
    R, K = X.shape
    lines = K // 64
    assert R * lines % 4 == 0  # a tile is a whole number of superblocks
    nsb = R * lines // 4
    warps = (nsb + 7) // 8
    # the stage as TMA writes it: logical 16-byte chunk c of line L at physical chunk c ^ (L & 7)
    stage = np.zeros((R * lines, 8, 8))
    for r in range(R):
        for ln in range(lines):
            L = r * lines + ln
            for c in range(8):
                stage[L, c ^ (L & 7)] = X[r, ln * 64 + c * 8: ln * 64 + c * 8 + 8]
    out = np.full((R, K), np.nan)
    written = np.zeros((R, K), dtype=int)
    bad_phases = 0
    bad_stores = 0
    for w in range(warps):
        a_off = np.zeros((32, 8), dtype=np.int64)
        for lane in range(32):
            ga, h, hf = lane & 7, (lane >> 3) & 1, lane >> 4
            sba = w * 8 + ga
            if sba >= nsb:
                sba = ga if ga < nsb else 0
            for u in range(8):
                j = (2 * u + h) ^ ga
                L = 4 * sba + (j >> 2)
                c = (2 * (j & 3) + hf) ^ (L & 7)
                a_off[lane, u] = L * 128 + c * 16
        full_warp = w * 8 + 7 < nsb
        for u in range(8):
            for m in range(4):
                banks = {(a_off[8 * m + i, u] // 16) % 8 for i in range(8)}
                bad_phases += full_warp and len(banks) != 8
        v = np.zeros((32, 16, 2, 2))
        for u in range(8):
            mats = [np.array([stage[a_off[8 * m + i, u] // 128, (a_off[8 * m + i, u] % 128) // 16]
                              for i in range(8)]) for m in range(4)]
            A = np.zeros((16, 16))
            A[0:8, 0:8], A[8:16, 0:8], A[0:8, 8:16], A[8:16, 8:16] = mats
            for nb in range(2):
                B = np.zeros((16, 8))
                for lane in range(32):
                    g, t = lane >> 2, lane & 3
                    p = 4 * (g >> 1) + 2 * nb + (g & 1)
                    for e in range(2):
                        B[2 * t + e, g] = h16_entry(G, p, 2 * t + e)
                        B[2 * t + 8 + e, g] = h16_entry(G, p, 2 * t + 8 + e)
                D = A @ B
                for lane in range(32):
                    g, t = lane >> 2, lane & 3
                    v[lane, 2 * u, nb] = D[g, 2 * t: 2 * t + 2]
                    v[lane, 2 * u + 1, nb] = D[g + 8, 2 * t: 2 * t + 2]
        for lane in range(32):
            for q in range(2):
                if G >= 64:
                    for a in range(0, 16, 4):
                        y = h4_stage(*[v[lane, a + i, q] for i in range(4)])
                        for i in range(4):
                            v[lane, a + i, q] = y[i]
                if G >= 256:
                    for b in range(4):
                        y = h4_stage(*[v[lane, b + 4 * i, q] for i in range(4)])
                        for i in range(4):
                            v[lane, b + 4 * i, q] = y[i]
        if G == 1024:
            # the 4-lane transpose (slot s with s & 3 = c from lane ^ 4c), then
            # the radix-4 stage on slots 4h .. 4h + 3
            v = np.array([[v[lane ^ (4 * (s & 3)), s] for s in range(16)] for lane in range(32)])
            for lane in range(32):
                for q in range(2):
                    for h in range(4):
                        y = h4_stage(*[v[lane, 4 * h + i, q] for i in range(4)])
                        for i in range(4):
                            v[lane, 4 * h + i, q] = y[i]

        def placed(lane, s):
            """(int8 staging offset, superblock, chunk) of slot s of the lane."""
            g, t = lane >> 2, lane & 3
            if G == 1024:
                g2, j = g >> 2, g & 3
                rel = 256 * (w * 8 + 4 * g2 + j) + 16 * (4 * g2 + j) + 4 * t
                addr = rel ^ (256 * (s & 3) + 16 * (s & 12))
                return addr, w * 8 + 4 * g2 + (j ^ (s & 3)), ((s & 12) ^ (4 * g2)) | j
            return ((256 * (w * 8 + g) + 4 * t) | (16 * g)) ^ (16 * s), w * 8 + g, s ^ g

        # int8 staging stores: lane (g, t) writes the 4 codes of slot s
        for s in range(16):
            banks = {(placed(lane, s)[0] // 4) % 32 for lane in range(32)}
            bad_stores += full_warp and len(banks) != 32
        for lane in range(32):
            g, t = lane >> 2, lane & 3
            sb0 = w * 8 + g
            if sb0 >= nsb:
                continue
            # the kernel's rows: the superblock's first and last line, and
            # bit h where slots 4h .. 4h + 3 (line h ^ (g >> 2)) lie in the second
            row1, row2 = 4 * sb0 // lines, (4 * sb0 + 3) // lines
            in2 = sum(1 << h for h in range(4) if (4 * sb0 + (h ^ (g >> 2))) // lines != row1)
            for s in range(16):
                addr, sb, chunk = placed(lane, s)
                assert sb < nsb
                assert addr == 256 * sb + 16 * chunk + 4 * t  # the dense output offset
                row, e = divmod(addr, K)
                if G <= 64:
                    assert row == (row2 if (in2 >> (s >> 2)) & 1 else row1)
                out[row, e:e + 2] = v[lane, s, 0]
                out[row, e + 2:e + 4] = v[lane, s, 1]
                written[row, e:e + 4] += 1
    return out, written, bad_phases, bad_stores


@pytest.mark.parametrize("K,G,R", [(3072, 256, 4), (6144, 256, 2), (4096, 1024, 1), (4096, 16, 3),
                                   (4096, 64, 1), (1024, 4, 12), (5376, 256, 3), (5376, 64, 3), (1024, 1024, 4),
                                   (3072, 1024, 1), (5120, 1024, 1),
                                   # K not a multiple of 256: superblocks across rows (G <= 64)
                                   (2688, 64, 6), (2688, 16, 2), (2688, 4, 4), (320, 64, 4), (1088, 64, 4),
                                   (2688, 64, 8)])
def test_replayed_layout_is_the_rotation(K, G, R):
    rng = np.random.default_rng(K + G + R)
    X = rng.standard_normal((R, K)).round(3)  # exactly representable sums in fp64
    got, written, bad_phases, bad_stores = replay(X, G)
    assert np.all(written == 1)
    np.testing.assert_allclose(got, O.rotate_rows(X, G, "h4") * np.sqrt(G), rtol=0, atol=1e-9)
    assert bad_phases == 0 and bad_stores == 0
