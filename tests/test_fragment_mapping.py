"""CPU check of the lane-level data flow of the warp-level tensor-core decode
kernel (split_mma_kernel.cuh): the E4M3 path, which builds f16 MMA fragments
straight from staged codes (KV8 branches), and the 16-bit path's ldmatrix
addressing of the query rows and the swizzled K/V stages.

The kernel's address and permutation formulas are restated here and run through a
model of the warp-level instructions, taken from their PTX definitions:
ldmatrix (lane l receives row l/4, 16-bit columns 2(l%4), 2(l%4)+1 of each 8x8
matrix; .trans: rows 2(l%4), 2(l%4)+1 of column l/4), mma.m16n8k16 fragment
layouts, the byte permutation 0x3120 and the E4M3 -> f16 pair conversion (low
code -> low half).  The products must equal Q K^T and P V of the decoded codes,
with Q's A fragments in the permuted k order and O's columns put back in order
by the epilogue mapping.  This pins the index arithmetic, not the hardware."""
import numpy as np
import pytest
import torch


def _dec(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes).astype(np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _stage(codes, d):
    """[32][d] codes -> stage bytes: d/128 regions of [32 rows][128 B], chunk c of row r at c ^ (r & 7)."""
    buf = np.zeros((d // 128) * 4096, dtype=np.uint8)
    for r in range(32):
        for c in range(d // 16):
            off = (c >> 3) * 4096 + r * 128 + (((c & 7) ^ (r & 7)) << 4)
            buf[off:off + 16] = codes[r, 16 * c:16 * c + 16]
    return buf


def _ldmatrix_x4(buf, addrs, trans):
    regs = [[None] * 4 for _ in range(32)]
    for m in range(4):
        rows = [buf[addrs[8 * m + r]:addrs[8 * m + r] + 16] for r in range(8)]
        for lane in range(32):
            t, g = lane % 4, lane // 4
            if trans:
                lo, hi = rows[2 * t][2 * g:2 * g + 2], rows[2 * t + 1][2 * g:2 * g + 2]
            else:
                lo, hi = rows[g][4 * t:4 * t + 2], rows[g][4 * t + 2:4 * t + 4]
            regs[lane][m] = np.concatenate([lo, hi])
    return regs


def _cvt4(w):  # four codes -> (f16 pair of bytes 0, 1), (pair of bytes 2, 3)
    v = _dec(w)
    return (v[0], v[1]), (v[2], v[3])


def _mma(acc, a, b0, b1):
    A, B = np.zeros((16, 16)), np.zeros((16, 8))
    for lane in range(32):
        g, t = lane // 4, lane % 4
        A[g, 2 * t:2 * t + 2], A[g + 8, 2 * t:2 * t + 2] = a[lane][0], a[lane][1]
        A[g, 2 * t + 8:2 * t + 10], A[g + 8, 2 * t + 8:2 * t + 10] = a[lane][2], a[lane][3]
        B[2 * t:2 * t + 2, g], B[2 * t + 8:2 * t + 10, g] = b0[lane], b1[lane]
    C = A @ B
    for lane in range(32):
        g, t = lane // 4, lane % 4
        acc[lane] += np.array([C[g, 2 * t], C[g, 2 * t + 1], C[g + 8, 2 * t], C[g + 8, 2 * t + 1]])


@pytest.mark.parametrize("d", [128, 256])
def test_code_fragments_reproduce_qk_and_pv(d):
    rng = np.random.default_rng(d)
    kc = rng.integers(0, 256, size=(32, d), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(32, d), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x10  # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x22
    q = rng.standard_normal((16, d)).astype(np.float16).astype(np.float64)
    p = rng.random((16, 32))
    kbuf, vbuf = _stage(kc, d), _stage(vc, d)

    # S = Q K^T: one ldmatrix.x4 per 16-dim step, lane l addresses token l
    s_acc = [[np.zeros(4) for _ in range(4)] for _ in range(32)]
    for kk in range(d // 16):
        addrs = [(kk >> 3) * 4096 + lane * 128 + (((kk & 7) << 4) ^ ((lane & 7) << 4)) for lane in range(32)]
        regs = _ldmatrix_x4(kbuf, addrs, trans=False)
        qa = []
        for lane in range(32):  # A fragments in the permuted k order: dims 16 kk + 4 t .. + 3
            g, t = lane // 4, lane % 4
            r0, r1 = q[g, 16 * kk + 4 * t:16 * kk + 4 * t + 4], q[g + 8, 16 * kk + 4 * t:16 * kk + 4 * t + 4]
            qa.append(((r0[0], r0[1]), (r1[0], r1[1]), (r0[2], r0[3]), (r1[2], r1[3])))
        for j in range(4):
            frags = [_cvt4(regs[lane][j]) for lane in range(32)]
            acc = [s_acc[lane][j] for lane in range(32)]
            _mma(acc, qa, [f[0] for f in frags], [f[1] for f in frags])
    s = np.zeros((16, 32))
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for n in range(4):
            s[g, 8 * n + 2 * t:8 * n + 2 * t + 2] = s_acc[lane][n][:2]
            s[g + 8, 8 * n + 2 * t:8 * n + 2 * t + 2] = s_acc[lane][n][2:]
    assert np.allclose(s, q @ _dec(kc).T, rtol=1e-12, atol=1e-9)

    # O = P V: one ldmatrix.x4.trans per (16-token step, two 16-dim chunks)
    o_acc = [[np.zeros(4) for _ in range(d // 8)] for _ in range(32)]
    for k2 in range(2):
        pa = []
        for lane in range(32):
            g, t = lane // 4, lane % 4
            b = 16 * k2
            pa.append(((p[g, b + 2 * t], p[g, b + 2 * t + 1]), (p[g + 8, b + 2 * t], p[g + 8, b + 2 * t + 1]),
                       (p[g, b + 8 + 2 * t], p[g, b + 9 + 2 * t]), (p[g + 8, b + 8 + 2 * t], p[g + 8, b + 9 + 2 * t])))
        for c in range(0, d // 16, 2):
            addrs = [(c >> 3) * 4096 + (16 * k2 + 8 * ((lane >> 3) & 1) + (lane & 7)) * 128 +
                     (((c & 7) << 4) ^ ((((lane >> 4) & 1) ^ (lane & 7)) << 4)) for lane in range(32)]
            regs = _ldmatrix_x4(vbuf, addrs, trans=True)
            ev = [[None] * 4 for _ in range(32)]
            od = [[None] * 4 for _ in range(32)]
            for lane in range(32):
                for m in range(4):
                    w = regs[lane][m]
                    ev[lane][m], od[lane][m] = _cvt4(np.array([w[0], w[2], w[1], w[3]], dtype=np.uint8))
            for tile, src, m0, m1 in ((2 * c, ev, 0, 1), (2 * c + 1, od, 0, 1), (2 * c + 2, ev, 2, 3),
                                      (2 * c + 3, od, 2, 3)):
                acc = [o_acc[lane][tile] for lane in range(32)]
                _mma(acc, pa, [src[lane][m0] for lane in range(32)], [src[lane][m1] for lane in range(32)])
    o = np.zeros((16, d))
    for lane in range(32):  # the epilogue's column order: dims 16c + 4t + (even c0, odd c0, even c1, odd c1)
        g, t = lane // 4, lane % 4
        for c in range(d // 16):
            e, od_ = o_acc[lane][2 * c], o_acc[lane][2 * c + 1]
            o[g, 16 * c + 4 * t:16 * c + 4 * t + 4] = [e[0], od_[0], e[1], od_[1]]
            o[g + 8, 16 * c + 4 * t:16 * c + 4 * t + 4] = [e[2], od_[2], e[3], od_[3]]
    assert np.allclose(o, p @ _dec(vc), rtol=1e-12, atol=1e-9)


def _stage16(vals, d):
    """[32][d] f16 values -> stage bytes: d/64 regions of [32 rows][128 B], 8-element chunk c at c ^ (r & 7)."""
    raw = np.ascontiguousarray(vals.astype(np.float16)).view(np.uint8).reshape(32, 2 * d)
    buf = np.zeros((d // 64) * 4096, dtype=np.uint8)
    for r in range(32):
        for c in range(d // 8):
            off = (c >> 3) * 4096 + r * 128 + (((c & 7) ^ (r & 7)) << 4)
            buf[off:off + 16] = raw[r, 16 * c:16 * c + 16]
    return buf


def _pairs16(w):  # 4 bytes -> the two f16 values (low half first)
    v = np.frombuffer(np.ascontiguousarray(w).tobytes(), dtype=np.float16).astype(np.float64)
    return (v[0], v[1])


@pytest.mark.parametrize("d", [64, 128, 256])
def test_16bit_fragments_reproduce_qk_and_pv(d):
    """The same check for the 16-bit cache path: Q fragments by ldmatrix from the query
    rows, K by ldmatrix and V by ldmatrix.trans from the swizzled stage."""
    rng = np.random.default_rng(d + 1)
    k = rng.standard_normal((32, d)).astype(np.float16).astype(np.float64)
    v = rng.standard_normal((32, d)).astype(np.float16).astype(np.float64)
    q = rng.standard_normal((16, d)).astype(np.float16).astype(np.float64)
    p = rng.random((16, 32)).astype(np.float16).astype(np.float64)
    kbuf, vbuf = _stage16(k, d), _stage16(v, d)
    qbuf = np.ascontiguousarray(q.astype(np.float16)).view(np.uint8).reshape(-1)  # [16][d] rows, unswizzled
    lanes = range(32)
    mi = [lane >> 3 for lane in lanes]
    q_lane = [((mi[lane] & 1) * 8 + (lane & 7)) * (d * 2) + (mi[lane] >> 1) * 16 for lane in lanes]
    kb_row = [[(8 * (2 * j + (mi[lane] >> 1)) + (lane & 7)) * 128 for lane in lanes] for j in range(2)]
    kb_x = [[((2 * j + (mi[lane] & 1)) ^ (lane & 7)) << 4 for lane in lanes] for j in range(4)]
    vb_row = [[(16 * j + 8 * (mi[lane] & 1) + (lane & 7)) * 128 for lane in lanes] for j in range(2)]
    vb_x = [[((2 * j + (mi[lane] >> 1)) ^ (lane & 7)) << 4 for lane in lanes] for j in range(4)]

    s_acc = [[np.zeros(4) for _ in range(4)] for _ in range(32)]
    for kk in range(d // 16):
        qr = _ldmatrix_x4(qbuf, [q_lane[lane] + 2 * kk * 16 for lane in lanes], trans=False)
        qa = [tuple(_pairs16(qr[lane][m]) for m in range(4)) for lane in lanes]
        for pr in range(2):
            kr = _ldmatrix_x4(kbuf, [(kk >> 2) * 4096 + kb_row[pr][lane] + kb_x[kk & 3][lane] for lane in lanes],
                              trans=False)
            for half, (m0, m1) in enumerate(((0, 1), (2, 3))):
                acc = [s_acc[lane][2 * pr + half] for lane in lanes]
                _mma(acc, qa, [_pairs16(kr[lane][m0]) for lane in lanes], [_pairs16(kr[lane][m1]) for lane in lanes])
    s = np.zeros((16, 32))
    for lane in lanes:
        g, t = lane // 4, lane % 4
        for n in range(4):
            s[g, 8 * n + 2 * t:8 * n + 2 * t + 2] = s_acc[lane][n][:2]
            s[g + 8, 8 * n + 2 * t:8 * n + 2 * t + 2] = s_acc[lane][n][2:]
    assert np.allclose(s, q @ k.T, rtol=1e-12, atol=1e-9)

    o_acc = [[np.zeros(4) for _ in range(d // 8)] for _ in range(32)]
    for k2 in range(2):
        pa = []
        for lane in lanes:
            g, t = lane // 4, lane % 4
            b = 16 * k2
            pa.append(((p[g, b + 2 * t], p[g, b + 2 * t + 1]), (p[g + 8, b + 2 * t], p[g + 8, b + 2 * t + 1]),
                       (p[g, b + 8 + 2 * t], p[g, b + 9 + 2 * t]), (p[g + 8, b + 8 + 2 * t], p[g + 8, b + 9 + 2 * t])))
        for jp in range(d // 16):
            vr = _ldmatrix_x4(vbuf, [(jp >> 2) * 4096 + vb_row[k2][lane] + vb_x[jp & 3][lane] for lane in lanes],
                              trans=True)
            for half, (m0, m1) in enumerate(((0, 1), (2, 3))):
                acc = [o_acc[lane][2 * jp + half] for lane in lanes]
                _mma(acc, pa, [_pairs16(vr[lane][m0]) for lane in lanes], [_pairs16(vr[lane][m1]) for lane in lanes])
    o = np.zeros((16, d))
    for lane in lanes:
        g, t = lane // 4, lane % 4
        for n in range(d // 8):
            o[g, 8 * n + 2 * t:8 * n + 2 * t + 2] = o_acc[lane][n][:2]
            o[g + 8, 8 * n + 2 * t:8 * n + 2 * t + 2] = o_acc[lane][n][2:]
    assert np.allclose(o, p @ v, rtol=1e-12, atol=1e-9)
