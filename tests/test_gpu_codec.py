"""GPU quantiser / dequantiser vs the oracle: bit-exact (integer and byte work)."""
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import num, parse_golden
from nvfp4_weight_mixture_gb300 import moe

pytestmark = pytest.mark.gpu


def frag_to_canonical(q, s, n, rows, k, w13=False):
    """Undo the fragment layout (as documented in include/moe_nvfp4.h): block
    b = ((m * rows/256 + G) * k/64 + ks) * 16 + j holds tile rt = 16 G + j."""
    q = q.reshape(n, rows // 256, k // 64, 16, 32, 2, 8)   # [m][G][ks][j][L][half][8 bytes]
    s = s.reshape(n, rows // 256, k // 64, 16, 32, 2)
    L = np.arange(32)
    g, c = L // 4, L % 4
    qc = np.zeros((n, rows, k // 2), np.uint8)
    sc = np.zeros((n, rows, k // 16), np.uint8)
    for rt in range(rows // 16):
        G, j = divmod(rt, 16)
        for ks in range(k // 64):
            for half in range(2):
                r = rt * 16 + g + 8 * half
                for b in range(8):
                    qc[:, r, ks * 32 + 8 * c + b] = q[:, G, ks, j, L, half, b]
                sc[:, r, ks * 4 + c] = s[:, G, ks, j, L, half]
    if w13:
        I = rows // 2
        canon_rows = []
        for rp in range(rows):
            t, r16 = rp // 16, rp % 16
            base = 16 * (t // 2) + r16
            canon_rows.append(I + base if t % 2 else base)
        out_q = np.zeros_like(qc)
        out_s = np.zeros_like(sc)
        out_q[:, canon_rows] = qc
        out_s[:, canon_rows] = sc
        return out_q, out_s
    return qc, sc


def _weights(seed, n, rows, k):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((n, rows, k)) * 0.02).astype(np.float32)
    # edge cases: heavy tails, tiny blocks (subnormal / zero scales), zeros, signed zeros
    w[0, 0, :16] = [2688, 224, -1344, 100, -100, 0, 672, -896] + [0] * 8
    w[0, 1, :16] *= 1e-7
    w[0, 2, 16:32] = 0.0
    w[0, 3, 32:48] = -0.0
    w[-1, 5, :] *= 40.0
    w[-1, 6, 64:80] = rng.standard_normal(16).astype(np.float32) * 1e-5
    return w


@pytest.mark.parametrize("layout", [moe.LAYOUT_CANONICAL, moe.LAYOUT_FRAGMENT,
                                    moe.LAYOUT_FRAGMENT_W13])
@pytest.mark.parametrize("shape", [(3, 256, 256), (2, 256, 2048), (1, 1024, 128)])
def test_quantize_bit_exact(layout, shape):
    n, rows, k = shape
    w = _weights(7 + rows, n, rows, k)
    qo, so, go, st = oracle.quantize(w)
    assert st == 0
    q, s, g = moe.quantize(torch.from_numpy(w).cuda(), layout)
    q, s, g = q.cpu().numpy(), s.cpu().numpy(), g.cpu().numpy()
    np.testing.assert_array_equal(g.view(np.uint32), go.view(np.uint32))
    if layout == moe.LAYOUT_CANONICAL:
        np.testing.assert_array_equal(q.reshape(qo.shape), qo)
        np.testing.assert_array_equal(s.reshape(so.shape), so)
    else:
        qc, sc = frag_to_canonical(q, s, n, rows, k, w13=(layout == moe.LAYOUT_FRAGMENT_W13))
        np.testing.assert_array_equal(qc, qo)
        np.testing.assert_array_equal(sc, so)


def test_quantize_small_canonical_shapes():
    """Canonical layout only needs rows % 16 == 0."""
    w = _weights(3, 2, 48, 128)
    qo, so, go, st = oracle.quantize(w)
    q, s, g = moe.quantize(torch.from_numpy(w).cuda(), moe.LAYOUT_CANONICAL)
    np.testing.assert_array_equal(q.cpu().numpy().reshape(qo.shape), qo)
    np.testing.assert_array_equal(s.cpu().numpy().reshape(so.shape), so)
    np.testing.assert_array_equal(g.cpu().numpy().view(np.uint32), go.view(np.uint32))


def test_quantize_worked_case(golden_dir):
    rows = parse_golden(os.path.join(golden_dir, "quantize_worked_case.txt"))
    x = np.zeros((16, 64), np.float32)   # the 4 x 16 case embedded in a 16 x 64 matrix
    for r in rows:
        if r[0] == "x":
            x[int(r[1]), :16] = [float(v) for v in r[2:]]
    q, s, g = moe.quantize(torch.from_numpy(x).cuda(), moe.LAYOUT_CANONICAL)
    q = q.cpu().numpy().reshape(16, 32)
    s = s.cpu().numpy().reshape(16, 4)
    assert float(g.cpu()[0]) == 1.0
    codes = np.stack([q & 15, q >> 4], -1).reshape(16, 64)
    for r in rows:
        if r[0] == "q":
            assert [int(v, 16) for v in r[2:]] == list(codes[int(r[1]), :16]), r
        if r[0] == "s":
            assert int(r[2], 16) == s[int(r[1]), 0], r


def test_quantize_nonfinite_sets_status():
    w = np.ones((1, 16, 64), np.float32)
    w[0, 2, 3] = np.nan
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.quantize(torch.from_numpy(w).cuda(), moe.LAYOUT_CANONICAL, status=st)
    assert int(st.item()) & moe.ST_NONFINITE


@pytest.mark.parametrize("layout", [moe.LAYOUT_CANONICAL, moe.LAYOUT_FRAGMENT,
                                    moe.LAYOUT_FRAGMENT_W13])
def test_dequantize_bit_exact_all_codes(layout):
    """Every (E2M1, E4M3) pair through the GPU decode vs the oracle's exact FP16."""
    n, rows, k = 1, 256, 256
    rng = np.random.default_rng(11)
    q = np.zeros((rows, k // 2), np.uint8)
    s = np.zeros((rows, k // 16), np.uint8)
    # rows 0..255: scale code = row for every block (0x7F/0xFF NaN codes skipped)
    for r in range(rows):
        s[r, :] = r if r not in (0x7F, 0xFF) else 0x7E
        codes = np.arange(k) % 16
        rng.shuffle(codes)
        q[r] = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    ref = oracle.dequant(q, s).view(np.uint16)
    if layout != moe.LAYOUT_CANONICAL:
        # build the fragment layout from the canonical bytes (the inverse map)
        qf = np.zeros((rows // 256, k // 64, 16, 32, 2, 8), np.uint8)
        sf = np.zeros((rows // 256, k // 64, 16, 32, 2), np.uint8)
        L = np.arange(32)
        g, c = L // 4, L % 4
        if layout == moe.LAYOUT_FRAGMENT_W13:
            I = rows // 2
            packed_src = []
            for rp in range(rows):
                t, r16 = rp // 16, rp % 16
                base = 16 * (t // 2) + r16
                packed_src.append(I + base if t % 2 else base)
            qp, sp = q[packed_src], s[packed_src]
        else:
            qp, sp = q, s
        for rt in range(rows // 16):
            G, j = divmod(rt, 16)
            for ks in range(k // 64):
                for half in range(2):
                    r = rt * 16 + g + 8 * half
                    for b in range(8):
                        qf[G, ks, j, L, half, b] = qp[r, ks * 32 + 8 * c + b]
                    sf[G, ks, j, L, half] = sp[r, ks * 4 + c]
        qd, sd = qf.reshape(-1), sf.reshape(-1)
    else:
        qd, sd = q.reshape(-1), s.reshape(-1)
    out = moe.dequantize(torch.from_numpy(qd).cuda(), torch.from_numpy(sd).cuda(), n, rows, k, layout)
    got = out.cpu().numpy().view(np.uint16).reshape(rows, k)
    np.testing.assert_array_equal(got, ref)
