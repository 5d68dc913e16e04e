"""Pins of the oracle's NVFP4 codecs: hand-worked cases, library routines,
exhaustive enumeration and brute-force nearest-code search."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import E2M1_VALUES, e4m3_table_torch, num, parse_golden


def _same(a, b):
    if math.isnan(b):
        return math.isnan(a)
    return a == b and math.copysign(1, a) == math.copysign(1, b)


def test_golden_codec_cases(golden_dir):
    rows = parse_golden(os.path.join(golden_dir, "nvfp4_codec_cases.txt"))
    assert len(rows) > 60
    for r in rows:
        kind = r[0]
        if kind == "e2m1_value":
            assert _same(oracle.e2m1_value(num(r[1])), num(r[2])), r
        elif kind == "e4m3_value":
            assert _same(oracle.e4m3_value(num(r[1])), num(r[2])), r
        elif kind == "dequant_f16":
            assert oracle.dequant_f16(num(r[1]), num(r[2])) == num(r[3]), r
        elif kind == "e2m1_encode":
            assert oracle.e2m1_encode(num(r[1])) == num(r[2]), r
        elif kind == "e4m3_encode":
            assert oracle.e4m3_encode(num(r[1])) == num(r[2]), r
        elif kind == "f16_from_double":
            assert oracle.f16_from_double(num(r[1])) == num(r[2]), r
        else:
            raise AssertionError(kind)


def test_e2m1_table_closed_form():
    for c in range(16):
        assert _same(oracle.e2m1_value(c), E2M1_VALUES[c])


def test_e4m3_all_codes_match_torch():
    tab = e4m3_table_torch()
    for c in range(256):
        assert _same(oracle.e4m3_value(c), float(tab[c])), hex(c)


def test_f16_conversion_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
        (rng.integers(0, 1 << 16, 2000)).astype(np.uint16).view(np.float16).astype(np.float64),
    ])
    vals = vals[np.isfinite(vals)]
    for v in vals:
        assert oracle.f16_from_double(float(v)) == int(np.float16(v).view(np.uint16)), v
    for b in range(0, 1 << 16, 7):
        d = oracle.f16_to_double(b)
        ref = float(np.uint16(b).view(np.float16))
        assert _same(d, ref) or (math.isnan(d) and math.isnan(ref))


def test_dequant_products_exact_in_fp16():
    """All 16 x 254 finite products are FP16-representable, signs of zero XOR."""
    tab = e4m3_table_torch()
    for s in range(256):
        if math.isnan(tab[s]):
            continue
        for q in range(16):
            v = E2M1_VALUES[q] * tab[s]
            bits = oracle.dequant_f16(q, s)
            back = float(np.uint16(bits).view(np.float16))
            assert back == v, (q, s)
            assert math.copysign(1, back) == math.copysign(1, v) or v != 0
            if v == 0:
                neg = (q >= 8) != (s >= 128)
                assert bits == (0x8000 if neg else 0), (q, s)


def _nearest(table, x):
    """Brute-force round-to-nearest, ties to even code (mantissa LSB 0)."""
    d = np.abs(table - abs(x))
    best = d.min()
    cand = [c for c in np.where(d == best)[0]]
    if len(cand) > 1:
        cand = [c for c in cand if c % 2 == 0]
    return int(cand[0])


def test_e2m1_encode_brute_force():
    mags = E2M1_VALUES[:8]
    rng = np.random.default_rng(2)
    xs = list(rng.uniform(-8, 8, 20000).astype(np.float32))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for m in mids:
        for dx in (-1, 0, 1):
            v = np.float32(m)
            if dx:
                v = np.nextafter(v, np.float32(dx * np.inf), dtype=np.float32)
            xs += [v, -v]
    for x in xs:
        x = np.float32(x)
        ref = 7 if abs(x) > 6 else _nearest(mags, float(x))
        if np.signbit(x):
            ref |= 8
        assert oracle.e2m1_encode(x) == ref, x


def test_e4m3_encode_brute_force_and_torch():
    tab = e4m3_table_torch()[:127]
    rng = np.random.default_rng(3)
    xs = np.concatenate([
        rng.uniform(0, 460, 5000),
        rng.uniform(0, 1, 20000) * 2.0 ** rng.integers(-16, 9, 20000),
    ]).astype(np.float32)
    # exact midpoints of all neighbouring finite codes
    mids = ((tab[1:] + tab[:-1]) / 2).astype(np.float32)
    xs = np.concatenate([xs, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    ref_torch = torch.from_numpy(xs.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, rt in zip(xs, ref_torch):
        got = oracle.e4m3_encode(x)
        if float(x) <= 448.0:
            assert got == _nearest(tab, float(x)), x
            assert got == int(rt), x
        else:
            assert got == 0x7E
    assert oracle.e4m3_encode(np.float32(-1.0)) == 0xB8


# ---- oracle_dequant (canonical rows -> FP16) ---------------------------------------

def _dequant_golden(golden_dir):
    rows = parse_golden(os.path.join(golden_dir, "dequant_worked_rows.txt"))
    q, s, y = {}, {}, {}
    for r in rows:
        vals = [int(t, 16) for t in r[2:]]
        {"q": q, "s": s, "y": y}[r[0]][int(r[1])] = vals
    n = len(q)
    return (np.array([q[i] for i in range(n)], np.uint8), np.array([s[i] for i in range(n)], np.uint8),
            np.array([y[i] for i in range(n)], np.uint16))


def test_dequant_worked_rows(golden_dir):
    """Hand-worked rows fix the nibble order (element 2i in the low nibble),
    the scale index (element c uses scale c // 16) and the zero signs."""
    q, s, y = _dequant_golden(golden_dir)
    assert q.shape == (2, 16) and s.shape == (2, 2) and y.shape == (2, 32)
    got = oracle.dequant(q, s).view(np.uint16)
    np.testing.assert_array_equal(got, y)


def test_dequant_matches_library_decode():
    """Random canonical rows (every code and every finite scale) against the
    test-side decode built from torch's float8_e4m3fn and the E2M1 closed
    form; both are exact in FP16, so the bit patterns (zero signs included)
    must agree."""
    from helpers import dequant_np
    rng = np.random.default_rng(7)
    rows, k = 64, 256
    q = rng.integers(0, 256, (rows, k // 2), dtype=np.uint8)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    s = finite[rng.integers(0, len(finite), (rows, k // 16))]
    s[0, :len(finite) // 16] = finite[:len(finite) // 16]     # a run of distinct scales
    got = oracle.dequant(q, s)
    ref = dequant_np(q, s).astype(np.float16)
    np.testing.assert_array_equal(got.view(np.uint16), ref.view(np.uint16))
    # 3-D input (matrices x rows) keeps its leading shape
    got3 = oracle.dequant(q.reshape(4, 16, k // 2), s.reshape(4, 16, k // 16))
    assert got3.shape == (4, 16, k)
    np.testing.assert_array_equal(got3.reshape(rows, k).view(np.uint16), ref.view(np.uint16))
