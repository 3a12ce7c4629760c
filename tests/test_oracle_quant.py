"""Pins for the oracle's number formats and quantisers (CPU only).

- bf16 rounding against torch's float32 -> bfloat16 cast (round to nearest even);
- e4m3 / e5m2 decode tables against torch's float8 types, and encoding against
  torch's float8 casts inside the finite range (torch maps overflow to NaN/inf,
  the oracle saturates, so saturation is pinned separately);
- e2m1 against the format's value table and an independent rounding route
  (frexp + rint to one mantissa bit);
- int8 (CANN aclnnMoeDistributeDispatchV2, quantMode 2) against hand-worked rows,
  exact rational arithmetic with IEEE rounding at each step, and the bound that
  every nonzero row reaches |q| = 127;
- MX (quantMode 4) against hand-worked blocks, the scale exponent from
  math.frexp, and the range of the largest code in each block.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMT = {"e4m3": oracle.Q_E4M3, "e5m2": oracle.Q_E5M2, "e2m1": oracle.Q_E2M1}


def read_cases(name):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            else:
                cur[key] = vals
    return cases


def bf16_bits(values):
    t = torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32_bits(x):
    return int(np.float32(x).view(np.uint32))


# ---------------------------------------------------------------- bf16

def test_bf16_matches_torch_cast():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e30).astype(np.float32),
        (rng.standard_normal(5000) * 1e-38).astype(np.float32),   # subnormals
        np.array([0.0, -0.0, 3.3895314e38, 3.4028235e38, -3.4028235e38, 1e-45], np.float32),
    ])
    # exact ties: bf16 value plus half a bf16 ulp
    b = rng.integers(0, 0x7f7f, 5000, dtype=np.uint32)
    ties = ((b << 16) | 0x8000).view(np.float32)
    v = np.concatenate([v, ties, -ties])
    got = oracle.bf16_from_f32(v)
    want = bf16_bits(v)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- fp8 tables and casts

@pytest.mark.parametrize("name,tdt,maxcode", [("e4m3", torch.float8_e4m3fn, 0x7e),
                                              ("e5m2", torch.float8_e5m2, 0x7b)])
def test_fp8_decode_table_matches_torch(name, tdt, maxcode):
    q = FMT[name]
    codes = np.arange(0, maxcode + 1)
    codes = np.concatenate([codes, codes | 0x80])
    want = torch.tensor(codes.astype(np.uint8)).view(tdt).float().numpy().astype(np.float64)
    got = oracle.mini_decode(q, codes)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("name,tdt,maxcode", [("e4m3", torch.float8_e4m3fn, 0x7e),
                                              ("e5m2", torch.float8_e5m2, 0x7b)])
def test_fp8_encode_matches_torch_in_range(name, tdt, maxcode):
    q = FMT[name]
    table = torch.arange(0, maxcode + 1, dtype=torch.uint8).view(tdt).float().numpy()
    mids = ((table[:-1].astype(np.float64) + table[1:]) / 2).astype(np.float32)  # exact ties
    rng = np.random.default_rng(11)
    top = float(table[-1])
    rnd = (rng.random(20000) * top).astype(np.float32)
    small = (rng.random(5000) * float(table[8])).astype(np.float32)
    v = np.concatenate([table, mids, rnd, small])
    v = v[np.abs(v) <= top]
    v = np.concatenate([v, -v])
    want = torch.tensor(v).to(tdt).view(torch.uint8).numpy().astype(np.int32)
    got = oracle.mini_encode(q, v)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("name,maxval", [("e4m3", 448.0), ("e5m2", 57344.0), ("e2m1", 6.0)])
def test_saturation(name, maxval):
    q = FMT[name]
    sbit = 0x8 if name == "e2m1" else 0x80
    big = np.array([maxval * 1.01, maxval * 4, 1e30, 3.0e38], np.float32)
    pos = oracle.mini_encode(q, big)
    neg = oracle.mini_encode(q, -big)
    dec = oracle.mini_decode(q, pos)
    assert np.all(dec == maxval)
    assert np.all(neg == pos | sbit)


def test_e2m1_table_from_definition():
    with open(os.path.join(GOLDEN, "formats.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    table = [float(v) for v in next(r for r in rows if r[0] == "e2m1")[1:]]
    assert np.array_equal(oracle.mini_decode(oracle.Q_E2M1, np.arange(8)), table)
    assert np.array_equal(oracle.mini_decode(oracle.Q_E2M1, np.arange(8) | 8), -np.array(table))
    for r in rows:
        if r[0] == "max":
            q, mx = FMT[r[1]], float(r[2])
            assert max(oracle.mini_decode(q, np.arange(0, {"e4m3": 0x7f, "e5m2": 0x7c, "e2m1": 8}[r[1]]))) == mx
            assert math.frexp(mx)[1] - 1 == int(r[3])


def e2m1_by_rounding(v):
    """Round to one mantissa bit with frexp/rint (normal range >= 1), or to the
    subnormal grid 0.5 below 1, then saturate at 6: a route independent of the
    oracle's table search."""
    a = abs(float(v))
    if a >= 1.0:
        m, e = math.frexp(a)          # a = m * 2^e, m in [0.5, 1)
        r = np.rint(m * 4.0) / 4.0 * 2.0 ** e   # 2 significant bits
    else:
        r = np.rint(a * 2.0) / 2.0
    return math.copysign(min(r, 6.0), v)


def test_e2m1_encode_matches_rounding_route():
    rng = np.random.default_rng(5)
    table = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    v = np.concatenate([table, mids, (rng.random(20000) * 7.5).astype(np.float32)])
    v = np.concatenate([v, -v])
    got = oracle.mini_decode(oracle.Q_E2M1, oracle.mini_encode(oracle.Q_E2M1, v))
    want = np.array([e2m1_by_rounding(x) for x in v])
    assert np.array_equal(got, want)
    # -0 for negative values that round to zero
    codes = oracle.mini_encode(oracle.Q_E2M1, np.array([-0.25, -0.1, -0.0], np.float32))
    assert codes.tolist() == [8, 8, 8]


# ---------------------------------------------------------------- int8 (quantMode 2)

def _row(vals, H):
    x = np.zeros(H, np.float32)
    x[:len(vals)] = vals
    return bf16_bits(x)


@pytest.mark.parametrize("case", read_cases("int8_rows.txt"), ids=lambda c: c["name"])
def test_int8_golden(case):
    H = int(case["H"][0])
    x = _row([float(v) for v in case["x"]], H)
    q, inv = oracle.quant_int8_row(x)
    assert q.tolist() == [int(v) for v in case["q"]]
    assert f32_bits(inv) == int(case["inv"][0], 16)


def _rne_f32(q: Fraction) -> Fraction:
    """Exact round-to-nearest-even of a rational to binary32 (normal range)."""
    if q == 0:
        return Fraction(0)
    sgn = -1 if q < 0 else 1
    a = abs(q)
    e = math.frexp(float(a))[1] - 1
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    m = a / ulp
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sgn * fl * ulp


def _rne_int(q: Fraction) -> int:
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def test_int8_exact_arithmetic():
    rng = np.random.default_rng(3)
    for trial in range(30):
        H = 64
        scale = 10.0 ** rng.uniform(-3, 3)
        x = bf16_bits((rng.standard_normal(H) * scale).astype(np.float32))
        xf = [Fraction(float(v)) for v in (x.astype(np.uint32) << 16).view(np.float32)]
        amax = max(abs(v) for v in xf)
        s = _rne_f32(Fraction(127) / amax)
        want = [max(-127, min(127, _rne_int(_rne_f32(v * s)))) for v in xf]
        inv = _rne_f32(1 / s)
        q, ginv = oracle.quant_int8_row(x)
        assert q.tolist() == want
        assert Fraction(float(ginv)) == inv


def test_int8_range_and_error_bound():
    rng = np.random.default_rng(9)
    for trial in range(200):
        H = int(rng.choice([8, 32, 1024]))
        x = bf16_bits((rng.standard_normal(H) * 10.0 ** rng.uniform(-20, 20)).astype(np.float32))
        q, inv = oracle.quant_int8_row(x)
        xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.max(np.abs(q.astype(int))) == 127
        # |q - x s| <= 1/2 + 127 * 2^-24 (the product rounds once), and inv = (1/s)(1 + d),
        # |d| <= 2^-24, so |x - q inv| <= inv (1/2 + 254 * 2^-24)(1 + 2^-24) < inv/2 (1 + 2^-14)
        err = np.abs(xf - q.astype(np.float64) * float(inv))
        assert np.all(err <= 0.5 * float(inv) * (1 + 2.0 ** -14))


# ---------------------------------------------------------------- MX (quantMode 4)

@pytest.mark.parametrize("case", read_cases("mx_blocks.txt"), ids=lambda c: c["name"])
def test_mx_golden(case):
    q = FMT[case["fmt"][0]]
    x = _row([float(v) for v in case["x"]], 32)
    codes, scales = oracle.quant_mx_row(q, x)
    assert scales.tolist() == [int(case["scale"][0], 16)]
    want = [int(v, 16) for v in case["codes"]]
    if q == oracle.Q_E2M1:
        nib = [(codes[i // 2] >> (4 * (i % 2))) & 0xF for i in range(32)]
        assert nib[:len(want)] == want and all(c == 0 for c in nib[len(want):])
    else:
        assert codes[:len(want)].tolist() == want and np.all(codes[len(want):] == 0)


def test_e2m1_nibble_order():
    # element 0 -> low nibble, element 1 -> high nibble (packing reading)
    x = _row([1.0, 0.625], 32)
    codes, _ = oracle.quant_mx_row(oracle.Q_E2M1, x)
    assert codes[0] == 0x46


@pytest.mark.parametrize("name", ["e4m3", "e5m2", "e2m1"])
def test_mx_scale_exponent_and_block_max(name):
    q = FMT[name]
    emax, maxval = {"e4m3": (8, 448.0), "e5m2": (15, 57344.0), "e2m1": (2, 6.0)}[name]
    rng = np.random.default_rng(21)
    H = 256
    for trial in range(100):
        x = bf16_bits((rng.standard_normal(H) * 10.0 ** rng.uniform(-30, 30)).astype(np.float32))
        codes, scales = oracle.quant_mx_row(q, x)
        xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        for b in range(H // 32):
            amax = np.max(np.abs(xf[b * 32:(b + 1) * 32]))
            se = math.frexp(amax)[1] - 1 - emax if amax >= 2.0 ** -126 else -127
            se = max(se, -127)
            assert scales[b] == se + 127
            if q == oracle.Q_E2M1:
                c = [(codes[(b * 32 + i) // 2] >> (4 * (i % 2))) & 0xF for i in range(32)]
            else:
                c = codes[b * 32:(b + 1) * 32]
            vals = np.abs(oracle.mini_decode(q, c))
            if amax >= 2.0 ** -126:
                assert 2.0 ** emax <= vals.max() <= maxval
            # each code is the nearest representable value (or saturated) to x / 2^se
            scaled = xf[b * 32:(b + 1) * 32] / 2.0 ** se
            dec = oracle.mini_decode(q, c)
            table = np.abs(oracle.mini_decode(q, np.arange(0, {"e4m3": 0x7f, "e5m2": 0x7c, "e2m1": 8}[name])))
            for sv, dv in zip(scaled, dec):
                best = np.min(np.abs(table - min(abs(sv), maxval)))
                assert abs(abs(dv) - min(abs(sv), maxval)) == best
