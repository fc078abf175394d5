"""Pins of the oracle's format codecs against the published format tables,
torch's own conversions (an independent library) and brute-force nearest search."""
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            c, v = line.split()
            rows.append((int(c, 16), float(v)))
    return rows


def test_e4m3_decode_matches_ocp_table():
    for code, val in _read_table("ocp_e4m3_values.txt"):
        got = O.e4m3_decode(np.array([code], np.uint8))[0]
        if np.isnan(val):
            assert np.isnan(got)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)


def test_e2m1_decode_matches_ocp_table():
    for code, val in _read_table("ocp_e2m1_values.txt"):
        got = O.e2m1_decode(np.array([code]))[0]
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin])


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    fin = np.isfinite(vals)
    assert np.array_equal(O.e4m3_encode(vals[fin].astype(np.float32)), codes[fin])


def _e4m3_brute(v):
    """Nearest finite e4m3 by exhaustive search; ties to the even code; saturating."""
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    pos = [(c, x) for c, x in zip(codes, vals) if np.isfinite(x) and c < 0x80]
    out = []
    for x in np.asarray(v, np.float64):
        a = min(abs(x), 448.0)
        best = min(pos, key=lambda cv: (abs(cv[1] - a), cv[0] & 1))
        c = int(best[0]) | (0x80 if np.signbit(x) else 0)
        out.append(c)
    return np.array(out, np.uint8)


def test_e4m3_encode_midpoints_and_neighbours():
    vals = np.sort(O.e4m3_decode(np.arange(0x7F, dtype=np.uint8)))   # 0 .. 448, positive finite
    mids = (vals[:-1] + vals[1:]) / 2                                 # exact in float32 (<= 5 significant bits)
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)
    probes = np.concatenate([m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9))])
    probes = np.concatenate([probes, -probes])
    assert np.array_equal(O.e4m3_encode(probes), _e4m3_brute(probes))


def test_e4m3_encode_matches_torch_random():
    r = np.random.default_rng(1)
    v = (r.standard_normal(200000) * np.exp2(r.uniform(-12, 9, 200000))).astype(np.float32)
    v = v[np.abs(v) < 464]           # torch's cast is not saturating above 464
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(v), ref)


def test_e4m3_saturates():
    v = np.array([448.0, 464.0, 470.0, 1e6, 3e38, -500.0, -1e30], np.float32)
    assert O.e4m3_encode(v).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e4m3_signed_zero_and_tiny():
    v = np.array([0.0, -0.0, 2.0 ** -11, -(2.0 ** -11), 2.0 ** -10 * 1.0000001], np.float32)
    assert O.e4m3_encode(v).tolist() == [0x00, 0x80, 0x00, 0x80, 0x01]


def test_e2m1_tie_table():
    v = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.25, -0.1, -5.0], np.float32)
    # 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4, >=7 saturates to 6
    assert O.e2m1_decode(O.e2m1_encode(v)).tolist() == [0, 1, 1, 2, 2, 4, 4, 6, 6, -0.0, -0.0, -4]
    assert O.e2m1_encode(np.array([-0.1], np.float32))[0] == 0x8


def test_e2m1_matches_brute_force():
    grid = O.e2m1_decode(np.arange(8))
    r = np.random.default_rng(2)
    v = np.concatenate([r.uniform(-8, 8, 20000), np.arange(-7, 7.01, 0.25)]).astype(np.float32)
    got = O.e2m1_encode(v)
    for x, c in zip(v.astype(np.float64), got):
        a = min(abs(x), 6.0)
        best = min(range(8), key=lambda i: (abs(grid[i] - a), i & 1))
        assert c == (best | (8 if np.signbit(x) else 0)), (x, c, best)


def test_bf16_encode_matches_torch():
    r = np.random.default_rng(3)
    v = np.concatenate([
        r.standard_normal(100000) * np.exp2(r.uniform(-140, 125, 100000)),
        [0.0, -0.0, 1.0, -1.0, 3.3895313892515355e38, 1e-45, -1e-40],
    ]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_encode(v), ref)
    assert np.array_equal(O.bf16_decode(ref), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_encoders_reject_nonfinite():
    with pytest.raises(ValueError):
        O.e4m3_encode(np.array([np.nan], np.float32))
    with pytest.raises(ValueError):
        O.e2m1_encode(np.array([np.inf], np.float32))
