"""Pins of the oracle's number formats against sources outside the oracle:
torch's own e4m3 and bf16 casts, the OCP E2M1 code table, brute-force
nearest-value search, and the round-trip property the MX scale rule gives."""
import math
import os

import numpy as np
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    rows = []
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def torch_e4m3(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    for c in codes:
        v = O.e4m3_decode(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(v)
        else:
            assert v == ref[c], (c, v, ref[c])
    assert O.e4m3_decode(0x7E) == 448.0 and O.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne_below_saturation():
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(4000) * s for s in (1e-3, 0.05, 1, 30, 150)]
    # exact midpoints between neighbouring representable values (tie cases)
    reps = np.array(sorted({O.e4m3_decode(c) for c in range(0x7F)}))
    mids = (reps[:-1] + reps[1:]) / 2
    x = np.concatenate(vals + [mids, -mids, reps, -reps]).astype(np.float32)
    x = x[np.abs(x) < 464]
    ref = torch_e4m3(x)
    got = np.array([O.e4m3_encode(v) for v in x], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(x[i], got[i], ref[i]) for i in bad[:5]]


def test_e4m3_encode_saturates_and_keeps_zero_sign():
    # the writer's cast is saturating ("unit-scale saturating cast", ATOM 2962)
    for v in (448.0, 448.5, 463.99, 464.0, 465.0, 480.0, 1e6, 3e38):
        assert O.e4m3_encode(v) == 0x7E
        assert O.e4m3_encode(-v) == 0xFE
    assert O.e4m3_encode(0.0) == 0x00
    assert O.e4m3_encode(-0.0) == 0x80
    assert O.e4m3_encode(-1e-30) == 0x80


def test_e2m1_decode_matches_ocp_table():
    for code, val in _gold("e2m1_codes.txt"):
        v = O.e2m1_decode(int(code))
        assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val))


def test_e2m1_encode_ties_and_saturation_table():
    for x, expect in _gold("e2m1_ties.txt"):
        c = O.e2m1_encode(float(x))
        v = O.e2m1_decode(c)
        assert v == float(expect) and math.copysign(1, v) == math.copysign(1, float(expect)), (x, c)


def test_e2m1_encode_is_nearest_by_brute_force():
    table = {int(c): float(v) for c, v in _gold("e2m1_codes.txt")}
    pos = sorted((v, c) for c, v in table.items() if c < 8)
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.uniform(-7, 7, 5000), np.linspace(-6.5, 6.5, 2601)])
    for x in xs:
        a = abs(x)
        best = min(pos, key=lambda vc: (abs(vc[0] - a), vc[1] & 1))  # nearest, then even mantissa bit
        if a > 6:
            best = (6.0, 7)
        c = O.e2m1_encode(x)
        assert (c & 7) == best[1], (x, c, best)
        assert (c >> 3) == (1 if math.copysign(1, x) < 0 else 0)


def test_bf16_matches_torch():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        # exact ties: low 16 bits 0x8000
                        (rng.integers(0, 2**31, 2000).astype(np.uint32) & 0xFFFF0000 | 0x8000).view(np.float32)])
    x = x[np.isfinite(x)]
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.bf16_encode(v) for v in x], np.uint16)
    assert np.array_equal(got, ref)
    back = torch.from_numpy(ref[:500].view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    for b, r in zip(ref[:500], back):
        assert O.bf16_decode(b) == r


def test_mx_scale_round_trips_e2m1_grid():
    """Groups of e2m1-representable values times 2^k holding both a top
    element (4 or 6 times 2^k) and 0.5 * 2^k round-trip exactly only when the
    shared exponent is exactly k: one too small saturates the top element,
    one too large flushes the 0.5 * 2^k element."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    rng = np.random.default_rng(3)
    for k in (-20, -3, -1, 0, 1, 5, 30):
        for top in (4.0, 6.0):
            g = rng.choice(mags, 32) * rng.choice([-1, 1], 32)
            g[0] = top
            g[1] = -0.5
            x = (g * 2.0 ** k).astype(np.float32)
            sb = O.mx_scale_byte(x)
            assert sb == k + 127, (k, top, sb)
            e = sb - 127
            back = [O.e2m1_decode(O.e2m1_encode(float(v) * 2.0 ** -e)) * 2.0 ** e for v in x]
            assert np.array_equal(np.array(back), x.astype(np.float64))


def test_mx_scale_zero_group_and_error_bound():
    assert O.mx_scale_byte(np.zeros(32, np.float32)) == 0
    rng = np.random.default_rng(4)
    for _ in range(200):
        x = (rng.standard_normal(32) * np.exp(rng.normal(0, 3))).astype(np.float32)
        e = O.mx_scale_byte(x) - 127
        amax = np.abs(x).max()
        # the largest element lands in [4, 8) after scaling, so it is not
        # flushed and saturates by at most 2^e * 2
        assert 4.0 <= amax * 2.0 ** -e < 8.0
        for v in x:
            q = O.e2m1_decode(O.e2m1_encode(float(v) * 2.0 ** -e)) * 2.0 ** e
            assert abs(q - v) <= 2.0 ** e * 2.0 + 1e-300


def test_cast_e4m3_array():
    x = np.array([0.0, 1.0, -2.5, 500.0, -1000.0, 0.001], np.float32)
    xb = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.cast_e4m3(xb)
    xf = torch.tensor(xb.view(np.int16)).view(torch.bfloat16).float().numpy()
    ref = torch_e4m3(np.clip(xf, -448, 448))
    assert np.array_equal(got, ref)
