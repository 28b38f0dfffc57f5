"""Pins of the oracle's number formats: E4M3, BF16, the SiLU exponential and the group scale.

Each check compares the oracle with something other than itself: the OCP E4M3 table, torch's
float8_e4m3fn / bfloat16 casts (library routines), double-precision math, or brute force
over all 256 codes."""
import json
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def _all_codes():
    return np.arange(256, dtype=np.uint8)


def test_e4m3_golden_points(orc):
    with open(os.path.join(HERE, "golden", "e4m3_points.json")) as f:
        pts = json.load(f)["points"]
    for p in pts:
        code = int(p["code"], 16)
        v = float(orc.e4m3_decode(np.array([code], np.uint8))[0])
        if p["value"] == "nan":
            assert math.isnan(v), p
        else:
            assert v == p["value"] and math.copysign(1, v) == math.copysign(1, p["value"]), p
            assert int(orc.e4m3_encode(np.array([p["value"]], np.float32))[0]) == code, p


def test_e4m3_decode_all_codes_match_torch(orc):
    codes = _all_codes()
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()
    # sign of zero
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def _finite_values():
    vals = torch.from_numpy(_all_codes()).view(torch.float8_e4m3fn).float().numpy()
    return np.unique(vals[np.isfinite(vals)])


def test_e4m3_encode_matches_torch_cast_in_range(orc):
    vals = _finite_values()
    pos = vals[vals >= 0]
    mids = (pos[1:] + pos[:-1]) / 2  # exact ties in fp32
    near = np.concatenate([np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf))])
    r = np.random.default_rng(0)
    rnd = np.concatenate([
        r.uniform(-448, 448, 200000),
        np.exp(r.uniform(np.log(1e-6), np.log(448), 200000)) * r.choice([-1, 1], 200000),
    ])
    x = np.concatenate([vals, mids, -mids, near, -near, rnd]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ours = orc.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (ours == ref).all(), x[ours != ref][:10]


def test_e4m3_encode_is_nearest_with_ties_to_even_bruteforce(orc):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    r = np.random.default_rng(1)
    x = np.concatenate([r.uniform(-448, 448, 4000), r.uniform(-0.02, 0.02, 4000)]).astype(np.float32)
    q = orc.e4m3_encode(x)
    for xi, qi in zip(x.astype(np.float64), q):
        d = np.abs(dec - xi)
        best = d.min()
        cands = codes[d == best]
        if cands.size == 1:
            assert qi == cands[0] or (best == 0 and (qi & 0x7F) == 0)
        else:  # a tie: the even mantissa wins
            assert qi in cands and (qi & 1) == 0


def test_e4m3_encode_saturation_and_specials(orc):
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e30, np.inf, -449.0, -np.inf, np.nan,
                  -0.0, -1e-30, 1e-30, 0.0009765625, 0.0009765626, 0.0029296875], np.float32)
    q = orc.e4m3_encode(x)
    want = [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F,
            0x80, 0x80, 0x00, 0x00, 0x01, 0x02]
    # 2^-10 is the tie between 0 and 2^-9 -> even (0); just above -> 2^-9; 1.5*2^-9 ties to 2*2^-9
    assert [int(v) for v in q] == want


def test_bf16_round_matches_torch(orc):
    r = np.random.default_rng(2)
    x = np.concatenate([
        r.standard_normal(300000).astype(np.float32) * np.float32(3.0),
        (r.integers(0, 2**31, 100000, dtype=np.uint64).astype(np.uint32)).view(np.float32),
    ])
    # exact ties: low 16 bits = 0x8000
    t = (r.integers(0, 2**15, 20000).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, t, -t])
    x = x[np.isfinite(x)]
    ours = orc.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (ours == ref).all()


def test_bf16_from_double_is_nearest(orc):
    r = np.random.default_rng(3)
    x = np.concatenate([r.standard_normal(20000) * 5, r.standard_normal(2000) * 1e-39,
                        r.standard_normal(2000) * 1e37])
    h = orc.bf16_round_double(x)
    v = orc.bf16_to_f32(h).astype(np.float64)
    up = orc.bf16_to_f32((h.astype(np.int64) + 1).astype(np.uint16)).astype(np.float64)
    dn = orc.bf16_to_f32((h.astype(np.int64) - 1).astype(np.uint16)).astype(np.float64)
    err = np.abs(v - x)
    # a neighbour code that is NaN (0xFFFF below +0) never beats the chosen value
    d_up = np.nan_to_num(np.abs(up - x), nan=np.inf)
    d_dn = np.nan_to_num(np.abs(dn - x), nan=np.inf)
    ok = (err <= d_up) & (err <= d_dn)
    assert ok.all()


def test_exp_within_one_ulp_of_double(orc):
    xs = np.concatenate([np.linspace(-103.9, 88.7, 400001), np.linspace(-1, 1, 100001)]).astype(np.float32)
    y = orc.exp_f32(xs).astype(np.float64)
    ref = np.exp(xs.astype(np.float64))
    normal = (ref > 1.2e-38) & (ref < 3.0e38)
    ulp = np.spacing(ref[normal].astype(np.float32)).astype(np.float64)
    assert (np.abs(y[normal] - ref[normal]) / ulp).max() < 1.0
    sub = ref < 1.2e-38  # subnormal results: one rounding at the subnormal grid
    assert (np.abs(y[sub] - ref[sub]) <= 2.0 ** -149).all()
    sp = orc.exp_f32(np.array([0.0, -0.0, 89.5, 1e30, -104.5, -1e30, np.inf, -np.inf], np.float32))
    assert sp[0] == 1.0 and sp[1] == 1.0
    assert np.isinf(sp[2]) and np.isinf(sp[3]) and np.isinf(sp[6])
    assert sp[4] == 0 and sp[5] == 0 and sp[7] == 0
    assert np.isnan(orc.exp_f32(np.array([np.nan], np.float32))[0])


def test_silu_close_to_double(orc):
    g = np.concatenate([np.linspace(-30, 30, 200001), [-200.0, -100.0, 100.0, 200.0]]).astype(np.float32)
    y = orc.silu_f32(g).astype(np.float64)
    gd = g.astype(np.float64)
    ref = gd / (1.0 + np.exp(-gd))
    big = np.abs(ref) > 1e-30
    rel = np.abs(y[big] - ref[big]) / np.abs(ref[big])
    assert rel.max() < 4 * 2.0 ** -24
    assert orc.silu_f32(np.array([0.0], np.float32))[0] == 0.0
    # large negative: exp overflows, silu -> -0
    assert orc.silu_f32(np.array([-1000.0], np.float32))[0] == 0.0


def test_group_scale_fp32_and_ue8m0_invariants(orc):
    r = np.random.default_rng(4)
    amax = np.exp(r.uniform(np.log(1e-8), np.log(1e6), 100000)).astype(np.float32)
    s32 = orc.group_scale(amax, orc.SCALE_F32)
    assert (s32 == (np.maximum(amax, np.float32(1e-10)) / np.float32(448.0))).all()
    s8 = orc.group_scale(amax, orc.SCALE_UE8M0)
    m, e = np.frexp(s8.astype(np.float64))
    assert (m == 0.5).all(), "UE8M0 scales are powers of two"
    assert (s8 >= s32).all() and (s8 < 2 * s32.astype(np.float64)).all()
    ratio = amax.astype(np.float64) / s8
    assert (ratio <= 448).all() and (ratio > 224).all()
    # all-zero group: the epsilon floor
    z = orc.group_scale(np.zeros(1, np.float32), orc.SCALE_F32)
    assert z[0] == np.float32(1e-10) / np.float32(448.0)
