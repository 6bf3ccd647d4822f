"""Pins of the oracle's number formats (bf16, FP8 E4M3, FP4 E2M1) against
library routines and brute force -- no GPU needed."""
import numpy as np
import pytest
import torch


def minifloat_decode(code: int, ebits: int, mbits: int, bias: int) -> float:
    """A generic sign/exponent/fraction decoder (IEEE-style subnormals, no specials).

    Validated below on formats torch implements, then used to pin E2M1, which
    torch cannot convert on the CPU.
    """
    sign = -1.0 if (code >> (ebits + mbits)) & 1 else 1.0
    ex = (code >> mbits) & ((1 << ebits) - 1)
    man = code & ((1 << mbits) - 1)
    if ex == 0:
        return sign * (man / (1 << mbits)) * 2.0 ** (1 - bias)
    return sign * (1.0 + man / (1 << mbits)) * 2.0 ** (ex - bias)


def test_generic_decoder_matches_torch_formats():
    codes = torch.arange(256, dtype=torch.uint8)
    e4m3 = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    e5m2 = codes.view(torch.float8_e5m2).to(torch.float64).numpy()
    for c in range(256):
        if not np.isnan(e4m3[c]):
            assert minifloat_decode(c, 4, 3, 7) == e4m3[c]
        if np.isfinite(e5m2[c]):
            assert minifloat_decode(c, 5, 2, 15) == e5m2[c]
    bf = torch.arange(0, 1 << 16, 97, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    bfv = bf.to(torch.float64).numpy()
    for c, v in zip(torch.arange(0, 1 << 16, 97).tolist(), bfv):
        if np.isfinite(v):
            assert minifloat_decode(c, 8, 7, 127) == v


def test_e4m3_decode_all_codes(oracle):
    ours = oracle.e4m3_decode(np.arange(256))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.nanmax(ours) == 448.0


def test_e4m3_encode_roundtrip_all_codes(oracle):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_e4m3_encode_matches_torch_cast(oracle):
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(400_000) * 10.0,
        rng.standard_normal(300_000) * 1e-2,
        rng.uniform(-447.9, 447.9, 200_000),
        rng.standard_normal(100_000) * 1e-3,
    ]).astype(np.float32)
    # exact midpoints between neighbouring codes exercise ties-to-even
    fin = np.array([c for c in range(127)], np.uint8)
    mids = ((oracle.e4m3_decode(fin[:-1]) + oracle.e4m3_decode(fin[1:])) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v), ref)


def test_e4m3_saturates(oracle):
    v = np.array([448.0, 449.0, 464.0, 500.0, 1e9, -1e9, -448.5], np.float32)
    assert oracle.e4m3_encode(v).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e2m1_decode_matches_generic_minifloat(oracle):
    ours = oracle.e2m1_decode(np.arange(16))
    ref = np.array([minifloat_decode(c, 2, 1, 1) for c in range(16)])
    assert np.array_equal(ours, ref)
    assert ours.max() == 6.0


def test_e2m1_encode_is_nearest_even(oracle):
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(-7, 7, 20000), np.arange(-6.5, 6.75, 0.25)]).astype(np.float32)
    got = oracle.e2m1_encode(v)
    grid = oracle.e2m1_decode(np.arange(16))
    for x, c in zip(v, got):
        xc = float(np.clip(x, -6.0, 6.0))
        d = np.abs(grid - xc)
        best = np.flatnonzero(d == d.min())
        best = [b for b in best if (b & 8) == (8 if np.signbit(x) else 0)] or list(best)
        if len(best) > 1:  # tie: the even code
            best = [b for b in best if (b & 7) % 2 == 0]
        assert grid[c] == grid[best[0]], (x, c, best)


def test_bf16_rounding_of_float32_matches_torch(oracle):
    rng = np.random.default_rng(2)
    v = np.concatenate([
        rng.standard_normal(300_000) * np.exp(rng.uniform(-30, 30, 300_000)),
        rng.standard_normal(1000) * 1e-39,   # bf16/fp32 subnormal range
    ]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(v.astype(np.float64)), ref)


def test_bf16_rounding_of_double_is_nearest_even(oracle):
    rng = np.random.default_rng(3)
    v = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))
    # values exactly halfway between two bf16 neighbours (only reachable from double)
    base = oracle.bf16_to_f64(rng.integers(0x0080, 0x7F00, 2000).astype(np.uint16))
    half = base * (1 + 2.0 ** -8)
    v = np.concatenate([v, half, -half])
    got = oracle.bf16_to_f64(oracle.f64_to_bf16(v))
    # neighbours by direct bit stepping of the truncation
    trunc = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    for x, g, tb in zip(v, got, trunc):
        cands = [oracle.bf16_to_f64(np.array([c], np.uint16))[0] for c in (tb - 1, tb, tb + 1)]
        dists = [abs(c - x) for c in cands]
        dmin = min(dists)
        assert abs(g - x) == dmin, (x, g, cands)
        if dists.count(dmin) > 1:
            bits = oracle.f64_to_bf16(np.array([x]))[0]
            assert bits % 2 == 0


def test_capacity_golden(oracle):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "capacity.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        rows, factor, align, cap = line.split()
        assert oracle.capacity(int(rows), float(factor), int(align)) == int(cap)


@pytest.mark.parametrize("rows,factor,expect", [(1, 1.0, 4), (4, 1.0, 4), (5, 1.0, 8), (10, 1.5, 16), (0, 2.0, 0)])
def test_capacity_small_cases(oracle, rows, factor, expect):
    assert oracle.capacity(rows, factor, 4) == expect
