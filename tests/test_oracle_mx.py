"""Pins of the oracle's MX combine formats (E4M3 or E2M1 elements with one E8M0
power-of-two scale per 32 elements): the E8M0 decode against its closed form,
the shared exponent against frexp, E4M3 element codes against torch's
float8_e4m3fn cast of the exactly scaled values, exact round trips of blocks
built from representable values, saturation, all-zero blocks, the MX combine
against the bf16 combine of the same decoded values, and the FC2 output in MX
against a float64 FFN."""
import numpy as np
import pytest
import torch

import workloads


def test_e8m0_decode_closed_form(oracle):
    codes = np.arange(255, dtype=np.uint8)
    assert np.array_equal(oracle.e8m0_decode(codes), np.ldexp(1.0, codes.astype(np.int64) - 127))
    assert np.isnan(oracle.e8m0_decode(np.array([255], np.uint8))[0])


def _blocks(rng, R, H, spread=6):
    """fp32 rows whose 32-blocks span several binades (and some zero blocks)."""
    x = rng.standard_normal((R, H)) * np.exp2(rng.integers(-spread, spread, (R, H // 32)).repeat(32, axis=1))
    x[0, :32] = 0.0
    return x.astype(np.float32)


def test_mx_e4m3_scale_and_codes(oracle):
    rng = np.random.default_rng(0)
    x = _blocks(rng, 64, 256)
    codes, scales = oracle.quantize_mx_rows(x, oracle.MX_E4M3)
    blocks = x.reshape(64, 8, 32).astype(np.float64)
    amax = np.abs(blocks).max(-1)
    _, e = np.frexp(amax)
    X = np.where(amax > 0, np.clip(e - 1 - 8, -127, 127), 0)
    assert np.array_equal(scales.astype(np.int64) - 127, X)
    q = (blocks / np.ldexp(1.0, X)[..., None]).astype(np.float32).reshape(64, 256)
    ref = torch.from_numpy(np.clip(q, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    # the largest element of every non-zero block lands in the top binade [256, 448]
    dec = oracle.mx_decode_rows(codes, scales, oracle.MX_E4M3).reshape(64, 8, 32)
    top = np.abs(dec).max(-1) / np.ldexp(1.0, X)
    assert np.all((top[amax > 0] >= 256) & (top[amax > 0] <= 448))
    assert scales[0, 0] == 127 and not codes[0, :32].any()  # all-zero block: scale 1, codes 0


@pytest.mark.parametrize("elem", [0, 1])
def test_mx_exact_round_trip_of_representable_blocks(oracle, elem):
    """Blocks of element-grid values times 2^s whose largest magnitude has the
    format's top exponent decode back bit for bit (the shared exponent is s)."""
    rng = np.random.default_rng(1)
    grid = (oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)) if elem == 0
            else oracle.e2m1_decode(np.arange(8, dtype=np.uint8)))
    top = grid[(grid >= (256 if elem == 0 else 4))]
    R, H = 16, 128
    vals = rng.choice(grid, (R, H)) * rng.choice([-1.0, 1.0], (R, H))
    vals.reshape(R, H // 32, 32)[:, :, 0] = rng.choice(top, (R, H // 32))
    s = rng.integers(-20, 20, (R, H // 32))
    x = (vals * np.ldexp(1.0, s).repeat(32, axis=1)).astype(np.float32)
    codes, scales = oracle.quantize_mx_rows(x, elem)
    assert np.array_equal(scales.astype(np.int64) - 127, s)
    assert np.array_equal(oracle.mx_decode_rows(codes, scales, elem), x.astype(np.float64))


def test_mx_saturates_at_the_largest_element(oracle):
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 500.0    # 500 / 2^0 lies above 448: saturates (X = floor(log2 500) - 8 = 0)
    x[0, 1] = -470.0
    x[0, 2] = 1.0
    codes, scales = oracle.quantize_mx_rows(x, oracle.MX_E4M3)
    dec = oracle.mx_decode_rows(codes, scales, oracle.MX_E4M3)[0]
    assert scales[0, 0] == 127 and dec[0] == 448.0 and dec[1] == -448.0 and dec[2] == 1.0
    x2 = np.zeros((1, 32), np.float32)
    x2[0, 0] = 7.5     # E2M1: X = floor(log2 7.5) - 2 = 0; 7.5 saturates to 6
    c2, s2 = oracle.quantize_mx_rows(x2, oracle.MX_E2M1)
    assert s2[0, 0] == 127 and oracle.mx_decode_rows(c2, s2, oracle.MX_E2M1)[0, 0] == 6.0


@pytest.mark.parametrize("elem", [0, 1])
def test_combine_mx_equals_bf16_combine_of_decoded_rows(oracle, elem):
    """MX values have at most 4 significant bits, so they are exact in bf16: the
    MX combine must equal the bf16 combine of the decoded rows bit for bit."""
    w = workloads.scaled(workloads.WORKLOADS["permute"], T=120, H=256, E=6, K=3)
    fmt, rmap, p = workloads.routing_inputs(w, 2)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    _, yp = oracle.dispatch(fmt, rmap, p, pre, np.zeros((w.T, 1), np.uint8), cap, w.E, w.K)
    rows = _blocks(np.random.default_rng(3), cap, w.H, spread=4)
    codes, scales = oracle.quantize_mx_rows(rows, elem)
    dec = oracle.mx_decode_rows(codes, scales, elem)
    as_bf16 = oracle.f64_to_bf16(dec)
    assert np.array_equal(oracle.bf16_to_f64(as_bf16), dec)
    assert np.array_equal(oracle.combine_mx(codes, scales, elem, pre["row_of"], yp),
                          oracle.combine(as_bf16, pre["row_of"], yp))


@pytest.mark.parametrize("elem", [0, 1])
def test_fc2_in_mx_matches_float64_ffn(oracle, elem):
    """Single expert: the MX FC2 rows equal the MX encoding (shared exponent
    from frexp, E4M3 codes from torch's cast) of torch float64 FC2 sums rounded
    to fp32, except where the two summation orders straddle a rounding
    boundary."""
    w = workloads.scaled(workloads.WORKLOADS["tiny"], T=24, H=256, E=1, K=1, I=128)
    x = workloads.bf16_bits(workloads.activations(w, 0))
    w13, w2 = workloads.expert_weights(w, 0)
    off = np.array([0, w.T], np.int32)
    _, act = oracle.grouped_mlp_rows(0, x, None, w.H, w.I, 1, off, workloads.bf16_bits(w13), None,
                                     workloads.bf16_bits(w2), None, np.arange(w.T), want_act=True)
    codes, scales = oracle.grouped_mlp_rows_mx(0, x, None, w.H, w.I, 1, off, workloads.bf16_bits(w13), None,
                                               workloads.bf16_bits(w2), None, np.arange(w.T), elem)
    fc2 = (torch.from_numpy(act) @ w2[0].double().T).numpy().astype(np.float32)
    blocks = fc2.reshape(w.T, w.H // 32, 32).astype(np.float64)
    _, e = np.frexp(np.abs(blocks).max(-1))
    X = e - 1 - (8 if elem == 0 else 2)
    assert np.mean(scales.astype(np.int64) - 127 == X) > 0.99
    dec = oracle.mx_decode_rows(codes, scales, elem)
    # the top binade's element step is 2^(X+5) for E4M3 (3 fraction bits over [256, 512)) and 2^(X+1)
    # for E2M1; rounding moves an element by at most half a step, saturation (above 448 / 6) by two
    step = np.ldexp(1.0, X + (5 if elem == 0 else 1)).repeat(32, axis=1)
    assert np.all(np.abs(dec - fc2) <= 2 * step)
    if elem == 0:
        ref = torch.from_numpy(np.clip((blocks / np.ldexp(1.0, X)[..., None]).astype(np.float32), -448, 448)
                               .reshape(w.T, w.H)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.mean(codes == ref) > 0.995
