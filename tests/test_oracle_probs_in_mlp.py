"""Pins of the oracle's probs-in-MLP variant: the grouped MLP multiplies each
FC2 row by its route's probability before rounding, and the combine then sums
the rows without weights.  Checked against torch float64 matmuls, exact
power-of-two scaling, the zero probability and the weighted combine."""
import numpy as np
import pytest
import torch

import workloads


def _bits(t):
    return workloads.bf16_bits(t)


def _single_expert(T=40, H=256, I=128, seed=0):
    w = workloads.scaled(workloads.WORKLOADS["tiny"], T=T, H=H, E=1, K=1, I=I)
    x = workloads.activations(w, seed)
    w13, w2 = workloads.expert_weights(w, seed)
    return w, x, w13, w2, np.array([0, w.T], np.int32)


def test_bf16_fc2_rows_scaled_by_probability_match_torch_matmul(oracle):
    w, x, w13, w2, off = _single_expert()
    p = np.random.default_rng(1).uniform(0.02, 1.0, w.T).astype(np.float32)
    out, act = oracle.grouped_mlp_rows(0, _bits(x), None, w.H, w.I, 1, off, _bits(w13), None, _bits(w2), None,
                                       np.arange(w.T), want_act=True, row_probs=p)
    ref = p.astype(np.float64)[:, None] * (torch.from_numpy(act) @ w2[0].double().T).numpy()
    got = oracle.bf16_to_f64(out)
    # one rounding to bf16 (8 significant bits) of the scaled float64 sum
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-12)
    # the probability is applied before the single rounding, not to the rounded row
    plain, _ = oracle.grouped_mlp_rows(0, _bits(x), None, w.H, w.I, 1, off, _bits(w13), None, _bits(w2), None,
                                       np.arange(w.T))
    twice = oracle.f64_to_bf16(p.astype(np.float64)[:, None] * oracle.bf16_to_f64(plain))
    assert np.mean(twice != out) > 0.01


def _format_inputs(oracle, fmt, x, w13, w2):
    xb = _bits(x)
    if fmt == 0:
        return xb, None, _bits(w13), None, _bits(w2), None, {}
    if fmt == 1:
        xq, xs = oracle.quantize_fp8_rows(xb)
        a13, s13 = oracle.quantize_fp8_weight(_bits(w13))
        a2, s2 = oracle.quantize_fp8_weight(_bits(w2))
        return xq, xs, a13, s13, a2, s2, {}
    g1 = float(np.float32(np.abs(oracle.bf16_to_f64(xb)).max() / 2688.0))
    xq, xs = oracle.quantize_nvfp4_rows(xb, g1)
    g13 = np.float32(np.abs(w13.float().numpy()).max() / 2688.0)
    g2 = np.float32(np.abs(w2.float().numpy()).max() / 2688.0)
    a13, s13 = oracle.quantize_nvfp4_rows(_bits(w13[0:1]), float(g13))
    a2, s2 = oracle.quantize_nvfp4_rows(_bits(w2[0:1]), float(g2))
    return xq, xs, a13, s13, a2, s2, dict(w13_global=np.array([g13], np.float32),
                                          w2_global=np.array([g2], np.float32), fc1_in_global=g1,
                                          fc2_in_global=0.004)


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_power_of_two_probabilities_scale_rows_exactly(oracle, fmt):
    """p = 2^k commutes with rounding: the row is exactly 2^k times the plain row;
    p = 1 changes nothing and p = 0 gives a zero row."""
    w, x, w13, w2, off = _single_expert(T=24)
    xa, xs, a13, s13, a2, s2, globs = _format_inputs(oracle, fmt, x, w13, w2)
    rows = np.arange(w.T)
    plain, _ = oracle.grouped_mlp_rows(fmt, xa, xs, w.H, w.I, 1, off, a13, s13, a2, s2, rows, **globs)
    k = np.array([-3, -1, 0, 1, 2, -6] * 4, np.int64)
    p = np.ldexp(1.0, k).astype(np.float32)
    p[5] = 0.0
    out, _ = oracle.grouped_mlp_rows(fmt, xa, xs, w.H, w.I, 1, off, a13, s13, a2, s2, rows, row_probs=p, **globs)
    assert np.abs(oracle.bf16_to_f64(plain)).max() > 0
    assert np.array_equal(oracle.bf16_to_f64(out), p.astype(np.float64)[:, None] * oracle.bf16_to_f64(plain))
    assert np.array_equal(out[k == 0], plain[k == 0])
    assert not oracle.bf16_to_f64(out[5]).any()


@pytest.mark.parametrize("elem", [0, 1])
def test_mx_fc2_power_of_two_probability_shifts_the_shared_exponent(oracle, elem):
    """MX FC2 rows: p = 2^k leaves every element code unchanged and adds k to
    every block's E8M0 exponent byte."""
    w, x, w13, w2, off = _single_expert(T=16)
    rows = np.arange(w.T)
    args = (0, _bits(x), None, w.H, w.I, 1, off, _bits(w13), None, _bits(w2), None, rows, elem)
    c0, s0 = oracle.grouped_mlp_rows_mx(*args)
    k = np.array([-2, 3, 1, -5] * 4, np.int64)
    c1, s1 = oracle.grouped_mlp_rows_mx(*args, row_probs=np.ldexp(1.0, k).astype(np.float32))
    assert np.array_equal(c1, c0)
    assert np.array_equal(s1.astype(np.int64), s0.astype(np.int64) + k[:, None])


def test_probs_in_mlp_layer_matches_weighted_combine_within_rounding(oracle):
    """Scaling the FC2 rows and summing unweighted equals the weighted combine
    of unscaled rows up to where each side rounds: one bf16 step of the token's
    output and of every row it sums."""
    w = workloads.scaled(workloads.WORKLOADS["tiny"], T=64, H=256, E=6, K=3, I=128)
    rfmt, rmap, p = workloads.routing_inputs(w, 5)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    pre = oracle.preprocess(rfmt, rmap, w.T, w.E, w.K, w.m, cap)
    x = _bits(workloads.activations(w, 5))
    w13, w2 = workloads.expert_weights(w, 5)
    y, yp = oracle.dispatch(rfmt, rmap, p, pre, x, cap, w.E, w.K)
    rows = np.arange(pre["valid_rows"])
    o, _ = oracle.grouped_mlp_rows(0, y, None, w.H, w.I, w.E, pre["offsets"], _bits(w13), None, _bits(w2), None,
                                   rows)
    op, _ = oracle.grouped_mlp_rows(0, y, None, w.H, w.I, w.E, pre["offsets"], _bits(w13), None, _bits(w2), None,
                                    rows, row_probs=yp[rows])
    weighted = oracle.bf16_to_f64(oracle.combine(o, pre["row_of"], yp))
    inside = oracle.bf16_to_f64(oracle.combine(op, pre["row_of"], None))
    ro = pre["row_of"]
    keep = ro >= 0
    r = np.where(keep, ro, 0)

    def ulp(v):
        a = np.abs(v)
        return np.ldexp(1.0, (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7).astype(np.int64))

    rows_o = oracle.bf16_to_f64(o)[r] * keep[..., None]
    rows_op = oracle.bf16_to_f64(op)[r] * keep[..., None]
    wts = yp[r].astype(np.float64) * keep
    bound = (ulp(weighted) + np.einsum("tk,tkh->th", np.abs(wts), ulp(rows_o) * (rows_o != 0))
             + np.einsum("tkh->th", ulp(rows_op) * (rows_op != 0)))
    assert np.abs(weighted).max() > 0
    assert np.all(np.abs(inside - weighted) <= bound)
    # a dropped or unrouted probability is never applied twice: K=1 rows come back unchanged
    assert np.array_equal(oracle.combine(op, pre["row_of"][:, :1], None)[keep[:, 0]],
                          op[pre["row_of"][:, 0][keep[:, 0]]])
