"""Pins of the oracle's dispatch, quantizers, grouped MLP and combine against
invariants, closed forms and library routines (torch CPU float64 matmul)."""
import numpy as np
import pytest
import torch

import workloads


def _bits(t):
    return workloads.bf16_bits(t)


def _setup(oracle, w, seed=0, routing=None, cap=None):
    fmt, rmap, p = workloads.routing_inputs(w, seed, routing)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m) if cap is None else cap
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    return fmt, rmap, p, cap, pre


def test_dispatch_rows_are_bitwise_copies_and_pads_zero(oracle):
    w = workloads.scaled(workloads.WORKLOADS["tiny"], T=300, H=64)
    fmt, rmap, p, cap, pre = _setup(oracle, w)
    x = _bits(workloads.activations(w, 0))
    y, yp = oracle.dispatch(fmt, rmap, p, pre, x, cap, w.E, w.K)
    for t in range(w.T):
        for k in range(w.K):
            r = pre["row_of"][t, k]
            assert np.array_equal(y[r], x[t])
            assert yp[r] == p[t, k]
    for e in range(w.E):
        for r in range(pre["offsets"][e] + pre["counts"][e], pre["offsets"][e + 1]):
            assert not y[r].any() and yp[r] == 0.0 and pre["token_of"][r] == -1


def test_combine_round_trip_is_exact_with_power_of_two_probs(oracle):
    """Identity experts and p = 1/8 for every route: x/8 is exact and a sum of
    eight equal terms is exact, so combine(dispatch(x)) == x bit for bit."""
    w = workloads.scaled(workloads.WORKLOADS["permute"], T=256, H=128)
    fmt, rmap, _, cap, pre = _setup(oracle, w)
    p = np.full((w.T, w.K), 1.0 / 8.0, np.float32)
    x = _bits(workloads.activations(w, 1))
    y, yp = oracle.dispatch(fmt, rmap, p, pre, x, cap, w.E, w.K)
    assert np.array_equal(oracle.combine(y, pre["row_of"], yp), x)


def test_combine_round_trip_renormalised_probs_within_one_ulp(oracle):
    w = workloads.scaled(workloads.WORKLOADS["permute"], T=256, H=128)
    fmt, rmap, p, cap, pre = _setup(oracle, w)
    x = _bits(workloads.activations(w, 1))
    y, yp = oracle.dispatch(fmt, rmap, p, pre, x, cap, w.E, w.K)
    out = oracle.bf16_to_f64(oracle.combine(y, pre["row_of"], yp))
    ref = oracle.bf16_to_f64(x)
    ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(out - ref) <= ulp)


def test_combine_without_probs_k1_is_inverse_permutation(oracle):
    w = workloads.scaled(workloads.WORKLOADS["permute"], T=200, H=32, K=1)
    fmt, rmap, p, cap, pre = _setup(oracle, w)
    x = _bits(workloads.activations(w, 3))
    y, _ = oracle.dispatch(fmt, rmap, None, pre, x, cap, w.E, w.K)
    assert np.array_equal(oracle.combine(y, pre["row_of"], None), x)


def test_combine_skips_dropped_routes(oracle):
    """Under overflow a dropped route contributes nothing."""
    w = workloads.scaled(workloads.WORKLOADS["permute"], T=128, H=16)
    fmt, rmap, p, _, full = _setup(oracle, w)
    cap = full["total_rows"] // 2
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    x = _bits(workloads.activations(w, 4))
    y, yp = oracle.dispatch(fmt, rmap, p, pre, x, cap, w.E, w.K)
    out = oracle.bf16_to_f64(oracle.combine(y, pre["row_of"], yp))
    xd = oracle.bf16_to_f64(x)
    for t in range(w.T):
        kept = pre["row_of"][t] >= 0
        ref = (p[t][kept].astype(np.float64)[:, None] * xd[t][None, :]).sum(0)
        assert np.array_equal(out[t], oracle.bf16_to_f64(oracle.f64_to_bf16(ref)))


def _torch_ffn(x, w13, w2, I):
    """Single-expert SwiGLU FFN with torch float64 matmuls (library routine)."""
    h = x @ w13.T
    up, gate = h[:, :I], h[:, I:]
    return (gate * torch.sigmoid(gate)) * up


def test_bf16_mlp_single_expert_matches_torch_matmul(oracle):
    w = workloads.scaled(workloads.WORKLOADS["tiny"], T=40, H=256, E=1, K=1, I=128)
    x = workloads.activations(w, 0)
    w13, w2 = workloads.expert_weights(w, 0)
    offsets = np.array([0, w.T], np.int32)
    out, act = oracle.grouped_mlp_rows(0, _bits(x), None, w.H, w.I, 1, offsets, _bits(w13), None,
                                       _bits(w2), None, np.arange(w.T), want_act=True)
    a = _torch_ffn(x.double(), w13[0].double(), w2[0].double(), w.I)
    a_bf = torch.from_numpy(oracle.bf16_to_f64(oracle.f64_to_bf16(a.numpy())))
    assert torch.allclose(torch.from_numpy(act), a_bf, rtol=2.0 ** -7, atol=1e-12)
    ref = (torch.from_numpy(act) @ w2[0].double().T).numpy()
    got = oracle.bf16_to_f64(out)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-12)


def test_fp8_quantizers_closed_form(oracle):
    w = workloads.scaled(workloads.WORKLOADS["dsv3"], T=16, H=512)
    x = _bits(workloads.activations(w, 0))
    q, s = oracle.quantize_fp8_rows(x)
    xd = oracle.bf16_to_f64(x).astype(np.float32)
    blocks = xd.reshape(w.T, w.H // 128, 128)
    amax = np.abs(blocks).max(-1)
    assert np.array_equal(s, np.where(amax == 0, np.float32(1), amax / np.float32(448)))
    # the codes are the library E4M3 cast of the fp32 quotient (in range by construction)
    quot = (blocks / s[..., None]).astype(np.float32).reshape(w.T, w.H)
    ref = torch.from_numpy(quot).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    # every block hits +-448 at its amax element
    dec = oracle.e4m3_decode(q).reshape(w.T, w.H // 128, 128)
    assert np.all(np.abs(dec).max(-1) == 448.0)
    # zero block -> scale 1, codes 0
    z = np.zeros((1, 128), np.uint16)
    qz, sz = oracle.quantize_fp8_rows(z)
    assert sz[0, 0] == 1.0 and not qz.any()


def test_fp8_weight_quantizer_blocks(oracle):
    rng = np.random.default_rng(0)
    wt = torch.from_numpy(rng.standard_normal((2, 256, 384)).astype(np.float32) * 0.02).to(torch.bfloat16)
    q, s = oracle.quantize_fp8_weight(_bits(wt))
    assert s.shape == (2, 2, 3)
    wd = wt.float().numpy()
    for g in range(2):
        for nb in range(2):
            for kb in range(3):
                blk = wd[g, nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
                sc = np.float32(np.abs(blk).max()) / np.float32(448)
                assert s[g, nb, kb] == sc
                ref = torch.from_numpy((blk / sc).astype(np.float32)).to(torch.float8_e4m3fn)
                assert np.array_equal(q[g, nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128],
                                      ref.view(torch.uint8).numpy())


def test_fp8_mlp_single_expert_matches_torch_matmul(oracle):
    w = workloads.scaled(workloads.WORKLOADS["dsv3"], T=24, H=256, E=1, K=1, I=128)
    x = _bits(workloads.activations(w, 0))
    w13, w2 = workloads.expert_weights(w, 0)
    xq, xs = oracle.quantize_fp8_rows(x)
    q13, s13 = oracle.quantize_fp8_weight(_bits(w13))
    q2, s2 = oracle.quantize_fp8_weight(_bits(w2))
    out, act = oracle.grouped_mlp_rows(1, xq, xs, w.H, w.I, 1, np.array([0, w.T], np.int32), q13, s13,
                                       q2, s2, np.arange(w.T), want_act=True)
    # dequantize with the library FP8 decode and recompute in float64
    def deq(q, s, bs):
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).double()
        return v * torch.from_numpy(np.kron(s, np.ones(bs))).double()
    xdq = deq(xq, xs, (1, 128))
    w13d = deq(q13[0], s13[0], (128, 128))
    a = _torch_ffn(xdq, w13d, None, w.I).numpy().astype(np.float32)
    # the intermediate is re-encoded per 1x128 block: compare after the same encoding
    aq, as_ = [], []
    for b in range(w.I // 128):
        blk = a[:, b * 128:(b + 1) * 128]
        sc = np.abs(blk).max(1).astype(np.float32) / np.float32(448)
        sc = np.where(sc == 0, np.float32(1), sc)
        code = torch.from_numpy((blk / sc[:, None]).astype(np.float32)).to(torch.float8_e4m3fn)
        aq.append(code.double().numpy() * sc[:, None])
    a_deq = np.concatenate(aq, 1)
    close = np.abs(act - a_deq) <= np.abs(a_deq) * 2.0 ** -3 + 1e-9  # a code may differ by rounding order
    assert close.mean() > 0.999
    ref = act @ deq(q2[0], s2[0], (128, 128)).numpy().T
    got = oracle.bf16_to_f64(out)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-12)


def test_nvfp4_quantizer_closed_form(oracle):
    rng = np.random.default_rng(4)
    x = torch.from_numpy(rng.standard_normal((8, 64)).astype(np.float32)).to(torch.bfloat16)
    g = float(np.float32(np.abs(x.float().numpy()).max() / (6 * 448)))
    packed, sc = oracle.quantize_nvfp4_rows(_bits(x), g)
    xd = x.float().numpy()
    for r in range(8):
        for b in range(4):
            blk = xd[r, b * 16:(b + 1) * 16]
            want = torch.tensor(np.float32(np.abs(blk).max()) / np.float32(6 * np.float32(g)),
                                dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).item()
            assert sc[r, b] == want
            sval = np.float32(oracle.e4m3_decode(np.array([want]))[0])
            denom = np.float32(sval * np.float32(g))
            codes = oracle.e2m1_encode((blk / denom).astype(np.float32))
            got = np.array([(packed[r, b * 8 + i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)])
            assert np.array_equal(got, codes)
    # decoded values stay within half a grid step of the input (relative to the block scale)
    dec = np.zeros_like(xd)
    for r in range(8):
        for i in range(64):
            c = (packed[r, i // 2] >> (4 * (i % 2))) & 0xF
            dec[r, i] = oracle.e2m1_decode(np.array([c]))[0] * oracle.e4m3_decode(np.array([sc[r, i // 16]]))[0] * g
    blockmax = np.repeat(np.abs(xd).reshape(8, 4, 16).max(-1), 16, axis=1)
    assert np.all(np.abs(dec - xd) <= blockmax * 0.25 + 1e-6)


def test_nvfp4_mlp_single_expert_matches_torch_matmul(oracle):
    w = workloads.scaled(workloads.WORKLOADS["decode64"], T=8, H=128, E=1, K=1, I=64)
    x = _bits(workloads.activations(w, 0))
    w13, w2 = workloads.expert_weights(w, 0)
    g1 = float(np.float32(np.abs(oracle.bf16_to_f64(x)).max() / 2688.0))
    g13 = np.array([np.abs(w13.float().numpy()).max() / 2688.0], np.float32)
    g2w = np.array([np.abs(w2.float().numpy()).max() / 2688.0], np.float32)
    xq, xs = oracle.quantize_nvfp4_rows(x, g1)
    q13, s13 = oracle.quantize_nvfp4_rows(_bits(w13), float(g13[0]))
    q2, s2 = oracle.quantize_nvfp4_rows(_bits(w2), float(g2w[0]))
    g2a = 0.01
    out, act = oracle.grouped_mlp_rows(2, xq, xs, w.H, w.I, 1, np.array([0, w.T], np.int32), q13, s13,
                                       q2, s2, np.arange(w.T), w13_global=g13, w2_global=g2w,
                                       fc1_in_global=g1, fc2_in_global=g2a, want_act=True)

    def deq(packed, sc, glob):
        R, half = packed.shape
        codes = np.stack([packed & 0xF, packed >> 4], -1).reshape(R, half * 2)
        return oracle.e2m1_decode(codes) * np.repeat(oracle.e4m3_decode(sc), 16, axis=1) * glob

    xdq = torch.from_numpy(deq(xq, xs, g1))
    w13d = torch.from_numpy(deq(q13[0], s13[0], float(g13[0])))
    a = _torch_ffn(xdq, w13d, None, w.I).numpy()
    # the intermediate is re-encoded to NVFP4 with the FC2 input global scale
    a32 = a.astype(np.float32)
    want = np.zeros_like(a)
    for r in range(w.T):
        for b in range(w.I // 16):
            blk = a32[r, b * 16:(b + 1) * 16]
            sc = torch.tensor(np.float32(np.abs(blk).max()) / np.float32(6 * np.float32(g2a)),
                              dtype=torch.float32).to(torch.float8_e4m3fn).double().item()
            den = np.float32(np.float32(sc) * np.float32(g2a))
            codes = oracle.e2m1_encode((blk / den).astype(np.float32)) if den != 0 else np.zeros(16, np.uint8)
            want[r, b * 16:(b + 1) * 16] = oracle.e2m1_decode(codes) * sc * g2a
    assert np.mean(act == want) > 0.99  # a code may differ only through summation order
    ref = act @ deq(q2[0], s2[0], float(g2w[0])).T
    got = oracle.bf16_to_f64(out)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-12)


def _nvfp4_per_expert(oracle, wt):
    """NVFP4 encoding of bf16 expert weights [E][N][K], each expert with its own
    global scale (amax / (6 * 448), so its largest block scale is E4M3's maximum)."""
    wf = wt.float().numpy()
    g = np.array([np.abs(wf[e]).max() / 2688.0 for e in range(wt.shape[0])], np.float32)
    packs, scs = zip(*[oracle.quantize_nvfp4_rows(_bits(wt[e:e + 1]), float(g[e])) for e in range(wt.shape[0])])
    return np.concatenate(packs), np.concatenate(scs), g


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_grouped_equals_unpermuted_per_token_layer(oracle, fmt):
    """The whole permuted pipeline equals the per-token formulation bit for bit."""
    w = workloads.scaled(workloads.WORKLOADS["tiny"], T=48, H=256, E=6, K=3, I=128)
    rfmt, rmap, p, cap, pre = _setup(oracle, w, seed=7)
    x = _bits(workloads.activations(w, 7))
    w13, w2 = workloads.expert_weights(w, 7)
    g13 = g2w = None
    g1 = g2a = 0.0
    if fmt == 0:
        xa, xsc, a13, s13, a2, s2 = x, None, _bits(w13), None, _bits(w2), None
    elif fmt == 1:
        xa, xsc = oracle.quantize_fp8_rows(x)
        a13, s13 = oracle.quantize_fp8_weight(_bits(w13))
        a2, s2 = oracle.quantize_fp8_weight(_bits(w2))
    else:
        g1 = float(np.float32(np.abs(oracle.bf16_to_f64(x)).max() / 2688.0))
        g2a = 0.004
        xa, xsc = oracle.quantize_nvfp4_rows(x, g1)
        a13, s13, g13 = _nvfp4_per_expert(oracle, w13)
        a2, s2, g2w = _nvfp4_per_expert(oracle, w2)
    globs = dict(w13_global=g13, w2_global=g2w, fc1_in_global=g1, fc2_in_global=g2a)
    y, yp = oracle.dispatch(rfmt, rmap, p, pre, xa, cap, w.E, w.K)
    ys = oracle.dispatch(rfmt, rmap, None, pre, xsc, cap, w.E, w.K)[0] if xsc is not None else None
    rows = np.arange(pre["valid_rows"])
    o, _ = oracle.grouped_mlp_rows(fmt, y, ys, w.H, w.I, w.E, pre["offsets"], a13, s13, a2, s2, rows, **globs)
    out = oracle.combine(o, pre["row_of"], yp)
    ref = oracle.layer_per_token(fmt, rfmt, rmap, p, w.E, w.K, xa, xsc, w.H, w.I, a13, s13, a2, s2,
                                 np.arange(w.T), **globs)
    assert np.array_equal(out, ref)
    assert np.abs(oracle.bf16_to_f64(out)).max() > 0  # a non-trivial layer
    # pad rows (zero input) give exactly zero output
    for e in range(w.E):
        for r in range(pre["offsets"][e] + pre["counts"][e], pre["offsets"][e + 1]):
            assert not o[r].any()


def test_zero_weights_give_zero_output(oracle):
    w = workloads.scaled(workloads.WORKLOADS["tiny"], T=8, H=128, E=2, K=1, I=128)
    x = _bits(workloads.activations(w, 0))
    w13, w2 = workloads.expert_weights(w, 0)
    z13 = np.zeros_like(_bits(w13))
    out, act = oracle.grouped_mlp_rows(0, x, None, w.H, w.I, 2, np.array([0, 4, 8], np.int32), z13, None,
                                       _bits(w2), None, np.arange(8), want_act=True)
    assert not act.any() and not out.any()
    # gate rows zero -> silu(0) = 0 -> zero; up rows zero -> zero
    half = _bits(w13).copy()
    half[:, w.I:, :] = 0
    out, _ = oracle.grouped_mlp_rows(0, x, None, w.H, w.I, 2, np.array([0, 4, 8], np.int32), half, None,
                                     _bits(w2), None, np.arange(8))
    assert not out.any()


def _e4m3_round_trip_blocks(a32, block, glob=None):
    """Re-encode an fp32 intermediate [rows][I] the way the method stores it,
    using library casts: FP8 (block None) per 1x128 block with scale amax/448;
    NVFP4 (block 16) with E4M3 block scales under the global scale ``glob``."""
    import oracle as o

    out = np.zeros(a32.shape, np.float64)
    if glob is None:
        for b in range(a32.shape[1] // 128):
            blk = a32[:, b * 128:(b + 1) * 128]
            sc = np.abs(blk).max(1).astype(np.float32) / np.float32(448)
            sc = np.where(sc == 0, np.float32(1), sc)
            code = torch.from_numpy((blk / sc[:, None]).astype(np.float32)).to(torch.float8_e4m3fn)
            out[:, b * 128:(b + 1) * 128] = code.double().numpy() * sc[:, None]
        return out
    for r in range(a32.shape[0]):
        for b in range(a32.shape[1] // 16):
            blk = a32[r, b * 16:(b + 1) * 16]
            sc = torch.tensor(np.float32(np.abs(blk).max()) / np.float32(6 * np.float32(glob)),
                              dtype=torch.float32).to(torch.float8_e4m3fn).double().item()
            den = np.float32(np.float32(sc) * np.float32(glob))
            codes = o.e2m1_encode((blk / den).astype(np.float32)) if den != 0 else np.zeros(16, np.uint8)
            out[r, b * 16:(b + 1) * 16] = o.e2m1_decode(codes) * sc * glob
    return out


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_grouped_mlp_picks_each_experts_own_weights_scales_and_globals(oracle, fmt):
    """Several experts with different weights (and so different FP8 block scales
    and NVFP4 global scales), one of them empty: every row's output equals a
    torch float64 FFN of that row with the slice of its own expert, dequantized
    by library casts with that expert's scales.  Pins the expert lookup from the
    offsets, the per-expert weight row offset, the FP8 scale-block index and the
    per-expert NVFP4 global, none of which a single-expert case exercises."""
    H, I, E = 256, 128, 4
    offsets = np.array([0, 6, 12, 12, 18], np.int32)  # expert 2 receives no rows
    rng = np.random.default_rng(11)
    y_bf = torch.from_numpy(rng.standard_normal((18, H)).astype(np.float32)).to(torch.bfloat16)
    # expert e's weights have magnitude 0.02 * (1 + e): scales and globals differ by expert
    mag = torch.tensor([0.02 * (1 + e) for e in range(E)]).view(E, 1, 1)
    w13 = (torch.from_numpy(rng.standard_normal((E, 2 * I, H)).astype(np.float32)) * mag).to(torch.bfloat16)
    w2 = (torch.from_numpy(rng.standard_normal((E, H, I)).astype(np.float32)) * mag).to(torch.bfloat16)
    rows = np.arange(18)
    globs = {}
    if fmt == 0:
        ya, ys, a13, s13, a2, s2 = _bits(y_bf), None, _bits(w13), None, _bits(w2), None
        y_d = y_bf.double()
        w13_d = [w13[e].double() for e in range(E)]
        w2_d = [w2[e].double() for e in range(E)]
    elif fmt == 1:
        ya, ys = oracle.quantize_fp8_rows(_bits(y_bf))
        a13, s13 = oracle.quantize_fp8_weight(_bits(w13))
        a2, s2 = oracle.quantize_fp8_weight(_bits(w2))
        assert len({float(s13[e].max()) for e in range(E)}) == E

        def deq(q, s, bs):
            v = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).double()
            return v * torch.from_numpy(np.kron(s, np.ones(bs))).double()

        y_d = deq(ya, ys, (1, 128))
        w13_d = [deq(a13[e], s13[e], (128, 128)) for e in range(E)]
        w2_d = [deq(a2[e], s2[e], (128, 128)) for e in range(E)]
    else:
        g1 = float(np.float32(np.abs(y_bf.float().numpy()).max() / 2688.0))
        ya, ys = oracle.quantize_nvfp4_rows(_bits(y_bf), g1)
        a13, s13, g13 = _nvfp4_per_expert(oracle, w13)
        a2, s2, g2w = _nvfp4_per_expert(oracle, w2)
        assert len(set(g13.tolist())) == E
        globs = dict(w13_global=g13, w2_global=g2w, fc1_in_global=g1, fc2_in_global=0.004)

        def deq(packed, sc, glob):
            R, half = packed.shape
            codes = np.stack([packed & 0xF, packed >> 4], -1).reshape(R, half * 2)
            v = torch.from_numpy(np.ascontiguousarray(codes)).to(torch.uint8)
            # E2M1 magnitudes from the format's definition: 0, .5, 1, 1.5, 2, 3, 4, 6; bit 3 the sign
            mags = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=torch.float64)
            val = mags[(v & 7).long()] * torch.where((v & 8) != 0, -1.0, 1.0).double()
            scl = torch.from_numpy(np.ascontiguousarray(sc)).view(torch.float8_e4m3fn).double()
            return val * scl.repeat_interleave(16, dim=1) * float(glob)

        y_d = deq(ya, ys, g1)
        w13_d = [deq(a13[e], s13[e], g13[e]) for e in range(E)]
        w2_d = [deq(a2[e], s2[e], g2w[e]) for e in range(E)]
    out, act = oracle.grouped_mlp_rows(fmt, ya, ys, H, I, E, offsets, a13, s13, a2, s2, rows, want_act=True,
                                       **globs)
    got = oracle.bf16_to_f64(out)
    for e in range(E):
        r = np.arange(offsets[e], offsets[e + 1])
        if len(r) == 0:
            continue
        a = _torch_ffn(y_d[r], w13_d[e], None, I).numpy()
        if fmt == 0:
            want_act = oracle.bf16_to_f64(oracle.f64_to_bf16(a))
            assert np.all(np.abs(act[r] - want_act) <= np.abs(want_act) * 2.0 ** -7 + 1e-12), e
        else:
            want_act = _e4m3_round_trip_blocks(a.astype(np.float32), None if fmt == 1 else 16,
                                               None if fmt == 1 else globs["fc2_in_global"])
            # a code may differ only where the fp32 product lies at a rounding boundary
            assert np.mean(np.abs(act[r] - want_act) <= np.abs(want_act) * 2.0 ** -3 + 1e-9) > 0.99, e
        ref = act[r] @ w2_d[e].numpy().T
        assert np.all(np.abs(got[r] - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-12), e
        # and the expert's own weights matter: another expert's FC2 gives a different result
        other = act[r] @ w2_d[(e + 1) % E].numpy().T
        assert np.abs(got[r] - other).max() > 10 * np.abs(ref).max() * 2.0 ** -8
