"""GPU parity of the probs-in-MLP variant: the grouped MLP multiplies each FC2
row by its route's dispatched probability before rounding (fc2_row_probs of
moe_grouped_mlp_ex) and the combine sums the rows without weights.  Every
kernel family (bf16 on single SMs, bf16 on SM pairs, FP8 with bf16 and MX
outputs, NVFP4) against the oracle's probs-in-MLP rows, plus exact
power-of-two scaling at full size."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import (bits, fill_pattern, gather_rows, largest_expert_rows, layer_rel_err, moe_mod,
                      oracle_rows_chunked, preprocess, rel_err, segment_edge_rows)

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp8": 5e-2, "nvfp4": 5e-2}
FC2_IN_GLOBAL = 0.01  # calibration constant of the NVFP4 intermediate, an input to both sides


@pytest.fixture(scope="module")
def moe():
    return moe_mod()


def _nvfp4_globals(x, w13, w2):
    gx = np.float32(x.float().abs().max().item() / 2688.0)
    g13 = (w13.float().abs().amax(dim=(1, 2)) / 2688.0).cpu().numpy().astype(np.float32)
    g2 = (w2.float().abs().amax(dim=(1, 2)) / 2688.0).cpu().numpy().astype(np.float32)
    return gx, g13, g2


def prepare(moe, w, dtype, seed):
    """Preprocess and dispatch seeded inputs, weights in the library's format."""
    dev = "cuda"
    fmt, rmap, probs = workloads.routing_inputs(w, seed)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    x = workloads.activations(w, seed)
    w13, w2 = workloads.expert_weights(w, seed, device=dev)
    shape, layout, routing_t, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    P = dict(w=w, dtype=dtype, fmt=fmt, rmap=rmap, probs=probs, cap=cap, x=x, w13=w13, w2=w2, shape=shape,
             layout=layout, handle=handle, globals=None, ys=None, s13=None, s2=None)
    yp = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
    if dtype == "bf16":
        P["mlp_dtype"] = moe.DTYPE_BF16
        P["q13"], P["q2"] = w13, w2
        y = torch.empty(max(cap, 1), w.H, dtype=torch.bfloat16, device=dev)
        moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16, x.to(dev), None, routing_t, y, yp)
    elif dtype == "fp8":
        P["mlp_dtype"] = moe.DTYPE_FP8_E4M3_B128
        P["q13"] = torch.empty(w13.shape, dtype=torch.uint8, device=dev)
        P["s13"] = torch.empty(w.E, 2 * w.I // 128, w.H // 128, dtype=torch.float32, device=dev)
        P["q2"] = torch.empty(w2.shape, dtype=torch.uint8, device=dev)
        P["s2"] = torch.empty(w.E, w.H // 128, w.I // 128, dtype=torch.float32, device=dev)
        moe.moe_quantize_fp8_blocks(w13, P["q13"], P["s13"])
        moe.moe_quantize_fp8_blocks(w2, P["q2"], P["s2"])
        y = torch.empty(max(cap, 1), w.H, dtype=torch.uint8, device=dev)
        P["ys"] = torch.empty(max(cap, 1), w.H // 128, dtype=torch.float32, device=dev)
        moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16_TO_FP8, x.to(dev), None, routing_t, y, yp,
                                 P["ys"])
    else:
        P["mlp_dtype"] = moe.DTYPE_NVFP4
        gx, g13, g2 = _nvfp4_globals(x, w13, w2)
        P.update(gx=gx, g13=g13, g2=g2)
        P["q13"] = torch.empty(w.E, 2 * w.I, w.H // 2, dtype=torch.uint8, device=dev)
        P["s13"] = torch.empty(w.E, 2 * w.I, w.H // 16, dtype=torch.uint8, device=dev)
        P["q2"] = torch.empty(w.E, w.H, w.I // 2, dtype=torch.uint8, device=dev)
        P["s2"] = torch.empty(w.E, w.H, w.I // 16, dtype=torch.uint8, device=dev)
        g13_d, g2_d = torch.from_numpy(g13).to(dev), torch.from_numpy(g2).to(dev)
        for e in range(w.E):
            moe.moe_quantize_nvfp4_rows(w13[e], g13_d[e:e + 1], P["q13"][e], P["s13"][e])
            moe.moe_quantize_nvfp4_rows(w2[e], g2_d[e:e + 1], P["q2"][e], P["s2"][e])
        gx_d = torch.tensor([gx], device=dev)
        P["globals"] = moe.Nvfp4Globals(gx_d, torch.tensor([FC2_IN_GLOBAL], dtype=torch.float32, device=dev), g13_d,
                                        g2_d)
        y = torch.empty(max(cap, 1), w.H // 2, dtype=torch.uint8, device=dev)
        P["ys"] = torch.empty(max(cap, 1), w.H // 16, dtype=torch.uint8, device=dev)
        moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16_TO_NVFP4, x.to(dev), gx_d, routing_t, y, yp,
                                 P["ys"])
    P["y"], P["yp"] = y, yp
    P["ws"] = torch.empty(moe.moe_grouped_mlp_workspace_size(shape, layout, P["mlp_dtype"]), dtype=torch.uint8,
                          device=dev)
    return P


def run_mlp(moe, P, row_probs, out_format=None, combine=True):
    """moe_grouped_mlp_ex with the given FC2 row probabilities; then the
    combine without weights.  Returns (rows, MX scales or None, combined)."""
    w = P["w"]
    out_format = moe.COMBINE_BF16 if out_format is None else out_format
    cap = max(P["cap"], 1)
    if out_format == moe.COMBINE_BF16:
        o, osc = fill_pattern(torch.empty(cap, w.H, dtype=torch.bfloat16, device="cuda")), None
    else:
        o = fill_pattern(torch.empty(cap, w.H if out_format == moe.COMBINE_MXFP8 else w.H // 2, dtype=torch.uint8,
                                     device="cuda"))
        osc = fill_pattern(torch.empty(cap, w.H // 32, dtype=torch.uint8, device="cuda"))
    moe.moe_grouped_mlp_ex(P["handle"], P["shape"], P["layout"], P["mlp_dtype"], P["y"], P["ys"], P["q13"],
                           P["s13"], P["q2"], P["s2"], P["globals"], P["ws"], out_format, o, osc, row_probs)
    out = None
    if combine:
        out = fill_pattern(torch.empty(max(w.T, 1), w.H, dtype=torch.bfloat16, device="cuda"))
        moe.moe_combine_unpermute_fmt(P["handle"], P["shape"], P["layout"], out_format, o, osc, None, out)
    torch.cuda.synchronize()
    return o, osc, out


def oracle_inputs(oracle, P, pre):
    """Oracle-format dispatched rows, the oracle's perm probabilities and an
    expert-weight quantizer in the oracle's format."""
    w = P["w"]
    xb = workloads.bf16_bits(P["x"])
    if P["dtype"] == "bf16":
        xq, xs, fmt, globs = xb, None, 0, {}
    elif P["dtype"] == "fp8":
        (xq, xs), fmt, globs = oracle.quantize_fp8_rows(xb), 1, {}
    else:
        (xq, xs), fmt = oracle.quantize_nvfp4_rows(xb, float(P["gx"])), 2
        globs = dict(fc1_in_global=float(P["gx"]), fc2_in_global=float(np.float32(FC2_IN_GLOBAL)))
    yq, po = oracle.dispatch(P["fmt"], P["rmap"], P["probs"], pre, xq, P["cap"], w.E, w.K)
    ys = oracle.dispatch(P["fmt"], P["rmap"], None, pre, xs, P["cap"], w.E, w.K)[0] if xs is not None else None

    def weights(ex):
        a13, a2 = workloads.bf16_bits(P["w13"][ex]), workloads.bf16_bits(P["w2"][ex])
        if P["dtype"] == "bf16":
            return a13, None, a2, None, None, None
        if P["dtype"] == "fp8":
            return (*oracle.quantize_fp8_weight(a13), *oracle.quantize_fp8_weight(a2), None, None)
        q13, s13, q2, s2 = [], [], [], []
        for i, e in enumerate(ex):
            a, b = oracle.quantize_nvfp4_rows(a13[i], float(P["g13"][e]))
            c, d = oracle.quantize_nvfp4_rows(a2[i], float(P["g2"][e]))
            q13.append(a), s13.append(b), q2.append(c), s2.append(d)
        return np.stack(q13), np.stack(s13), np.stack(q2), np.stack(s2), P["g13"][ex], P["g2"][ex]

    return fmt, yq, ys, po, weights, globs


def check_rows_and_layer(oracle, P, o, out, rows=None, toks=None):
    """Oracle probs-in-MLP rows (default: every routed row) and the unweighted
    combine of the given tokens (default: all)."""
    w = P["w"]
    pre = oracle.preprocess(P["fmt"], P["rmap"], w.T, w.E, w.K, w.m, P["cap"])
    fmt, yq, ys, po, weights, globs = oracle_inputs(oracle, P, pre)
    if rows is None:
        rows = np.arange(pre["valid_rows"])[pre["token_of"] >= 0]
    toks = np.arange(w.T) if toks is None else toks
    tok_rows = pre["row_of"][toks]
    rows = np.unique(np.concatenate([np.asarray(rows, np.int64), tok_rows[tok_rows >= 0]]))
    sel, ob = oracle_rows_chunked(oracle, fmt, yq, ys, pre, rows, w.H, w.I, weights, perm_probs=po, **globs)
    got = bits(o[torch.from_numpy(sel).cuda()])
    assert rel_err(oracle.bf16_to_f64(got), oracle.bf16_to_f64(ob)) <= TOL[P["dtype"]]
    # pad rows hold zero input and stay zero after scaling
    o_all = bits(o)
    for e in range(w.E):
        pads = range(pre["offsets"][e] + pre["counts"][e], min(pre["offsets"][e + 1], P["cap"]))
        assert all(not o_all[r].any() for r in pads)
    # the layer: unweighted combine of the scaled rows
    o_full = np.zeros((P["cap"], w.H), np.uint16)
    o_full[sel] = ob
    yref = oracle.combine(o_full, tok_rows, None)
    o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), tok_rows, None)
    assert layer_rel_err(oracle.bf16_to_f64(bits(out[torch.from_numpy(toks).cuda()])), oracle.bf16_to_f64(yref),
                         o_rows, wts) <= TOL[P["dtype"]]


CASES = [
    ("bf16_fused_ragged", "bf16", workloads.scaled(workloads.WORKLOADS["tiny"], T=300, H=384, E=5, K=2, I=128)),
    ("bf16_fused_pad8", "bf16", workloads.scaled(workloads.WORKLOADS["tiny"], T=513, H=256, E=12, K=3, I=256, m=8)),
    ("bf16_pair", "bf16", workloads.scaled(workloads.WORKLOADS["tiny"], T=4160, H=512, E=2, K=2, I=256)),
    ("fp8", "fp8", workloads.scaled(workloads.WORKLOADS["dsv3"], T=256, H=512, E=8, K=2, I=256)),
    ("fp8_ragged_h384", "fp8", workloads.scaled(workloads.WORKLOADS["dsv3"], T=300, H=384, E=6, K=3, I=128)),
    ("nvfp4", "nvfp4", workloads.scaled(workloads.WORKLOADS["decode256"], T=77, H=512, E=6, K=3, I=512, m=8)),
]


@pytest.mark.parametrize("name,dtype,w", CASES, ids=[c[0] for c in CASES])
def test_probs_in_mlp_matches_oracle(oracle, moe, name, dtype, w):
    P = prepare(moe, w, dtype, seed=83)
    o, _, out = run_mlp(moe, P, P["yp"])
    if name == "bf16_pair":
        assert moe.moe_grouped_mlp_kernel_count(P["shape"], P["layout"], moe.DTYPE_BF16) == 2  # SM-pair kernels
        pre = oracle.preprocess(P["fmt"], P["rmap"], w.T, w.E, w.K, w.m, P["cap"])
        head, _ = largest_expert_rows(pre, P["cap"], 192)
        rows = np.concatenate([head, segment_edge_rows(pre, P["cap"])])
        toks = np.sort(np.random.default_rng(2).choice(w.T, 24, replace=False))
        check_rows_and_layer(oracle, P, o, out, rows, toks)
    else:
        check_rows_and_layer(oracle, P, o, out)


@pytest.mark.parametrize("elem", [0, 1])
def test_probs_in_mlp_mx_output_matches_oracle(oracle, moe, elem):
    """FP8 path writing MXFP8 / MXFP4 FC2 rows with the probabilities applied
    before the MX encoding: the oracle's codes and E8M0 scales, and the
    unweighted MX combine."""
    w = workloads.scaled(workloads.WORKLOADS["dsv3"], T=192, H=512, E=6, K=2, I=256)
    P = prepare(moe, w, "fp8", seed=84)
    ofmt = moe.COMBINE_MXFP8 if elem == 0 else moe.COMBINE_MXFP4
    oc, osc, out = run_mlp(moe, P, P["yp"], ofmt)
    pre = oracle.preprocess(P["fmt"], P["rmap"], w.T, w.E, w.K, w.m, P["cap"])
    fmt, yq, ys, po, weights, _ = oracle_inputs(oracle, P, pre)
    rows = np.arange(pre["valid_rows"])
    rows = rows[pre["token_of"] >= 0]
    q13, s13, q2, s2, _, _ = weights(list(range(w.E)))
    codes, scales = oracle.grouped_mlp_rows_mx(fmt, yq, ys, w.H, w.I, w.E, pre["offsets"], q13, s13, q2, s2, rows,
                                               elem, row_probs=po[rows])
    got_c, got_s = oc.cpu().numpy()[rows], osc.cpu().numpy()[rows]
    # fp32 sums in another order may land on the other side of a code boundary
    assert np.mean(got_s == scales) > 0.99
    dec_got = oracle.mx_decode_rows(got_c, got_s, elem)
    dec_ref = oracle.mx_decode_rows(codes, scales, elem)
    assert rel_err(dec_got, dec_ref) <= TOL["fp8"] * 2
    ref = oracle.combine_mx(_place(codes, rows, P["cap"]), _place(scales, rows, P["cap"]), elem, pre["row_of"])
    o_full = np.zeros((P["cap"], w.H))
    o_full[rows] = dec_ref
    o_rows, wts = gather_rows(o_full, pre["row_of"], None)
    assert layer_rel_err(oracle.bf16_to_f64(bits(out[:w.T])), oracle.bf16_to_f64(ref), o_rows, wts) <= TOL["fp8"] * 2


def _place(a, rows, cap):
    full = np.zeros((cap,) + a.shape[1:], a.dtype)
    full[rows] = a
    return full


@pytest.mark.parametrize("name,dtype,out_format", [
    ("dsv3_fp8", "fp8", "bf16"),
    ("dsv3_fp8", "fp8", "mxfp8"),
    ("mid_layer_bf16", "bf16", "bf16"),
    ("decode64_nvfp4", "nvfp4", "bf16"),
])
def test_power_of_two_probs_scale_rows_exactly_full_size(moe, name, dtype, out_format):
    """Full-size shapes (unbounded capacity): with p = 2^k per row every bf16
    FC2 row is exactly 2^k times the row written without probabilities (MX
    rows: identical codes, E8M0 byte + k), and with the dispatched
    probabilities each row is within one rounding of p times the fp32 sum,
    i.e. within two bf16 steps of p times the unscaled row."""
    w = workloads.WORKLOADS[{"dsv3_fp8": "dsv3", "mid_layer_bf16": "mid", "decode64_nvfp4": "decode64"}[name]]
    assert w.dtype == dtype
    P = prepare(moe, w, dtype, seed=0)
    ofmt = {"bf16": moe.COMBINE_BF16, "mxfp8": moe.COMBINE_MXFP8}[out_format]
    o0, s0, _ = run_mlp(moe, P, None, ofmt, combine=False)
    valid = min(int(P["handle"].total_rows.item()), P["cap"])
    k = torch.from_numpy(np.random.default_rng(5).integers(-4, 3, max(P["cap"], 1))).cuda()
    p2 = torch.ldexp(torch.ones_like(k, dtype=torch.float32), k)
    o1, s1, _ = run_mlp(moe, P, p2, ofmt, combine=False)
    if ofmt == moe.COMBINE_BF16:
        a0 = o0[:valid].float()
        assert torch.equal(o1[:valid].float(), a0 * p2[:valid, None])
        assert a0.abs().max().item() > 0
        # the dispatched probabilities: one rounding of p x the fp32 sum against p x the rounded row
        o2, _, _ = run_mlp(moe, P, P["yp"], ofmt, combine=False)
        p = P["yp"][:valid, None]
        scaled = a0 * p
        ulp = torch.ldexp(torch.ones_like(scaled), torch.floor(torch.log2(scaled.abs().clamp_min(2.0 ** -126)))
                          .to(torch.int32) - 7)
        assert torch.all((o2[:valid].float() - scaled).abs() <= 2 * ulp)
    else:
        # routed rows (pad rows are all-zero blocks, whose exponent byte does not move)
        routed = (P["handle"].token_of[:valid] >= 0).nonzero().squeeze(1)
        assert torch.equal(o1[routed], o0[routed])
        assert torch.equal(s1[routed].to(torch.int32), s0[routed].to(torch.int32) + k[routed, None].to(torch.int32))
