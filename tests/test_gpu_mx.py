"""GPU parity of the MX combine formats (E4M3 or E2M1 elements with one E8M0
scale per 32): the bf16 -> MX row quantizer bit for bit against the oracle, the
combine reading MX rows against the oracle's combine of the same codes, and the
FP8 layer whose FC2 epilogue writes MX rows against the oracle's MX layer.
Where the GPU (fp32 sums) and the oracle (double sums) encode a value that
sits at an element-grid boundary differently, the two codes are one element
step apart: the FP8 / NVFP4 budget of 5e-2 of the output RMS applies beyond
that step."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import bf16_ulp, bits, fill_pattern, moe_mod, preprocess

pytestmark = pytest.mark.gpu

TOL = 5e-2


@pytest.fixture(scope="module")
def moe():
    return moe_mod()


def _elem_step(oracle, dec, scales, elem):
    """Spacing of the element grid at each decoded value (in value units)."""
    X = np.repeat(scales.astype(np.int64) - 127, 32, axis=1)
    q = np.abs(dec) / np.ldexp(1.0, X)
    if elem == 0:
        e = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
        step = np.ldexp(1.0, (e - 3).astype(np.int64))
    else:
        step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    return step * np.ldexp(1.0, X)


@pytest.mark.parametrize("elem", [0, 1])
def test_quantize_mx_rows_bit_exact(oracle, moe, elem):
    rng = np.random.default_rng(elem)
    R, H = 300, 512
    x = torch.from_numpy((rng.standard_normal((R, H)) * np.exp2(rng.integers(-8, 8, (R, H // 32)))
                          .repeat(32, axis=1)).astype(np.float32)).to(torch.bfloat16)
    x[0, :32] = 0
    fmt = moe.COMBINE_MXFP8 if elem == 0 else moe.COMBINE_MXFP4
    codes = fill_pattern(torch.empty(R, H if elem == 0 else H // 2, dtype=torch.uint8, device="cuda"))
    scales = fill_pattern(torch.empty(R, H // 32, dtype=torch.uint8, device="cuda"))
    moe.moe_quantize_mx_rows(x.cuda(), fmt, codes, scales)
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_mx_rows(x.float().numpy(), elem)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("elem", [0, 1])
@pytest.mark.parametrize("routing", ["dense", "sparse"])
def test_combine_from_mx_rows(oracle, moe, elem, routing):
    w = workloads.scaled(workloads.WORKLOADS["permute"], T=700, H=512, E=12, K=4)
    fmt, rmap, probs = workloads.routing_inputs(w, 9, routing)
    cap = int(oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"] * 0.8)  # some routes drop
    shape, layout, routing_t, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    _, yp = oracle.dispatch(fmt, rmap, probs, pre, np.zeros((w.T, 1), np.uint8), cap, w.E, w.K)
    rng = np.random.default_rng(4)
    rows = (rng.standard_normal((cap, w.H)) * np.exp2(rng.integers(-4, 4, (cap, w.H // 32))).repeat(32, axis=1))
    codes, scales = oracle.quantize_mx_rows(rows.astype(np.float32), elem)
    y = fill_pattern(torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda"))
    moe.moe_combine_unpermute_fmt(handle, shape, layout, moe.COMBINE_MXFP8 if elem == 0 else moe.COMBINE_MXFP4,
                                  torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(),
                                  torch.from_numpy(yp).cuda(), y)
    torch.cuda.synchronize()
    ref = oracle.bf16_to_f64(oracle.combine_mx(codes, scales, elem, pre["row_of"], yp))
    got = oracle.bf16_to_f64(bits(y))
    # fp32 accumulation of at most K exact products: within one bf16 step of the double sum
    assert np.all(np.abs(got - ref) <= bf16_ulp(ref))


def _run_fp8_layer_mx(moe, w, seed, elem, cap=None):
    fmt, rmap, probs = workloads.routing_inputs(w, seed)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m) if cap is None else cap
    x = workloads.activations(w, seed)
    w13, w2 = workloads.expert_weights(w, seed, device="cuda")
    q13 = torch.empty(w13.shape, dtype=torch.uint8, device="cuda")
    s13 = torch.empty(w.E, 2 * w.I // 128, w.H // 128, dtype=torch.float32, device="cuda")
    q2 = torch.empty(w2.shape, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(w.E, w.H // 128, w.I // 128, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_blocks(w13, q13, s13)
    moe.moe_quantize_fp8_blocks(w2, q2, s2)
    shape, layout, routing_t, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    y = torch.empty(cap, w.H, dtype=torch.uint8, device="cuda")
    ys = torch.empty(cap, w.H // 128, dtype=torch.float32, device="cuda")
    yp = torch.empty(cap, dtype=torch.float32, device="cuda")
    moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16_TO_FP8, x.cuda(), None, routing_t, y, yp, ys)
    ws = torch.empty(moe.moe_grouped_mlp_workspace_size(shape, layout, moe.DTYPE_FP8_E4M3_B128), dtype=torch.uint8,
                     device="cuda")
    oc = fill_pattern(torch.empty(cap, w.H if elem == 0 else w.H // 2, dtype=torch.uint8, device="cuda"))
    osc = fill_pattern(torch.empty(cap, w.H // 32, dtype=torch.uint8, device="cuda"))
    ofmt = moe.COMBINE_MXFP8 if elem == 0 else moe.COMBINE_MXFP4
    moe.moe_grouped_mlp_ex(handle, shape, layout, moe.DTYPE_FP8_E4M3_B128, y, ys, q13, s13, q2, s2, None, ws, ofmt,
                            oc, osc)
    out = fill_pattern(torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda"))
    moe.moe_combine_unpermute_fmt(handle, shape, layout, ofmt, oc, osc, yp, out)
    torch.cuda.synchronize()
    return dict(fmt=fmt, rmap=rmap, probs=probs, cap=cap, x=x, w13=w13, w2=w2, oc=oc.cpu().numpy(),
                osc=osc.cpu().numpy(), out=out)


def _check_fp8_layer_mx(oracle, w, r, elem, toks):
    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, r["cap"])
    xq, xs = oracle.quantize_fp8_rows(workloads.bf16_bits(r["x"]))
    yq, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xq, r["cap"], w.E, w.K)
    ys, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xs, r["cap"], w.E, w.K)
    rows = pre["row_of"][toks]
    rows = np.unique(rows[rows >= 0])
    owner = np.searchsorted(pre["offsets"], rows, side="right") - 1
    experts = sorted(set(owner.tolist()))
    q13, s13 = oracle.quantize_fp8_weight(workloads.bf16_bits(r["w13"][experts]))
    q2, s2 = oracle.quantize_fp8_weight(workloads.bf16_bits(r["w2"][experts]))
    sel, off = [], [0]
    for e in experts:
        rr = rows[owner == e]
        sel.append(rr)
        off.append(off[-1] + len(rr))
    sel = np.concatenate(sel)
    rc, rs = oracle.grouped_mlp_rows_mx(1, yq[sel], ys[sel], w.H, w.I, len(experts), np.array(off, np.int32), q13,
                                        s13, q2, s2, np.arange(len(sel)), elem)
    ref = oracle.mx_decode_rows(rc, rs, elem)
    got = oracle.mx_decode_rows(r["oc"][sel], r["osc"][sel], elem)
    assert np.mean(r["osc"][sel] == rs) > 0.99
    step = np.maximum(_elem_step(oracle, ref, rs, elem), _elem_step(oracle, got, r["osc"][sel], elem))
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.maximum(np.abs(got - ref) - step, 0).max() <= TOL * rms
    # the layer output: the combine of the oracle's MX rows, with each route's one-step allowance carried
    c_full = np.zeros((r["cap"],) + rc.shape[1:], np.uint8)
    s_full = np.full((r["cap"], w.H // 32), 127, np.uint8)
    c_full[sel], s_full[sel] = rc, rs
    _, po = oracle.dispatch(r["fmt"], r["rmap"], r["probs"], pre, np.zeros((w.T, 1), np.uint8), r["cap"], w.E, w.K)
    yref = oracle.bf16_to_f64(oracle.combine_mx(c_full, s_full, elem, pre["row_of"][toks], po))
    ygot = oracle.bf16_to_f64(bits(r["out"][torch.from_numpy(toks).cuda()]))
    st_full = np.zeros((r["cap"], w.H))
    st_full[sel] = step
    ro = pre["row_of"][toks]
    keep = ro >= 0
    carried = np.einsum("tk,tkh->th", np.abs(po[np.where(keep, ro, 0)]) * keep, st_full[np.where(keep, ro, 0)])
    yrms = np.sqrt(np.mean(yref ** 2))
    assert np.maximum(np.abs(ygot - yref) - bf16_ulp(yref) - carried, 0).max() <= TOL * yrms


@pytest.mark.parametrize("elem", [0, 1])
def test_fp8_layer_with_mx_fc2_output(oracle, moe, elem):
    w = workloads.scaled(workloads.WORKLOADS["dsv3"], T=256, H=512, E=8, K=2, I=256)
    r = _run_fp8_layer_mx(moe, w, 61, elem)
    _check_fp8_layer_mx(oracle, w, r, elem, np.arange(w.T))


@pytest.mark.parametrize("elem", [0, 1])
def test_fp8_layer_mx_output_ragged_hidden(oracle, moe, elem):
    """H = 384: FC2's last 256-column tile is half past the rows' end; its second
    half is computed but neither codes nor scales are written."""
    w = workloads.scaled(workloads.WORKLOADS["dsv3"], T=200, H=384, E=6, K=3, I=256)
    r = _run_fp8_layer_mx(moe, w, 62, elem)
    _check_fp8_layer_mx(oracle, w, r, elem, np.arange(w.T))


@pytest.mark.parametrize("elem", [0, 1])
def test_fp8_layer_mx_output_capacity_cut(oracle, moe, elem):
    """A capacity below the padded total: kept rows match the oracle, rows from
    the capacity on are never written (their 0xFF pre-fill stays), and the
    combine skips the dropped routes."""
    w = workloads.scaled(workloads.WORKLOADS["dsv3"], T=256, H=512, E=8, K=2, I=256)
    fmt, rmap, _ = workloads.routing_inputs(w, 63)
    total = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
    cap = int(total * 0.7) // 4 * 4
    r = _run_fp8_layer_mx(moe, w, 63, elem, cap=cap)
    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, cap)
    assert pre["overflow"] == 1
    _check_fp8_layer_mx(oracle, w, r, elem, np.arange(w.T))
    assert np.all(r["oc"][pre["valid_rows"]:] == 0xFF) and np.all(r["osc"][pre["valid_rows"]:] == 0xFF)


def test_dsv3_layer_with_mxfp8_combine_full_size_sampled(oracle, moe):
    """8192 tokens, hidden 7168, 256 Zipf-skewed experts, FP8 GEMMs, FC2 writing
    MXFP8 and the combine reading it: the rows of 6 sampled tokens."""
    w = workloads.WORKLOADS["dsv3"]
    r = _run_fp8_layer_mx(moe, w, 0, 0)
    toks = np.sort(np.random.default_rng(3).choice(w.T, 6, replace=False))
    _check_fp8_layer_mx(oracle, w, r, 0, toks)


def test_mx_output_unsupported_on_bf16_path(moe):
    w = workloads.scaled(workloads.WORKLOADS["tiny"], T=64, H=256, E=4, K=2, I=128)
    shape, layout = moe.Shape(w.T, w.H, w.E, w.K, w.I), moe.Layout(32, 256)
    h = moe.Handle.empty(shape, layout)
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_grouped_mlp_ex(h, shape, layout, moe.DTYPE_BF16, buf, None, buf, None, buf, None, None, buf,
                                moe.COMBINE_MXFP8, buf, buf)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
