"""GPU parity of the NVFP4 decode path (W4A4: E2M1 values, E4M3 scale per 16
elements, fp32 global per tensor): fused bf16 -> NVFP4 dispatch, the NVFP4
grouped SwiGLU MLP (NVFP4 intermediate) and the bf16 combine, against the CPU
oracle (max-abs-error beyond one bf16 step <= 5e-2 of the output RMS)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import bits, fill_pattern, gather_rows, layer_rel_err, moe_mod, preprocess, rel_err

pytestmark = pytest.mark.gpu

TOL_FP4 = 5e-2
FC2_IN_GLOBAL = 0.01  # calibration constant of the intermediate, an input to both sides


@pytest.fixture(scope="module")
def moe():
    return moe_mod()


def _case(**kw):
    return workloads.scaled(workloads.WORKLOADS["decode256"], **kw)


def _globals(x, w13, w2):
    """fp32 global scales amax / (6 * 448), computed once on the host (inputs to both sides)."""
    gx = np.float32(x.float().abs().max().item() / 2688.0)
    g13 = (w13.float().abs().amax(dim=(1, 2)) / 2688.0).cpu().numpy().astype(np.float32)
    g2 = (w2.float().abs().amax(dim=(1, 2)) / 2688.0).cpu().numpy().astype(np.float32)
    return gx, g13, g2


def run_layer_nvfp4(moe, w, seed, cap=None):
    fmt, rmap, probs = workloads.routing_inputs(w, seed)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m) if cap is None else cap
    x = workloads.activations(w, seed)
    w13, w2 = workloads.expert_weights(w, seed, device="cuda")
    gx, g13, g2 = _globals(x, w13, w2)
    dev = "cuda"
    q13 = torch.empty(w.E, 2 * w.I, w.H // 2, dtype=torch.uint8, device=dev)
    s13 = torch.empty(w.E, 2 * w.I, w.H // 16, dtype=torch.uint8, device=dev)
    q2 = torch.empty(w.E, w.H, w.I // 2, dtype=torch.uint8, device=dev)
    s2 = torch.empty(w.E, w.H, w.I // 16, dtype=torch.uint8, device=dev)
    g13_d, g2_d = torch.from_numpy(g13).to(dev), torch.from_numpy(g2).to(dev)
    for e in range(w.E):
        moe.moe_quantize_nvfp4_rows(w13[e], g13_d[e:e + 1], q13[e], s13[e])
        moe.moe_quantize_nvfp4_rows(w2[e], g2_d[e:e + 1], q2[e], s2[e])
    gx_d = torch.tensor([gx], device=dev)
    globals_ = moe.Nvfp4Globals(gx_d, torch.tensor([FC2_IN_GLOBAL], dtype=torch.float32, device=dev), g13_d, g2_d)
    shape, layout, routing_t, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    y = fill_pattern(torch.empty(max(cap, 1), w.H // 2, dtype=torch.uint8, device=dev))
    ys = fill_pattern(torch.empty(max(cap, 1), w.H // 16, dtype=torch.uint8, device=dev))
    yp = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
    moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16_TO_NVFP4, x.to(dev), gx_d, routing_t, y, yp, ys)
    ws = fill_pattern(torch.empty(moe.moe_grouped_mlp_workspace_size(shape, layout, moe.DTYPE_NVFP4),
                                  dtype=torch.uint8, device=dev))
    o = fill_pattern(torch.empty(max(cap, 1), w.H, dtype=torch.bfloat16, device=dev))
    moe.moe_grouped_mlp(handle, shape, layout, moe.DTYPE_NVFP4, y, ys, q13, s13, q2, s2, globals_, ws, o)
    out = fill_pattern(torch.empty(max(w.T, 1), w.H, dtype=torch.bfloat16, device=dev))
    moe.moe_combine_unpermute(handle, shape, layout, o, yp, out)
    torch.cuda.synchronize()
    return dict(fmt=fmt, rmap=rmap, probs=probs, cap=cap, x=x, w13=w13, w2=w2, gx=gx, g13=g13, g2=g2, o=o,
                out=out[:w.T])


def _oracle_rows(oracle, w, r, rows, pre):
    xq, xs = oracle.quantize_nvfp4_rows(workloads.bf16_bits(r["x"]), float(r["gx"]))
    yq, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xq, r["cap"], w.E, w.K)
    ys, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xs, r["cap"], w.E, w.K)
    experts = sorted({int(np.searchsorted(pre["offsets"], rr, side="right") - 1) for rr in rows})
    q13, s13, q2, s2 = [], [], [], []
    for e in experts:
        a, b = oracle.quantize_nvfp4_rows(workloads.bf16_bits(r["w13"][e]), float(r["g13"][e]))
        c, d = oracle.quantize_nvfp4_rows(workloads.bf16_bits(r["w2"][e]), float(r["g2"][e]))
        q13.append(a), s13.append(b), q2.append(c), s2.append(d)
    sel, off = [], [0]
    for e in experts:
        rr = rows[(rows >= pre["offsets"][e]) & (rows < pre["offsets"][e + 1])]
        sel.append(rr)
        off.append(off[-1] + len(rr))
    sel = np.concatenate(sel)
    ob, _ = oracle.grouped_mlp_rows(2, yq[sel], ys[sel], w.H, w.I, len(experts), np.array(off, np.int32),
                                    np.stack(q13), np.stack(s13), np.stack(q2), np.stack(s2), np.arange(len(sel)),
                                    w13_global=r["g13"][experts], w2_global=r["g2"][experts],
                                    fc1_in_global=float(r["gx"]), fc2_in_global=float(np.float32(FC2_IN_GLOBAL)))
    return sel, ob


def _check(oracle, w, r, toks):
    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, r["cap"])
    rows = pre["row_of"][toks]
    rows = np.unique(rows[rows >= 0])
    sel, ob = _oracle_rows(oracle, w, r, rows, pre)
    got = bits(r["o"][torch.from_numpy(sel).cuda()])
    assert rel_err(oracle.bf16_to_f64(got), oracle.bf16_to_f64(ob)) <= TOL_FP4
    _, po = oracle.dispatch(r["fmt"], r["rmap"], r["probs"], pre, np.zeros((w.T, 1), np.uint8), r["cap"], w.E, w.K)
    o_full = np.zeros((r["cap"], w.H), np.uint16)
    o_full[sel] = ob
    yref = oracle.combine(o_full, pre["row_of"][toks], po)
    o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), pre["row_of"][toks], po)
    assert layer_rel_err(oracle.bf16_to_f64(bits(r["out"][torch.from_numpy(toks).cuda()])),
                         oracle.bf16_to_f64(yref), o_rows, wts) <= TOL_FP4
    return pre


@pytest.mark.parametrize("name,w", [
    ("small", _case(T=64, H=512, E=8, K=2, I=256)),
    ("many_token_tiles", _case(T=512, H=256, E=4, K=2, I=256)),
    ("pad8_ragged", _case(T=77, H=512, E=6, K=3, I=512, m=8)),
    ("one_expert", _case(T=40, H=256, E=1, K=1, I=256)),
], ids=lambda v: v if isinstance(v, str) else "")
def test_nvfp4_layer_all_tokens(oracle, moe, name, w):
    r = run_layer_nvfp4(moe, w, seed=71)
    pre = _check(oracle, w, r, np.arange(w.T))
    o_all = bits(r["o"])
    for e in range(w.E):
        for row in range(pre["offsets"][e] + pre["counts"][e], min(pre["offsets"][e + 1], r["cap"])):
            assert not o_all[row].any()


@pytest.mark.parametrize("name,n_tokens", [("decode64", 64), ("decode256", 32)])
def test_decode_full_size(oracle, moe, name, n_tokens):
    """64 / 256 tokens, hidden 7168, 256 experts, top-8, intermediate 2048,
    NVFP4, in the launch configuration the benchmark times: the oracle
    recomputes every route of every token (decode64) or of 32 sampled tokens
    (decode256), and their combined outputs."""
    from gpu_util import oracle_rows_chunked

    w = workloads.WORKLOADS[name]
    r = run_layer_nvfp4(moe, w, seed=0)
    toks = np.arange(w.T) if n_tokens >= w.T else np.sort(
        np.random.default_rng(5).choice(w.T, n_tokens, replace=False))
    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, r["cap"])
    rows = pre["row_of"][toks]
    rows = np.unique(rows[rows >= 0])
    xq, xs = oracle.quantize_nvfp4_rows(workloads.bf16_bits(r["x"]), float(r["gx"]))
    yq, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xq, r["cap"], w.E, w.K)
    ys, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xs, r["cap"], w.E, w.K)

    def weights(ex):
        q13, s13, q2, s2 = [], [], [], []
        for e in ex:
            a, b = oracle.quantize_nvfp4_rows(workloads.bf16_bits(r["w13"][e]), float(r["g13"][e]))
            c, d = oracle.quantize_nvfp4_rows(workloads.bf16_bits(r["w2"][e]), float(r["g2"][e]))
            q13.append(a), s13.append(b), q2.append(c), s2.append(d)
        return np.stack(q13), np.stack(s13), np.stack(q2), np.stack(s2), r["g13"][ex], r["g2"][ex]

    sel, ob = oracle_rows_chunked(oracle, 2, yq, ys, pre, rows, w.H, w.I, weights,
                                  fc1_in_global=float(r["gx"]), fc2_in_global=float(np.float32(FC2_IN_GLOBAL)))
    got = bits(r["o"][torch.from_numpy(sel).cuda()])
    assert rel_err(oracle.bf16_to_f64(got), oracle.bf16_to_f64(ob)) <= TOL_FP4
    _, po = oracle.dispatch(r["fmt"], r["rmap"], r["probs"], pre, np.zeros((w.T, 1), np.uint8), r["cap"], w.E, w.K)
    o_full = np.zeros((r["cap"], w.H), np.uint16)
    o_full[sel] = ob
    yref = oracle.combine(o_full, pre["row_of"][toks], po)
    o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), pre["row_of"][toks], po)
    assert layer_rel_err(oracle.bf16_to_f64(bits(r["out"][torch.from_numpy(toks).cuda()])),
                         oracle.bf16_to_f64(yref), o_rows, wts) <= TOL_FP4


def test_nvfp4_overflowed_capacity(oracle, moe):
    """Capacity at half the padded rows, cutting an expert segment inside a
    token tile: kept routes match the oracle (rows and layer), pad rows are
    zero and rows past the capacity's end of the segments are never written."""
    w = _case(T=160, H=512, E=6, K=3, I=256)
    fmt, rmap, _ = workloads.routing_inputs(w, 73)
    total = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
    cap = oracle.capacity(total // 2 + 6, 1.0)
    r = run_layer_nvfp4(moe, w, seed=73, cap=cap)
    pre = _check(oracle, w, r, np.arange(w.T))
    assert pre["overflow"] == 1 and cap % 32 != 0
    o_all = bits(r["o"])
    for e in range(w.E):
        for row in range(pre["offsets"][e] + pre["counts"][e], min(pre["offsets"][e + 1], cap)):
            assert not o_all[row].any()
    assert np.all(o_all[pre["valid_rows"]:] == 0xFFFF)
