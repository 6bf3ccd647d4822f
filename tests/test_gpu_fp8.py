"""GPU parity of the FP8 path (E4M3 with fp32 block scales: 1x128 for
activations, 128x128 for weights): fused bf16 -> FP8 dispatch, the FP8 grouped
SwiGLU MLP (FP8 intermediate) and the bf16 combine, against the CPU oracle
(max-abs-error beyond one bf16 step <= 5e-2 of the output RMS)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import bits, fill_pattern, gather_rows, layer_rel_err, moe_mod, preprocess, rel_err

pytestmark = pytest.mark.gpu

TOL_FP8 = 5e-2


@pytest.fixture(scope="module")
def moe():
    return moe_mod()


def _case(**kw):
    return workloads.scaled(workloads.WORKLOADS["dsv3"], **kw)


def run_layer_fp8(moe, w, seed, cap=None):
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
    y = fill_pattern(torch.empty(max(cap, 1), w.H, dtype=torch.uint8, device="cuda"))
    ys = fill_pattern(torch.empty(max(cap, 1), w.H // 128, dtype=torch.float32, device="cuda"))
    yp = torch.empty(max(cap, 1), dtype=torch.float32, device="cuda")
    moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16_TO_FP8, x.cuda(), None, routing_t, y, yp, ys)
    ws = fill_pattern(torch.empty(moe.moe_grouped_mlp_workspace_size(shape, layout, moe.DTYPE_FP8_E4M3_B128),
                                  dtype=torch.uint8, device="cuda"))
    o = fill_pattern(torch.empty(max(cap, 1), w.H, dtype=torch.bfloat16, device="cuda"))
    moe.moe_grouped_mlp(handle, shape, layout, moe.DTYPE_FP8_E4M3_B128, y, ys, q13, s13, q2, s2, None, ws, o)
    out = fill_pattern(torch.empty(max(w.T, 1), w.H, dtype=torch.bfloat16, device="cuda"))
    moe.moe_combine_unpermute(handle, shape, layout, o, yp, out)
    torch.cuda.synchronize()
    return dict(fmt=fmt, rmap=rmap, probs=probs, cap=cap, x=x, w13=w13, w2=w2, o=o, out=out[:w.T])


def _oracle_rows(oracle, w, r, rows, pre):
    """Oracle FP8 FFN of the given permuted rows (weights quantized by the oracle)."""
    xq, xs = oracle.quantize_fp8_rows(workloads.bf16_bits(r["x"]))
    yq, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xq, r["cap"], w.E, w.K)
    ys, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xs, r["cap"], w.E, w.K)
    experts = sorted({int(np.searchsorted(pre["offsets"], rr, side="right") - 1) for rr in rows})
    q13, s13 = oracle.quantize_fp8_weight(workloads.bf16_bits(r["w13"][experts]))
    q2, s2 = oracle.quantize_fp8_weight(workloads.bf16_bits(r["w2"][experts]))
    sel, off = [], [0]
    for e in experts:
        rr = rows[(rows >= pre["offsets"][e]) & (rows < pre["offsets"][e + 1])]
        sel.append(rr)
        off.append(off[-1] + len(rr))
    sel = np.concatenate(sel)
    ob, _ = oracle.grouped_mlp_rows(1, yq[sel], ys[sel], w.H, w.I, len(experts), np.array(off, np.int32), q13, s13,
                                    q2, s2, np.arange(len(sel)))
    return sel, ob


@pytest.mark.parametrize("name,w", [
    ("small", _case(T=256, H=512, E=8, K=2, I=256)),
    ("ragged_h384", _case(T=300, H=384, E=6, K=3, I=128)),
    ("skewed_e32", _case(T=1024, H=256, E=32, K=4, I=384)),
    ("max_experts_1024", _case(T=600, H=256, E=1024, K=2, I=128, m=8)),
    ("one_expert", _case(T=300, H=256, E=1, K=1, I=128)),
], ids=lambda v: v if isinstance(v, str) else "")
def test_fp8_layer_all_rows(oracle, moe, name, w):
    r = run_layer_fp8(moe, w, seed=61)
    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, r["cap"])
    v = pre["valid_rows"]
    rows = np.arange(v)
    nonpad = rows[pre["token_of"] >= 0]
    sel, ob = _oracle_rows(oracle, w, r, nonpad, pre)
    got = bits(r["o"][torch.from_numpy(sel).cuda()])
    assert rel_err(oracle.bf16_to_f64(got), oracle.bf16_to_f64(ob)) <= TOL_FP8
    # pad rows: zero input rows give exactly zero output
    o_all = bits(r["o"])
    for e in range(w.E):
        for row in range(pre["offsets"][e] + pre["counts"][e], min(pre["offsets"][e + 1], r["cap"])):
            assert not o_all[row].any()
    _, po = oracle.dispatch(r["fmt"], r["rmap"], r["probs"], pre, np.zeros((w.T, 1), np.uint8), r["cap"], w.E, w.K)
    o_full = np.zeros((r["cap"], w.H), np.uint16)
    o_full[sel] = ob
    yref = oracle.combine(o_full, pre["row_of"], po)
    o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), pre["row_of"], po)
    assert layer_rel_err(oracle.bf16_to_f64(bits(r["out"])), oracle.bf16_to_f64(yref), o_rows, wts) <= TOL_FP8


def test_dsv3_layer_full_size_sampled(oracle, moe):
    """8192 tokens, hidden 7168, 256 Zipf(1.2)-skewed experts, top-8,
    intermediate 2048, FP8, in the launch configuration the benchmark times.
    The oracle recomputes: every route of 6 sampled tokens (and their combined
    outputs); the first and the last valid row of every expert segment (the
    first token tile and the ragged last tile of all 256 experts, across every
    CTA's share of the tile list); 128 rows spread over the largest expert
    (thousands of rows, dozens of token tiles)."""
    from gpu_util import largest_expert_rows, oracle_rows_chunked, segment_edge_rows

    w = workloads.WORKLOADS["dsv3"]
    r = run_layer_fp8(moe, w, seed=0)
    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, r["cap"])
    assert pre["counts"].max() > 10 * np.median(pre["counts"])
    toks = np.sort(np.random.default_rng(3).choice(w.T, 6, replace=False))
    tok_rows = np.unique(pre["row_of"][toks][pre["row_of"][toks] >= 0])
    head_rows, head = largest_expert_rows(pre, r["cap"], 128)
    assert pre["counts"][head] > 50 * 128  # the Zipf head spans dozens of token tiles
    edge_rows = segment_edge_rows(pre, r["cap"])
    assert len(edge_rows) >= 2 * 250
    rows = np.unique(np.concatenate([tok_rows, head_rows, edge_rows]))

    xq, xs = oracle.quantize_fp8_rows(workloads.bf16_bits(r["x"]))
    yq, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xq, r["cap"], w.E, w.K)
    ys, _ = oracle.dispatch(r["fmt"], r["rmap"], None, pre, xs, r["cap"], w.E, w.K)

    def weights(ex):
        q13, s13 = oracle.quantize_fp8_weight(workloads.bf16_bits(r["w13"][ex]))
        q2, s2 = oracle.quantize_fp8_weight(workloads.bf16_bits(r["w2"][ex]))
        return q13, s13, q2, s2, None, None

    sel, ob = oracle_rows_chunked(oracle, 1, yq, ys, pre, rows, w.H, w.I, weights)
    got = bits(r["o"][torch.from_numpy(sel).cuda()])
    for name, subset in (("edges", edge_rows), ("largest expert", head_rows), ("sampled tokens", tok_rows)):
        m = np.isin(sel, subset)
        assert rel_err(oracle.bf16_to_f64(got[m]), oracle.bf16_to_f64(ob[m])) <= TOL_FP8, name
    _, po = oracle.dispatch(r["fmt"], r["rmap"], r["probs"], pre, np.zeros((w.T, 1), np.uint8), r["cap"], w.E, w.K)
    o_full = np.zeros((r["cap"], w.H), np.uint16)
    o_full[sel] = ob
    yref = oracle.combine(o_full, pre["row_of"][toks], po)
    o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), pre["row_of"][toks], po)
    assert layer_rel_err(oracle.bf16_to_f64(bits(r["out"][torch.from_numpy(toks).cuda()])),
                         oracle.bf16_to_f64(yref), o_rows, wts) <= TOL_FP8


def test_fp8_overflowed_capacity(oracle, moe):
    """Capacity at half the padded rows (4-aligned, cutting an expert segment
    inside a token tile): the kept rows match the oracle, pad rows are zero,
    rows at or past the capacity's end of the segments are never written, and
    dropped routes contribute nothing to the layer."""
    w = _case(T=256, H=512, E=8, K=2, I=256)
    fmt, rmap, _ = workloads.routing_inputs(w, 63)
    total = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
    cap = oracle.capacity(total // 2 + 6, 1.0)
    r = run_layer_fp8(moe, w, seed=63, cap=cap)
    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, cap)
    assert pre["overflow"] == 1 and cap % 32 != 0
    v = pre["valid_rows"]
    rows = np.arange(v)[pre["token_of"] >= 0]
    sel, ob = _oracle_rows(oracle, w, r, rows, pre)
    got = bits(r["o"][torch.from_numpy(sel).cuda()])
    assert rel_err(oracle.bf16_to_f64(got), oracle.bf16_to_f64(ob)) <= TOL_FP8
    o_all = bits(r["o"])
    for e in range(w.E):
        for row in range(pre["offsets"][e] + pre["counts"][e], min(pre["offsets"][e + 1], cap)):
            assert not o_all[row].any()
    assert np.all(o_all[v:] == 0xFFFF)
    _, po = oracle.dispatch(r["fmt"], r["rmap"], r["probs"], pre, np.zeros((w.T, 1), np.uint8), cap, w.E, w.K)
    o_full = np.zeros((cap, w.H), np.uint16)
    o_full[sel] = ob
    yref = oracle.combine(o_full, pre["row_of"], po)
    o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), pre["row_of"], po)
    assert layer_rel_err(oracle.bf16_to_f64(bits(r["out"])), oracle.bf16_to_f64(yref), o_rows, wts) <= TOL_FP8
