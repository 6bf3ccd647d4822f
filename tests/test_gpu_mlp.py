"""GPU parity of the grouped SwiGLU expert MLP (tcgen05 grouped GEMMs) and of
the whole layer against the CPU oracle: max-abs-error / RMS of the output
<= 1e-2 for bf16 (<= 5e-2 for FP8 / NVFP4), fp32 accumulation on the GPU."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import bits, fill_pattern, gather_rows, handle_np, layer_rel_err, moe_mod, preprocess, rel_err

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2


@pytest.fixture(scope="module")
def moe():
    return moe_mod()


def _case(name, **kw):
    return workloads.scaled(workloads.WORKLOADS[name], **kw)


def run_layer_bf16(moe, w, seed, cap=None, routing=None):
    """The four calls on seeded inputs; returns everything the checks need."""
    fmt, rmap, probs = workloads.routing_inputs(w, seed, routing)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m) if cap is None else cap
    x = workloads.activations(w, seed)
    w13, w2 = workloads.expert_weights(w, seed, device="cuda")
    shape, layout, routing_t, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    y = fill_pattern(torch.empty(max(cap, 1), w.H, dtype=torch.bfloat16, device="cuda"))
    yp = torch.empty(max(cap, 1), dtype=torch.float32, device="cuda")
    moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16, x.cuda(), None, routing_t, y, yp)
    ws = fill_pattern(torch.empty(moe.moe_grouped_mlp_workspace_size(shape, layout, moe.DTYPE_BF16),
                                  dtype=torch.uint8, device="cuda"))
    o = fill_pattern(torch.empty(max(cap, 1), w.H, dtype=torch.bfloat16, device="cuda"))
    moe.moe_grouped_mlp(handle, shape, layout, moe.DTYPE_BF16, y, None, w13, None, w2, None, None, ws, o)
    out = fill_pattern(torch.empty(max(w.T, 1), w.H, dtype=torch.bfloat16, device="cuda"))
    moe.moe_combine_unpermute(handle, shape, layout, o, yp, out)
    torch.cuda.synchronize()
    return dict(fmt=fmt, rmap=rmap, probs=probs, cap=cap, x=x, w13=w13, w2=w2, handle=handle, o=o, out=out[:w.T])


@pytest.mark.parametrize("name,w", [
    ("tiny", _case("tiny")),
    ("ragged_h384", _case("tiny", T=200, H=384, E=5, K=2, I=128)),
    ("one_expert", _case("tiny", T=300, H=256, E=1, K=1, I=256)),
    ("m1_no_padding", _case("tiny", T=257, H=256, E=7, K=3, I=128, m=1)),
    ("many_experts_pad8", _case("tiny", T=1024, H=512, E=24, K=3, I=256, m=8)),
    ("max_experts_1024", _case("tiny", T=600, H=128, E=1024, K=2, I=128, m=8)),
    ("pair_large_experts", _case("tiny", T=4160, H=512, E=2, K=2, I=256)),
    ("pair_ragged_h384", _case("tiny", T=8400, H=384, E=4, K=2, I=128)),
], ids=lambda v: v if isinstance(v, str) else "")
def test_grouped_mlp_bf16_all_rows(oracle, moe, name, w):
    r = run_layer_bf16(moe, w, seed=21)
    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, r["cap"])
    yo, po = oracle.dispatch(r["fmt"], r["rmap"], r["probs"], pre, workloads.bf16_bits(r["x"]), r["cap"], w.E, w.K)
    v = pre["valid_rows"]
    w13b, w2b = workloads.bf16_bits(r["w13"]), workloads.bf16_bits(r["w2"])
    ob, _ = oracle.grouped_mlp_rows(0, yo, None, w.H, w.I, w.E, pre["offsets"], w13b, None, w2b, None,
                                    np.arange(v))
    got = bits(r["o"])
    assert rel_err(oracle.bf16_to_f64(got[:v]), oracle.bf16_to_f64(ob)) <= TOL_BF16
    # pad rows are exactly zero; rows past the segments untouched
    for e in range(w.E):
        for row in range(pre["offsets"][e] + pre["counts"][e], min(pre["offsets"][e + 1], r["cap"])):
            assert not got[row].any()
    assert np.all(got[v:] == 0xFFFF)
    # whole layer vs the unpermuted per-token formulation of the oracle
    ref = oracle.layer_per_token(0, r["fmt"], r["rmap"], r["probs"], w.E, w.K, workloads.bf16_bits(r["x"]), None,
                                 w.H, w.I, w13b, None, w2b, None, np.arange(w.T))
    o_full = np.zeros((r["cap"], w.H), np.uint16)
    o_full[:v] = ob
    o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), pre["row_of"], po)
    assert layer_rel_err(oracle.bf16_to_f64(bits(r["out"])), oracle.bf16_to_f64(ref), o_rows, wts) <= TOL_BF16


def _sampled_check(oracle, w, r, n_tokens=48, seed=0, edges=False):
    """Oracle on a sample of tokens (all their routes) at full size; with
    edges, also the first and last valid row of every expert segment."""
    from gpu_util import segment_edge_rows

    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, r["cap"])
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(w.T, n_tokens, replace=False))
    rows = np.unique(pre["row_of"][toks][pre["row_of"][toks] >= 0])
    if edges:
        rows = np.unique(np.concatenate([rows, segment_edge_rows(pre, r["cap"])]))
    xb = workloads.bf16_bits(r["x"])
    yo, po = oracle.dispatch(r["fmt"], r["rmap"], r["probs"], pre, xb, r["cap"], w.E, w.K)
    experts = sorted({int(np.searchsorted(pre["offsets"], rr, side="right") - 1) for rr in rows})
    # oracle weights for the experts involved only, remapped to local ids
    w13l = workloads.bf16_bits(r["w13"][experts])
    w2l = workloads.bf16_bits(r["w2"][experts])
    local_off = np.zeros(len(experts) + 1, np.int32)
    # give each involved expert its own contiguous block of the sampled rows
    sel_rows, blocks = [], []
    for j, e in enumerate(experts):
        rr = rows[(rows >= pre["offsets"][e]) & (rows < pre["offsets"][e + 1])]
        sel_rows.append(rr)
        local_off[j + 1] = local_off[j] + len(rr)
    sel = np.concatenate(sel_rows)
    ob, _ = oracle.grouped_mlp_rows(0, yo[sel], None, w.H, w.I, len(experts), local_off, w13l, None, w2l, None,
                                    np.arange(len(sel)))
    got = bits(r["o"][torch.from_numpy(sel).cuda()])
    assert rel_err(oracle.bf16_to_f64(got), oracle.bf16_to_f64(ob)) <= TOL_BF16
    # combine of the sampled tokens from the oracle's own expert rows
    o_full = np.zeros((r["cap"], w.H), np.uint16)
    o_full[sel] = ob
    yref = oracle.combine(o_full, pre["row_of"][toks], po)
    o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), pre["row_of"][toks], po)
    assert layer_rel_err(oracle.bf16_to_f64(bits(r["out"][torch.from_numpy(toks).cuda()])),
                         oracle.bf16_to_f64(yref), o_rows, wts) <= TOL_BF16


def test_mid_layer_full_size_sampled(oracle, moe):
    """4096 tokens, hidden 2048, 64 experts, top-8, sparse map, intermediate 1024,
    capacity factor 1.5 from a calibration pass: flag 0; sampled rows match."""
    w = workloads.WORKLOADS["mid"]
    fmt, rmap, probs = workloads.routing_inputs(w, 31)
    rows = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
    cap = oracle.capacity(rows, w.cap_factor)
    r = run_layer_bf16(moe, w, seed=31, cap=cap)
    assert handle_np(r["handle"], w.T, w.K, cap)["overflow"] == 0
    _sampled_check(oracle, w, r, edges=True)


def test_skewed_experts_with_empty_ones(oracle, moe):
    """Zipf-skewed popularity over 64 experts (some empty, one very large)."""
    w = _case("dsv3", T=2048, H=512, E=64, K=4, I=256, dtype="bf16")
    r = run_layer_bf16(moe, w, seed=41)
    pre = oracle.preprocess(r["fmt"], r["rmap"], w.T, w.E, w.K, w.m, r["cap"])
    assert pre["counts"].max() > 8 * np.median(pre["counts"])
    _sampled_check(oracle, w, r, n_tokens=64)


def test_overflowed_capacity_layer(oracle, moe):
    """Capacity below the routed rows: dropped routes contribute nothing."""
    w = _case("tiny", T=256, H=256, E=8, K=2, I=128)
    fmt, rmap, probs = workloads.routing_inputs(w, 51)
    rows = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
    cap = oracle.capacity(rows // 2, 1.0)
    r = run_layer_bf16(moe, w, seed=51, cap=cap)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    assert pre["overflow"] == 1
    yo, po = oracle.dispatch(fmt, rmap, probs, pre, workloads.bf16_bits(r["x"]), cap, w.E, w.K)
    v = pre["valid_rows"]
    ob, _ = oracle.grouped_mlp_rows(0, yo, None, w.H, w.I, w.E, pre["offsets"], workloads.bf16_bits(r["w13"]), None,
                                    workloads.bf16_bits(r["w2"]), None, np.arange(v))
    o_full = np.zeros((cap, w.H), np.uint16)
    o_full[:v] = ob
    yref = oracle.combine(o_full, pre["row_of"], po)
    o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), pre["row_of"], po)
    assert layer_rel_err(oracle.bf16_to_f64(bits(r["out"])), oracle.bf16_to_f64(yref), o_rows, wts) <= TOL_BF16


def test_whole_layer_in_one_cuda_graph(oracle, moe):
    """preprocess -> dispatch -> fused grouped MLP -> combine captured once and
    replayed with new routing and activations written into the same input
    buffers: the MLP's claim and completion counters are re-zeroed inside the
    graph, and every replay matches the oracle's per-token layer."""
    w = _case("tiny", T=384, H=512, E=8, K=2, I=256)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    fmt, rmap, probs = workloads.routing_inputs(w, seed=0)
    shape, layout = moe.Shape(w.T, w.H, w.E, w.K, w.I), moe.Layout(w.m, cap)
    assert moe.moe_grouped_mlp_kernel_count(shape, layout, moe.DTYPE_BF16) == 1
    map_d, probs_d = torch.from_numpy(rmap).cuda(), torch.from_numpy(probs).cuda()
    x_d = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    w13, w2 = workloads.expert_weights(w, 0, device="cuda")
    routing = moe.Routing(fmt, map_d, probs_d)
    handle = moe.Handle.empty(shape, layout)
    ws = torch.empty(moe.moe_preprocess_workspace_size(shape), dtype=torch.uint8, device="cuda")
    mlp_ws = torch.empty(moe.moe_grouped_mlp_workspace_size(shape, layout, moe.DTYPE_BF16), dtype=torch.uint8,
                         device="cuda")
    y = torch.zeros(cap, w.H, dtype=torch.bfloat16, device="cuda")
    yp = torch.zeros(cap, dtype=torch.float32, device="cuda")
    o = torch.zeros(cap, w.H, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")

    def layer(s):
        moe.moe_preprocess(routing, shape, layout, handle, ws, stream=s)
        moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16, x_d, None, routing, y, yp, stream=s)
        moe.moe_grouped_mlp(handle, shape, layout, moe.DTYPE_BF16, y, None, w13, None, w2, None, None, mlp_ws, o,
                            stream=s)
        moe.moe_combine_unpermute(handle, shape, layout, o, yp, out, stream=s)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        x_d.copy_(workloads.activations(w, 0).cuda())
        layer(s)  # eager warm-up (one-time attribute set-up happens outside the capture)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            layer(s)
    torch.cuda.synchronize()
    w13b, w2b = workloads.bf16_bits(w13), workloads.bf16_bits(w2)
    for cycle in range(3):
        fmt, rmap, probs = workloads.routing_inputs(w, seed=200 + cycle)
        x = workloads.activations(w, 200 + cycle)
        map_d.copy_(torch.from_numpy(rmap))
        probs_d.copy_(torch.from_numpy(probs))
        x_d.copy_(x.cuda())
        g.replay()
        torch.cuda.synchronize()
        assert int(handle.status.item()) == 0
        pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
        v = pre["valid_rows"]
        yo, po = oracle.dispatch(fmt, rmap, probs, pre, workloads.bf16_bits(x), cap, w.E, w.K)
        ob, _ = oracle.grouped_mlp_rows(0, yo, None, w.H, w.I, w.E, pre["offsets"], w13b, None, w2b, None,
                                        np.arange(v))
        assert rel_err(oracle.bf16_to_f64(bits(o)[:v]), oracle.bf16_to_f64(ob)) <= TOL_BF16
        ref = oracle.layer_per_token(0, fmt, rmap, probs, w.E, w.K, workloads.bf16_bits(x), None, w.H, w.I, w13b,
                                     None, w2b, None, np.arange(w.T))
        o_full = np.zeros((cap, w.H), np.uint16)
        o_full[:v] = ob
        o_rows, wts = gather_rows(oracle.bf16_to_f64(o_full), pre["row_of"], po)
        assert layer_rel_err(oracle.bf16_to_f64(bits(out)), oracle.bf16_to_f64(ref), o_rows, wts) <= TOL_BF16


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "nvfp4"])
def test_zero_token_layer(moe, dtype):
    """T = 0: all four calls run (the grouped MLP claims no tiles), the status
    word stays clear and nothing is written."""
    w = _case("tiny", T=0, H=256, E=8, K=2, I=256 if dtype == "nvfp4" else 128)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    fmt, rmap, probs = workloads.routing_inputs(w, seed=1)
    shape, layout, routing_t, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    rows = max(cap, 1)
    if dtype == "bf16":
        w13, w2 = workloads.expert_weights(w, 1, device="cuda")
        y = fill_pattern(torch.empty(rows, w.H, dtype=torch.bfloat16, device="cuda"))
        ys = None
        wd, w13_s, w2_s, in_dtype = moe.DTYPE_BF16, None, None, moe.DTYPE_BF16
        x = torch.empty(1, w.H, dtype=torch.bfloat16, device="cuda")
    elif dtype == "nvfp4":
        w13b, w2b = workloads.expert_weights(w, 1, device="cuda")
        g13 = (w13b.float().abs().amax(dim=(1, 2)) / 2688.0).contiguous()
        g2 = (w2b.float().abs().amax(dim=(1, 2)) / 2688.0).contiguous()
        w13 = torch.empty(w.E, 2 * w.I, w.H // 2, dtype=torch.uint8, device="cuda")
        w13_s = torch.empty(w.E, 2 * w.I, w.H // 16, dtype=torch.uint8, device="cuda")
        w2 = torch.empty(w.E, w.H, w.I // 2, dtype=torch.uint8, device="cuda")
        w2_s = torch.empty(w.E, w.H, w.I // 16, dtype=torch.uint8, device="cuda")
        for e in range(w.E):
            moe.moe_quantize_nvfp4_rows(w13b[e], g13[e:e + 1], w13[e], w13_s[e])
            moe.moe_quantize_nvfp4_rows(w2b[e], g2[e:e + 1], w2[e], w2_s[e])
        one = torch.ones(1, dtype=torch.float32, device="cuda")
        glob = moe.Nvfp4Globals(one, one, g13, g2)
        y = fill_pattern(torch.empty(rows, w.H // 2, dtype=torch.uint8, device="cuda"))
        ys = torch.empty(rows, w.H // 16, dtype=torch.uint8, device="cuda")
        wd, in_dtype = moe.DTYPE_NVFP4, moe.DTYPE_BF16_TO_NVFP4
        x = torch.empty(1, w.H, dtype=torch.bfloat16, device="cuda")
    else:
        w13b, w2b = workloads.expert_weights(w, 1, device="cuda")
        w13 = torch.empty(w13b.shape, dtype=torch.uint8, device="cuda")
        w2 = torch.empty(w2b.shape, dtype=torch.uint8, device="cuda")
        w13_s = torch.empty(w.E, 2 * w.I // 128, w.H // 128, dtype=torch.float32, device="cuda")
        w2_s = torch.empty(w.E, w.H // 128, w.I // 128, dtype=torch.float32, device="cuda")
        moe.moe_quantize_fp8_blocks(w13b, w13, w13_s)
        moe.moe_quantize_fp8_blocks(w2b, w2, w2_s)
        y = fill_pattern(torch.empty(rows, w.H, dtype=torch.uint8, device="cuda"))
        ys = torch.empty(rows, w.H // 128, dtype=torch.float32, device="cuda")
        wd, in_dtype = moe.DTYPE_FP8_E4M3_B128, moe.DTYPE_BF16_TO_FP8
        x = torch.empty(1, w.H, dtype=torch.bfloat16, device="cuda")
    yp = torch.empty(rows, dtype=torch.float32, device="cuda")
    moe.moe_dispatch_permute(handle, shape, layout, in_dtype, x, one if dtype == "nvfp4" else None, routing_t, y,
                             yp, ys)
    ws = torch.empty(max(moe.moe_grouped_mlp_workspace_size(shape, layout, wd), 256), dtype=torch.uint8,
                     device="cuda")
    o = fill_pattern(torch.empty(rows, w.H, dtype=torch.bfloat16, device="cuda"))
    before = bits(o).copy()
    moe.moe_grouped_mlp(handle, shape, layout, wd, y, ys, w13, w13_s, w2, w2_s, glob if dtype == "nvfp4" else None,
                        ws, o)
    out = fill_pattern(torch.empty(1, w.H, dtype=torch.bfloat16, device="cuda"))
    moe.moe_combine_unpermute(handle, shape, layout, o, yp, out)
    torch.cuda.synchronize()
    assert int(handle.status.item()) == 0
    assert int(handle.total_rows.item()) == 0
    # every expert segment is empty, so no expert row is written
    assert np.array_equal(bits(o), before)
