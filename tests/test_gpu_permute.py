"""GPU parity of preprocess, dispatch and combine against the CPU oracle
(bit-exact for counts, offsets, row maps, flags, permuted rows, FP8 / NVFP4
codes and scales; max-abs-error / RMS <= 1e-2 for the bf16 combine)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import (assert_handle_equal, bits, fill_pattern, handle_np, mismatch_fraction, moe_mod, preprocess,
                      rel_err)

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2


@pytest.fixture(scope="module")
def moe():
    return moe_mod()


def _case(name, **kw):
    return workloads.scaled(workloads.WORKLOADS[name], **kw)


PRE_CASES = [
    ("tiny", _case("tiny"), None, None),
    ("mid_sparse", _case("mid"), None, 1.5),
    ("permute_1x", _case("permute"), None, 1.0),
    ("permute_2x", _case("permute"), None, 2.0),
    ("permute_half", _case("permute"), None, 0.5),
    ("permute_m1", _case("permute", m=1), None, 1.0),
    ("stress_dense", _case("stress"), "dense", None),
    ("stress_sparse", _case("stress"), "sparse", None),
    ("k_equals_e", _case("tiny", T=333, E=4, K=4), None, None),
    ("one_expert", _case("tiny", T=1000, E=1, K=1), None, None),
    ("max_experts", _case("stress", T=3000, E=1024, K=8), None, None),
    ("ragged_tiles", _case("stress", T=4099, K=36), "sparse", None),
    ("zero_tokens", _case("tiny", T=0), None, None),
    ("max_topk_128", _case("stress", T=300, E=256, K=128), "dense", None),
    ("max_topk_128_sparse", _case("stress", T=300, E=256, K=128), "sparse", None),
]


@pytest.mark.parametrize("name,w,routing,factor", PRE_CASES, ids=[c[0] for c in PRE_CASES])
def test_preprocess_bit_exact(oracle, moe, name, w, routing, factor):
    fmt, rmap, probs = workloads.routing_inputs(w, seed=11, routing=routing)
    if factor is None:
        cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    else:
        rows = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
        cap = oracle.capacity(rows, factor)
    ref = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    _, _, _, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    got = handle_np(handle, w.T, w.K, cap)
    assert_handle_equal(got, ref)
    if factor is not None:
        assert got["overflow"] == int(factor < 1.0)


@pytest.mark.parametrize("cap_delta", [0, -1, -100])
def test_capacity_edges(oracle, moe, cap_delta):
    w = _case("permute", T=2048, H=128)
    fmt, rmap, probs = workloads.routing_inputs(w, seed=3)
    rows = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
    cap = rows + cap_delta
    ref = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    _, _, _, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    got = handle_np(handle, w.T, w.K, cap)
    assert_handle_equal(got, ref)
    assert got["overflow"] == int(cap_delta < 0)


def test_malformed_routing_sets_status(oracle, moe):
    w = _case("tiny", T=64, E=8, K=2)
    idx = np.random.default_rng(0).integers(0, 8, (64, 2)).astype(np.int16)
    idx[3, 1] = 9
    idx[10, 0] = -5
    idx[11, 0] = -1
    cap = 1000
    ref = oracle.preprocess(0, idx, w.T, w.E, w.K, w.m, cap)
    _, _, _, handle, _ = preprocess(moe, w, 0, idx, None, cap)
    got = handle_np(handle, w.T, w.K, cap)
    assert ref["status"] == moe.DEV_ERR_BAD_EXPERT
    assert_handle_equal(got, ref)
    sm = np.zeros((40, 8), np.uint8)
    sm[:, :3] = 1
    sm[5, :] = 1
    ref = oracle.preprocess(1, sm, 40, 8, 3, w.m, cap)
    _, _, _, handle, _ = preprocess(moe, _case("tiny", T=40, E=8, K=3), 1, sm, None, cap)
    got = handle_np(handle, 40, 3, cap)
    assert ref["status"] == moe.DEV_ERR_TOO_MANY_ROUTES
    assert_handle_equal(got, ref)


def _dispatch(moe, w, fmt, rmap, probs, cap, x, in_dtype=None, x_scales=None, nvfp4_global=None):
    shape, layout, routing, handle, ws = preprocess(moe, w, fmt, rmap, probs, cap)
    dev = "cuda"
    in_dtype = moe.DTYPE_BF16 if in_dtype is None else in_dtype
    rows = max(cap, 1)
    if in_dtype == moe.DTYPE_BF16:
        out = fill_pattern(torch.empty(rows, w.H, dtype=torch.bfloat16, device=dev))
        out_s = None
    elif in_dtype in (moe.DTYPE_BF16_TO_FP8, moe.DTYPE_FP8_E4M3_B128):
        out = fill_pattern(torch.empty(rows, w.H, dtype=torch.uint8, device=dev))
        out_s = fill_pattern(torch.empty(rows, w.H // 128, dtype=torch.float32, device=dev))
    else:
        out = fill_pattern(torch.empty(rows, w.H // 2, dtype=torch.uint8, device=dev))
        out_s = fill_pattern(torch.empty(rows, w.H // 16, dtype=torch.uint8, device=dev))
    out_p = fill_pattern(torch.empty(rows, dtype=torch.float32, device=dev)) if probs is not None else None
    xs = x_scales if nvfp4_global is None else nvfp4_global
    moe.moe_dispatch_permute(handle, shape, layout, in_dtype, x, xs, routing, out, out_p, out_s)
    torch.cuda.synchronize()
    return handle, out, out_p, out_s


@pytest.mark.parametrize("name,w,routing", [
    ("tiny", _case("tiny"), None),
    ("mid_sparse", _case("mid"), None),
    ("permute", _case("permute", T=2048), None),
    ("k36_sparse", _case("stress", T=1500, H=256), "sparse"),
    ("zero_tokens", _case("tiny", T=0), None),
    ("max_topk_128", _case("stress", T=200, H=256, E=256, K=128), None),
], ids=lambda v: v if isinstance(v, str) else "")
def test_dispatch_bf16_bitwise(oracle, moe, name, w, routing):
    fmt, rmap, probs = workloads.routing_inputs(w, seed=5, routing=routing)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    x = workloads.activations(w, 5)
    handle, out, out_p, _ = _dispatch(moe, w, fmt, rmap, probs, cap, x.cuda())
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    yo, po = oracle.dispatch(fmt, rmap, probs, pre, workloads.bf16_bits(x), cap, w.E, w.K)
    v = pre["valid_rows"]
    got = bits(out)
    assert np.array_equal(got[:v], yo[:v])
    assert np.array_equal(out_p.cpu().numpy()[:v].view(np.uint32), po[:v].view(np.uint32))
    # rows past the last segment are untouched
    assert np.all(got[v:] == 0xFFFF)


@pytest.mark.parametrize("factor", [1.0, 1.5, 2.0, 0.5])
def test_dispatch_capacity_modes_match_unbounded(oracle, moe, factor):
    """Capacity 1x / 1.5x / 2x: flag 0 and rows equal to the unbounded dispatch;
    capacity 1/2x: flag 1 and only the rows below the capacity written."""
    w = _case("permute", T=2048, H=512)
    fmt, rmap, probs = workloads.routing_inputs(w, seed=8)
    rows = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
    cap = oracle.capacity(rows, factor)
    x = workloads.activations(w, 8)
    handle, out, out_p, _ = _dispatch(moe, w, fmt, rmap, probs, cap, x.cuda())
    got = handle_np(handle, w.T, w.K, cap)
    assert got["overflow"] == int(factor < 1)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    yo, po = oracle.dispatch(fmt, rmap, probs, pre, workloads.bf16_bits(x), cap, w.E, w.K)
    v = pre["valid_rows"]
    assert np.array_equal(bits(out)[:v], yo[:v])
    assert np.array_equal(out_p.cpu().numpy()[:v], po[:v])


def test_dispatch_stress_full_size_sampled(oracle, moe):
    """65536 tokens x top-36 x 256 experts, hidden 1024: 2.36 M rows (4.8 GB,
    int64 offsets).  Row maps bit-exact in full; dispatched rows checked on a
    sample of rows against the oracle's token_of."""
    w = workloads.WORKLOADS["stress"]
    for routing in ("dense", "sparse"):
        fmt, rmap, probs = workloads.routing_inputs(w, seed=1, routing=routing)
        cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
        x = workloads.activations(w, 1).cuda()
        handle, out, out_p, _ = _dispatch(moe, w, fmt, rmap, probs, cap, x)
        ref = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
        got = handle_np(handle, w.T, w.K, cap)
        assert_handle_equal(got, ref)
        rng = np.random.default_rng(0)
        rows = np.sort(rng.choice(ref["valid_rows"], 4096, replace=False))
        rows = np.concatenate([rows, [ref["valid_rows"] - 1]])
        tok = ref["token_of"][rows]
        xr = workloads.bf16_bits(x[torch.from_numpy(np.maximum(tok, 0)).cuda()])
        gr = bits(out[torch.from_numpy(rows).cuda()])
        for i, t in enumerate(tok):
            if t >= 0:
                assert np.array_equal(gr[i], xr[i])
            else:
                assert not gr[i].any()
        del out, out_p, x
        torch.cuda.empty_cache()


def test_dispatch_fp8_quantize_bit_exact(oracle, moe):
    w = _case("dsv3", T=1024, H=1024)
    fmt, rmap, probs = workloads.routing_inputs(w, seed=2)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    x = workloads.activations(w, 2)
    x[5, :128] = 0  # an all-zero block takes scale 1
    handle, out, out_p, out_s = _dispatch(moe, w, fmt, rmap, probs, cap, x.cuda(), moe.DTYPE_BF16_TO_FP8)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    q, s = oracle.quantize_fp8_rows(workloads.bf16_bits(x))
    yq, _ = oracle.dispatch(fmt, rmap, None, pre, q, cap, w.E, w.K)
    ys, _ = oracle.dispatch(fmt, rmap, None, pre, s, cap, w.E, w.K)
    v = pre["valid_rows"]
    assert np.array_equal(out.cpu().numpy()[:v], yq[:v])
    assert np.array_equal(out_s.cpu().numpy()[:v].view(np.uint32), ys[:v].view(np.uint32))
    # FP8 passthrough (codes + scales quantized beforehand) copies bit for bit
    handle2, out2, _, out2_s = _dispatch(moe, w, fmt, rmap, probs, cap, torch.from_numpy(q).cuda(),
                                         moe.DTYPE_FP8_E4M3_B128, x_scales=torch.from_numpy(s).cuda())
    assert np.array_equal(out2.cpu().numpy()[:v], yq[:v])
    assert np.array_equal(out2_s.cpu().numpy()[:v], ys[:v])


def test_dispatch_nvfp4_quantize_bit_exact(oracle, moe):
    w = _case("decode256", T=200, H=1024)
    fmt, rmap, probs = workloads.routing_inputs(w, seed=4)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    x = workloads.activations(w, 4)
    g = np.float32(np.abs(x.float().numpy()).max() / (6 * 448))
    handle, out, out_p, out_s = _dispatch(moe, w, fmt, rmap, probs, cap, x.cuda(), moe.DTYPE_BF16_TO_NVFP4,
                                          nvfp4_global=torch.tensor([g], device="cuda"))
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    packed, sc = oracle.quantize_nvfp4_rows(workloads.bf16_bits(x), float(g))
    yq, _ = oracle.dispatch(fmt, rmap, None, pre, packed, cap, w.E, w.K)
    ys, _ = oracle.dispatch(fmt, rmap, None, pre, sc, cap, w.E, w.K)
    v = pre["valid_rows"]
    assert np.array_equal(out.cpu().numpy()[:v], yq[:v])
    assert np.array_equal(out_s.cpu().numpy()[:v], ys[:v])


def test_quantize_fp8_weights_bit_exact(oracle, moe):
    rng = np.random.default_rng(9)
    wt = torch.from_numpy(rng.standard_normal((3, 256, 640)).astype(np.float32) * 0.02).to(torch.bfloat16)
    wt[1, :128, :128] = 0
    codes = torch.empty(3, 256, 640, dtype=torch.uint8, device="cuda")
    scales = torch.empty(3, 2, 5, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_blocks(wt.cuda(), codes, scales)
    q, s = oracle.quantize_fp8_weight(workloads.bf16_bits(wt))
    assert np.array_equal(codes.cpu().numpy(), q)
    assert np.array_equal(scales.cpu().numpy(), s)


def test_quantize_nvfp4_rows_bit_exact(oracle, moe):
    rng = np.random.default_rng(10)
    wt = torch.from_numpy(rng.standard_normal((77, 512)).astype(np.float32)).to(torch.bfloat16)
    g = np.float32(np.abs(wt.float().numpy()).max() / 2688)
    packed = torch.empty(77, 256, dtype=torch.uint8, device="cuda")
    sc = torch.empty(77, 32, dtype=torch.uint8, device="cuda")
    moe.moe_quantize_nvfp4_rows(wt.cuda(), torch.tensor([g], device="cuda"), packed, sc)
    p, s = oracle.quantize_nvfp4_rows(workloads.bf16_bits(wt), float(g))
    assert np.array_equal(packed.cpu().numpy(), p)
    assert np.array_equal(sc.cpu().numpy(), s)


def _combine(moe, handle, shape, layout, o, perm_probs, T, H):
    y = fill_pattern(torch.empty(max(T, 1), H, dtype=torch.bfloat16, device="cuda"))
    moe.moe_combine_unpermute(handle, shape, layout, o, perm_probs, y)
    torch.cuda.synchronize()
    return y[:T]


@pytest.mark.parametrize("name,w,routing,use_probs", [
    ("tiny", _case("tiny"), None, True),
    ("mid_sparse", _case("mid"), None, True),
    ("k36_sparse", _case("stress", T=700, H=512), "sparse", True),
    ("no_probs", _case("tiny", T=300), None, False),
    ("max_topk_128", _case("stress", T=200, H=256, E=256, K=128), None, True),
], ids=lambda v: v if isinstance(v, str) else "")
def test_combine_random_expert_rows(oracle, moe, name, w, routing, use_probs):
    fmt, rmap, probs = workloads.routing_inputs(w, seed=6, routing=routing)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    shape, layout, routing_t, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    _, po = oracle.dispatch(fmt, rmap, probs, pre, np.zeros((w.T, 1), np.uint8), cap, w.E, w.K)
    o = (torch.randn(cap, w.H, generator=torch.Generator().manual_seed(6))).to(torch.bfloat16)
    pp = torch.from_numpy(po).cuda() if use_probs else None
    y = _combine(moe, handle, shape, layout, o.cuda(), pp, w.T, w.H)
    ref = oracle.combine(workloads.bf16_bits(o), pre["row_of"], po if use_probs else None)
    assert rel_err(oracle.bf16_to_f64(bits(y)), oracle.bf16_to_f64(ref)) <= TOL_BF16
    # fp32 accumulation in ascending k: only rare one-step rounding differences
    assert mismatch_fraction(bits(y), ref) < 1e-3


@pytest.mark.parametrize("factor", [1.0, 1.5, 2.0])
def test_combine_round_trip_identity_experts(oracle, moe, factor):
    """Identity experts at the 8192 x 7168, 32-expert top-8 shape: combine(dispatch(x))
    returns x (renormalised probs) and equals the oracle within tolerance."""
    w = workloads.WORKLOADS["permute"]
    fmt, rmap, probs = workloads.routing_inputs(w, seed=12)
    rows = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
    cap = oracle.capacity(rows, factor)
    x = workloads.activations(w, 12)
    handle, out, out_p, _ = _dispatch(moe, w, fmt, rmap, probs, cap, x.cuda())
    shape, layout = moe.Shape(w.T, w.H, w.E, w.K), moe.Layout(w.m, cap)
    y = _combine(moe, handle, shape, layout, out, out_p, w.T, w.H)
    xd = oracle.bf16_to_f64(workloads.bf16_bits(x))
    assert rel_err(oracle.bf16_to_f64(bits(y)), xd) <= TOL_BF16
    # power-of-two probs make the round trip exact
    p8 = np.full_like(probs, 1.0 / 8.0)
    handle, out, out_p, _ = _dispatch(moe, w, fmt, rmap, p8, cap, x.cuda())
    y = _combine(moe, handle, shape, layout, out, out_p, w.T, w.H)
    assert np.array_equal(bits(y), workloads.bf16_bits(x))


def test_combine_under_overflow_skips_dropped(oracle, moe):
    w = _case("permute", T=1024, H=256)
    fmt, rmap, probs = workloads.routing_inputs(w, seed=13)
    rows = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, 1 << 30)["total_rows"]
    cap = oracle.capacity(rows // 4, 1.0)
    x = workloads.activations(w, 13)
    handle, out, out_p, _ = _dispatch(moe, w, fmt, rmap, probs, cap, x.cuda())
    shape, layout = moe.Shape(w.T, w.H, w.E, w.K), moe.Layout(w.m, cap)
    y = _combine(moe, handle, shape, layout, out, out_p, w.T, w.H)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    yo, po = oracle.dispatch(fmt, rmap, probs, pre, workloads.bf16_bits(x), cap, w.E, w.K)
    ref = oracle.combine(yo, pre["row_of"], po)
    assert rel_err(oracle.bf16_to_f64(bits(y)), oracle.bf16_to_f64(ref)) <= TOL_BF16
    # tokens with every route dropped come back as zeros
    dead = np.all(pre["row_of"] < 0, axis=1)
    assert dead.any() and not bits(y)[dead].any()


def test_three_cycles_in_one_cuda_graph(oracle, moe):
    """preprocess -> dispatch -> combine captured once and replayed with new
    routing and activations written into the same input buffers; every replay
    matches the oracle (dense and sparse)."""
    for routing_kind in ("dense", "sparse"):
        w = _case("tiny", T=512, H=512)
        cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
        fmt, rmap, probs = workloads.routing_inputs(w, seed=0, routing=routing_kind)
        shape, layout = moe.Shape(w.T, w.H, w.E, w.K), moe.Layout(w.m, cap)
        map_d = torch.from_numpy(rmap).cuda()
        probs_d = torch.from_numpy(probs).cuda()
        x_d = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        routing = moe.Routing(fmt, map_d, probs_d)
        handle = moe.Handle.empty(shape, layout)
        ws = torch.empty(moe.moe_preprocess_workspace_size(shape), dtype=torch.uint8, device="cuda")
        yperm = torch.zeros(cap, w.H, dtype=torch.bfloat16, device="cuda")
        pperm = torch.zeros(cap, dtype=torch.float32, device="cuda")
        out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            x_d.copy_(workloads.activations(w, 0).cuda())
            moe.moe_preprocess(routing, shape, layout, handle, ws, stream=s)  # eager warm-up
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                moe.moe_preprocess(routing, shape, layout, handle, ws, stream=s)
                moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16, x_d, None, routing, yperm, pperm,
                                         stream=s)
                moe.moe_combine_unpermute(handle, shape, layout, yperm, pperm, out, stream=s)
        torch.cuda.synchronize()
        for cycle in range(3):
            fmt, rmap, probs = workloads.routing_inputs(w, seed=100 + cycle, routing=routing_kind)
            x = workloads.activations(w, 100 + cycle)
            map_d.copy_(torch.from_numpy(rmap))
            probs_d.copy_(torch.from_numpy(probs))
            x_d.copy_(x.cuda())
            g.replay()
            torch.cuda.synchronize()
            ref = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
            assert_handle_equal(handle_np(handle, w.T, w.K, cap), ref)
            yo, po = oracle.dispatch(fmt, rmap, probs, ref, workloads.bf16_bits(x), cap, w.E, w.K)
            v = ref["valid_rows"]
            assert np.array_equal(bits(yperm)[:v], yo[:v])
            yref = oracle.combine(yo, ref["row_of"], po)
            assert rel_err(oracle.bf16_to_f64(bits(out)), oracle.bf16_to_f64(yref)) <= TOL_BF16


def test_ring_with_stream_events(moe):
    r = moe.Ring(2, use_events=True)
    s = torch.cuda.Stream()
    a = r.acquire(s)
    b = r.acquire(s)
    r.release(a, s)
    assert r.acquire(s) == a
    r.release(b, s)
    r.release(a, s)
    torch.cuda.synchronize()
    r.close()
