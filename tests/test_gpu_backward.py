"""GPU parity of the backward of combine and of dispatch against the CPU oracle:
gradient rows within one bf16 step of the oracle's (each side rounds its own
fp32 / exact product or sum once), probability gradients of the combine within
the fp32 accumulation bound of their dot products, gathered probability
gradients bit for bit; pad rows zero and rows past the valid region untouched."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import bf16_ulp, bits, fill_pattern, moe_mod, preprocess

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return moe_mod()


def _bf16(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)


def _within_one_step(oracle, got_bits, ref_bits):
    got, ref = oracle.bf16_to_f64(got_bits), oracle.bf16_to_f64(ref_bits)
    return bool(np.all(np.abs(got - ref) <= bf16_ulp(ref)))


def _setup(oracle, moe, w, seed, routing=None, cap_frac=None):
    fmt, rmap, probs = workloads.routing_inputs(w, seed, routing)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    if cap_frac is not None:
        cap = int(oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)["total_rows"] * cap_frac)
    shape, layout, routing_t, handle, _ = preprocess(moe, w, fmt, rmap, probs, cap)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    _, yp = oracle.dispatch(fmt, rmap, probs, pre, np.zeros((w.T, 1), np.uint8), cap, w.E, w.K)
    return fmt, rmap, probs, cap, shape, layout, handle, pre, yp


CASES = [
    ("dense", workloads.scaled(workloads.WORKLOADS["permute"], T=500, H=384, E=12, K=4), "dense", None),
    ("sparse", workloads.scaled(workloads.WORKLOADS["mid"], T=333, H=256, E=16, K=3), "sparse", None),
    ("dense_overflow", workloads.scaled(workloads.WORKLOADS["permute"], T=400, H=256, E=8, K=3), "dense", 0.5),
    ("sparse_overflow", workloads.scaled(workloads.WORKLOADS["mid"], T=300, H=128, E=10, K=4), "sparse", 0.6),
    ("zero_tokens", workloads.scaled(workloads.WORKLOADS["permute"], T=0, H=128, E=4, K=2), "dense", None),
    # hidden sizes at and past the token-per-warp kernels' register rows (1024, 2048) and the route-per-warp
    # kernel beyond; top-36 takes the token kernel through a second 32-route pass
    ("h1024_top36", workloads.scaled(workloads.WORKLOADS["stress"], T=200, H=1024, E=64, K=36), "dense", None),
    ("h1152_sparse", workloads.scaled(workloads.WORKLOADS["mid"], T=257, H=1152, E=16, K=4), "sparse", None),
    ("h2048_overflow", workloads.scaled(workloads.WORKLOADS["mid"], T=300, H=2048, E=16, K=8), "sparse", 0.7),
    ("h2176", workloads.scaled(workloads.WORKLOADS["permute"], T=130, H=2176, E=8, K=3), "dense", None),
    # the largest top-k the API takes: four 32-route passes of the token kernel
    ("h256_top128", workloads.scaled(workloads.WORKLOADS["stress"], T=150, H=256, E=256, K=128), "dense", None),
]


@pytest.mark.parametrize("name,w,routing,cap_frac", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("with_probs", [True, False])
def test_combine_backward(oracle, moe, name, w, routing, cap_frac, with_probs):
    fmt, rmap, probs, cap, shape, layout, handle, pre, yp = _setup(oracle, moe, w, 17, routing, cap_frac)
    rng = np.random.default_rng(3)
    o = _bf16(rng, (max(cap, 1), w.H))
    gy = _bf16(rng, (max(w.T, 1), w.H))
    pp = torch.from_numpy(yp if yp is not None else np.zeros(max(cap, 1), np.float32)).cuda()
    g_o = fill_pattern(torch.empty(max(cap, 1), w.H, dtype=torch.bfloat16, device="cuda"))
    g_w = fill_pattern(torch.empty(max(cap, 1), dtype=torch.float32, device="cuda"))
    moe.moe_combine_backward(handle, shape, layout, gy.cuda(), o.cuda(), pp if with_probs else None, g_o,
                             g_w if with_probs else None)
    torch.cuda.synchronize()
    ref_o, ref_w = oracle.combine_backward(bits(gy)[:w.T], pre, cap, o=bits(o)[:cap],
                                           perm_probs=yp if with_probs else None)
    v = pre["valid_rows"]
    got_o = bits(g_o)
    assert _within_one_step(oracle, got_o[:v], ref_o[:v])
    assert np.all(got_o[v:cap] == 0xFFFF)  # rows past the valid region untouched
    if with_probs:
        gw = g_w.cpu().numpy()
        # fp32 accumulation of H products: bound each row by 2^-24 * H/4 * sum_h |gy * o|
        l1 = np.zeros(cap)
        ro = pre["row_of"]
        gyd, od = oracle.bf16_to_f64(bits(gy)), oracle.bf16_to_f64(bits(o))
        for t, k in zip(*np.nonzero(ro >= 0)):
            l1[ro[t, k]] = np.abs(gyd[t] * od[ro[t, k]]).sum()
        assert np.all(np.abs(gw[:v] - ref_w[:v]) <= l1[:v] * 2.0 ** -24 * w.H / 4 + 1e-30)
        assert np.all(gw[v:cap].view(np.uint32) == 0xFFFFFFFF)
        for e in range(w.E):
            for r in range(pre["offsets"][e] + pre["counts"][e], min(pre["offsets"][e + 1], cap)):
                assert gw[r] == 0.0 and not got_o[r].any()


@pytest.mark.parametrize("name,w,routing,cap_frac", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("with_probs", [True, False])
def test_dispatch_backward(oracle, moe, name, w, routing, cap_frac, with_probs):
    fmt, rmap, probs, cap, shape, layout, handle, pre, yp = _setup(oracle, moe, w, 23, routing, cap_frac)
    rng = np.random.default_rng(5)
    g_y = _bf16(rng, (max(cap, 1), w.H))
    g_yp = rng.standard_normal(max(cap, 1)).astype(np.float32)
    g_x = fill_pattern(torch.empty(max(w.T, 1), w.H, dtype=torch.bfloat16, device="cuda"))
    g_p = fill_pattern(torch.empty(max(w.T, 1), w.K if fmt == 0 else w.E, dtype=torch.float32, device="cuda"))
    moe.moe_dispatch_backward(handle, shape, layout, fmt, g_y.cuda(),
                              torch.from_numpy(g_yp).cuda() if with_probs else None, g_x,
                              g_p if with_probs else None)
    torch.cuda.synchronize()
    ref_x, ref_p = oracle.dispatch_backward(fmt, rmap, pre["row_of"], w.E, bits(g_y)[:cap],
                                            g_yp[:cap] if with_probs else None)
    assert _within_one_step(oracle, bits(g_x)[:w.T], ref_x)
    if with_probs:
        assert np.array_equal(g_p.cpu().numpy()[:w.T], ref_p)


@pytest.mark.parametrize("routing", ["dense", "sparse"])
def test_backward_full_size(oracle, moe, routing):
    """8192 tokens, hidden 7168, 32 experts, top-8 (the dispatch/combine shape),
    capacity 1.5x: both backward calls against the oracle on every row."""
    w = workloads.WORKLOADS["permute"]
    fmt, rmap, probs, cap, shape, layout, handle, pre, yp = _setup(oracle, moe, w, 0, routing, 1.5)
    rng = np.random.default_rng(8)
    o = _bf16(rng, (cap, w.H))
    gy = _bf16(rng, (w.T, w.H))
    g_o = fill_pattern(torch.empty(cap, w.H, dtype=torch.bfloat16, device="cuda"))
    g_w = torch.empty(cap, dtype=torch.float32, device="cuda")
    moe.moe_combine_backward(handle, shape, layout, gy.cuda(), o.cuda(), torch.from_numpy(yp).cuda(), g_o, g_w)
    g_yr = _bf16(rng, (cap, w.H))
    g_ypr = rng.standard_normal(cap).astype(np.float32)
    g_x = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    g_p = torch.empty(w.T, w.K if fmt == 0 else w.E, dtype=torch.float32, device="cuda")
    moe.moe_dispatch_backward(handle, shape, layout, fmt, g_yr.cuda(), torch.from_numpy(g_ypr).cuda(), g_x, g_p)
    torch.cuda.synchronize()
    ref_o, ref_w = oracle.combine_backward(bits(gy), pre, cap, o=bits(o), perm_probs=yp)
    v = pre["valid_rows"]
    got_o = bits(g_o)
    assert _within_one_step(oracle, got_o[:v], ref_o[:v])
    gw = g_w.cpu().numpy()[:v]
    scale = np.abs(ref_w[:v]).max()
    assert np.abs(gw - ref_w[:v]).max() <= 1e-4 * scale
    ref_x, ref_p = oracle.dispatch_backward(fmt, rmap, pre["row_of"], w.E, bits(g_yr), g_ypr)
    assert _within_one_step(oracle, bits(g_x), ref_x)
    assert np.array_equal(g_p.cpu().numpy(), ref_p)
