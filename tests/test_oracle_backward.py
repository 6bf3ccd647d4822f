"""Pins of the oracle's backward of combine and of dispatch against torch
autograd (a library routine) through an independently written float64 forward
of the same two steps, and against special cases: with one route per token and
no probabilities the dispatch backward is the inverse permutation; dropped
routes and pad rows carry no gradient."""
import numpy as np
import pytest
import torch

import workloads


def _bits(t):
    return workloads.bf16_bits(t)


def _routes(fmt, rmap, T, E, K):
    """Expert of every slot (t, k) straight from the routing map, -1 for none."""
    if fmt == 0:
        return np.asarray(rmap, np.int64).reshape(T, K)
    out = np.full((T, K), -1, np.int64)
    for t in range(T):
        ex = np.nonzero(np.asarray(rmap)[t])[0][:K]
        out[t, :len(ex)] = ex
    return out


def _case(oracle, name, T, H, E, K, seed, routing=None, cap_frac=None):
    w = workloads.scaled(workloads.WORKLOADS[name], T=T, H=H, E=E, K=K)
    fmt, rmap, p = workloads.routing_inputs(w, seed, routing)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    if cap_frac is not None:
        full = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
        cap = int(full["total_rows"] * cap_frac)
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    return w, fmt, rmap, p, cap, pre


def _bf16(rng, shape, scale=1.0):
    return torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("routing,cap_frac", [("dense", None), ("sparse", None), ("dense", 0.5), ("sparse", 0.6)])
def test_combine_backward_matches_autograd(oracle, routing, cap_frac):
    w, fmt, rmap, p, cap, pre = _case(oracle, "mid", T=96, H=128, E=8, K=3, seed=5, routing=routing,
                                      cap_frac=cap_frac)
    rng = np.random.default_rng(1)
    o = _bf16(rng, (cap, w.H))
    gy = _bf16(rng, (w.T, w.H))
    _, yp = oracle.dispatch(fmt, rmap, p, pre, np.zeros((w.T, 1), np.uint8), cap, w.E, w.K)
    g_o, g_w = oracle.combine_backward(_bits(gy), pre, cap, o=_bits(o), perm_probs=yp)

    # float64 forward of the combine, written with torch indexing, differentiated by autograd
    ro = torch.from_numpy(pre["row_of"].astype(np.int64))
    keep = ro >= 0
    O = o.double().requires_grad_(True)
    W = torch.from_numpy(yp.astype(np.float64)).requires_grad_(True)
    rows = torch.where(keep, ro, torch.zeros_like(ro))
    y = (O[rows] * (W[rows] * keep)[..., None]).sum(1)
    (y * gy.double()).sum().backward()
    v = pre["valid_rows"]
    exact_go, exact_gw = O.grad.numpy()[:v], W.grad.numpy()[:v]
    got_go = oracle.bf16_to_f64(g_o[:v])
    # gO is the exact product rounded once to bf16: within half a bf16 step
    ulp = np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(exact_go), 2.0 ** -126))) - 7).astype(np.int64))
    assert np.all(np.abs(got_go - exact_go) <= ulp / 2)
    # gw is the dot product rounded to fp32
    assert np.all(np.abs(g_w[:v] - exact_gw) <= np.abs(exact_gw) * 2.0 ** -23 + 1e-30)
    assert np.abs(exact_gw).max() > 0
    # pad rows carry no gradient; dropped routes have no row at all
    for e in range(w.E):
        for r in range(pre["offsets"][e] + pre["counts"][e], min(pre["offsets"][e + 1], cap)):
            assert not g_o[r].any() and g_w[r] == 0.0
    if cap_frac is not None:
        assert (pre["row_of"] < 0).any()


@pytest.mark.parametrize("routing,cap_frac", [("dense", None), ("sparse", None), ("dense", 0.5), ("sparse", 0.6)])
def test_dispatch_backward_matches_autograd(oracle, routing, cap_frac):
    w, fmt, rmap, p, cap, pre = _case(oracle, "mid", T=80, H=128, E=8, K=3, seed=9, routing=routing,
                                      cap_frac=cap_frac)
    rng = np.random.default_rng(2)
    g_y = _bf16(rng, (cap, w.H))
    g_yp = rng.standard_normal(cap).astype(np.float32)
    g_x, g_p = oracle.dispatch_backward(fmt, rmap, pre["row_of"], w.E, _bits(g_y), g_yp)

    # float64 forward of the dispatch: Y[r] = x[t], Yp[r] = p(t, expert of slot k)
    ex = _routes(fmt, rmap, w.T, w.E, w.K)
    X = torch.zeros(w.T, w.H, dtype=torch.float64, requires_grad=True)
    P = torch.from_numpy(np.asarray(p, np.float64)).requires_grad_(True)
    loss = 0.0
    for t in range(w.T):
        for k in range(w.K):
            r = pre["row_of"][t, k]
            if r < 0:
                continue
            pv = P[t, k] if fmt == 0 else P[t, ex[t, k]]
            loss = loss + (X[t] * g_y[r].double()).sum() + pv * float(g_yp[r])
    loss.backward()
    exact_gx = X.grad.numpy()
    ulp = np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(exact_gx), 2.0 ** -126))) - 7).astype(np.int64))
    assert np.all(np.abs(oracle.bf16_to_f64(g_x) - exact_gx) <= ulp / 2)
    assert np.array_equal(g_p, P.grad.numpy().astype(np.float32))
    if cap_frac is not None:
        dropped = pre["row_of"] < 0
        assert dropped.any()
        if fmt == 0:
            assert not g_p[dropped].any()


def test_dispatch_backward_k1_without_probs_is_inverse_permutation(oracle):
    w, fmt, rmap, p, cap, pre = _case(oracle, "permute", T=150, H=64, E=6, K=1, seed=3)
    g_y = _bits(_bf16(np.random.default_rng(4), (cap, w.H)))
    g_x, g_p = oracle.dispatch_backward(fmt, rmap, pre["row_of"], w.E, g_y)
    assert g_p is None
    assert np.array_equal(g_x, g_y[pre["row_of"][:, 0]])


def test_combine_backward_without_probs_k1_is_the_dispatch(oracle):
    """Weight 1 and one route per token: the combine's backward dispatches gy."""
    w, fmt, rmap, p, cap, pre = _case(oracle, "permute", T=150, H=64, E=6, K=1, seed=6)
    gy = _bits(_bf16(np.random.default_rng(7), (w.T, w.H)))
    g_o, g_w = oracle.combine_backward(gy, pre, cap)
    y, _ = oracle.dispatch(fmt, rmap, None, pre, gy, cap, w.E, w.K)
    assert g_w is None
    assert np.array_equal(g_o, y)
