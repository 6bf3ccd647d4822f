"""The seeded synthetic input recipe (input generation only, no arithmetic of
the path): routing shapes and invariants, the Zipf skew of the DeepSeek-V3-like
workload, determinism, and per-expert weight independence."""
import numpy as np
import torch

import workloads as W


def test_router_invariants_renormalised():
    w = W.scaled(W.WORKLOADS["mid"], T=300)
    idx, p = W.router(w, seed=5)
    assert idx.shape == (300, w.K) and p.shape == (300, w.K) and idx.dtype == np.int16
    assert np.all(np.diff(idx.astype(np.int64), axis=1) > 0)  # K distinct ids, ascending
    assert idx.min() >= 0 and idx.max() < w.E
    assert np.all(p > 0) and np.allclose(p.sum(axis=1), 1.0, atol=1e-5)


def test_router_top_k_of_softmax_over_all_experts():
    w = W.scaled(W.WORKLOADS["tiny"], T=200)  # probs: the top-K values of a softmax over all E
    idx, p = W.router(w, seed=3)
    assert np.all(p.sum(axis=1) < 1.0) and np.all(p > 0)
    assert np.all(np.diff(idx.astype(np.int64), axis=1) > 0)


def test_dsv3_popularity_is_zipf_skewed():
    w = W.WORKLOADS["dsv3"]
    idx, _ = W.router(w, seed=0)
    counts = np.bincount(idx.reshape(-1).astype(np.int64), minlength=w.E)
    assert counts.sum() == w.T * w.K
    assert counts.max() > 50 * np.median(counts)  # a heavy head over a long tail
    assert np.all(np.diff(np.sort(idx.astype(np.int64), axis=1), axis=1) > 0)  # sampled without replacement


def test_inputs_are_seeded():
    w = W.scaled(W.WORKLOADS["tiny"], T=64)
    a = W.routing_inputs(w, seed=11)
    b = W.routing_inputs(w, seed=11)
    c = W.routing_inputs(w, seed=12)
    assert a[0] == b[0] and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert not np.array_equal(a[1], c[1])
    assert torch.equal(W.activations(w, 11), W.activations(w, 11))
    assert not torch.equal(W.activations(w, 11), W.activations(w, 12))


def test_expert_weights_do_not_depend_on_the_other_experts():
    w = W.scaled(W.WORKLOADS["tiny"], E=6, H=128, I=64)
    w13, w2 = W.expert_weights(w, seed=2)
    s13, s2 = W.expert_weights(w, seed=2, experts=[4, 1])
    assert torch.equal(s13[0], w13[4]) and torch.equal(s13[1], w13[1])
    assert torch.equal(s2[0], w2[4]) and torch.equal(s2[1], w2[1])


def test_sparse_encoding_holds_the_same_routes():
    w = W.scaled(W.WORKLOADS["mid"], T=50)
    idx, p = W.router(w, seed=9)
    m, ps = W.to_sparse(idx, p, w.E)
    assert m.shape == (50, w.E) and m.sum() == 50 * w.K
    for t in range(50):
        assert np.array_equal(np.flatnonzero(m[t]), idx[t].astype(np.int64))
        assert np.array_equal(ps[t, idx[t].astype(np.int64)], p[t])
