"""Pins of the oracle's metadata preprocessing (counts, padded offsets, row map,
capacity / overflow) against brute force and the invariants the pages fix."""
import itertools
import os

import numpy as np
import pytest

import workloads


def brute_force(routes: np.ndarray, E: int, m: int, cap: int):
    """Independent restatement via a library stable sort of (expert, token, slot)."""
    T, K = routes.shape
    triples = [(int(routes[t, k]), t, k) for t in range(T) for k in range(K) if routes[t, k] >= 0]
    order = sorted(triples)  # textbook sort; the tuples are distinct so order is total
    counts = np.bincount([e for e, _, _ in triples], minlength=E).astype(np.int32)
    padded = -(-counts // m) * m
    offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
    row_of = -np.ones((T, K), np.int32)
    seen = np.zeros(E, np.int64)
    for e, t, k in order:
        dest = offsets[e] + seen[e]
        seen[e] += 1
        if dest < cap:
            row_of[t, k] = dest
    return counts, offsets, row_of


def dense_cases(T, E, K):
    """Every dense routing of T tokens with K distinct experts each (or a -1 slot)."""
    per_token = list(itertools.permutations(list(range(E)) + [-1], K))
    for combo in itertools.product(per_token, repeat=T):
        yield np.array(combo, np.int16).reshape(T, K)


@pytest.mark.parametrize("T,E,K,m", [(2, 3, 2, 1), (2, 3, 2, 2), (3, 2, 1, 3), (2, 4, 2, 4)])
def test_brute_force_every_dense_routing(oracle, T, E, K, m):
    n = 0
    for idx in dense_cases(T, E, K):
        cap = workloads.unbounded_capacity(T, K, E, m)
        pre = oracle.preprocess(0, idx, T, E, K, m, cap)
        counts, offsets, row_of = brute_force(idx.astype(np.int64), E, m, cap)
        assert np.array_equal(pre["counts"], counts)
        assert np.array_equal(pre["offsets"], offsets)
        assert np.array_equal(pre["row_of"], row_of)
        assert pre["overflow"] == 0 and pre["status"] == 0
        n += 1
    assert n > 10


@pytest.mark.parametrize("T,E,K,m", [(3, 3, 2, 2), (4, 2, 2, 1)])
def test_brute_force_every_capacity(oracle, T, E, K, m):
    rng = np.random.default_rng(5)
    for _ in range(30):
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int16)
        r_pad = int(brute_force(idx, E, m, 10**9)[1][-1])
        for cap in range(0, r_pad + 5):
            pre = oracle.preprocess(0, idx, T, E, K, m, cap)
            counts, offsets, row_of = brute_force(idx, E, m, cap)
            assert pre["overflow"] == int(r_pad > cap)  # flips exactly below R_pad
            assert pre["total_rows"] == r_pad            # unclamped
            assert np.array_equal(pre["counts"], counts)  # real counts, never clamped
            assert np.array_equal(pre["row_of"], row_of)
            # token_of / slot_of invert row_of on the valid region, pads are -1
            tok = -np.ones(min(cap, r_pad), np.int32)
            slot = -np.ones(min(cap, r_pad), np.int32)
            for t in range(T):
                for k in range(K):
                    if row_of[t, k] >= 0:
                        tok[row_of[t, k]] = t
                        slot[row_of[t, k]] = k
            assert np.array_equal(pre["token_of"], tok)
            assert np.array_equal(pre["slot_of"], slot)


def test_invariants_stress_shape(oracle):
    w = workloads.scaled(workloads.WORKLOADS["stress"], T=4096)
    fmt, idx, _ = workloads.routing_inputs(w, seed=0, routing="dense")
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    pre = oracle.preprocess(fmt, idx, w.T, w.E, w.K, w.m, cap)
    R = w.T * w.K
    assert pre["counts"].sum() == R                       # counts sum to tokens x topk
    assert pre["total_rows"] <= R + w.E * (w.m - 1)        # padding bound
    assert np.all(np.diff(pre["offsets"]) % w.m == 0)
    # row map: a bijection from routes onto the non-pad rows
    rows = pre["row_of"].reshape(-1)
    assert len(np.unique(rows)) == R and rows.min() >= 0
    nonpad = np.flatnonzero(pre["token_of"] >= 0)
    assert np.array_equal(np.sort(rows), nonpad)
    # stability: within each expert, source tokens ascend
    for e in range(w.E):
        seg = pre["token_of"][pre["offsets"][e]:pre["offsets"][e] + pre["counts"][e]]
        assert np.all(np.diff(seg) > 0)


def test_dense_and_sparse_encodings_agree(oracle):
    w = workloads.scaled(workloads.WORKLOADS["mid"], T=512)
    idx, p = workloads.router(w, seed=1)
    sm, sp = workloads.to_sparse(idx, p, w.E)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    a = oracle.preprocess(0, idx, w.T, w.E, w.K, w.m, cap)
    b = oracle.preprocess(1, sm, w.T, w.E, w.K, w.m, cap)
    for key in ("counts", "offsets", "row_of", "token_of", "slot_of"):
        assert np.array_equal(a[key], b[key]), key
    x = np.arange(w.T * 8, dtype=np.uint16).reshape(w.T, 8)
    ya, pa = oracle.dispatch(0, idx, p, a, x, cap, w.E, w.K)
    yb, pb = oracle.dispatch(1, sm, sp, b, x, cap, w.E, w.K)
    assert np.array_equal(ya, yb) and np.array_equal(pa, pb)


def test_capacity_modes_match_unbounded(oracle):
    """Capacity 1x / 1.5x / 2x of the actual rows: flag 0 and identical rows;
    capacity = actual / 2: flag set, rows past the capacity dropped."""
    w = workloads.scaled(workloads.WORKLOADS["permute"], T=1024, H=64)
    fmt, idx, p = workloads.routing_inputs(w, seed=2)
    big = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    ref = oracle.preprocess(fmt, idx, w.T, w.E, w.K, w.m, big)
    x = np.random.default_rng(0).integers(0, 65535, (w.T, w.H)).astype(np.uint16)
    yref, pref = oracle.dispatch(fmt, idx, p, ref, x, big, w.E, w.K)
    rows = ref["total_rows"]
    for f in (1.0, 1.5, 2.0):
        cap = oracle.capacity(rows, f)
        pre = oracle.preprocess(fmt, idx, w.T, w.E, w.K, w.m, cap)
        assert pre["overflow"] == 0
        for key in ("counts", "offsets", "row_of", "token_of", "slot_of"):
            assert np.array_equal(pre[key], ref[key])
        y, pp = oracle.dispatch(fmt, idx, p, pre, x, cap, w.E, w.K)
        assert np.array_equal(y[:rows], yref[:rows]) and np.array_equal(pp[:rows], pref[:rows])
    cap = oracle.capacity(rows // 2, 1.0)
    pre = oracle.preprocess(fmt, idx, w.T, w.E, w.K, w.m, cap)
    assert pre["overflow"] == 1
    kept = ref["row_of"] < cap
    assert np.array_equal(pre["row_of"][kept], ref["row_of"][kept])
    assert np.all(pre["row_of"][~kept] == -1)


def test_malformed_routing_is_reported(oracle):
    idx = np.array([[0, 5], [1, -1], [-3, 2]], np.int16)
    pre = oracle.preprocess(0, idx, 3, 4, 2, 1, 100)
    assert pre["status"] == oracle.ERR_BAD_EXPERT
    assert pre["counts"].tolist() == [1, 1, 1, 0]
    sm = np.array([[1, 1, 1, 0], [0, 1, 0, 0]], np.uint8)
    pre = oracle.preprocess(1, sm, 2, 4, 2, 1, 100)
    assert pre["status"] == oracle.ERR_TOO_MANY_ROUTES
    assert pre["counts"].tolist() == [1, 2, 0, 0]
    assert pre["row_of"].tolist() == [[0, 1], [2, -1]]


def test_empty_and_degenerate(oracle):
    # no tokens
    pre = oracle.preprocess(0, np.zeros((0, 2), np.int16), 0, 3, 2, 4, 0)
    assert pre["counts"].tolist() == [0, 0, 0] and pre["total_rows"] == 0 and pre["overflow"] == 0
    # one expert takes everything, K = E
    idx = np.tile(np.arange(3, dtype=np.int16), (5, 1))
    pre = oracle.preprocess(0, idx, 5, 3, 3, 32, 1000)
    assert pre["counts"].tolist() == [5, 5, 5] and pre["offsets"].tolist() == [0, 32, 64, 96]
    # capacity zero drops everything
    pre = oracle.preprocess(0, idx, 5, 3, 3, 1, 0)
    assert pre["overflow"] == 1 and np.all(pre["row_of"] == -1)


def test_routing_layout_bytes_golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "routing_bytes.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        layout, T, E, K, nbytes = line.split()
        T, E, K, nbytes = int(T), int(E), int(K), int(nbytes)
        w = workloads.scaled(workloads.WORKLOADS["stress"], T=T, E=E, K=K)
        fmt, rmap, _ = workloads.routing_inputs(w, seed=0, routing=layout)
        assert rmap.nbytes == nbytes
