"""Helpers shared by the GPU parity tests: run the library on seeded inputs and
read its device outputs back as numpy arrays for comparison with the oracle."""
import numpy as np
import torch

import workloads


def moe_mod():
    import __graft_entry__

    __graft_entry__.build_library()
    import permute_grouped_expert_gb300 as moe

    return moe


def fill_pattern(t: torch.Tensor) -> torch.Tensor:
    """Pre-fill an output with 0xFF bytes so untouched rows are recognisable."""
    t.view(torch.uint8).fill_(0xFF)
    return t


def preprocess(moe, w, fmt, rmap, probs, cap, dev="cuda"):
    shape = moe.Shape(w.T, w.H, w.E, w.K, w.I)
    layout = moe.Layout(w.m, cap)
    routing = moe.Routing(fmt, torch.from_numpy(np.ascontiguousarray(rmap)).to(dev),
                          None if probs is None else torch.from_numpy(probs).to(dev))
    handle = moe.Handle.empty(shape, layout, dev)
    for f in ("row_of", "token_of", "slot_of"):
        getattr(handle, f).fill_(-7)
    ws = torch.empty(moe.moe_preprocess_workspace_size(shape), dtype=torch.uint8, device=dev)
    moe.moe_preprocess(routing, shape, layout, handle, ws)
    return shape, layout, routing, handle, ws


def handle_np(handle, T, K, cap):
    torch.cuda.synchronize()
    total = int(handle.total_rows.item())
    valid = min(total, cap)
    return dict(counts=handle.tokens_per_expert.cpu().numpy(), offsets=handle.padded_offsets.cpu().numpy(),
                row_of=handle.row_of.cpu().numpy()[:T * K].reshape(T, K),
                token_of=handle.token_of.cpu().numpy()[:valid], slot_of=handle.slot_of.cpu().numpy()[:valid],
                total_rows=total, overflow=int(handle.overflow.item()), status=int(handle.status.item()),
                valid_rows=valid)


def assert_handle_equal(got, ref):
    for key in ("counts", "offsets", "row_of", "token_of", "slot_of"):
        assert np.array_equal(got[key], ref[key]), key
    for key in ("total_rows", "overflow", "status"):
        assert got[key] == ref[key], (key, got[key], ref[key])


def bits(t: torch.Tensor) -> np.ndarray:
    return workloads.bf16_bits(t.cpu())


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at each value (8 significant bits; subnormal floor 2^-133)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """Tolerance measure for bf16 outputs against the oracle's bf16 outputs:
    max over elements of (|got - ref| - ulp_bf16(ref)), clamped at 0, divided by
    rms(ref).  Both sides round their own result to bf16, so two correct results
    can differ by one bf16 step at any element; the 1e-2 (bf16) / 5e-2 (FP8,
    NVFP4) budget applies beyond that step."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(np.square(ref))))
    excess = float(np.maximum(np.abs(got - ref) - bf16_ulp(ref), 0.0).max())
    return excess / rms if rms > 0 else excess


def layer_rel_err(got_y, ref_y, ref_o_rows, weights) -> float:
    """Tolerance measure for the layer output y = bf16(sum_k w_k * O_k): beyond
    one bf16 step of y itself, each stored expert row O_k may differ by one
    bf16 step of its own, which the combine carries with weight |w_k|.
    ref_o_rows: [T, K, H] oracle expert rows (float64, 0 for dropped routes);
    weights: [T, K] combine weights (0 for dropped routes)."""
    got_y = np.asarray(got_y, np.float64)
    ref_y = np.asarray(ref_y, np.float64)
    if ref_y.size == 0:
        return 0.0
    carried = np.einsum("tk,tkh->th", np.abs(weights), bf16_ulp(ref_o_rows) * (ref_o_rows != 0))
    rms = float(np.sqrt(np.mean(np.square(ref_y))))
    excess = float(np.maximum(np.abs(got_y - ref_y) - bf16_ulp(ref_y) - carried, 0.0).max())
    return excess / rms if rms > 0 else excess


def gather_rows(o_full, row_of, perm_probs):
    """Oracle expert rows and combine weights per (token, slot) for layer_rel_err."""
    ro = np.asarray(row_of)
    keep = ro >= 0
    rows = np.where(keep, ro, 0)
    o = np.asarray(o_full, np.float64)[rows] * keep[..., None]
    wts = (np.asarray(perm_probs, np.float64)[rows] if perm_probs is not None else np.ones(ro.shape)) * keep
    return o, wts


def mismatch_fraction(got: np.ndarray, ref: np.ndarray) -> float:
    """Fraction of elements that are not bit-identical."""
    return float(np.mean(np.asarray(got) != np.asarray(ref))) if np.asarray(ref).size else 0.0


def expert_of_rows(offsets, rows):
    """Expert owning each permuted row (offsets[e] <= row < offsets[e+1])."""
    return np.searchsorted(np.asarray(offsets), np.asarray(rows), side="right") - 1


def segment_edge_rows(pre, cap):
    """First and last valid (routed) row of every non-empty expert segment below the capacity."""
    off, cnt = pre["offsets"], pre["counts"]
    rows = []
    for e in range(len(cnt)):
        if cnt[e] == 0 or off[e] >= cap:
            continue
        last = min(off[e] + cnt[e], cap) - 1
        rows += [off[e], last]
    return np.unique(np.array(rows, np.int64))


def largest_expert_rows(pre, cap, n):
    """n rows spread evenly over the largest expert's valid rows (all its token tiles)."""
    e = int(np.argmax(pre["counts"]))
    beg, end = int(pre["offsets"][e]), int(min(pre["offsets"][e] + pre["counts"][e], cap))
    return np.unique(np.linspace(beg, end - 1, n).astype(np.int64)), e


def oracle_rows_chunked(oracle, fmt, yq, ys, pre, rows, H, I, expert_weights, chunk=16, perm_probs=None, **globs):
    """Oracle FFN of the given permuted rows, a chunk of experts at a time so
    that only that chunk's oracle-format weights are in host memory.
    expert_weights(experts) -> (w13, w13_scales, w2, w2_scales, g13, g2) for
    those experts in the oracle's format (g13 / g2 None except NVFP4).
    perm_probs ([cap], optional): probabilities applied to the FC2 rows inside
    the MLP.  Returns (rows in evaluation order, bf16 outputs [n, H])."""
    rows = np.unique(np.asarray(rows, np.int64))
    owner = expert_of_rows(pre["offsets"], rows)
    experts = sorted(set(owner.tolist()))
    sel_all, out_all = [], []
    for i in range(0, len(experts), chunk):
        ex = experts[i:i + chunk]
        q13, s13, q2, s2, g13, g2 = expert_weights(ex)
        sel, off = [], [0]
        for e in ex:
            rr = rows[owner == e]
            sel.append(rr)
            off.append(off[-1] + len(rr))
        sel = np.concatenate(sel)
        extra = dict(globs)
        if g13 is not None:
            extra.update(w13_global=g13, w2_global=g2)
        if perm_probs is not None:
            extra["row_probs"] = np.asarray(perm_probs, np.float32)[sel]
        ob, _ = oracle.grouped_mlp_rows(fmt, yq[sel], None if ys is None else ys[sel], H, I, len(ex),
                                        np.array(off, np.int32), q13, s13, q2, s2, np.arange(len(sel)), **extra)
        sel_all.append(sel)
        out_all.append(ob)
    return np.concatenate(sel_all), np.concatenate(out_all)
