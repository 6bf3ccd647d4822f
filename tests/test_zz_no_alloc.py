"""moe_preprocess_noalloc: the preprocess entry point for callers that cannot
allocate device memory (a plugin whose host application owns all device
memory, a loop that must not call cudaMalloc).  Its results must equal the
ordinary entry point's, on consecutive calls that share the library's fixed
scratch array.  This file sorts last so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_util import handle_np, moe_mod

pytestmark = pytest.mark.gpu


def _run(moe, fn, w, fmt, rmap, probs, cap):
    shape = moe.Shape(w.T, w.H, w.E, w.K, w.I)
    layout = moe.Layout(w.m, cap)
    routing = moe.Routing(fmt, torch.from_numpy(np.ascontiguousarray(rmap)).cuda(), torch.from_numpy(probs).cuda())
    handle = moe.Handle.empty(shape, layout)
    for f in ("row_of", "token_of", "slot_of"):
        getattr(handle, f).fill_(-7)
    if fn == "noalloc":
        # straight through the C ABI
        rc = moe.library().moe_preprocess_noalloc(ctypes.byref(routing.c()), ctypes.byref(shape.c()),
                                                  ctypes.byref(layout.c()), ctypes.byref(handle.c()),
                                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == moe.MOE_OK, rc
    else:
        ws = torch.empty(moe.moe_preprocess_workspace_size(shape), dtype=torch.uint8, device="cuda")
        moe.moe_preprocess(routing, shape, layout, handle, ws)
    torch.cuda.synchronize()
    return handle_np(handle, w.T, w.K, cap)


@pytest.mark.parametrize("case", ["dense_tight_capacity", "sparse_k36"])
def test_noalloc_matches_workspace_entry_point_twice(case):
    moe = moe_mod()
    if case == "dense_tight_capacity":
        w = workloads.scaled(workloads.WORKLOADS["permute"], T=4096)
        seeds = (1, 2)
    else:
        w = workloads.scaled(workloads.WORKLOADS["stress"], T=8192)
        seeds = (3, 4)
    routing = "sparse" if case == "sparse_k36" else "dense"
    for seed in seeds:  # two calls in a row share the scratch array
        fmt, rmap, probs = workloads.routing_inputs(w, seed, routing)
        cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
        if case == "dense_tight_capacity":
            cap = int(_run(moe, "workspace", w, fmt, rmap, probs, cap)["total_rows"]) - 17
        ref = _run(moe, "workspace", w, fmt, rmap, probs, cap)
        got = _run(moe, "noalloc", w, fmt, rmap, probs, cap)
        for key in ("counts", "offsets", "row_of", "token_of", "slot_of"):
            assert np.array_equal(got[key], ref[key]), (case, seed, key)
        for key in ("total_rows", "overflow", "status"):
            assert got[key] == ref[key], (case, seed, key)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """Only the size rule fails here: the routing, layout and handle are valid
    device buffers of the oversized shape, so the status names the scratch."""
    moe = moe_mod()
    big = moe.Shape(T=1 << 20, H=128, E=64, K=8)   # needs about 17 MiB of scratch
    assert moe.moe_preprocess_workspace_size(big) > 8 << 20
    cap = workloads.unbounded_capacity(big.T, big.K, big.E, 32)
    layout = moe.Layout(32, cap)
    rmap = torch.zeros(big.T, big.K, dtype=torch.int16, device="cuda")
    routing = moe.Routing(moe.ROUTING_DENSE_I16, rmap)
    handle = moe.Handle.empty(big, layout)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_preprocess_noalloc(routing, big, layout, handle)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    # a malformed argument is reported as such, before the size rule
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_preprocess_noalloc(routing, big, moe.Layout(0, cap), handle)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
