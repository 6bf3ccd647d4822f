"""Failure detection on the GPU without a GPU fault: a preprocessing tile that
never publishes its lookback words makes every later tile's bounded wait run
out; the kernel records MOE_DEV_ERR_TIMEOUT in the device status word and
returns, and the next ordinary call on the same context is correct."""
import time

import numpy as np
import pytest
import torch

import workloads
from gpu_util import assert_handle_equal, handle_np, moe_mod, preprocess

pytestmark = pytest.mark.gpu


def test_bounded_lookback_wait_reports_timeout_and_context_survives(oracle):
    moe = moe_mod()
    w = workloads.scaled(workloads.WORKLOADS["permute"], T=2048, H=128)
    fmt, rmap, probs = workloads.routing_inputs(w, seed=9)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    shape, layout, routing, handle, ws = preprocess(moe, w, fmt, rmap, probs, cap)
    torch.cuda.synchronize()
    t0 = time.time()
    # a tile after the first stays silent: its own lookback completes, and every later
    # tile's wait runs out (tile 0 would publish the chain's first inclusive prefix)
    moe.moe_debug_preprocess_silent_tile(routing, shape, layout, handle, ws, silent_tile=1)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    status = int(handle.status.item())
    assert status & moe.DEV_ERR_TIMEOUT, status
    assert elapsed < 30.0
    # the context is intact: an ordinary call right after is bit-exact
    moe.moe_preprocess(routing, shape, layout, handle, ws)
    ref = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    assert_handle_equal(handle_np(handle, w.T, w.K, cap), ref)


def test_fused_mlp_bounded_wait_reports_timeout_and_context_survives(oracle):
    """The fused bf16 grouped MLP: FC1 tiles of token tile 0 withhold their
    completion publication (testing hook), so the FC2 tiles waiting on them give
    up after their bounded wait; the status word reports the timeout, the kernel
    returns, and the next ordinary layer on the same context matches the oracle."""
    from gpu_util import bits, rel_err

    moe = moe_mod()
    w = workloads.scaled(workloads.WORKLOADS["tiny"], T=512, H=256, E=4, K=2, I=256)
    fmt, rmap, probs = workloads.routing_inputs(w, seed=13)
    cap = workloads.unbounded_capacity(w.T, w.K, w.E, w.m)
    x = workloads.activations(w, 13)
    w13, w2 = workloads.expert_weights(w, 13, device="cuda")
    shape, layout, routing, handle, ws = preprocess(moe, w, fmt, rmap, probs, cap)
    assert moe.moe_grouped_mlp_kernel_count(shape, layout, moe.DTYPE_BF16) == 1
    y = torch.zeros(cap, w.H, dtype=torch.bfloat16, device="cuda")
    yp = torch.zeros(cap, dtype=torch.float32, device="cuda")
    mlp_ws = torch.empty(moe.moe_grouped_mlp_workspace_size(shape, layout, moe.DTYPE_BF16), dtype=torch.uint8,
                         device="cuda")
    o = torch.zeros(cap, w.H, dtype=torch.bfloat16, device="cuda")

    def layer(silent):
        moe.moe_preprocess(routing, shape, layout, handle, ws)
        moe.moe_dispatch_permute(handle, shape, layout, moe.DTYPE_BF16, x.cuda(), None, routing, y, yp)
        if silent is not None:
            moe.moe_debug_next_grouped_mlp_silent_token_tile(silent)
        moe.moe_grouped_mlp(handle, shape, layout, moe.DTYPE_BF16, y, None, w13, None, w2, None, None, mlp_ws, o)
        torch.cuda.synchronize()

    t0 = time.time()
    layer(silent=0)
    elapsed = time.time() - t0
    status = int(handle.status.item())
    assert status & moe.DEV_ERR_TIMEOUT, status
    assert elapsed < 30.0
    # the context is intact: an ordinary layer right after matches the oracle
    layer(silent=None)
    assert int(handle.status.item()) == 0
    pre = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    yo, _ = oracle.dispatch(fmt, rmap, probs, pre, workloads.bf16_bits(x), cap, w.E, w.K)
    v = pre["valid_rows"]
    ob, _ = oracle.grouped_mlp_rows(0, yo, None, w.H, w.I, w.E, pre["offsets"], workloads.bf16_bits(w13), None,
                                    workloads.bf16_bits(w2), None, np.arange(v))
    assert rel_err(oracle.bf16_to_f64(bits(o)[:v]), oracle.bf16_to_f64(ob)) <= 1e-2
