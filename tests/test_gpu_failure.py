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
    moe.moe_debug_preprocess_silent_tile(routing, shape, layout, handle, ws, silent_tile=0)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    status = int(handle.status.item())
    assert status & moe.DEV_ERR_TIMEOUT, status
    assert elapsed < 30.0
    # the context is intact: an ordinary call right after is bit-exact
    moe.moe_preprocess(routing, shape, layout, handle, ws)
    ref = oracle.preprocess(fmt, rmap, w.T, w.E, w.K, w.m, cap)
    assert_handle_equal(handle_np(handle, w.T, w.K, cap), ref)
