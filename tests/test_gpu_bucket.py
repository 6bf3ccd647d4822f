"""Decode buckets: a CUDA graph of the whole layer captured once at a bucket's
token count and replayed for smaller batches padded with "no route" tokens
gives every real token exactly the output of the unpadded batch, and the
padding tokens zero rows (bf16 and NVFP4 layers)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import bits, moe_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return moe_mod()


class Layer:
    """The four calls at a fixed token count T (buffers sized for T), bf16 or NVFP4."""

    def __init__(self, moe, w, T, weights, fc2_global):
        self.moe, self.w, self.T = moe, w, T
        self.shape = moe.Shape(T, w.H, w.E, w.K, w.I)
        self.cap = workloads.unbounded_capacity(T, w.K, w.E, w.m)
        self.layout = moe.Layout(w.m, self.cap)
        self.map = torch.full((T, w.K), -1, dtype=torch.int16, device="cuda")
        self.probs = torch.zeros(T, w.K, dtype=torch.float32, device="cuda")
        self.x = torch.zeros(T, w.H, dtype=torch.bfloat16, device="cuda")
        self.routing = moe.Routing(moe.ROUTING_DENSE_I16, self.map, self.probs)
        self.handle = moe.Handle.empty(self.shape, self.layout)
        self.ws = torch.empty(moe.moe_preprocess_workspace_size(self.shape), dtype=torch.uint8, device="cuda")
        self.nvfp4 = w.dtype == "nvfp4"
        if self.nvfp4:
            self.y = torch.empty(self.cap, w.H // 2, dtype=torch.uint8, device="cuda")
            self.ys = torch.empty(self.cap, w.H // 16, dtype=torch.uint8, device="cuda")
            self.in_dtype, self.w_dtype = moe.DTYPE_BF16_TO_NVFP4, moe.DTYPE_NVFP4
        else:
            self.y = torch.empty(self.cap, w.H, dtype=torch.bfloat16, device="cuda")
            self.ys = None
            self.in_dtype, self.w_dtype = moe.DTYPE_BF16, moe.DTYPE_BF16
        self.yp = torch.empty(self.cap, dtype=torch.float32, device="cuda")
        self.weights, self.fc2_global = weights, fc2_global
        self.mlp_ws = torch.empty(moe.moe_grouped_mlp_workspace_size(self.shape, self.layout, self.w_dtype),
                                  dtype=torch.uint8, device="cuda")
        self.o = torch.empty(self.cap, w.H, dtype=torch.bfloat16, device="cuda")
        self.out = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")

    def load(self, x, rmap, probs, n):
        """The first n tokens real, the rest "no route" with zero activations."""
        self.map.fill_(-1)
        self.probs.zero_()
        self.x.zero_()
        self.map[:n].copy_(torch.from_numpy(rmap[:n]))
        self.probs[:n].copy_(torch.from_numpy(probs[:n]))
        self.x[:n].copy_(x[:n])

    def run(self, stream):
        m, W = self.moe, self.weights
        m.moe_preprocess(self.routing, self.shape, self.layout, self.handle, self.ws, stream=stream)
        m.moe_dispatch_permute(self.handle, self.shape, self.layout, self.in_dtype, self.x,
                               W["gx"] if self.nvfp4 else None, self.routing, self.y, self.yp, self.ys, stream=stream)
        m.moe_grouped_mlp(self.handle, self.shape, self.layout, self.w_dtype, self.y, self.ys, W["w13"], W["s13"],
                          W["w2"], W["s2"], W["globals"], self.mlp_ws, self.o, stream=stream)
        m.moe_combine_unpermute(self.handle, self.shape, self.layout, self.o, self.yp, self.out, stream=stream)


def _weights(moe, w):
    w13, w2 = workloads.expert_weights(w, 3, device="cuda")
    if w.dtype != "nvfp4":
        return dict(w13=w13, w2=w2, s13=None, s2=None, globals=None, gx=None)
    g13 = (w13.float().abs().amax(dim=(1, 2)) / 2688.0).contiguous()
    g2 = (w2.float().abs().amax(dim=(1, 2)) / 2688.0).contiguous()
    q13 = torch.empty(w.E, 2 * w.I, w.H // 2, dtype=torch.uint8, device="cuda")
    s13 = torch.empty(w.E, 2 * w.I, w.H // 16, dtype=torch.uint8, device="cuda")
    q2 = torch.empty(w.E, w.H, w.I // 2, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(w.E, w.H, w.I // 16, dtype=torch.uint8, device="cuda")
    for e in range(w.E):
        moe.moe_quantize_nvfp4_rows(w13[e], g13[e:e + 1], q13[e], s13[e])
        moe.moe_quantize_nvfp4_rows(w2[e], g2[e:e + 1], q2[e], s2[e])
    gx = torch.tensor([4.0 / 2688.0], dtype=torch.float32, device="cuda")  # a fixed calibration constant
    return dict(w13=q13, w2=q2, s13=s13, s2=s2, gx=gx,
                globals=moe.Nvfp4Globals(gx, torch.tensor([0.01], device="cuda"), g13, g2))


@pytest.mark.parametrize("dtype", ["bf16", "nvfp4"])
def test_bucketed_graph_replay_equals_unpadded_batches(moe, dtype):
    base = workloads.WORKLOADS["decode64"] if dtype == "nvfp4" else workloads.WORKLOADS["tiny"]
    w = workloads.scaled(base, T=64, H=1024, E=32, K=8, I=512)
    ladder = [1, 2, 4, 8, 16, 32, 64, 128]
    W = _weights(moe, w)
    stream = torch.cuda.Stream()
    bucket = moe.moe_decode_bucket(37, ladder)
    assert bucket == 64 and moe.moe_decode_bucket(50, ladder) == 64
    padded = Layer(moe, w, bucket, W, 0.01)
    with torch.cuda.stream(stream):  # warm the path once before capture
        padded.run(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        padded.run(stream)
    for n, seed in ((37, 11), (50, 12)):
        wn = workloads.scaled(w, T=n)
        _, rmap, probs = workloads.routing_inputs(wn, seed, "dense")
        x = workloads.activations(wn, seed).cuda()
        exact = Layer(moe, w, n, W, 0.01)
        exact.load(x, rmap, probs, n)
        with torch.cuda.stream(stream):
            exact.run(stream)
        padded.load(x, rmap, probs, n)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        assert int(padded.handle.status.item()) == 0 and int(padded.handle.overflow.item()) == 0
        got = bits(padded.out)
        assert np.array_equal(got[:n], bits(exact.out)), n
        assert not got[n:].any()
