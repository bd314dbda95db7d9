"""CUDA-graph decode replay ("PagedAttention - CUDA Design Document", section
17.6): capture one pa_forward, then replay it for several decode steps while
every sequence's context grows, writing each step's new Q/K/V and lengths
into the same device buffers.  Every step is checked against the oracle, so
a launch extent or mask bound frozen at capture fails from step 2 on."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("window,softcap", [(-1, 0.0), (40, 30.0)])
def test_graph_replay_with_growing_context(window, softcap):
    steps = 6
    past0 = [10, 100, 31, 0, 63]
    H, Hk, D, bs = 8, 2, 128, 16
    # lay out blocks for the final lengths; step i adds one token per sequence
    shape = workloads.custom_shape("graph", H, Hk, D, bs, [p + steps for p in past0], [1] * 5,
                                   local_window_size=window, softcap=softcap, seed=21)
    full = workloads.make_step(shape, device="cpu")
    B, T = 5, 5
    bt = full["block_table"]
    # the pool holds the first past0[b] positions; later ones start as sentinels
    host_k, host_v = full["key_cache"].clone(), full["value_cache"].clone()
    for b in range(B):
        for p in range(past0[b], past0[b] + steps + 1):
            blk = int(bt[b, p // bs])
            host_k[blk, p % bs] = torch.tensor(workloads.NAN_SENTINEL_BITS, dtype=torch.int16).view(torch.float16)
            host_v[blk, p % bs] = torch.tensor(workloads.NAN_SENTINEL_BITS, dtype=torch.int16).view(torch.float16)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in full.items()}
    dev["key_cache"].copy_(host_k)
    dev["value_cache"].copy_(host_v)
    dev["past_sequence_lengths"].copy_(torch.tensor(past0, dtype=torch.int32))
    op = pa.PagedAttention.for_step(dev, max_batch=B, max_tokens=T)
    out = torch.zeros(T, H * D, dtype=torch.float16, device="cuda")

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    op.forward(dev, out, stream=s.cuda_stream)  # warm-up (capture must not be the first call)
    torch.cuda.synchronize()
    dev["key_cache"].copy_(host_k)
    dev["value_cache"].copy_(host_v)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        op.forward(dev, out, stream=s.cuda_stream)
    torch.cuda.synchronize()

    gen = torch.Generator().manual_seed(5)
    kc, vc = bits(host_k), bits(host_v)
    for i in range(steps):
        past = torch.tensor([p + i for p in past0], dtype=torch.int32)
        q = torch.randn(T, H * D, generator=gen).half()
        k = torch.randn(T, Hk * D, generator=gen).half()
        v = torch.randn(T, Hk * D, generator=gen).half()
        for name, val in (("query", q), ("key", k), ("value", v), ("past_sequence_lengths", past)):
            dev[name].copy_(val)
        g.replay()
        torch.cuda.synchronize()
        assert op.device_error() == 0
        kc, vc = oracle.cache_write(k, v, kc, vc, bt, full["cumulative_sequence_lengths"], past, Hk, D, bs)
        ref = oracle.attention(q, kc, vc, bt, full["cumulative_sequence_lengths"], past, H, Hk, D, bs,
                               0.0, softcap, window)
        assert np.array_equal(bits(dev["key_cache"]), kc), f"step {i}: key pool"
        assert np.array_equal(bits(dev["value_cache"]), vc), f"step {i}: value pool"
        assert_close(out.float().cpu().numpy().reshape(T, H, D), ref, what=f"step {i}")


@pytest.mark.parametrize("heads", [128, 32])
def test_latent_step_replays_in_a_graph(heads):
    """A latent step (tcgen05 kernel at 128 heads, mma.sync at 32) captured
    once and replayed with new query values gives the eager outputs bit for
    bit (the cache write is idempotent for the same new rows)."""
    shape = workloads.custom_shape("latent_graph", heads, 1, 576, 64, [300, 2500, 17, 1200], [1] * 4,
                                   scale=0.0723, do_rotary=1, rotary_dim=64, seed=23)
    dev = workloads.make_step(shape, device="cuda", gen_device="cpu", latent_v_head_size=512)
    op = pa.PagedAttention.for_step(dev, max_query_len_bound=1)
    out = torch.zeros(4, heads * 512, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    op.forward(dev, out, stream=s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        op.forward(dev, out, stream=s.cuda_stream)
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(7)
    for _ in range(2):
        dev["query"].copy_(torch.randn(dev["query"].shape, generator=gen).half())
        eager = torch.zeros_like(out)
        op.forward(dev, eager, stream=s.cuda_stream)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert op.device_error() == 0
        assert torch.equal(out, eager)
