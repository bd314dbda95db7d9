"""Pins for the oracle's multi-head latent attention ("PagedAttention - CUDA
Design Document", section 12), each against something other than the oracle:

  * latent attention -> torch scaled_dot_product_attention in fp64 with K the
                        576-channel latent rows (one kv head shared by every
                        query head) and V their first 512 channels
  * window + softcap -> the masks and cap * tanh(scale * q.k / cap) written
                        out on the dense latent rows, fp64 softmax
  * offset rotary    -> complex multiplication of the channels
                        [offset, offset + R) by the tables' cos + i sin (numpy
                        complex128) within one fp16 ulp, every other channel
                        copied bit for bit
"""

import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import workloads
from test_oracle_pins import _complex_rotary, _ulp16


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_latent_attention_matches_sdpa():
    H, D, Dv, bs = 8, 576, 512, 16
    shape = workloads.custom_shape("mla_pin", H, 1, D, bs, [0, 40, 7], [3, 1, 2], scale=0.07, seed=61)
    step = workloads.make_step(shape, latent_v_head_size=Dv)
    res = oracle.forward(step)
    # dense reference per sequence from the written pool
    kc = torch.from_numpy(res["key_cache"].view(np.float16).astype(np.float32)).double()  # [NB, bs, 1, D]
    bt, cum, past = step["block_table"], step["cumulative_sequence_lengths"], step["past_sequence_lengths"]
    q = torch.from_numpy(res["query_rot"].view(np.float16).astype(np.float32)).double().view(-1, H, D)
    for b in range(step["batch"]):
        L = int(past[b]) + int(cum[b + 1] - cum[b])
        rows = torch.stack([kc[int(bt[b, p // bs]), p % bs, 0] for p in range(L)])  # [L, D]
        t0, t1 = int(cum[b]), int(cum[b + 1])
        qb = q[t0:t1].transpose(0, 1)[None]                       # [1, H, q, D]
        kb = rows[None, None].expand(1, H, L, D)
        vb = rows[None, None, :, :Dv].expand(1, H, L, Dv)
        j = torch.arange(t1 - t0)[:, None]
        mask = torch.arange(L)[None, :] <= int(past[b]) + j
        ref = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=0.07)[0].transpose(0, 1)
        np.testing.assert_allclose(res["out"][t0:t1], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_latent_attention_with_window_and_softcap():
    """Window (each row admits [pos + 1 - W, pos]) and softcap
    (cap * tanh(scale * q.k / cap)) written out on the dense latent rows:
    explicit fp64 scores, masks and softmax, V = the first 512 channels."""
    H, D, Dv, bs, W, cap, scale = 4, 576, 512, 16, 20, 5.0, 0.07
    shape = workloads.custom_shape("mla_pin_wc", H, 1, D, bs, [50, 3], [2, 1], scale=scale, softcap=cap,
                                   local_window_size=W, seed=62)
    step = workloads.make_step(shape, latent_v_head_size=Dv)
    res = oracle.forward(step)
    kc = torch.from_numpy(res["key_cache"].view(np.float16).astype(np.float32)).double()
    bt, cum, past = step["block_table"], step["cumulative_sequence_lengths"], step["past_sequence_lengths"]
    q = torch.from_numpy(res["query_rot"].view(np.float16).astype(np.float32)).double().view(-1, H, D)
    for b in range(step["batch"]):
        t0, t1 = int(cum[b]), int(cum[b + 1])
        L = int(past[b]) + (t1 - t0)
        rows = torch.stack([kc[int(bt[b, p // bs]), p % bs, 0] for p in range(L)])  # [L, D]
        for j in range(t1 - t0):
            pos = int(past[b]) + j
            keys = torch.arange(L)
            ok = (keys <= pos) & (keys >= pos + 1 - W)
            sc = cap * torch.tanh(scale * (q[t0 + j] @ rows.T) / cap)                # [H, L]
            sc = sc.masked_fill(~ok[None, :], float("-inf"))
            p = torch.softmax(sc, dim=-1)
            ref = p @ rows[:, :Dv]                                                     # [H, Dv]
            np.testing.assert_allclose(res["out"][t0 + j], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_offset_rotary_matches_complex_rotation():
    T, nh, D, R, off = 3, 2, 576, 64, 512
    g = torch.Generator().manual_seed(62)
    x = torch.randn(T, nh * D, generator=g).half()
    past = torch.tensor([5, 100, 0], dtype=torch.int32)
    cum = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    cos, sin = workloads.rotary_tables(256, R)
    y = oracle.rotary(_bits(x), cum, past, _bits(cos), _bits(sin), nh, D, 0, offset=off)
    xb = _bits(x).reshape(T, nh, D)
    yb = y.reshape(T, nh, D)
    assert np.array_equal(yb[:, :, :off], xb[:, :, :off])  # channels outside the range are copied
    # the range itself: the pinned offset-0 rotation of the sliced channels
    ref = _complex_rotary(x.double().numpy().reshape(T, nh, D)[:, :, off:off + R], past.numpy(), cos.numpy(),
                          sin.numpy(), R // 2, 0)
    got = y.view(np.float16).astype(np.float64).reshape(T, nh, D)[:, :, off:off + R]
    assert np.all(np.abs(got - ref) <= _ulp16(ref) + 1e-12)


def test_separate_layout_step_rotates_at_its_offset():
    # a step with separate K/V caches and rotary_offset 32, rotary_dim 64 on
    # head_size 128: Q and K rows are rotated over channels [32, 96) exactly
    # as the pinned offset rotation does, every other channel is copied, and
    # the cached K rows are those rotated rows
    shape = workloads.custom_shape("sep_offset", 8, 2, 128, 16, [5, 40], [1, 3], do_rotary=1, rotary_dim=64,
                                   seed=63)
    step = workloads.make_step(shape)
    step["rotary_offset"] = 32
    res = oracle.forward(step)
    cum, past = step["cumulative_sequence_lengths"], step["past_sequence_lengths"]
    for name, nh, got in (("query", 8, res["query_rot"]), ("key", 2, res["key_rot"])):
        x = _bits(step[name])
        ref = oracle.rotary(x, cum, past, _bits(step["cos_cache"]), _bits(step["sin_cache"]), nh, 128, 0, offset=32)
        assert np.array_equal(got, ref)
        xb, gb = x.reshape(-1, nh, 128), got.reshape(-1, nh, 128)
        assert np.array_equal(gb[:, :, :32], xb[:, :, :32]) and np.array_equal(gb[:, :, 96:], xb[:, :, 96:])
        assert not np.array_equal(gb[:, :, 32:96], xb[:, :, 32:96])
    kc = res["key_cache"].reshape(-1, 2 * 128)
    bt = step["block_table"].numpy()
    for b, (p0, q) in enumerate(((5, 1), (40, 3))):
        for j in range(q):
            pos = p0 + j
            slot = bt[b, pos // 16] * 16 + pos % 16
            t = int(cum[b]) + j
            assert np.array_equal(kc[slot], res["key_rot"].reshape(-1, 256)[t])
