"""Pins for bfloat16 activations over 8-bit caches (the kernel is registered
for fp16 and bfloat16 activations with int8 and float8 caches, "PagedAttention
- CUDA Design Document", section 8.2), each against something other than the
oracle.

  * quantize from bfloat16 -> numpy float32 division / rint / clip (int8) and
                              torch's float8_e4m3fn conversion (e4m3), on
                              values decoded by torch from bfloat16
  * attention, bfloat16 query -> torch SDPA in fp64 on the dequantized KV with
                              the query decoded by torch from bfloat16
  * head_sink in bfloat16  -> the fp16 sink path (pinned in
                              test_oracle_quant_pins.py) on sink values exact
                              in both formats
  * whole step             -> written codes equal numpy quantization of the
                              torch-decoded bfloat16 key / value rows; the
                              output equals SDPA on the dequantized pools
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from test_oracle_pins import _rand_case, _sdpa_reference, bits
from test_oracle_quant_pins import _dequant_dense, _numpy_quant, _quant_pools

INT8, FP8 = oracle.CACHE_INT8, oracle.CACHE_FP8


def _bf16_values(n, seed, spread=4.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, generator=g) * spread).to(torch.bfloat16)


@pytest.mark.parametrize("scale", [1.0, 0.03125, 0.0371, 7.5])
def test_bf16_int8_quantize_matches_numpy(scale):
    x = torch.cat([_bf16_values(5000, 11),
                   (torch.tensor([0.5, 1.5, 2.5, -0.5, -2.5, 1e3, -1e3, 3e38]) * scale).to(torch.bfloat16)])
    y = x.float().numpy() / np.float32(scale)
    ref = np.clip(np.rint(y), -128, 127).astype(np.int8).view(np.uint8)
    got = oracle.quantize(bits(x), scale, INT8 | oracle.ACT_BF16)
    assert np.array_equal(got, ref)
    # the same bits read as fp16 quantize differently (the flag is not ignored)
    assert not np.array_equal(oracle.quantize(bits(x), scale, INT8), ref)


@pytest.mark.parametrize("scale", [1.0, 0.0123, 0.25])
def test_bf16_fp8_quantize_matches_torch(scale):
    x = _bf16_values(5000, 12, spread=3.0)
    y = x.float().numpy() / np.float32(scale)
    keep = np.abs(y) <= 448.0
    ref = torch.from_numpy(y[keep]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.quantize(bits(x)[keep], scale, FP8 | oracle.ACT_BF16)
    assert np.array_equal(got, ref)
    # beyond the range the code saturates, as for fp16 inputs
    big = torch.tensor([1e4, -1e4, 3e38], dtype=torch.bfloat16)
    assert list(oracle.quantize(bits(big), 1.0, FP8 | oracle.ACT_BF16)) == [0x7E, 0xFE, 0x7E]


@pytest.mark.parametrize("cache_dtype", [INT8, FP8])
@pytest.mark.parametrize("per_channel", [False, True])
def test_bf16_query_quant_attention_matches_sdpa(cache_dtype, per_channel):
    H, Hk, D, bs = 8, 2, 32, 16
    past, new = [0, 29, 70], [4, 1, 2]
    Ks, Vs, _, cum, pst = _rand_case(H, Hk, D, bs, past, new, seed=13)
    q = torch.randn(int(cum[-1]), H * D, generator=torch.Generator().manual_seed(14)).to(torch.bfloat16)
    g = torch.Generator().manual_seed(15)
    n_s = Hk * D if per_channel else 1
    ks = (torch.rand(n_s, generator=g) * 0.04 + 0.02).numpy().astype(np.float32)
    vs = (torch.rand(n_s, generator=g) * 0.04 + 0.02).numpy().astype(np.float32)
    ksb = np.broadcast_to(ks if per_channel else ks[0], (Hk * D,)).copy()
    vsb = np.broadcast_to(vs if per_channel else vs[0], (Hk * D,)).copy()
    kq, vq, bt = _quant_pools(Ks, Vs, bs, Hk, D, cache_dtype, ksb, vsb)
    got = oracle.attention(bits(q), kq, vq, bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1,
                           cache_dtype=cache_dtype | oracle.ACT_BF16, k_scale=ks, v_scale=vs,
                           per_channel=per_channel)
    Kd, Vd = [], []
    for k, v in zip(Ks, Vs):
        kcode = _numpy_quant(k.numpy(), np.broadcast_to(ksb.reshape(Hk, D), k.shape), cache_dtype)
        vcode = _numpy_quant(v.numpy(), np.broadcast_to(vsb.reshape(Hk, D), v.shape), cache_dtype)
        Kd.append(torch.from_numpy(_dequant_dense(kcode, ksb.reshape(Hk, D), cache_dtype)))
        Vd.append(torch.from_numpy(_dequant_dense(vcode, vsb.reshape(Hk, D), cache_dtype)))
    ref = _sdpa_reference(q, Kd, Vd, cum, pst, H, Hk, D, 1.0 / math.sqrt(D))
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("cache_dtype", [INT8, FP8])
def test_bf16_sink_equals_fp16_sink_on_shared_values(cache_dtype):
    """Sink and query values exact in both formats: the bfloat16 call equals
    the fp16 call, which is pinned to the log-sum-exp epilogue."""
    H, Hk, D, bs = 4, 2, 16, 16
    past, new = [0, 17, 40], [5, 1, 3]
    Ks, Vs, _, cum, pst = _rand_case(H, Hk, D, bs, past, new, seed=16)
    g = torch.Generator().manual_seed(17)
    qv = (torch.randint(-64, 65, (int(cum[-1]), H * D), generator=g).double() / 32.0)
    sv = torch.tensor([1.5, -2.25, 0.0, 3.0], dtype=torch.float64)
    ks = vs = np.array([0.03125], dtype=np.float32)
    kq, vq, bt = _quant_pools(Ks, Vs, bs, Hk, D, cache_dtype, np.full(Hk * D, ks[0], np.float32),
                              np.full(Hk * D, vs[0], np.float32))
    args = (kq, vq, bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1)
    ref = oracle.attention(bits(qv.half()), *args, cache_dtype=cache_dtype, k_scale=ks, v_scale=vs,
                           head_sink=bits(sv.half()))
    got = oracle.attention(bits(qv.to(torch.bfloat16)), *args, cache_dtype=cache_dtype | oracle.ACT_BF16,
                           k_scale=ks, v_scale=vs, head_sink=bits(sv.to(torch.bfloat16)))
    assert np.array_equal(got, ref)
    # reading the bfloat16 sink bits as fp16 would change the result
    bad = oracle.attention(bits(qv.to(torch.bfloat16)), *args, cache_dtype=cache_dtype | oracle.ACT_BF16,
                           k_scale=ks, v_scale=vs, head_sink=bits(sv.half()))
    assert not np.array_equal(bad, ref)


@pytest.mark.parametrize("cache_dtype", [INT8, FP8])
@pytest.mark.parametrize("quant_type", [workloads.QUANT_PER_TENSOR, workloads.QUANT_PER_CHANNEL])
def test_bf16_quant_step_codes_and_output(cache_dtype, quant_type):
    shape = workloads.custom_shape("pin_bf16_q8", 4, 2, 32, 16, [0, 21, 40], [3, 1, 17], seed=18)
    step = workloads.make_step(shape, cache_dtype=cache_dtype, quant_type=quant_type, act_bf16=True)
    assert step["query"].dtype == torch.bfloat16 and step["key_cache"].dtype == torch.uint8
    res = oracle.forward(step)
    Hk, D, bs = 2, 32, 16
    ks = np.broadcast_to(step["k_scale"].numpy(), (Hk * D,)).reshape(Hk, D)
    vs = np.broadcast_to(step["v_scale"].numpy(), (Hk * D,)).reshape(Hk, D)
    bt = step["block_table"]
    cum, past = step["cumulative_sequence_lengths"], step["past_sequence_lengths"]
    kc0, vc0 = step["key_cache"].numpy(), step["value_cache"].numpy()
    ekc, evc = kc0.copy(), vc0.copy()
    kd = step["key"].float().numpy().reshape(-1, Hk, D)
    vd = step["value"].float().numpy().reshape(-1, Hk, D)
    for b in range(3):
        for t in range(int(cum[b]), int(cum[b + 1])):
            pos = int(past[b]) + t - int(cum[b])
            blk, off = int(bt[b, pos // bs]), pos % bs
            ekc[blk, off] = _numpy_quant(kd[t], ks, cache_dtype)
            evc[blk, off] = _numpy_quant(vd[t], vs, cache_dtype)
    assert np.array_equal(res["key_cache"], ekc) and np.array_equal(res["value_cache"], evc)
    # output: SDPA on the dequantized written pools with the bfloat16 query
    Kd, Vd = [], []
    for b in range(3):
        L = int(past[b]) + int(cum[b + 1]) - int(cum[b])
        ids = [int(bt[b, p // bs]) for p in range(L)]
        offs = [p % bs for p in range(L)]
        Kd.append(torch.from_numpy(_dequant_dense(np.stack([ekc[i, o] for i, o in zip(ids, offs)]), ks, cache_dtype)))
        Vd.append(torch.from_numpy(_dequant_dense(np.stack([evc[i, o] for i, o in zip(ids, offs)]), vs, cache_dtype)))
    ref = _sdpa_reference(step["query"], Kd, Vd, cum, past, 4, Hk, D, 1.0 / math.sqrt(D))
    np.testing.assert_allclose(res["out"], ref.numpy(), rtol=1e-10, atol=1e-12)
