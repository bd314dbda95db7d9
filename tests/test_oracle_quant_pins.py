"""Pins for the oracle's quantized cache and head_sink, each against something
other than the oracle.

  * e4m3fn decode     -> torch.float8_e4m3fn (all 256 codes)
  * e4m3fn encode     -> torch's float -> float8_e4m3fn conversion (round to
                         nearest-even) on every tie and on random values in
                         range; saturation to +-448 (the saturating reading of
                         the CUDA design, section 8) on hand-picked values
  * int8 encode       -> numpy float32 division, rint and clip
  * quantized write   -> the fp16 write (pinned in test_oracle_pins.py) with
                         numpy / torch quantization of the written rows
  * quantized attention -> exactly representable codes reduce to the fp16
                         attention; random codes against torch SDPA in fp64 on
                         the dequantized dense KV
  * head_sink         -> the exact log-sum-exp epilogue of the CUDA design,
                         section 6.2: o_sink = o / (1 + exp(s - lse)), with lse
                         from scipy's logsumexp of torch-computed logits;
                         s = -inf reduces to no sink
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle
from test_oracle_pins import _paged_from_dense, _rand_case, _sdpa_reference, bits


# ------------------------------------------------------------- e4m3fn -----

def test_e4m3_decode_table_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_to_double(np.arange(256))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # landmarks of the format: largest finite, smallest normal and subnormal, one
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e4m3_encode_ties_and_random_match_torch():
    vals = oracle.e4m3_to_double(np.arange(0x7F))            # finite non-negative codes, ascending
    mids = ((vals[:-1] + vals[1:]) / 2)                       # exact ties in fp32
    rng = np.random.default_rng(1)
    rand = rng.standard_normal(20000) * 10.0 ** rng.integers(-4, 3, 20000)
    x = np.concatenate([vals, mids, -mids, rand]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.float_to_e4m3(x)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates():
    x = np.array([448.0, 450.0, 463.9, 464.0, 500.0, 1e9, np.inf], dtype=np.float32)
    assert np.all(oracle.float_to_e4m3(x) == 0x7E)
    assert np.all(oracle.float_to_e4m3(-x) == 0xFE)
    assert oracle.float_to_e4m3(np.array([np.nan], dtype=np.float32))[0] == 0x7F


# --------------------------------------------------------------- int8 -----

@pytest.mark.parametrize("scale", [1.0, 0.03125, 0.0371, 7.5])
def test_int8_quantize_matches_numpy(scale):
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(5000) * 4).astype(np.float16)
    x = np.concatenate([x, np.array([0.5, 1.5, 2.5, -0.5, -2.5, 1e3, -1e3], np.float16) * np.float16(scale)])
    ref = np.clip(np.rint(x.astype(np.float32) / np.float32(scale)), -128, 127).astype(np.int8).view(np.uint8)
    got = oracle.quantize(x.view(np.uint16), scale, oracle.CACHE_INT8)
    assert np.array_equal(got, ref)


def test_int8_quantize_nan_and_infinity():
    x = np.array([np.nan, np.inf, -np.inf], dtype=np.float16).view(np.uint16)
    assert list(oracle.quantize(x, 0.5, oracle.CACHE_INT8)) == [0, 127, 128]


@pytest.mark.parametrize("scale", [1.0, 0.0123, 0.25])
def test_fp8_quantize_matches_torch(scale):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(5000) * 3).astype(np.float16)
    y = x.astype(np.float32) / np.float32(scale)
    keep = np.abs(y) <= 448.0
    ref = torch.from_numpy(y[keep]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.quantize(x[keep].view(np.uint16), scale, oracle.CACHE_FP8)
    assert np.array_equal(got, ref)


# ------------------------------------------------------ quantized write -----

def _numpy_quant(vals_f16, scales, cache_dtype):
    y = vals_f16.astype(np.float32) / scales.astype(np.float32)
    if cache_dtype == oracle.CACHE_INT8:
        return np.clip(np.rint(y), -128, 127).astype(np.int8).view(np.uint8)
    return torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("cache_dtype", [oracle.CACHE_INT8, oracle.CACHE_FP8])
@pytest.mark.parametrize("per_channel", [False, True])
def test_quant_cache_write_matches_fp16_write_then_quantize(cache_dtype, per_channel):
    H, Hk, D, bs = 4, 2, 16, 16
    past, new = [0, 17, 40], [5, 1, 3]
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, past, new, seed=4)
    kc16, vc16, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    g = torch.Generator().manual_seed(5)
    n_s = Hk * D if per_channel else 1
    ks = (torch.rand(n_s, generator=g) * 0.05 + 0.01).numpy().astype(np.float32)
    vs = (torch.rand(n_s, generator=g) * 0.05 + 0.01).numpy().astype(np.float32)
    T = int(cum[-1])
    key = torch.randn(T, Hk * D, generator=g).half()
    val = torch.randn(T, Hk * D, generator=g).half()
    init_k = np.random.default_rng(6).integers(0, 256, kc16.shape, dtype=np.uint8)
    init_v = np.random.default_rng(7).integers(0, 256, vc16.shape, dtype=np.uint8)
    gk, gv = oracle.cache_write(bits(key), bits(val), init_k, init_v, bt, cum, pst, Hk, D, bs,
                                cache_dtype=cache_dtype, k_scale=ks, v_scale=vs, per_channel=per_channel)
    # fp16 write (pinned separately), then quantize the rows it wrote
    wk, wv = oracle.cache_write(bits(key), bits(val), np.zeros(kc16.shape, np.uint16),
                                np.zeros(vc16.shape, np.uint16), bt, cum, pst, Hk, D, bs)
    marker_k, _ = oracle.cache_write(np.full((T, Hk * D), 1, np.uint16), np.full((T, Hk * D), 1, np.uint16),
                                     np.zeros(kc16.shape, np.uint16), np.zeros(vc16.shape, np.uint16),
                                     bt, cum, pst, Hk, D, bs)
    written = marker_k == 1
    sk = np.broadcast_to(ks.reshape(-1) if per_channel else ks, (Hk * D,)).reshape(Hk, D)
    sv = np.broadcast_to(vs.reshape(-1) if per_channel else vs, (Hk * D,)).reshape(Hk, D)
    ek = np.where(written, _numpy_quant(wk.view(np.float16), np.broadcast_to(sk, wk.shape), cache_dtype), init_k)
    ev = np.where(written, _numpy_quant(wv.view(np.float16), np.broadcast_to(sv, wv.shape), cache_dtype), init_v)
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


# -------------------------------------------------- quantized attention -----

def _quant_pools(Ks, Vs, bs, Hk, D, cache_dtype, ks, vs):
    """Dense fp16 K/V -> paged 8-bit pools with numpy/torch quantization."""
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    kq = _numpy_quant(np.nan_to_num(kc.numpy()), np.broadcast_to(ks.reshape(Hk, D), kc.shape), cache_dtype)
    vq = _numpy_quant(np.nan_to_num(vc.numpy()), np.broadcast_to(vs.reshape(Hk, D), vc.shape), cache_dtype)
    return kq, vq, bt


def _dequant_dense(codes, scales, cache_dtype):
    if cache_dtype == oracle.CACHE_INT8:
        v = codes.view(np.int8).astype(np.float64)
    else:
        v = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    return v * scales.astype(np.float64)


@pytest.mark.parametrize("cache_dtype", [oracle.CACHE_INT8, oracle.CACHE_FP8])
def test_quant_attention_exact_codes_equal_fp16_attention(cache_dtype):
    H, Hk, D, bs = 4, 2, 16, 16
    past, new = [0, 17, 40], [5, 1, 3]
    g = torch.Generator().manual_seed(8)
    L = [p + n for p, n in zip(past, new)]
    # per-channel power-of-two scales and codes whose values are exact in fp16
    scales = (2.0 ** torch.randint(-6, 2, (Hk * D,), generator=g)).float()
    if cache_dtype == oracle.CACHE_INT8:
        code_vals = lambda n: torch.randint(-127, 128, (n, Hk, D), generator=g).double()
    else:
        finite = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double()
        finite = finite[~torch.isnan(finite)]
        code_vals = lambda n: finite[torch.randint(0, finite.numel(), (n, Hk, D), generator=g)]
    sc = scales.double().view(Hk, D)
    Ks = [(code_vals(l) * sc).half() for l in L]
    Vs = [(code_vals(l) * sc).half() for l in L]
    T = sum(new)
    q = torch.randn(T, H * D, generator=g).half()
    cum = torch.tensor([0] + list(np.cumsum(new)), dtype=torch.int32)
    pst = torch.tensor(past, dtype=torch.int32)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    ref = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1)
    ks = vs = scales.numpy()
    kq, vq, _ = _quant_pools(Ks, Vs, bs, Hk, D, cache_dtype, ks, vs)
    got = oracle.attention(bits(q), kq, vq, bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1,
                           cache_dtype=cache_dtype, k_scale=ks, v_scale=vs, per_channel=True)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("cache_dtype", [oracle.CACHE_INT8, oracle.CACHE_FP8])
@pytest.mark.parametrize("per_channel", [False, True])
def test_quant_attention_matches_sdpa_on_dequantized_kv(cache_dtype, per_channel):
    H, Hk, D, bs = 8, 2, 32, 16
    past, new = [0, 29, 70], [4, 1, 2]
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, past, new, seed=9)
    g = torch.Generator().manual_seed(10)
    n_s = Hk * D if per_channel else 1
    ks = (torch.rand(n_s, generator=g) * 0.04 + 0.02).numpy().astype(np.float32)
    vs = (torch.rand(n_s, generator=g) * 0.04 + 0.02).numpy().astype(np.float32)
    ksb = np.broadcast_to(ks if per_channel else ks[0], (Hk * D,)).copy()
    vsb = np.broadcast_to(vs if per_channel else vs[0], (Hk * D,)).copy()
    kq, vq, bt = _quant_pools(Ks, Vs, bs, Hk, D, cache_dtype, ksb, vsb)
    got = oracle.attention(bits(q), kq, vq, bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1,
                           cache_dtype=cache_dtype, k_scale=ks, v_scale=vs, per_channel=per_channel)
    # dense dequantized KV through SDPA: quantize the dense rows the same way
    Kd, Vd = [], []
    for k, v in zip(Ks, Vs):
        kcode = _numpy_quant(k.numpy(), np.broadcast_to(ksb.reshape(Hk, D), k.shape), cache_dtype)
        vcode = _numpy_quant(v.numpy(), np.broadcast_to(vsb.reshape(Hk, D), v.shape), cache_dtype)
        Kd.append(torch.from_numpy(_dequant_dense(kcode, ksb.reshape(Hk, D), cache_dtype)))
        Vd.append(torch.from_numpy(_dequant_dense(vcode, vsb.reshape(Hk, D), cache_dtype)))
    ref = _sdpa_reference(q, Kd, Vd, cum, pst, H, Hk, D, 1.0 / math.sqrt(D))
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------- head_sink -----

def _logits(q, Ks, cum, pst, H, Hk, D, scale, softcap, window):
    """Per (t, h): admitted logits as a torch fp64 vector."""
    G = H // Hk
    out = {}
    for b in range(len(Ks)):
        for t in range(int(cum[b]), int(cum[b + 1])):
            pos = int(pst[b]) + t - int(cum[b])
            lo = max(0, pos + 1 - window) if window >= 1 else 0
            for h in range(H):
                qv = q[t].double().view(H, D)[h]
                x = Ks[b][lo:pos + 1, h // G].double() @ qv * scale
                if softcap > 0:
                    x = softcap * torch.tanh(x / softcap)
                out[(t, h)] = x
    return out


@pytest.mark.parametrize("softcap,window", [(0.0, -1), (20.0, -1), (0.0, 9), (30.0, 5)])
def test_head_sink_is_the_lse_epilogue(softcap, window):
    H, Hk, D, bs = 4, 2, 16, 16
    past, new = [0, 33, 12], [6, 1, 2]
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, past, new, seed=11)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    sink = torch.tensor([-1.5, 0.0, 2.0, 7.0]).half()
    base = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, softcap, window)
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, softcap, window,
                           head_sink=bits(sink))
    lg = _logits(q, Ks, cum, pst, H, Hk, D, 1.0 / math.sqrt(D), softcap, window)
    for (t, h), x in lg.items():
        lse = logsumexp(x.numpy())
        f = 1.0 / (1.0 + math.exp(float(sink[h]) - lse))
        np.testing.assert_allclose(got[t, h], base[t, h] * f, rtol=1e-12, atol=1e-15)


def test_head_sink_minus_infinity_is_no_sink_and_empty_rows_stay_zero():
    H, Hk, D, bs = 4, 2, 16, 16
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, [5, 20], [2, 1], seed=12)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    base = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1)
    ninf = torch.full((H,), float("-inf")).half()
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1,
                           head_sink=bits(ninf))
    assert np.array_equal(got, base)
    bt[1, :] = -1   # sequence 1 has no admitted key
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1,
                           head_sink=bits(torch.zeros(H).half()))
    assert np.all(got[2] == 0.0) and not np.isnan(got).any()
