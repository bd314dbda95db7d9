"""Pins for the oracle's bfloat16 paths, each against something other than
the oracle.  The kernel is registered for fp16 and bfloat16 activations
("PagedAttention - CUDA Design Document", section 8.2).

  * bfloat16 decode    -> torch's bfloat16 -> float64 conversion, all 65536
                          patterns (library routine)
  * bfloat16 rounding  -> torch's float32 -> bfloat16 conversion on values
                          exact in float32 (one rounding, nearest-even) and
                          closed-form halfway points, overflow and subnormals
  * attention          -> torch SDPA in fp64 on the dense bfloat16 KV, with
                          and without a bfloat16 head_sink (the sink as the
                          log-sum-exp epilogue, closed form)
  * rotary             -> complex multiplication by the tables' exp(i*angle)
                          within one bfloat16 ulp, position-0 identity,
                          channels past the rotary dim copied
  * cache write        -> the pools after a step hold the rotated K and the
                          V bits unchanged at the derived slots
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

BF16 = oracle.CACHE_BF16


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


# ------------------------------------------------------------ conversions -----

def test_bf16_to_double_all_patterns(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = from_bits(pats).double().numpy()
    got = np.array([oracle_lib.oracle_bf16_to_double(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_double_to_bf16_rne_matches_torch(oracle_lib):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 38, 20000),
        rng.standard_normal(5000),
        [0.0, -0.0, 3.0e38, 3.3961e38, 3.4e38, 1e-39, -1e-40, 1e-45, np.inf, -np.inf],
    ]).astype(np.float32)   # exact in float32: torch's float32 -> bfloat16 is then a single rounding
    ref = bits(torch.from_numpy(vals).to(torch.bfloat16))
    got = np.array([oracle_lib.oracle_double_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_double_to_bf16_closed_form_ties_and_limits(oracle_lib):
    f = lambda v: int(oracle_lib.oracle_double_to_bf16(float(v)))
    # halfway between 1 + k/128 and 1 + (k+1)/128 rounds to the even fraction
    for k in range(0, 127):
        tie = 1.0 + (k + 0.5) / 128.0
        want = k if k % 2 == 0 else k + 1
        assert f(tie) == 0x3F80 + want, k
        assert f(-tie) == 0xBF80 + want, k
    # just above the halfway point always rounds up
    assert f(1.0 + 1.5 / 128.0 + 2.0 ** -30) == 0x3F82
    assert f(1.0 + 0.5 / 128.0 + 2.0 ** -30) == 0x3F81
    # largest finite (2 - 2^-7) * 2^127; halfway to 2^128 and beyond overflow
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert f(big) == 0x7F7F
    assert f((2.0 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80
    assert f((2.0 - 2.0 ** -8) * 2.0 ** 127 * (1 - 2.0 ** -40)) == 0x7F7F
    # subnormals: quantum 2^-133; half a quantum ties to zero, 1.5 quanta to 2
    assert f(2.0 ** -133) == 0x0001
    assert f(2.0 ** -134) == 0x0000
    assert f(1.5 * 2.0 ** -133) == 0x0002
    assert f(127.5 * 2.0 ** -133) == 0x0080   # rounds up into the smallest normal
    assert f(2.0 ** -126) == 0x0080
    assert f(float("nan")) & 0x7FFF == 0x7FC0


# -------------------------------------------------------------- attention -----

def _case(H, Hk, D, bs, past, new, seed):
    g = torch.Generator().manual_seed(seed)
    L = [p + n for p, n in zip(past, new)]
    Ks = [torch.randn(l, Hk, D, generator=g).bfloat16() for l in L]
    Vs = [torch.randn(l, Hk, D, generator=g).bfloat16() for l in L]
    q = torch.randn(sum(new), H * D, generator=g).bfloat16()
    cum = torch.tensor([0] + list(np.cumsum(new)), dtype=torch.int32)
    return Ks, Vs, q, cum, torch.tensor(past, dtype=torch.int32)


def _pool(Ks, Vs, bs, Hk, D, seed=0):
    need = [(k.shape[0] + bs - 1) // bs for k in Ks]
    NB = sum(need) + 2
    ids = torch.randperm(NB, generator=torch.Generator().manual_seed(seed))
    bt = torch.full((len(Ks), max(need)), -1, dtype=torch.int32)
    kc = torch.full((NB, bs, Hk, D), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    cur = 0
    for b, (k, v) in enumerate(zip(Ks, Vs)):
        for i in range(need[b]):
            blk = int(ids[cur]); cur += 1
            bt[b, i] = blk
            n = min(bs, k.shape[0] - i * bs)
            kc[blk, :n] = k[i * bs:i * bs + n]
            vc[blk, :n] = v[i * bs:i * bs + n]
    return kc, vc, bt


def _sdpa(q, Ks, Vs, cum, past, H, Hk, D, scale, window):
    G = H // Hk
    out = torch.zeros(q.shape[0], H, D, dtype=torch.float64)
    lse = torch.zeros(q.shape[0], H, dtype=torch.float64)
    for b in range(len(Ks)):
        t0, t1 = int(cum[b]), int(cum[b + 1])
        if t1 == t0:
            continue
        qb = q[t0:t1].double().view(t1 - t0, H, D).transpose(0, 1)
        kb = Ks[b].double().transpose(0, 1).repeat_interleave(G, 0)
        vb = Vs[b].double().transpose(0, 1).repeat_interleave(G, 0)
        qpos = int(past[b]) + torch.arange(t1 - t0)[:, None]
        p = torch.arange(Ks[b].shape[0])[None, :]
        mask = p <= qpos
        if window >= 1:
            mask &= p > qpos - window
        out[t0:t1] = F.scaled_dot_product_attention(qb[None], kb[None], vb[None], attn_mask=mask,
                                                    scale=scale)[0].transpose(0, 1)
        x = (qb @ kb.transpose(1, 2)) * scale
        lse[t0:t1] = torch.logsumexp(x.masked_fill(~mask, float("-inf")), dim=-1).transpose(0, 1)
    return out, lse


@pytest.mark.parametrize("H,Hk,D,bs,past,new,window", [
    (4, 2, 32, 16, [0, 17, 40], [5, 1, 1], -1),
    (8, 2, 64, 32, [100, 0, 65], [1, 40, 3], -1),
    (8, 2, 16, 16, [100, 0, 65], [1, 40, 3], 7),
])
def test_bf16_attention_matches_sdpa(H, Hk, D, bs, past, new, window):
    Ks, Vs, q, cum, pst = _case(H, Hk, D, bs, past, new, seed=H * D + 3)
    kc, vc, bt = _pool(Ks, Vs, bs, Hk, D)
    scale = 1.0 / math.sqrt(D)
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, window,
                           cache_dtype=BF16)
    ref, lse = _sdpa(q, Ks, Vs, cum, pst, H, Hk, D, scale, window)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)
    # a bfloat16 sink scales each row by 1 / (1 + exp(s_h - lse))
    sink = torch.tensor([-1.5, 0.25, 2.0, 7.0] * (H // 4)).bfloat16()
    got_s = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, window,
                             cache_dtype=BF16, head_sink=bits(sink))
    f = 1.0 / (1.0 + torch.exp(sink.double()[None, :] - lse))
    np.testing.assert_allclose(got_s, (ref * f[..., None]).numpy(), rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------- rotary -----

def _complex_rotary(x, pos, cos_t, sin_t, half, interleaved):
    if interleaved:
        z = x[..., 0:2 * half:2] + 1j * x[..., 1:2 * half:2]
    else:
        z = x[..., :half] + 1j * x[..., half:2 * half]
    zr = z * (cos_t[pos] + 1j * sin_t[pos])[:, None, :]
    y = x.copy()
    if interleaved:
        y[..., 0:2 * half:2], y[..., 1:2 * half:2] = zr.real, zr.imag
    else:
        y[..., :half], y[..., half:2 * half] = zr.real, zr.imag
    return y


def _ulp_bf16(v):
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("interleaved", [0, 1])
@pytest.mark.parametrize("R", [32, 16])
def test_bf16_rotary_matches_complex_rotation(interleaved, R):
    H, D = 3, 32
    past, new = [0, 5, 100], [2, 3, 1]
    T = sum(new)
    cum = torch.tensor([0] + list(np.cumsum(new)), dtype=torch.int32)
    pst = torch.tensor(past, dtype=torch.int32)
    cos_t, sin_t = workloads.rotary_tables(200, R, dtype=torch.bfloat16)
    x = torch.randn(T, H * D, generator=torch.Generator().manual_seed(R + 5)).bfloat16()
    y = oracle.rotary(bits(x), cum, pst, cos_t, sin_t, H, D, interleaved, bf16=True)
    yv = from_bits(y).double().numpy().reshape(T, H, D)
    pos = np.concatenate([np.arange(p, p + n) for p, n in zip(past, new)])
    ref = _complex_rotary(x.double().numpy().reshape(T, H, D), pos, cos_t.double().numpy(),
                          sin_t.double().numpy(), R // 2, interleaved)
    # fp32 evaluation + one bfloat16 rounding stays within one bfloat16 ulp
    assert np.all(np.abs(yv - ref) <= _ulp_bf16(ref) + 1e-30)
    # and is not the fp16 result: some outputs carry no more than 8 significant bits
    assert np.array_equal(yv, from_bits(oracle.double_to_bf16_bits(yv)).double().numpy())
    assert np.array_equal(y[0], bits(x)[0])                       # position 0: identity
    assert np.array_equal(y.reshape(T, H, D)[..., R:], bits(x).reshape(T, H, D)[..., R:])


# ------------------------------------------------------------- whole step -----

def test_bf16_step_writes_rotated_key_and_value_bits():
    shape = workloads.custom_shape("bf16_pin", 4, 2, 32, 16, [5, 0, 40], [2, 3, 1], do_rotary=1, seed=3)
    st = workloads.make_step(shape, cache_dtype=BF16)
    assert st["query"].dtype == torch.bfloat16 and st["cos_cache"].dtype == torch.bfloat16
    r = oracle.forward(st)
    k_rot = oracle.rotary(st["key"], st["cumulative_sequence_lengths"], st["past_sequence_lengths"],
                          st["cos_cache"], st["sin_cache"], 2, 32, 0, bf16=True)
    kc, vc = r["key_cache"].reshape(st["num_blocks"], 16, 64), r["value_cache"].reshape(st["num_blocks"], 16, 64)
    bt = st["block_table"].numpy()
    vb = bits(st["value"])
    t = 0
    for b, (p0, n) in enumerate(zip([5, 0, 40], [2, 3, 1])):
        for j in range(n):
            pos = p0 + j
            blk, off = bt[b, pos // 16], pos % 16
            assert np.array_equal(kc[blk, off], k_rot[t]) and np.array_equal(vc[blk, off], vb[t])
            t += 1
    # rotation changed something away from position 0, and the output is finite
    assert not np.array_equal(k_rot[2:], bits(st["key"])[2:])
    assert np.isfinite(r["out"]).all()


# --------------------------------------------------------------- QK-Norm -----

def test_bf16_qk_norm_matches_torch_rms_norm():
    """bfloat16 QK-Norm: fp32 arithmetic, one bfloat16 rounding: within one
    bfloat16 ulp of torch's rms_norm evaluated in fp64 (a weight or an
    epsilon left out, or an fp16 rounding, would miss it)."""
    g = torch.Generator().manual_seed(7)
    for D, nh in ((64, 3), (128, 4), (256, 2)):
        x = (torch.randn(7, nh * D, generator=g) * (0.1 + 3 * torch.rand(7, 1, generator=g))).bfloat16()
        w = (1 + 0.5 * torch.randn(D, generator=g)).bfloat16()
        got = from_bits(oracle.qk_norm(bits(x), nh, D, bits(w), 1e-6, bf16=True)).double().numpy()
        ref = F.rms_norm(x.double().view(7, nh, D), (D,), w.double(), eps=1e-6).view(7, nh * D).numpy()
        assert np.all(np.abs(got - ref) <= _ulp_bf16(ref) + 1e-30)
        assert np.array_equal(got, from_bits(oracle.double_to_bf16_bits(got)).double().numpy())


def test_bf16_qk_norm_constant_rows_closed_form():
    D = 128
    for a in (2.0, -0.375, 17.0):
        x = torch.full((1, D), a).bfloat16()
        w = torch.ones(D).bfloat16()
        got = from_bits(oracle.qk_norm(bits(x), 1, D, bits(w), 1e-6, bf16=True)).double().numpy()
        ref = torch.tensor(a / math.sqrt(a * a + 1e-6)).bfloat16().double().item()
        assert np.all(got == ref), (a, got[0, 0], ref)


def test_bf16_packed_qk_norm_step_pools():
    """A bfloat16 step with packed QKV rows and QK-Norm: the key pool holds
    the normalized, rotated K rows and the value pool the V bits."""
    shape = workloads.custom_shape("bf16_pk", 4, 2, 64, 16, [3, 20], [2, 1], do_rotary=1, seed=9)
    st = workloads.make_step(shape, cache_dtype=BF16, qk_norm=True, packed_qkv=True)
    assert st["key"] is None and st["q_norm_weight"].dtype == torch.bfloat16
    r = oracle.forward(st)
    q, k, v = oracle.split_packed_qkv(st["query"], 4, 2, 64)
    kn = oracle.qk_norm(k, 2, 64, st["k_norm_weight"], 1e-6, bf16=True)
    kr = oracle.rotary(kn, st["cumulative_sequence_lengths"], st["past_sequence_lengths"], st["cos_cache"],
                       st["sin_cache"], 2, 64, 0, bf16=True)
    assert np.array_equal(r["key_rot"], kr)
    bt = st["block_table"].numpy()
    kc = r["key_cache"].reshape(st["num_blocks"], 16, 128)
    vc = r["value_cache"].reshape(st["num_blocks"], 16, 128)
    t = 0
    for b, (p0, n) in enumerate(zip([3, 20], [2, 1])):
        for j in range(n):
            pos = p0 + j
            assert np.array_equal(kc[bt[b, pos // 16], pos % 16], kr[t])
            assert np.array_equal(vc[bt[b, pos // 16], pos % 16], v[t])
            t += 1
    assert np.isfinite(r["out"]).all()
