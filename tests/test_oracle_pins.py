"""Pins for the CPU oracle, each against something other than the oracle.

  * fp16 conversion   -> numpy's own float16 conversion (library routine)
  * cache write       -> hand-derived slots (tests/golden/cache_write_slots.txt)
  * attention core    -> torch scaled_dot_product_attention in fp64 on the
                         dense contiguous KV (the GQA <-> paged cross-parity
                         idea of the CUDA design, section 17.1), with GQA as
                         repeat_interleave of KV heads and an explicit mask
  * invariants        -> block permutation, constant V, one-token context,
                         window 1, window >= context, -1 blocks, empty rows
  * softcap           -> large-cap limit (no softcap) and a two-key closed form
  * rotary            -> complex multiplication by exp(i * pos * theta) (fp64
                         numpy), position-0 identity, relative-position property
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

SENT = workloads.NAN_SENTINEL_BITS


def h16(x):
    return torch.as_tensor(x, dtype=torch.float16)


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- fp16 -----

def test_half_to_double_all_patterns(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.oracle_half_to_double(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_double_to_half_rne(oracle_lib):
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
        # exact halfway points between neighbouring halves (ties to even)
        (np.arange(1, 3000, dtype=np.float64) + 0.5) * 2.0 ** -24,
        (np.arange(1024, 2048, dtype=np.float64) + 0.5) * 2.0 ** -3,
        [65504.0, 65519.99, 65520.0, 1e6, -0.0, 0.0, 2.0 ** -25, 2.0 ** -25 * 1.0001,
         6.0975552e-05, np.inf, -np.inf],
    ])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle_lib.oracle_double_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------- cache write -----

def _parse_golden(path):
    meta, rows = {}, []
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0].isalpha() or "_" in parts[0]:
            if parts[0] == "block_table":
                meta["block_table"] = [[int(x) for x in r.split()] for r in " ".join(parts[1:]).split("|")]
            else:
                meta[parts[0]] = [int(x) for x in parts[1:]]
        else:
            rows.append(parts)
    return meta, rows


def test_cache_write_golden_slots():
    meta, rows = _parse_golden("tests/golden/cache_write_slots.txt")
    bs, NB = meta["block_size"][0], meta["num_blocks"][0]
    Hk, D = meta["kv_num_heads"][0], meta["head_size"][0]
    bt = torch.tensor(meta["block_table"], dtype=torch.int32)
    past = torch.tensor(meta["past"], dtype=torch.int32)
    new = meta["new"]
    cum = torch.tensor([0] + list(np.cumsum(new)), dtype=torch.int32)
    T = int(cum[-1])
    # token t carries the value t+1 in K and -(t+1) in V in every element
    key = h16(np.repeat(np.arange(1, T + 1, dtype=np.float32)[:, None], Hk * D, 1))
    value = -key
    pool = np.full((NB, bs, Hk, D), SENT, dtype=np.uint16)
    kc, vc = oracle.cache_write(bits(key), bits(value), pool, pool, bt, cum, past, Hk, D, bs)
    kflat = kc.reshape(NB * bs, Hk * D)
    vflat = vc.reshape(NB * bs, Hk * D)
    written = set()
    for tok, seq, posn, brow, bid, slot in rows:
        tok = int(tok)
        if slot == "none":
            continue
        slot = int(slot)
        written.add(slot)
        assert np.all(kflat[slot].view(np.float16) == tok + 1)
        assert np.all(vflat[slot].view(np.float16) == -(tok + 1))
    for s in range(NB * bs):
        if s not in written:
            assert np.all(kflat[s] == SENT) and np.all(vflat[s] == SENT), s


def test_cache_write_touches_only_new_slots():
    sh = workloads.custom_shape("w", 4, 2, 32, 16, [3, 0, 40, 16], [2, 20, 1, 0])
    st = workloads.make_step(sh)
    kc, vc = oracle.cache_write(st["key"], st["value"], st["key_cache"], st["value_cache"],
                                st["block_table"], st["cumulative_sequence_lengths"],
                                st["past_sequence_lengths"], 2, 32, 16)
    k0 = bits(st["key_cache"])
    changed = np.any(kc != k0, axis=(2, 3))           # [NB, bs]
    # every changed slot is a sentinel slot that now holds a new row
    assert np.all(k0[changed] == SENT)
    assert changed.sum() == st["token_count"]
    # the new rows appear in the pool exactly (multiset of rows)
    new_rows = sorted(map(bytes, bits(st["key"]).reshape(st["token_count"], -1)))
    got_rows = sorted(map(bytes, kc[changed].reshape(st["token_count"], -1)))
    assert new_rows == got_rows


def test_cache_write_unmapped_and_empty():
    sh = workloads.custom_shape("e", 2, 1, 16, 16, [5, 0], [0, 3])
    st = workloads.make_step(sh)
    st["block_table"][1, 0] = -1
    kc, vc = oracle.cache_write(st["key"], st["value"], st["key_cache"], st["value_cache"],
                                st["block_table"], st["cumulative_sequence_lengths"],
                                st["past_sequence_lengths"], 1, 16, 16)
    assert np.array_equal(kc, bits(st["key_cache"]))
    assert np.array_equal(vc, bits(st["value_cache"]))
    # token_count == 0
    z = torch.zeros(0, 16, dtype=torch.float16)
    kc, _ = oracle.cache_write(z, z, st["key_cache"], st["value_cache"], st["block_table"][:1],
                               torch.tensor([0, 0], dtype=torch.int32), torch.tensor([5], dtype=torch.int32),
                               1, 16, 16)
    assert np.array_equal(kc, bits(st["key_cache"]))


# ------------------------------------------------------------ attention -----

def _paged_from_dense(Ks, Vs, bs, Hk, D, seed=0, extra_blocks=3, shuffle=True):
    """Lay dense per-sequence K/V [L_b, Hk, D] into a pool (test-side layout)."""
    need = [(k.shape[0] + bs - 1) // bs for k in Ks]
    NB = sum(need) + extra_blocks
    g = torch.Generator().manual_seed(seed)
    ids = torch.randperm(NB, generator=g) if shuffle else torch.arange(NB)
    MB = max(need)
    bt = torch.full((len(Ks), MB), -1, dtype=torch.int32)
    kc = torch.full((NB, bs, Hk, D), float("nan"), dtype=torch.float16)
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


def _rand_case(H, Hk, D, bs, past, new, seed=0):
    g = torch.Generator().manual_seed(seed)
    L = [p + n for p, n in zip(past, new)]
    Ks = [torch.randn(l, Hk, D, generator=g).half() for l in L]
    Vs = [torch.randn(l, Hk, D, generator=g).half() for l in L]
    T = sum(new)
    q = torch.randn(T, H * D, generator=g).half()
    cum = torch.tensor([0] + list(np.cumsum(new)), dtype=torch.int32)
    return Ks, Vs, q, cum, torch.tensor(past, dtype=torch.int32)


def _sdpa_reference(q, Ks, Vs, cum, past, H, Hk, D, scale, window=-1, unmapped=None):
    """torch SDPA (fp64) on the dense KV of each sequence."""
    G = H // Hk
    T = q.shape[0]
    out = torch.zeros(T, H, D, dtype=torch.float64)
    for b in range(len(Ks)):
        t0, t1 = int(cum[b]), int(cum[b + 1])
        if t1 == t0:
            continue
        Lb = Ks[b].shape[0]
        qb = q[t0:t1].double().view(t1 - t0, H, D).transpose(0, 1)[None]
        kb = Ks[b].double().transpose(0, 1).repeat_interleave(G, 0)[None]
        vb = Vs[b].double().transpose(0, 1).repeat_interleave(G, 0)[None]
        j = torch.arange(t1 - t0)[:, None]
        p = torch.arange(Lb)[None, :]
        qpos = int(past[b]) + j
        mask = p <= qpos
        if window >= 1:
            mask &= p > qpos - window
        if unmapped is not None and b in unmapped:
            mask &= ~unmapped[b][None, :]
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=scale)
        out[t0:t1] = o[0].transpose(0, 1)
    return out


@pytest.mark.parametrize("H,Hk,D,bs,past,new,window", [
    (4, 4, 16, 16, [0, 7, 33], [3, 1, 2], -1),          # MHA (G = 1)
    (4, 2, 32, 16, [0, 17, 40], [5, 1, 1], -1),         # tiny mixed shape
    (8, 2, 64, 32, [100, 0, 65], [1, 40, 3], -1),       # G = 4, prefill rows
    (8, 2, 16, 16, [100, 0, 65], [1, 40, 3], 7),        # sliding window
    (6, 3, 8, 16, [31, 32, 33], [2, 2, 2], 33),         # window near a block edge
])
def test_attention_matches_sdpa(H, Hk, D, bs, past, new, window):
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, past, new, seed=H + D)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    scale = 1.0 / math.sqrt(D)
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs,
                           0.0, 0.0, window, threads=2)
    ref = _sdpa_reference(q, Ks, Vs, cum, pst, H, Hk, D, scale, window)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_block_permutation_invariance():
    H, Hk, D, bs = 8, 2, 32, 16
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, [50, 3, 90], [1, 4, 2], seed=3)
    outs = []
    for seed in (0, 1, 2):
        kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D, seed=seed)
        outs.append(oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs,
                                     0.0, 0.0, -1))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_constant_v_returns_v():
    H, Hk, D, bs = 4, 2, 16, 16
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, [20, 0], [2, 3], seed=5)
    row = torch.randn(Hk, D).half()
    Vs = [row.expand(v.shape[0], Hk, D).clone() for v in Vs]
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1)
    expect = row.double().repeat_interleave(H // Hk, 0).numpy()
    for t in range(q.shape[0]):
        np.testing.assert_allclose(got[t], expect, rtol=1e-12, atol=1e-12)


def test_one_token_context_and_window_one():
    H, Hk, D, bs = 4, 2, 16, 16
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, [0, 30], [1, 3], seed=6)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1)
    # sequence 0: past 0, one new token -> output is that token's V row
    np.testing.assert_array_equal(got[0], Vs[0][0].double().repeat_interleave(2, 0).numpy())
    # window 1 -> every row returns its own V row
    got1 = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, 1)
    for j in range(3):
        np.testing.assert_array_equal(got1[1 + j], Vs[1][30 + j].double().repeat_interleave(2, 0).numpy())


def test_window_at_least_context_is_full():
    H, Hk, D, bs = 4, 1, 16, 16
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, [10, 45], [3, 1], seed=8)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    full = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1)
    for W in (46, 47, 1000):
        got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, W)
        assert np.array_equal(got, full)
    shorter = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, 45)
    assert not np.array_equal(shorter[3], full[3])  # row with kv_len 46 loses position 0


def test_unmapped_blocks_are_masked():
    H, Hk, D, bs = 4, 2, 16, 16
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, [60, 20], [2, 1], seed=9)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    bt[0, 1] = -1                       # positions 16..31 of sequence 0
    um = {0: (torch.arange(62) >= 16) & (torch.arange(62) < 32)}
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1)
    ref = _sdpa_reference(q, Ks, Vs, cum, pst, H, Hk, D, 1.0 / math.sqrt(D), unmapped=um)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)
    # below-window blocks unmapped: identical to the mapped run (section 9.3)
    kc2, vc2, bt2 = _paged_from_dense(Ks, Vs, bs, Hk, D)
    w_full = oracle.attention(bits(q), bits(kc2), bits(vc2), bt2, cum, pst, H, Hk, D, bs, 0.0, 0.0, 20)
    bt2[0, 0] = -1                      # positions 0..15, below 61 - 20 + 1
    bt2[0, 1] = -1                      # positions 16..31
    w_pruned = oracle.attention(bits(q), bits(kc2), bits(vc2), bt2, cum, pst, H, Hk, D, bs, 0.0, 0.0, 20)
    assert np.array_equal(w_full, w_pruned)


def test_fully_masked_row_outputs_zero():
    H, Hk, D, bs = 2, 1, 16, 16
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, [5, 3], [1, 1], seed=10)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    bt[1, :] = -1
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1)
    assert np.all(got[1] == 0.0) and not np.isnan(got).any()


def test_scale_zero_is_inverse_sqrt_head_size():
    H, Hk, D, bs = 4, 2, 64, 16
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, [9, 30], [2, 1], seed=11)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    a = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.0, 0.0, -1)
    b = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.125, 0.0, -1)
    assert np.array_equal(a, b)
    c = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.3, 0.0, -1)
    ref = _sdpa_reference(q, Ks, Vs, cum, pst, H, Hk, D, 0.3)
    np.testing.assert_allclose(c, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_softcap_large_limit():
    H, Hk, D, bs = 4, 2, 32, 16
    Ks, Vs, q, cum, pst = _rand_case(H, Hk, D, bs, [40, 8], [1, 2], seed=12)
    kc, vc, bt = _paged_from_dense(Ks, Vs, bs, Hk, D)
    ref = _sdpa_reference(q, Ks, Vs, cum, pst, H, Hk, D, 0.25)
    got = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.25, 1e7, -1)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-8, atol=1e-9)
    small = oracle.attention(bits(q), bits(kc), bits(vc), bt, cum, pst, H, Hk, D, bs, 0.25, 0.5, -1)
    assert np.abs(small - ref.numpy()).max() > 1e-3   # a small cap does change the result


def test_softcap_two_key_closed_form():
    # one kv head, D = 8, two cached keys e0 and -e0, q = a*e0:
    # raw scores +-scale*a, capped c = cap*tanh(scale*a/cap), weights are the
    # logistic function of the capped difference 2c.
    D, bs, cap, scale, a = 8, 16, 3.0, 0.5, 6.0
    K = torch.zeros(3, 1, D); K[0, 0, 0] = 1.0; K[1, 0, 0] = -1.0
    V = torch.zeros(3, 1, D); V[0, 0, 1] = 1.0; V[1, 0, 2] = 1.0
    K[2, 0, 0] = 0.0; V[2, 0, 3] = 1.0                   # the new token itself
    q = torch.zeros(1, D); q[0, 0] = a
    kc, vc, bt = _paged_from_dense([K.half()], [V.half()], bs, 1, D)
    cum = torch.tensor([0, 1], dtype=torch.int32)
    past = torch.tensor([2], dtype=torch.int32)
    got = oracle.attention(bits(q.half()), bits(kc), bits(vc), bt, cum, past, 1, 1, D, bs,
                           scale, cap, -1)[0, 0]
    c = cap * math.tanh(scale * a / cap)
    z = math.exp(c) + math.exp(-c) + 1.0
    np.testing.assert_allclose(got[1:4], [math.exp(c) / z, math.exp(-c) / z, 1.0 / z], rtol=1e-14)


# -------------------------------------------------------------- rotary -----

def _complex_rotary(x, pos, cos_t, sin_t, half, interleaved):
    """fp64 rotation by exp(i*angle) using the given cos/sin tables."""
    x = x.astype(np.float64)
    if interleaved:
        z = x[..., 0:2 * half:2] + 1j * x[..., 1:2 * half:2]
    else:
        z = x[..., :half] + 1j * x[..., half:2 * half]
    w = cos_t[pos].astype(np.float64) + 1j * sin_t[pos].astype(np.float64)
    zr = z * w[:, None, :]
    y = x.copy()
    if interleaved:
        y[..., 0:2 * half:2], y[..., 1:2 * half:2] = zr.real, zr.imag
    else:
        y[..., :half], y[..., half:2 * half] = zr.real, zr.imag
    return y


def _ulp16(v):
    a = np.abs(v).astype(np.float64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 10)


@pytest.mark.parametrize("interleaved", [0, 1])
@pytest.mark.parametrize("R", [32, 16])
def test_rotary_matches_complex_rotation(interleaved, R):
    H, D = 3, 32
    past, new = [0, 5, 100], [2, 3, 1]
    T = sum(new)
    cum = torch.tensor([0] + list(np.cumsum(new)), dtype=torch.int32)
    pst = torch.tensor(past, dtype=torch.int32)
    cos_t, sin_t = workloads.rotary_tables(200, R)
    x = torch.randn(T, H * D, generator=torch.Generator().manual_seed(R)).half()
    y = oracle.rotary(bits(x), cum, pst, cos_t, sin_t, H, D, interleaved)
    yv = y.view(np.float16).astype(np.float64).reshape(T, H, D)
    pos = np.concatenate([np.arange(p, p + n) for p, n in zip(past, new)])
    ref = _complex_rotary(x.double().numpy().reshape(T, H, D), pos, cos_t.numpy(), sin_t.numpy(),
                          R // 2, interleaved)
    # fp32 evaluation + one fp16 rounding stays within one fp16 ulp of exact
    assert np.all(np.abs(yv - ref) <= _ulp16(ref) + 1e-12)
    # position 0 is the identity (cos 1, sin 0)
    assert np.array_equal(y[0], bits(x)[0])
    # channels past the rotary dim are copied
    assert np.array_equal(y.reshape(T, H, D)[..., R:], bits(x).reshape(T, H, D)[..., R:])


def test_rotary_relative_position_property():
    # <R(m) q, R(n) k> depends only on m - n (up to fp16 rounding of outputs)
    D, R = 64, 64
    cos_t, sin_t = workloads.rotary_tables(400, R)
    g = torch.Generator().manual_seed(1)
    q = torch.randn(1, D, generator=g).half()
    k = torch.randn(1, D, generator=g).half()

    def rot(x, pos):
        cum = torch.tensor([0, 1], dtype=torch.int32)
        return oracle.rotary(bits(x), cum, torch.tensor([pos], dtype=torch.int32), cos_t, sin_t,
                             1, D, 0).view(np.float16).astype(np.float64)[0]

    base = rot(q, 7) @ rot(k, 3)
    for s in (10, 50, 200):
        other = rot(q, 7 + s) @ rot(k, 3 + s)
        assert abs(other - base) < 0.05 * (1 + abs(base))
    # and it genuinely depends on the offset
    assert abs(rot(q, 7) @ rot(k, 6) - base) > 1e-3


def test_full_forward_tiny_is_finite():
    st = workloads.make_step(workloads.config_shape(0))
    r = oracle.forward(st)
    assert r["out"].shape == (7, 4, 64) and np.isfinite(r["out"]).all()
