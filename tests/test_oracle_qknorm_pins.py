"""Pins for the oracle's QK-Norm and packed-QKV split ("PagedAttention -
CUDA Design Document", sections 7 and 4), each against something other than
the oracle:

  * QK-Norm       -> torch.nn.functional.rms_norm in fp64, within one fp16 ulp
                     (the fp32 sum of squares may round the other way);
                     bit for bit against numpy's float32 arithmetic with the
                     sum of squares as one running sum in channel order
                     (np.add.accumulate), on random rows and on rows built so
                     that the order of the sum (or an fp64 sum) changes the
                     fp16 result; constant rows against the closed form
                     a / sqrt(a^2 + eps); with eps = 0 a power-of-two scaling
                     of a row leaves its output bit-identical
  * packed QKV    -> a step whose query rows hold [Q | K | V] gives the same
                     pools and output as the unpacked step
"""

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import workloads


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_qk_norm_matches_torch_rms_norm():
    g = torch.Generator().manual_seed(1)
    for D, nh in ((64, 3), (128, 4), (256, 2)):
        x = (torch.randn(7, nh * D, generator=g) * (0.1 + 3 * torch.rand(7, 1, generator=g))).half()
        w = (1 + 0.5 * torch.randn(D, generator=g)).half()
        got = oracle.qk_norm(_bits(x), nh, D, _bits(w), 1e-6).view(np.float16).astype(np.float64)
        ref = F.rms_norm(x.double().view(7, nh, D), (D,), w.double(), eps=1e-6).view(7, nh * D)
        ref16 = ref.half().double().numpy()
        ulp = np.spacing(np.abs(ref16).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(got - ref16) <= ulp), np.max(np.abs(got - ref16) / ulp)


def _np_qk_norm(x16, w16, eps, reverse=False, acc=np.float32):
    """The plain fp32 definition in numpy: squares in float32, one running
    sum over the channels (reverse: from the last channel; acc: the sum's
    type), mean = sum * (1/D), r = 1 / sqrt(mean + eps), y = (x * r) * w."""
    D = x16.shape[-1]
    x = x16.astype(np.float32)
    sq = x * x
    if reverse:
        sq = sq[..., ::-1]
    s = np.add.accumulate(sq.astype(acc), axis=-1, dtype=acc)[..., -1].astype(np.float32)
    mean = s * np.float32(1.0 / D)
    r = np.float32(1.0) / np.sqrt(mean + np.float32(eps))
    return ((x * r[..., None]) * w16.astype(np.float32)).astype(np.float16)


def test_qk_norm_bitwise_against_numpy_running_sum():
    rng = np.random.default_rng(3)
    for D in (64, 128, 256):
        x = (rng.standard_normal((40, D)) * rng.uniform(0.05, 8.0, (40, 1))).astype(np.float16)
        w = (1 + 0.5 * rng.standard_normal(D)).astype(np.float16)
        got = oracle.qk_norm(x.view(np.uint16), 1, D, w.view(np.uint16), 1e-6).view(np.float16).reshape(40, D)
        assert np.array_equal(got.view(np.uint16), _np_qk_norm(x, w, 1e-6).view(np.uint16))


def test_qk_norm_sum_order_decides_rows_built_for_it():
    # One channel near the fp16 maximum among many small ones: its square is
    # about 2^32, where an fp32 ulp is 512, so the small squares (< 256)
    # vanish into the running sum once the large one is in it, and add up
    # when they come first; an fp64 sum keeps them all.  The rows kept are
    # those where numpy's three sums give different fp16 outputs.
    rng = np.random.default_rng(4)
    D = 256
    rows, n_order, n_f64 = [], 0, 0
    for _ in range(300):
        x = (rng.uniform(12.0, 15.9, D) * rng.choice([-1.0, 1.0], D)).astype(np.float16)
        x[rng.integers(0, 4)] = rng.choice([60000.0, 62000.0, 65504.0]) * rng.choice([-1.0, 1.0])
        w = rng.uniform(0.5, 1.5, D).astype(np.float16)
        plain = _np_qk_norm(x, w, 1e-6)
        rev = _np_qk_norm(x, w, 1e-6, reverse=True)
        f64 = _np_qk_norm(x, w, 1e-6, acc=np.float64)
        if not np.array_equal(plain, rev) or not np.array_equal(plain, f64):
            n_order += not np.array_equal(plain, rev)
            n_f64 += not np.array_equal(plain, f64)
            rows.append((x, w, plain))
    assert n_order >= 5 and n_f64 >= 5, (n_order, n_f64)
    for x, w, plain in rows:
        got = oracle.qk_norm(x.view(np.uint16)[None], 1, D, w.view(np.uint16), 1e-6).view(np.float16)
        assert np.array_equal(got.reshape(D).view(np.uint16), plain.view(np.uint16))


def test_qk_norm_constant_rows_closed_form():
    D = 128
    for a in (2.0, -0.375, 17.0, 1e-3):
        x = torch.full((1, D), a).half()
        w = torch.ones(D).half()
        got = oracle.qk_norm(_bits(x), 1, D, _bits(w), 1e-6).view(np.float16)
        a16 = float(x[0, 0])
        ref = np.float16(a16 / np.sqrt(a16 * a16 + 1e-6))
        assert np.all(got == ref), (a, got[0], ref)


def test_qk_norm_scale_invariance_without_eps():
    g = torch.Generator().manual_seed(2)
    D, nh = 128, 2
    x = torch.randn(5, nh * D, generator=g).half()
    w = torch.randn(D, generator=g).half()
    a = oracle.qk_norm(_bits(x), nh, D, _bits(w), 0.0)
    b = oracle.qk_norm(_bits(x * 4), nh, D, _bits(w), 0.0)
    assert np.array_equal(a, b)


def test_packed_qkv_equals_unpacked():
    shape = workloads.custom_shape("packed", 8, 2, 64, 16, [0, 17, 40], [5, 1, 2], do_rotary=1, seed=9)
    step = workloads.make_step(shape)
    packed = dict(step, query=torch.cat([step["query"], step["key"], step["value"]], dim=1), key=None, value=None)
    a = oracle.forward(step)
    b = oracle.forward(packed)
    assert np.array_equal(a["key_cache"], b["key_cache"]) and np.array_equal(a["value_cache"], b["value_cache"])
    assert np.array_equal(a["out"], b["out"])
