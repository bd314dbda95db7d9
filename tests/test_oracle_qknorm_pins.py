"""Pins for the oracle's QK-Norm and packed-QKV split ("PagedAttention -
CUDA Design Document", sections 7 and 4), each against something other than
the oracle:

  * QK-Norm       -> torch.nn.functional.rms_norm in fp64, within one fp16 ulp
                     (the oracle's fixed fp32 summation order may round the
                     other way); constant rows against the closed form
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
