"""GPU parity for packed QKV input and QK-Norm ("PagedAttention - CUDA
Design Document", sections 4 and 7): the fused prologue splits packed rows,
normalizes every head of Q and K (fixed fp32 reduction order), rotates and
writes the normalized K; pools bit-exact and output within tolerance of the
oracle, on the decode and both prefill kernels, and over an 8-bit cache."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import check_full, host_copy, make, raw, run

pytestmark = pytest.mark.gpu
cs = workloads.custom_shape

SHAPES = [
    cs("qkn_d128_g4_rotary", 8, 2, 128, 16, [0, 17, 300, 5], [3, 1, 2, 1], do_rotary=1, seed=51),
    cs("qkn_d64_mha", 4, 4, 64, 32, [0, 33, 100], [4, 1, 3], seed=52),
    cs("qkn_d256_window_cap", 4, 2, 256, 64, [700, 64, 5], [1, 1, 2], scale=1 / 16, softcap=50.0,
       local_window_size=100, seed=53),
    cs("qkn_prefill_pair_d128", 8, 2, 128, 32, [0, 40, 7], [300, 1, 129], do_rotary=1, seed=54),
    cs("qkn_prefill_single_d256", 4, 2, 256, 64, [0, 10], [200, 70], seed=55),
]


@pytest.mark.parametrize("mode", ["qk_norm", "packed", "packed_qk_norm"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_fused_prologue_matches_oracle(shape, mode):
    step = make(shape, device="cuda", gen_device="cpu", qk_norm="qk_norm" in mode, packed_qkv="packed" in mode)
    host = host_copy(step)
    _, out, err = run(step)
    assert err == 0
    check_full(host, step, out)


def test_packed_equals_unpacked_bitwise():
    shape = cs("qkn_packed_bitwise", 8, 2, 128, 16, [0, 60, 9], [4, 1, 1], do_rotary=1, seed=56)
    a = make(shape, device="cuda", gen_device="cpu", qk_norm=True)
    b = make(shape, device="cuda", gen_device="cpu", qk_norm=True, packed_qkv=True)
    _, out_a, ea = run(a)
    _, out_b, eb = run(b)
    assert ea == 0 and eb == 0
    assert np.array_equal(raw(a["key_cache"]), raw(b["key_cache"]))
    assert torch.equal(out_a, out_b)


@pytest.mark.parametrize("cache_dtype", [workloads.CACHE_INT8, workloads.CACHE_FP8], ids=["int8", "e4m3"])
def test_qk_norm_packed_over_8bit_cache(cache_dtype):
    shape = cs("qkn_q8", 8, 2, 128, 16, [0, 31, 333], [1, 2, 1], do_rotary=1, seed=57)
    step = make(shape, device="cuda", gen_device="cpu", cache_dtype=cache_dtype,
                quant_type=workloads.QUANT_PER_CHANNEL, head_sink=True, qk_norm=True, packed_qkv=True)
    host = host_copy(step)
    _, out, err = run(step, max_query_len_bound=2)
    assert err == 0
    check_full(host, step, out)


@pytest.mark.parametrize("mode", ["qk_norm", "packed", "packed_qk_norm"])
@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[2], SHAPES[3], SHAPES[4]], ids=lambda s: s.name)
def test_fused_prologue_bf16(shape, mode):
    """The same prologue on bfloat16 rows (bfloat16 weights, one bfloat16
    rounding per normalized and rotated value), on the decode kernel and
    both prefill kernels."""
    step = make(shape, device="cuda", gen_device="cpu", cache_dtype=workloads.CACHE_BF16, qk_norm="qk_norm" in mode,
                packed_qkv="packed" in mode)
    host = host_copy(step)
    _, out, err = run(step)
    assert err == 0
    assert out.dtype == torch.bfloat16
    check_full(host, step, out)
