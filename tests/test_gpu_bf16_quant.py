"""GPU parity of bfloat16 activations over int8 / e4m3fn caches (the kernel
is registered for fp16 and bfloat16 activations with int8 and float8 caches,
"PagedAttention - CUDA Design Document", section 8.2) against the CPU oracle.

Bars: both 8-bit pools bit-exact (the codes of the bfloat16 values, after
QK-Norm and rotary in bfloat16); the bfloat16 output within
|gpu - oracle| <= 2^-6 + 1e-2 |oracle| (the 8-bit path's contraction bound
with the bfloat16 output rounding; tests/gpu_util.py).  The cases cover the
decode kernel over codes (head sizes 128 and 256, GQA 1 to 16), prompt rows
in chunks, split-KV with the combine kernel, rotary (the bfloat16 query
rotated, then copied as fp16), per-tensor and per-channel scales, head_sink,
packed QKV with QK-Norm, and the Llama-3-8B-shaped decode at full size.
"""

import pytest
import torch

import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import check_full, check_sampled, host_copy, make, run

pytestmark = pytest.mark.gpu

cs = workloads.custom_shape
I8, F8 = workloads.CACHE_INT8, workloads.CACHE_FP8
PT, PC = workloads.QUANT_PER_TENSOR, workloads.QUANT_PER_CHANNEL
DT = pytest.mark.parametrize("cache_dtype", [I8, F8], ids=["int8", "e4m3"])
QT = pytest.mark.parametrize("quant_type", [PT, PC], ids=["per_tensor", "per_channel"])


def _full(shape, options=(), **kw):
    step = make(shape, device="cuda", gen_device="cpu", act_bf16=True, **kw)
    assert step["query"].dtype == torch.bfloat16 and step["key_cache"].dtype == torch.uint8
    host = host_copy(step)
    op, out, err = run(step, options=options, max_tokens=step["token_count"],
                       max_query_len_bound=max(shape.new_lens))
    assert out.dtype == torch.bfloat16
    assert err == 0, f"device error {err:#x}"
    check_full(host, step, out)
    return op, out


SHAPES = [
    cs("bq_d128_g4_bs16", 8, 2, 128, 16, [0, 1, 15, 16, 17, 63, 64, 300], [1] * 8, seed=121),
    cs("bq_d128_g8_bs32_multitok", 16, 2, 128, 32, [0, 33, 100, 7], [2, 1, 2, 1], seed=122),
    cs("bq_d256_g2_bs64_window_cap", 4, 2, 256, 64, [700, 64, 5, 129], [1, 1, 2, 1], scale=1 / 16,
       softcap=50.0, local_window_size=100, seed=123),
    cs("bq_d128_g4_rotary", 8, 2, 128, 16, [0, 5, 200, 999], [1, 2, 1, 2], do_rotary=1, seed=124),
    cs("bq_d128_g1_prompts", 4, 4, 128, 64, [5, 70, 0], [4, 16, 37], seed=125),
]


@DT
@QT
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_bf16_over_codes_matches_oracle(shape, cache_dtype, quant_type):
    _full(shape, cache_dtype=cache_dtype, quant_type=quant_type)


@DT
def test_bf16_over_codes_split_combine_with_sink(cache_dtype):
    shape = cs("bq_splits", 8, 2, 128, 16, [1000, 70, 2047, 300], [1, 1, 1, 2], seed=126)
    _full(shape, options=[(pa.PA_OPT_SPLIT_KEYS, 64)], cache_dtype=cache_dtype, quant_type=PC,
          head_sink=True)


@DT
def test_bf16_over_codes_sink_single_split(cache_dtype):
    shape = cs("bq_sink", 8, 2, 256, 16, [0, 31, 333], [1, 2, 1], seed=127)
    _full(shape, cache_dtype=cache_dtype, quant_type=PT, head_sink=True)


@DT
def test_bf16_over_codes_packed_qk_norm_rotary(cache_dtype):
    shape = cs("bq_packed_norm", 16, 4, 128, 16, [0, 40, 300], [3, 1, 9], do_rotary=1, seed=128)
    _full(shape, cache_dtype=cache_dtype, quant_type=PC, packed_qkv=True, qk_norm=True)


@DT
def test_bf16_over_codes_full_size_decode_config(cache_dtype):
    """The Llama-3-8B-shaped decode (64 sequences, 512..4096 context) with
    bfloat16 activations over 8-bit pools: pools in full, sampled rows."""
    shape = workloads.config_shape(1)
    step = make(shape, device="cuda", gen_device="cuda", cache_dtype=cache_dtype, quant_type=PT,
                act_bf16=True)
    host = host_copy(step)
    op, out, err = run(step)
    assert err == 0, f"device error {err:#x}"
    check_sampled(host, step, out, n_rows=160)


def test_bf16_over_codes_is_not_read_as_fp16():
    """The same draws with fp16 and with bfloat16 activations give different
    pools and outputs, each matching its own oracle."""
    shape = SHAPES[0]
    _, out_bf = _full(shape, cache_dtype=I8, quant_type=PT)
    step = make(shape, device="cuda", gen_device="cpu", cache_dtype=I8, quant_type=PT)
    host = host_copy(step)
    _, out_h, err = run(step)
    assert err == 0
    check_full(host, step, out_h)
    assert not torch.equal(out_bf.float(), out_h.float())
