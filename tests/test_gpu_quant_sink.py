"""GPU parity for the quantized cache and head_sink (CUDA design sections 8
and 6): int8 / e4m3fn pools written bit-exactly (quantize-on-write), decode
over the 8-bit pools at their stored width, and the sink term on every
kernel path (decode single split, split + combine, both prefill kernels).

Bars as everywhere: pools bit-exact, output within 2e-3 + 1e-2 |oracle|.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import check_full, check_sampled, host_copy, make, run

pytestmark = pytest.mark.gpu

cs = workloads.custom_shape
I8, F8 = workloads.CACHE_INT8, workloads.CACHE_FP8
PT, PC = workloads.QUANT_PER_TENSOR, workloads.QUANT_PER_CHANNEL


def _full(shape, options=(), **kw):
    step = make(shape, device="cuda", gen_device="cpu", **kw)
    host = host_copy(step)
    op, out, err = run(step, options=options, max_tokens=step["token_count"],
                       max_query_len_bound=max(shape.new_lens))
    assert err == 0, f"device error {err:#x}"
    check_full(host, step, out)
    return op, out


QUANT_SHAPES = [
    cs("q_d128_g4_bs16", 8, 2, 128, 16, [0, 1, 15, 16, 17, 63, 64, 300], [1] * 8, seed=21),
    cs("q_d128_g8_bs32_multitok", 16, 2, 128, 32, [0, 33, 100, 7], [2, 1, 2, 1], seed=22),
    cs("q_d128_g1_bs64_4tok", 4, 4, 128, 64, [5, 70, 129], [4, 16, 3], seed=23),
    cs("q_d256_g2_bs64_window_cap", 4, 2, 256, 64, [700, 64, 5, 129], [1, 1, 2, 1], scale=1 / 16,
       softcap=50.0, local_window_size=100, seed=24),
    cs("q_d128_g4_rotary", 8, 2, 128, 16, [0, 5, 200, 999], [1, 2, 1, 2], do_rotary=1, seed=25),
    cs("q_d128_g4_bs128_window", 8, 2, 128, 128, [0, 127, 128, 500], [1, 1, 1, 1], local_window_size=64,
       seed=26),
]


@pytest.mark.parametrize("cache_dtype", [I8, F8], ids=["int8", "e4m3"])
@pytest.mark.parametrize("quant_type", [PT, PC], ids=["per_tensor", "per_channel"])
@pytest.mark.parametrize("shape", QUANT_SHAPES, ids=lambda s: s.name)
def test_quantized_decode_matches_oracle(shape, cache_dtype, quant_type):
    _full(shape, cache_dtype=cache_dtype, quant_type=quant_type)


@pytest.mark.parametrize("cache_dtype", [I8, F8], ids=["int8", "e4m3"])
@pytest.mark.parametrize("split_keys", [64, 128])
def test_quantized_split_merge(cache_dtype, split_keys):
    shape = cs("q_splits", 8, 2, 128, 16, [1000, 70, 2047, 300], [1, 1, 1, 2], seed=27)
    _full(shape, options=[(pa.PA_OPT_SPLIT_KEYS, split_keys)], cache_dtype=cache_dtype, quant_type=PC,
          head_sink=True)


@pytest.mark.parametrize("cache_dtype", [I8, F8], ids=["int8", "e4m3"])
def test_quantized_with_sink(cache_dtype):
    shape = cs("q_sink", 8, 2, 256, 16, [0, 31, 333], [1, 2, 1], seed=28)
    _full(shape, cache_dtype=cache_dtype, quant_type=PT, head_sink=True)


def test_quantized_cache_write_alone_is_bit_exact():
    shape = cs("q_write", 8, 2, 128, 16, [3, 40, 0], [1, 1, 2], do_rotary=1, seed=29)
    step = make(shape, device="cuda", gen_device="cpu", cache_dtype=F8, quant_type=PC)
    host = host_copy(step)
    op = pa.PagedAttention.for_step(step, max_query_len_bound=2)
    op.cache_write(step)
    torch.cuda.synchronize()
    assert op.device_error() == 0
    import oracle
    from gpu_util import raw
    k = oracle.rotary(host["key"], host["cumulative_sequence_lengths"], host["past_sequence_lengths"],
                      host["cos_cache"], host["sin_cache"], 2, 128, 0)
    kc, vc = oracle.cache_write(k, host["value"], host["key_cache"], host["value_cache"], host["block_table"],
                                host["cumulative_sequence_lengths"], host["past_sequence_lengths"], 2, 128, 16,
                                cache_dtype=F8, k_scale=host["k_scale"], v_scale=host["v_scale"],
                                per_channel=True)
    assert np.array_equal(raw(step["key_cache"]), raw(kc)) and np.array_equal(raw(step["value_cache"]), raw(vc))


@pytest.mark.parametrize("index", [1])
def test_full_size_quantized_decode_config(index):
    """Llama-3-8B-shaped decode over an e4m3fn per-channel cache with sinks (sampled rows)."""
    shape = workloads.config_shape(index)
    step = make(shape, device="cuda", gen_device="cpu", cache_dtype=F8, quant_type=PC, head_sink=True)
    host = host_copy(step)
    op, out, err = run(step, max_query_len_bound=1)
    assert err == 0
    check_sampled(host, step, out)


# ------------------------------------------------------------- head_sink on fp16

SINK_SHAPES = [
    cs("sink_decode_single_split", 8, 2, 128, 16, [0, 15, 300], [1, 1, 1], seed=31),
    cs("sink_d64_multitok", 4, 4, 64, 32, [0, 33, 100], [4, 1, 3], seed=32),
    cs("sink_prefill_pair_d128", 8, 2, 128, 32, [0, 40, 7], [300, 1, 129], seed=33),
    cs("sink_prefill_single_d256", 4, 2, 256, 64, [0, 10], [200, 70], softcap=30.0, seed=34),
    cs("sink_window", 8, 2, 128, 16, [500, 0], [1, 90], local_window_size=64, seed=35),
]


@pytest.mark.parametrize("shape", SINK_SHAPES, ids=lambda s: s.name)
def test_head_sink_fp16_paths(shape):
    step = make(shape, device="cuda", gen_device="cpu", head_sink=True)
    host = host_copy(step)
    op, out, err = run(step)
    assert err == 0
    check_full(host, step, out)


def test_head_sink_split_combine():
    shape = cs("sink_splits", 8, 2, 128, 16, [1000, 2047], [1, 1], seed=36)
    step = make(shape, device="cuda", gen_device="cpu", head_sink=True)
    host = host_copy(step)
    op, out, err = run(step, options=[(pa.PA_OPT_SPLIT_KEYS, 128)])
    assert err == 0
    check_full(host, step, out)


# ------------------------------------------------------------- host rules on a live handle

def test_scales_required_and_routing_locked():
    shape = cs("q_rules", 8, 2, 128, 16, [10], [1], seed=37)
    step = make(shape, device="cuda", gen_device="cpu", cache_dtype=I8, quant_type=PT)
    op = pa.PagedAttention.for_step(step, max_query_len_bound=1)
    out = torch.empty_like(step["query"])
    no_scales = dict(step, k_scale=None)
    with pytest.raises(pa.PAError) as e:
        op.forward(no_scales, out)
    assert e.value.status == pa.PA_INVALID_ARGUMENT
    with pytest.raises(pa.PAError) as e:
        op.set_option(pa.PA_OPT_DECODE_MAX_ROWS, 4)
    assert e.value.status == pa.PA_NOT_SUPPORTED


@pytest.mark.parametrize("cache_dtype", [I8, F8], ids=["int8", "e4m3"])
@pytest.mark.parametrize("quant_type", [PT, PC], ids=["per_tensor", "per_channel"])
def test_quantized_rotary_at_an_offset(cache_dtype, quant_type):
    """Rotary over channels [32, 96) of head_size 128 (rotary_offset 32,
    rotary_dim 64): the quantized K rows and the scaled query copy rotate
    the same channels the oracle does."""
    shape = cs("q_rotary_offset", 8, 2, 128, 16, [3, 90, 400], [1, 2, 1], do_rotary=1, rotary_dim=64, seed=29)
    step = make(shape, device="cuda", gen_device="cpu", cache_dtype=cache_dtype, quant_type=quant_type)
    step["rotary_offset"] = 32
    host = host_copy(step)
    op, out, err = run(step, max_tokens=step["token_count"], max_query_len_bound=2)
    assert err == 0, f"device error {err:#x}"
    check_full(host, step, out)


QUANT_PROMPTS = [
    # q_len * G > 16: the rows run through the decode kernel in chunks of
    # 16 / G tokens, each chunk attending causally from its first token
    cs("q_prompt_d128_g4", 8, 2, 128, 16, [0, 70, 300, 5], [40, 1, 17, 3], seed=31),
    cs("q_prompt_d128_g8_bs32", 16, 2, 128, 32, [0, 33], [25, 9], seed=32),
    cs("q_prompt_d256_g2_window_cap", 4, 2, 256, 64, [0, 100], [60, 11], scale=1 / 16, softcap=50.0,
       local_window_size=45, seed=33),
    cs("q_prompt_d128_g1_rotary", 4, 4, 128, 16, [0, 9], [50, 20], do_rotary=1, seed=34),
]


@pytest.mark.parametrize("cache_dtype", [I8, F8], ids=["int8", "e4m3"])
@pytest.mark.parametrize("quant_type", [PT, PC], ids=["per_tensor", "per_channel"])
@pytest.mark.parametrize("shape", QUANT_PROMPTS, ids=lambda s: s.name)
def test_quantized_prompt_rows_match_oracle(shape, cache_dtype, quant_type):
    """Prompt and mixed steps over 8-bit pools (every token of a quantized
    cache goes through the decode kernel, which reads the codes at their
    stored width)."""
    op, _ = _full(shape, cache_dtype=cache_dtype, quant_type=quant_type, head_sink=True)
    counts = op.last_step_counts()
    assert counts["n_pre"] == 0


@pytest.mark.parametrize("split_keys", [64, 0])
def test_quantized_prompt_rows_with_splits(split_keys):
    shape = cs("q_prompt_splits", 8, 2, 128, 16, [0, 1500, 600], [64, 1, 8], seed=35)
    _full(shape, options=[(pa.PA_OPT_SPLIT_KEYS, split_keys)], cache_dtype=F8, quant_type=PC)


def test_quantized_prompt_rows_large_batch():
    """More sequences than one work-list block (the multi-pass builder)."""
    import numpy as np
    rng = np.random.default_rng(36)
    B = 1030
    new = [1] * B
    for b in rng.choice(B, 12, replace=False):
        new[b] = int(rng.integers(5, 40))
    shape = cs("q_prompt_b1030", 8, 2, 128, 16, rng.integers(0, 60, B), new, seed=36)
    _full(shape, cache_dtype=I8, quant_type=PT)
