"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point include/pa.h declares, and rejects each
invalid configuration / step with a message naming the argument (one test
per validation rule, "PagedAttention - CUDA Design Document" sections 15
and 17.5)."""

import ctypes
import os
import re

import pytest

import paged_kv_cache_reshape_gb300 as pa
from paged_kv_cache_reshape_gb300 import builder as pabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    pabuild.build()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    return sorted(set(re.findall(r"^PA_API\s+[\w\s\*]*?\b(pa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_binding_names():
    assert declared_symbols() == sorted(pa.EXPORTED)


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(pa.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(L, name), name


def good(**over):
    c = pa.make_config(32, 8, 128, 16, 1000, 257, 64, 64)
    for k, v in over.items():
        setattr(c, k, v)
    return c


def test_valid_config_passes():
    assert pa.pa_validate_config(good()) == (pa.PA_OK, "ok")


@pytest.mark.parametrize("field,value,status,word", [
    ("num_heads", 0, pa.PA_INVALID_ARGUMENT, "num_heads"),
    ("kv_num_heads", 0, pa.PA_INVALID_ARGUMENT, "kv_num_heads"),
    ("num_heads", 30, pa.PA_INVALID_ARGUMENT, "num_heads % kv_num_heads"),
    ("head_size", 100, pa.PA_INVALID_ARGUMENT, "head_size"),
    ("block_size", 8, pa.PA_INVALID_ARGUMENT, "block_size"),
    ("block_size", 48, pa.PA_INVALID_ARGUMENT, "block_size"),
    ("num_blocks", 0, pa.PA_INVALID_ARGUMENT, "num_blocks"),
    ("max_blocks_per_seq", 0, pa.PA_INVALID_ARGUMENT, "max_blocks_per_seq"),
    ("scale", -1.0, pa.PA_INVALID_ARGUMENT, "scale"),
    ("softcap", -0.5, pa.PA_INVALID_ARGUMENT, "softcap"),
    ("local_window_size", 0, pa.PA_INVALID_ARGUMENT, "local_window_size"),
    ("local_window_size", -2, pa.PA_INVALID_ARGUMENT, "local_window_size"),
    ("do_rotary", 2, pa.PA_INVALID_ARGUMENT, "do_rotary"),
    ("rotary_interleaved", 3, pa.PA_INVALID_ARGUMENT, "rotary_interleaved"),
    ("max_batch", 0, pa.PA_INVALID_ARGUMENT, "max_batch"),
    ("max_tokens", 0, pa.PA_INVALID_ARGUMENT, "max_tokens"),
    ("max_kv_len_bound", -1, pa.PA_INVALID_ARGUMENT, "max_kv_len_bound"),
    ("head_size", 96, pa.PA_NOT_SUPPORTED, "head_size"),
])
def test_config_rule(field, value, status, word):
    st, msg = pa.pa_validate_config(good(**{field: value}))
    assert st == status and word in msg, (st, msg)


@pytest.mark.parametrize("over,status,word", [
    (dict(cache_dtype=4), pa.PA_INVALID_ARGUMENT, "cache_dtype"),
    (dict(cache_dtype=-1), pa.PA_INVALID_ARGUMENT, "cache_dtype"),
    (dict(k_quant_type=4), pa.PA_INVALID_ARGUMENT, "k_quant_type"),
    (dict(k_quant_type=pa.PA_QUANT_PER_TENSOR, v_quant_type=pa.PA_QUANT_PER_TENSOR),
     pa.PA_INVALID_ARGUMENT, "16-bit cache"),
    (dict(cache_dtype=pa.PA_CACHE_BF16, k_quant_type=pa.PA_QUANT_PER_TENSOR, v_quant_type=pa.PA_QUANT_PER_TENSOR),
     pa.PA_INVALID_ARGUMENT, "16-bit cache"),
    (dict(cache_dtype=pa.PA_CACHE_INT8), pa.PA_INVALID_ARGUMENT, "8-bit cache needs"),
    (dict(cache_dtype=pa.PA_CACHE_INT8, k_quant_type=pa.PA_QUANT_PER_TENSOR,
          v_quant_type=pa.PA_QUANT_PER_CHANNEL, max_query_len_bound=1), pa.PA_NOT_SUPPORTED, "must match"),
    (dict(cache_dtype=pa.PA_CACHE_FP8_E4M3, k_quant_type=pa.PA_QUANT_PER_TENSOR,
          v_quant_type=pa.PA_QUANT_PER_TENSOR, head_size=64, max_query_len_bound=1), pa.PA_NOT_SUPPORTED,
     "head_size"),
    (dict(cache_dtype=pa.PA_CACHE_FP8_E4M3, k_quant_type=pa.PA_QUANT_PER_TENSOR,
          v_quant_type=pa.PA_QUANT_PER_TENSOR, num_heads=64, kv_num_heads=2), pa.PA_NOT_SUPPORTED,
     "num_heads / kv_num_heads <= 16"),
])
def test_quantized_cache_rules(over, status, word):
    st, msg = pa.pa_validate_config(good(**over))
    assert st == status and word in msg, (st, msg)


def test_bf16_config_passes_and_latent_rejects_it():
    assert pa.pa_validate_config(good(cache_dtype=pa.PA_CACHE_BF16)) == (pa.PA_OK, "ok")
    assert pa.pa_validate_config(good(cache_dtype=pa.PA_CACHE_BF16, packed_qkv=1, qk_norm=1)) == (pa.PA_OK, "ok")
    cfg = pa.make_config(128, 1, 576, 64, 100, 8, 4, 4, scale=0.1, cache_dtype=pa.PA_CACHE_BF16,
                         kv_cache_layout=pa.PA_LAYOUT_LATENT, v_head_size=512)
    st, msg = pa.pa_validate_config(cfg)
    assert st == pa.PA_NOT_SUPPORTED and "fp16" in msg, (st, msg)


Q8 = dict(cache_dtype=pa.PA_CACHE_INT8, k_quant_type=pa.PA_QUANT_PER_TENSOR, v_quant_type=pa.PA_QUANT_PER_TENSOR)


def test_bf16_activation_rules():
    """act_dtype: bfloat16 activations go with an 8-bit or a bfloat16 cache."""
    for cdt in (pa.PA_CACHE_INT8, pa.PA_CACHE_FP8_E4M3):
        for qt in (pa.PA_QUANT_PER_TENSOR, pa.PA_QUANT_PER_CHANNEL):
            assert pa.pa_validate_config(good(cache_dtype=cdt, k_quant_type=qt, v_quant_type=qt,
                                              act_dtype=pa.PA_ACT_BF16)) == (pa.PA_OK, "ok")
    assert pa.pa_validate_config(good(act_dtype=pa.PA_ACT_BF16, packed_qkv=1, qk_norm=1, **Q8)) == (pa.PA_OK, "ok")
    assert pa.pa_validate_config(good(cache_dtype=pa.PA_CACHE_BF16, act_dtype=pa.PA_ACT_BF16)) == (pa.PA_OK, "ok")
    st, msg = pa.pa_validate_config(good(act_dtype=pa.PA_ACT_BF16))
    assert st == pa.PA_INVALID_ARGUMENT and "PA_CACHE_BF16" in msg, (st, msg)
    for bad in (2, -1):
        st, msg = pa.pa_validate_config(good(act_dtype=bad, **Q8))
        assert st == pa.PA_INVALID_ARGUMENT and "act_dtype" in msg, (st, msg)


def test_no_alloc_rejects_bf16_activations():
    a = step_args()
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731
    cfg = good(act_dtype=pa.PA_ACT_BF16, **Q8)
    assert pa.pa_validate_config(cfg) == (pa.PA_OK, "ok")
    st = pa.lib().pa_forward_no_alloc(ctypes.byref(cfg), P(a["query"]), P(a["key"]),
                                      P(a["value"]), P(a["key_cache"]), P(a["value_cache"]), P(a["block_table"]),
                                      P(a["cumulative_sequence_lengths"]), P(a["past_sequence_lengths"]), 4, 4,
                                      None, None, P(a["output"]), None, ctypes.c_void_p(0))
    assert st == pa.PA_NOT_SUPPORTED


@pytest.mark.parametrize("over,status,word", [
    (dict(packed_qkv=2), pa.PA_INVALID_ARGUMENT, "packed_qkv"),
    (dict(qk_norm=3), pa.PA_INVALID_ARGUMENT, "qk_norm"),
    (dict(qk_norm=1, qk_norm_epsilon=0.0), pa.PA_INVALID_ARGUMENT, "qk_norm_epsilon"),
    (dict(qk_norm=1, qk_norm_epsilon=-1e-6), pa.PA_INVALID_ARGUMENT, "qk_norm_epsilon"),
    (dict(qk_norm=1, num_heads=64, kv_num_heads=64), pa.PA_NOT_SUPPORTED, "kv_num_heads <= 32"),
])
def test_packed_and_qk_norm_rules(over, status, word):
    st, msg = pa.pa_validate_config(good(**over))
    assert st == status and word in msg, (st, msg)


def test_packed_qkv_wants_no_key_or_value():
    cfg = good(packed_qkv=1)
    st, msg = pa.pa_check_step(cfg, **step_args())
    assert st == pa.PA_INVALID_ARGUMENT and "packed_qkv" in msg, msg
    assert pa.pa_check_step(cfg, **step_args(key=None, value=None))[0] == pa.PA_OK
    # the cache write alone still takes key and value
    assert pa.pa_check_step(cfg, **step_args(for_forward=0, query=None, output=None))[0] == pa.PA_OK


def latent(**over):
    c = pa.make_config(16, 1, 576, 64, 1000, 65, 32, 32, scale=0.07, kv_cache_layout=pa.PA_LAYOUT_LATENT,
                       v_head_size=512, max_query_len_bound=1)
    for k, v in over.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("over,status,word", [
    (dict(kv_cache_layout=2), pa.PA_INVALID_ARGUMENT, "kv_cache_layout"),
    (dict(kv_num_heads=2), pa.PA_INVALID_ARGUMENT, "kv_num_heads == 1"),
    (dict(scale=0.0), pa.PA_INVALID_ARGUMENT, "explicit scale"),
    (dict(v_head_size=600), pa.PA_INVALID_ARGUMENT, "v_head_size"),
    (dict(qk_norm=1), pa.PA_INVALID_ARGUMENT, "qk_norm"),
    (dict(rotary_offset=4), pa.PA_INVALID_ARGUMENT, "rotary_offset"),
    (dict(do_rotary=1, rotary_dim=64, rotary_offset=528, max_rotary_positions=100), pa.PA_INVALID_ARGUMENT,
     "rotary_offset"),
    (dict(cache_dtype=pa.PA_CACHE_FP8_E4M3, k_quant_type=1, v_quant_type=1), pa.PA_NOT_SUPPORTED, "latent"),
    (dict(head_size=512, v_head_size=448), pa.PA_NOT_SUPPORTED, "576"),
    (dict(num_heads=24), pa.PA_NOT_SUPPORTED, "multiple of 16"),
])
def test_latent_rules(over, status, word):
    st, msg = pa.pa_validate_config(latent(**over))
    assert st == status and word in msg, (st, msg)


def test_latent_config_passes_and_separate_rejects_other_v_width():
    assert pa.pa_validate_config(latent())[0] == pa.PA_OK
    assert pa.pa_validate_config(latent(num_heads=128))[0] == pa.PA_OK
    st, msg = pa.pa_validate_config(good(v_head_size=64))
    assert st == pa.PA_INVALID_ARGUMENT and "LATENT" in msg


def test_latent_step_wants_no_value():
    cfg = latent()
    st, msg = pa.pa_check_step(cfg, **step_args())
    assert st == pa.PA_INVALID_ARGUMENT and "LATENT" in msg
    assert pa.pa_check_step(cfg, **step_args(value=None, value_cache=None))[0] == pa.PA_OK


def test_no_alloc_rejects_latent_layout():
    """The handle-less entry point runs the separate K/V layout only; a latent
    step is refused on the host, before any device work."""
    a = step_args(value=None, value_cache=None)
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731
    st = pa.lib().pa_forward_no_alloc(ctypes.byref(latent()), P(a["query"]), P(a["key"]), None,
                                      P(a["key_cache"]), None, P(a["block_table"]),
                                      P(a["cumulative_sequence_lengths"]), P(a["past_sequence_lengths"]), 4, 4,
                                      None, None, P(a["output"]), None, ctypes.c_void_p(0))
    assert st == pa.PA_NOT_SUPPORTED
    assert "latent" in pa.lib().pa_last_error_message(None).decode()


def test_no_alloc_rejects_bf16_cache():
    a = step_args()
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731
    st = pa.lib().pa_forward_no_alloc(ctypes.byref(good(cache_dtype=pa.PA_CACHE_BF16)), P(a["query"]), P(a["key"]),
                                      P(a["value"]), P(a["key_cache"]), P(a["value_cache"]), P(a["block_table"]),
                                      P(a["cumulative_sequence_lengths"]), P(a["past_sequence_lengths"]), 4, 4,
                                      None, None, P(a["output"]), None, ctypes.c_void_p(0))
    assert st == pa.PA_NOT_SUPPORTED
    assert "bfloat16" in pa.lib().pa_last_error_message(None).decode()


def test_quantized_decode_config_passes():
    for cdt in (pa.PA_CACHE_INT8, pa.PA_CACHE_FP8_E4M3):
        for qt in (pa.PA_QUANT_PER_TENSOR, pa.PA_QUANT_PER_CHANNEL):
            st, msg = pa.pa_validate_config(good(cache_dtype=cdt, k_quant_type=qt, v_quant_type=qt,
                                                 max_query_len_bound=4))
            assert st == pa.PA_OK, msg


def test_rotary_rules():
    st, msg = pa.pa_validate_config(good(do_rotary=1, max_rotary_positions=0))
    assert st == pa.PA_INVALID_ARGUMENT and "max_rotary_positions" in msg
    st, msg = pa.pa_validate_config(good(do_rotary=1, max_rotary_positions=100, rotary_dim=130))
    assert st == pa.PA_INVALID_ARGUMENT and "rotary_dim" in msg
    st, msg = pa.pa_validate_config(good(do_rotary=1, max_rotary_positions=100, rotary_dim=24))
    assert st == pa.PA_NOT_SUPPORTED and "rotary_dim" in msg
    assert pa.pa_validate_config(good(do_rotary=1, max_rotary_positions=100))[0] == pa.PA_OK


A = 1 << 20  # a fake, suitably aligned "device address" (never dereferenced)


def step_args(**over):
    d = dict(for_forward=1, query=A, key=A + 4096, value=A + 8192, key_cache=A + 16384,
             value_cache=A + 32768, block_table=A + 65536, cumulative_sequence_lengths=A + 70000,
             past_sequence_lengths=A + 80000, batch=4, token_count=4, cos_cache=None,
             sin_cache=None, output=A + 90000)
    d.update(over)
    return d


def check(cfg=None, **over):
    return pa.pa_check_step(cfg or good(), **step_args(**over))


def test_valid_step_passes():
    assert check() == (pa.PA_OK, "ok")


@pytest.mark.parametrize("over,word", [
    (dict(batch=0), "batch"),
    (dict(batch=65), "batch"),
    (dict(token_count=-1), "token_count"),
    (dict(token_count=65), "token_count"),
    (dict(query=None), "query"),
    (dict(output=None), "output"),
    (dict(key=None), "key"),
    (dict(value=None), "value"),
    (dict(key_cache=None), "key_cache"),
    (dict(block_table=None), "block_table"),
    (dict(cumulative_sequence_lengths=None), "cumulative_sequence_lengths"),
    (dict(past_sequence_lengths=None), "past_sequence_lengths"),
    (dict(query=A + 2), "aligned"),
    (dict(value_cache=A + 16384), "distinct"),
    (dict(cos_cache=A + 100000), "both present"),
    (dict(cos_cache=A + 100000, sin_cache=A + 110000), "do_rotary == 0"),
])
def test_step_rule(over, word):
    st, msg = check(**over)
    assert st == pa.PA_INVALID_ARGUMENT and word in msg, (st, msg)


def test_rotary_tables_required():
    cfg = good(do_rotary=1, max_rotary_positions=100)
    st, msg = check(cfg)
    assert st == pa.PA_INVALID_ARGUMENT and "required" in msg
    assert check(cfg, cos_cache=A + 100000, sin_cache=A + 110000)[0] == pa.PA_OK


def test_cache_write_needs_no_query_or_output():
    assert check(for_forward=0, query=None, output=None)[0] == pa.PA_OK


def test_create_without_gpu_reports_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(pa.PAError) as e:
        pa.pa_create(good())
    assert e.value.status == pa.PA_CUDA_ERROR
    # an invalid config is rejected before any CUDA call
    with pytest.raises(pa.PAError) as e:
        pa.pa_create(good(block_size=24))
    assert e.value.status == pa.PA_INVALID_ARGUMENT and "block_size" in e.value.message


@pytest.mark.parametrize("over", [dict(), dict(max_query_len_bound=5), dict(max_query_len_bound=4096)])
def test_quantized_cache_takes_prompt_rows(over):
    # longer query rows run through the decode kernel in chunks of 16 / G tokens
    st, msg = pa.pa_validate_config(good(cache_dtype=pa.PA_CACHE_FP8_E4M3, k_quant_type=pa.PA_QUANT_PER_TENSOR,
                                         v_quant_type=pa.PA_QUANT_PER_TENSOR, **over))
    assert st == pa.PA_OK, msg


def test_latent_layout_takes_prompt_rows():
    # longer query rows run as one-token decode entries (the absorbed form)
    st, msg = pa.pa_validate_config(latent(max_query_len_bound=64))
    assert st == pa.PA_OK, msg
