"""Python binding of the GB300 PagedAttention step library (libpa_gb300.so).

Argument marshalling only: every function below forwards to the C entry
point of the same name declared in include/pa.h.  Tensors are passed by
`data_ptr()`; streams by `torch.cuda.Stream.cuda_stream`.  No computation
happens here, and there is no fallback: if the shared library is missing
or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa_gb300.so")

PA_OK, PA_INVALID_ARGUMENT, PA_NOT_SUPPORTED, PA_CUDA_ERROR, PA_DEVICE_DATA_ERROR = range(5)
STATUS_NAMES = {0: "PA_OK", 1: "PA_INVALID_ARGUMENT", 2: "PA_NOT_SUPPORTED", 3: "PA_CUDA_ERROR",
                4: "PA_DEVICE_DATA_ERROR"}

PA_DEVERR_CUM, PA_DEVERR_BLOCK_ID, PA_DEVERR_PAST = 1, 2, 4
PA_DEVERR_KV_BOUND, PA_DEVERR_Q_BOUND, PA_DEVERR_ROTARY_POS, PA_DEVERR_TIMEOUT = 8, 16, 32, 64
PA_DEVERR_SLOT = 128

PA_OPT_SPLIT_KEYS, PA_OPT_NO_WINDOW_PRUNE, PA_OPT_KERNEL_TIMING, PA_OPT_DECODE_MAX_ROWS = 1, 2, 3, 4
PA_OPT_DECODE_ITEMS_PER_CTA = 5
PA_OPT_LATENT_TCGEN05 = 6
PA_OPT_PREFILL_SMS, PA_OPT_WAIT_PROBE = 7, 8
PA_SITE_DECODE, PA_SITE_COMBINE, PA_SITE_PREFILL, PA_SITE_PREFILL_PAIR, PA_SITE_LATENT, PA_SITE_LATENT_TC = (
    k << 8 for k in range(1, 7))
PA_STEP_COUNTS = 6
STEP_COUNT_NAMES = ("n_dec", "n_pre", "n_comb", "split_keys", "pre_ctas", "dec_ctas")
PA_STAGE_WORKLIST, PA_STAGE_CACHE_WRITE, PA_STAGE_DECODE, PA_STAGE_PREFILL, PA_STAGE_COMBINE = range(5)
STAGES = ("worklist", "cache_write", "decode", "prefill", "combine")
PA_CACHE_FP16, PA_CACHE_INT8, PA_CACHE_FP8_E4M3, PA_CACHE_BF16 = 0, 1, 2, 3
PA_ACT_DEFAULT, PA_ACT_BF16 = 0, 1
PA_QUANT_NONE, PA_QUANT_PER_TENSOR, PA_QUANT_PER_CHANNEL = 0, 1, 2
PA_LAYOUT_SEPARATE, PA_LAYOUT_LATENT = 0, 1

EXPORTED = ("pa_config_init", "pa_validate_config", "pa_check_step", "pa_create", "pa_cache_write",
            "pa_forward", "pa_check_device_error", "pa_last_error_message", "pa_destroy",
            "pa_set_option", "pa_kernel_time_ms", "pa_last_launch_count", "pa_forward_no_alloc",
            "pa_cache_write_ex", "pa_forward_ex", "pa_last_wait_site", "pa_last_step_counts")


class pa_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("num_heads", "kv_num_heads", "head_size", "block_size",
                                            "num_blocks", "max_blocks_per_seq")] + [
        ("scale", ctypes.c_float), ("softcap", ctypes.c_float)] + [
        (n, ctypes.c_int) for n in ("local_window_size", "do_rotary", "rotary_interleaved",
                                    "rotary_dim", "max_rotary_positions", "max_batch", "max_tokens",
                                    "max_query_len_bound", "max_kv_len_bound", "cache_dtype",
                                    "k_quant_type", "v_quant_type", "packed_qkv", "qk_norm")] + [
        ("qk_norm_epsilon", ctypes.c_float)] + [
        (n, ctypes.c_int) for n in ("kv_cache_layout", "v_head_size", "rotary_offset", "act_dtype")]


class pa_extra_inputs(ctypes.Structure):
    _fields_ = [("head_sink", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("slot_mapping", ctypes.c_void_p), ("q_norm_weight", ctypes.c_void_p),
                ("k_norm_weight", ctypes.c_void_p)]


class PAError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


_lib = None


def lib():
    """The loaded library (builds nothing; call build() first)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; run paged_kv_cache_reshape_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        CFG = ctypes.POINTER(pa_config)
        L.pa_config_init.argtypes = [CFG]
        L.pa_config_init.restype = None
        L.pa_validate_config.argtypes = [CFG, ctypes.c_char_p, S]
        L.pa_check_step.argtypes = [CFG, I, P, P, P, P, P, P, P, P, I, I, P, P, P, ctypes.c_char_p, S]
        L.pa_create.argtypes = [CFG, ctypes.POINTER(P)]
        L.pa_cache_write.argtypes = [P, P, P, P, P, P, P, P, I, I, P, P, P]
        L.pa_forward.argtypes = [P, P, P, P, P, P, P, P, P, I, I, P, P, P, P]
        L.pa_check_device_error.argtypes = [P, ctypes.POINTER(I)]
        L.pa_last_error_message.argtypes = [P]
        L.pa_last_error_message.restype = ctypes.c_char_p
        L.pa_destroy.argtypes = [P]
        L.pa_set_option.argtypes = [P, I, I]
        L.pa_kernel_time_ms.argtypes = [P, I, ctypes.POINTER(ctypes.c_float)]
        L.pa_forward_no_alloc.argtypes = [CFG, P, P, P, P, P, P, P, P, I, I, P, P, P, P, P]
        X = ctypes.POINTER(pa_extra_inputs)
        L.pa_cache_write_ex.argtypes = [P, P, P, P, P, P, P, P, I, I, P, P, X, P]
        L.pa_forward_ex.argtypes = [P, P, P, P, P, P, P, P, P, I, I, P, P, X, P, P]
        L.pa_last_launch_count.argtypes = [P]
        L.pa_last_launch_count.restype = I
        L.pa_last_wait_site.argtypes = [P]
        L.pa_last_step_counts.argtypes = [P, ctypes.POINTER(I)]
        for n in EXPORTED:
            if n not in ("pa_config_init", "pa_last_error_message", "pa_last_launch_count"):
                getattr(L, n).restype = I
        _lib = L
    return _lib


def build(force: bool = False):
    from . import builder as _b
    return _b.build(force=force)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status, handle=None):
    if status != PA_OK:
        msg = lib().pa_last_error_message(handle).decode()
        raise PAError(status, msg)


def make_config(num_heads, kv_num_heads, head_size, block_size, num_blocks, max_blocks_per_seq,
                max_batch, max_tokens, scale=0.0, softcap=0.0, local_window_size=-1, do_rotary=0,
                rotary_interleaved=0, rotary_dim=0, max_rotary_positions=0, max_query_len_bound=0,
                max_kv_len_bound=0, cache_dtype=0, k_quant_type=0, v_quant_type=0, packed_qkv=0,
                qk_norm=0, qk_norm_epsilon=1e-6, kv_cache_layout=0, v_head_size=0,
                rotary_offset=0, act_dtype=0) -> pa_config:
    c = pa_config()
    lib().pa_config_init(ctypes.byref(c))
    for k, v in dict(num_heads=num_heads, kv_num_heads=kv_num_heads, head_size=head_size,
                     block_size=block_size, num_blocks=num_blocks,
                     max_blocks_per_seq=max_blocks_per_seq, max_batch=max_batch,
                     max_tokens=max_tokens, scale=scale, softcap=softcap,
                     local_window_size=local_window_size, do_rotary=do_rotary,
                     rotary_interleaved=rotary_interleaved, rotary_dim=rotary_dim,
                     max_rotary_positions=max_rotary_positions,
                     max_query_len_bound=max_query_len_bound,
                     max_kv_len_bound=max_kv_len_bound, cache_dtype=cache_dtype,
                     k_quant_type=k_quant_type, v_quant_type=v_quant_type, packed_qkv=packed_qkv,
                     qk_norm=qk_norm, qk_norm_epsilon=qk_norm_epsilon, kv_cache_layout=kv_cache_layout,
                     v_head_size=v_head_size, rotary_offset=rotary_offset, act_dtype=act_dtype).items():
        setattr(c, k, v)
    return c


def pa_validate_config(cfg: pa_config):
    buf = ctypes.create_string_buffer(512)
    st = lib().pa_validate_config(ctypes.byref(cfg), buf, 512)
    return st, buf.value.decode()


def pa_check_step(cfg: pa_config, for_forward, query, key, value, key_cache, value_cache,
                  block_table, cumulative_sequence_lengths, past_sequence_lengths, batch,
                  token_count, cos_cache, sin_cache, output):
    """Host-only argument check; pointer arguments are plain integers (or None)."""
    buf = ctypes.create_string_buffer(512)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    st = lib().pa_check_step(ctypes.byref(cfg), for_forward, vp(query), vp(key), vp(value),
                             vp(key_cache), vp(value_cache), vp(block_table),
                             vp(cumulative_sequence_lengths), vp(past_sequence_lengths), batch,
                             token_count, vp(cos_cache), vp(sin_cache), vp(output), buf, 512)
    return st, buf.value.decode()


def pa_create(cfg: pa_config):
    h = ctypes.c_void_p()
    _check(lib().pa_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h


def pa_destroy(h):
    _check(lib().pa_destroy(h))


def pa_set_option(h, option, value):
    _check(lib().pa_set_option(h, option, value), h)


def pa_cache_write(h, key, value, key_cache, value_cache, block_table,
                   cumulative_sequence_lengths, past_sequence_lengths, batch, token_count,
                   cos_cache=None, sin_cache=None, stream=None):
    _check(lib().pa_cache_write(h, _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                _ptr(block_table), _ptr(cumulative_sequence_lengths),
                                _ptr(past_sequence_lengths), batch, token_count, _ptr(cos_cache),
                                _ptr(sin_cache), ctypes.c_void_p(stream or 0)), h)


def pa_forward(h, query, key, value, key_cache, value_cache, block_table,
               cumulative_sequence_lengths, past_sequence_lengths, batch, token_count,
               cos_cache, sin_cache, output, stream=None):
    _check(lib().pa_forward(h, _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache),
                            _ptr(value_cache), _ptr(block_table),
                            _ptr(cumulative_sequence_lengths), _ptr(past_sequence_lengths),
                            batch, token_count, _ptr(cos_cache), _ptr(sin_cache), _ptr(output),
                            ctypes.c_void_p(stream or 0)), h)


def _extra(head_sink=None, k_scale=None, v_scale=None, slot_mapping=None, q_norm_weight=None,
           k_norm_weight=None):
    if all(v is None for v in (head_sink, k_scale, v_scale, slot_mapping, q_norm_weight, k_norm_weight)):
        return None
    x = pa_extra_inputs()
    x.q_norm_weight = None if q_norm_weight is None else q_norm_weight.data_ptr()
    x.k_norm_weight = None if k_norm_weight is None else k_norm_weight.data_ptr()
    x.head_sink = None if head_sink is None else head_sink.data_ptr()
    x.k_scale = None if k_scale is None else k_scale.data_ptr()
    x.v_scale = None if v_scale is None else v_scale.data_ptr()
    x.slot_mapping = None if slot_mapping is None else slot_mapping.data_ptr()
    return ctypes.byref(x)


def pa_cache_write_ex(h, key, value, key_cache, value_cache, block_table,
                      cumulative_sequence_lengths, past_sequence_lengths, batch, token_count,
                      cos_cache=None, sin_cache=None, head_sink=None, k_scale=None, v_scale=None,
                      slot_mapping=None, q_norm_weight=None, k_norm_weight=None, stream=None):
    _check(lib().pa_cache_write_ex(h, _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                   _ptr(block_table), _ptr(cumulative_sequence_lengths),
                                   _ptr(past_sequence_lengths), batch, token_count, _ptr(cos_cache),
                                   _ptr(sin_cache),
                                   _extra(head_sink, k_scale, v_scale, slot_mapping, q_norm_weight, k_norm_weight),
                                   ctypes.c_void_p(stream or 0)), h)


def pa_forward_ex(h, query, key, value, key_cache, value_cache, block_table,
                  cumulative_sequence_lengths, past_sequence_lengths, batch, token_count,
                  cos_cache, sin_cache, output, head_sink=None, k_scale=None, v_scale=None,
                  slot_mapping=None, q_norm_weight=None, k_norm_weight=None, stream=None):
    _check(lib().pa_forward_ex(h, _ptr(query), _ptr(key), _ptr(value), _ptr(key_cache),
                               _ptr(value_cache), _ptr(block_table),
                               _ptr(cumulative_sequence_lengths), _ptr(past_sequence_lengths),
                               batch, token_count, _ptr(cos_cache), _ptr(sin_cache),
                               _extra(head_sink, k_scale, v_scale, slot_mapping, q_norm_weight, k_norm_weight),
                               _ptr(output),
                               ctypes.c_void_p(stream or 0)), h)


def pa_forward_no_alloc(cfg: pa_config, query, key, value, key_cache, value_cache, block_table,
                        cumulative_sequence_lengths, past_sequence_lengths, batch, token_count,
                        cos_cache, sin_cache, output, device_error=None, stream=None):
    """The whole step without a handle or any device allocation (scratch in a
    static device array); see include/pa.h for its limits and sharing rules."""
    _check(lib().pa_forward_no_alloc(ctypes.byref(cfg), _ptr(query), _ptr(key), _ptr(value),
                                     _ptr(key_cache), _ptr(value_cache), _ptr(block_table),
                                     _ptr(cumulative_sequence_lengths),
                                     _ptr(past_sequence_lengths), batch, token_count,
                                     _ptr(cos_cache), _ptr(sin_cache), _ptr(output),
                                     _ptr(device_error), ctypes.c_void_p(stream or 0)))


def pa_check_device_error(h) -> int:
    code = ctypes.c_int(0)
    st = lib().pa_check_device_error(h, ctypes.byref(code))
    if st not in (PA_OK, PA_DEVICE_DATA_ERROR):
        _check(st, h)
    return code.value


def pa_kernel_time_ms(h, stage) -> float:
    ms = ctypes.c_float(-1.0)
    _check(lib().pa_kernel_time_ms(h, stage, ctypes.byref(ms)), h)
    return ms.value


def pa_last_launch_count(h) -> int:
    return lib().pa_last_launch_count(h)


def pa_last_wait_site(h) -> int:
    return lib().pa_last_wait_site(h)


def pa_last_step_counts(h) -> dict:
    out = (ctypes.c_int * PA_STEP_COUNTS)()
    _check(lib().pa_last_step_counts(h, out), h)
    return dict(zip(STEP_COUNT_NAMES, list(out)))


def pa_last_error_message(h=None) -> str:
    return lib().pa_last_error_message(h).decode()


class PagedAttention:
    """A handle bound to one layer configuration (owns the device workspace)."""

    def __init__(self, cfg: pa_config):
        self.cfg = cfg
        self.handle = pa_create(cfg)

    @classmethod
    def for_step(cls, step: dict, max_batch: Optional[int] = None, max_tokens: Optional[int] = None,
                 **bounds):
        cos = step.get("cos_cache")
        cfg = make_config(step["num_heads"], step["kv_num_heads"], step["head_size"],
                          step["block_size"], step["num_blocks"], step["max_blocks_per_seq"],
                          max_batch or step["batch"], max_tokens or max(step["token_count"], 1),
                          scale=step["scale"], softcap=step["softcap"],
                          local_window_size=step["local_window_size"],
                          do_rotary=step["do_rotary"],
                          rotary_interleaved=step["rotary_interleaved"],
                          rotary_dim=step.get("rotary_dim", 0) or 0,
                          max_rotary_positions=0 if cos is None else cos.shape[0],
                          cache_dtype=step.get("cache_dtype", 0),
                          k_quant_type=step.get("quant_type", 0), v_quant_type=step.get("quant_type", 0),
                          packed_qkv=int(step.get("key") is None),
                          kv_cache_layout=step.get("kv_cache_layout", 0), v_head_size=step.get("v_head_size", 0),
                          rotary_offset=step.get("rotary_offset", 0),
                          act_dtype=PA_ACT_BF16 if step.get("act_bf16") else PA_ACT_DEFAULT,
                          qk_norm=int(step.get("q_norm_weight") is not None),
                          qk_norm_epsilon=step.get("qk_norm_epsilon", 1e-6), **bounds)
        return cls(cfg)

    def forward(self, step: dict, output, stream=None):
        pa_forward_ex(self.handle, step["query"], step["key"], step["value"], step["key_cache"],
                      step["value_cache"], step["block_table"], step["cumulative_sequence_lengths"],
                      step["past_sequence_lengths"], step["batch"], step["token_count"],
                      step.get("cos_cache"), step.get("sin_cache"), output,
                      head_sink=step.get("head_sink"), k_scale=step.get("k_scale"),
                      v_scale=step.get("v_scale"), slot_mapping=step.get("slot_mapping"),
                      q_norm_weight=step.get("q_norm_weight"), k_norm_weight=step.get("k_norm_weight"),
                      stream=stream)

    def cache_write(self, step: dict, stream=None):
        pa_cache_write_ex(self.handle, step["key"], step["value"], step["key_cache"],
                          step["value_cache"], step["block_table"],
                          step["cumulative_sequence_lengths"], step["past_sequence_lengths"],
                          step["batch"], step["token_count"], step.get("cos_cache"),
                          step.get("sin_cache"), head_sink=step.get("head_sink"),
                          k_scale=step.get("k_scale"), v_scale=step.get("v_scale"),
                          slot_mapping=step.get("slot_mapping"), q_norm_weight=step.get("q_norm_weight"),
                          k_norm_weight=step.get("k_norm_weight"), stream=stream)

    def set_option(self, option, value):
        pa_set_option(self.handle, option, value)

    def device_error(self) -> int:
        return pa_check_device_error(self.handle)

    def kernel_time_ms(self, stage) -> float:
        return pa_kernel_time_ms(self.handle, stage)

    def last_launch_count(self) -> int:
        return pa_last_launch_count(self.handle)

    def last_wait_site(self) -> int:
        return pa_last_wait_site(self.handle)

    def last_step_counts(self) -> dict:
        return pa_last_step_counts(self.handle)

    def close(self):
        if self.handle is not None:
            pa_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
