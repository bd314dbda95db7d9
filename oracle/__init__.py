"""Python access to the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by
the CPU-baseline leg of bench.py.  The library under test never imports it.

The C file is compiled with gcc (-O2 -ffp-contract=off, so that the fp32
rotary keeps one rounding per operation) into liboracle.so beside it.
Arrays cross the boundary as numpy buffers; fp16 and bfloat16 tensors travel
as their uint16 bit patterns.  A step whose cache_dtype is CACHE_BF16 has
bfloat16 activations throughout (query, key, value, both pools, the rotary
tables and head_sink); a step with an 8-bit cache and "act_bf16" set has
bfloat16 activations over 8-bit pools (ACT_BF16 is then added to the cache
type handed to the C functions).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# PA_ORACLE_SOURCE names another copy of oracle.c (the pin-strength test runs
# the pins against deliberately broken copies); its library is built beside it.
_SRC = os.environ.get("PA_ORACLE_SOURCE") or os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(os.path.dirname(os.path.abspath(_SRC)), "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, BAD_ARGUMENT, BAD_DEVICE_DATA = 0, 1, 2
CACHE_FP16, CACHE_INT8, CACHE_FP8, CACHE_BF16 = 0, 1, 2, 3
ACT_BF16 = 16  # added to an 8-bit cache type: bfloat16 activations


def act_bf16(step) -> bool:
    """True when the step's activations (query, key, value, tables, sink,
    norm weights and the output) are bfloat16."""
    return step.get("cache_dtype", CACHE_FP16) == CACHE_BF16 or bool(step.get("act_bf16", False))


def step_cache_dtype(step) -> int:
    """The cache type handed to the C functions for a step: its cache_dtype,
    plus ACT_BF16 for bfloat16 activations over an 8-bit cache."""
    cdt = step.get("cache_dtype", CACHE_FP16)
    if act_bf16(step) and cdt in (CACHE_INT8, CACHE_FP8):
        cdt |= ACT_BF16
    return cdt


def build(force: bool = False) -> str:
    """Compile oracle.c -> liboracle.so (plain gcc, no CUDA)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math",
                           "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I, LL, Dd = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_double
            L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_half_to_double.restype = Dd
            L.oracle_double_to_half.argtypes = [Dd]
            L.oracle_double_to_half.restype = ctypes.c_uint16
            L.oracle_rotary.argtypes = [P, P, I, I, I, P, P, I, P, P, I, I, I]
            L.oracle_rotary.restype = I
            L.oracle_cache_write.argtypes = [P, P, P, P, P, I, P, P, I, I, I, I, I, I, P]
            L.oracle_cache_write.restype = I
            L.oracle_attention.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, I, I,
                                           Dd, Dd, I, LL, LL, P]
            L.oracle_attention.restype = I
            L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_double.restype = Dd
            L.oracle_float_to_e4m3.argtypes = [ctypes.c_float]
            L.oracle_float_to_e4m3.restype = ctypes.c_uint8
            L.oracle_quantize.argtypes = [ctypes.c_uint16, ctypes.c_float, I]
            L.oracle_quantize.restype = ctypes.c_uint8
            L.oracle_cache_write_quant.argtypes = [P, P, P, P, P, P, I, I, P, I, P, P, I, I, I, I, I, I, P]
            L.oracle_cache_write_quant.restype = I
            L.oracle_attention_ex.argtypes = [P, P, P, I, P, P, I, P, P, I, P, P, I, I, I, I, I, I, I,
                                              Dd, Dd, I, LL, LL, P]
            L.oracle_attention_ex.restype = I
            L.oracle_qk_norm.argtypes = [P, P, I, I, I, P, ctypes.c_float]
            L.oracle_qk_norm.restype = I
            L.oracle_rotary_offset.argtypes = [P, P, I, I, I, P, P, I, P, P, I, I, I, I]
            L.oracle_rotary_offset.restype = I
            L.oracle_attention_latent.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, Dd, Dd, I, LL, LL, P]
            L.oracle_attention_latent.restype = I
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = Dd
            L.oracle_double_to_bf16.argtypes = [Dd]
            L.oracle_double_to_bf16.restype = ctypes.c_uint16
            L.oracle_rotary_bf16.argtypes = [P, P, I, I, I, P, P, I, P, P, I, I, I, I]
            L.oracle_rotary_bf16.restype = I
            L.oracle_qk_norm_bf16.argtypes = [P, P, I, I, I, P, ctypes.c_float]
            L.oracle_qk_norm_bf16.restype = I
            _lib = L
    return _lib


def _np(x, dtype):
    """torch tensor / numpy array -> C-contiguous numpy array of `dtype`."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if dtype == np.uint16:
            import torch
            x = x.contiguous().view(torch.int16).numpy().view(np.uint16)
        else:
            x = x.contiguous().numpy()
    return np.ascontiguousarray(x).astype(dtype, copy=False)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _check(st, what):
    if st != OK:
        raise ValueError(f"oracle {what} failed with status {st}")


def half_bits_to_double(bits: np.ndarray) -> np.ndarray:
    f = np.vectorize(lib().oracle_half_to_double, otypes=[np.float64])
    return f(bits.astype(np.uint16))


def double_to_half_bits(x: np.ndarray) -> np.ndarray:
    f = np.vectorize(lambda v: lib().oracle_double_to_half(float(v)), otypes=[np.uint16])
    return f(np.asarray(x, dtype=np.float64))


def bf16_bits_to_double(bits: np.ndarray) -> np.ndarray:
    f = np.vectorize(lib().oracle_bf16_to_double, otypes=[np.float64])
    return f(np.asarray(bits, dtype=np.uint16))


def double_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    f = np.vectorize(lambda v: lib().oracle_double_to_bf16(float(v)), otypes=[np.uint16])
    return f(np.asarray(x, dtype=np.float64))


def e4m3_to_double(codes: np.ndarray) -> np.ndarray:
    f = np.vectorize(lambda c: lib().oracle_e4m3_to_double(int(c)), otypes=[np.float64])
    return f(np.asarray(codes, dtype=np.uint8))


def float_to_e4m3(x: np.ndarray) -> np.ndarray:
    f = np.vectorize(lambda v: lib().oracle_float_to_e4m3(float(v)), otypes=[np.uint8])
    return f(np.asarray(x, dtype=np.float32))


def quantize(bits: np.ndarray, scale: float, cache_dtype: int) -> np.ndarray:
    """8-bit codes of fp16 values (bit patterns; bfloat16 with ACT_BF16 added
    to cache_dtype) under one scale."""
    f = np.vectorize(lambda h: lib().oracle_quantize(int(h), float(scale), int(cache_dtype)),
                     otypes=[np.uint8])
    return f(np.asarray(bits, dtype=np.uint16))


def qk_norm(x, nheads, head_size, weight, eps, bf16=False):
    """Per-head RMS-normalized copy of x ([T, nheads*D] fp16 bits, or
    bfloat16 bits with a bfloat16 weight when bf16)."""
    xa = _np(x, np.uint16)
    wa = _np(weight, np.uint16)
    y = np.empty_like(xa)
    fn = lib().oracle_qk_norm_bf16 if bf16 else lib().oracle_qk_norm
    _check(fn(_p(xa), _p(y), xa.shape[0], nheads, head_size, _p(wa), float(eps)), "qk_norm")
    return y


def split_packed_qkv(query, num_heads, kv_num_heads, head_size):
    """(q, k, v) views of packed rows [T, (H + 2*Hk) * D] (fp16 bits)."""
    qa = _np(query, np.uint16)
    H, Hk, D = num_heads, kv_num_heads, head_size
    return (np.ascontiguousarray(qa[:, :H * D]), np.ascontiguousarray(qa[:, H * D:(H + Hk) * D]),
            np.ascontiguousarray(qa[:, (H + Hk) * D:]))


def rotary(x, cum, past, cos_cache, sin_cache, nheads, head_size, interleaved, offset=0, bf16=False):
    """Rotated copy of x ([T, nheads*D] fp16 bits, or bfloat16 bits with
    bfloat16 tables when bf16) at positions past_b + j; the rotated channels
    are [offset, offset + 2 * cos_cache.shape[1])."""
    xa = _np(x, np.uint16)
    cum_a, past_a = _np(cum, np.int32), _np(past, np.int32)
    cos_a, sin_a = _np(cos_cache, np.uint16), _np(sin_cache, np.uint16)
    T = xa.shape[0]
    y = np.empty_like(xa)
    fn = lib().oracle_rotary_bf16 if bf16 else lib().oracle_rotary_offset
    st = fn(_p(xa), _p(y), T, nheads, head_size, _p(cum_a), _p(past_a), past_a.shape[0], _p(cos_a), _p(sin_a),
            cos_a.shape[1], cos_a.shape[0], interleaved, int(offset))
    _check(st, "rotary")
    return y


def attention_latent(query, latent_cache, block_table, cum, past, num_heads, head_size, v_head_size,
                     block_size, scale, softcap, window, rows=None, threads=None):
    """fp64 absorbed latent attention ([T, H, Dv], or [len(rows), Dv])."""
    qa = _np(query, np.uint16)
    lc = _np(latent_cache, np.uint16)
    bt = _np(block_table, np.int32)
    cum_a, past_a = _np(cum, np.int32), _np(past, np.int32)
    T, H, D, Dv = qa.shape[0], num_heads, head_size, v_head_size
    B, MB, NB = past_a.shape[0], bt.shape[1], lc.shape[0]
    L = lib()

    def run(r0, r1, out):
        st = L.oracle_attention_latent(_p(qa), _p(lc), _p(bt), MB, _p(cum_a), _p(past_a), B, T, H, D, Dv,
                                       block_size, NB, float(scale), float(softcap), int(window), r0, r1,
                                       _p(out))
        _check(st, "attention_latent")

    threads = threads or 1
    if rows is None:
        n = T * H
        out = np.zeros((n, Dv), dtype=np.float64)
        bounds = np.linspace(0, n, max(1, min(threads, n)) + 1).astype(np.int64)
        with ThreadPoolExecutor(max(1, threads)) as ex:
            list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1]), out[bounds[i]:bounds[i + 1]]),
                        range(len(bounds) - 1)))
        return out.reshape(T, H, Dv)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.shape[0], Dv), dtype=np.float64)
    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(lambda i: run(int(rows[i]), int(rows[i]) + 1, out[i:i + 1]), range(rows.shape[0])))
    return out


def cache_write(key, value, key_cache, value_cache, block_table, cum, past,
                kv_num_heads, head_size, block_size, cache_dtype=CACHE_FP16,
                k_scale=None, v_scale=None, per_channel=False, slot_mapping=None):
    """Returns (key_cache', value_cache') after writing the new tokens' rows.

    key/value are fp16 bit arrays [T, Hk*D] (key already rotated when rotary
    is on); the input caches are copied, not modified.  With an 8-bit
    cache_dtype the caches are uint8 code arrays and k_scale / v_scale fp32
    arrays ([1], or [Hk*D] when per_channel); ACT_BF16 added to it reads key
    and value as bfloat16 bits.  slot_mapping ([T] int32, -1 =
    no write) replaces the slot derivation when given."""
    sm = _np(slot_mapping, np.int32) if slot_mapping is not None else None
    if cache_dtype not in (CACHE_FP16, CACHE_BF16):  # a 16-bit write is a copy of the bits
        ka, va = _np(key, np.uint16), _np(value, np.uint16)
        kc = _np(key_cache, np.uint8).copy()
        vc = _np(value_cache, np.uint8).copy()
        ks, vs = _np(k_scale, np.float32), _np(v_scale, np.float32)
        bt = _np(block_table, np.int32)
        cum_a, past_a = _np(cum, np.int32), _np(past, np.int32)
        st = lib().oracle_cache_write_quant(_p(ka), _p(va), _p(kc), _p(vc), _p(ks), _p(vs),
                                            int(bool(per_channel)), int(cache_dtype), _p(bt),
                                            bt.shape[1], _p(cum_a), _p(past_a), past_a.shape[0],
                                            ka.shape[0], kv_num_heads, head_size, block_size,
                                            kc.shape[0], _p(sm))
        _check(st, "cache_write_quant")
        return kc, vc
    ka, va = _np(key, np.uint16), _np(value, np.uint16)
    kc = _np(key_cache, np.uint16).copy()
    vc = _np(value_cache, np.uint16).copy()
    bt = _np(block_table, np.int32)
    cum_a, past_a = _np(cum, np.int32), _np(past, np.int32)
    st = lib().oracle_cache_write(_p(ka), _p(va), _p(kc), _p(vc), _p(bt), bt.shape[1],
                                  _p(cum_a), _p(past_a), past_a.shape[0], ka.shape[0],
                                  kv_num_heads, head_size, block_size, kc.shape[0], _p(sm))
    _check(st, "cache_write")
    return kc, vc


def attention(query, key_cache, value_cache, block_table, cum, past, num_heads,
              kv_num_heads, head_size, block_size, scale, softcap, window,
              rows=None, threads=None, cache_dtype=CACHE_FP16, k_scale=None,
              v_scale=None, per_channel=False, head_sink=None):
    """fp64 attention output.

    rows=None computes every (t, h) row and returns [T, H, D]; otherwise
    `rows` is an int array of r = t*H + h and the result is [len(rows), D].
    Row ranges run on `threads` Python threads (the C call releases the GIL).
    8-bit caches are code arrays dequantized with k_scale / v_scale;
    CACHE_BF16 reads query, both caches and head_sink as bfloat16 bits;
    ACT_BF16 added to an 8-bit type reads query and head_sink so;
    head_sink ([H] fp16) adds the sink term to every row's denominator.
    """
    qa = _np(query, np.uint16)
    cdt = np.uint16 if cache_dtype in (CACHE_FP16, CACHE_BF16) else np.uint8
    kc, vc = _np(key_cache, cdt), _np(value_cache, cdt)
    ks = _np(k_scale, np.float32) if k_scale is not None else None
    vs = _np(v_scale, np.float32) if v_scale is not None else None
    sk = _np(head_sink, np.uint16) if head_sink is not None else None
    bt = _np(block_table, np.int32)
    cum_a, past_a = _np(cum, np.int32), _np(past, np.int32)
    T, H, D = qa.shape[0], num_heads, head_size
    B, MB, NB = past_a.shape[0], bt.shape[1], kc.shape[0]
    L = lib()

    def run(r0, r1, out):
        st = L.oracle_attention_ex(_p(qa), _p(kc), _p(vc), int(cache_dtype), _p(ks), _p(vs),
                                   int(bool(per_channel)), _p(sk), _p(bt), MB, _p(cum_a),
                                   _p(past_a), B, T, H, kv_num_heads, D, block_size, NB,
                                   float(scale), float(softcap), int(window), r0, r1, _p(out))
        _check(st, "attention")

    threads = threads or 1
    if rows is None:
        out = np.zeros((T * H, D), dtype=np.float64)
        n = T * H
        if threads <= 1 or n < 2:
            run(0, n, out)
        else:
            bounds = np.linspace(0, n, min(threads, n) + 1).astype(np.int64)
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(lambda i: run(int(bounds[i]), int(bounds[i + 1]),
                                          out[bounds[i]:bounds[i + 1]]), range(len(bounds) - 1)))
        return out.reshape(T, H, D)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.shape[0], D), dtype=np.float64)

    def one(i):
        run(int(rows[i]), int(rows[i]) + 1, out[i:i + 1])

    if threads <= 1:
        for i in range(rows.shape[0]):
            one(i)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(one, range(rows.shape[0])))
    return out


def forward(step, threads=None, rows=None):
    """Whole step on the CPU: rotary (if on), cache write, attention.

    `step` is a dict as produced by workloads.make_step.  Returns a dict with
    the rotated query bits, the updated caches (uint16 bits) and the fp64
    output ([T, H, D], or [len(rows), D] when rows is given).
    """
    H, Hk, D = step["num_heads"], step["kv_num_heads"], step["head_size"]
    cum, past = step["cumulative_sequence_lengths"], step["past_sequence_lengths"]
    if step.get("kv_cache_layout", 0) == 1:  # one latent cache (CUDA design section 12)
        q, k = _np(step["query"], np.uint16), _np(step["key"], np.uint16)
        if step["do_rotary"]:
            off = step.get("rotary_offset", 0)
            q = rotary(q, cum, past, step["cos_cache"], step["sin_cache"], H, D, step["rotary_interleaved"], off)
            k = rotary(k, cum, past, step["cos_cache"], step["sin_cache"], 1, D, step["rotary_interleaved"], off)
        kc, _ = cache_write(k, k, step["key_cache"], step["key_cache"], step["block_table"], cum, past, 1, D,
                            step["block_size"], slot_mapping=step.get("slot_mapping"))
        out = attention_latent(q, kc, step["block_table"], cum, past, H, D, step["v_head_size"],
                               step["block_size"], step["scale"], step["softcap"], step["local_window_size"],
                               rows=rows, threads=threads)
        return dict(query_rot=q, key_rot=k, key_cache=kc, value_cache=None, out=out)
    if step.get("key") is None:  # packed QKV rows
        q, k, v = split_packed_qkv(step["query"], H, Hk, D)
    else:
        q, k, v = _np(step["query"], np.uint16), _np(step["key"], np.uint16), _np(step["value"], np.uint16)
    if step.get("q_norm_weight") is not None:
        eps = step.get("qk_norm_epsilon", 1e-6)
        bf = act_bf16(step)
        q = qk_norm(q, H, D, step["q_norm_weight"], eps, bf16=bf)
        k = qk_norm(k, Hk, D, step["k_norm_weight"], eps, bf16=bf)
    cdt = step_cache_dtype(step)
    bf = act_bf16(step)
    if step["do_rotary"]:
        off = step.get("rotary_offset", 0)  # first rotated channel of a head
        q = rotary(q, cum, past, step["cos_cache"], step["sin_cache"], H, D,
                   step["rotary_interleaved"], off, bf16=bf)
        k = rotary(k, cum, past, step["cos_cache"], step["sin_cache"], Hk, D,
                   step["rotary_interleaved"], off, bf16=bf)
    quant = dict(cache_dtype=cdt, k_scale=step.get("k_scale"), v_scale=step.get("v_scale"),
                 per_channel=step.get("quant_type", 0) == 2)
    kc, vc = cache_write(k, v, step["key_cache"], step["value_cache"],
                         step["block_table"], cum, past, Hk, D, step["block_size"],
                         slot_mapping=step.get("slot_mapping"), **quant)
    out = attention(q, kc, vc, step["block_table"], cum, past, H, Hk, D,
                    step["block_size"], step["scale"], step["softcap"],
                    step["local_window_size"], rows=rows, threads=threads,
                    head_sink=step.get("head_sink"), **quant)
    return dict(query_rot=q, key_rot=k, key_cache=kc, value_cache=vc, out=out)
