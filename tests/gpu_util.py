"""Helpers shared by the GPU parity tests: run one step through the C ABI
and compare it with the CPU oracle."""

import numpy as np
import torch

import oracle
import paged_kv_cache_reshape_gb300 as pa
import workloads

RTOL, ATOL = 1e-2, 2e-3   # |gpu - oracle| <= ATOL + RTOL * |oracle|
# bfloat16 activations: the output's own rounding is at most 2^-9 |o|, and
# the P*V contraction takes P rounded to bfloat16 (relative error 2^-9 per
# weight) while the denominator sums the unrounded P, so the output moves by
# at most 2^-9 max|V| (|V| < 8 for the N(0,1) draws); hence
# |gpu - oracle| <= 2^-6 + 2^-8 |oracle|.
RTOL_BF16, ATOL_BF16 = 2.0 ** -8, 2.0 ** -6
# bfloat16 activations over an 8-bit cache: the contractions are those of the
# fp16 8-bit path (fp16 operands, P in fp16) and only the output is rounded
# to bfloat16, so the bar is the looser of the two.


def tolerance(step):
    """(rtol, atol) for a step's output."""
    if step.get("cache_dtype", 0) == workloads.CACHE_BF16:
        return RTOL_BF16, ATOL_BF16
    if oracle.act_bf16(step):
        return max(RTOL, RTOL_BF16), max(ATOL, ATOL_BF16)
    return RTOL, ATOL


def out_dtype(step):
    return torch.bfloat16 if oracle.act_bf16(step) else torch.float16


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def raw(t):
    """Bytes of a tensor or numpy array (fp16 pools and 8-bit code pools alike)."""
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().contiguous().view(torch.uint8).numpy().reshape(-1)
    return np.ascontiguousarray(t).view(np.uint8).reshape(-1)


def ensure_built():
    from paged_kv_cache_reshape_gb300 import builder as build
    build.build()


def make(shape, device="cuda", gen_device=None, **kw):
    return workloads.make_step(shape, device=device, gen_device=gen_device, **kw)


def host_copy(step):
    """CPU copy of every tensor of a step (the oracle's inputs)."""
    return {k: (v.detach().cpu().clone() if isinstance(v, torch.Tensor) else v) for k, v in step.items()}


def run(step, options=(), max_batch=None, max_tokens=None, **bounds):
    """pa_forward on `step` (device tensors, pools updated in place)."""
    ensure_built()
    op = pa.PagedAttention.for_step(step, max_batch=max_batch, max_tokens=max_tokens, **bounds)
    for k, v in options:
        op.set_option(k, v)
    width = step.get("v_head_size") or step["head_size"]
    out = torch.full((step["token_count"], step["num_heads"] * width), float("nan"),
                     dtype=out_dtype(step), device=step["query"].device)
    op.forward(step, out)
    torch.cuda.synchronize()
    err = op.device_error()
    return op, out, err


def assert_close(got, ref, what="output", rtol=RTOL, atol=ATOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    # (a NaN reference would pass every comparison below vacuously)
    assert not np.isnan(ref).any(), f"{what}: NaN in the oracle's result (the step reads a NaN input)"
    assert not np.isnan(got).any(), f"{what}: NaN in GPU result"
    diff = np.abs(got - ref)
    bad = diff > atol + rtol * np.abs(ref)
    big = np.abs(ref) >= 1e-3
    rel = (diff[big] / np.abs(ref[big])).max() if big.any() else 0.0
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements outside tolerance; "
                           f"max abs {diff.max():.3g}, max rel {rel:.3g}")
    return diff.max(), rel


def check_full(step_host, step_dev, out, threads=8):
    """Whole-step parity: both pools bit-exact, every output row within tolerance."""
    ref = oracle.forward(step_host, threads=threads)
    assert np.array_equal(raw(step_dev["key_cache"]), raw(ref["key_cache"])), "key_cache pool differs"
    if ref["value_cache"] is not None:
        assert np.array_equal(raw(step_dev["value_cache"]), raw(ref["value_cache"])), "value_cache pool differs"
    T, H = step_host["token_count"], step_host["num_heads"]
    D = step_host.get("v_head_size") or step_host["head_size"]
    rtol, atol = tolerance(step_host)
    return assert_close(out.float().cpu().numpy().reshape(T, H, D), ref["out"], rtol=rtol, atol=atol)


def check_sampled(step_host, step_dev, out, n_rows=192, seed=0, threads=16):
    """Large-step parity: pools bit-exact, a seeded sample of (t, h) rows."""
    T, H = step_host["token_count"], step_host["num_heads"]
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([rng.integers(0, T * H, n_rows), [0, T * H - 1]]))
    return check_rows(step_host, step_dev, out, rows, threads=threads)


def check_rows(step_host, step_dev, out, rows, threads=16):
    """Large-step parity: pools bit-exact, the given (t, h) rows (t * H + h)."""
    ref = oracle.forward(step_host, threads=threads, rows=np.zeros(0, dtype=np.int64))
    assert np.array_equal(raw(step_dev["key_cache"]), raw(ref["key_cache"])), "key_cache pool differs"
    assert np.array_equal(raw(step_dev["value_cache"]), raw(ref["value_cache"])), "value_cache pool differs"
    T, H, D = step_host["token_count"], step_host["num_heads"], step_host["head_size"]
    rows = np.asarray(rows, dtype=np.int64)
    o = oracle.attention(ref["query_rot"], ref["key_cache"], ref["value_cache"],
                         step_host["block_table"], step_host["cumulative_sequence_lengths"],
                         step_host["past_sequence_lengths"], H, step_host["kv_num_heads"], D,
                         step_host["block_size"], step_host["scale"], step_host["softcap"],
                         step_host["local_window_size"], rows=rows, threads=threads,
                         cache_dtype=oracle.step_cache_dtype(step_host), k_scale=step_host.get("k_scale"),
                         v_scale=step_host.get("v_scale"), per_channel=step_host.get("quant_type", 0) == 2,
                         head_sink=step_host.get("head_sink"))
    got = out.float().cpu().numpy().reshape(T * H, D)[rows]
    rtol, atol = tolerance(step_host)
    return assert_close(got, o, rtol=rtol, atol=atol)
