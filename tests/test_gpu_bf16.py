"""GPU parity of bfloat16 steps (bfloat16 activations and pools; the kernel
is registered for fp16 and bfloat16 activations, "PagedAttention - CUDA
Design Document", section 8.2) against the CPU oracle.

Bars: both pools bit-exact (the write copies or rotates with the oracle's
fp32 steps and one bfloat16 rounding); the bfloat16 output within
|gpu - oracle| <= 2^-6 + 2^-8 |oracle| (the bound is derived in
tests/gpu_util.py).  The cases cover every kernel a bfloat16 step can take:
split-KV decode with and without the combine kernel (head sizes 64, 128,
256; GQA groups 1 to 16), chunked short prompts, the two-tile tensor-core
prefill (head sizes 64 and 128), the one-tile prefill (256), rotary,
window, softcap, head_sink, -1 blocks and an explicit slot_mapping.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import check_full, check_sampled, host_copy, make, run

pytestmark = pytest.mark.gpu

cs = workloads.custom_shape
BF16 = workloads.CACHE_BF16


def _full(shape, options=(), **kw):
    step = make(shape, device="cuda", gen_device="cpu", cache_dtype=BF16, **kw)
    host = host_copy(step)
    op, out, err = run(step, options=options)
    assert out.dtype == torch.bfloat16
    assert err == 0, f"device error {err:#x}"
    check_full(host, step, out)
    return op, out


DECODE = [
    workloads.config_shape(0),
    cs("bf_d128_g4_bs16_decode", 8, 2, 128, 16, [0, 1, 15, 16, 17, 63, 64, 300], [1] * 8, seed=81),
    cs("bf_d64_mha_bs32_multitok", 4, 4, 64, 32, [0, 33, 100, 7, 64], [4, 1, 3, 2, 4], seed=82),
    cs("bf_d256_g2_bs64_window_cap", 4, 2, 256, 64, [700, 64, 5, 129], [1, 1, 2, 1], scale=1 / 16,
       softcap=50.0, local_window_size=100, seed=83),
    cs("bf_d128_g8_bs16_rotary", 16, 2, 128, 16, [0, 5, 200, 999], [1, 2, 1, 2], do_rotary=1, seed=84),
    cs("bf_d128_g4_rotary_interleaved_r64", 8, 2, 128, 16, [10, 300], [1, 3], do_rotary=1,
       rotary_interleaved=1, rotary_dim=64, seed=85),
    cs("bf_d128_g16_splits", 32, 2, 128, 16, [2000, 70, 4000, 1], [1, 1, 1, 1], seed=86),
    cs("bf_zero_len_rows", 8, 4, 128, 16, [40, 0, 90, 12], [1, 0, 1, 0], seed=87),
]


@pytest.mark.parametrize("shape", DECODE, ids=lambda s: s.name)
def test_bf16_decode_step_matches_oracle(shape):
    _full(shape)


@pytest.mark.parametrize("split_keys", [64, 0])
def test_bf16_split_kv_combine(split_keys):
    shape = cs("bf_splits", 8, 2, 128, 16, [1000, 70, 2047, 300], [1, 1, 1, 2], seed=88)
    _full(shape, options=[(pa.PA_OPT_SPLIT_KEYS, split_keys)])


PREFILL = [
    cs("bf_pf_d128_g4_bs32_long", 8, 2, 128, 32, [0, 70, 5], [300, 45, 129], seed=91),
    cs("bf_pf_d64_mha_bs16", 4, 4, 64, 16, [0, 200], [150, 33], seed=92),
    cs("bf_pf_d256_g2_bs64_window_cap", 4, 2, 256, 64, [0, 100], [200, 70], scale=1 / 16, softcap=50.0,
       local_window_size=97, seed=93),
    cs("bf_pf_d128_g8_bs16_rotary", 16, 2, 128, 16, [3, 0], [40, 17], do_rotary=1, seed=94),
]


@pytest.mark.parametrize("shape", PREFILL, ids=lambda s: s.name)
def test_bf16_prefill_step_matches_oracle(shape):
    op, _ = _full(shape)
    assert op.last_step_counts()["n_pre"] > 0


def test_bf16_all_rows_through_prefill_kernel():
    op, _ = _full(DECODE[1], options=[(pa.PA_OPT_DECODE_MAX_ROWS, 0)])
    assert op.last_step_counts()["n_dec"] == 0


def test_bf16_short_prompts_take_chunked_decode_entries():
    op, _ = _full(workloads.config_shape(0))
    counts = op.last_step_counts()
    assert counts["n_pre"] == 0 and counts["n_dec"] >= 4


@pytest.mark.parametrize("shape", [DECODE[1], PREFILL[0]], ids=lambda s: s.name)
def test_bf16_head_sink(shape):
    _full(shape, head_sink=True)


def test_bf16_unmapped_blocks_and_slot_mapping():
    shape = cs("bf_unmapped", 8, 2, 128, 16, [200, 150], [1, 3], local_window_size=48, seed=95)
    step = make(shape, device="cpu", cache_dtype=BF16)
    step["block_table"][0, 2] = -1       # inside sequence 0's context, below its window
    step["block_table"][1, 3] = -1       # inside sequence 1's window: positions 48..63 masked
    # explicit slots: token 0 as derived, token 1 skipped (-1), tokens 2, 3 as derived
    bt, bs = step["block_table"], shape.block_size
    slots = [int(bt[0, 200 // bs]) * bs + 200 % bs, -1,
             int(bt[1, 151 // bs]) * bs + 151 % bs, int(bt[1, 152 // bs]) * bs + 152 % bs]
    step["slot_mapping"] = torch.tensor(slots, dtype=torch.int32)
    # the skipped token's derived slot is still read through the block table
    # (its own position): finite stale content instead of the NaN sentinel
    skipped = int(bt[1, 150 // bs]) * bs + 150 % bs
    for pool in (step["key_cache"], step["value_cache"]):
        pool.view(-1, *pool.shape[2:])[skipped] = torch.randn(pool.shape[2:]).to(torch.bfloat16)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in step.items()}
    op, out, err = run(dev)
    assert err == 0
    check_full(step, dev, out)


def test_bf16_full_size_decode_config():
    """The Llama-3-8B-shaped decode (64 sequences, 512..4096 context) in
    bfloat16: both pools in full and a seeded sample of output rows."""
    shape = workloads.config_shape(1)
    step = make(shape, device="cuda", gen_device="cuda", cache_dtype=BF16)
    host = host_copy(step)
    op, out, err = run(step)
    assert err == 0, f"device error {err:#x}"
    check_sampled(host, step, out, n_rows=160)


def test_bf16_is_not_read_as_fp16():
    """The same draws as fp16 and as bfloat16 give different outputs, each
    matching its own oracle (a kernel that ignored the type would match at
    most one of them)."""
    shape = DECODE[1]
    _, out_bf = _full(shape)
    step = make(shape, device="cuda", gen_device="cpu")
    host = host_copy(step)
    _, out_h, err = run(step)
    assert err == 0
    check_full(host, step, out_h)
    assert not torch.equal(out_bf.float(), out_h.float())
