"""GPU parity: the C-ABI path against the CPU oracle, element by element.

Bars: the paged pools are bit-exact; the fp16 output is within
|gpu - oracle| <= 2e-3 + 1e-2 |oracle| (oracle in fp64).
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import assert_close, bits, check_full, check_rows, check_sampled, host_copy, make, run

pytestmark = pytest.mark.gpu

cs = workloads.custom_shape


def _full(shape, options=(), **kw):
    step = make(shape, device="cuda", gen_device="cpu")
    host = host_copy(step)
    op, out, err = run(step, options=options, **kw)
    assert err == 0, f"device error {err:#x}"
    check_full(host, step, out)
    return op, out


SMALL = [
    workloads.config_shape(0),
    cs("d128_g4_bs16_decode", 8, 2, 128, 16, [0, 1, 15, 16, 17, 63, 64, 300], [1] * 8, seed=1),
    cs("d64_mha_bs32_multitok", 4, 4, 64, 32, [0, 33, 100, 7, 64], [4, 1, 3, 2, 4], seed=2),
    cs("d256_g2_bs64_window_cap", 4, 2, 256, 64, [700, 64, 5, 129], [1, 1, 2, 1], scale=1 / 16,
       softcap=50.0, local_window_size=100, seed=3),
    cs("d128_g8_bs16_rotary", 16, 2, 128, 16, [0, 5, 200, 999], [1, 2, 1, 2], do_rotary=1, seed=4),
    cs("d128_g4_rotary_interleaved_r64", 8, 2, 128, 16, [10, 300], [1, 3], do_rotary=1,
       rotary_interleaved=1, rotary_dim=64, seed=5),
    cs("d128_g2_bs128", 4, 2, 128, 128, [0, 127, 128, 500], [1, 1, 1, 1], seed=6),
    cs("d64_g4_bs256_window1", 8, 2, 64, 256, [300, 600], [1, 2], local_window_size=1, seed=7),
    cs("zero_len_rows", 8, 4, 128, 16, [40, 0, 90, 12], [1, 0, 1, 0], seed=8),
    cs("softcap_small_window_edge", 2, 1, 64, 16, [63, 64, 65, 200], [1, 1, 1, 1], softcap=5.0,
       local_window_size=64, seed=9),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_small_step_matches_oracle(shape):
    _full(shape)


@pytest.mark.parametrize("split_keys", [64, 128, 0])
def test_split_counts_agree(split_keys):
    shape = cs("splits", 8, 2, 128, 16, [1000, 70, 2047, 300], [1, 1, 1, 2], seed=11)
    _full(shape, options=[(pa.PA_OPT_SPLIT_KEYS, split_keys)])


def test_unmapped_blocks_are_masked():
    shape = cs("unmapped", 8, 2, 128, 16, [200, 150], [1, 1], local_window_size=48, seed=12)
    step = make(shape, device="cpu")
    step["block_table"][0, 2] = -1       # inside sequence 0's context, below its window
    step["block_table"][1, 3] = -1       # inside sequence 1's window: positions 48..63 masked
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in step.items()}
    op, out, err = run(dev)
    assert err == 0
    check_full(step, dev, out)


def test_large_batch_worklist_chunks():
    B = 1100
    rng = np.random.default_rng(13)
    shape = cs("b1100", 4, 2, 64, 16, rng.integers(0, 40, B), [1] * B, seed=13)
    _full(shape)


def test_empty_step_launches_nothing():
    shape = cs("empty", 4, 2, 64, 16, [5, 9], [0, 0], seed=14)
    step = make(shape, device="cuda", gen_device="cpu")
    op = pa.PagedAttention.for_step(step, max_tokens=4)
    out = torch.empty(0, 4 * 64, dtype=torch.float16, device="cuda")
    before = bits(step["key_cache"]).copy()
    op.forward(step, out)
    torch.cuda.synchronize()
    assert op.last_launch_count() == 0
    assert np.array_equal(before, bits(step["key_cache"]))


def test_bad_device_data_is_flagged_not_faulting():
    shape = cs("bad", 4, 2, 64, 16, [30, 40], [1, 1], seed=15)
    step = make(shape, device="cpu")
    step["block_table"][0, 0] = 10_000                   # outside the pool
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in step.items()}
    op, out, err = run(dev)
    assert err & pa.PA_DEVERR_BLOCK_ID
    # cum not ending at token_count
    step2 = make(shape, device="cpu")
    step2["cumulative_sequence_lengths"][2] = 1
    dev2 = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in step2.items()}
    op2, out2, err2 = run(dev2)
    assert err2 & pa.PA_DEVERR_CUM


def test_window_pruning_bit_matches_unpruned():
    shape = cs("prune", 8, 2, 128, 16, [3000, 1500], [1, 1], local_window_size=256, seed=16)
    outs = []
    for no_prune in (0, 1):
        step = make(shape, device="cuda", gen_device="cpu")
        op, out, err = run(step, options=[(pa.PA_OPT_NO_WINDOW_PRUNE, no_prune),
                                          (pa.PA_OPT_SPLIT_KEYS, 4096)])
        assert err == 0
        outs.append(bits(out))
    assert np.array_equal(outs[0], outs[1])


def test_metadata_bound_invariance():
    shape = cs("bounds", 8, 2, 128, 16, [100, 1000, 37], [1, 1, 1], seed=17)
    outs = []
    for bounds in ({}, dict(max_query_len_bound=1, max_kv_len_bound=1001),
                   dict(max_query_len_bound=64, max_kv_len_bound=4000)):
        step = make(shape, device="cuda", gen_device="cpu")
        op, out, err = run(step, max_tokens=64, max_batch=16, **bounds)
        assert err == 0
        outs.append(bits(out))
    # split sizes follow the device-side work, not the bounds
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


@pytest.mark.parametrize("index", [1, 3, 4])
def test_full_size_decode_config(index):
    shape = workloads.config_shape(index)
    step = make(shape, device="cuda", gen_device="cuda")
    host = host_copy(step)
    op, out, err = run(step)
    assert err == 0, f"device error {err:#x}"
    check_sampled(host, step, out, n_rows=160)


# ------------------------------------------------------------ prefill path
PREFILL = [
    cs("pf_d128_g4_bs32_long", 8, 2, 128, 32, [0, 70, 5], [300, 45, 129], seed=31),
    cs("pf_d64_mha_bs16", 4, 4, 64, 16, [0, 200], [150, 33], seed=32),
    cs("pf_d256_g2_bs64_window_cap", 4, 2, 256, 64, [0, 100], [200, 70], scale=1 / 16, softcap=50.0,
       local_window_size=97, seed=33),
    cs("pf_d128_g8_bs16_rotary", 16, 2, 128, 16, [3, 0], [40, 17], do_rotary=1, seed=34),
    cs("pf_d128_g1_bs128_window", 4, 4, 128, 128, [0, 250], [260, 7], local_window_size=130, seed=35),
    cs("pf_d128_g4_bs256", 8, 2, 128, 256, [0, 511], [257, 2], seed=36),
    cs("pf_g3_rows_not_pow2", 6, 2, 64, 16, [0, 9], [50, 20], seed=37),
]


@pytest.mark.parametrize("shape", PREFILL, ids=lambda s: s.name)
def test_prefill_step_matches_oracle(shape):
    _full(shape)


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_small_step_through_prefill_kernel(shape):
    _full(shape, options=[(pa.PA_OPT_DECODE_MAX_ROWS, 0)])


def test_mixed_routing_in_one_step():
    # tiny mixed step with decode for <= 4 rows: sequence 0 (5 tokens x 2 heads)
    # goes to the tensor-core prefill kernel, the others to split-KV decode
    _full(workloads.config_shape(0), options=[(pa.PA_OPT_DECODE_MAX_ROWS, 4)])


def test_short_prompts_take_chunked_decode_entries():
    """Multi-token sequences of at most two decode items' rows run as two
    decode entries (chunks of 8 / G tokens) instead of a prefill tile: the
    tiny step's 5-token sequence (10 rows at G = 2) and, at G = 4, prompts
    of 3 and 4 tokens, while a 5-token prompt (20 rows) takes the prefill
    kernel."""
    op, _ = _full(workloads.config_shape(0))
    counts = op.last_step_counts()
    assert counts["n_pre"] == 0 and counts["n_dec"] >= 4
    op, _ = _full(cs("short_prompts_g4", 8, 2, 128, 16, [0, 100, 37, 5], [4, 5, 3, 1], seed=73))
    counts = op.last_step_counts()
    assert counts["n_pre"] > 0 and counts["n_dec"] >= 5


def test_full_size_mixed_step():
    """The 16 x 1024-token prompts beside 240 decodes, as the benchmark runs
    it (prefill and decode kernels side by side on an SM split): both pools
    in full, every decode row, every row of two prompts and a seeded sample
    of the rest."""
    shape = workloads.config_shape(2)
    step = make(shape, device="cuda", gen_device="cuda")
    host = host_copy(step)
    op, out, err = run(step)
    assert err == 0, f"device error {err:#x}"
    counts = op.last_step_counts()
    assert counts["n_pre"] > 0 and counts["n_dec"] > 0
    assert counts["pre_ctas"] + counts["dec_ctas"] // 2 <= torch.cuda.get_device_properties(0).multi_processor_count
    H = shape.num_heads
    cum = host["cumulative_sequence_lengths"].tolist()
    dec = [b for b in range(shape.batch) if shape.new_lens[b] == 1]
    prompts = [b for b in range(shape.batch) if shape.new_lens[b] > 1][:2]
    rows = [np.arange(cum[b] * H, cum[b + 1] * H) for b in dec + prompts]
    rng = np.random.default_rng(0)
    rows.append(rng.integers(0, shape.token_count * H, 512))
    rows = np.unique(np.concatenate(rows))
    assert len(dec) == 240 and np.isin(np.arange(cum[dec[0]] * H, cum[dec[0]] * H + H), rows).all()
    check_rows(host, step, out, rows)


def _mid_mixed():
    rng = np.random.default_rng(71)
    past = [0] * 4 + rng.integers(300, 3000, 60).tolist()
    new = [300] * 4 + [1] * 60
    order = rng.permutation(64)
    return cs("mid_mixed_4x300_60dec", 32, 8, 128, 16, [past[i] for i in order], [new[i] for i in order], seed=72)


@pytest.mark.parametrize("prefill_sms", [40, -1])
def test_mid_mixed_step_with_and_without_sm_split(prefill_sms):
    """4 prompts of 300 tokens beside 60 decodes, every row against the
    oracle: once with the prefill kernel held to 40 SMs and the decode
    kernel beside it on the rest (the split shown active in the work list's
    counts), once with no split."""
    shape = _mid_mixed()
    step = make(shape, device="cuda", gen_device="cpu")
    host = host_copy(step)
    op, out, err = run(step, options=[(pa.PA_OPT_PREFILL_SMS, prefill_sms)])
    assert err == 0, f"device error {err:#x}"
    counts = op.last_step_counts()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert counts["n_pre"] > 0 and counts["n_dec"] > 0
    if prefill_sms > 0:
        assert counts["pre_ctas"] == prefill_sms
        assert counts["dec_ctas"] <= 2 * (sms - prefill_sms)
    else:
        assert counts["pre_ctas"] == sms
    check_full(host, step, out)


@pytest.mark.parametrize("items", [0, 1, 2, 7, 8])
def test_items_per_cta_option(items):
    """PA_OPT_DECODE_ITEMS_PER_CTA: 0 (chosen per step from the batch) and
    fixed counts size the splits differently; every choice is correct."""
    shape = cs("items_per_cta", 8, 2, 128, 16, [3000, 70, 2047, 300, 1], [1, 1, 2, 1, 1], seed=91)
    _full(shape, options=[(pa.PA_OPT_DECODE_ITEMS_PER_CTA, items)])


def test_items_per_cta_option_range():
    step = make(cs("items_rule", 8, 2, 128, 16, [10], [1], seed=92), device="cuda", gen_device="cpu")
    op = pa.PagedAttention.for_step(step, max_query_len_bound=1)
    for bad in (-1, 9):
        with pytest.raises(pa.PAError) as e:
            op.set_option(pa.PA_OPT_DECODE_ITEMS_PER_CTA, bad)
        assert e.value.status == pa.PA_INVALID_ARGUMENT


@pytest.mark.parametrize("shape", [
    cs("rot_off_decode", 8, 2, 128, 16, [5, 260, 31], [1, 2, 1], do_rotary=1, rotary_dim=64, seed=81),
    cs("rot_off_prefill", 8, 2, 128, 32, [0, 40], [150, 70], do_rotary=1, rotary_dim=64, seed=82),
    cs("rot_off_interleaved_d256", 4, 2, 256, 64, [0, 300], [90, 1], do_rotary=1, rotary_interleaved=1,
       rotary_dim=128, seed=83),
], ids=lambda s: s.name)
def test_rotary_at_an_offset(shape):
    """rotary_offset on separate K/V caches: channels [off, off + R) of every
    Q and K head are rotated, the others copied; pools bit-exact."""
    step = make(shape, device="cuda", gen_device="cpu")
    step["rotary_offset"] = 32 if shape.head_size == 128 else 64
    host = host_copy(step)
    op, out, err = run(step)
    assert err == 0, f"device error {err:#x}"
    check_full(host, step, out)
