"""GPU parity for multi-head latent attention decode ("PagedAttention - CUDA
Design Document", section 12): one latent cache [NB, bs, 1, 576] written
bit-exactly (rotary over channels 512..575), every query head attending with
576 channels and reading the first 512 as V; output within 2e-3 + 1e-2
|oracle| of the fp64 oracle, on single-split items, split + combine, 16-head
groups, fewer than 16 heads, windows and softcap, and a full-size step."""

import pytest
import torch

import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import check_full, check_sampled, host_copy, make, run

pytestmark = pytest.mark.gpu
cs = workloads.custom_shape
SCALE = 0.0723  # explicit: the latent width is not the model's head width


def _step(shape, **kw):
    return make(shape, device="cuda", gen_device="cpu", latent_v_head_size=512, **kw)


SHAPES = [
    cs("mla_h16_bs64", 16, 1, 576, 64, [0, 1, 63, 64, 65, 700], [1] * 6, scale=SCALE, seed=71),
    cs("mla_h16_bs16_rotary", 16, 1, 576, 16, [0, 5, 200, 999], [1] * 4, scale=SCALE, do_rotary=1,
       rotary_dim=64, seed=72),
    cs("mla_h8", 8, 1, 576, 64, [10, 300], [1, 1], scale=SCALE, seed=73),
    cs("mla_h128_groups", 128, 1, 576, 64, [40, 513], [1, 1], scale=SCALE, do_rotary=1, rotary_dim=64, seed=74),
    cs("mla_h16_window_cap", 16, 1, 576, 64, [700, 64, 129], [1, 1, 1], scale=SCALE, softcap=30.0,
       local_window_size=100, seed=75),
    # 48 heads: the second 32-head group of an item holds one valid 16-head half
    cs("mla_h48_half_group", 48, 1, 576, 32, [0, 100, 1500], [1, 1, 1], scale=SCALE, do_rotary=1,
       rotary_dim=64, seed=77),
    # multiples of 128 heads also run the tcgen05 kernel (option): two pages
    # per 32-key tile, window + softcap, unmapped and partly filled pages;
    # 256 heads
    cs("mla_tc_h128_bs16_window_cap", 128, 1, 576, 16, [700, 5, 129, 0, 31], [1] * 5, scale=SCALE, softcap=30.0,
       local_window_size=100, do_rotary=1, rotary_dim=64, seed=78),
    cs("mla_tc_h128_bs64", 128, 1, 576, 64, [0, 1, 31, 32, 63, 64, 65, 1000], [1] * 8, scale=SCALE, seed=79),
    cs("mla_tc_h256_bs32", 256, 1, 576, 32, [300, 1000, 17], [1, 1, 1], scale=SCALE, do_rotary=1, rotary_dim=64,
       seed=80),
]


def _kernel_options(kernel, heads):
    if kernel == "tcgen05":
        if heads % 128:
            pytest.skip("the tcgen05 latent kernel serves multiples of 128 heads")
        return [(pa.PA_OPT_LATENT_TCGEN05, 1)]
    return [(pa.PA_OPT_LATENT_TCGEN05, 0)]


@pytest.mark.parametrize("kernel", ["mma", "tcgen05"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_latent_decode_matches_oracle(shape, kernel):
    opts = _kernel_options(kernel, shape.num_heads)
    step = _step(shape)
    host = host_copy(step)
    _, out, err = run(step, options=opts, max_query_len_bound=1)
    assert err == 0
    check_full(host, step, out)


@pytest.mark.parametrize("kernel", ["mma", "tcgen05"])
@pytest.mark.parametrize("heads", [32, 48, 128])
@pytest.mark.parametrize("split_keys", [64, 192])
def test_latent_split_merge(split_keys, heads, kernel):
    opts = _kernel_options(kernel, heads)
    shape = cs("mla_splits", heads, 1, 576, 64, [1000, 70, 2047, 300], [1] * 4, scale=SCALE, do_rotary=1,
               rotary_dim=64, seed=76)
    step = _step(shape)
    host = host_copy(step)
    _, out, err = run(step, options=[(pa.PA_OPT_SPLIT_KEYS, split_keys)] + opts, max_query_len_bound=1)
    assert err == 0
    check_full(host, step, out)


def test_tcgen05_latent_option_rules():
    step = _step(cs("mla_opt_h32", 32, 1, 576, 64, [10], [1], scale=SCALE, seed=81))
    op = pa.PagedAttention.for_step(step, max_query_len_bound=1)
    with pytest.raises(pa.PAError) as e:
        op.set_option(pa.PA_OPT_LATENT_TCGEN05, 1)
    assert e.value.status == pa.PA_NOT_SUPPORTED
    op.set_option(pa.PA_OPT_LATENT_TCGEN05, 0)


@pytest.mark.parametrize("kernel", ["mma", "tcgen05"])
def test_latent_full_size_step_sampled(kernel):
    """DeepSeek-V3-shaped decode: 128 heads, 576/512 latent, block_size 64,
    32 sequences with past lengths U{512..4096} (sampled rows)."""
    g = torch.Generator().manual_seed(77)
    past = torch.randint(512, 4097, (32,), generator=g).tolist()
    shape = cs("mla_deepseek_b32", 128, 1, 576, 64, past, [1] * 32, scale=SCALE, do_rotary=1, rotary_dim=64,
               seed=77)
    step = _step(shape)
    host = host_copy(step)
    _, out, err = run(step, options=_kernel_options(kernel, 128), max_query_len_bound=1)
    assert err == 0
    from gpu_util import assert_close, raw
    import numpy as np
    import oracle
    ref = oracle.forward(host, threads=16, rows=np.zeros(0, dtype=np.int64))
    assert np.array_equal(raw(step["key_cache"]), raw(ref["key_cache"]))
    rng = np.random.default_rng(0)
    T, H = host["token_count"], host["num_heads"]
    rows = np.unique(rng.integers(0, T * H, 160))
    o = oracle.attention_latent(ref["query_rot"], ref["key_cache"], host["block_table"],
                                host["cumulative_sequence_lengths"], host["past_sequence_lengths"], H, 576, 512,
                                64, SCALE, 0.0, -1, rows=rows, threads=16)
    assert_close(out.float().cpu().numpy().reshape(T * H, 512)[rows], o)


LATENT_PROMPTS = [
    # several new tokens per sequence: each token is its own decode entry,
    # attending causally over the cached rows and the step's earlier tokens
    cs("mla_h16_prompts", 16, 1, 576, 64, [0, 50, 700], [20, 3, 1], scale=SCALE, do_rotary=1, rotary_dim=64,
       seed=82),
    cs("mla_h48_prompts_window_cap", 48, 1, 576, 32, [0, 300], [70, 5], scale=SCALE, softcap=30.0,
       local_window_size=40, seed=83),
    cs("mla_tc_h128_prompts", 128, 1, 576, 64, [0, 129, 2000], [33, 2, 1], scale=SCALE, do_rotary=1, rotary_dim=64,
       seed=84),
]


@pytest.mark.parametrize("kernel", ["mma", "tcgen05"])
@pytest.mark.parametrize("shape", LATENT_PROMPTS, ids=lambda s: s.name)
def test_latent_prompt_rows_match_oracle(shape, kernel):
    """Chunked prefill / prefix caching on the latent layout: sequences with
    many new tokens run in the absorbed form, one token per decode entry."""
    opts = _kernel_options(kernel, shape.num_heads)
    step = _step(shape)
    host = host_copy(step)
    op, out, err = run(step, options=opts)
    assert err == 0
    counts = op.last_step_counts()
    assert counts["n_pre"] == 0 and counts["n_dec"] >= shape.token_count
    check_full(host, step, out)


def test_latent_prompt_rows_with_splits():
    shape = cs("mla_prompts_splits", 32, 1, 576, 64, [0, 1000], [40, 2], scale=SCALE, seed=85)
    step = _step(shape)
    host = host_copy(step)
    _, out, err = run(step, options=[(pa.PA_OPT_SPLIT_KEYS, 128), (pa.PA_OPT_LATENT_TCGEN05, 0)])
    assert err == 0
    check_full(host, step, out)
