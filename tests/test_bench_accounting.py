"""The benchmark's algorithmic work (the numerators of every roofline
fraction and throughput it reports), checked against counts written out by
hand for small steps:

  * decode: each admitted key's K and V row is read once per kv head
    (Hk * D * 2 elements), the query rows are read and the output rows
    written once (2 * q * H * D elements); 8-bit pools count one byte per
    element;
  * a window W admits min(L, W) keys for the last token;
  * latent steps read each admitted 576-channel row once (it serves as K
    and V) and do 2 * H * (576 + 512) FLOP per admitted key;
  * a prompt (q * G > 16 rows) counts 4 * D * H FLOP per admitted
    (query token, key) pair, causal: token j of a sequence with past p
    admits min(p + j + 1, W) keys.
"""

import bench
import workloads

cs = workloads.custom_shape


def _step(shape, **kw):
    return workloads.make_step(shape, device="cpu", **kw)


def test_gqa_decode_bytes():
    H, Hk, D = 8, 2, 128
    step = _step(cs("acct_dec", H, Hk, D, 16, [10, 100, 0], [1, 1, 1], seed=1))
    w = bench.work_of(step)
    keys = (10 + 1) + (100 + 1) + (0 + 1)
    assert w["dec_kv_bytes"] == keys * Hk * D * 2 * 2
    assert w["kv_bytes"] == w["dec_kv_bytes"]
    assert w["dec_qo_bytes"] == 3 * 2 * H * D * 2
    assert w["pre_flops"] == 0 and w["tokens"] == 3


def test_window_caps_the_admitted_keys():
    H, Hk, D, W = 4, 2, 64, 50
    step = _step(cs("acct_win", H, Hk, D, 16, [10, 100], [1, 1], local_window_size=W, seed=2))
    w = bench.work_of(step)
    assert w["dec_kv_bytes"] == (11 + W) * Hk * D * 2 * 2


def test_eight_bit_pools_count_one_byte_per_element():
    H, Hk, D = 8, 2, 128
    shape = cs("acct_q8", H, Hk, D, 16, [30, 7], [1, 1], seed=3)
    w16 = bench.work_of(_step(shape))
    w8 = bench.work_of(_step(shape, cache_dtype=workloads.CACHE_FP8, quant_type=workloads.QUANT_PER_TENSOR))
    assert w8["dec_kv_bytes"] * 2 == w16["dec_kv_bytes"]
    assert w8["dec_kv_bytes"] == (31 + 8) * Hk * D * 2


def test_latent_rows_are_read_once():
    H = 16
    step = _step(cs("acct_mla", H, 1, 576, 64, [40, 3], [1, 1], scale=0.07, seed=4), latent_v_head_size=512)
    w = bench.work_of(step)
    keys = 41 + 4
    assert w["dec_kv_bytes"] == keys * 576 * 2
    assert w["dec_flops"] == 2 * H * keys * (576 + 512)
    assert w["dec_qo_bytes"] == 2 * H * (576 + 512) * 2


def test_prompt_flops_are_causal_pairs():
    H, Hk, D, W = 8, 2, 64, 9
    step = _step(cs("acct_pre", H, Hk, D, 16, [5], [20], local_window_size=W, seed=5))
    w = bench.work_of(step)
    pairs = sum(min(5 + j + 1, W) for j in range(20))
    assert w["pre_flops"] == 4 * D * H * pairs
    assert w["dec_kv_bytes"] == 0 and w["tokens"] == 20
