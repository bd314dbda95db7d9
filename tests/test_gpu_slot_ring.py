"""GPU parity for the explicit slot_mapping write and the rolling (ring
buffer) sliding-window cache ("PagedAttention - CUDA Design Document",
sections 5.2 and 9.3).

  * slot_mapping equal to the derived slots: pools and output bit-identical
    to the derived run, and equal to the oracle;
  * -1 entries skip, other entries redirect rows to blocks no table row
    names: pools bit-exact against the oracle;
  * out-of-range entries are flagged (PA_DEVERR_SLOT) and write nothing;
  * ring buffer (section 9.3.5): each sequence holds N = ceil(W/bs) + 1
    recycled blocks, table entries below the live range are -1; over several
    decode steps the output is bit-identical to the full-cache run with the
    same window, in a batch where some sequences are past the window and some
    are not, also over an e4m3 cache with head_sink.
"""

import math

import numpy as np
import pytest
import torch

import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import check_full, host_copy, make, raw, run

pytestmark = pytest.mark.gpu
cs = workloads.custom_shape


def _derived_slots(step):
    bt = step["block_table"].cpu()
    cum = step["cumulative_sequence_lengths"].cpu().tolist()
    past = step["past_sequence_lengths"].cpu().tolist()
    bs = step["block_size"]
    out = []
    for b in range(len(past)):
        for j in range(cum[b + 1] - cum[b]):
            p = past[b] + j
            blk = int(bt[b, p // bs])
            out.append(-1 if blk < 0 else blk * bs + p % bs)
    return torch.tensor(out, dtype=torch.int32)


def test_explicit_slots_equal_derived_write():
    shape = cs("slots_derived", 8, 2, 128, 16, [0, 17, 300, 5], [3, 1, 2, 1], do_rotary=1, seed=41)
    a = make(shape, device="cuda", gen_device="cpu")
    b = make(shape, device="cuda", gen_device="cpu")
    b["slot_mapping"] = _derived_slots(b).cuda()
    host_b = host_copy(b)
    _, out_a, err_a = run(a)
    _, out_b, err_b = run(b)
    assert err_a == 0 and err_b == 0
    assert np.array_equal(raw(a["key_cache"]), raw(b["key_cache"]))
    assert np.array_equal(raw(a["value_cache"]), raw(b["value_cache"]))
    assert torch.equal(out_a, out_b)
    check_full(host_b, b, out_b)


@pytest.mark.parametrize("cache", ["fp16", "e4m3"])
def test_slot_mapping_skips_and_redirects(cache):
    kw = dict(cache_dtype=workloads.CACHE_FP8, quant_type=workloads.QUANT_PER_TENSOR) if cache == "e4m3" else {}
    shape = cs("slots_redirect", 8, 2, 128, 16, [0, 40, 90], [1, 1, 1], seed=42)
    step = make(shape, device="cuda", gen_device="cpu", **kw)
    NB, bs = step["num_blocks"], step["block_size"]
    used = set(int(x) for x in step["block_table"].flatten().tolist() if x >= 0)
    spare = [x for x in range(NB) if x not in used][0]
    # token 0: redirected into a block no table row names; token 1: no write;
    # token 2: its derived slot
    s = _derived_slots(step)
    # the derived slots of tokens 0 and 1 are not written but still read
    # through the block table (the tokens' own positions): give them finite
    # stale content instead of the NaN sentinel
    for slot in s[:2].tolist():
        for pool in (step["key_cache"], step["value_cache"]):
            row = pool.view(-1, *pool.shape[2:])[slot]
            row.copy_(torch.randn(row.shape, generator=torch.Generator().manual_seed(slot)).to(row.device).to(
                row.dtype) if cache == "fp16" else torch.randint(0, 0x70, row.shape, dtype=torch.uint8).to(row.device))
    s[0], s[1] = spare * bs + 3, -1
    step["slot_mapping"] = s.cuda()
    host = host_copy(step)
    _, out, err = run(step, max_query_len_bound=1)
    assert err == 0
    check_full(host, step, out)


def test_out_of_range_slot_is_flagged_and_skipped():
    shape = cs("slots_bad", 4, 2, 64, 16, [10, 20], [1, 1], seed=43)
    step = make(shape, device="cuda", gen_device="cpu")
    before = raw(step["key_cache"]).copy()
    step["slot_mapping"] = torch.tensor([step["num_blocks"] * 16, -7], dtype=torch.int32, device="cuda")
    _, out, err = run(step)
    assert err & pa.PA_DEVERR_SLOT
    assert np.array_equal(raw(step["key_cache"]), before)


def _ring_case(shape, steps, W, seed, **kw):
    """(full-cache steps, ring-cache steps) of `steps` one-token decode steps."""
    S = steps
    base = make(cs(shape.name, shape.num_heads, shape.kv_num_heads, shape.head_size, shape.block_size,
                   shape.past_lens, [S] * shape.batch, local_window_size=W, seed=seed),
                device="cuda", gen_device="cpu", **kw)
    B, bs, H, Hk, D = base["batch"], base["block_size"], base["num_heads"], base["kv_num_heads"], base["head_size"]
    L0 = list(shape.past_lens)
    N = math.ceil(W / bs) + 1
    bt_full = base["block_table"]
    MB = bt_full.shape[1]
    ring_ids = [[b * N + r for r in range(N)] for b in range(B)]
    kc_r = torch.empty((B * N + 1,) + tuple(base["key_cache"].shape[1:]), dtype=base["key_cache"].dtype,
                       device="cuda")
    vc_r = torch.empty_like(kc_r)
    for t in (kc_r, vc_r):  # the unused-slot patterns of workloads.make_step
        if t.dtype == torch.float16:
            t.view(torch.int16).fill_(workloads.NAN_SENTINEL_BITS)
        else:
            t.fill_(0x7F if kw.get("cache_dtype") == workloads.CACHE_FP8 else 0x80)
    for b in range(B):
        live0 = max(0, L0[b] - W + 1) // bs
        for i in range(live0, math.ceil(L0[b] / bs)):
            kc_r[ring_ids[b][i % N]] = base["key_cache"][int(bt_full[b, i])]
            vc_r[ring_ids[b][i % N]] = base["value_cache"][int(bt_full[b, i])]
    g = torch.Generator().manual_seed(seed + 1)
    full_steps, ring_steps = [], []
    for s in range(S):
        past = torch.tensor([L0[b] + s for b in range(B)], dtype=torch.int32)
        cum = torch.arange(B + 1, dtype=torch.int32)
        q = torch.randn(B, H * D, generator=g).half()
        k = torch.randn(B, Hk * D, generator=g).half()
        v = torch.randn(B, Hk * D, generator=g).half()
        common = {key: val for key, val in base.items()
                  if key not in ("query", "key", "value", "cumulative_sequence_lengths", "past_sequence_lengths",
                                 "block_table", "key_cache", "value_cache")}
        common.update(query=q.cuda(), key=k.cuda(), value=v.cuda(), cumulative_sequence_lengths=cum.cuda(),
                      past_sequence_lengths=past.cuda(), batch=B, token_count=B)
        full_steps.append(dict(common, block_table=bt_full, key_cache=base["key_cache"],
                               value_cache=base["value_cache"]))
        bt_r = torch.full((B, MB), -1, dtype=torch.int32)
        slots = []
        for b in range(B):
            p = L0[b] + s
            live0 = max(0, p - W + 1) // bs
            for j in range(live0, p // bs + 1):
                bt_r[b, j] = ring_ids[b][j % N]
            slots.append(ring_ids[b][(p // bs) % N] * bs + p % bs)
        ring_steps.append(dict(common, block_table=bt_r.cuda(), key_cache=kc_r, value_cache=vc_r,
                               num_blocks=B * N + 1, slot_mapping=torch.tensor(slots, dtype=torch.int32).cuda()))
    return full_steps, ring_steps


@pytest.mark.parametrize("variant", ["fp16", "e4m3_sink"])
def test_ring_buffer_cache_bit_matches_full_cache(variant):
    kw = dict(cache_dtype=workloads.CACHE_FP8, quant_type=workloads.QUANT_PER_CHANNEL, head_sink=True) \
        if variant == "e4m3_sink" else {}
    # W = 100: sequences 0-2 are past the window, sequence 3 is not
    shape = cs("ring", 8, 2, 128, 16, [260, 1000, 131, 40], [1, 1, 1, 1])
    full, ring = _ring_case(shape, steps=5, W=100, seed=44, **kw)
    op_f = pa.PagedAttention.for_step(full[0], max_query_len_bound=1)
    op_r = pa.PagedAttention.for_step(ring[0], max_query_len_bound=1)
    for s in range(len(full)):
        host_r = host_copy(ring[s])
        out_f = torch.full_like(full[s]["query"], float("nan"))
        out_r = torch.full_like(ring[s]["query"], float("nan"))
        op_f.forward(full[s], out_f)
        op_r.forward(ring[s], out_r)
        torch.cuda.synchronize()
        assert op_f.device_error() == 0 and op_r.device_error() == 0
        assert torch.equal(out_f, out_r), f"step {s}: ring output differs from the full cache"
        if s in (0, len(full) - 1):
            check_full(host_r, ring[s], out_r)
