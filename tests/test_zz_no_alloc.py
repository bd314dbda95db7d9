"""pa_forward_no_alloc: the step for callers that cannot allocate device
memory (scratch lives in a static device array instead of a handle's
workspace).  Two calls in a row, with different layers and batches, must
reproduce what pa_forward computes on the same inputs: the paged pools
bit for bit and the outputs within the parity tolerance.

This file is collected last on purpose: a failure here leaves every other
test already run."""

import numpy as np
import pytest
import torch

import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import assert_close, bits, make

pytestmark = pytest.mark.gpu

cs = workloads.custom_shape


def _config(step):
    cos = step.get("cos_cache")
    return pa.make_config(step["num_heads"], step["kv_num_heads"], step["head_size"], step["block_size"],
                          step["num_blocks"], step["max_blocks_per_seq"], step["batch"],
                          max(step["token_count"], 1), scale=step["scale"], softcap=step["softcap"],
                          local_window_size=step["local_window_size"], do_rotary=step["do_rotary"],
                          rotary_interleaved=step["rotary_interleaved"],
                          rotary_dim=step.get("rotary_dim", 0) or 0,
                          max_rotary_positions=0 if cos is None else cos.shape[0])


def _both(shape):
    """(pools, output) from pa_forward and from pa_forward_no_alloc on copies
    of the same step."""
    ref_step = make(shape, device="cuda", gen_device="cpu")
    step = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in ref_step.items()}
    op = pa.PagedAttention.for_step(ref_step)
    ref_out = torch.zeros_like(ref_step["query"])
    op.forward(ref_step, ref_out)
    out = torch.full_like(step["query"], float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_forward_no_alloc(_config(step), step["query"], step["key"], step["value"], step["key_cache"],
                           step["value_cache"], step["block_table"], step["cumulative_sequence_lengths"],
                           step["past_sequence_lengths"], step["batch"], step["token_count"],
                           step.get("cos_cache"), step.get("sin_cache"), out, device_error=err)
    torch.cuda.synchronize()
    assert op.device_error() == 0
    assert int(err.item()) == 0
    return ref_step, ref_out, step, out


def test_no_alloc_matches_forward_twice_in_a_row():
    shapes = [
        workloads.config_shape(0),                                   # mixed decode rows, G = 2, D = 64
        cs("no_alloc_decode", 16, 4, 128, 16, [900, 33, 2047, 400], [1, 2, 1, 1], seed=41),
    ]
    for shape in shapes:
        ref_step, ref_out, step, out = _both(shape)
        assert np.array_equal(bits(step["key_cache"]), bits(ref_step["key_cache"]))
        assert np.array_equal(bits(step["value_cache"]), bits(ref_step["value_cache"]))
        assert_close(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), what=shape.name)


def test_no_alloc_rejects_capacities_beyond_scratch():
    c = pa.make_config(64, 8, 128, 16, 1000, 64, max_batch=4096, max_tokens=1 << 20, do_rotary=1,
                       max_rotary_positions=1024)
    z = torch.zeros(16, dtype=torch.float16, device="cuda")
    i = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_forward_no_alloc(c, z, z, z, z, z.clone(), i, i, i, 1, 1, z, z, z)
    assert e.value.status == pa.PA_INVALID_ARGUMENT and "scratch" in e.value.message
