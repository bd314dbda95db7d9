"""pa_forward_no_alloc: the step for callers that cannot allocate device
memory (scratch lives in a static device array instead of a handle's
workspace).  Every shape runs twice in a row through both entry points on
copies of the same inputs: the paged pools must agree bit for bit with
pa_forward's and with the CPU oracle's, and the outputs must be within the
parity tolerance of pa_forward's and of the oracle's.

The shapes reach every kernel the entry point launches: decode rows only,
prompts long enough for prefill tiles beside decode rows, full and partial
rotary (partial at a channel offset), and a window with softcap.

This file is collected last on purpose: a failure here leaves every other
test already run."""

import numpy as np
import pytest
import torch

import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import assert_close, bits, check_full, host_copy, make

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
                          rotary_offset=step.get("rotary_offset", 0),
                          max_rotary_positions=0 if cos is None else cos.shape[0])


def _copy(step):
    return {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in step.items()}


def _step(shape, rotary_offset=0):
    step = make(shape, device="cuda", gen_device="cpu")
    if rotary_offset:
        step["rotary_offset"] = rotary_offset
    return step


SHAPES = [
    (workloads.config_shape(0), 0),                                                   # decode rows, G = 2, D = 64
    (cs("na_decode", 16, 4, 128, 16, [900, 33, 2047, 400], [1, 2, 1, 1], seed=41), 0),
    (cs("na_prompts_beside_decode", 8, 2, 128, 16, [0, 700, 40, 1500], [200, 1, 96, 1], seed=42), 0),
    (cs("na_rotary_full", 8, 2, 128, 32, [0, 300, 77], [130, 1, 3], do_rotary=1, seed=43), 0),
    (cs("na_rotary_partial_offset", 8, 2, 128, 16, [5, 260, 0], [1, 2, 70], do_rotary=1, rotary_dim=64,
        seed=44), 32),
    (cs("na_window_softcap_d256", 4, 2, 256, 64, [0, 900, 130], [150, 1, 2], scale=1 / 16, softcap=30.0,
        local_window_size=120, seed=45), 0),
]


@pytest.mark.parametrize("shape,rotary_offset", SHAPES, ids=lambda v: getattr(v, "name", str(v)))
def test_no_alloc_matches_forward_and_oracle_twice_in_a_row(shape, rotary_offset):
    base = _step(shape, rotary_offset)
    host = host_copy(base)
    for call in range(2):
        ref_step, step = _copy(base), _copy(base)
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
        assert int(err.item()) == 0, f"call {call}: device error {int(err.item()):#x}"
        assert np.array_equal(bits(step["key_cache"]), bits(ref_step["key_cache"])), f"call {call}: key_cache"
        assert np.array_equal(bits(step["value_cache"]), bits(ref_step["value_cache"])), f"call {call}: value_cache"
        assert_close(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), what=f"{shape.name} call {call}")
        check_full(host, step, out)
        op.close()


def test_no_alloc_rejects_capacities_beyond_scratch():
    c = pa.make_config(64, 8, 128, 16, 1000, 64, max_batch=4096, max_tokens=1 << 20, do_rotary=1,
                       max_rotary_positions=1024)
    z = torch.zeros(16, dtype=torch.float16, device="cuda")
    i = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_forward_no_alloc(c, z, z, z, z, z.clone(), i, i, i, 1, 1, z, z, z)
    assert e.value.status == pa.PA_INVALID_ARGUMENT and "scratch" in e.value.message
