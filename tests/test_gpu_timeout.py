"""The timeout path of the kernels' bounded waits, made to run out safely.

PA_OPT_WAIT_PROBE makes the combine kernel (the step's last kernel, which
holds no asynchronous copies or tensor memory) run one more bounded wait, on
a flag that nothing sets, limited to 2 ms by the global timer.  The step
must end with PA_DEVERR_TIMEOUT in the device error word, the wait's site id
(PA_SITE_COMBINE | 1) beside it and named in the message, its outputs still
correct, and the context still usable: the next step, with the probe off,
is clean.  No GPU fault, trap or hang is involved.
"""

import pytest

import paged_kv_cache_reshape_gb300 as pa
import workloads
from gpu_util import check_full, host_copy, make, run

pytestmark = pytest.mark.gpu

cs = workloads.custom_shape


@pytest.mark.parametrize("shape", [
    workloads.config_shape(0),
    cs("probe_prompts_beside_decode", 8, 2, 128, 16, [0, 600, 31], [150, 1, 1], seed=61),
], ids=lambda s: s.name)
def test_wait_that_runs_out_is_reported_and_the_step_stays_correct(shape):
    step = make(shape, device="cuda", gen_device="cpu")
    host = host_copy(step)
    op, out, err = run(step, options=[(pa.PA_OPT_WAIT_PROBE, 1)])
    assert err & pa.PA_DEVERR_TIMEOUT, f"device error {err:#x}"
    assert op.last_wait_site() == pa.PA_SITE_COMBINE | 1
    assert "combine kernel, wait 1" in pa.pa_last_error_message(op.handle)
    check_full(host, step, out)

    # the same handle, probe off: a clean step on a usable context
    op.set_option(pa.PA_OPT_WAIT_PROBE, 0)
    step2 = make(shape, device="cuda", gen_device="cpu")
    host2 = host_copy(step2)
    out2 = out.clone().fill_(float("nan"))
    op.forward(step2, out2)
    assert op.device_error() == 0
    assert op.last_wait_site() == 0
    check_full(host2, step2, out2)
