"""The tensor-core decode's timeout path, run on purpose: every pipeline wait
is given a limit of a few SM cycles (pa_set_decode_wait_limit), so waits run
out while the first work item is still being loaded.  The call must record
PA_DEVERR_TIMEOUT and return with the GPU context intact (each CTA drains its
own TMA loads and MMAs, with the default limit, before it frees its tensor
memory and exits), leave the workspace's work counters at zero, and the next
call with the same workspace and the default limit must match the oracle."""
import pytest
import torch

import paged_kv_cache_78_gb300 as pa
import workloads
from gpu_util import DeviceCase, assert_close, oracle_reference, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("partition", [0, pa.PA_PARTITION_BALANCED])
def test_wait_limit_timeout_is_reported_and_the_next_call_is_exact(partition):
    pa.pa_get_device_error()
    case = workloads.custom(6, 16, 4, 128, 16, [700, 1500, 64, 1, 900, 2500], "bf16", seed=81)
    dc = DeviceCase(case)
    nbytes = pa.pa_decode_workspace_size(dc.cache, case.num_seqs, case.num_heads,
                                         case.max_seq_len, partition)
    ws = pa.alloc_workspace(nbytes, "cuda")
    pa.pa_set_decode_wait_limit(8)
    try:
        dc.step(partition, ws, kernel=pa.PA_KERNEL_TENSOR)
        flags = pa.pa_get_device_error()
    finally:
        pa.pa_set_decode_wait_limit(0)
    assert flags & pa.PA_DEVERR_TIMEOUT
    # The work counters (next item, CTAs finished) are back at zero.
    assert int(ws[:8].view(torch.int32).abs().sum()) == 0
    ref, _ = oracle_reference(case)
    for _ in range(2):
        dc.out.zero_()
        out = dc.step(partition, ws, kernel=pa.PA_KERNEL_TENSOR)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        assert_close(to_f64(out), ref, case.dtype, "decode after a timed-out call")

