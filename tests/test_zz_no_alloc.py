"""pa_decode_no_alloc, the decode entry point that allocates nothing: its
split-KV scratch lives in a device array the library owns, for callers that
cannot allocate device memory (an engine that reserves all memory for its
block pool at start-up, or a C caller without a caching allocator, for whom a
cudaMalloc around each step would synchronise the device).

Checked through the C ABI against the oracle and, bit for bit, against
pa_decode with a caller-provided workspace (the same kernels on the same
inputs), on two calls in a row: the second with shorter sequences than the
first, so that piece counts or partials the first call left in the shared
array would show.  Every partition mode is covered, the automatic choice and
the balanced split included; a call without a split still uses the array's
header (the tensor-core kernel's work counters).  This file is collected last
on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_78_gb300 as pa
import workloads
from gpu_util import DeviceCase, assert_close, to_f64

pytestmark = pytest.mark.gpu


def call_no_alloc(dc, seq_lens, partition):
    c = dc.case
    desc = pa.cache_desc(dc.cache)
    return pa.lib.pa_decode_no_alloc(
        dc.out.data_ptr(), dc.query.data_ptr(), dc.cache.data_ptr(), ctypes.byref(desc),
        dc.block_tables.data_ptr(), dc.block_tables.shape[1], seq_lens.data_ptr(),
        c.num_seqs, c.num_heads, ctypes.c_float(c.scale), c.max_seq_len, partition,
        torch.cuda.current_stream().cuda_stream)


def with_workspace(dc, seq_lens, partition):
    """pa_decode with its own zeroed workspace, on the same inputs."""
    c = dc.case
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(dc.cache, c.num_seqs, c.num_heads,
                                                        c.max_seq_len, partition), "cuda")
    out = torch.empty_like(dc.out)
    pa.pa_decode(out, dc.query, dc.cache, dc.block_tables, seq_lens, c.scale, c.max_seq_len,
                 partition, ws)
    return out


@pytest.mark.parametrize("args,partition", [
    ((3, 32, 8, 128, 16, [3000, 5000, 100], "bf16"), 512),   # fixed partitions
    ((3, 32, 8, 128, 16, [3000, 5000, 100], "bf16"), -1),    # automatic choice (balanced)
    ((3, 32, 8, 128, 16, [3000, 5000, 100], "bf16"), pa.PA_PARTITION_BALANCED),
    ((4, 14, 2, 64, 16, [200, 1500, 1, 900], "bf16"), 128),
    ((4, 14, 2, 64, 16, [200, 1500, 1, 900], "bf16"), -1),
    ((4, 14, 2, 64, 16, [200, 1500, 1, 900], "bf16"), pa.PA_PARTITION_BALANCED),
    ((2, 8, 2, 128, 8, [700, 2100], "fp32"), 256),           # CUDA-core kernel
    ((2, 8, 2, 128, 8, [700, 2100], "fp32"), -1),
    ((2, 4, 4, 64, 16, [60, 90], "bf16"), 0),                # no split: only the header is used
])
def test_no_alloc_matches_oracle_and_pa_decode_on_two_calls(args, partition):
    pa.pa_get_device_error()
    case = workloads.custom(*args[:5], args[5], args[6], seed=77)
    dc = DeviceCase(case)
    dc.step(0)  # writes the step's new tokens; the decode below reads all of them
    cache = oracle.fill_cache(case)
    full = case.seq_lens
    short = np.maximum(1, full // 3).astype(np.int32)
    for lens in (full, short):
        lens_dev = torch.from_numpy(lens).cuda()
        want = oracle.decode(case.query, cache, case.block_tables, lens, case.scale)
        same = with_workspace(dc, lens_dev, partition)
        dc.out.zero_()
        assert call_no_alloc(dc, lens_dev, partition) == pa.PA_OK
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        assert_close(to_f64(dc.out), want, case.dtype, "pa_decode_no_alloc vs oracle")
        assert torch.equal(dc.out.view(torch.uint8), same.view(torch.uint8)), \
            "pa_decode_no_alloc differs from pa_decode"


def test_no_alloc_rejects_partials_beyond_its_array():
    # One sequence bounded by 131072 tokens in 64-token partitions: 32 heads x
    # 2048 partitions x 129 floats = 33.8 MB of partials, above the 16 MiB array.
    case = workloads.custom(1, 32, 8, 128, 16, [40], "bf16", seed=3)
    dc = DeviceCase(case)
    desc = pa.cache_desc(dc.cache)
    max_len, part = 131072, 64
    need = pa.pa_decode_workspace_size(desc, 1, 32, max_len, part)
    assert need > pa.NO_ALLOC_WORKSPACE_BYTES
    st = pa.lib.pa_decode_no_alloc(
        dc.out.data_ptr(), dc.query.data_ptr(), dc.cache.data_ptr(), ctypes.byref(desc),
        dc.block_tables.data_ptr(), dc.block_tables.shape[1], dc.seq_lens.data_ptr(),
        1, 32, ctypes.c_float(case.scale), max_len, part, torch.cuda.current_stream().cuda_stream)
    assert st == pa.PA_ERR_INVALID_ARG
