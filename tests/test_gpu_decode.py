"""GPU parity of paged decode attention against the oracle: every head size,
query-group size and block size the library supports, ragged tails, zero and
one-token sequences, split-KV with many partitions, garbage in stale slots,
block relabelling, and device-side error recording."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_78_gb300 as pa
import workloads
from gpu_util import DeviceCase, assert_close, oracle_reference, to_device, to_f64, to_host_bits

pytestmark = pytest.mark.gpu


def bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.fixture(autouse=True)
def clean_error_word():
    pa.pa_get_device_error()
    yield


def kernels_for(case):
    """CUDA-core kernel always; tensor-core kernel where it applies."""
    tc = (case.dtype == "bf16" and case.head_size in (64, 128) and case.block_size >= 8
          and case.num_heads // case.num_kv_heads <= 16)
    simt = case.num_heads // case.num_kv_heads <= 8
    return ([pa.PA_KERNEL_SIMT] if simt else []) + ([pa.PA_KERNEL_TENSOR] if tc else [])


def check(case, partitions=(0, -1)):
    # Every case also runs the balanced split (on the CUDA-core kernel it
    # becomes equal partitions sized to the same workspace).
    ref, cache_ref = oracle_reference(case)
    for kernel in kernels_for(case):
        for p in tuple(partitions) + (pa.PA_PARTITION_BALANCED,):
            dc = DeviceCase(case)
            out = dc.step(p, kernel=kernel)
            torch.cuda.synchronize()
            assert pa.pa_get_device_error() == 0
            assert np.array_equal(bits(to_host_bits(dc.cache)), bits(cache_ref)), "cache differs"
            assert_close(to_f64(out), ref, case.dtype,
                         "%s kernel=%d partition=%s" % (case.name, kernel, p))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_tiny_config(dtype):
    check(workloads.tiny(dtype), partitions=(0, 16, 32, -1))


# (Hq, Hkv, head_size, block_size, lengths, dtype, partitions)
SHAPES = [
    (14, 2, 64, 16, [1, 15, 16, 17, 33, 255, 700], "bf16", (0, 64)),
    (4, 4, 128, 8, [0, 1, 31, 32, 33, 129], "bf16", (0, 32)),
    (32, 8, 128, 16, [5, 100, 511, 512, 513, 1500], "bf16", (0, 512, 128)),
    (32, 8, 128, 16, [7, 300, 1029], "fp32", (0, 256)),
    (8, 1, 256, 32, [3, 64, 200], "bf16", (0, 64)),
    (8, 1, 256, 32, [3, 64, 200], "fp32", (0, 96)),
    (6, 2, 64, 1, [1, 2, 45, 90], "bf16", (0, 8)),
    (4, 2, 128, 2, [3, 40], "fp32", (0, 16)),
    (10, 2, 64, 64, [63, 64, 65, 300], "bf16", (0, 128)),
    (3, 1, 128, 128, [1, 127, 128, 260], "bf16", (0, 256)),
    (2, 1, 64, 256, [255, 256, 257, 600], "fp32", (0, 256)),
    (9, 3, 64, 4, [17, 41], "bf16", (0, 8)),
    (5, 1, 128, 16, [77], "bf16", (0, 16)),
    (12, 2, 256, 16, [150, 33], "bf16", (0, 32)),
    (40, 40, 128, 16, [1, 2048], "bf16", (0, 512)),
    (16, 2, 64, 16, [5000], "bf16", (32, 256)),
    # tensor-core kernel specifics: groups up to 16, stage (128-token) edges,
    # boxes of 128 rows (block size 256), 8-token blocks
    (32, 2, 64, 16, [1, 127, 128, 129, 255, 256, 257, 1000], "bf16", (0, 128, 384)),
    (24, 2, 128, 8, [8, 9, 300, 777], "bf16", (0, 256)),
    (16, 16, 128, 256, [100, 256, 700], "bf16", (0, 512)),
    (12, 1, 64, 32, [2, 4096], "bf16", (0, 640)),
    # many partitions per sequence (the tensor-core kernel numbers only the
    # real items), empty sequences first and last
    (16, 4, 64, 16, [0, 1, 700, 3000, 129, 0], "bf16", (128, 512)),
    # groups of two (the tensor-core kernel's GP = 2), 20-partition rows
    (8, 4, 128, 16, [77, 500, 1025, 2560], "bf16", (0, 128, 256)),
]


@pytest.mark.parametrize("hq,hkv,d,bs,lens,dtype,parts", SHAPES,
                         ids=["hq%d_hkv%d_d%d_bs%d_%s" % (s[0], s[1], s[2], s[3], s[5])
                              for s in SHAPES])
def test_decode_shapes(hq, hkv, d, bs, lens, dtype, parts):
    case = workloads.custom(len(lens), hq, hkv, d, bs, lens, dtype,
                            seed=hq * 1000 + d + bs, cache_fill="garbage")
    check(case, partitions=parts)


@pytest.mark.parametrize("kernel", [pa.PA_KERNEL_SIMT, pa.PA_KERNEL_TENSOR])
def test_block_relabelling_gives_identical_output(kernel):
    case = workloads.custom(3, 8, 2, 128, 16, [70, 300, 33], "bf16", seed=3)
    a = DeviceCase(case).step(0, kernel=kernel).clone()
    perm = np.random.default_rng(2).permutation(case.num_blocks)
    case2 = workloads.custom(3, 8, 2, 128, 16, [70, 300, 33], "bf16", seed=3)
    case2.block_tables = perm[case.block_tables].astype(np.int32)
    b = DeviceCase(case2).step(0, kernel=kernel)
    assert torch.equal(a, b)


@pytest.mark.parametrize("kernel", [pa.PA_KERNEL_SIMT, pa.PA_KERNEL_TENSOR])
def test_repeated_calls_are_deterministic(kernel):
    case = workloads.custom(4, 14, 2, 64, 16, [100, 900, 2000, 1], "bf16", seed=8)
    dc = DeviceCase(case)
    a = dc.step(128, kernel=kernel).clone()
    b = dc.step(128, kernel=kernel).clone()
    assert torch.equal(a, b)


def test_tensor_kernel_rejects_shapes_it_has_no_kernel_for():
    for args in [(4, 4, 64, 4, [9, 9], "bf16"),     # block size below 8
                 (4, 4, 64, 16, [9, 9], "fp32"),    # fp32
                 (4, 4, 256, 16, [9, 9], "bf16")]:  # head size 256
        case = workloads.custom(2, *args[:4], args[4], args[5], seed=1)
        dc = DeviceCase(case)
        with pytest.raises(pa.PAError):
            dc.step(0, kernel=pa.PA_KERNEL_TENSOR)


def test_bad_block_id_is_recorded_and_reads_zeros():
    case = workloads.custom(2, 4, 4, 64, 16, [40, 20], "bf16", seed=4, cache_fill="zeros")
    case.block_tables[0, 1] = case.num_blocks + 3
    dc = DeviceCase.__new__(DeviceCase)
    dc.case, dc.device = case, "cuda"
    cache = oracle.fill_cache(workloads.custom(2, 4, 4, 64, 16, [40, 20], "bf16", seed=4,
                                               cache_fill="zeros"))
    dc.cache = to_device(cache)
    bt = to_device(case.block_tables)
    out = torch.empty_like(to_device(case.query))
    pa.pa_decode(out, to_device(case.query), dc.cache, bt, to_device(case.seq_lens),
                 case.scale, case.max_seq_len, 0, None)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_BLOCK_ID
    assert torch.isfinite(out).all()
    # sequence 1 is untouched by the bad entry
    ref = oracle.decode(case.query[1:], cache, case.block_tables[1:], case.seq_lens[1:], case.scale)
    assert_close(to_f64(out[1:]), ref, "bf16")


def test_seq_len_beyond_table_is_recorded():
    case = workloads.custom(2, 4, 4, 64, 16, [40, 20], "bf16", seed=6, max_blocks=3)
    dc = DeviceCase(case)
    sl = torch.tensor([40, 49], dtype=torch.int32, device="cuda")   # 49 > 3 * 16
    pa.pa_decode(dc.out, dc.query, dc.cache, dc.block_tables, sl, case.scale, 49, 0, None)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_SEQ_LEN


def test_decode_on_side_stream():
    case = workloads.custom(3, 8, 2, 64, 16, [10, 400, 77], "bf16", seed=12)
    ref, _ = oracle_reference(case)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dc = DeviceCase(case)
        out = dc.step(64)
    s.synchronize()
    assert_close(to_f64(out), ref, "bf16")


def test_decode_trace_records_the_pipeline():
    case = workloads.custom(3, 8, 2, 64, 16, [300, 40, 700], "bf16", seed=21)
    dc = DeviceCase(case)
    per_role, warps = 256, 6
    buf = torch.zeros(304 * warps * per_role * 2, dtype=torch.int64, device="cuda")
    pa.pa_set_decode_trace(buf, per_role)
    try:
        out = dc.step(128, kernel=pa.PA_KERNEL_TENSOR)
        torch.cuda.synchronize()
    finally:
        pa.pa_set_decode_trace(None)
    ref, _ = oracle_reference(case)
    assert_close(to_f64(out), ref, "bf16")
    ev = buf.view(-1, warps, per_role, 2).cpu().numpy()
    tags = (ev[..., 1] >> 32) & 0xFFFFFFFF
    starts = int((tags[:, 0, :] == 9).sum())
    assert starts >= 1
    items = 2 * sum(-(-int(n) // 128) for n in case.seq_lens)    # (seq, kv head, 128-token partition)
    stages = 2 * sum(-(-int(n) // 128) for n in case.seq_lens)   # one 128-token stage per partition
    count = lambda w, tag: int((tags[:, w, :] == tag).sum())
    assert count(2, 7) == items
    assert count(0, 2) == stages and count(0, 20) == stages
    assert count(1, 3) == stages and count(1, 4) == stages and count(1, 17) == stages
    assert count(2, 6) == stages
    assert all(count(w, 19) == stages for w in (3, 4, 5))
    for cta in range(ev.shape[0]):
        for w in range(warps):
            t = ev[cta, w, :, 0][tags[cta, w] != 0]
            assert np.all(np.diff(t) >= 0)



def test_large_batch_without_the_length_cache():
    # More sequences than the tensor-core kernel keeps lengths of in shared
    # memory (256): lengths come from global memory, items are numbered sparsely.
    rng = np.random.default_rng(77)
    lens = [int(x) for x in rng.integers(0, 300, size=300)]
    case = workloads.custom(300, 14, 2, 64, 16, lens, "bf16", seed=78)
    check(case, partitions=(0, 64))


@pytest.mark.parametrize("n", [128, 129])
def test_longest_first_ranks_every_sequence(n):
    # The CUDA-core kernel takes batches of up to 128 sequences in decreasing
    # length order: many equal lengths (ties broken by index), empty
    # sequences and one long one must each land on exactly one grid slot;
    # 129 sequences take the unranked order.
    rng = np.random.default_rng(n)
    lens = [int(x) for x in rng.choice([0, 1, 5, 16, 17, 40], size=n)]
    lens[n // 2] = 700
    case = workloads.custom(n, 4, 4, 128, 16, lens, "bf16", seed=n + 1, cache_fill="garbage")
    ref, cache_ref = oracle_reference(case)
    for p in (0, 64, -1):
        dc = DeviceCase(case)
        out = dc.step(p, kernel=pa.PA_KERNEL_SIMT)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        assert np.array_equal(bits(to_host_bits(dc.cache)), bits(cache_ref)), "cache differs"
        assert_close(to_f64(out), ref, case.dtype, "%d sequences partition=%d" % (n, p))


@pytest.mark.parametrize("hq,hkv,d,fused", [(32, 8, 128, False), (32, 8, 128, True),
                                            (14, 2, 64, False), (14, 2, 64, True)])
def test_balanced_ranges_longer_than_the_stage_ring(hq, hkv, d, fused):
    # Enough stages that every balanced range holds more than the three the
    # ring keeps in flight (the first stage past the ring is prefetched into
    # L2), with ragged ends, garbage in stale slots, and the newest token
    # written by the decode itself in the fused form.
    rng = np.random.default_rng(hq + d)
    n = 8 if d == 128 else 64
    lens = [int(x) for x in rng.integers(700, 2100, size=n)]
    lens[1] = 1
    case = workloads.custom(n, hq, hkv, d, 16, lens, "bf16", seed=hq * d + 5, cache_fill="garbage")
    ref, cache_ref = oracle_reference(case)
    dc = DeviceCase(case)
    B = pa.PA_PARTITION_BALANCED
    out = (dc.step_fused(B, kernel=pa.PA_KERNEL_TENSOR) if fused
           else dc.step(B, kernel=pa.PA_KERNEL_TENSOR))
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert np.array_equal(bits(to_host_bits(dc.cache)), bits(cache_ref)), "cache differs"
    assert_close(to_f64(out), ref, case.dtype, "balanced, long ranges, fused=%s" % fused)


def test_automatic_partition_choices():
    # Tensor-core path: no split when pairs give 4+ items per CTA and no
    # sequence is long, else the balanced split (long items beyond 256
    # sequences); CUDA-core path: no split for batches it takes longest first
    # with pairs for 4 CTAs per SM and lengths up to 2048, else 512 halved
    # toward 64.
    cache = torch.zeros((2, 4, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = pa.PA_PARTITION_BALANCED
    assert pa.pa_decode_partition_size(cache, 64, 14, 2011, -1) == B        # Qwen2 shape
    assert pa.pa_decode_partition_size(cache, 4 * sms, 14, 2011, -1) == 0    # 8 pairs per SM
    assert pa.pa_decode_partition_size(cache, 4 * sms, 14, 8192, -1) == 1024  # > 256 sequences
    assert pa.pa_decode_partition_size(cache, 64, 14, 1000, -1) == B         # 128 pairs: split
    assert pa.pa_decode_partition_size(cache, 64, 14, 100, -1) == 0          # one partition
    c128 = torch.zeros((2, 4, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    assert pa.pa_decode_partition_size(c128, 8, 32, 32768, -1) == B         # long context
    mha = torch.zeros((2, 4, 16, 40, 128), dtype=torch.bfloat16, device="cuda")
    assert pa.pa_decode_partition_size(mha, 32, 40, 2048, -1) == 0          # CUDA cores, G = 1
    assert pa.pa_decode_partition_size(mha, 32, 40, 2049, -1) == 512        # a longer sequence
    assert pa.pa_decode_partition_size(mha, 129, 40, 2048, -1) == 512       # not ranked
    f32 = torch.zeros((2, 4, 16, 8, 128), dtype=torch.float32, device="cuda")
    few = -(-4 * sms // 8) - 1                                               # pairs < 4 per SM
    assert pa.pa_decode_partition_size(f32, few + 1, 8, 2048, -1) == 0
    assert pa.pa_decode_partition_size(f32, few, 8, 2048, -1) > 0


def test_balanced_split_applies_to_the_tensor_core_kernel_only():
    B = pa.PA_PARTITION_BALANCED
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cache = torch.zeros((2, 4, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    assert pa.pa_decode_partition_size(cache, 64, 14, 2011, B) == B
    assert pa.pa_decode_partition_size(cache, 256, 14, 2011, B) == B
    # more sequences than the kernel keeps lengths of, a CUDA-core shape, fp32:
    # the automatic rule
    assert pa.pa_decode_partition_size(cache, 257, 14, 2011, B) == \
        pa.pa_decode_partition_size(cache, 257, 14, 2011, -1)
    mha = torch.zeros((2, 4, 16, 40, 128), dtype=torch.bfloat16, device="cuda")
    assert pa.pa_decode_partition_size(mha, 32, 40, 2048, B) == 0
    assert pa.pa_decode_partition_size(mha, 32, 40, 4096, B) == 512
    f32 = torch.zeros((2, 4, 16, 2, 64), dtype=torch.float32, device="cuda")
    assert pa.pa_decode_partition_size(f32, 64, 14, 2011, B) == \
        pa.pa_decode_partition_size(f32, 64, 14, 2011, -1)
    # workspace: partials for min(ceil(len / 128), ceil(ranges / Hkv) + 1)
    # per row, then one piece count per (sequence, KV head)
    for (hkv, d, s, hq, max_len) in [(2, 64, 64, 14, 2011), (8, 128, 8, 32, 32768),
                                     (1, 64, 3, 8, 100000)]:
        c = torch.zeros((2, 4, 16, hkv, d), dtype=torch.bfloat16, device="cuda")
        ranges = sms * (2 if d == 64 else 1)
        mp = min(-(-max_len // 128), -(-ranges // hkv) + 1)
        rows = s * hq * mp
        up = lambda n: -(-n // 256) * 256
        assert pa.pa_decode_workspace_size(c, s, hq, max_len, B) == \
            256 + up(rows * d * 4) + up(rows * 4) + up(s * hkv * 4)


# (Hq, Hkv, head_size, block_size, lengths): the balanced split's cuts
BALANCED_SHAPES = [
    # one long sequence among short ones: with fewer stages than ranges
    # every stage is its own piece, and the long pair has 157 partials
    (8, 1, 64, 16, [1] * 40 + [20000]),
    # empty sequences among others, four KV heads (pieces span pairs)
    (16, 4, 128, 16, [0, 129, 0, 3000, 1, 0, 7000]),
    # everything fits in one stage per pair: one piece each, no partials
    (14, 2, 64, 16, [5, 128, 1, 77]),
    # many pairs per range: ranges cut pairs at arbitrary stages
    (14, 2, 64, 16, [int(x) for x in np.random.default_rng(5).integers(1, 4000, size=200)]),
    # the largest batch the split covers, with empty sequences
    (14, 2, 64, 16, [int(x) * (i % 7 != 3) for i, x in
                     enumerate(np.random.default_rng(6).integers(1, 600, size=256))]),
    # groups of 16, block size 8 and 256
    (32, 2, 64, 8, [3000, 5, 900, 129]),
    (16, 16, 128, 256, [100, 256, 700, 5000]),
]


@pytest.mark.parametrize("hq,hkv,d,bs,lens", BALANCED_SHAPES,
                         ids=["hq%d_hkv%d_d%d_bs%d_n%d" % (s[0], s[1], s[2], s[3], len(s[4]))
                              for s in BALANCED_SHAPES])
def test_balanced_split(hq, hkv, d, bs, lens):
    case = workloads.custom(len(lens), hq, hkv, d, bs, lens, "bf16",
                            seed=hq * 31 + d + bs + len(lens), cache_fill="garbage")
    ref, cache_ref = oracle_reference(case)
    for fused in (False, True):
        dc = DeviceCase(case)
        out = (dc.step_fused if fused else dc.step)(pa.PA_PARTITION_BALANCED,
                                                     kernel=pa.PA_KERNEL_TENSOR)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        assert np.array_equal(to_host_bits(dc.cache), cache_ref), "cache differs"
        assert_close(to_f64(out), ref, "bf16", "balanced fused=%s" % fused)


@pytest.mark.parametrize("hkv,d,lens", [
    (2, 64, None),                                   # the Qwen2-shaped batch
    (8, 128, [3000] * 8),                            # long sequences, equal lengths
    (4, 128, [0, 1, 700, 3000, 129, 0, 5000, 64]),   # empty sequences between others
])
def test_balanced_split_piece_counts_follow_the_rule(hkv, d, lens):
    # The kernel records each (sequence, KV head) pair's piece count in the
    # workspace (after the partials); it must be the number of stage ranges
    # the pair meets: stages laid end to end, cut every ceil(total / ranges).
    if lens is None:
        case = workloads.qwen2_gqa()
    else:
        case = workloads.custom(len(lens), 4 * hkv, hkv, d, 16, lens, "bf16", seed=51)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ranges = sms * (2 if d == 64 else 1)
    dc = DeviceCase(case)
    nbytes = pa.pa_decode_workspace_size(dc.cache, case.num_seqs, case.num_heads,
                                         case.max_seq_len, pa.PA_PARTITION_BALANCED)
    ws = pa.alloc_workspace(nbytes, "cuda")
    dc.step(pa.PA_PARTITION_BALANCED, workspace=ws, kernel=pa.PA_KERNEL_TENSOR)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    pairs = case.num_seqs * case.num_kv_heads
    region = -(-pairs * 4 // 256) * 256
    counts = ws[nbytes - region:nbytes - region + pairs * 4].view(torch.int32).cpu().numpy()
    n = (case.seq_lens.astype(np.int64) + 127) // 128
    per_pair = np.repeat(n, case.num_kv_heads)
    q = max(1, -(-int(per_pair.sum()) // ranges))
    start = np.concatenate([[0], np.cumsum(per_pair)[:-1]])
    want = np.where(per_pair > 0, (start + per_pair - 1) // q - start // q + 1, 0)
    assert np.array_equal(counts, want)
    # every CTA's range holds at most q stages: the split is balanced
    assert q == max(1, -(-int(per_pair.sum()) // ranges))


def test_balanced_split_is_deterministic():
    case = workloads.custom(5, 14, 2, 64, 16, [100, 900, 2000, 1, 0], "bf16", seed=18)
    dc = DeviceCase(case)
    a = dc.step(pa.PA_PARTITION_BALANCED, kernel=pa.PA_KERNEL_TENSOR).clone()
    b = dc.step(pa.PA_PARTITION_BALANCED, kernel=pa.PA_KERNEL_TENSOR).clone()
    assert torch.equal(a, b)



FUSED_SHAPES = [
    (14, 2, 64, 16, [1, 15, 16, 17, 33, 255, 700, 0], "bf16", (0, 64)),
    (32, 8, 128, 16, [5, 100, 511, 512, 513, 1500], "bf16", (0, 512)),
    (4, 4, 128, 8, [0, 1, 31, 32, 33, 129], "bf16", (0, 32)),
    (32, 8, 128, 16, [7, 300, 1029], "fp32", (0, 256)),
    (6, 2, 64, 1, [1, 2, 45, 90], "bf16", (0, 8)),
    (16, 16, 128, 256, [100, 256, 700], "bf16", (0, 512)),
    (16, 4, 64, 16, [0, 1, 700, 3000, 129, 0], "bf16", (128, 512)),
]


@pytest.mark.parametrize("hq,hkv,d,bs,lens,dtype,parts", FUSED_SHAPES,
                         ids=["hq%d_hkv%d_d%d_bs%d_%s" % (s[0], s[1], s[2], s[3], s[5])
                              for s in FUSED_SHAPES])
def test_decode_with_fused_cache_write(hq, hkv, d, bs, lens, dtype, parts):
    # pa_decode_append writes each sequence's newest token itself: the cache
    # ends bit-identical to the separate write, the output matches the oracle.
    case = workloads.custom(len(lens), hq, hkv, d, bs, lens, dtype,
                            seed=hq * 100 + d + bs + 7, cache_fill="garbage")
    ref, cache_ref = oracle_reference(case)
    for kernel in kernels_for(case):
        for p in tuple(parts) + (pa.PA_PARTITION_BALANCED,):
            dc = DeviceCase(case)
            out = dc.step_fused(p, kernel=kernel)
            torch.cuda.synchronize()
            assert pa.pa_get_device_error() == 0
            assert np.array_equal(bits(to_host_bits(dc.cache)), bits(cache_ref)), "cache differs"
            assert_close(to_f64(out), ref, case.dtype, "fused kernel=%d partition=%s" % (kernel, p))


@pytest.mark.parametrize("fused", [False, True])
def test_steps_through_host_buffers(fused):
    # A serving loop's form: each step's inputs come from page-locked host
    # memory through pa_copy_bytes, the step runs, and its output goes back to
    # page-locked host memory the same way, all chained on one stream with
    # no synchronisation between steps.  Step i's query is the base query
    # times a power of two, so each step's output is checked bit for bit
    # against the same step on device-resident inputs, and step 0 against
    # the oracle: an input copy that overtook the previous step's decode, or
    # an output copy that overtook its own, would show.
    lens = [1, 15, 16, 17, 33, 255, 700, 2048, 129, 1000]
    case = workloads.custom(len(lens), 14, 2, 64, 16, lens, "bf16", seed=808,
                            cache_fill="garbage")
    ref, _ = oracle_reference(case)
    dc = DeviceCase(case)
    factors = (1.0, 2.0, 0.5, 4.0)
    base_q = dc.query.clone()
    want = []
    for f in factors:
        dc.query.copy_(base_q * f)
        want.append((dc.step_fused() if fused else dc.step()).clone())
    torch.cuda.synchronize()
    assert_close(to_f64(want[0]), ref, case.dtype, "device-resident step")
    # Host-side inputs of every step, and the device buffers they land in.
    names = ("query", "block_tables", "seq_lens") + (
        ("new_keys", "new_values") if fused else ("step_keys", "step_values", "step_slots"))
    host = [{n: (base_q * f if n == "query" else getattr(dc, n)).cpu().pin_memory()
             for n in names} for f in factors]
    for n in names:
        getattr(dc, n).view(torch.uint8).fill_(0x7f)
    outs = [torch.full(tuple(base_q.shape), 7.0, dtype=base_q.dtype).pin_memory()
            for _ in factors]
    nbytes = pa.pa_decode_workspace_size(dc.cache, case.num_seqs, case.num_heads,
                                         case.max_seq_len, -1)
    ws = pa.alloc_workspace(nbytes, "cuda")
    for i in range(len(factors)):
        for n in names:
            pa.pa_copy_bytes(getattr(dc, n), host[i][n])
        out = dc.step_fused(workspace=ws) if fused else dc.step(workspace=ws)
        pa.pa_copy_bytes(outs[i], out)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    for i in range(len(factors)):
        assert torch.equal(outs[i].view(torch.int16), want[i].cpu().view(torch.int16)), \
            "step %d through host buffers differs" % i
