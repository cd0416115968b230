"""Parity on the five workload configurations at full size, in the launch
configuration the benchmark times (the library's partition choice, or
512-token partitions for long context).  The cache after every write is
compared bit for bit with the oracle's; decode outputs are compared on
sampled sequences the oracle computes one by one (all sequences where that is
cheap)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_78_gb300 as pa
import workloads
from gpu_util import DeviceCase, assert_close, to_device, to_f64, to_host_bits
from oracle.pool_replay import PoolReplay

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(autouse=True)
def clean_error_word():
    pa.pa_get_device_error()
    yield


def run_case(case, partition, sample):
    dc = DeviceCase(case)
    out = dc.step(partition)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    cache_ref = oracle.fill_cache(case)
    assert np.array_equal(to_host_bits(dc.cache), cache_ref), "cache differs from the oracle"
    seqs = np.arange(case.num_seqs) if sample is None else np.asarray(sample)
    ref = oracle.decode(np.ascontiguousarray(case.query[seqs]), cache_ref,
                        np.ascontiguousarray(case.block_tables[seqs]),
                        np.ascontiguousarray(case.seq_lens[seqs]), case.scale)
    return assert_close(to_f64(out)[seqs], ref, case.dtype, case.name)


def test_tiny_full_step():
    run_case(workloads.tiny("bf16"), -1, None)


def test_qwen2_gqa_all_sequences():
    run_case(workloads.qwen2_gqa("bf16"), -1, None)


@pytest.mark.parametrize("block_size", [8, 16, 32])
def test_opt13b_mha_block_size_sweep(block_size):
    case = workloads.opt13b_mha(block_size=block_size)
    lens = case.seq_lens
    sample = sorted({0, 1, int(np.argmax(lens)), int(np.argmin(lens)), case.num_seqs - 1})
    run_case(case, -1, sample)


@pytest.fixture(scope="module", params=[False, True], ids=["uniform_8x32768", "mixed_to_131072"])
def long_context_case(request):
    """The long-context batch on the device, with the oracle's cache and its
    decode of every sequence (computed once for every partition mode)."""
    case = workloads.long_context(mixed=request.param)
    dc = DeviceCase(case)
    cache_ref = oracle.fill_cache(case)
    ref = oracle.decode(case.query, cache_ref, case.block_tables, case.seq_lens, case.scale)
    return case, dc, cache_ref, ref


@pytest.mark.parametrize("fused", [False, True], ids=["write_then_decode", "fused_write"])
@pytest.mark.parametrize("partition", [512, -1, pa.PA_PARTITION_BALANCED])
def test_long_context_every_sequence(long_context_case, partition, fused):
    # 512-token partitions (the workload's statement), the automatic choice
    # and the balanced split (what -1 resolves to here), with the step's
    # cache write as its own call or fused into the decode; every sequence of
    # the batch against the oracle.
    case, dc, cache_ref, ref = long_context_case
    if partition == -1:
        assert pa.pa_decode_partition_size(dc.cache, case.num_seqs, case.num_heads,
                                           case.max_seq_len, -1) == pa.PA_PARTITION_BALANCED
    dc.out.zero_()
    out = dc.step_fused(partition) if fused else dc.step(partition)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert_close(to_f64(out), ref, case.dtype, "%s partition %d" % (case.name, partition))
    if fused:
        assert np.array_equal(to_host_bits(dc.cache), cache_ref), "cache differs from the oracle"


def replay_script(script, num_heads, num_kv_heads, head_size, seed):
    """Drive the library's pool and the oracle's replay with the same
    operations; the GPU cache gets the library's copies and writes (batched
    per run of appends), the oracle cache the oracle's, one op at a time."""
    rng = np.random.default_rng(seed)
    nb, bs = script.num_blocks, script.block_size
    ours = pa.Pool(nb, bs, script.free_order)
    ref = PoolReplay(nb, bs, script.free_order)
    shape = (2, nb, bs, num_kv_heads, head_size)
    cache_dev = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    cache_ref = np.zeros(shape, dtype=np.uint16)
    ops = script.ops
    i = 0
    copies = 0
    while i < len(ops):
        kind, arg = ops[i]
        if kind == "add":
            sid = ours.add_seq(arg)
            assert ref.add_seq(arg) == sid
            k = workloads.random_values(rng, (arg, num_kv_heads, head_size), "bf16")
            v = workloads.random_values(rng, (arg, num_kv_heads, head_size), "bf16")
            slots = np.array([ours.slot(sid, p) for p in range(arg)], dtype=np.int64)
            assert slots.tolist() == [ref.slot(sid, p) for p in range(arg)]
            pa.pa_reshape_and_cache(cache_dev, to_device(k), to_device(v), to_device(slots))
            oracle.reshape_and_cache(cache_ref, k, v, slots)
            i += 1
        elif kind == "fork":
            assert ours.fork(arg) == ref.fork(arg)
            i += 1
        else:
            j = i
            while j < len(ops) and ops[j][0] == "append":
                j += 1
            seqs = [a for _, a in ops[i:j]]
            slots, pairs = ours.append_tokens(seqs)
            k = workloads.random_values(rng, (len(seqs), num_kv_heads, head_size), "bf16")
            v = workloads.random_values(rng, (len(seqs), num_kv_heads, head_size), "bf16")
            ref_pairs = []
            for t, sid in enumerate(seqs):
                slot, pair = ref.append_token(sid)
                assert slot == int(slots[t])
                if pair is not None:
                    ref_pairs.append(pair)
                    oracle.copy_blocks(cache_ref, np.array([pair]))
                oracle.reshape_and_cache(cache_ref, k[t:t + 1], v[t:t + 1], np.array([slot]))
            assert pairs.tolist() == [list(p) for p in ref_pairs]
            copies += len(ref_pairs)
            pa.pa_copy_blocks(cache_dev, pairs.to("cuda"))
            pa.pa_reshape_and_cache(cache_dev, to_device(k), to_device(v), slots.to("cuda"))
            i = j
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert np.array_equal(to_host_bits(cache_dev), cache_ref), "cache differs from the oracle"
    seqs = script.decode_seqs
    mb = max(len(ref.table(s)[0]) for s in seqs)
    bt, sl = ours.fill_tables(seqs, mb)
    for r, s in enumerate(seqs):
        t, n = ref.table(s)
        assert bt[r, :len(t)].tolist() == t and int(sl[r]) == n
    q = workloads.random_values(rng, (len(seqs), num_heads, head_size), "bf16")
    out = torch.empty((len(seqs), num_heads, head_size), dtype=torch.bfloat16, device="cuda")
    max_len = int(sl.max())
    part = pa.pa_decode_partition_size(cache_dev, len(seqs), num_heads, max_len, -1)
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(cache_dev, len(seqs), num_heads,
                                                        max_len, part), "cuda")
    scale = 1.0 / np.sqrt(head_size)
    pa.pa_decode(out, to_device(q), cache_dev, bt.cuda(), sl.cuda(), scale, max_len, part, ws)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    want = oracle.decode(q, cache_ref, bt.numpy(), sl.numpy(), scale)
    assert_close(to_f64(out), want, "bf16", "shared prefix decode")
    # The same batch through the shared-prefix decode: the blocks the pool
    # shares are attended once per group of sharers.
    plan = pa.SharedPlan(bt, sl, bs, num_heads, num_kv_heads)
    ws2 = pa.alloc_workspace(pa.pa_decode_shared_workspace_size(cache_dev, len(seqs), num_heads,
                                                                max_len, plan), "cuda")
    out2 = torch.empty_like(out)
    pa.pa_decode_shared(out2, to_device(q), cache_dev, bt.cuda(), sl.cuda(), scale, max_len, plan,
                        plan.upload(), ws2)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert_close(to_f64(out2), want, "bf16", "shared-prefix decode (shared blocks once per group)")
    return copies, plan.num_chunks


def test_parallel_sampling_with_copy_on_write():
    script = workloads.shared_prefix_script(variant="fork", prompt_len=1018)
    copies, chunks = replay_script(script, 32, 8, 128, seed=30)
    assert copies == 16 * 7  # the partly filled last prompt block: one copy per extra sample
    assert chunks == 16


def test_parallel_sampling_full_prompt_blocks_need_no_copy():
    script = workloads.shared_prefix_script(variant="fork", prompt_len=1024, num_requests=4)
    assert replay_script(script, 32, 8, 128, seed=31) == (0, 4)


def test_shared_prefix_requests():
    script = workloads.shared_prefix_script(variant="prefix")
    assert replay_script(script, 32, 8, 128, seed=32) == (0, 4)
