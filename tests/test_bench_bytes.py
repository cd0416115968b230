"""The bench's byte accounting (bench.step_bytes), from which every bench
line's roofline is computed: checked on CPU against closed forms written
here from the workloads' shapes, and against a stage-by-stage walk of the
balanced split.  The decode call must move each attended K/V row once, the
queries and outputs once, one table entry per block and one length per
sequence, plus the split-KV partials (head_size values and a log-sum-exp per
query head, in fp32) written once and read once for every row that is split."""
import numpy as np
import pytest

import bench
import paged_kv_cache_78_gb300 as pa
import workloads


def lengths_case(lens, hq, hkv, d, bs, dtype="bf16", meta=None):
    """A batch described by its lengths only (step_bytes reads no data)."""
    lens = np.asarray(lens, dtype=np.int32)
    mb = max(1, int(((lens.astype(np.int64) + bs - 1) // bs).max()) if lens.size else 1)
    empty = np.zeros(0, dtype=np.uint16)
    return workloads.DecodeCase("lengths", 0, hq, hkv, d, bs, 1, dtype, d ** -0.5, lens,
                                np.zeros((len(lens), mb), dtype=np.int32), empty, empty, empty,
                                np.zeros(len(lens) + 1, dtype=np.int64), meta=meta or {})


def test_long_context_with_512_token_partitions():
    # 8 sequences of 32768 tokens, 32 query / 8 KV heads of 128, bf16, 16-token
    # blocks: K and V 8 * 32768 * 8 * 128 * 2 * 2 B, q and o 8 * 32 * 128 * 2 * 2,
    # 2048 table entries per sequence, 8 lengths; 64 partitions per row, each
    # 129 fp32 values written and read.
    case = lengths_case([32768] * 8, 32, 8, 128, 16)
    kv = 8 * 32768 * 8 * 128 * 2 * 2
    qo = 8 * 32 * 128 * 2 * 2
    tables = 8 * 2048 * 4
    partials = 8 * 32 * 64 * 129 * 4 * 2
    b = bench.step_bytes(case, 512)
    assert b["partials"] == partials == 16908288
    assert b["decode"] == kv + qo + tables + 8 * 4 + partials == 1090846752
    # The step counts the workload's bytes (no partials) and the cache write
    # of one new token per sequence: read and write its K and V rows, read
    # its slot.
    assert b["write"] == 8 * 8 * 128 * 2 * 2 * 2 + 8 * 8
    assert b["step"] == kv + qo + tables + 8 * 4 + b["write"]


def test_partitions_only_count_rows_that_split():
    # A row of one partition is written as the final output: no partials.
    case = lengths_case([512, 513, 1, 0, 4096], 16, 4, 64, 16, "fp32")
    b = bench.step_bytes(case, 512)
    parts = [1, 2, 1, 0, 8]
    assert b["partials"] == (2 + 8) * 16 * 65 * 4 * 2
    blocks = 32 + 33 + 1 + 0 + 256
    kv = (512 + 513 + 1 + 4096) * 4 * 64 * 2 * 4
    assert b["decode"] == kv + 5 * 16 * 64 * 4 * 2 + blocks * 4 + 5 * 4 + b["partials"]
    assert sum(p for p in parts if p > 1) == 10
    # Unsplit: the same bytes without partials; the step is the same either way.
    b0 = bench.step_bytes(case, 0)
    assert b0["partials"] == 0 and b0["decode"] == b["decode"] - b["partials"]
    assert b0["step"] == b["step"]


def walk_balanced(lens, hkv, ranges):
    """Pieces per (sequence, KV head) pair, stage by stage: the pairs' stages
    laid end to end (sequence-major, KV heads fastest) and cut into ranges of
    ceil(total / ranges) stages; a pair's pieces are the ranges it meets."""
    owners = []
    for s, n in enumerate(lens):
        for h in range(hkv):
            owners += [s * hkv + h] * (-(-int(n) // 128))
    q = max(1, -(-len(owners) // ranges))
    pieces = np.zeros(len(lens) * hkv, dtype=np.int64)
    for r0 in range(0, len(owners), q):
        for pair in set(owners[r0:r0 + q]):
            pieces[pair] += 1
    return pieces


@pytest.mark.parametrize("ranges", [1, 7, 304, 5000])
def test_balanced_split_pieces_match_a_stage_walk(ranges):
    rng = np.random.default_rng(ranges)
    lens = rng.integers(0, 2049, size=23)
    lens[3] = 0
    case = lengths_case(lens, 14, 2, 64, 16)
    want = walk_balanced(lens, 2, ranges)
    assert np.array_equal(bench.balanced_pieces(case, ranges), want)
    b = bench.step_bytes(case, bench.BALANCED, ranges)
    assert b["partials"] == int(want[want > 1].sum()) * 7 * 65 * 4 * 2


def test_shared_prefix_counts_unique_rows_and_the_group_kernels_ranges():
    # Four sequences on 4 common blocks (16-token blocks), two own blocks
    # each, plus one sequence outside the group; 8 query / 2 KV heads of 128.
    bs = 16
    tables = [[0, 1, 2, 3, 4 + 2 * i, 5 + 2 * i] for i in range(4)] + [[20, 21, 22, 23, 24, 25]]
    lens = np.array([80, 90, 70, 96, 81], dtype=np.int32)
    bt = np.array(tables, dtype=np.int32)
    # Distinct (block, offset) slots the batch attends: the shared 64 tokens
    # once, then every sequence's own tokens.
    unique = 64 + sum(int(n) - 64 for n in lens[:4]) + int(lens[4])
    case = lengths_case(lens, 8, 2, 128, bs, meta={"unique_slots": unique})
    plan = pa.SharedPlan(bt, lens, bs, 8, 2, 1)
    assert plan.num_chunks == 1 and plan.members() == [0, 1, 2, 3]
    kv_unique = unique * 2 * 128 * 2 * 2
    for sms, r_want in ((152, min(152 // 2, plan.info.min_chunk_stages, 16)), (2, 1)):
        r = bench.shared_ranges(case, plan, sms)
        assert r == max(1, r_want)
        b = bench.step_bytes(case, plan=plan, sms=sms)
        assert b["unique_kv"] == kv_unique
        assert b["logical_kv"] == int(lens.sum()) * 2 * 128 * 2 * 2
        member_partials = 4 * 8 * r * 129 * 4 * 2 if r > 1 else 0
        # The non-member (one sequence of 81 tokens: one stage per pair) is
        # never split, whatever the balanced ranges.
        assert b["partials"] == member_partials
        blocks = 5 + 6 + 5 + 6 + 6  # ceil(L / 16) of each sequence
        assert b["decode"] == kv_unique + 5 * 8 * 128 * 2 * 2 + blocks * 4 + 5 * 4 + member_partials
