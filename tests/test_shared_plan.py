"""The shared-prefix plan (pa_decode_shared_plan, host only): groups of
sequences by common leading block ids, the shared length capped so that every
member keeps its newest token, chunks of up to 128 query rows; checked on
hand-built tables and on the shared-prefix pool scripts (forked samples of
one prompt, requests forked from one common prefix)."""
import numpy as np
import pytest

import paged_kv_cache_78_gb300 as pa
import workloads


def plan_of(tables, lens, bs, hq, hkv, min_blocks=1):
    mb = max(len(t) for t in tables)
    bt = np.full((len(tables), mb), 0, dtype=np.int32)
    for r, t in enumerate(tables):
        bt[r, :len(t)] = t
    return pa.SharedPlan(bt, np.asarray(lens, dtype=np.int32), bs, hq, hkv, min_blocks)


def test_group_shares_the_common_leading_blocks():
    # Block size 4.  Sequences 0 and 1 share blocks [7, 1, 3]; sequence 2
    # shares only [7, 1]; sequence 3 starts elsewhere.
    tables = [[7, 1, 3, 10], [7, 1, 3, 11], [7, 1, 12], [5, 6]]
    lens = [14, 13, 9, 6]
    p = plan_of(tables, lens, 4, 4, 2)
    assert p.num_chunks == 1
    assert p.chunks() == [(0, 3, 8, 0)]             # 2 shared blocks = 8 tokens
    assert p.members() == [0, 1, 2]
    assert p.seq_start() == [8, 8, 8, 0]
    assert p.info.num_members == 3 and p.info.min_shared_tokens == 8 and p.info.group_size == 2
    assert p.info.plan_ints == 4 + 4 + 4 + 3
    # Stages: one for the 8 shared tokens, then own boxes of 4 tokens, 8 to
    # each warp's 32-column word: members 0, 1, 2 (one per warp) hold 2, 2, 1.
    assert p.info.min_chunk_stages == 2


def test_shared_length_leaves_every_member_its_newest_token():
    # Both hold blocks [2, 4, 6]; sequence 1 has exactly 12 tokens, so its
    # newest token is in block 6: at most floor((12 - 1) / 4) = 2 blocks are shared.
    p = plan_of([[2, 4, 6, 8], [2, 4, 6]], [16, 12], 4, 2, 2)
    assert p.chunks() == [(0, 2, 8, 0)]
    assert p.seq_start() == [8, 8]
    # One token past a block boundary: the full blocks before it are shared.
    p = plan_of([[2, 4, 6, 8], [2, 4, 6, 9]], [13, 13], 4, 2, 2)
    assert p.chunks() == [(0, 2, 12, 0)]


def test_short_groups_and_singletons_are_dropped():
    tables = [[1, 2, 3], [1, 2, 4], [9, 8, 7], [5, 6]]
    lens = [12, 12, 12, 8]
    assert plan_of(tables, lens, 4, 8, 8, min_blocks=3).num_chunks == 0   # only 2 shared
    p = plan_of(tables, lens, 4, 8, 8, min_blocks=2)
    assert p.chunks() == [(0, 2, 8, 0)]
    assert p.seq_start() == [8, 8, 0, 0]
    # One-token sequences have no full block before their newest token.
    assert plan_of([[1], [1]], [1, 1], 4, 2, 1).num_chunks == 0


def test_groups_are_cut_into_chunks_of_128_query_rows():
    # 70 members with 4 query heads per KV head: 32 members (128 rows) per chunk.
    tables = [[3, 5, 100 + r] for r in range(70)] + [[40, 41, 42]]
    lens = [10] * 70 + [10]
    p = plan_of(tables, lens, 4, 8, 2)
    assert p.chunks() == [(0, 32, 8, 0), (32, 32, 8, 0), (64, 6, 8, 0)]
    assert p.members() == list(range(70))
    # Two groups; the plan lists them in order of their first member.
    tables = [[1, 2, 9], [7, 8, 9], [1, 2, 10], [7, 8, 11], [7, 8, 12]]
    p = plan_of(tables, [11] * 5, 4, 2, 2)
    assert p.chunks() == [(0, 2, 8, 0), (2, 3, 8, 1)]
    assert p.members() == [0, 2, 1, 3, 4]
    # G = 16: 8 members per chunk (two to each 32-row warp); G = 7: 16
    # (four to a warp: 28 rows), not floor(128 / 7) = 18.
    p = plan_of([[1, 2, 50 + r] for r in range(9)], [9] * 9, 4, 32, 2)
    assert [c[1] for c in p.chunks()] == [8, 1]
    p = plan_of([[1, 2, 50 + r] for r in range(40)], [9] * 40, 4, 14, 2)
    assert [c[1] for c in p.chunks()] == [16, 16, 8]


def _script_tables(variant, **kw):
    script = workloads.shared_prefix_script(variant=variant, **kw)
    pool = pa.Pool(script.num_blocks, script.block_size, script.free_order)
    for kind, arg in script.ops:
        if kind == "add":
            pool.add_seq(arg)
        elif kind == "fork":
            pool.fork(arg)
        else:
            pool.append_token(arg)
    seqs = script.decode_seqs
    mb = max(len(pool.table(x)[0]) for x in seqs)
    bt, sl = pool.fill_tables(seqs, mb)
    return bt, sl


def test_forked_samples_share_their_prompt_blocks():
    # 16 requests of a 1018-token prompt, 8 samples each: the 63 full prompt
    # blocks are shared; the partly filled 64th was copied on write.
    bt, sl = _script_tables("fork", prompt_len=1018)
    p = pa.SharedPlan(bt, sl, 16, 32, 8)
    assert p.num_chunks == 16
    assert all(c[1] == 8 and c[2] == 63 * 16 for c in p.chunks())
    assert sorted(p.members()) == list(range(128))
    # A 1024-token prompt: all 64 prompt blocks are shared.
    bt, sl = _script_tables("fork", prompt_len=1024, num_requests=4)
    p = pa.SharedPlan(bt, sl, 16, 32, 8)
    assert [c[2] for c in p.chunks()] == [1024] * 4


def test_requests_on_a_common_prefix_share_it():
    # 128 requests forked from one 512-token prefix: one group, 32 blocks,
    # 4 chunks of 32 members (G = 4).
    bt, sl = _script_tables("prefix")
    p = pa.SharedPlan(bt, sl, 16, 32, 8)
    assert p.chunks() == [(0, 32, 512, 0), (32, 32, 512, 0), (64, 32, 512, 0), (96, 32, 512, 0)]
    assert p.seq_start() == [512] * 128
    assert p.info.min_shared_tokens == 512
    # 4 shared stages, then each warp's queue (8 members) in 16-token boxes,
    # 2 boxes to the warp's 32-column word in each stage.
    own = [(int(n) - 512 + 15) // 16 for n in sl]
    stages = [4 + -(-max(sum(own[c * 32 + w * 8:c * 32 + w * 8 + 8]) for w in range(4)) // 2)
              for c in range(4)]
    assert p.info.min_chunk_stages == min(stages)


def test_plan_argument_checks():
    bt = np.zeros((2, 2), dtype=np.int32)
    with pytest.raises(pa.PAError):
        pa.SharedPlan(bt, np.array([4, 40], dtype=np.int32), 16, 4, 2)   # table too short
    with pytest.raises(pa.PAError):
        pa.SharedPlan(bt, np.array([4, 4], dtype=np.int32), 12, 4, 2)    # block size
    with pytest.raises(pa.PAError):
        pa.SharedPlan(bt, np.array([4, 4], dtype=np.int32), 16, 5, 2)    # heads
    with pytest.raises(pa.PAError):
        pa.SharedPlan(bt, np.array([4, 4], dtype=np.int32), 16, 4, 2, 0)  # min blocks
    empty = pa.SharedPlan(np.zeros((0, 1), dtype=np.int32), np.zeros(0, dtype=np.int32), 16, 4, 2)
    assert empty.num_chunks == 0 and empty.info.plan_ints == 4
