"""The library's C++ block pool against the oracle's independent replay:
the pages' worked examples, random operation sequences step by step, the
all-or-nothing batch append, and slot mapping from block tables."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_78_gb300 as pa
import workloads
from oracle.pool_replay import BadState, OutOfBlocks, PoolReplay

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def head_order(n, head):
    return list(head) + [b for b in range(n) if b not in head]


def test_worked_example_matches_pages():
    g = golden("worked_example.json")
    pool = pa.Pool(8, g["block_size"], head_order(8, g["free_order_head"]))
    sid = pool.add_seq(g["prompt_tokens"])
    assert pool.table(sid) == (g["after_prompt"]["table"], 7)
    assert pool.append_token(sid) == (g["after_decode_1"]["slot"], None)
    assert pool.table(sid)[0] == g["after_decode_1"]["table"]
    assert pool.append_token(sid) == (g["after_decode_2"]["slot"], None)
    assert pool.table(sid)[0] == g["after_decode_2"]["table"]


def test_cow_example_matches_pages():
    g = golden("cow_example.json")
    pool = pa.Pool(8, g["block_size"], head_order(8, g["free_order_head"]))
    a1 = pool.add_seq(g["prompt_tokens"])
    a2 = pool.fork(a1)
    assert pool.ref_count(7) == 2 and pool.ref_count(1) == 2
    slot, pair = pool.append_token(a1)
    assert list(pair) == g["a1_write"]["pair"] and slot == g["a1_write"]["slot"]
    assert pool.table(a1)[0] == g["a1_write"]["table"]
    slot, pair = pool.append_token(a2)
    assert pair is None and slot == g["a2_write"]["slot"]
    for b, r in g["a2_write"]["refs"].items():
        assert pool.ref_count(int(b)) == r


def test_allocation_example_matches_pages():
    g = golden("allocation_example.json")
    pool = pa.Pool(128, g["block_size"], head_order(128, g["free_order_head"]))
    sid = pool.add_seq(g["prompt_tokens"])
    assert pool.table(sid)[0] == g["after_prompt"]["table"]
    for _ in range(g["appends_without_new_block"]):
        pool.append_token(sid)
    slot, _ = pool.append_token(sid)
    assert pool.table(sid)[0] == g["after_full"]["table"] and slot == g["after_full"]["slot"]


def _prefix_timeline(pool):
    """Drive `pool` (the library's or the oracle's) through the pages' prefix
    cache timeline and check every state the page states."""
    g = golden("prefix_cache_example.json")
    r0, cached = pool.add_seq_tokens(g["t1"]["tokens"])
    assert cached == g["t1"]["num_cached_tokens"]
    assert pool.table(r0)[0] == g["t1"]["table"]
    assert [b for b in range(g["num_blocks"]) if pool.is_cached(b)] == g["t1"]["cached_blocks"]
    for t in g["t2"]["append"]:
        pool.append_token(r0, t) if isinstance(pool, PoolReplay) else pool.append_token_id(r0, t)
    assert pool.table(r0)[0] == g["t2"]["table"]
    assert [b for b in range(g["num_blocks"]) if pool.is_cached(b)] == g["t2"]["cached_blocks"]
    r1, cached = pool.add_seq_tokens(g["t3"]["tokens"])
    assert cached == g["t3"]["num_cached_tokens"]
    assert pool.table(r1)[0] == g["t3"]["table"]
    refs = pool.ref if isinstance(pool, PoolReplay) else None
    for b, r in g["t3"]["refs"].items():
        assert (refs[int(b)] if refs else pool.ref_count(int(b))) == r
    pool.free_seq(r0)
    assert pool.free_queue() == g["t4"]["free_queue"]
    assert all(pool.is_cached(b) for b in g["t4"]["still_cached"])
    pool.free_seq(r1)
    assert pool.free_queue() == g["t5"]["free_queue"]
    r2, cached = pool.add_seq_tokens(g["t6"]["tokens"])
    assert cached == g["t6"]["num_cached_tokens"]
    assert pool.table(r2)[0] == g["t6"]["table"]
    assert pool.free_queue() == g["t6"]["free_queue"]
    return pool


def test_prefix_cache_timeline_matches_pages():
    g = golden("prefix_cache_example.json")
    pool = _prefix_timeline(pa.Pool(g["num_blocks"], g["block_size"]))
    assert not pool.is_cached(3)  # reused for request 2's partial last block: its hash is gone


def test_prefix_cache_timeline_matches_pages_in_the_oracle_replay():
    g = golden("prefix_cache_example.json")
    pool = _prefix_timeline(PoolReplay(g["num_blocks"], g["block_size"]))
    pool.check_invariants()
    assert not pool.is_cached(3)


def test_prefix_cache_never_shares_the_last_prompt_token():
    pool = pa.Pool(16, 4)
    a, _ = pool.add_seq_tokens(range(8))         # two full blocks, both registered
    b, cached = pool.add_seq_tokens(range(8))    # same 8 tokens: only (8 - 1) // 4 = 1 block shared
    assert cached == 4
    assert pool.table(b)[0][0] == pool.table(a)[0][0] and pool.table(b)[0][1] != pool.table(a)[0][1]
    c, cached = pool.add_seq_tokens(list(range(8)) + [99])
    assert cached == 8 and pool.table(c)[0][:2] == pool.table(a)[0]
    d, cached = pool.add_seq_tokens([1] + list(range(1, 9)))  # differs in the first token
    assert cached == 0


def test_prefix_cache_out_of_blocks_changes_nothing():
    pool = pa.Pool(5, 4)
    a, _ = pool.add_seq_tokens(range(12))        # blocks 0,1,2
    pool.free_seq(a)                             # queue 3 4 2 1 0, all three cached
    before = pool.free_queue()
    with pytest.raises(pa.OutOfBlocks):
        pool.add_seq_tokens(list(range(12)) + list(range(100, 112)))  # 3 shared + 3 new > 5
    assert pool.free_queue() == before and all(pool.is_cached(b) for b in (0, 1, 2))
    b, cached = pool.add_seq_tokens(list(range(12)) + [7])
    assert cached == 12 and pool.free_queue() == [4]  # 3 shared + one new block (3)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_operations_match_replay(seed):
    rng = np.random.default_rng(seed)
    nb, bs = 40, 4
    order = rng.permutation(nb)
    ours, ref = pa.Pool(nb, bs, order), PoolReplay(nb, bs, order)
    ours.set_cpu_blocks(nb // 2)
    ref.set_cpu_blocks(nb // 2)
    live = []
    resident = lambda: [x for x in live if x not in ref.swapped]
    pick = lambda xs: xs[int(rng.integers(len(xs)))]
    prompts = [[int(t) for t in rng.integers(0, 3, size=24)] for _ in range(4)]
    for step in range(1500):
        op = int(rng.integers(0, 8))
        if op == 5 and live:
            # prefix caching: prompts drawn as prefixes of a few shared streams
            base = prompts[int(rng.integers(len(prompts)))]
            toks = base[:int(rng.integers(0, len(base) + 1))] + \
                [int(t) for t in rng.integers(0, 3, size=int(rng.integers(0, 3)))]
            try:
                want = ref.add_seq_tokens(toks)
            except OutOfBlocks:
                with pytest.raises(pa.OutOfBlocks):
                    ours.add_seq_tokens(toks)
                continue
            assert ours.add_seq_tokens(toks) == want
            live.append(want[0])
        elif op == 6 and resident():
            sid = pick(resident())
            tok = int(rng.integers(0, 3))
            try:
                want = ref.append_token(sid, tok)
            except OutOfBlocks:
                with pytest.raises(pa.OutOfBlocks):
                    ours.append_token_id(sid, tok)
                continue
            assert ours.append_token_id(sid, tok) == want
        elif op == 7 and step % 97 == 0:
            ref.reset_prefix_cache()
            ours.reset_prefix_cache()
        elif op == 7 and live:
            # swap a sequence group out (all sequences sharing blocks with one) or back in
            sid = live[int(rng.integers(len(live)))]
            out = not ref.tables[sid] or sid not in ref.swapped
            group, frontier = {sid}, [sid]
            while frontier:
                x = frontier.pop()
                for y in live:
                    if y not in group and (y in ref.swapped) == (x in ref.swapped) and \
                            set(ref.tables[y]) & set(ref.tables[x]):
                        group.add(y)
                        frontier.append(y)
            group = sorted(group)
            try:
                want = ref.swap_out(group) if out else ref.swap_in(group)
            except (OutOfBlocks, BadState) as exc:
                with pytest.raises(pa.OutOfBlocks if isinstance(exc, OutOfBlocks) else pa.PAError):
                    ours.swap_out(group) if out else ours.swap_in(group)
                continue
            assert _pairs(ours.swap_out(group) if out else ours.swap_in(group)) == want
        elif op == 0 or not live:
            n = int(rng.integers(0, 14))
            try:
                want = ref.add_seq(n)
            except OutOfBlocks:
                with pytest.raises(pa.OutOfBlocks):
                    ours.add_seq(n)
                continue
            assert ours.add_seq(n) == want
            live.append(want)
        elif op == 1 and resident():
            p = pick(resident())
            want = ref.fork(p)
            assert ours.fork(p) == want
            live.append(want)
        elif op in (2, 3) and resident():
            sid = pick(resident())
            try:
                want = ref.append_token(sid)
            except OutOfBlocks:
                with pytest.raises(pa.OutOfBlocks):
                    ours.append_token(sid)
                continue
            assert ours.append_token(sid) == want
        elif op == 4:
            sid = live.pop(int(rng.integers(len(live))))
            ref.free_seq(sid)
            ours.free_seq(sid)
        assert ours.num_free() == ref.num_free()
        assert ours.num_free_cpu() == len(ref.cpu_free)
        assert ours.free_queue() == ref.free_queue()
        for sid in live:
            assert ours.table(sid) == ref.table(sid)
        for b in range(nb):
            assert ours.ref_count(b) == ref.ref[b]
            assert ours.is_cached(b) == ref.is_cached(b)
        ref.check_invariants()


def test_batch_append_is_all_or_nothing():
    pool = pa.Pool(6, 4)
    a = pool.add_seq(4)      # block 0 full
    b = pool.fork(a)         # shares block 0
    c = pool.add_seq(6)      # blocks 1, 2
    d = pool.fork(c)         # shares 1, 2 (block 2 half full)
    before = [pool.table(x) for x in (a, b, c, d)], pool.num_free()
    # a: new block, b: new block, c: copy-on-write of block 2, d: in place -> 3 blocks; 3 free
    slots, pairs = pool.append_tokens([a, b, c, d])
    assert pairs.tolist() == [[2, pool.table(c)[0][1]]]
    assert pool.num_free() == 0
    for x in (a, b, c, d):
        pool.free_seq(x)
    pool2 = pa.Pool(5, 4)
    a = pool2.add_seq(4)
    b = pool2.fork(a)
    c = pool2.add_seq(6)
    d = pool2.fork(c)
    before = [pool2.table(x) for x in (a, b, c, d)], pool2.num_free(), \
        [pool2.ref_count(i) for i in range(5)]
    with pytest.raises(pa.OutOfBlocks):
        pool2.append_tokens([a, b, c, d])       # needs 3 blocks, 2 free
    after = [pool2.table(x) for x in (a, b, c, d)], pool2.num_free(), \
        [pool2.ref_count(i) for i in range(5)]
    assert after == before
    # and the free list order survived: the next allocation takes the same block
    ref = PoolReplay(5, 4)
    ra = ref.add_seq(4); rb = ref.fork(ra); rc = ref.add_seq(6); ref.fork(rc)
    assert pool2.append_token(a) == ref.append_token(ra)


def test_fill_tables_and_slot_mapping_agree_with_oracle():
    script = workloads.shared_prefix_script(variant="fork", num_requests=3, samples=4,
                                            prompt_len=37)
    pool = pa.Pool(script.num_blocks, script.block_size, script.free_order)
    ref = PoolReplay(script.num_blocks, script.block_size, script.free_order)
    for op, arg in script.ops:
        if op == "add":
            assert pool.add_seq(arg) == ref.add_seq(arg)
        elif op == "fork":
            assert pool.fork(arg) == ref.fork(arg)
        else:
            assert pool.append_token(arg) == ref.append_token(arg)
    seqs = script.decode_seqs
    mb = max(len(ref.table(s)[0]) for s in seqs) + 1
    bt, sl = pool.fill_tables(seqs, mb)
    for i, s in enumerate(seqs):
        t, n = ref.table(s)
        assert bt[i, :len(t)].tolist() == t and int(sl[i]) == n
    rng = np.random.default_rng(0)
    si = rng.integers(0, len(seqs), size=50)
    pos = np.array([rng.integers(0, int(sl[i])) for i in si])
    ours = pa.pa_slot_mapping(bt, script.block_size, script.num_blocks,
                              torch.from_numpy(si), torch.from_numpy(pos))
    want = oracle.slot_mapping(bt.numpy(), si, pos, script.block_size)
    assert ours.tolist() == want.tolist()
    for k in range(10):
        assert pool.slot(seqs[si[k]], int(pos[k])) == ref.slot(seqs[si[k]], int(pos[k]))


def test_slot_mapping_rejects_out_of_table_positions():
    bt = torch.tensor([[3, 1]], dtype=torch.int32)
    with pytest.raises(pa.PAError):
        pa.pa_slot_mapping(bt, 4, 8, torch.tensor([0]), torch.tensor([8]))
    with pytest.raises(pa.PAError):
        pa.pa_slot_mapping(bt, 4, 8, torch.tensor([1]), torch.tensor([0]))


def test_pool_errors():
    pool = pa.Pool(4, 4)
    with pytest.raises(pa.PAError):
        pool.fork(5)
    with pytest.raises(pa.PAError):
        pool.free_seq(0)
    with pytest.raises(pa.PAError):
        pa.Pool(4, 4, [0, 1, 1, 2])


def test_usage_counts_tokens_and_blocks():
    pool = pa.Pool(32, 16)
    a = pool.add_seq(50)            # 4 blocks, 14 slots unused in the last
    assert pool.usage() == (50, 4)
    b = pool.fork(a)                # shared blocks count once, tokens per sequence
    assert pool.usage() == (100, 4)
    pool.append_token(b)            # copy-on-write of the partly filled last block
    assert pool.usage() == (101, 5)
    pool.free_seq(a)
    assert pool.usage() == (51, 4)
    # waste stays within the last block: at most block_size - 1 slots per sequence
    c = pool.add_seq(33)
    tokens, blocks = pool.usage()
    assert blocks * 16 - tokens == (64 - 51) + (48 - 33)



def _pairs(t):
    return [tuple(int(x) for x in row) for row in t.tolist()]


def test_swap_preempts_a_sequence_group_whole():
    # Two samples of one request share a prompt; a second request needs the
    # GPU blocks, so the group is swapped out whole, and back in after.
    ours, ref = pa.Pool(8, 4), PoolReplay(8, 4)
    for p in (ours, ref):
        p.set_cpu_blocks(8)
    a = ours.add_seq(10); assert ref.add_seq(10) == a          # blocks 0,1,2 (2 tokens in 2)
    a2 = ours.fork(a); assert ref.fork(a) == a2
    b = ours.add_seq(16); assert ref.add_seq(16) == b          # blocks 3..6; one block left
    with pytest.raises(pa.PAError) as e:
        ours.swap_out([a])                                      # would split the group
    assert e.value.status == pa.PA_ERR_BAD_STATE
    got = _pairs(ours.swap_out([a, a2]))
    assert got == ref.swap_out([a, a2]) == [(0, 0), (1, 1), (2, 2)]
    assert ours.num_free() == ref.num_free() == 4 and ours.num_free_cpu() == 5
    assert ours.is_swapped(a) and ours.table(a)[0] == ref.table(a)[0] == [0, 1, 2]
    for call in (lambda: ours.append_token(a), lambda: ours.fork(a2),
                 lambda: ours.fill_tables([a], 8), lambda: ours.slot(a, 0)):
        with pytest.raises(pa.PAError) as e:
            call()
        assert e.value.status == pa.PA_ERR_BAD_STATE
    for _ in range(5):                                          # the other request grows
        assert ours.append_token(b) == ref.append_token(b)
    ours.free_seq(b); ref.free_seq(b)
    got = _pairs(ours.swap_in([a2, a]))
    assert got == ref.swap_in([a2, a])
    assert ours.table(a) == ref.table(a) and ours.table(a2) == ref.table(a2)
    assert all(ours.ref_count(x) == 2 for x in ours.table(a)[0])
    slot, pair = ours.append_token(a2)                          # copy-on-write still works
    assert (slot, pair) == ref.append_token(a2) and pair is not None
    assert ours.num_free_cpu() == 8
    ref.check_invariants()


def test_swap_limits():
    pool = pa.Pool(6, 4)
    with pytest.raises(pa.PAError) as e:
        pool.set_cpu_blocks(7)                                  # never more than the GPU has
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    pool.set_cpu_blocks(2)
    a = pool.add_seq(12)
    with pytest.raises(pa.OutOfBlocks):
        pool.swap_out([a])                                      # 3 blocks, 2 CPU blocks
    assert not pool.is_swapped(a) and pool.num_free() == 3 and pool.num_free_cpu() == 2
    b = pool.add_seq(8)
    pool.swap_out([b])
    with pytest.raises(pa.PAError) as e:
        pool.set_cpu_blocks(4)                                  # not while swapped
    assert e.value.status == pa.PA_ERR_BAD_STATE
    pool.free_seq(b)                                            # frees its CPU blocks
    assert pool.num_free_cpu() == 2 and pool.num_free() == 3
