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
from oracle.pool_replay import OutOfBlocks, PoolReplay

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


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_operations_match_replay(seed):
    rng = np.random.default_rng(seed)
    nb, bs = 40, 4
    order = rng.permutation(nb)
    ours, ref = pa.Pool(nb, bs, order), PoolReplay(nb, bs, order)
    live = []
    for step in range(1500):
        op = int(rng.integers(0, 5))
        if op == 0 or not live:
            n = int(rng.integers(0, 14))
            try:
                want = ref.add_seq(n)
            except OutOfBlocks:
                with pytest.raises(pa.OutOfBlocks):
                    ours.add_seq(n)
                continue
            assert ours.add_seq(n) == want
            live.append(want)
        elif op == 1:
            p = live[int(rng.integers(len(live)))]
            want = ref.fork(p)
            assert ours.fork(p) == want
            live.append(want)
        elif op in (2, 3):
            sid = live[int(rng.integers(len(live)))]
            try:
                want = ref.append_token(sid)
            except OutOfBlocks:
                with pytest.raises(pa.OutOfBlocks):
                    ours.append_token(sid)
                continue
            assert ours.append_token(sid) == want
        else:
            sid = live.pop(int(rng.integers(len(live))))
            ref.free_seq(sid)
            ours.free_seq(sid)
        assert ours.num_free() == ref.num_free()
        for sid in live:
            assert ours.table(sid) == ref.table(sid)
        for b in range(nb):
            assert ours.ref_count(b) == ref.ref[b]


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
