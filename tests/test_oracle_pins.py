"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here checks the oracle against itself: each test compares it with a
value the pages print (tests/golden/*.json), a library routine (torch's
scaled_dot_product_attention in float64, numpy indexing), a closed form or
an invariant that holds exactly.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import sizing
from oracle.pool_replay import OutOfBlocks, PoolReplay

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def pool_with_head(num_blocks, block_size, head):
    rest = [b for b in range(num_blocks) if b not in head]
    return PoolReplay(num_blocks, block_size, free_order=list(head) + rest)


# --------------------------------------------------------------------------
# sizing closed forms
# --------------------------------------------------------------------------

def test_sizing_opt13b():
    g = golden("sizing.json")["opt13b"]
    per_tok = sizing.kv_bytes_per_token(g["num_layers"], g["hidden_size"], g["dtype_bytes"])
    assert per_tok == g["kv_bytes_per_token"] == 800 * 1024
    req = per_tok * g["request_tokens"]
    assert req == g["request_bytes"]
    assert abs(req / 1e9 - 1.6) < 0.1          # "about 1.6 GB"
    lo, hi = g["requests_range"]
    assert lo <= g["gpu_bytes"] / req <= hi     # "40 to 50 requests on 80 GB"


def test_sizing_qwen2_page_and_tensor():
    g = golden("sizing.json")["qwen2_0_5b"]
    page = sizing.page_size_bytes(g["block_size"], g["num_kv_heads"], g["head_size"],
                                  g["dtype_bytes"])
    assert page == g["page_size"] == 8192
    assert sizing.layer_tensor_bytes(page, g["num_blocks"]) == g["layer_tensor_bytes"]
    shape = sizing.cache_shape(g["num_blocks"], g["block_size"], g["num_kv_heads"],
                               g["head_size"])
    assert list(shape) == g["cache_shape"]
    assert int(np.prod(shape)) * g["dtype_bytes"] == g["layer_tensor_bytes"]


def test_blocks_for_tokens():
    for n, bs, want in golden("sizing.json")["blocks_for_tokens"]["cases"]:
        assert sizing.blocks_for_tokens(n, bs) == want


# --------------------------------------------------------------------------
# host block bookkeeping: the pages' worked examples
# --------------------------------------------------------------------------

def test_worked_example_allocation():
    g = golden("worked_example.json")
    pool = pool_with_head(8, g["block_size"], g["free_order_head"])
    sid = pool.add_seq(g["prompt_tokens"])
    assert pool.table(sid)[0] == g["after_prompt"]["table"]
    assert pool.filled(sid) == g["after_prompt"]["filled"]
    slot, pair = pool.append_token(sid)
    assert pair is None and slot == g["after_decode_1"]["slot"]
    assert pool.table(sid)[0] == g["after_decode_1"]["table"]
    assert pool.filled(sid) == g["after_decode_1"]["filled"]
    slot, pair = pool.append_token(sid)
    assert pair is None and slot == g["after_decode_2"]["slot"]
    assert pool.table(sid)[0] == g["after_decode_2"]["table"]
    assert pool.filled(sid) == g["after_decode_2"]["filled"]
    pool.check_invariants()


def test_cow_example():
    g = golden("cow_example.json")
    pool = pool_with_head(8, g["block_size"], g["free_order_head"])
    a1 = pool.add_seq(g["prompt_tokens"])
    a2 = pool.fork(a1)
    for b, r in g["after_fork"]["refs"].items():
        assert pool.ref[int(b)] == r
    assert pool.table(a2)[0] == g["after_fork"]["table"]
    slot, pair = pool.append_token(a1)
    assert list(pair) == g["a1_write"]["pair"] and slot == g["a1_write"]["slot"]
    assert pool.table(a1)[0] == g["a1_write"]["table"]
    for b, r in g["a1_write"]["refs"].items():
        assert pool.ref[int(b)] == r
    slot, pair = pool.append_token(a2)
    assert pair is None and slot == g["a2_write"]["slot"]
    assert pool.table(a2)[0] == g["a2_write"]["table"]
    for b, r in g["a2_write"]["refs"].items():
        assert pool.ref[int(b)] == r
    pool.check_invariants()


def test_allocation_example():
    g = golden("allocation_example.json")
    pool = pool_with_head(128, g["block_size"], g["free_order_head"])
    sid = pool.add_seq(g["prompt_tokens"])
    assert pool.table(sid)[0] == g["after_prompt"]["table"]
    for _ in range(g["appends_without_new_block"]):
        _, pair = pool.append_token(sid)
        assert pair is None
        assert pool.table(sid)[0] == g["after_prompt"]["table"]
    slot, _ = pool.append_token(sid)
    assert pool.table(sid)[0] == g["after_full"]["table"]
    assert slot == g["after_full"]["slot"]


def test_pool_out_of_blocks_is_transactional():
    pool = PoolReplay(3, 4)
    a = pool.add_seq(8)
    with pytest.raises(OutOfBlocks):
        pool.add_seq(5)
    assert pool.num_free() == 1
    pool.append_token(a)  # position 8 -> third block
    b = pool.fork(a)
    before = (pool.table(a), pool.table(b), list(pool.ref), pool.num_free())
    with pytest.raises(OutOfBlocks):
        pool.append_token(b)  # would copy-on-write block 2 but nothing is free
    assert (pool.table(a), pool.table(b), list(pool.ref), pool.num_free()) == before
    pool.check_invariants()


def test_pool_random_ops_invariants():
    rng = np.random.default_rng(11)
    pool = PoolReplay(48, 4, free_order=rng.permutation(48))
    live = []
    for _ in range(3000):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                live.append(pool.add_seq(int(rng.integers(0, 12))))
            elif op == 1:
                live.append(pool.fork(live[rng.integers(len(live))]))
            elif op == 2:
                pool.append_token(live[rng.integers(len(live))])
            else:
                pool.free_seq(live.pop(rng.integers(len(live))))
        except OutOfBlocks:
            pass
        pool.check_invariants()
    for sid in live:
        pool.free_seq(sid)
    assert pool.num_free() == 48


# --------------------------------------------------------------------------
# decode attention
# --------------------------------------------------------------------------

def contiguous_keys_values(case, s):
    a, b = case.seq_starts[s], case.seq_starts[s + 1]
    return oracle.to_f64(case.keys[a:b]), oracle.to_f64(case.values[a:b])


def sdpa_reference(case):
    """torch's scaled_dot_product_attention in float64 over the unpaged tokens."""
    out = np.zeros((case.num_seqs, case.num_heads, case.head_size))
    g = case.num_heads // case.num_kv_heads
    for s in range(case.num_seqs):
        k, v = contiguous_keys_values(case, s)
        if k.shape[0] == 0:
            continue
        q = torch.from_numpy(oracle.to_f64(case.query[s]))[None, :, None, :]
        kt = torch.from_numpy(k.transpose(1, 0, 2).copy())[None]
        vt = torch.from_numpy(v.transpose(1, 0, 2).copy())[None]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, kt, vt, scale=case.scale, enable_gqa=(g > 1))
        out[s] = o[0, :, 0, :].numpy()
    return out


CASES = [
    lambda: workloads.tiny("bf16"),
    lambda: workloads.tiny("fp32"),
    lambda: workloads.custom(5, 8, 2, 64, 16, [1, 15, 16, 17, 200], "bf16", seed=5),
    lambda: workloads.custom(3, 6, 3, 128, 8, [9, 64, 130], "fp32", seed=6),
    lambda: workloads.custom(2, 7, 1, 64, 32, [33, 97], "bf16", seed=7),
]


@pytest.mark.parametrize("make", CASES)
def test_decode_equals_contiguous_sdpa(make):
    case = make()
    cache = oracle.fill_cache(case)
    got = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    np.testing.assert_allclose(got, sdpa_reference(case), rtol=1e-12, atol=1e-12)


def test_decode_indexes_blocks_like_numpy_gather():
    """Page 4's kv_cache[:, table, ...]: gathering the table's blocks with numpy
    fancy indexing and flattening gives the sequence's tokens in order."""
    case = workloads.tiny("bf16")
    cache = oracle.fill_cache(case)
    for s in range(case.num_seqs):
        n = int(case.seq_lens[s])
        nblk = -(-n // case.block_size)
        table = case.block_tables[s, :nblk]
        gathered = cache[:, table].reshape(2, nblk * case.block_size, case.num_kv_heads,
                                           case.head_size)[:, :n]
        a, b = case.seq_starts[s], case.seq_starts[s + 1]
        assert np.array_equal(gathered[0], case.keys[a:b])
        assert np.array_equal(gathered[1], case.values[a:b])


def test_decode_block_relabelling_is_bit_identical():
    case = workloads.custom(4, 4, 2, 64, 8, [5, 40, 64, 77], "bf16", seed=9)
    cache = oracle.fill_cache(case)
    ref = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    perm = np.random.default_rng(1).permutation(case.num_blocks)
    cache2 = np.empty_like(cache)
    cache2[:, perm] = cache
    tables2 = perm[case.block_tables].astype(np.int32)
    got = oracle.decode(case.query, cache2, tables2, case.seq_lens, case.scale)
    assert np.array_equal(got, ref)


def test_decode_does_not_depend_on_the_thread_count():
    # The baseline times the oracle on every core and on one; each (sequence,
    # query head) row is computed by one thread in a fixed order, so both
    # give the same bits.
    case = workloads.custom(4, 8, 2, 64, 8, [5, 40, 64, 77], "bf16", seed=19)
    cache = oracle.fill_cache(case)
    ref = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    every = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        assert oracle.num_threads() == 1
        got = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    finally:
        oracle.set_num_threads(every)
    assert oracle.num_threads() == every
    assert np.array_equal(got, ref)


def test_unpaged_layout_of_the_same_tokens_gives_the_same_output():
    # The bench's paging-overhead run: consecutive physical blocks are one more
    # relabelling of the same tokens.
    case = workloads.custom(4, 4, 2, 64, 8, [5, 40, 64, 77], "bf16", seed=9)
    flat = workloads.contiguous(case)
    assert [list(r[:-(-int(n) // 8)]) for r, n in zip(flat.block_tables, flat.seq_lens)] == \
        [[0], [1, 2, 3, 4, 5], [6, 7, 8, 9, 10, 11, 12, 13], list(range(14, 24))]
    ref = oracle.decode(case.query, oracle.fill_cache(case), case.block_tables, case.seq_lens,
                        case.scale)
    got = oracle.decode(flat.query, oracle.fill_cache(flat), flat.block_tables, flat.seq_lens,
                        flat.scale)
    assert np.array_equal(got, ref)


def test_decode_single_token_returns_its_value():
    case = workloads.custom(3, 4, 4, 64, 4, [1, 1, 1], "bf16", seed=3)
    cache = oracle.fill_cache(case)
    got = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    for s in range(3):
        _, v = contiguous_keys_values(case, s)
        assert np.array_equal(got[s], v[0])


def test_decode_equal_keys_average_values():
    case = workloads.custom(2, 2, 2, 64, 4, [13, 30], "fp32", seed=4)
    case.keys[:] = case.keys[0:1]
    cache = oracle.fill_cache(case)
    got = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    for s in range(2):
        _, v = contiguous_keys_values(case, s)
        np.testing.assert_allclose(got[s], np.broadcast_to(v.mean(axis=0), got[s].shape),
                                   rtol=0, atol=1e-12)


def test_decode_dominant_logit_selects_its_value():
    case = workloads.custom(2, 2, 2, 64, 4, [21, 50], "fp32", seed=8)
    cache = oracle.fill_cache(case)
    scale = 1e4
    got = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, scale)
    for s in range(2):
        k, v = contiguous_keys_values(case, s)
        q = oracle.to_f64(case.query[s])
        for h in range(2):
            j = int(np.argmax(k[:, h] @ q[h]))
            np.testing.assert_allclose(got[s, h], v[j, h], rtol=0, atol=1e-9)


def test_decode_gqa_equals_repeated_kv_heads():
    case = workloads.custom(3, 12, 3, 64, 8, [17, 48, 99], "bf16", seed=12)
    cache = oracle.fill_cache(case)
    got = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    rep = np.ascontiguousarray(np.repeat(cache, 4, axis=3))  # head h -> heads 4h..4h+3
    mha = oracle.decode(case.query, rep, case.block_tables, case.seq_lens, case.scale)
    assert np.array_equal(got, mha)


def test_decode_zero_length_gives_zero_row():
    case = workloads.custom(3, 4, 2, 64, 4, [0, 5, 0], "bf16", seed=13)
    cache = oracle.fill_cache(case)
    got = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    np.testing.assert_allclose(got, sdpa_reference(case), rtol=1e-12, atol=1e-12)


def test_decode_ignores_stale_slots_past_seq_len():
    """The garbage-filled tail of a last block (NaN and Inf patterns included)
    must not reach the output."""
    case = workloads.custom(2, 4, 4, 64, 16, [3, 21], "bf16", seed=14, cache_fill="garbage")
    cache = oracle.fill_cache(case)
    got = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, sdpa_reference(case), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("partition", [4, 8, 12, 32, 64, 1000])
def test_split_partials_combine_to_single_pass(partition):
    case = workloads.custom(4, 8, 2, 64, 4, [1, 31, 64, 150], "bf16", seed=15)
    cache = oracle.fill_cache(case)
    ref = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    parts = -(-150 // partition)
    m, l, acc = oracle.decode_partials(case.query, cache, case.block_tables, case.seq_lens,
                                       case.scale, partition, parts)
    got = oracle.combine_partials(m, l, acc)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_worked_example_decode_steps_match_contiguous_attention():
    """Replay the worked example end to end: prompt of 7 tokens in blocks 7 and
    1, then two decode steps; after each step the paged decode over 8 and 9
    tokens equals attention over the same tokens laid out contiguously."""
    g = golden("worked_example.json")
    bs = g["block_size"]
    rng = np.random.default_rng(21)
    toks_k = workloads.random_values(rng, (9, 1, 64), "fp32")
    toks_v = workloads.random_values(rng, (9, 1, 64), "fp32")
    q = workloads.random_values(rng, (1, 1, 64), "fp32")
    pool = pool_with_head(8, bs, g["free_order_head"])
    sid = pool.add_seq(7)
    cache = np.zeros((2, 8, bs, 1, 64), dtype=np.float32)
    oracle.reshape_and_cache(cache, toks_k[:7], toks_v[:7],
                             np.array([pool.slot(sid, p) for p in range(7)]))
    for n in (8, 9):
        slot, _ = pool.append_token(sid)
        oracle.reshape_and_cache(cache, toks_k[n - 1:n], toks_v[n - 1:n], np.array([slot]))
        table, length = pool.table(sid)
        assert length == n
        bt = np.array([table + [0] * (4 - len(table))], dtype=np.int32)
        got = oracle.decode(q, cache, bt, np.array([n], dtype=np.int32), 0.125)
        qq = torch.from_numpy(q.astype(np.float64))[None, :, :, :].transpose(1, 2)
        kk = torch.from_numpy(toks_k[:n].astype(np.float64)).transpose(0, 1)[None]
        vv = torch.from_numpy(toks_v[:n].astype(np.float64)).transpose(0, 1)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=0.125)
        np.testing.assert_allclose(got[0, 0], ref[0, 0, 0].numpy(), rtol=1e-12, atol=1e-12)
    assert pool.table(sid)[0] == g["after_decode_2"]["table"]


def test_reshape_and_cache_places_worked_example_token():
    """The first decode token of the worked example lands at physical block 1,
    offset 3 (the free place of logical block 1)."""
    cache = np.zeros((2, 8, 4, 2, 64), dtype=np.uint16)
    k = np.arange(2 * 64, dtype=np.uint16).reshape(1, 2, 64) + 1
    v = k + 1000
    oracle.reshape_and_cache(cache, k, v, np.array([7]))
    assert np.array_equal(cache[0, 1, 3], k[0]) and np.array_equal(cache[1, 1, 3], v[0])
    cache[0, 1, 3] = 0
    cache[1, 1, 3] = 0
    assert not cache.any()


def test_reshape_and_cache_skips_padding_and_matches_numpy_assignment():
    rng = np.random.default_rng(3)
    nb, bs, h, d = 16, 8, 3, 64
    cache = workloads.garbage_values(rng, (2, nb, bs, h, d), "bf16")
    ref = cache.copy()
    slots = rng.choice(nb * bs, size=40, replace=False).astype(np.int64)
    slots[::7] = -1
    k = workloads.random_values(rng, (40, h, d), "bf16")
    v = workloads.random_values(rng, (40, h, d), "bf16")
    oracle.reshape_and_cache(cache, k, v, slots)
    flat = ref.reshape(2, nb * bs, h, d)
    keep = slots >= 0
    flat[0, slots[keep]] = k[keep]
    flat[1, slots[keep]] = v[keep]
    assert np.array_equal(cache, ref)


def test_copy_blocks_matches_numpy_assignment():
    rng = np.random.default_rng(4)
    cache = workloads.random_values(rng, (2, 20, 4, 2, 64), "fp32")
    ref = cache.copy()
    pairs = np.array([[3, 11], [5, 0], [19, 7]], dtype=np.int64)
    oracle.copy_blocks(cache, pairs)
    for src, dst in pairs:
        ref[:, dst] = ref[:, src]
    assert np.array_equal(cache, ref)


def test_copy_on_write_copy_keeps_decode_of_the_sharer():
    """After the copy, a sequence reading the copy sees the same attention as
    one reading the original block."""
    case = workloads.custom(1, 4, 2, 64, 4, [10], "bf16", seed=16, spare_blocks=4)
    cache = oracle.fill_cache(case)
    ref = oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale)
    used = set(case.block_tables[0, :3].tolist())
    dst = next(b for b in range(case.num_blocks) if b not in used)
    src = int(case.block_tables[0, 2])
    oracle.copy_blocks(cache, np.array([[src, dst]]))
    bt = case.block_tables.copy()
    bt[0, 2] = dst
    got = oracle.decode(case.query, cache, bt, case.seq_lens, case.scale)
    assert np.array_equal(got, ref)
