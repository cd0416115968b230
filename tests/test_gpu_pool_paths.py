"""GPU parity of the host pool's prefix caching and swapping, end to end: the
library's pool and the oracle's replay are driven with the same operations,
the GPU cache gets only the writes and copies the library's pool asks for,
and the decode over the pool's tables is compared with the oracle.

Prefix caching (itan.pw "vLLMにおけるKVCacheマネージャーの詳細解説", sections
"KVCacheManagerの処理詳細" and "プレイフィックスキャッシュの詳細"): a request
admitted with token ids shares the cached blocks of its longest known prefix,
and only its other tokens' K/V are computed and written.  A token's K/V here
is a seeded function of the token ids up to it (as a model's would be), so
the decode over the shared blocks must equal attention over each sequence's
own tokens laid out contiguously.

Swapping (studying-code.tistory.com/16, sections "All-or-Nothing Eviction"
and "스와핑(Swapping)"): a sequence group leaves for page-locked host blocks
and comes back to other GPU blocks; the copies are checked against the
oracle's block copy and the returning group's decode against the oracle."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_78_gb300 as pa
import workloads
from gpu_util import assert_close, to_device, to_f64, to_host_bits
from oracle.pool_replay import PoolReplay

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS = 8, 2, 128, 16


@pytest.fixture(autouse=True)
def clean_error_word():
    pa.pa_get_device_error()
    yield


def kv_of_prefix(tokens):
    """K and V rows of the last token of `tokens`, drawn from a generator
    seeded by the whole prefix (the same prefix always gives the same rows)."""
    key = np.asarray(tokens, dtype=np.int64)
    rng = np.random.default_rng([len(tokens), zlib.crc32(key.tobytes())])
    return (workloads.random_values(rng, (HKV, D), "bf16"),
            workloads.random_values(rng, (HKV, D), "bf16"))


class Side:
    """The GPU cache with the library's pool, and the oracle's cache with the
    oracle's replay, fed the same operations."""

    def __init__(self, num_blocks, seed):
        self.rng = np.random.default_rng(seed)
        order = self.rng.permutation(num_blocks).astype(np.int32)
        self.pool = pa.Pool(num_blocks, BS, order)
        self.ref = PoolReplay(num_blocks, BS, order)
        shape = (2, num_blocks, BS, HKV, D)
        self.cache_dev = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        self.cache_ref = np.zeros(shape, dtype=np.uint16)
        self.tokens = {}

    def write(self, slots, rows):
        """K/V rows (list of (k, v)) to their slots, on both sides."""
        if not rows:
            return
        k = np.stack([r[0] for r in rows])
        v = np.stack([r[1] for r in rows])
        s = np.asarray(slots, dtype=np.int64)
        pa.pa_reshape_and_cache(self.cache_dev, to_device(k), to_device(v), to_device(s))
        oracle.reshape_and_cache(self.cache_ref, k, v, s)

    def admit(self, tokens):
        """A request by token ids: only the tokens past the cached prefix get
        their K/V computed and written.  Returns (sequence id, cached tokens)."""
        sid, cached = self.pool.add_seq_tokens(tokens)
        rsid, rcached = self.ref.add_seq_tokens(tokens)
        assert (sid, cached) == (rsid, rcached)
        slots = [self.pool.slot(sid, p) for p in range(cached, len(tokens))]
        assert slots == [self.ref.slot(sid, p) for p in range(cached, len(tokens))]
        self.write(slots, [kv_of_prefix(tokens[:p + 1]) for p in range(cached, len(tokens))])
        self.tokens[sid] = list(tokens)
        return sid, cached

    def generate(self, sid, token):
        """One decode-step token of a sequence: slot (and any copy-on-write
        pair) from the pool, its K/V written."""
        slot, pair = self.pool.append_token_id(sid, token)
        rslot, rpair = self.ref.append_token(sid, token)
        assert (slot, pair) == (rslot, rpair)
        if pair is not None:
            pairs = np.array([pair], dtype=np.int64)
            pa.pa_copy_blocks(self.cache_dev, to_device(pairs))
            oracle.copy_blocks(self.cache_ref, pairs)
        self.tokens[sid].append(int(token))
        self.write([slot], [kv_of_prefix(self.tokens[sid])])

    def free(self, sid):
        self.pool.free_seq(sid)
        self.ref.free_seq(sid)
        del self.tokens[sid]

    def tables(self, seqs):
        mb = max(len(self.ref.table(s)[0]) for s in seqs)
        bt, sl = self.pool.fill_tables(seqs, mb)
        for r, s in enumerate(seqs):
            t, n = self.ref.table(s)
            assert bt[r, :len(t)].tolist() == t and int(sl[r]) == n
        return bt, sl

    def decode(self, seqs, q, partition=-1):
        """The library's decode over its pool's tables, and the oracle's over
        the replay's tables and cache (the tables were checked equal)."""
        bt, sl = self.tables(seqs)
        out = torch.empty((len(seqs), HQ, D), dtype=torch.bfloat16, device="cuda")
        max_len = int(sl.max())
        ws = pa.alloc_workspace(pa.pa_decode_workspace_size(self.cache_dev, len(seqs), HQ,
                                                            max_len, partition), "cuda")
        scale = 1.0 / np.sqrt(D)
        pa.pa_decode(out, to_device(q), self.cache_dev, bt.cuda(), sl.cuda(), scale, max_len,
                     partition, ws)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        want = oracle.decode(q, self.cache_ref, bt.numpy(), sl.numpy(), scale)
        return to_f64(out), want, bt.numpy(), sl.numpy()

    def check_cache(self):
        torch.cuda.synchronize()
        assert np.array_equal(to_host_bits(self.cache_dev), self.cache_ref), \
            "cache differs from the oracle"


def contiguous_reference(tokens_of_seqs, q):
    """Attention over each sequence's own tokens, K/V recomputed from its
    token ids and laid out on consecutive blocks (no sharing at all)."""
    lens = np.array([len(t) for t in tokens_of_seqs], dtype=np.int32)
    blocks = [-(-int(n) // BS) for n in lens]
    cache = np.zeros((2, sum(blocks), BS, HKV, D), dtype=np.uint16)
    bt = np.zeros((len(lens), max(blocks)), dtype=np.int32)
    b0 = 0
    for r, toks in enumerate(tokens_of_seqs):
        bt[r, :blocks[r]] = np.arange(b0, b0 + blocks[r])
        rows = [kv_of_prefix(toks[:p + 1]) for p in range(len(toks))]
        slots = np.arange(len(toks), dtype=np.int64) + b0 * BS
        oracle.reshape_and_cache(cache, np.stack([x[0] for x in rows]),
                                 np.stack([x[1] for x in rows]), slots)
        b0 += blocks[r]
    return oracle.decode(q, cache, bt, lens, 1.0 / np.sqrt(D))


@pytest.mark.parametrize("partition", [-1, 0, 32])
def test_prefix_cache_hits_decode_against_the_oracle(partition):
    side = Side(num_blocks=48, seed=61)
    rng = np.random.default_rng(62)
    prompt_a = rng.integers(0, 32000, size=50).tolist()
    a, hit = side.admit(prompt_a)
    assert hit == 0
    # B shares A's first 40 tokens: two full blocks are hits (block 2 differs
    # at token 40).
    prompt_b = prompt_a[:40] + rng.integers(0, 32000, size=10).tolist()
    b, hit = side.admit(prompt_b)
    assert hit == 32
    # C repeats A's prompt: (50 - 1) // 16 = 3 blocks are hits.
    c, hit = side.admit(list(prompt_a))
    assert hit == 48
    # Decode steps: A fills its fourth block (tokens 50..63 and one more),
    # which registers it; B and C generate their own tokens.
    for step in range(15):
        side.generate(a, 1000 + step)
        side.generate(b, 2000 + step)
        side.generate(c, 3000 + step)
    full_a = list(side.tokens[a])
    assert len(full_a) == 65
    # A finishes: its blocks return to the free queue and stay cached.
    blocks_a = side.ref.table(a)[0]
    side.free(a)
    assert side.pool.is_cached(blocks_a[3]) and blocks_a[3] in side.pool.free_queue()
    # D continues A's whole text: it re-hits A's freed, still cached fourth
    # block (taken back out of the free queue) on top of the three shared ones.
    d, hit = side.admit(full_a[:64] + [4242, 4343])
    assert hit == 64
    assert side.ref.table(d)[0][:4] == blocks_a[:4]
    assert blocks_a[3] not in side.pool.free_queue()
    # A new request takes blocks from the free queue: the cached blocks of D
    # are not among them, so D's rows survive.
    e, hit = side.admit(rng.integers(0, 32000, size=40).tolist())
    assert hit == 0
    side.generate(d, 4444)
    side.check_cache()
    seqs = [b, c, d, e]
    q = workloads.random_values(np.random.default_rng(63), (len(seqs), HQ, D), "bf16")
    got, want, bt, sl = side.decode(seqs, q, partition)
    assert_close(got, want, "bf16", "decode over prefix-cache hits vs oracle")
    # Shared blocks hold exactly the rows each sequence's own tokens give.
    plain = contiguous_reference([side.tokens[s] for s in seqs], q)
    assert np.allclose(want, plain, rtol=0, atol=1e-12)
    # The sharing is real: B, C and D hold A's first two blocks.
    assert bt[0, 0] == bt[1, 0] == bt[2, 0] == blocks_a[0]


def test_swap_round_trip_against_the_oracle_then_decode():
    # Group {x, x2} (a fork) and requests y, z share a 12-block pool.  The
    # group leaves for page-locked host blocks, z finishes, y generates into
    # freed blocks (the group's among them), the group comes back to other
    # GPU blocks and the batch is decoded.
    ncpu, nb = 8, 12
    side = Side(num_blocks=nb, seed=71)
    rng = np.random.default_rng(72)
    side.pool.set_cpu_blocks(ncpu)
    side.ref.set_cpu_blocks(ncpu)
    x, _ = side.admit(rng.integers(0, 32000, size=3 * BS + 5).tolist())
    x2 = side.pool.fork(x)
    assert side.ref.fork(x) == x2
    side.tokens[x2] = list(side.tokens[x])
    for t in range(3):
        side.generate(x, 10 + t)     # the first write into the shared last block copies it
        side.generate(x2, 20 + t)
    y, _ = side.admit(rng.integers(0, 32000, size=2 * BS).tolist())
    z, _ = side.admit(rng.integers(0, 32000, size=2 * BS + 8).tolist())
    side.check_cache()
    group_blocks = set(side.ref.table(x)[0]) | set(side.ref.table(x2)[0])
    assert len(group_blocks) == 5 and side.pool.num_free() == 2
    # The host pool, one canary-filled page-locked buffer; the oracle sees the
    # GPU and CPU pools as one block index space (CPU block c = nb + c).
    canary = workloads.garbage_values(rng, (2, ncpu, BS, HKV, D), "bf16")
    cpu = torch.from_numpy(canary.view(np.int16)).view(torch.bfloat16).pin_memory()
    both = np.concatenate([side.cache_ref, canary], axis=1)
    out = side.pool.swap_out([x, x2])
    assert out.tolist() == [list(p) for p in side.ref.swap_out([x, x2])]
    pa.pa_swap_blocks(cpu, side.cache_dev, out.cuda())
    oracle.copy_blocks(both, out.numpy() + np.array([0, nb]))
    torch.cuda.synchronize()
    assert np.array_equal(cpu.view(torch.int16).numpy().view(np.uint16), both[:, nb:])
    assert pa.pa_get_device_error() == 0
    # z finishes and y generates four blocks' worth while the group is out:
    # two blocks were free before, so y also takes two the group left.
    side.free(z)
    for t in range(4 * BS):
        side.generate(y, 30 + t)
    assert len(set(side.ref.table(y)[0]) & group_blocks) == 2
    both[:, :nb] = side.cache_ref
    back = side.pool.swap_in([x, x2])
    assert back.tolist() == [list(p) for p in side.ref.swap_in([x, x2])]
    pa.pa_swap_blocks(side.cache_dev, cpu, back.cuda())
    oracle.copy_blocks(both, back.numpy() + np.array([nb, 0]))
    side.cache_ref[...] = both[:, :nb]
    side.check_cache()
    side.generate(x, 99)
    side.check_cache()
    seqs = [x, x2, y]
    q = workloads.random_values(np.random.default_rng(73), (len(seqs), HQ, D), "bf16")
    got, want, _, _ = side.decode(seqs, q)
    assert_close(got, want, "bf16", "decode after swap-in vs oracle")
    plain = contiguous_reference([side.tokens[s] for s in seqs], q)
    assert np.allclose(want, plain, rtol=0, atol=1e-12)
