"""Seeded synthetic workloads for the paged decode hot path.

This module only draws inputs: token data, queries, sequence lengths and
random, non-contiguous block tables.  It holds none of the method's
arithmetic (no scatter, no slot formula, no attention); both the CUDA path and
the CPU oracle receive the same arrays and derive everything else with their
own code.  Shapes follow the workloads the pages size their caches for:

* ``tiny``: 4 sequences of {7, 16, 33, 100} tokens, 4 heads of 64, block size
  4, a pool of 64 blocks; sequence 0 maps logical blocks 0 -> 7 and 1 -> 1 as in
  the worked decode example of studying-code.tistory.com/16 (section
  "① 초기 단계").
* ``qwen2_gqa``: the Qwen2-0.5B attention shape of the itan.pw page (2 KV heads
  of 64, block size 16; 14 query heads), batch 64, lengths U[128, 2048], pool
  of 16384 blocks.
* ``opt13b_mha``: OPT-13B attention (40 heads of 128, studying-code.tistory.com/16
  sizes its cache at about 800 KB per token), batch 32, lengths U[1, 2048],
  block size 8, 16 or 32 on the same token data.
* ``shared_prefix``: 32 query / 8 KV heads of 128, block size 16; forked
  samples sharing prompt blocks, and requests sharing a common prefix.
* ``long_context``: the same head shape, batch 8 at 32768 tokens, and a mixed
  batch {512, 4096, 32768, 131072}.

Values are N(0, 1) rounded to bf16 (round to nearest even) or kept in fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def random_values(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0, 1) values: bf16 bit patterns (uint16) or float32."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def garbage_values(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """Arbitrary bit patterns (NaN and Inf included) standing in for stale cache memory."""
    if dtype == "bf16":
        return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
    return rng.integers(0, 1 << 32, size=shape, dtype=np.uint32).view(np.float32)


def np_dtype(dtype: str):
    return np.uint16 if dtype == "bf16" else np.float32


def elem_bytes(dtype: str) -> int:
    return 2 if dtype == "bf16" else 4


@dataclass
class DecodeCase:
    """One decode batch over a paged pool.

    ``seq_lens`` count every token the decode attends to; the last token of
    each sequence (position seq_len - 1) is the one the decode step writes.
    ``keys``/``values`` hold the token data of all sequences back to back
    (sequence s occupies rows seq_starts[s] .. seq_starts[s+1]).
    """

    name: str
    seed: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    dtype: str
    scale: float
    seq_lens: np.ndarray
    block_tables: np.ndarray
    query: np.ndarray
    keys: np.ndarray
    values: np.ndarray
    seq_starts: np.ndarray
    cache_fill: str = "zeros"
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.seq_lens.size else 0

    def cache_shape(self):
        return (2, self.num_blocks, self.block_size, self.num_kv_heads, self.head_size)

    def initial_cache(self) -> np.ndarray:
        """The pool before any token is written: zeros, or stale garbage."""
        shape = self.cache_shape()
        if self.cache_fill == "garbage":
            return garbage_values(np.random.default_rng([self.seed, 7]), shape, self.dtype)
        return np.zeros(shape, dtype=np_dtype(self.dtype))

    def token_positions(self, last_only: bool = False, exclude_last: bool = False):
        """(seq index, position) of tokens, sequence-major, as int32 arrays, and
        the matching row indices into keys/values."""
        seqs, poss, rows = [], [], []
        for s in range(self.num_seqs):
            n = int(self.seq_lens[s])
            if n == 0:
                continue
            if last_only:
                p = np.array([n - 1])
            elif exclude_last:
                p = np.arange(n - 1)
            else:
                p = np.arange(n)
            seqs.append(np.full(p.shape, s, dtype=np.int32))
            poss.append(p.astype(np.int32))
            rows.append(self.seq_starts[s] + p)
        if not seqs:
            e = np.zeros(0, dtype=np.int32)
            return e, e, np.zeros(0, dtype=np.int64)
        return (np.concatenate(seqs), np.concatenate(poss),
                np.concatenate(rows).astype(np.int64))

    def kv_bytes(self) -> int:
        """Bytes of K and V the decode must read once: sum_s L_s * Hkv * D * 2 * elem."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_size * 2 * elem_bytes(self.dtype)


def _tables_from_permutation(perm: np.ndarray, seq_lens: np.ndarray, block_size: int,
                             max_blocks: int | None = None):
    counts = [-(-int(n) // block_size) for n in seq_lens]
    mb = max(max(counts) if counts else 0, 1) if max_blocks is None else max_blocks
    tables = np.zeros((len(seq_lens), mb), dtype=np.int32)
    off = 0
    for s, c in enumerate(counts):
        tables[s, :c] = perm[off:off + c]
        off += c
    if off > perm.shape[0]:
        raise ValueError("pool too small for the sequences")
    return tables


def contiguous(case: "DecodeCase") -> "DecodeCase":
    """The same tokens with each sequence's logical blocks on consecutive
    physical blocks (sequence after sequence from block 0): the unpaged
    layout, for measuring what scattering the blocks costs."""
    tables = _tables_from_permutation(np.arange(case.num_blocks, dtype=np.int32), case.seq_lens,
                                      case.block_size, max_blocks=case.block_tables.shape[1])
    return DecodeCase(**{**case.__dict__, "name": case.name + "_contiguous",
                         "block_tables": tables})


def _token_data(rng, seq_lens, hkv, d, dtype):
    starts = np.zeros(len(seq_lens) + 1, dtype=np.int64)
    starts[1:] = np.cumsum(seq_lens.astype(np.int64))
    total = int(starts[-1])
    keys = random_values(rng, (total, hkv, d), dtype)
    values = random_values(rng, (total, hkv, d), dtype)
    return keys, values, starts


def tiny(dtype: str = "bf16", seed: int = 0) -> DecodeCase:
    rng = np.random.default_rng(seed)
    seq_lens = np.array([7, 16, 33, 100], dtype=np.int32)
    nb, bs, h, d = 64, 4, 4, 64
    perm = rng.permutation(nb)
    rest = [b for b in perm if b not in (7, 1)]
    perm = np.array([7, 1] + rest, dtype=np.int64)
    tables = _tables_from_permutation(perm, seq_lens, bs)
    keys, values, starts = _token_data(rng, seq_lens, h, d, dtype)
    q = random_values(rng, (4, h, d), dtype)
    return DecodeCase("tiny", seed, h, h, d, bs, nb, dtype, 1.0 / math.sqrt(d), seq_lens,
                      tables, q, keys, values, starts, cache_fill="garbage")


def qwen2_gqa(dtype: str = "bf16", seed: int = 1, num_seqs: int = 64) -> DecodeCase:
    rng = np.random.default_rng(seed)
    nb, bs, hq, hkv, d = 16384, 16, 14, 2, 64
    seq_lens = rng.integers(128, 2048, size=num_seqs, endpoint=True).astype(np.int32)
    tables = _tables_from_permutation(rng.permutation(nb), seq_lens, bs)
    keys, values, starts = _token_data(rng, seq_lens, hkv, d, dtype)
    q = random_values(rng, (num_seqs, hq, d), dtype)
    return DecodeCase("qwen2_gqa", seed, hq, hkv, d, bs, nb, dtype, 1.0 / math.sqrt(d),
                      seq_lens, tables, q, keys, values, starts)


def opt13b_mha(block_size: int = 16, dtype: str = "bf16", seed: int = 2,
               num_seqs: int = 32) -> DecodeCase:
    rng = np.random.default_rng(seed)
    h, d = 40, 128
    seq_lens = rng.integers(1, 2048, size=num_seqs, endpoint=True).astype(np.int32)
    keys, values, starts = _token_data(rng, seq_lens, h, d, dtype)
    q = random_values(rng, (num_seqs, h, d), dtype)
    nb = num_seqs * 2048 // block_size
    trng = np.random.default_rng([seed, block_size])
    tables = _tables_from_permutation(trng.permutation(nb), seq_lens, block_size)
    return DecodeCase("opt13b_mha_bs%d" % block_size, seed, h, h, d, block_size, nb, dtype,
                      1.0 / math.sqrt(d), seq_lens, tables, q, keys, values, starts)


def long_context(mixed: bool = False, dtype: str = "bf16", seed: int = 4) -> DecodeCase:
    rng = np.random.default_rng([seed, int(mixed)])
    hq, hkv, d, bs = 32, 8, 128, 16
    if mixed:
        seq_lens = np.array([512, 4096, 32768, 131072], dtype=np.int32)
    else:
        seq_lens = np.full(8, 32768, dtype=np.int32)
    need = sum(-(-int(n) // bs) for n in seq_lens)
    nb = max(need, 16384) if not mixed else need
    tables = _tables_from_permutation(rng.permutation(nb), seq_lens, bs)
    keys, values, starts = _token_data(rng, seq_lens, hkv, d, dtype)
    q = random_values(rng, (len(seq_lens), hq, d), dtype)
    return DecodeCase("long_context_mixed" if mixed else "long_context", seed, hq, hkv, d, bs,
                      nb, dtype, 1.0 / math.sqrt(d), seq_lens, tables, q, keys, values, starts)


def custom(num_seqs: int, num_heads: int, num_kv_heads: int, head_size: int,
           block_size: int, seq_lens, dtype: str = "bf16", seed: int = 0,
           spare_blocks: int = 3, cache_fill: str = "garbage",
           max_blocks: int | None = None) -> DecodeCase:
    """A small case with explicit lengths (edge cases, ragged tails)."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (num_seqs,)
    need = sum(-(-int(n) // block_size) for n in seq_lens)
    nb = need + spare_blocks
    tables = _tables_from_permutation(rng.permutation(nb), seq_lens, block_size, max_blocks)
    keys, values, starts = _token_data(rng, seq_lens, num_kv_heads, head_size, dtype)
    q = random_values(rng, (num_seqs, num_heads, head_size), dtype)
    return DecodeCase("custom", seed, num_heads, num_kv_heads, head_size, block_size, nb,
                      dtype, 1.0 / math.sqrt(head_size), seq_lens, tables, q, keys, values,
                      starts, cache_fill=cache_fill)


# ---------------------------------------------------------------------------
# Shared-prefix / parallel sampling: an operation script for the block pools.
# ---------------------------------------------------------------------------

@dataclass
class PoolScript:
    """Operations on a block pool; each side replays them with its own pool.

    ops: ("add", n_tokens) -> new sequence id (ids count up from 0 in creation order)
         ("fork", parent_id) -> new sequence id
         ("append", seq_id)  -> one token written at the sequence's end
    ``decode_seqs`` lists the sequences the decode step attends for.
    """

    num_blocks: int
    block_size: int
    free_order: np.ndarray
    ops: list
    decode_seqs: list


def shared_prefix_script(seed: int = 3, variant: str = "fork", prompt_len: int = 1018,
                         num_requests: int | None = None, samples: int = 8,
                         prefix_len: int = 512) -> PoolScript:
    """``fork``: requests with a prompt forked into ``samples`` samples, each
    then generating 1..64 private tokens.  A prompt length that is not a
    multiple of the block size leaves a shared, partly filled last block that
    the first write of all but one sample copies.
    ``prefix``: requests share a ``prefix_len``-token prefix (forked from one
    parent) and then append distinct 64..512-token suffixes."""
    rng = np.random.default_rng([seed, 0 if variant == "fork" else 1])
    bs = 16
    ops: list = []
    decode_seqs: list = []
    if variant == "fork":
        nreq = 16 if num_requests is None else num_requests
        priv = rng.integers(1, 64, size=(nreq, samples), endpoint=True)
        need = 0
        next_id = 0
        for r in range(nreq):
            ops.append(("add", prompt_len))
            parent = next_id
            next_id += 1
            ids = [parent]
            for _ in range(samples - 1):
                ops.append(("fork", parent))
                ids.append(next_id)
                next_id += 1
            # generation steps: every sample writes one token per step until done
            for step in range(int(priv[r].max())):
                for k, sid in enumerate(ids):
                    if step < priv[r, k]:
                        ops.append(("append", sid))
            decode_seqs += ids
            need += -(-prompt_len // bs) + samples * (-(-(prompt_len % bs + 64) // bs) + 1)
    else:
        nreq = 128 if num_requests is None else num_requests
        suffix = rng.integers(64, 512, size=nreq, endpoint=True)
        ops.append(("add", prefix_len))
        root = 0
        next_id = 1
        need = -(-prefix_len // bs)
        for r in range(nreq):
            ops.append(("fork", root))
            sid = next_id
            next_id += 1
            for _ in range(int(suffix[r])):
                ops.append(("append", sid))
            decode_seqs.append(sid)
            need += -(-int(suffix[r]) // bs) + 1
    nb = int(need * 1.1) + 16
    free_order = np.random.default_rng([seed, 2]).permutation(nb).astype(np.int32)
    return PoolScript(nb, bs, free_order, ops, decode_seqs)
