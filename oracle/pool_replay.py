"""Block bookkeeping of the paged KV cache, replayed in plain Python.

TEST INFRASTRUCTURE ONLY (part of the oracle).  It is written independently
of the library's C++ block pool and is compared with it step by step.

Rules, in the pages' terms:

* A request's KV cache is a list of logical blocks filled left to right; a
  block table maps each logical block to a physical block.  A new physical
  block is taken only when the last one is full, so all waste sits in the last
  block (studying-code.tistory.com/16, sections "vLLM의 메모리 관리" and
  "물리적 블록 할당"; tech.blogsailing.com/?p=100 section 2, ``append_token``:
  logical block = token_idx // BLOCK_SIZE, offset = token_idx % BLOCK_SIZE,
  a new block is popped from the front of the free pool only when the logical
  block does not exist yet).
* A prompt of n tokens takes ceil(n / block_size) blocks
  (itan.pw "vLLMにおけるKVCacheマネージャーの詳細解説", section
  "ブロック割当のロジック": cdiv(num_tokens, block_size)).
* Forking a sequence shares all its physical blocks and raises each block's
  reference count (studying-code.tistory.com/16, the two-sample example before
  "생성 단계에서의 Copy-on-Write"; tech.blogsailing.com/?p=100 section 3,
  ``fork_sequence``).
* Copy-on-write: a sequence about to write into a block whose reference count
  is above 1 takes a new block, the old block's content is copied to it, and
  the old block's count drops by one; a holder that finds the count at 1
  writes in place (studying-code.tistory.com/16, section "생성 단계에서의
  Copy-on-Write"; tech.blogsailing.com/?p=100 section 3, ``resolve_cow``).
  The copy is reported as a (src, dst) pair for the block-copy kernel.
* Freeing a sequence lowers the count of each of its blocks; blocks that
  reach 0 go back to the free pool (studying-code.tistory.com/16, sections
  "요청 완료 후 메모리 관리" and "물리적 블록 해제와 참조 카운트").  They are
  returned last block first, as in the prefix-cache timeline of the itan.pw
  page (time 4: a finished request's blocks enter the free queue in reverse
  order), and appended at the tail of the FIFO free list (the front is where
  ``pop(0)`` takes new blocks in tech.blogsailing.com/?p=100).
* Running out of free blocks is reported and leaves the state unchanged.

Prefix caching (itan.pw page, sections "KVCacheManagerの処理詳細" and
"プレイフィックスキャッシュの詳細"), written here with the exact token prefix as
the key instead of a chained hash:

* a full block of a sequence whose token ids are known is registered under
  the tuple of all tokens up to its end (that is what the chained hash
  identifies); a partly filled block is not;
* a new request shares the longest run of leading registered blocks, at most
  (num_tokens - 1) // block_size (the page's ``max_length = num_tokens - 1``
  and ``max_num_blocks = max_length // block_size``), stopping at the first
  miss; shared blocks leave the free queue before any block is taken for the
  rest of the request (time 6 of the page's timeline);
* freed blocks stay registered until the free queue hands them out again
  (time 4: blocks 2 and 3 are free and still cached).

Swapping (studying-code.tistory.com/16, sections "All-or-Nothing Eviction"
and "스와핑(Swapping)"):

* a preempted sequence group leaves the GPU whole: every block of its
  sequences is copied to a block of a CPU allocator whose size never exceeds
  the GPU's block count, then the GPU blocks are released; a block shared
  with a sequence outside the group cannot leave (the group would be split);
* swapping in takes GPU blocks for the group's CPU blocks and releases those;
* the order of the copies (first use, sequences in the given order, blocks
  in table order) and of the releases (each sequence's last block first, to
  the tail of the free list) follows the rest of this replay.
"""
from __future__ import annotations

from collections import deque


class OutOfBlocks(Exception):
    pass


class BadState(Exception):
    pass


class PoolReplay:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad pool geometry")
        self.block_size = block_size
        self.num_blocks = num_blocks
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the block ids")
        self.free = deque(order)
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self.next_id = 0
        self.toks: dict[int, list[int] | None] = {}  # token ids of tracked sequences
        self.cpu_free: deque = deque()
        self.cpu_ref: list[int] = []
        self.swapped: set[int] = set()
        self.cache: dict[tuple, int] = {}            # token prefix -> registered block
        self.block_key: dict[int, tuple] = {}        # registered block -> its prefix

    def _take(self) -> int:
        b = self.free.popleft()
        key = self.block_key.pop(b, None)
        if key is not None:
            del self.cache[key]
        self.ref[b] = 1
        return b

    def _register(self, b: int, key: tuple) -> None:
        if key not in self.cache and b not in self.block_key:
            self.cache[key] = b
            self.block_key[b] = key

    # -- operations -------------------------------------------------------
    def add_seq(self, num_tokens: int) -> int:
        need = -(-num_tokens // self.block_size)
        if need > len(self.free):
            raise OutOfBlocks()
        blocks = [self._take() for _ in range(need)]
        sid = self.next_id
        self.next_id += 1
        self.tables[sid] = blocks
        self.lens[sid] = num_tokens
        self.toks[sid] = None
        return sid

    def add_seq_tokens(self, tokens):
        """Returns (sid, number of leading tokens whose blocks were shared)."""
        tokens = [int(t) for t in tokens]
        n, bs = len(tokens), self.block_size
        need = -(-n // bs)
        hits = []
        for i in range((n - 1) // bs if n > 0 else 0):
            b = self.cache.get(tuple(tokens[:(i + 1) * bs]))
            if b is None:
                break
            hits.append(b)
        in_free = sum(1 for b in hits if b in self.free)
        if need - len(hits) > len(self.free) - in_free:
            raise OutOfBlocks()
        for b in hits:
            if b in self.free:
                self.free.remove(b)
            self.ref[b] += 1
        blocks = hits + [self._take() for _ in range(need - len(hits))]
        for i in range(len(hits), n // bs):
            self._register(blocks[i], tuple(tokens[:(i + 1) * bs]))
        sid = self.next_id
        self.next_id += 1
        self.tables[sid] = blocks
        self.lens[sid] = n
        self.toks[sid] = tokens
        return sid, len(hits) * bs

    def fork(self, parent: int) -> int:
        if parent in self.swapped:
            raise BadState()
        blocks = list(self.tables[parent])
        for b in blocks:
            self.ref[b] += 1
        sid = self.next_id
        self.next_id += 1
        self.tables[sid] = blocks
        self.lens[sid] = self.lens[parent]
        toks = self.toks[parent]
        self.toks[sid] = None if toks is None else list(toks)
        return sid

    def append_token(self, sid: int, token=None):
        """Returns (slot, pair) where pair is (src, dst) of a copy-on-write or
        None.  With a token id a tracked sequence records it and registers the
        block it fills; without one the sequence stops being tracked."""
        if sid in self.swapped:
            raise BadState()
        table = self.tables[sid]
        pos = self.lens[sid]
        logical, offset = divmod(pos, self.block_size)
        pair = None
        if logical == len(table):
            if not self.free:
                raise OutOfBlocks()
            b = self._take()
            table.append(b)
        else:
            b = table[logical]
            if self.ref[b] > 1:
                if not self.free:
                    raise OutOfBlocks()
                nb = self._take()
                self.ref[b] -= 1
                table[logical] = nb
                pair = (b, nb)
                b = nb
        self.lens[sid] = pos + 1
        toks = self.toks[sid]
        if toks is not None:
            if token is None:
                self.toks[sid] = None
            else:
                toks.append(int(token))
                if offset == self.block_size - 1:
                    self._register(b, tuple(toks[:(logical + 1) * self.block_size]))
        return b * self.block_size + offset, pair

    def free_seq(self, sid: int) -> None:
        swapped = sid in self.swapped
        ref, free = (self.cpu_ref, self.cpu_free) if swapped else (self.ref, self.free)
        for b in reversed(self.tables.pop(sid)):
            ref[b] -= 1
            if ref[b] == 0:
                free.append(b)
        del self.lens[sid]
        del self.toks[sid]
        self.swapped.discard(sid)

    # -- swapping ------------------------------------------------------------
    def set_cpu_blocks(self, n: int) -> None:
        if n < 0 or n > self.num_blocks:
            raise ValueError("the CPU region may not exceed the GPU block count")
        if self.swapped:
            raise BadState()
        self.cpu_free = deque(range(n))
        self.cpu_ref = [0] * n

    def _move(self, sids, out: bool):
        if len(set(sids)) != len(sids):
            raise ValueError("sequence listed twice")
        for sid in sids:
            if sid not in self.tables or (sid in self.swapped) == out:
                raise BadState()
        src_ref = self.ref if out else self.cpu_ref
        dst_free = self.cpu_free if out else self.free
        uses: dict[int, int] = {}
        for sid in sids:
            for b in self.tables[sid]:
                uses[b] = uses.get(b, 0) + 1
        if any(uses[b] != src_ref[b] for b in uses):
            raise BadState()
        if len(uses) > len(dst_free):
            raise OutOfBlocks()
        where, pairs = {}, []
        for b in uses:  # dicts keep first-use order
            if out:
                d = self.cpu_free.popleft()
                self.cpu_ref[d] = self.ref[b]
            else:
                r = self.cpu_ref[b]
                d = self._take()
                self.ref[d] = r
            where[b] = d
            pairs.append((b, d))
        for sid in sids:
            for b in reversed(self.tables[sid]):
                src_ref[b] -= 1
                if src_ref[b] == 0:
                    (self.free if out else self.cpu_free).append(b)
            self.tables[sid] = [where[b] for b in self.tables[sid]]
            if out:
                self.swapped.add(sid)
            else:
                self.swapped.discard(sid)
        return pairs

    def swap_out(self, sids):
        return self._move(list(sids), True)

    def swap_in(self, sids):
        return self._move(list(sids), False)

    def reset_prefix_cache(self) -> None:
        self.cache.clear()
        self.block_key.clear()

    # -- views -------------------------------------------------------------
    def table(self, sid: int):
        return list(self.tables[sid]), self.lens[sid]

    def filled(self, sid: int):
        """#filled of every block-table entry (the pages' per-entry fill count)."""
        n, bs = self.lens[sid], self.block_size
        return [min(bs, n - i * bs) for i in range(len(self.tables[sid]))]

    def slot(self, sid: int, pos: int) -> int:
        return self.tables[sid][pos // self.block_size] * self.block_size + pos % self.block_size

    def num_free(self) -> int:
        return len(self.free)

    def is_cached(self, b: int) -> bool:
        return b in self.block_key

    def free_queue(self):
        return list(self.free)

    def check_invariants(self) -> None:
        used = [b for b in range(self.num_blocks) if self.ref[b] > 0]
        cpu_used = [b for b in range(len(self.cpu_ref)) if self.cpu_ref[b] > 0]
        assert len(cpu_used) + len(self.cpu_free) == len(self.cpu_ref), "CPU block lost"
        assert set(cpu_used).isdisjoint(self.cpu_free), "CPU block both used and free"
        assert sum(self.cpu_ref) == sum(len(self.tables[s]) for s in self.swapped)
        assert set(used).isdisjoint(self.free), "block both used and free"
        assert len(used) + len(self.free) == self.num_blocks, "block lost"
        assert len(set(self.free)) == len(self.free), "block twice in the free list"
        total_refs = sum(self.ref)
        total_entries = sum(len(t) for s, t in self.tables.items() if s not in self.swapped)
        assert total_refs == total_entries, "ref counts disagree with the tables"
        for key, b in self.cache.items():
            assert self.block_key[b] == key and len(key) % self.block_size == 0
