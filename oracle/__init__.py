"""CPU oracle for the paged KV-cache hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The library in
``paged_kv_cache_78_gb300`` never imports it and shares no code with it.

Contents
  * ``pa_oracle.c`` (built into ``_pa_oracle.so`` with gcc): scatter through
    slot_mapping, copy-on-write block copy, paged decode attention in binary64
    (two-pass softmax), split-KV partials and their log-sum-exp combination.
  * ``pool_replay.py``: the block bookkeeping of the pages (allocation,
    fork with reference counts, copy-on-write, free), written independently of
    the C++ pool.
  * ``sizing.py``: the KV-cache sizing closed forms the pages print.

Arrays use numpy.  bf16 tensors are carried as ``uint16`` bit patterns,
fp32 tensors as ``float32``.  The cache of one layer is an array of shape
``[2, num_blocks, block_size, num_kv_heads, head_size]`` (0 = K, 1 = V).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_pa_oracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP32 = 1


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (OpenMP when available).  Returns the .so path."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC,
            "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    p, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_num_threads.restype = i32
    lib.oracle_set_num_threads.argtypes = [i32]
    lib.oracle_set_num_threads.restype = None
    lib.oracle_reshape_and_cache.argtypes = [p, i64, i32, i32, i32, i32, p, p, p, i64]
    lib.oracle_reshape_and_cache.restype = i32
    lib.oracle_copy_blocks.argtypes = [p, i64, i32, i32, i32, i32, p, i64]
    lib.oracle_copy_blocks.restype = i32
    lib.oracle_decode.argtypes = [p, p, p, i64, i32, i32, i32, i32, p, i32, p, i32, i32, dbl]
    lib.oracle_decode.restype = i32
    lib.oracle_decode_partials.argtypes = [p, p, p, p, p, i64, i32, i32, i32, i32, p, i32,
                                           p, i32, i32, dbl, i32, i32]
    lib.oracle_decode_partials.restype = i32
    lib.oracle_combine_partials.argtypes = [p, p, p, p, i32, i32, i32, i32]
    lib.oracle_combine_partials.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
        return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.float32:
        return FP32
    raise TypeError("oracle arrays are bf16 bit patterns (uint16) or float32, got %s" % arr.dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of later oracle calls from this thread (timing only)."""
    _load().oracle_set_num_threads(int(n))


def reshape_and_cache(cache: np.ndarray, key: np.ndarray, value: np.ndarray,
                      slot_mapping: np.ndarray) -> None:
    """In place: cache[0, slot // BS, slot % BS] = key[t]; the same for value at 1."""
    two, nb, bs, hkv, d = cache.shape
    assert two == 2 and key.shape == value.shape and key.shape[1:] == (hkv, d)
    assert key.dtype == cache.dtype == value.dtype
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = _load().oracle_reshape_and_cache(_ptr(cache), nb, bs, hkv, d, dtype_code(cache),
                                          _ptr(np.ascontiguousarray(key)),
                                          _ptr(np.ascontiguousarray(value)), _ptr(slots),
                                          slots.shape[0])
    if rc != 0:
        raise IndexError("slot outside the pool")


def copy_blocks(cache: np.ndarray, pairs: np.ndarray) -> None:
    """In place, in list order: cache[:, dst] = cache[:, src] for each (src, dst)."""
    two, nb, bs, hkv, d = cache.shape
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    rc = _load().oracle_copy_blocks(_ptr(cache), nb, bs, hkv, d, dtype_code(cache), _ptr(pr),
                                    pr.shape[0])
    if rc != 0:
        raise IndexError("block index outside the pool")


def decode(query: np.ndarray, cache: np.ndarray, block_tables: np.ndarray,
           seq_lens: np.ndarray, scale: float) -> np.ndarray:
    """Paged decode attention in binary64; returns [num_seqs, num_heads, head_size] float64."""
    two, nb, bs, hkv, d = cache.shape
    s, hq, dq = query.shape
    assert dq == d and query.dtype == cache.dtype
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert bt.shape[0] == s and sl.shape == (s,)
    out = np.zeros((s, hq, d), dtype=np.float64)
    rc = _load().oracle_decode(_ptr(out), _ptr(np.ascontiguousarray(query)), _ptr(cache), nb,
                               bs, hkv, d, dtype_code(cache), _ptr(bt), bt.shape[1], _ptr(sl),
                               s, hq, float(scale))
    if rc != 0:
        raise IndexError("block table or seq_len outside the pool")
    return out


def decode_partials(query: np.ndarray, cache: np.ndarray, block_tables: np.ndarray,
                    seq_lens: np.ndarray, scale: float, partition_size: int,
                    max_parts: int):
    """Split-KV partials (m, l, acc) in binary64, one entry per partition."""
    two, nb, bs, hkv, d = cache.shape
    s, hq, _ = query.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    m = np.empty((s, hq, max_parts), dtype=np.float64)
    l = np.empty((s, hq, max_parts), dtype=np.float64)
    acc = np.empty((s, hq, max_parts, d), dtype=np.float64)
    rc = _load().oracle_decode_partials(_ptr(m), _ptr(l), _ptr(acc),
                                        _ptr(np.ascontiguousarray(query)), _ptr(cache), nb, bs,
                                        hkv, d, dtype_code(cache), _ptr(bt), bt.shape[1],
                                        _ptr(sl), s, hq, float(scale), int(partition_size),
                                        int(max_parts))
    if rc != 0:
        raise IndexError("bad index, seq_len or partition count")
    return m, l, acc


def combine_partials(m: np.ndarray, l: np.ndarray, acc: np.ndarray) -> np.ndarray:
    """Log-sum-exp combination of split-KV partials (binary64)."""
    s, hq, p, d = acc.shape
    out = np.empty((s, hq, d), dtype=np.float64)
    _load().oracle_combine_partials(_ptr(out), _ptr(np.ascontiguousarray(m)),
                                    _ptr(np.ascontiguousarray(l)),
                                    _ptr(np.ascontiguousarray(acc)), s, hq, d, p)
    return out


def to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) or float32 to float64."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if a.dtype == np.float32:
        return a.astype(np.float64)
    raise TypeError(a.dtype)


def slot_mapping(block_tables: np.ndarray, seq_idx: np.ndarray, positions: np.ndarray,
                 block_size: int) -> np.ndarray:
    """Physical slot of token ``positions[i]`` of sequence ``seq_idx[i]``:
    table[pos // block_size] * block_size + pos % block_size
    (tech.blogsailing.com/?p=100 section 2: a token index splits into a
    logical block and an offset; the block table maps the logical block to a
    physical one)."""
    bt = np.asarray(block_tables)
    s = np.asarray(seq_idx, dtype=np.int64)
    p = np.asarray(positions, dtype=np.int64)
    return bt[s, p // block_size].astype(np.int64) * block_size + p % block_size


def fill_cache(case, cache: np.ndarray | None = None, exclude_last: bool = False) -> np.ndarray:
    """The pool of a workload with every token written through the oracle's
    own scatter (tokens at position seq_len - 1 left out when ``exclude_last``)."""
    if cache is None:
        cache = case.initial_cache()
    seqs, pos, rows = case.token_positions(exclude_last=exclude_last)
    if rows.size:
        slots = slot_mapping(case.block_tables, seqs, pos, case.block_size)
        reshape_and_cache(cache, case.keys[rows], case.values[rows], slots)
    return cache
