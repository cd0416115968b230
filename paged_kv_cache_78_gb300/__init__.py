"""Python binding of libpa.so, the GB300 paged KV-cache library.

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels (or, for the block pool, its C++ host code).  Names follow the
C ABI in include/pa.h.  Tensors are torch tensors; PyTorch provides device
memory and streams.  If libpa.so is missing this module raises on import:
there is no fallback path.

Cache layout (one layer): a contiguous tensor [2, num_blocks, block_size,
num_kv_heads, head_size] of bf16 or fp32, index 0 = keys, 1 = values.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_CUDA = 3
PA_ERR_OUT_OF_BLOCKS = 4
PA_ERR_BAD_STATE = 5
PA_ERR_DEVICE_CHECK = 6
PA_ERR_TIMEOUT = 7
PA_BF16 = 0
PA_FP32 = 1
PA_KERNEL_AUTO = 0
PA_KERNEL_SIMT = 1
PA_KERNEL_TENSOR = 2
PA_DEVERR_SLOT = 0x1
PA_DEVERR_BLOCK_ID = 0x2
PA_DEVERR_SEQ_LEN = 0x4
PA_DEVERR_TIMEOUT = 0x8
PA_PARTITION_BALANCED = -2

# Every function include/pa.h declares.
EXPORTS = (
    "pa_reshape_and_cache", "pa_copy_blocks", "pa_decode", "pa_decode_ex", "pa_decode_no_alloc",
    "pa_decode_partition_size", "pa_decode_select_kernel",
    "pa_decode_workspace_size", "pa_slot_mapping", "pa_pool_create", "pa_pool_destroy",
    "pa_pool_add_seq", "pa_pool_fork", "pa_pool_append_token", "pa_pool_append_tokens",
    "pa_pool_free_seq", "pa_pool_block_table", "pa_pool_fill_tables", "pa_pool_slot",
    "pa_pool_ref_count", "pa_pool_num_free", "pa_get_device_error", "pa_status_string",
    "pa_version", "pa_set_decode_trace", "pa_pool_add_seq_tokens", "pa_pool_append_token_id",
    "pa_pool_is_cached", "pa_pool_free_queue", "pa_pool_reset_prefix_cache", "pa_pool_usage",
    "pa_swap_blocks", "pa_pool_set_cpu_blocks", "pa_pool_swap_out", "pa_pool_swap_in",
    "pa_pool_is_swapped", "pa_pool_num_free_cpu", "pa_decode_append", "pa_copy_bytes",
    "pa_set_decode_wait_limit", "pa_decode_shared_plan", "pa_decode_shared_workspace_size",
    "pa_decode_shared",
)


class PAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (where, _status_string(status), status))


class OutOfBlocks(PAError):
    pass


class SharedPlanInfo(ctypes.Structure):
    _fields_ = [("num_chunks", ctypes.c_int32), ("num_members", ctypes.c_int32),
                ("min_shared_tokens", ctypes.c_int32), ("min_chunk_stages", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("plan_ints", ctypes.c_int32)]


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_size", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("libpa.so is not built (%s); run python paged_kv_cache_78_gb300/_build.py"
                          % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    sz = ctypes.c_size_t
    desc = ctypes.POINTER(CacheDesc)
    p_i32, p_i64, p_sz = ctypes.POINTER(i32), ctypes.POINTER(i64), ctypes.POINTER(sz)
    sig = {
        "pa_reshape_and_cache": [vp, desc, vp, vp, vp, i32, vp],
        "pa_copy_blocks": [vp, desc, vp, i32, vp],
        "pa_decode": [vp, vp, vp, desc, vp, i32, vp, i32, i32, f32, i32, i32, vp, sz, vp],
        "pa_decode_ex": [vp, vp, vp, desc, vp, i32, vp, i32, i32, f32, i32, i32, vp, sz, i32, vp],
        "pa_decode_no_alloc": [vp, vp, vp, desc, vp, i32, vp, i32, i32, f32, i32, i32, vp],
        "pa_decode_append": [vp, vp, vp, desc, vp, i32, vp, i32, i32, f32, i32, i32, vp, vp, vp,
                             sz, i32, vp],
        "pa_decode_partition_size": [desc, i32, i32, i32, i32, p_i32],
        "pa_decode_select_kernel": [desc, i32, i32, vp, i32, p_i32],
        "pa_decode_workspace_size": [desc, i32, i32, i32, i32, p_sz],
        "pa_slot_mapping": [vp, i32, i32, i32, i32, vp, vp, i32, vp],
        "pa_pool_create": [i32, i32, vp, ctypes.POINTER(vp)],
        "pa_pool_add_seq": [vp, i64, p_i64],
        "pa_pool_fork": [vp, i64, p_i64],
        "pa_pool_append_token": [vp, i64, p_i64, vp],
        "pa_pool_append_tokens": [vp, vp, i32, vp, vp, p_i32],
        "pa_pool_free_seq": [vp, i64],
        "pa_pool_block_table": [vp, i64, vp, i32, p_i32, p_i64],
        "pa_pool_fill_tables": [vp, vp, i32, vp, i32, vp],
        "pa_pool_slot": [vp, i64, i64, p_i64],
        "pa_pool_ref_count": [vp, i32, p_i32],
        "pa_get_device_error": [ctypes.POINTER(ctypes.c_uint32), vp],
        "pa_set_decode_trace": [vp, sz, i32],
        "pa_set_decode_wait_limit": [i64],
        "pa_decode_shared_plan": [vp, i32, vp, i32, i32, i32, i32, i32, vp, sz,
                                  ctypes.POINTER(SharedPlanInfo)],
        "pa_decode_shared_workspace_size": [desc, i32, i32, i32, ctypes.POINTER(SharedPlanInfo),
                                            p_sz],
        "pa_decode_shared": [vp, vp, vp, desc, vp, i32, vp, i32, i32, f32, i32, vp,
                             ctypes.POINTER(SharedPlanInfo), vp, vp, vp, sz, vp],
        "pa_pool_add_seq_tokens": [vp, vp, i64, p_i64, p_i64],
        "pa_pool_append_token_id": [vp, i64, i32, p_i64, vp],
        "pa_pool_is_cached": [vp, i32, p_i32],
        "pa_pool_free_queue": [vp, vp, i32, p_i32],
        "pa_pool_reset_prefix_cache": [vp],
        "pa_pool_usage": [vp, p_i64, p_i64],
        "pa_swap_blocks": [vp, desc, vp, desc, vp, i32, vp],
        "pa_copy_bytes": [vp, vp, sz, vp],
        "pa_pool_set_cpu_blocks": [vp, i32],
        "pa_pool_swap_out": [vp, vp, i32, vp, p_i32],
        "pa_pool_swap_in": [vp, vp, i32, vp, p_i32],
        "pa_pool_is_swapped": [vp, i64, p_i32],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.pa_pool_destroy.argtypes = [vp]
    lib.pa_pool_destroy.restype = None
    lib.pa_pool_num_free.argtypes = [vp]
    lib.pa_pool_num_free.restype = i32
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_version.argtypes = []
    lib.pa_version.restype = ctypes.c_char_p
    return lib


lib = _load()


def _status_string(status: int) -> str:
    return lib.pa_status_string(status).decode()


def _check(status: int, where: str) -> None:
    if status == PA_OK:
        return
    if status == PA_ERR_OUT_OF_BLOCKS:
        raise OutOfBlocks(status, where)
    raise PAError(status, where)


def version() -> str:
    return lib.pa_version().decode()


# ---------------------------------------------------------------------------
# tensor helpers
# ---------------------------------------------------------------------------

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float32:
        return PA_FP32
    raise TypeError("tensors must be bfloat16 or float32, got %s" % t.dtype)


def cache_desc(cache: torch.Tensor) -> CacheDesc:
    """Descriptor of a [2, num_blocks, block_size, num_kv_heads, head_size] pool."""
    if cache.dim() != 5 or cache.shape[0] != 2:
        raise ValueError("cache must be [2, num_blocks, block_size, num_kv_heads, head_size]")
    if not cache.is_contiguous():
        raise ValueError("cache must be contiguous")
    _, nb, bs, hkv, d = cache.shape
    return CacheDesc(nb, bs, hkv, d, _dtype_code(cache))


def _dev_ptr(t: torch.Tensor, name: str, dtype=None) -> int:
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ---------------------------------------------------------------------------
# kernels
# ---------------------------------------------------------------------------

def pa_reshape_and_cache(cache: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                         slot_mapping: torch.Tensor, stream=None) -> None:
    """cache[0/1, slot // bs, slot % bs] = key/value[t] for every slot >= 0."""
    desc = cache_desc(cache)
    n = key.shape[0]
    if key.shape != value.shape or tuple(key.shape[1:]) != (desc.num_kv_heads, desc.head_size):
        raise ValueError("key/value must be [num_tokens, num_kv_heads, head_size]")
    if key.dtype != cache.dtype or value.dtype != cache.dtype:
        raise TypeError("key/value dtype must match the cache")
    if slot_mapping.shape != (n,):
        raise ValueError("slot_mapping must be [num_tokens]")
    _check(lib.pa_reshape_and_cache(_dev_ptr(cache, "cache"), ctypes.byref(desc),
                                    _dev_ptr(key, "key") if n else None,
                                    _dev_ptr(value, "value") if n else None,
                                    _dev_ptr(slot_mapping, "slot_mapping", torch.int64) if n else None,
                                    n, _stream(stream)), "pa_reshape_and_cache")


def pa_copy_blocks(cache: torch.Tensor, pairs: torch.Tensor, stream=None) -> None:
    """Copy block pairs[i, 0] to block pairs[i, 1] (keys and values)."""
    desc = cache_desc(cache)
    n = pairs.shape[0] if pairs.numel() else 0
    if n and (pairs.dim() != 2 or pairs.shape[1] != 2):
        raise ValueError("pairs must be [num_pairs, 2]")
    _check(lib.pa_copy_blocks(_dev_ptr(cache, "cache"), ctypes.byref(desc),
                              _dev_ptr(pairs, "pairs", torch.int64) if n else None, n,
                              _stream(stream)), "pa_copy_blocks")


def _dev_or_pinned_ptr(t: torch.Tensor, name: str, dtype=None) -> int:
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("%s must be a CUDA tensor or page-locked host memory" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def pa_copy_bytes(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    """Copy src's bytes into dst with a library kernel; either side may be
    page-locked host memory.  Both contiguous, with the same byte size."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src differ in byte size")
    if nbytes == 0:
        return
    _check(lib.pa_copy_bytes(_dev_or_pinned_ptr(dst, "dst"), _dev_or_pinned_ptr(src, "src"),
                             nbytes, _stream(stream)), "pa_copy_bytes")


def pa_swap_blocks(dst_cache: torch.Tensor, src_cache: torch.Tensor, pairs: torch.Tensor,
                   stream=None) -> None:
    """Copy block pairs[i, 0] of src_cache to block pairs[i, 1] of dst_cache
    (keys and values); either pool may be page-locked host memory."""
    n = pairs.shape[0] if pairs.numel() else 0
    if n and (pairs.dim() != 2 or pairs.shape[1] != 2):
        raise ValueError("pairs must be [num_pairs, 2]")
    dd, sd = cache_desc(dst_cache), cache_desc(src_cache)
    _check(lib.pa_swap_blocks(_dev_or_pinned_ptr(dst_cache, "dst_cache"), ctypes.byref(dd),
                              _dev_or_pinned_ptr(src_cache, "src_cache"), ctypes.byref(sd),
                              _dev_or_pinned_ptr(pairs, "pairs", torch.int64) if n else None, n,
                              _stream(stream)), "pa_swap_blocks")


def pa_decode_partition_size(cache_or_desc, num_seqs: int, num_heads: int, max_seq_len: int,
                             partition_size: int = -1) -> int:
    desc = cache_or_desc if isinstance(cache_or_desc, CacheDesc) else cache_desc(cache_or_desc)
    out = ctypes.c_int32()
    _check(lib.pa_decode_partition_size(ctypes.byref(desc), num_seqs, num_heads, max_seq_len,
                                        partition_size, ctypes.byref(out)),
           "pa_decode_partition_size")
    return out.value


def pa_decode_select_kernel(cache_or_desc, num_seqs: int, num_heads: int, query_ptr: int = 0,
                            kernel: int = 0) -> int:
    """The kernel family (PA_KERNEL_SIMT or PA_KERNEL_TENSOR) pa_decode runs
    for these arguments; `query_ptr` is the query's device address (only its
    alignment matters), or 0 to assume a 256-byte aligned buffer."""
    desc = cache_or_desc if isinstance(cache_or_desc, CacheDesc) else cache_desc(cache_or_desc)
    out = ctypes.c_int32()
    _check(lib.pa_decode_select_kernel(ctypes.byref(desc), num_seqs, num_heads,
                                       ctypes.c_void_p(query_ptr or 256), kernel,
                                       ctypes.byref(out)),
           "pa_decode_select_kernel")
    return out.value


def pa_decode_workspace_size(cache_or_desc, num_seqs: int, num_heads: int, max_seq_len: int,
                             partition_size: int = -1) -> int:
    desc = cache_or_desc if isinstance(cache_or_desc, CacheDesc) else cache_desc(cache_or_desc)
    out = ctypes.c_size_t()
    _check(lib.pa_decode_workspace_size(ctypes.byref(desc), num_seqs, num_heads, max_seq_len,
                                        partition_size, ctypes.byref(out)),
           "pa_decode_workspace_size")
    return out.value


def alloc_workspace(nbytes: int, device) -> torch.Tensor | None:
    """Caller-owned decode workspace: zeroed (its header must start at zero),
    256-byte aligned by the caching allocator."""
    if nbytes == 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def pa_decode(out: torch.Tensor, query: torch.Tensor, cache: torch.Tensor,
              block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
              max_seq_len: int, partition_size: int = -1, workspace: torch.Tensor | None = None,
              stream=None, kernel: int = PA_KERNEL_AUTO) -> None:
    """out[s, hq] = softmax(scale * q[s, hq] . K_s) V_s over the paged tokens.
    kernel: PA_KERNEL_AUTO, PA_KERNEL_SIMT or PA_KERNEL_TENSOR (pa_decode_ex)."""
    desc = cache_desc(cache)
    s, hq, d = query.shape
    if out.shape != query.shape or d != desc.head_size:
        raise ValueError("query/out must be [num_seqs, num_heads, head_size]")
    if query.dtype != cache.dtype or out.dtype != cache.dtype:
        raise TypeError("query/out dtype must match the cache")
    if block_tables.dim() != 2 or block_tables.shape[0] != s or seq_lens.shape != (s,):
        raise ValueError("block_tables must be [num_seqs, max_blocks], seq_lens [num_seqs]")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()
    _check(lib.pa_decode_ex(_dev_ptr(out, "out"), _dev_ptr(query, "query"),
                            _dev_ptr(cache, "cache"), ctypes.byref(desc),
                            _dev_ptr(block_tables, "block_tables", torch.int32),
                            block_tables.shape[1], _dev_ptr(seq_lens, "seq_lens", torch.int32), s,
                            hq, float(scale), int(max_seq_len), int(partition_size), ws_ptr,
                            ws_bytes, int(kernel), _stream(stream)), "pa_decode")


def pa_decode_append(out: torch.Tensor, query: torch.Tensor, cache: torch.Tensor,
                     block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                     max_seq_len: int, key_new: torch.Tensor, value_new: torch.Tensor,
                     partition_size: int = -1, workspace: torch.Tensor | None = None,
                     stream=None, kernel: int = PA_KERNEL_AUTO) -> None:
    """pa_decode that first writes each sequence's newest token (position
    seq_lens[s] - 1; key_new / value_new [num_seqs, num_kv_heads, head_size])
    into its cache slot."""
    desc = cache_desc(cache)
    s, hq, d = query.shape
    if out.shape != query.shape or d != desc.head_size:
        raise ValueError("query/out must be [num_seqs, num_heads, head_size]")
    for name, t in (("query", query), ("out", out), ("key_new", key_new), ("value_new", value_new)):
        if t.dtype != cache.dtype:
            raise TypeError("%s dtype must match the cache" % name)
    if key_new.shape != (s, desc.num_kv_heads, d) or value_new.shape != key_new.shape:
        raise ValueError("key_new/value_new must be [num_seqs, num_kv_heads, head_size]")
    if block_tables.dim() != 2 or block_tables.shape[0] != s or seq_lens.shape != (s,):
        raise ValueError("block_tables must be [num_seqs, max_blocks], seq_lens [num_seqs]")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()
    _check(lib.pa_decode_append(_dev_ptr(out, "out"), _dev_ptr(query, "query"),
                                _dev_ptr(cache, "cache"), ctypes.byref(desc),
                                _dev_ptr(block_tables, "block_tables", torch.int32),
                                block_tables.shape[1], _dev_ptr(seq_lens, "seq_lens", torch.int32),
                                s, hq, float(scale), int(max_seq_len), int(partition_size),
                                _dev_ptr(key_new, "key_new"), _dev_ptr(value_new, "value_new"),
                                ws_ptr, ws_bytes, int(kernel), _stream(stream)), "pa_decode_append")


SHARED_TILE_ROWS = 128


class SharedPlan:
    """pa_decode_shared_plan on host block tables and lengths: the plan
    (int32, host) and its sizes; `upload` gives the device copy the decode
    reads."""

    def __init__(self, block_tables, seq_lens, block_size: int, num_heads: int,
                 num_kv_heads: int, min_shared_blocks: int = 8):
        bt = torch.as_tensor(block_tables).to(torch.int32).contiguous().cpu()
        sl = torch.as_tensor(seq_lens).to(torch.int32).contiguous().cpu()
        if bt.dim() != 2 or sl.shape != (bt.shape[0],):
            raise ValueError("block_tables must be [num_seqs, max_blocks], seq_lens [num_seqs]")
        n = bt.shape[0]
        self.plan = torch.zeros(4 + 6 * n, dtype=torch.int32)
        self.info = SharedPlanInfo()
        _check(lib.pa_decode_shared_plan(bt.data_ptr(), bt.shape[1], sl.data_ptr(), n, block_size,
                                         num_heads, num_kv_heads, min_shared_blocks,
                                         self.plan.data_ptr(), self.plan.numel(),
                                         ctypes.byref(self.info)), "pa_decode_shared_plan")
        self.plan = self.plan[:self.info.plan_ints].clone()

    @property
    def num_chunks(self) -> int:
        return int(self.info.num_chunks)

    def chunks(self):
        """[(first member index, members, shared tokens, group)] per chunk."""
        nc = self.num_chunks
        return [tuple(int(x) for x in self.plan[4 + 4 * c:8 + 4 * c]) for c in range(nc)]

    def seq_start(self):
        nc, n = self.num_chunks, int(self.plan[1])
        return self.plan[4 + 4 * nc:4 + 4 * nc + n].tolist()

    def members(self):
        nc, n = self.num_chunks, int(self.plan[1])
        return self.plan[4 + 4 * nc + n:].tolist()

    def upload(self, device="cuda") -> torch.Tensor:
        return self.plan.to(device)


def pa_decode_shared_workspace_size(cache_or_desc, num_seqs: int, num_heads: int,
                                    max_seq_len: int, plan: SharedPlan) -> int:
    desc = cache_or_desc if isinstance(cache_or_desc, CacheDesc) else cache_desc(cache_or_desc)
    out = ctypes.c_size_t()
    _check(lib.pa_decode_shared_workspace_size(ctypes.byref(desc), num_seqs, num_heads,
                                               int(max_seq_len), ctypes.byref(plan.info),
                                               ctypes.byref(out)),
           "pa_decode_shared_workspace_size")
    return out.value


def pa_decode_shared(out: torch.Tensor, query: torch.Tensor, cache: torch.Tensor,
                     block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                     max_seq_len: int, plan: SharedPlan, plan_dev: torch.Tensor,
                     workspace: torch.Tensor | None, key_new: torch.Tensor | None = None,
                     value_new: torch.Tensor | None = None, stream=None) -> None:
    """pa_decode with the blocks the plan's groups share attended once per
    group (plan_dev: the plan's device copy, SharedPlan.upload)."""
    desc = cache_desc(cache)
    s, hq, d = query.shape
    if out.shape != query.shape or d != desc.head_size:
        raise ValueError("query/out must be [num_seqs, num_heads, head_size]")
    if query.dtype != cache.dtype or out.dtype != cache.dtype:
        raise TypeError("query/out dtype must match the cache")
    if block_tables.dim() != 2 or block_tables.shape[0] != s or seq_lens.shape != (s,):
        raise ValueError("block_tables must be [num_seqs, max_blocks], seq_lens [num_seqs]")
    if (key_new is None) != (value_new is None):
        raise ValueError("key_new and value_new go together")
    kn = vn = None
    if key_new is not None:
        if key_new.shape != (s, desc.num_kv_heads, d) or value_new.shape != key_new.shape:
            raise ValueError("key_new/value_new must be [num_seqs, num_kv_heads, head_size]")
        kn, vn = _dev_ptr(key_new, "key_new"), _dev_ptr(value_new, "value_new")
    if plan_dev.numel() < plan.info.plan_ints:
        raise ValueError("plan_dev is shorter than the plan")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()
    _check(lib.pa_decode_shared(_dev_ptr(out, "out"), _dev_ptr(query, "query"),
                                _dev_ptr(cache, "cache"), ctypes.byref(desc),
                                _dev_ptr(block_tables, "block_tables", torch.int32),
                                block_tables.shape[1], _dev_ptr(seq_lens, "seq_lens", torch.int32),
                                s, hq, float(scale), int(max_seq_len),
                                _dev_ptr(plan_dev, "plan", torch.int32), ctypes.byref(plan.info),
                                kn, vn, ws_ptr, ws_bytes, _stream(stream)), "pa_decode_shared")


NO_ALLOC_WORKSPACE_BYTES = 16 << 20


def pa_decode_no_alloc(out: torch.Tensor, query: torch.Tensor, cache: torch.Tensor,
                       block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                       max_seq_len: int, partition_size: int = -1, stream=None) -> None:
    """pa_decode with the split-KV scratch in the library's own device array
    (for callers that cannot allocate device memory; see include/pa.h)."""
    desc = cache_desc(cache)
    s, hq, d = query.shape
    if out.shape != query.shape or d != desc.head_size:
        raise ValueError("query/out must be [num_seqs, num_heads, head_size]")
    if block_tables.dim() != 2 or block_tables.shape[0] != s or seq_lens.shape != (s,):
        raise ValueError("block_tables must be [num_seqs, max_blocks], seq_lens [num_seqs]")
    _check(lib.pa_decode_no_alloc(_dev_ptr(out, "out"), _dev_ptr(query, "query"),
                                  _dev_ptr(cache, "cache"), ctypes.byref(desc),
                                  _dev_ptr(block_tables, "block_tables", torch.int32),
                                  block_tables.shape[1],
                                  _dev_ptr(seq_lens, "seq_lens", torch.int32), s, hq,
                                  float(scale), int(max_seq_len), int(partition_size),
                                  _stream(stream)), "pa_decode_no_alloc")


def pa_slot_mapping(block_tables: torch.Tensor, block_size: int, num_blocks: int,
                    seq_idx: torch.Tensor, positions: torch.Tensor) -> torch.Tensor:
    """Host: physical slots of (sequence, position) pairs through CPU block tables."""
    bt = block_tables.to(torch.int32).contiguous().cpu()
    si = seq_idx.to(torch.int32).contiguous().cpu()
    po = positions.to(torch.int32).contiguous().cpu()
    n = si.numel()
    out = torch.empty(n, dtype=torch.int64)
    _check(lib.pa_slot_mapping(bt.data_ptr(), bt.shape[0], bt.shape[1], block_size, num_blocks,
                               si.data_ptr(), po.data_ptr(), n, out.data_ptr()), "pa_slot_mapping")
    return out


def pa_get_device_error(stream=None) -> int:
    """Synchronise, return and clear the device error word (PA_DEVERR_* bits)."""
    flags = ctypes.c_uint32()
    st = lib.pa_get_device_error(ctypes.byref(flags), _stream(stream))
    if st not in (PA_OK, PA_ERR_DEVICE_CHECK, PA_ERR_TIMEOUT):
        _check(st, "pa_get_device_error")
    return flags.value


# ---------------------------------------------------------------------------
# host block pool
# ---------------------------------------------------------------------------

class Pool:
    """The C++ block pool (pa_pool_*): block tables, slots, copy-on-write pairs."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self._h = ctypes.c_void_p()
        order = None
        if free_order is not None:
            self._order = (ctypes.c_int32 * num_blocks)(*[int(b) for b in free_order])
            order = ctypes.cast(self._order, ctypes.c_void_p)
        _check(lib.pa_pool_create(num_blocks, block_size, order, ctypes.byref(self._h)),
               "pa_pool_create")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib.pa_pool_destroy(h)
            self._h = None

    def add_seq(self, num_tokens: int) -> int:
        out = ctypes.c_int64()
        _check(lib.pa_pool_add_seq(self._h, num_tokens, ctypes.byref(out)), "pa_pool_add_seq")
        return out.value

    def fork(self, parent: int) -> int:
        out = ctypes.c_int64()
        _check(lib.pa_pool_fork(self._h, parent, ctypes.byref(out)), "pa_pool_fork")
        return out.value

    def append_token(self, seq: int):
        """Returns (slot, pair) with pair = (src, dst) of a copy-on-write, or None."""
        slot = ctypes.c_int64()
        pair = (ctypes.c_int64 * 2)()
        _check(lib.pa_pool_append_token(self._h, seq, ctypes.byref(slot), pair),
               "pa_pool_append_token")
        return slot.value, (None if pair[0] < 0 else (pair[0], pair[1]))

    def append_tokens(self, seqs):
        """append_token for each sequence, all or nothing: (slots int64[n], pairs int64[k,2])."""
        n = len(seqs)
        s = torch.tensor(list(seqs), dtype=torch.int64)
        slots = torch.empty(n, dtype=torch.int64)
        pairs = torch.empty((max(n, 1), 2), dtype=torch.int64)
        k = ctypes.c_int32()
        _check(lib.pa_pool_append_tokens(self._h, s.data_ptr(), n, slots.data_ptr(),
                                         pairs.data_ptr(), ctypes.byref(k)),
               "pa_pool_append_tokens")
        return slots, pairs[:k.value].clone()

    def free_seq(self, seq: int) -> None:
        _check(lib.pa_pool_free_seq(self._h, seq), "pa_pool_free_seq")

    # -- prefix caching --------------------------------------------------------
    def add_seq_tokens(self, tokens):
        """New sequence from prompt token ids, sharing cached prefix blocks:
        (seq id, number of leading tokens whose KV is already cached)."""
        t = torch.tensor([int(x) for x in tokens], dtype=torch.int32)
        sid = ctypes.c_int64()
        cached = ctypes.c_int64()
        _check(lib.pa_pool_add_seq_tokens(self._h, t.data_ptr() if t.numel() else None, t.numel(),
                                          ctypes.byref(sid), ctypes.byref(cached)),
               "pa_pool_add_seq_tokens")
        return sid.value, cached.value

    def append_token_id(self, seq: int, token: int):
        """append_token that records the token id: (slot, pair or None)."""
        slot = ctypes.c_int64()
        pair = (ctypes.c_int64 * 2)()
        _check(lib.pa_pool_append_token_id(self._h, seq, int(token), ctypes.byref(slot), pair),
               "pa_pool_append_token_id")
        return slot.value, (None if pair[0] < 0 else (pair[0], pair[1]))

    def is_cached(self, block: int) -> bool:
        out = ctypes.c_int32()
        _check(lib.pa_pool_is_cached(self._h, block, ctypes.byref(out)), "pa_pool_is_cached")
        return bool(out.value)

    def free_queue(self):
        """The free queue, front (next handed out) first."""
        buf = (ctypes.c_int32 * max(self.num_blocks, 1))()
        n = ctypes.c_int32()
        _check(lib.pa_pool_free_queue(self._h, buf, self.num_blocks, ctypes.byref(n)),
               "pa_pool_free_queue")
        return list(buf[:n.value])

    def usage(self):
        """(tokens held by live sequences, physical blocks in use)."""
        t, b = ctypes.c_int64(), ctypes.c_int64()
        _check(lib.pa_pool_usage(self._h, ctypes.byref(t), ctypes.byref(b)), "pa_pool_usage")
        return t.value, b.value

    # -- swapping ---------------------------------------------------------------
    def set_cpu_blocks(self, n: int) -> None:
        _check(lib.pa_pool_set_cpu_blocks(self._h, n), "pa_pool_set_cpu_blocks")
        self.num_cpu_blocks = n

    def _swap(self, fn, name, seqs):
        s = torch.tensor([int(x) for x in seqs], dtype=torch.int64)
        cap = max(1, self.num_blocks)
        pairs = torch.empty((cap, 2), dtype=torch.int64)
        k = ctypes.c_int32()
        _check(fn(self._h, s.data_ptr() if s.numel() else None, s.numel(), pairs.data_ptr(),
                  ctypes.byref(k)), name)
        return pairs[:k.value].clone()

    def swap_out(self, seqs):
        """Move a sequence group to CPU blocks: int64 [k, 2] (GPU block, CPU block) pairs."""
        return self._swap(lib.pa_pool_swap_out, "pa_pool_swap_out", seqs)

    def swap_in(self, seqs):
        """Move a swapped group back: int64 [k, 2] (CPU block, GPU block) pairs."""
        return self._swap(lib.pa_pool_swap_in, "pa_pool_swap_in", seqs)

    def is_swapped(self, seq: int) -> bool:
        out = ctypes.c_int32()
        _check(lib.pa_pool_is_swapped(self._h, seq, ctypes.byref(out)), "pa_pool_is_swapped")
        return bool(out.value)

    def num_free_cpu(self) -> int:
        return int(lib.pa_pool_num_free_cpu(self._h))

    def reset_prefix_cache(self) -> None:
        _check(lib.pa_pool_reset_prefix_cache(self._h), "pa_pool_reset_prefix_cache")

    def table(self, seq: int):
        n = ctypes.c_int32()
        length = ctypes.c_int64()
        cap = 16
        while True:
            buf = (ctypes.c_int32 * cap)()
            st = lib.pa_pool_block_table(self._h, seq, buf, cap, ctypes.byref(n),
                                         ctypes.byref(length))
            if st == PA_OK:
                return list(buf[:n.value]), length.value
            if st == PA_ERR_INVALID_ARG and n.value > cap:
                cap = n.value
                continue
            _check(st, "pa_pool_block_table")

    def fill_tables(self, seqs, max_blocks_per_seq: int):
        """Dense int32 [n, max_blocks_per_seq] tables and int32 [n] lengths (host)."""
        n = len(seqs)
        s = torch.tensor(list(seqs), dtype=torch.int64)
        bt = torch.empty((n, max_blocks_per_seq), dtype=torch.int32)
        sl = torch.empty(n, dtype=torch.int32)
        _check(lib.pa_pool_fill_tables(self._h, s.data_ptr(), n, bt.data_ptr(),
                                       max_blocks_per_seq, sl.data_ptr()), "pa_pool_fill_tables")
        return bt, sl

    def slot(self, seq: int, pos: int) -> int:
        out = ctypes.c_int64()
        _check(lib.pa_pool_slot(self._h, seq, pos, ctypes.byref(out)), "pa_pool_slot")
        return out.value

    def ref_count(self, block: int) -> int:
        out = ctypes.c_int32()
        _check(lib.pa_pool_ref_count(self._h, block, ctypes.byref(out)), "pa_pool_ref_count")
        return out.value

    def num_free(self) -> int:
        return int(lib.pa_pool_num_free(self._h))


def tensor_core_supported(cache: torch.Tensor, num_heads: int) -> bool:
    """Whether PA_KERNEL_TENSOR has a kernel for this cache and head count."""
    try:
        pa_decode_select_kernel(cache, 1, num_heads, kernel=PA_KERNEL_TENSOR)
    except PAError as e:
        if e.status == PA_ERR_UNSUPPORTED:
            return False
        raise
    return True


def pa_set_decode_trace(buffer: torch.Tensor | None, events_per_role: int = 0) -> None:
    """Record the tensor-core decode's timeline into `buffer` (a CUDA tensor;
    see include/pa.h for the record format), or stop recording (None)."""
    if buffer is None:
        _check(lib.pa_set_decode_trace(None, 0, 0), "pa_set_decode_trace")
        return
    _check(lib.pa_set_decode_trace(_dev_ptr(buffer, "buffer"),
                                   buffer.numel() * buffer.element_size(), int(events_per_role)),
           "pa_set_decode_trace")


def pa_set_decode_wait_limit(cycles: int) -> None:
    """Limit (SM clock cycles) of the tensor-core decode's pipeline waits;
    0 restores the default.  A test hook: see include/pa.h."""
    _check(lib.pa_set_decode_wait_limit(int(cycles)), "pa_set_decode_wait_limit")
