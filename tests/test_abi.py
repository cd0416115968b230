"""The C-ABI library loads and exports every symbol include/pa.h declares;
host-side argument checks reject bad calls before any CUDA work."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_cache_78_gb300 as pa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for required in ("pa_reshape_and_cache", "pa_decode", "pa_copy_blocks", "pa_pool_create"):
        assert required in names
    assert set(names) == set(pa.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(pa.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings():
    assert pa.version().count(".") == 2
    assert pa.lib.pa_status_string(pa.PA_ERR_OUT_OF_BLOCKS) == b"out of blocks"
    assert pa.lib.pa_status_string(99) == b"unknown status"


def desc(**kw):
    d = dict(num_blocks=16, block_size=16, num_kv_heads=2, head_size=64, dtype=pa.PA_BF16)
    d.update(kw)
    return pa.CacheDesc(**d)


@pytest.mark.parametrize("bad", [dict(block_size=12), dict(block_size=512), dict(num_blocks=0),
                                 dict(dtype=7), dict(head_size=0), dict(num_kv_heads=0)])
def test_bad_cache_desc_rejected_without_launch(bad):
    d = desc(**bad)
    st = pa.lib.pa_reshape_and_cache(ctypes.c_void_p(16), ctypes.byref(d), ctypes.c_void_p(16),
                                     ctypes.c_void_p(16), ctypes.c_void_p(16), 4, None)
    assert st == pa.PA_ERR_INVALID_ARG


def test_decode_argument_checks():
    d = desc()
    p = ctypes.c_void_p(256)
    call = lambda **kw: pa.lib.pa_decode(
        kw.get("out", p), p, kw.get("cache", p), ctypes.byref(kw.get("desc", d)), p,
        kw.get("mb", 4), p, kw.get("s", 2), kw.get("hq", 14), kw.get("scale", 0.125),
        kw.get("max_len", 64), kw.get("part", 0), None, 0, None)
    assert call(hq=13) == pa.PA_ERR_INVALID_ARG            # heads not a multiple of kv heads
    assert call(out=None) == pa.PA_ERR_INVALID_ARG
    assert call(cache=ctypes.c_void_p(258)) == pa.PA_ERR_INVALID_ARG   # cache not 16-byte aligned
    assert call(scale=float("nan")) == pa.PA_ERR_INVALID_ARG
    assert call(mb=0) == pa.PA_ERR_INVALID_ARG
    assert call(s=0) == pa.PA_OK                           # empty batch: no-op
    assert call(desc=desc(head_size=96)) == pa.PA_ERR_UNSUPPORTED
    assert call(hq=2 * 17) == pa.PA_ERR_UNSUPPORTED        # group of 17
    assert call(hq=2 * 9, desc=desc(dtype=pa.PA_FP32)) == pa.PA_ERR_UNSUPPORTED  # fp32, group 9
    assert call(hq=2 * 9, desc=desc(block_size=4)) == pa.PA_ERR_UNSUPPORTED     # 4-token blocks


def test_kernel_selection_rule():
    sel = pa.pa_decode_select_kernel
    qwen = desc(block_size=16, num_kv_heads=2, head_size=64)
    assert sel(qwen, 64, 14) == pa.PA_KERNEL_TENSOR                  # G = 7
    opt = desc(block_size=16, num_kv_heads=40, head_size=128)
    assert sel(opt, 32, 40) == pa.PA_KERNEL_SIMT                     # G = 1
    assert sel(opt, 32, 40, kernel=pa.PA_KERNEL_TENSOR) == pa.PA_KERNEL_TENSOR
    assert sel(qwen, 64, 14, kernel=pa.PA_KERNEL_SIMT) == pa.PA_KERNEL_SIMT
    assert sel(qwen, 64, 14, query_ptr=256 + 8) == pa.PA_KERNEL_SIMT  # query not 16-byte aligned
    assert sel(desc(block_size=4, num_kv_heads=2, head_size=64), 4, 8) == pa.PA_KERNEL_SIMT
    f32 = desc(block_size=16, num_kv_heads=2, head_size=64, dtype=pa.PA_FP32)
    assert sel(f32, 4, 8) == pa.PA_KERNEL_SIMT
    with pytest.raises(pa.PAError) as e:
        sel(f32, 4, 8, kernel=pa.PA_KERNEL_TENSOR)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    assert sel(qwen, 4, 2 * 12) == pa.PA_KERNEL_TENSOR               # G = 12: tensor cores only
    with pytest.raises(pa.PAError) as e:
        sel(qwen, 4, 2 * 12, kernel=pa.PA_KERNEL_SIMT)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    with pytest.raises(pa.PAError) as e:
        sel(qwen, 4, 15)                                             # 15 % 2 != 0
    assert e.value.status == pa.PA_ERR_INVALID_ARG


def test_partition_and_workspace_sizes():
    d = desc(block_size=16, num_kv_heads=8, head_size=128)
    assert pa.pa_decode_partition_size(d, 8, 32, 32768, 512) == 512
    assert pa.pa_decode_partition_size(d, 8, 32, 300, 512) == 0      # one partition: no split
    assert pa.pa_decode_partition_size(d, 8, 32, 32768, 0) == 0
    with pytest.raises(pa.PAError):
        pa.pa_decode_partition_size(d, 8, 32, 32768, 520)           # not a multiple of 16
    nbytes = pa.pa_decode_workspace_size(d, 8, 32, 32768, 512)
    rows = 8 * 32 * 64
    assert nbytes == 256 + -(-rows * 128 * 4 // 256) * 256 + -(-rows * 4 // 256) * 256
    assert pa.pa_decode_workspace_size(d, 8, 32, 300, 512) == 256   # header only


def test_zero_work_calls_are_noops():
    d = desc()
    assert pa.lib.pa_reshape_and_cache(None, ctypes.byref(d), None, None, None, 0, None) == pa.PA_OK
    assert pa.lib.pa_copy_blocks(None, ctypes.byref(d), None, 0, None) == pa.PA_OK


def test_copy_pair_count_limit():
    # Two CTAs per pair along grid x: more than 2^30 - 1 pairs is refused
    # before any CUDA call.
    d = desc()
    p = ctypes.c_void_p(256)
    assert pa.lib.pa_copy_blocks(p, ctypes.byref(d), p, 1 << 30, None) == pa.PA_ERR_INVALID_ARG
    assert pa.lib.pa_swap_blocks(p, ctypes.byref(d), p, ctypes.byref(d), p, 1 << 30,
                                 None) == pa.PA_ERR_INVALID_ARG
    assert pa.lib.pa_copy_blocks(p, ctypes.byref(d), p, -1, None) == pa.PA_ERR_INVALID_ARG


def test_wait_limit_argument_checks():
    # A host-side setting: a negative limit is refused, 0 restores the default.
    assert pa.lib.pa_set_decode_wait_limit(-1) == pa.PA_ERR_INVALID_ARG
    assert pa.lib.pa_set_decode_wait_limit(0) == pa.PA_OK


def test_copy_bytes_argument_checks():
    # Validated before any CUDA call: zero bytes is a no-op, null pointers
    # and sizes past 2^40 are refused; the Python wrapper refuses tensors of
    # different byte sizes and host tensors that are not page-locked.
    assert pa.lib.pa_copy_bytes(None, None, 0, None) == pa.PA_OK
    assert pa.lib.pa_copy_bytes(None, ctypes.c_void_p(64), 16, None) == pa.PA_ERR_INVALID_ARG
    assert pa.lib.pa_copy_bytes(ctypes.c_void_p(64), None, 16, None) == pa.PA_ERR_INVALID_ARG
    assert pa.lib.pa_copy_bytes(ctypes.c_void_p(64), ctypes.c_void_p(128), (1 << 40) + 1,
                                None) == pa.PA_ERR_INVALID_ARG
    a = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(ValueError):
        pa.pa_copy_bytes(a, torch.zeros(8, dtype=torch.uint8))
    with pytest.raises(ValueError):
        pa.pa_copy_bytes(a, torch.zeros(16, dtype=torch.uint8))   # pageable host memory
    pa.pa_copy_bytes(a[:0], a[:0])                                 # nothing to copy
