"""GPU parity of the cache write and the copy-on-write block copy: bit-exact
against the oracle, including padding slots, untouched bytes and ids outside
the pool (skipped and recorded, never faulting)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_78_gb300 as pa
import workloads
from gpu_util import to_device, to_host_bits

pytestmark = pytest.mark.gpu


def bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.fixture(autouse=True)
def clean_error_word():
    pa.pa_get_device_error()
    yield


@pytest.mark.parametrize("dtype,nb,bs,hkv,d,ntok", [
    ("bf16", 64, 4, 4, 64, 4),
    ("bf16", 512, 16, 2, 64, 64),
    ("bf16", 300, 16, 40, 128, 200),
    ("fp32", 128, 8, 8, 128, 77),
    ("bf16", 40, 1, 3, 256, 33),
    ("fp32", 16, 256, 1, 64, 1000),
])
def test_reshape_and_cache_bit_exact(dtype, nb, bs, hkv, d, ntok):
    rng = np.random.default_rng(nb + bs + d)
    cache = workloads.garbage_values(rng, (2, nb, bs, hkv, d), dtype)
    slots = rng.choice(nb * bs, size=ntok, replace=False).astype(np.int64)
    slots[::5] = -1
    k = workloads.random_values(rng, (ntok, hkv, d), dtype)
    v = workloads.random_values(rng, (ntok, hkv, d), dtype)
    dev = to_device(cache)
    pa.pa_reshape_and_cache(dev, to_device(k), to_device(v), to_device(slots))
    oracle.reshape_and_cache(cache, k, v, slots)
    assert np.array_equal(bits(to_host_bits(dev)), bits(cache))
    assert pa.pa_get_device_error() == 0


def test_reshape_and_cache_slot_outside_pool_is_skipped_and_recorded():
    rng = np.random.default_rng(5)
    nb, bs, hkv, d = 8, 4, 2, 64
    cache = workloads.random_values(rng, (2, nb, bs, hkv, d), "bf16")
    slots = np.array([3, nb * bs, 7, nb * bs + 100], dtype=np.int64)
    k = workloads.random_values(rng, (4, hkv, d), "bf16")
    v = workloads.random_values(rng, (4, hkv, d), "bf16")
    dev = to_device(cache)
    pa.pa_reshape_and_cache(dev, to_device(k), to_device(v), to_device(slots))
    assert pa.pa_get_device_error() & pa.PA_DEVERR_SLOT
    keep = slots < nb * bs
    oracle.reshape_and_cache(cache, k[keep], v[keep], slots[keep])
    assert np.array_equal(to_host_bits(dev), cache)


@pytest.mark.parametrize("dtype,nb,bs,hkv,d", [
    ("bf16", 64, 16, 8, 128), ("fp32", 32, 4, 2, 64), ("bf16", 12, 256, 1, 256)])
def test_copy_blocks_bit_exact(dtype, nb, bs, hkv, d):
    rng = np.random.default_rng(nb * 7 + bs)
    cache = workloads.garbage_values(rng, (2, nb, bs, hkv, d), dtype)
    perm = rng.permutation(nb)
    n = nb // 3
    pairs = np.stack([perm[:n], perm[n:2 * n]], axis=1).astype(np.int64)
    dev = to_device(cache)
    pa.pa_copy_blocks(dev, to_device(pairs))
    oracle.copy_blocks(cache, pairs)
    assert np.array_equal(bits(to_host_bits(dev)), bits(cache))
    assert pa.pa_get_device_error() == 0


def test_copy_blocks_bad_id_is_skipped_and_recorded():
    rng = np.random.default_rng(9)
    cache = workloads.random_values(rng, (2, 10, 4, 2, 64), "fp32")
    pairs = np.array([[1, 2], [3, 10], [-1, 4], [5, 6]], dtype=np.int64)
    dev = to_device(cache)
    pa.pa_copy_blocks(dev, to_device(pairs))
    assert pa.pa_get_device_error() & pa.PA_DEVERR_BLOCK_ID
    oracle.copy_blocks(cache, pairs[[0, 3]])
    assert np.array_equal(to_host_bits(dev), cache)


def test_zero_token_and_zero_pair_calls():
    cache = torch.zeros((2, 4, 4, 1, 64), dtype=torch.bfloat16, device="cuda")
    empty = torch.empty((0, 1, 64), dtype=torch.bfloat16, device="cuda")
    pa.pa_reshape_and_cache(cache, empty, empty, torch.empty(0, dtype=torch.int64, device="cuda"))
    pa.pa_copy_blocks(cache, torch.empty((0, 2), dtype=torch.int64, device="cuda"))
    assert not cache.any()


def _pinned_like(rng, shape, dtype):
    host = workloads.garbage_values(rng, shape, dtype)
    if dtype == "bf16":
        t = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(host)
    return host, t.pin_memory()


def _host_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
        else t.numpy().view(np.uint32)


@pytest.mark.parametrize("dtype,nb,ncpu,bs,hkv,d", [
    ("bf16", 64, 32, 16, 2, 64),
    ("bf16", 40, 40, 8, 8, 128),
    ("fp32", 24, 12, 4, 4, 64),
])
def test_swap_round_trip_bit_exact(dtype, nb, ncpu, bs, hkv, d):
    # A sequence group leaves the GPU for page-locked host blocks and comes
    # back to other GPU blocks; every byte matches a plain block assignment
    # and CPU blocks outside the pairs keep their canary bytes.
    rng = np.random.default_rng(nb + ncpu + d)
    gpu_host = workloads.garbage_values(rng, (2, nb, bs, hkv, d), dtype)
    gpu = to_device(gpu_host)
    cpu_ref, cpu = _pinned_like(rng, (2, ncpu, bs, hkv, d), dtype)
    pool = pa.Pool(nb, bs)
    pool.set_cpu_blocks(ncpu)
    a = pool.add_seq(3 * bs + 1)
    a2 = pool.fork(a)
    pool.add_seq(2 * bs)                              # another request keeps its blocks
    out = pool.swap_out([a, a2])                      # (GPU block, CPU block)
    for pairs in (out.cuda(), out.pin_memory()):      # pair lists on the device or pinned
        pa.pa_swap_blocks(cpu, gpu, pairs)
        torch.cuda.synchronize()
        expect = cpu_ref.copy()
        expect[:, out[:, 1].numpy()] = gpu_host[:, out[:, 0].numpy()]
        assert np.array_equal(_host_bits(cpu), bits(expect))
    back = pool.swap_in([a, a2])                      # (CPU block, GPU block)
    assert sorted(back[:, 0].tolist()) == sorted(out[:, 1].tolist())
    pa.pa_swap_blocks(gpu, cpu, back.cuda())
    torch.cuda.synchronize()
    now = to_host_bits(gpu)
    old_of_new = {int(c): int(g) for g, c in out.tolist()}
    for c, g in back.tolist():
        assert np.array_equal(bits(now[:, g]), bits(gpu_host[:, old_of_new[c]]))
    assert pa.pa_get_device_error() == 0


def test_swap_refuses_pageable_host_memory():
    cache = torch.zeros((2, 4, 4, 2, 64), dtype=torch.bfloat16, device="cuda")
    pageable = torch.zeros((2, 4, 4, 2, 64), dtype=torch.bfloat16)
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    desc = pa.cache_desc(cache)
    st = pa.lib.pa_swap_blocks(pageable.data_ptr(), ctypes.byref(desc), cache.data_ptr(),
                               ctypes.byref(desc), pairs.data_ptr(), 1, None)
    assert st == pa.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("nbytes,dst_off,src_off", [
    (1, 0, 0), (15, 0, 0), (16, 0, 0), (17, 0, 0), (4096 + 3, 0, 0),
    ((1 << 20) + 5, 0, 0), ((1 << 22) + 48, 16, 32),      # vectors, 4 in flight, ragged tail
    (1000, 1, 0), (70001, 3, 5),                          # misaligned: byte by byte
])
@pytest.mark.parametrize("route", ["h2d", "d2h", "d2d", "h2h"])
def test_copy_bytes_bit_exact(nbytes, dst_off, src_off, route):
    # Every byte of the range arrives; the bytes around it keep their canary.
    rng = np.random.default_rng(nbytes + dst_off + src_off)
    src_np = rng.integers(0, 256, size=nbytes + src_off + 64, dtype=np.uint8)
    dst_np = rng.integers(0, 256, size=nbytes + dst_off + 64, dtype=np.uint8)

    def place(a, where):
        t = torch.from_numpy(a)
        return t.pin_memory() if where == "h" else t.cuda()

    src = place(src_np, route[0])
    dst = place(dst_np.copy(), route[-1])
    pa.pa_copy_bytes(dst[dst_off:dst_off + nbytes], src[src_off:src_off + nbytes])
    torch.cuda.synchronize()
    expect = dst_np.copy()
    expect[dst_off:dst_off + nbytes] = src_np[src_off:src_off + nbytes]
    assert np.array_equal(dst.cpu().numpy(), expect)


def test_copy_bytes_refuses_pageable_and_overlapping_ranges():
    dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(4096, dtype=torch.uint8)
    assert pa.lib.pa_copy_bytes(dev.data_ptr(), pageable.data_ptr(), 4096, None) == \
        pa.PA_ERR_INVALID_ARG
    assert pa.lib.pa_copy_bytes(pageable.data_ptr(), dev.data_ptr(), 4096, None) == \
        pa.PA_ERR_INVALID_ARG
    assert pa.lib.pa_copy_bytes(dev.data_ptr() + 16, dev.data_ptr(), 64, None) == \
        pa.PA_ERR_INVALID_ARG
    assert pa.lib.pa_copy_bytes(dev.data_ptr(), dev.data_ptr() + 64, 64, None) == pa.PA_OK
    assert pa.lib.pa_copy_bytes(dev.data_ptr(), None, 0, None) == pa.PA_OK
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
