"""GPU parity of the cache write and the copy-on-write block copy: bit-exact
against the oracle, including padding slots, untouched bytes and ids outside
the pool (skipped and recorded, never faulting)."""
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
