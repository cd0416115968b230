"""GPU parity of the shared-prefix decode (pa_decode_shared): sequences that
share leading blocks have those blocks attended once per group, their own
tokens by the tensor-core decode, and the two combined by the log-sum-exp
reduce.  Every output row is compared with the oracle's paged decode of the
whole sequence, over ragged shared lengths, groups cut into several chunks,
every query-group size the tile takes (1, 4, 7, 16), head sizes 64 and 128,
block sizes 8 to 64, and with the step's cache write fused in."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_78_gb300 as pa
import workloads
from gpu_util import assert_close, to_device, to_f64, to_host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clean_error_word():
    pa.pa_get_device_error()
    yield


def shared_case(groups, singles, hq, hkv, d, bs, seed):
    """A pool of random rows and tables where each group's members share
    their first `shared` blocks; members and singles then have 1..`own`
    tokens of their own.  groups: [(members, shared blocks, own max)]."""
    rng = np.random.default_rng(seed)
    lens = []
    for members, shared, own in groups:
        for _ in range(members):
            lens.append(shared * bs + int(rng.integers(1, own, endpoint=True)))
    lens += [int(x) for x in rng.integers(1, 700, size=singles, endpoint=True)]
    need = sum(sh for _, sh, _ in groups) + sum(
        -(-(n - (groups_shared(groups, i) * bs)) // bs) for i, n in enumerate(lens))
    nb = need + 5
    perm = iter(rng.permutation(nb).tolist())
    tables = []
    i = 0
    for members, shared, _ in groups:
        common = [next(perm) for _ in range(shared)]
        for _ in range(members):
            own = -(-(lens[i] - shared * bs) // bs)
            tables.append(common + [next(perm) for _ in range(own)])
            i += 1
    for n in lens[i:]:
        tables.append([next(perm) for _ in range(-(-n // bs))])
    order = rng.permutation(len(lens))  # groups interleaved with the rest
    lens = np.array([lens[j] for j in order], dtype=np.int32)
    mb = max(len(t) for t in tables)
    bt = np.zeros((len(lens), mb), dtype=np.int32)
    for r, j in enumerate(order):
        bt[r, :len(tables[j])] = tables[j]
    cache = workloads.random_values(rng, (2, nb, bs, hkv, d), "bf16")
    q = workloads.random_values(rng, (len(lens), hq, d), "bf16")
    return cache, bt, lens, q


def groups_shared(groups, i):
    """Shared blocks of sequence i (0 for the singles after the groups)."""
    for members, shared, _ in groups:
        if i < members:
            return shared
        i -= members
    return 0


def run_shared(cache, bt, lens, q, hq, hkv, bs, min_blocks=1, new_kv=None):
    d = cache.shape[-1]
    plan = pa.SharedPlan(bt, lens, bs, hq, hkv, min_blocks)
    dev_cache = to_device(cache)
    out = torch.empty((len(lens), hq, d), dtype=torch.bfloat16, device="cuda")
    ws = pa.alloc_workspace(pa.pa_decode_shared_workspace_size(dev_cache, len(lens), hq,
                                                               int(lens.max()), plan), "cuda")
    kn = vn = None
    if new_kv is not None:
        kn, vn = to_device(new_kv[0]), to_device(new_kv[1])
    pa.pa_decode_shared(out, to_device(q), dev_cache, to_device(bt), to_device(lens),
                        1.0 / np.sqrt(d), int(lens.max()), plan, plan.upload(), ws, kn, vn)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    return to_f64(out), plan, dev_cache


@pytest.mark.parametrize("d,hq,hkv,bs,groups,singles", [
    (128, 32, 8, 16, [(8, 63, 64), (3, 10, 200)], 4),    # forked samples, G = 4
    (64, 14, 2, 16, [(40, 20, 300)], 3),                  # 3 chunks of 16/16/8, ragged stage
    (128, 8, 8, 32, [(130, 5, 40)], 0),                   # G = 1: 2 chunks of 128/2 rows
    (128, 32, 2, 8, [(9, 40, 100)], 2),                   # G = 16: 8 members a chunk
    (64, 16, 4, 64, [(5, 9, 500), (2, 2, 60)], 5),        # 64-token blocks
], ids=["g4_d128_bs16", "g7_d64_bs16", "g1_d128_bs32", "g16_d128_bs8", "g4_d64_bs64"])
def test_shared_decode_matches_the_oracle(d, hq, hkv, bs, groups, singles):
    cache, bt, lens, q = shared_case(groups, singles, hq, hkv, d, bs, seed=hq * d + bs)
    got, plan, _ = run_shared(cache, bt, lens, q, hq, hkv, bs)
    assert plan.num_chunks >= len(groups)
    want = oracle.decode(q, cache, bt, lens, 1.0 / np.sqrt(d))
    assert_close(got, want, "bf16", "shared-prefix decode vs oracle")


def test_shared_decode_with_the_fused_cache_write():
    hq, hkv, d, bs = 32, 8, 128, 16
    cache, bt, lens, q = shared_case([(6, 30, 90)], 3, hq, hkv, d, bs, seed=5)
    rng = np.random.default_rng(6)
    new_k = workloads.random_values(rng, (len(lens), hkv, d), "bf16")
    new_v = workloads.random_values(rng, (len(lens), hkv, d), "bf16")
    got, _, dev_cache = run_shared(cache, bt, lens, q, hq, hkv, bs, new_kv=(new_k, new_v))
    slots = oracle.slot_mapping(bt, np.arange(len(lens)), lens - 1, bs)
    oracle.reshape_and_cache(cache, new_k, new_v, slots)
    assert np.array_equal(to_host_bits(dev_cache), cache)
    want = oracle.decode(q, cache, bt, lens, 1.0 / np.sqrt(d))
    assert_close(got, want, "bf16", "shared-prefix decode with the fused write vs oracle")


def test_shared_decode_without_sharing_is_the_plain_decode():
    hq, hkv, d, bs = 16, 4, 64, 16
    cache, bt, lens, q = shared_case([], 6, hq, hkv, d, bs, seed=8)
    got, plan, _ = run_shared(cache, bt, lens, q, hq, hkv, bs)
    assert plan.num_chunks == 0
    want = oracle.decode(q, cache, bt, lens, 1.0 / np.sqrt(d))
    assert_close(got, want, "bf16", "decode with an empty plan vs oracle")


def test_two_calls_reuse_the_workspace():
    # The second call finds the first call's piece counts and partials in the
    # workspace; a batch where fewer sequences share must not combine them.
    hq, hkv, d, bs = 32, 8, 128, 16
    cache, bt, lens, q = shared_case([(10, 12, 80)], 4, hq, hkv, d, bs, seed=11)
    plan = pa.SharedPlan(bt, lens, bs, hq, hkv)
    dev_cache = to_device(cache)
    ws = pa.alloc_workspace(pa.pa_decode_shared_workspace_size(dev_cache, len(lens), hq,
                                                               int(lens.max()), plan), "cuda")
    scale = 1.0 / np.sqrt(d)
    for lens_now in (lens, np.minimum(lens, 5 * bs + 3).astype(np.int32)):
        p = pa.SharedPlan(bt, lens_now, bs, hq, hkv, 3)
        need = pa.pa_decode_shared_workspace_size(dev_cache, len(lens), hq, int(lens.max()), p)
        assert need <= ws.numel()
        out = torch.zeros((len(lens), hq, d), dtype=torch.bfloat16, device="cuda")
        pa.pa_decode_shared(out, to_device(q), dev_cache, to_device(bt), to_device(lens_now),
                            scale, int(lens.max()), p, p.upload(), ws)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        want = oracle.decode(q, cache, bt, lens_now, scale)
        assert_close(to_f64(out), want, "bf16", "second call vs oracle")


def test_plan_inconsistent_with_the_lengths_is_refused_on_the_device():
    # A plan claiming more shared tokens than a member holds: the unit is
    # refused and recorded, nothing outside the buffers is touched.
    hq, hkv, d, bs = 16, 4, 128, 16
    cache, bt, lens, q = shared_case([(4, 8, 30)], 2, hq, hkv, d, bs, seed=13)
    plan = pa.SharedPlan(bt, lens, bs, hq, hkv)
    assert plan.num_chunks == 1
    bad = plan.plan.clone()
    bad[4 + 2] = int(lens.max()) + bs * 4   # shared tokens of chunk 0
    dev_cache = to_device(cache)
    out = torch.zeros((len(lens), hq, d), dtype=torch.bfloat16, device="cuda")
    ws = pa.alloc_workspace(pa.pa_decode_shared_workspace_size(dev_cache, len(lens), hq,
                                                               int(lens.max()), plan), "cuda")
    pa.pa_decode_shared(out, to_device(q), dev_cache, to_device(bt), to_device(lens),
                        1.0 / np.sqrt(d), int(lens.max()), plan, bad.cuda(), ws)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_SEQ_LEN
    # Rows of sequences outside the group are still exact.
    singles = [r for r in range(len(lens)) if r not in set(plan.members())]
    want = oracle.decode(q, cache, bt, lens, 1.0 / np.sqrt(d))
    assert_close(to_f64(out)[singles], want[singles], "bf16", "rows outside the refused group")
