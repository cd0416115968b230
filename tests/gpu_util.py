"""Helpers for the GPU parity tests: move seeded workloads to the device, run
the library's path (cache fill, step write, decode) through the C ABI, and
compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_78_gb300 as pa

# bf16 mode: |o - ref| <= 8e-3 + 1e-2 |ref|.
BF16_ATOL, BF16_RTOL = 8e-3, 1e-2
# fp32 mode: |o - ref| <= 1e-5 |ref| + 1e-5 max_row |ref|.
FP32_RTOL = 1e-5


def to_device(a: np.ndarray, device="cuda") -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    """Device tensor back to the oracle's representation (bf16 -> uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).cpu().numpy()


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "") -> float:
    """Tolerance check; returns the largest error relative to the bound."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output " + what
    err = np.abs(got - ref)
    if dtype == "bf16":
        bound = BF16_ATOL + BF16_RTOL * np.abs(ref)
    else:
        rowmax = np.max(np.abs(ref), axis=-1, keepdims=True)
        bound = FP32_RTOL * np.abs(ref) + FP32_RTOL * rowmax + 1e-30
    worst = float(np.max(err / bound)) if err.size else 0.0
    if worst > 1.0:
        idx = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError("%s: error %.3g at %s exceeds bound %.3g (got %r, ref %r)" % (
            what, err[idx], idx, bound[idx], got[idx], ref[idx]))
    return worst


class DeviceCase:
    """A workload's pool, tables and step inputs on the GPU, filled through
    the library's own slot mapping and cache write."""

    def __init__(self, case, device="cuda"):
        self.case = case
        self.device = device
        self.cache = to_device(case.initial_cache(), device)
        self.block_tables = to_device(case.block_tables, device)
        self.seq_lens = to_device(case.seq_lens, device)
        self.query = to_device(case.query, device)
        self.out = torch.empty_like(self.query)
        bt_host = torch.from_numpy(case.block_tables)
        # prefill: every token but the last of each sequence
        seqs, pos, rows = case.token_positions(exclude_last=True)
        if rows.size:
            slots = pa.pa_slot_mapping(bt_host, case.block_size, case.num_blocks,
                                       torch.from_numpy(seqs), torch.from_numpy(pos))
            pa.pa_reshape_and_cache(self.cache, to_device(case.keys[rows], device),
                                    to_device(case.values[rows], device), slots.to(device))
        # the decode step's new tokens
        seqs, pos, rows = case.token_positions(last_only=True)
        self.step_slots = pa.pa_slot_mapping(bt_host, case.block_size, case.num_blocks,
                                             torch.from_numpy(seqs),
                                             torch.from_numpy(pos)).to(device)
        self.step_keys = to_device(case.keys[rows], device)
        self.step_values = to_device(case.values[rows], device)
        # the same tokens as one row per sequence (zeros where a sequence is empty)
        new_k = np.zeros((case.num_seqs,) + case.keys.shape[1:], dtype=case.keys.dtype)
        new_v = np.zeros_like(new_k)
        new_k[seqs] = case.keys[rows]
        new_v[seqs] = case.values[rows]
        self.new_keys = to_device(new_k, device)
        self.new_values = to_device(new_v, device)

    def step(self, partition_size=-1, workspace=None, kernel=pa.PA_KERNEL_AUTO):
        c = self.case
        pa.pa_reshape_and_cache(self.cache, self.step_keys, self.step_values, self.step_slots)
        if workspace is None:
            nbytes = pa.pa_decode_workspace_size(self.cache, c.num_seqs, c.num_heads,
                                                 c.max_seq_len, partition_size)
            workspace = pa.alloc_workspace(nbytes, self.device)
        pa.pa_decode(self.out, self.query, self.cache, self.block_tables, self.seq_lens,
                     c.scale, c.max_seq_len, partition_size, workspace, kernel=kernel)
        return self.out


    def step_fused(self, partition_size=-1, workspace=None, kernel=pa.PA_KERNEL_AUTO):
        """The same step with the cache write fused into the decode."""
        c = self.case
        if workspace is None:
            nbytes = pa.pa_decode_workspace_size(self.cache, c.num_seqs, c.num_heads,
                                                 c.max_seq_len, partition_size)
            workspace = pa.alloc_workspace(nbytes, self.device)
        pa.pa_decode_append(self.out, self.query, self.cache, self.block_tables, self.seq_lens,
                            c.scale, c.max_seq_len, self.new_keys, self.new_values,
                            partition_size, workspace, kernel=kernel)
        return self.out


def oracle_reference(case, seqs=None):
    """Oracle output for the listed sequences (all by default), with the
    cache filled through the oracle's own scatter."""
    cache = oracle.fill_cache(case)
    if seqs is None:
        return oracle.decode(case.query, cache, case.block_tables, case.seq_lens, case.scale), cache
    seqs = np.asarray(seqs)
    return oracle.decode(np.ascontiguousarray(case.query[seqs]), cache,
                         np.ascontiguousarray(case.block_tables[seqs]),
                         np.ascontiguousarray(case.seq_lens[seqs]), case.scale), cache
