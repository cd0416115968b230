"""Benchmark of the paged decode hot path on GB300.

One step = the whole hot path over one batch: the cache write of the step's
new tokens (pa_reshape_and_cache through slot_mapping), any copy-on-write
block copies, then paged decode attention (pa_decode: single pass, or
split-KV partitions plus the log-sum-exp reduce).

Default workload: the long-context batch (8 sequences of 32768 tokens, 32
query / 8 KV heads of 128, block size 16, split-KV in 512-token partitions
with the log-sum-exp reduce, one new token per sequence per step): the
largest single-GPU configuration, and one of the two the >= 70 % of HBM
bandwidth target names.  Other workloads (the Qwen2-0.5B-shaped GQA batch,
the OPT-13B-shaped MHA batch at block sizes 8/16/32, the mixed-length
long-context batch, the shared-prefix batches): --workload.

Printed: one JSON line (rank 0).  `value` is algorithmic GB/s of the whole
step (bytes the step must move, divided by its device time); `roofline`
reports the decode call alone against the measured HBM copy bandwidth;
`e2e` repeats the step through the C ABI with host buffers (pinned H2D of
the step's inputs, D2H of the output) inside the timed region;
`cpu_baseline` times the CPU oracle on this host, on all its cores and on
one.  L2 is flushed before every timed step: a 256 MB write, then a 256 MB
read so that the written lines are evicted (and written back) before the step
starts.  Right before the timed steps the step runs untimed for a quarter of
a second, so the first timed steps do not start from an idle clock.

`--impl reference` times the CPU oracle as the reference arm, on the same
workload, metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged decode attn: achieved HBM GB/s (% of GB300 peak), µs per batch step"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20
PREROLL_S = 0.25


def spread_us(times_ms):
    """Mean, median, min and max of per-launch event times, in µs."""
    if not times_ms:
        return None
    return {"mean": round(sum(times_ms) / len(times_ms) * 1e3, 2),
            "median": round(statistics.median(times_ms) * 1e3, 2),
            "min": round(min(times_ms) * 1e3, 2), "max": round(max(times_ms) * 1e3, 2),
            "first": round(times_ms[0] * 1e3, 2)}


def make_workload(name: str):
    if name == "qwen2_gqa":
        return workloads.qwen2_gqa()
    if name.startswith("opt13b_mha_bs"):
        return workloads.opt13b_mha(block_size=int(name[len("opt13b_mha_bs"):]))
    if name == "long_context":
        return workloads.long_context(mixed=False)
    if name == "long_context_mixed":
        return workloads.long_context(mixed=True)
    if name == "tiny":
        return workloads.tiny()
    if name in ("shared_prefix_fork", "shared_prefix_prefix"):
        return shared_prefix_case(name[len("shared_prefix_"):])
    raise SystemExit("unknown workload %s" % name)


def shared_prefix_case(variant: str):
    """The shared-prefix / parallel-sampling batch: the seeded pool script
    (16 requests of a 1018-token prompt forked into 8 samples with 1-64 private
    tokens each, or 128 requests forked from one 512-token prefix with 64-512
    private tokens) replayed on the library's host pool, so forks share blocks
    by reference count and a write into a shared, partly filled block moves
    the writer to a copy.  K/V are drawn once per physical slot and gathered
    per sequence, so every sequence sharing a block sees the same rows."""
    import paged_kv_cache_78_gb300 as pa

    script = workloads.shared_prefix_script(variant=variant)
    pool = pa.Pool(script.num_blocks, script.block_size, script.free_order)
    for kind, arg in script.ops:
        if kind == "add":
            pool.add_seq(arg)
        elif kind == "fork":
            pool.fork(arg)
        else:
            pool.append_token(arg)
    seqs = script.decode_seqs
    mb = max(len(pool.table(x)[0]) for x in seqs)
    bt, sl = pool.fill_tables(seqs, mb)
    bt, sl = bt.numpy().astype(np.int32), sl.numpy().astype(np.int32)
    hq, hkv, d, bs, nb = 32, 8, 128, script.block_size, script.num_blocks
    rng = np.random.default_rng([3, 9, int(variant == "fork")])
    slot_k = workloads.random_values(rng, (nb * bs, hkv, d), "bf16")
    slot_v = workloads.random_values(rng, (nb * bs, hkv, d), "bf16")
    idx = np.concatenate([bt[r, np.arange(n) // bs].astype(np.int64) * bs + np.arange(n) % bs
                          for r, n in enumerate(sl)])
    starts = np.zeros(len(seqs) + 1, dtype=np.int64)
    starts[1:] = np.cumsum(sl.astype(np.int64))
    q = workloads.random_values(rng, (len(seqs), hq, d), "bf16")
    return workloads.DecodeCase("shared_prefix_" + variant, 3, hq, hkv, d, bs, nb, "bf16",
                                1.0 / math.sqrt(d), sl, bt, q, slot_k[idx], slot_v[idx], starts,
                                meta={"unique_slots": int(np.unique(idx).size)})


# Workloads whose statement fixes the split-KV partition (512-token partitions
# for the long-context batches); the others take the library's choice.
WORKLOAD_PARTITION = {"long_context": 512, "long_context_mixed": 512}


# The largest length each workload's statement allows (what a contiguous
# max-length preallocation reserves per sequence).
WORKLOAD_MAX_LEN = {"qwen2_gqa": 2048, "long_context": 32768, "long_context_mixed": 131072,
                    "shared_prefix_fork": 2048, "shared_prefix_prefix": 2048}


def memory_report(pa, case, workload: str) -> dict:
    """KV memory the workload's sequences leave allocated but unused: paged
    (the library's host pool, block sizes 8/16/32; the waste sits in each
    sequence's last block) against reserving the largest allowed length per
    sequence in one contiguous region."""
    lens = [int(n) for n in case.seq_lens]
    max_len = WORKLOAD_MAX_LEN.get(workload, 2048)
    paged = {}
    for bs in (8, 16, 32):
        pool = pa.Pool(sum(-(-n // bs) for n in lens) + 1, bs)
        for n in lens:
            pool.add_seq(n)
        tokens, blocks = pool.usage()
        paged[str(bs)] = {"waste": round(1.0 - tokens / max(1, blocks * bs), 5),
                          "unused_slots_per_seq": round((blocks * bs - tokens) / len(lens), 2)}
    used = sum(lens)
    return {"paged": paged, "contiguous_reserved_len": max_len,
            "contiguous_waste": round(1.0 - used / (len(lens) * max_len), 5)}


BALANCED = -2  # the library's PA_PARTITION_BALANCED


def balanced_pieces(case, ranges: int, start=None) -> np.ndarray:
    """Pieces of each (sequence, KV head) pair under the balanced split: the
    pairs' 128-token stages (of tokens [start, L) when given) laid end to
    end, cut every ceil(total / ranges) stages."""
    lens = case.seq_lens.astype(np.int64)
    if start is not None:
        lens = np.where(lens > 0, lens - np.minimum(start, lens - 1), 0)
    n = (lens + 127) // 128
    per_pair = np.repeat(n, case.num_kv_heads)
    total = int(per_pair.sum())
    q = max(1, -(-total // ranges))
    start = np.concatenate([[0], np.cumsum(per_pair)[:-1]])
    pieces = np.where(per_pair > 0, (start + per_pair - 1) // q - start // q + 1, 0)
    return pieces


def shared_ranges(case, plan, sms: int) -> int:
    """Stage ranges per (chunk, KV head) of the shared-prefix decode's group
    kernel: the library's rule (fill the SMs, no more than the shortest
    chunk's stages, at most 16)."""
    units = plan.num_chunks * case.num_kv_heads
    r = sms // units if units else 1
    r = min(r, plan.info.min_chunk_stages, 16)
    return max(1, r)


def step_bytes(case, partition: int = 0, ranges: int = 0, plan=None, sms: int = 0) -> dict:
    """Algorithmic bytes of one step: what the operations must read and write
    once.  With split-KV partitions, each sequence of more than one partition
    also writes and reads its fp32 partials (head_size values and a log-sum-exp
    per query head and partition); the balanced split (over `ranges` stage
    ranges) writes and reads those of every pair cut into several pieces; the
    shared-prefix decode those of every member row (its shared ranges and its
    own part)."""
    eb = workloads.elem_bytes(case.dtype)
    s, hq, hkv, d = case.num_seqs, case.num_heads, case.num_kv_heads, case.head_size
    lens = case.seq_lens.astype(np.int64)
    blocks = int(((lens + case.block_size - 1) // case.block_size).sum())
    logical_kv = case.kv_bytes()
    # Sequences sharing blocks read each shared K/V row once (from DRAM; the
    # other readers find it in L2): the roofline counts the distinct slots.
    kv = logical_kv
    if "unique_slots" in case.meta:
        kv = case.meta["unique_slots"] * hkv * d * 2 * eb
    decode = kv + 2 * s * hq * d * eb + 4 * blocks + 4 * s
    partials = 0
    if plan is not None and plan.num_chunks:
        # Member rows: one partial per range of the group kernel when it has
        # several; the other sequences: the balanced split's pieces.
        r = shared_ranges(case, plan, sms)
        member = np.array(plan.seq_start(), dtype=np.int64) > 0
        if r > 1:
            partials += int(member.sum()) * hq * r * (d + 1) * 4 * 2
        if not member.all():
            pieces = balanced_pieces(case, sms * (2 if d == 64 else 1))
            pieces = np.where(np.repeat(member, hkv), 0, pieces)
            partials += int(pieces[pieces > 1].sum()) * (hq // hkv) * (d + 1) * 4 * 2
    elif partition > 0:
        parts = (lens + partition - 1) // partition
        partials = int(parts[parts > 1].sum()) * hq * (d + 1) * 4 * 2
    elif partition == BALANCED:
        pieces = balanced_pieces(case, ranges)
        partials = int(pieces[pieces > 1].sum()) * (hq // hkv) * (d + 1) * 4 * 2
    t = int((lens > 0).sum())  # one new token per sequence
    write = t * hkv * d * eb * 2 * 2 + 8 * t  # read new K/V, write them, read slots
    # "step": the workload's bytes, the same whatever partitions a run uses;
    # "decode": what the decode call moves, partials included.
    return {"decode": int(decode + partials), "partials": partials, "write": int(write),
            "step": int(decode + write), "logical_kv": int(logical_kv), "unique_kv": int(kv)}


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest() -> str:
    csrc = os.path.join(ROOT, "paged_kv_cache_78_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.startswith("decode") or f in ("pa_device.cuh", "pa_tcgen05.cuh", "api.cu"):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, partition: int):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu
    summary, when it was taken on the current kernel source and at the same
    resolved partition (another split is another kernel variant)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    entry = data.get(workload)
    if not entry or entry.get("kernel_digest") != kernel_source_digest():
        return None
    if entry.get("partition") != partition:
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = [p for t, p in self.samples if t0 <= t <= t1] or [p for _, p in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def bf16_or_f32_to_device(torch, a, device):
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class GpuStep:
    """A workload resident on the device, and its step through the C ABI.
    With `shared`, the decode is pa_decode_shared over a plan of the blocks
    the batch's sequences share (built on the host from the block tables)."""

    def __init__(self, torch, pa, case, device, partition, kernel=0, shared=False):
        self.torch, self.pa, self.case, self.device = torch, pa, case, device
        self.kernel = kernel
        self.plan = None
        to_dev = lambda a: bf16_or_f32_to_device(torch, a, device)
        self.cache = to_dev(case.initial_cache())
        bt_host = torch.from_numpy(case.block_tables)
        seqs, pos, rows = case.token_positions(exclude_last=True)
        chunk = 1 << 16
        for i in range(0, rows.size, chunk):  # prefill, through the library's own write
            sl = slice(i, i + chunk)
            slots = pa.pa_slot_mapping(bt_host, case.block_size, case.num_blocks,
                                       torch.from_numpy(seqs[sl]), torch.from_numpy(pos[sl]))
            pa.pa_reshape_and_cache(self.cache, to_dev(case.keys[rows[sl]]),
                                    to_dev(case.values[rows[sl]]), slots.to(device))
        seqs, pos, rows = case.token_positions(last_only=True)
        self.slots_host = pa.pa_slot_mapping(bt_host, case.block_size, case.num_blocks,
                                             torch.from_numpy(seqs), torch.from_numpy(pos))
        self.k_host = case.keys[rows]
        self.v_host = case.values[rows]
        self.slots = self.slots_host.to(device)
        self.k = to_dev(self.k_host)
        self.v = to_dev(self.v_host)
        self.q = to_dev(case.query)
        self.bt = to_dev(case.block_tables)
        self.sl = to_dev(case.seq_lens)
        self.out = torch.empty_like(self.q)
        self.partition = pa.pa_decode_partition_size(self.cache, case.num_seqs, case.num_heads,
                                                     case.max_seq_len, partition)
        nbytes = pa.pa_decode_workspace_size(self.cache, case.num_seqs, case.num_heads,
                                             case.max_seq_len, self.partition)
        split = self.partition > 0 or (self.partition == BALANCED and case.max_seq_len > 128)
        self.launches = 2 + (1 if split else 0)
        if shared:
            self.plan = pa.SharedPlan(case.block_tables, case.seq_lens, case.block_size,
                                      case.num_heads, case.num_kv_heads)
            self.plan_dev = self.plan.upload(device)
            nbytes = pa.pa_decode_shared_workspace_size(self.cache, case.num_seqs, case.num_heads,
                                                        case.max_seq_len, self.plan)
            sms = torch.cuda.get_device_properties(device).multi_processor_count
            others = self.plan.info.num_members < case.num_seqs
            self.launches = 1 + (1 + int(others) + int(others or shared_ranges(
                case, self.plan, sms) > 1) if self.plan.num_chunks else 1)
        self.ws = pa.alloc_workspace(nbytes, device)
        if int((case.seq_lens > 0).sum()) != case.num_seqs:
            raise SystemExit("the bench's workloads give every sequence a new token")
        family = pa.pa_decode_select_kernel(self.cache, case.num_seqs, case.num_heads,
                                            self.q.data_ptr(), kernel)
        self.kernel_name = ("paged_decode_tc_kernel" if family == pa.PA_KERNEL_TENSOR
                            else "paged_decode_kernel")
        if self.plan is not None:
            self.kernel_name = "paged_decode_shared_kernel + paged_decode_tc_kernel"

    def write(self):
        self.pa.pa_reshape_and_cache(self.cache, self.k, self.v, self.slots)

    def decode(self):
        c = self.case
        if self.plan is not None:
            self.pa.pa_decode_shared(self.out, self.q, self.cache, self.bt, self.sl, c.scale,
                                     c.max_seq_len, self.plan, self.plan_dev, self.ws)
            return
        self.pa.pa_decode(self.out, self.q, self.cache, self.bt, self.sl, c.scale, c.max_seq_len,
                          self.partition, self.ws, kernel=self.kernel)

    def write_and_decode(self):
        """The step as one call: the decode writes each sequence's newest
        token itself (pa_decode_append, or pa_decode_shared with the new
        tokens)."""
        c = self.case
        if self.plan is not None:
            self.pa.pa_decode_shared(self.out, self.q, self.cache, self.bt, self.sl, c.scale,
                                     c.max_seq_len, self.plan, self.plan_dev, self.ws, self.k,
                                     self.v)
            return
        self.pa.pa_decode_append(self.out, self.q, self.cache, self.bt, self.sl, c.scale,
                                 c.max_seq_len, self.k, self.v, self.partition, self.ws,
                                 kernel=self.kernel)

    def inputs(self):
        """Names of the step's host-supplied inputs (the plan too when shared)."""
        return STEP_INPUTS + (("plan_dev",) if self.plan is not None else ())


STEP_INPUTS = ("q", "k", "v", "slots", "bt", "sl")


def pack_step_inputs(torch, st, device):
    """Place the step's inputs (query, new K/V, slots, block tables, lengths)
    in one device arena, each 256-byte aligned, with a page-locked host copy
    of the same bytes: a step's host-to-device traffic is then one copy.
    The step's tensors become views into the arena."""
    spans, off = {}, 0
    names = st.inputs()
    for name in names:
        t = getattr(st, name)
        nbytes = t.numel() * t.element_size()
        spans[name] = (off, nbytes)
        off += (nbytes + 255) // 256 * 256
    arena = torch.zeros(off, dtype=torch.uint8, device=device)
    for name in names:
        t = getattr(st, name)
        o, nbytes = spans[name]
        view = arena[o:o + nbytes].view(t.dtype).view(t.shape)
        view.copy_(t)
        setattr(st, name, view)
    host = arena.cpu().pin_memory()
    return arena, host


def sms_of(torch, device) -> int:
    return torch.cuda.get_device_properties(device).multi_processor_count


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over all ranks of the default
    process group (each replica's time; the job takes as long as its slowest
    rank)."""
    import torch

    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def run_gpu(args, rank, world, device):
    import torch

    import paged_kv_cache_78_gb300 as pa

    torch.cuda.set_device(device)
    case = make_workload(args.workload)
    partition = args.partition if args.partition != -1 else WORKLOAD_PARTITION.get(args.workload, -1)
    shared = args.shared == 1 or (args.shared == -1 and args.workload.startswith("shared_prefix"))
    st = GpuStep(torch, pa, case, device, partition, args.kernel, shared)
    arena, arena_host = pack_step_inputs(torch, st, device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    nbytes = step_bytes(case, st.partition, ranges=sms * (2 if case.head_size == 64 else 1),
                        plan=st.plan, sms=sms)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()

    class _Flush:
        # Write a buffer larger than L2, then read another one: the read
        # evicts the written lines (their write-back happens here, not in the
        # timed step) and leaves L2 holding clean, unrelated data.
        @staticmethod
        def zero_():
            flush_w.zero_()
            flush_r.sum()

    flush = _Flush

    graphs = None
    if args.graph:
        # One graph for the whole step (its kernels chained by programmatic
        # dependent launch), and one for the decode call alone.
        st.write()
        st.decode()
        torch.cuda.synchronize()
        g_step, g_write, g_decode = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                     torch.cuda.CUDAGraph())
        with torch.cuda.graph(g_step):
            if args.fused:
                st.write_and_decode()
            else:
                st.write()
                st.decode()
        with torch.cuda.graph(g_write):
            st.write()
        with torch.cuda.graph(g_decode):
            st.decode()
        graphs = (g_step, g_write, g_decode)

    def step():
        if graphs:
            graphs[0].replay()
        elif args.fused:
            st.write_and_decode()
        else:
            st.write()
            st.decode()

    def write():
        graphs[1].replay() if graphs else st.write()

    def decode():
        graphs[2].replay() if graphs else st.decode()

    for _ in range(args.warmup):
        flush.zero_()
        step()
        flush.zero_()
        write()
        decode()
    torch.cuda.synchronize()
    flags = pa.pa_get_device_error()
    if flags:
        raise RuntimeError("device error word 0x%x after warm-up" % flags)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # Keep the GPU busy up to the timed region (the sleep above lets its
    # clock fall to idle, and the first steps after an idle spell run slow).
    t_pre = time.time()
    while time.time() - t_pre < PREROLL_S:
        for _ in range(8):
            flush.zero_()
            step()
        torch.cuda.synchronize()
    mk = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    ev = [mk() for _ in range(args.steps)]
    ev_dec = [mk() for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    # The K timed steps: cache write + decode, L2 evicted before each.
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    # The decode call alone (the roofline's kernel), K more times, the step's
    # cache write done untimed before each.
    for e0, e1 in ev_dec:
        flush.zero_()
        write()
        e0.record(stream)
        decode()
        e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    step_each = [a.elapsed_time(b) for a, b in ev]
    decode_each = [a.elapsed_time(b) for a, b in ev_dec]
    step_ms = sum(step_each)
    decode_ms = sum(decode_each)
    if world > 1:
        step_ms, decode_ms = max_over_ranks([step_ms, decode_ms], device)
    spread = {"step_us": spread_us(step_each), "decode_us": spread_us(decode_each)}

    # Outside the timed steps: the decode call warm (no eviction, inputs left
    # in L2 by the previous call), and the same tokens in the unpaged layout
    # (consecutive blocks), L2 evicted, to report what paging costs.
    paging = None
    if args.paging and world == 1 and "unique_slots" in case.meta:
        paging = {"skipped": "sequences share blocks: a consecutive-block layout would duplicate "
                             "the shared blocks and read more bytes"}
    elif args.paging and world == 1:
        n = max(50, args.steps // 4)
        warm = [mk() for _ in range(n)]
        for e0, e1 in warm:
            e0.record(stream)
            decode()
            e1.record(stream)
        st_c = GpuStep(torch, pa, workloads.contiguous(case), device, st.partition, args.kernel)
        st_c.write()
        st_c.decode()
        g_c = None
        if args.graph:
            torch.cuda.synchronize()
            g_c = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_c):
                st_c.decode()
        cont = [mk() for _ in range(n)]
        for _ in range(3):
            flush.zero_()
            g_c.replay() if g_c else st_c.decode()
        for e0, e1 in cont:
            flush.zero_()
            st_c.write()
            e0.record(stream)
            g_c.replay() if g_c else st_c.decode()
            e1.record(stream)
        torch.cuda.synchronize()
        warm_us = sum(a.elapsed_time(b) for a, b in warm) / n * 1e3
        cont_us = sum(a.elapsed_time(b) for a, b in cont) / n * 1e3
        paged_us = decode_ms / args.steps * 1e3
        paging = {"paged_us_per_launch": round(paged_us, 2),
                  "contiguous_us_per_launch": round(cont_us, 2),
                  "overhead": round(paged_us / cont_us - 1.0, 4),
                  "warm_us_per_launch": round(warm_us, 2),
                  "launches": n,
                  "note": "decode call on the same tokens with consecutive physical blocks "
                          "(L2 evicted), and the paged call without eviction (warm)"}
        del st_c, g_c
    flags = pa.pa_get_device_error()
    if flags:
        raise RuntimeError("device error word 0x%x after the timed region" % flags)

    # End to end through the C ABI with host buffers: pinned H2D of the
    # step's inputs, the step, D2H of the output, all inside the timed region.
    # The host side holds the step's inputs in one page-locked arena (query,
    # new K/V, slots, block tables, lengths: pack_step_inputs), copied in with
    # one transfer per step.  By default both transfers are the library's
    # copy kernel (pa_copy_bytes), chained with the step's kernels by
    # programmatic dependent launch; --e2e-copy dma takes the copy engine.
    out_host = torch.empty(st.out.numel() * st.out.element_size(), dtype=torch.uint8).pin_memory()
    h2d = arena_host.numel()
    d2h = out_host.numel()

    out_bytes = st.out.view(torch.uint8).view(-1)

    def e2e_step():
        if args.e2e_copy == "kernel":
            pa.pa_copy_bytes(arena, arena_host)
        else:
            arena.copy_(arena_host, non_blocking=True)
        if args.fused:
            st.write_and_decode()
        else:
            st.write()
            st.decode()
        if args.e2e_copy == "kernel":
            pa.pa_copy_bytes(out_host, out_bytes)
        else:
            out_host.copy_(out_bytes, non_blocking=True)

    if not args.e2e:
        clocks = sampler.summary(t0, t1) if sampler else None
        if sampler:
            sampler.stop()
        return {"case": case, "step": st, "bytes": nbytes, "step_ms": step_ms / args.steps,
                "decode_ms": decode_ms / args.steps, "e2e_ms": None, "clocks": clocks,
                "h2d": h2d, "d2h": d2h, "paging": paging, "spread": spread}
    for _ in range(max(3, args.warmup // 4)):
        flush.zero_()
        e2e_step()
    torch.cuda.synchronize()
    if args.graph:
        # The serving loop's form: the step with its copies from and to the
        # pinned host buffers captured once and replayed every step.
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_step()
        e2e_call = g_e2e.replay
        for _ in range(3):
            flush.zero_()
            e2e_call()
        torch.cuda.synchronize()
    else:
        e2e_call = e2e_step
    e2e_steps = max(10, args.steps // 4)
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(e2e_steps)]
    for a, b in ev2:
        flush.zero_()
        a.record(stream)
        e2e_call()
        b.record(stream)
    torch.cuda.synchronize()
    e2e_each = [a.elapsed_time(b) for a, b in ev2]
    e2e_ms = sum(e2e_each) / e2e_steps
    spread["e2e_us"] = spread_us(e2e_each)
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()

    if world > 1:
        e2e_ms = max_over_ranks([e2e_ms], device)[0]
    return {"case": case, "step": st, "bytes": nbytes, "step_ms": step_ms / args.steps,
            "decode_ms": decode_ms / args.steps, "e2e_ms": e2e_ms, "clocks": clocks,
            "h2d": h2d, "d2h": d2h, "paging": paging, "spread": spread}


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

class OracleStep:
    """The step on the CPU oracle for the first `n` sequences of the batch."""

    def __init__(self, case, n=None):
        import oracle

        self.oracle = oracle
        self.case = case
        n = case.num_seqs if n is None else n
        self.n = n
        self.cache = oracle.fill_cache(case, exclude_last=True)
        seqs, pos, rows = case.token_positions(last_only=True)
        keep = seqs < n
        self.slots = oracle.slot_mapping(case.block_tables, seqs[keep], pos[keep], case.block_size)
        self.k = np.ascontiguousarray(case.keys[rows[keep]])
        self.v = np.ascontiguousarray(case.values[rows[keep]])
        self.q = np.ascontiguousarray(case.query[:n])
        self.bt = np.ascontiguousarray(case.block_tables[:n])
        self.sl = np.ascontiguousarray(case.seq_lens[:n])

    def run(self):
        self.oracle.reshape_and_cache(self.cache, self.k, self.v, self.slots)
        return self.oracle.decode(self.q, self.cache, self.bt, self.sl, self.case.scale)

    def bytes(self):
        sub = workloads.DecodeCase(**{**self.case.__dict__, "seq_lens": self.sl,
                                      "block_tables": self.bt, "query": self.q})
        return step_bytes(sub)["step"]


def oracle_sample(case, per_step_s: float):
    """An OracleStep over the longest prefix of sequences whose estimated
    oracle time fits per_step_s (at least one sequence)."""
    probe = OracleStep(case, 1)
    probe.run()
    t = time.perf_counter()
    probe.run()
    per_token = (time.perf_counter() - t) / max(1, int(case.seq_lens[0]))
    cum = np.cumsum(case.seq_lens.astype(np.float64)) * per_token
    n = int(max(1, np.searchsorted(cum, per_step_s, side="right")))
    return probe if n == 1 else OracleStep(case, min(n, case.num_seqs))


def time_oracle(case, budget_s: float, steps: int = 0, threads: int = 0):
    """Per-step times of the oracle on a bounded sample of the batch: `steps`
    runs, or as many as fit budget_s; on `threads` threads (0 = all of the
    host's cores, the oracle's default).  Returns (times, sample, threads)."""
    import oracle

    every = oracle.num_threads()
    if threads:
        oracle.set_num_threads(threads)
    try:
        per_step = budget_s / max(1, steps) if steps else budget_s / 5
        step = oracle_sample(case, per_step)
        times = []
        t_start = time.time()
        while (steps and len(times) < steps) or \
                (not steps and (not times or time.time() - t_start < budget_s)):
            t = time.perf_counter()
            step.run()
            times.append(time.perf_counter() - t)
        used = oracle.num_threads()
    finally:
        oracle.set_num_threads(every)
    return times, step, used


def config_for(case, name, partition=0):
    lens = case.seq_lens
    return {"workload": name, "num_seqs": case.num_seqs, "num_heads": case.num_heads,
            "num_kv_heads": case.num_kv_heads, "head_size": case.head_size,
            "block_size": case.block_size, "num_blocks": case.num_blocks,
            "seq_len_min": int(lens.min()), "seq_len_max": int(lens.max()),
            "seq_len_mean": round(float(lens.mean()), 1),
            "new_tokens_per_step": int((lens > 0).sum()),
            "bytes_per_step": step_bytes(case)["step"],
            "l2": "flushed before every timed step (256 MB write, then 256 MB read)"}


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_context")
    ap.add_argument("--partition", type=int, default=-1,
                    help="tokens per split-KV partition; 0 = no split, -1 = library's choice")
    ap.add_argument("--graph", type=int, default=0,
                    help="replay the step as CUDA graphs (default: plain launches on the "
                         "stream, chained by programmatic dependent launch; measured faster "
                         "on GB300: 27.2 vs 28.0 us per Qwen2-shape step, e2e 41.8 vs 46.3)")
    ap.add_argument("--kernel", type=int, default=0,
                    help="decode kernel family: 0 = library's choice, 1 = CUDA cores, 2 = tensor cores")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the CPU baseline (0 = skip)")
    ap.add_argument("--e2e", type=int, default=1, help="also time the step with host buffers")
    ap.add_argument("--e2e-copy", choices=("kernel", "dma"), default="kernel",
                    help="host<->device transfers of the end-to-end step: the library's copy "
                         "kernel (pa_copy_bytes) or the copy engine")
    ap.add_argument("--fused", type=int, default=1,
                    help="1: the step is one pa_decode_append (the decode writes the new tokens); "
                         "0: pa_reshape_and_cache, then pa_decode")
    ap.add_argument("--shared", type=int, default=-1,
                    help="1: decode with pa_decode_shared (blocks the sequences share attended "
                         "once per group), 0: pa_decode; -1 (default): 1 for the shared-prefix "
                         "workloads")
    ap.add_argument("--paging", type=int, default=1,
                    help="also time the decode warm and on the unpaged (consecutive-block) layout")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        case = make_workload(args.workload)
        total = args.steps + args.warmup
        times, step, cores = time_oracle(case, budget_s=min(150.0, 2.0 * total), steps=total)
        timed = times[args.warmup:]
        sec = sum(timed) / len(timed)
        value = step.bytes() / sec / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16" if case.dtype == "bf16" else "f32",
                "data": "synthetic", "config": config_for(case, args.workload),
                "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                                 "kind": "oracle",
                                 "sample": "per step: cache write of the new tokens and binary64 "
                                           "decode of the first %d of %d sequences (%d bytes)"
                                           % (step.n, case.num_seqs, step.bytes())},
                "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch

    import paged_kv_cache_78_gb300 as pa

    if world > 1:
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local_rank)
    r = run_gpu(args, rank, world, device)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return

    case, st, nbytes = r["case"], r["step"], r["bytes"]
    step_s = r["step_ms"] / 1e3
    value = world * nbytes["step"] / step_s / 1e9
    decode_gbs = nbytes["decode"] / (r["decode_ms"] / 1e3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    e2e = None
    if r["e2e_ms"] is not None:
        e2e = {"value": round(world * nbytes["step"] / (r["e2e_ms"] / 1e3) / 1e9, 2),
               "unit": "GB/s", "us_per_step": round(r["e2e_ms"] * 1e3, 2),
               "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
               "cuda_graph": bool(args.graph),
               "transfers": ("pa_copy_bytes kernels" if args.e2e_copy == "kernel"
                             else "copy engine")}

    cpu = None
    if args.cpu_budget > 0:
        def oracle_leg(threads):
            times, ostep, cores = time_oracle(case, budget_s=args.cpu_budget, threads=threads)
            sec = statistics.median(times)
            return {"value": round(ostep.bytes() / sec / 1e9, 4), "unit": "GB/s", "cores": cores,
                    "kind": "oracle",
                    "sample": "cache write of the new tokens and binary64 decode of the first %d "
                              "of %d sequences, median of %d runs in %.0f s"
                              % (ostep.n, case.num_seqs, len(times), sum(times)),
                    "ms_per_step": round(sec * 1e3, 2)}

        # All of the host's cores (the oracle's OpenMP loop over sequences and
        # query heads), then one core.
        cpu = oracle_leg(0)
        cpu["single_core"] = oracle_leg(1)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(r["step_ms"], 5),
        "us_per_step": round(r["step_ms"] * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if case.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": config_for(case, args.workload, st.partition),
        "run": {"partition_size": st.partition, "cuda_graph": bool(args.graph),
                "step_calls": ("pa_decode_shared (new tokens written by the decode)"
                               if st.plan is not None and args.fused else
                               "pa_reshape_and_cache + pa_decode_shared" if st.plan is not None
                               else "pa_decode_append" if args.fused else
                               "pa_reshape_and_cache + pa_decode"),
                "shared_plan": None if st.plan is None else {
                    "chunks": st.plan.num_chunks, "members": st.plan.info.num_members,
                    "min_shared_tokens": st.plan.info.min_shared_tokens,
                    "ranges": shared_ranges(case, st.plan, sms_of(torch, st.device))},
                "decode_kernel": {0: "auto", 1: "cuda cores", 2: "tensor cores"}[args.kernel] +
                                 " -> " + st.kernel_name,
                "decode_bytes": nbytes["decode"],
                "kv_bytes_logical": nbytes["logical_kv"],
                "kv_bytes_unique": nbytes["unique_kv"],
                "parallelism": "replicas" if world > 1 else "single GPU"},
        "gpu_launches": (st.launches - (1 if args.fused else 0)) * args.steps,
        "roofline": {
            "kernel": "%s (%s%s)" % ("pa_decode_shared" if st.plan is not None else "pa_decode",
                                     st.kernel_name,
                                     " + the log-sum-exp reduce"
                                     if st.partition or (st.plan is not None and
                                                         st.plan.num_chunks) else ""),
            "timed": "the decode call alone, %d launches after the timed steps, L2 evicted "
                     "before each" % args.steps,
            "bound": "hbm",
            "achieved": round(decode_gbs, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(decode_gbs / peak, 4),
            "us_per_launch": round(r["decode_ms"] * 1e3, 2),
            "traffic": ncu_traffic(args.workload + ("_shared" if st.plan is not None else ""),
                                   st.partition),
        },
        "e2e": e2e,
        "spread": r["spread"],
        "paging": r["paging"],
        "memory": memory_report(pa, case, args.workload),
        "clocks": r["clocks"],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
