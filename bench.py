#!/usr/bin/env python
"""Benchmark of the paged decode hot path on GB300.

One step = one decode step of the whole hot path over one batch: the work
list is planned once from the context lengths, then for every layer one fused
launch stores the batch's new K/V rows in their paged slots and runs paged
decode attention over the block tables (copy-on-write block copies are part of
the path but the default workload never forks, so none are due).

Default workload: 7B-shaped MHA decode -- batch 64, 32 query / 32 KV heads,
head_dim 128, fp16, block size 16, context lengths log-uniform in [16, 2048],
block tables as random disjoint draws from a pool of the needed blocks + 10 %,
32 layers with separate caches (timed as 32 fused append + attention
launches).  ``--workload gqa_8b`` runs the 8B-shaped GQA batch (128 sequences,
32 / 8 heads, bf16, lengths log-uniform in [128, 8192] plus 4 x 8192, one layer).
Other workloads: ``prefill_8b`` (chunked prefill), ``prefix_8b`` [``--cascade``]
(shared-prefix batch), ``sampling_8b`` (decode of 128 branches forked 4 ways
from 32 prompts), ``block_copy_8b`` (copy-on-write at a 4-way fork),
``swap_8b`` (device <-> host block swap) and ``pool_churn`` (host pool).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle (the
reference arm of this method: there is no other implementation) on bounded
samples of the same workload.
"""

from __future__ import annotations

import os

# The oracle baseline is timed single-threaded; pin BLAS before numpy loads.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from pagedattention_decode_attention_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attention tokens/s and KV-read GB/s (% of GB300 HBM peak), 1 GPU"
DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
ELEM = {"f16": 2, "bf16": 2, "f32": 4}
L2_BYTES = 126 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload",
                    choices=["mha_7b", "gqa_8b", "prefix_8b", "sampling_8b", "prefill_8b",
                             "swap_8b", "block_copy_8b", "pool_churn"],
                    default="mha_7b")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="override the workload's layer count (profiling at a small footprint)")
    ap.add_argument("--warmup-seconds", type=float, default=1.0,
                    help="keep warming up until this much wall time has passed")
    ap.add_argument("--no-secondary", action="store_true",
                    help="default workload only: skip the other configurations' lines")
    ap.add_argument("--cascade", action="store_true",
                    help="prefix_8b / sampling_8b: time the (grouped) shared-prefix decode "
                         "against the plain one")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def make_batch(name: str, rank: int, model_pool: bool = False) -> wl.DecodeBatch:
    """The workload's batch; each rank decodes its own independent batch
    (replicas; no exchange).  Tables of pool-built batches come from the
    native pool, or with ``model_pool`` from the oracle's model of it (the
    reference arm runs nothing of this library)."""
    if name == "mha_7b":
        return wl.mha_7b(seed=wl.SEED_BASE + 2 + 100 * rank)
    if name == "prefill_8b":
        return wl.prefill_8b(seed=wl.SEED_BASE + 6 + 100 * rank)
    if name == "prefix_8b":
        return prefix_batch(wl.prefix_mix(seed=wl.SEED_BASE + 5 + 100 * rank), model_pool)
    if name == "sampling_8b":
        return sampling_batch(wl.sampling_cow(seed=wl.SEED_BASE + 4 + 100 * rank), model_pool)
    return wl.gqa_8b(seed=wl.SEED_BASE + 3 + 100 * rank)


def make_pool(script, model_pool: bool):
    if model_pool:
        from oracle.pool import BlockPool as ModelPool
        return ModelPool(script.num_blocks, 16, script.initial_order)
    import pagedattention_decode_attention_gb300 as pa
    return pa.BlockPool(script.num_blocks, 16, script.initial_order)


def pool_tables(pool, seqs):
    """Block tables (int32, -1 padded to the longest) and context lengths."""
    rows = [pool.block_table(s) for s in seqs]
    tab = np.full((len(rows), max(len(t) for t, _ in rows)), -1, dtype=np.int32)
    for i, (t, _) in enumerate(rows):
        tab[i, :len(t)] = t
    return tab, np.array([c for _, c in rows], dtype=np.int32)


def sampling_batch(script, model_pool: bool = False) -> wl.DecodeBatch:
    """Parallel sampling after the divergence: the branches of every prompt,
    sharing all of their prompt's blocks but the last (each branch's own
    copy, or the block its last holder kept).  Eight layer caches rotate so
    a step reads about 1.1 GB of distinct K/V (one layer's 138 MB would
    nearly fit in L2)."""
    pool = make_pool(script, model_pool)
    branches, _ = cow_divergence(pool, script)
    tables, lens = pool_tables(pool, branches)
    # each prompt's branches are one group: contiguous, sharing the prompt's
    # whole blocks (the leading table entries all members agree on)
    starts = np.arange(0, len(branches) + 1, script.branches, dtype=np.int32)
    shared = []
    for a, b in zip(starts[:-1], starts[1:]):
        rows = tables[a:b]
        n = 0
        while n < rows.shape[1] and rows[0, n] >= 0 and (rows[:, n] == rows[0, n]).all():
            n += 1
        shared.append(n)
    return wl.DecodeBatch("sampling_8b_bf16", 32, 8, 128, "bf16", lens, tables, script.num_blocks,
                          num_layers=8, seed=script.seed,
                          extra={"group_start": starts,
                                 "group_blocks": np.array(shared, dtype=np.int32)})


def prefix_batch(script, model_pool: bool = False) -> wl.DecodeBatch:
    """The prefix-mix decode batch, tables from the pool: one pinned prefix
    sequence, then every request shares its blocks and appends its own
    suffix (the request's newest token last)."""
    pool = make_pool(script, model_pool)
    root = pool.new_seq()
    for _ in range(script.prefix_len):
        pool.append_slot(root)
    pool.pin(root, script.prefix_len)
    seqs = []
    for n in script.suffix_lens:
        s = pool.new_seq()
        pool.share_prefix(root, s, script.prefix_len)
        for _ in range(int(n)):
            pool.append_slot(s)
        seqs.append(s)
    tables, lens = pool_tables(pool, seqs)
    return wl.DecodeBatch("prefix_8b_bf16", 32, 8, 128, "bf16", lens, tables, script.num_blocks,
                          num_layers=script.num_layers, seed=script.seed,
                          extra={"prefix_blocks": script.prefix_len // 16})


def unique_kv_bytes(batch: wl.DecodeBatch) -> int:
    """K/V bytes of one call counting every physical block once (the tokens of
    a block any sequence attends, at most 16)."""
    used = {}
    for b, ctx in enumerate(batch.context_lens):
        for j in range((int(ctx) + 15) // 16):
            blk = int(batch.block_tables[b, j])
            used[blk] = max(used.get(blk, 0), min(16, int(ctx) - 16 * j))
    return sum(used.values()) * 2 * batch.num_kv_heads * batch.head_dim * ELEM[batch.dtype]


def prefill_flops(batch: wl.DecodeBatch) -> float:
    """Flops of one chunked-prefill attention call: every query row (token x
    query head) does 2 d flops for q.k and 2 d for p.v per attended token, and
    the query at position p attends p + 1 tokens."""
    total = 0.0
    for ctx, qlen in zip(batch.context_lens.astype(np.int64), batch.extra["query_lens"]):
        first = ctx - int(qlen)
        attended = int(qlen) * (first + 1) + int(qlen) * (int(qlen) - 1) // 2
        total += attended
    return total * 4 * batch.head_dim * batch.num_q_heads


def run_prefill_bench(args):
    """Chunked-prefill attention: each step is one attention call (plan +
    kernel) over the batch's chunks, rotating over the layer caches."""
    import pagedattention_decode_attention_gb300 as pa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    batch = make_batch("prefill_8b", 0)
    if args.layers > 0:
        batch.num_layers = args.layers
    dt = DTYPES[batch.dtype]
    hq, hkv, d, nb, L = (batch.num_q_heads, batch.num_kv_heads, batch.head_dim, batch.num_blocks,
                         batch.num_layers)
    qlens = batch.extra["query_lens"]
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    total_q = int(qs[-1])
    s0 = batch.seed * 1000
    kc = [wl.normal((nb, hkv, 16, d), dt, s0 + 4 * i, device) for i in range(L)]
    vc = [wl.normal((nb, hkv, 16, d), dt, s0 + 4 * i + 1, device) for i in range(L)]
    q = wl.normal((L, total_q, hq, d), dt, s0 + 7, device)
    out = torch.empty_like(q)
    bt = torch.from_numpy(batch.block_tables).to(device)
    cl = torch.from_numpy(batch.context_lens).to(device)
    qs_d = torch.from_numpy(qs).to(device)
    ws = pa.alloc_prefill_workspace(batch.num_seqs, total_q, hq, hkv, d, device)

    def step():
        """One model step: the work list is planned once from the chunk
        lengths (the same in every layer), then each layer runs attention."""
        pa.prefill_plan(cl, qs_d, total_q, hq, hkv, d, batch.max_blocks, batch.scale, dt, ws)
        for layer in range(L):
            pa.paged_attention_prefill_run(q[layer], kc[layer], vc[layer], bt, cl, qs_d,
                                           batch.scale, ws, out=out[layer])

    # The chunk's own K/V rows, appended to their paged slots in every layer
    # before its attention (a model step does this; the attention-only pass
    # above it is the kernel's roofline).
    pos = np.concatenate([np.arange(c - n, c) for c, n in zip(batch.context_lens, qlens)])
    seq = np.repeat(np.arange(batch.num_seqs), qlens)
    slots = torch.from_numpy((batch.block_tables[seq, pos // 16].astype(np.int64) * 16
                              + pos % 16)).to(device)
    k_new = wl.normal((L, total_q, hkv, d), dt, s0 + 8, device)
    v_new = wl.normal((L, total_q, hkv, d), dt, s0 + 9, device)
    appends = [pa.prepare_kv_append(k_new[i], v_new[i], kc[i], vc[i], slots) for i in range(L)]

    def step_with_append():
        pa.prefill_plan(cl, qs_d, total_q, hq, hkv, d, batch.max_blocks, batch.scale, dt, ws)
        for layer in range(L):
            appends[layer]()
            pa.paged_attention_prefill_run(q[layer], kc[layer], vc[layer], bt, cl, qs_d,
                                           batch.scale, ws, out=out[layer])

    def timed(fn):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(args.steps):
            fn()
        end.record()
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3

    for _ in range(max(args.warmup, 3)):
        step()
        step_with_append()
    torch.cuda.synchronize()
    pa.check_status()
    clocks = ClockSampler(device)
    clocks.start()
    secs = timed(step)
    secs_append = timed(step_with_append)
    clk = clocks.stop()
    pa.check_status()
    per_call = secs / (args.steps * L)     # one layer's share of a step
    per_layer_append = secs_append / (args.steps * L)
    append_bytes = 2 * 2 * total_q * hkv * d * ELEM[batch.dtype] + total_q * 8
    flops = prefill_flops(batch)
    kv_bytes = int(batch.context_lens.astype(np.int64).sum()) * 2 * hkv * d * ELEM[batch.dtype]
    peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"]) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 1900.0
    line = {
        "metric": "paged chunked-prefill attention query tokens/s per layer, 1 GPU",
        "value": total_q / per_call, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": per_call * L * 1e3,
        "ms_per_layer": per_call * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": batch.dtype,
        "data": "synthetic (seeded N(0,1) Q/K/V, seeded lengths and placements)",
        "config": {"workload": batch.name, "num_seqs": batch.num_seqs,
                   "num_q_heads": hq, "num_kv_heads": hkv, "head_dim": d, "block_size": 16,
                   "query_tokens": total_q, "context_tokens": int(batch.context_lens.sum()),
                   "layers_rotated": L,
                   "step": "one model step: one plan, then one chunked-prefill attention "
                           "call per layer (value and roofline per layer)",
                   "l2": f"layers rotate: each layer's {kv_bytes / 1e6:.0f} MB of K/V "
                         f"comes from HBM ({L} layers > L2)"},
        "roofline": {"bound": "tensor", "achieved": flops / per_call / 1e12, "peak": peak,
                     "unit": "TFLOP/s", "frac": flops / per_call / 1e12 / peak,
                     "flops_per_launch": flops, "peak_source": "measured bf16_tflops (burst)",
                     "kv_read_gbs_unique": kv_bytes / per_call / 1e9},
        "with_append": {"ms_per_layer": per_layer_append * 1e3,
                        "tokens_per_s": total_q / per_layer_append,
                        "append_ms_per_layer": (per_layer_append - per_call) * 1e3,
                        "append_bytes": append_bytes,
                        "append_gbs": append_bytes / max(per_layer_append - per_call, 1e-9) / 1e9,
                        "step": "per layer: kv_append of the chunk's K/V, then attention"},
        "gpu_launches": (1 + L) * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_prefill_baseline(batch, args.cpu_seconds / 2)
    print(json.dumps(line))


def algorithmic_bytes(batch: wl.DecodeBatch) -> dict:
    """Bytes one fused append + attention call must move at minimum: the K and
    V rows of every attended token, the queries, the outputs, the used table
    entries, the context lengths, and the append (new K/V rows read, written
    to their slots, and the slots)."""
    e = ELEM[batch.dtype]
    toks = int(batch.context_lens.astype(np.int64).sum())
    kv = toks * 2 * batch.num_kv_heads * batch.head_dim * e
    qo = 2 * batch.num_seqs * batch.num_q_heads * batch.head_dim * e
    tables = int(wl.num_blocks_for(batch.context_lens).sum()) * 4 + batch.num_seqs * 4
    append = 2 * 2 * batch.num_seqs * batch.num_kv_heads * batch.head_dim * e + batch.num_seqs * 8
    return {"kv": kv, "total": kv + qo + tables + append, "tokens": toks}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "pagedattention_decode_attention_gb300", "csrc")
    for name in ("decode.cu", "decode.cuh", "device_common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def copy_kernel_source_hash() -> str:
    h = hashlib.sha256()
    with open(os.path.join(ROOT, "pagedattention_decode_attention_gb300", "csrc",
                           "copy_kernels.cu"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "dram_traffic.json")


def _recorded_traffic(key: str, source_hash: str):
    """DRAM bytes per launch (``dram__bytes_read.sum + dram__bytes_write.sum``)
    of one kernel on one workload from the committed ncu record, if it was
    taken on the current kernel source (else None)."""
    if not os.path.exists(TRAFFIC_RECORD):
        return None
    with open(TRAFFIC_RECORD) as f:
        rec = json.load(f).get(key)
    if not rec or rec.get("kernel_source_sha256_16") != source_hash:
        return None
    return float(rec["dram_bytes_per_launch"])


def profiled_copy_traffic():
    """Steady-state DRAM bytes per block_copy launch of the block_copy_8b
    workload (current kernel source only)."""
    return _recorded_traffic("block_copy_8b", copy_kernel_source_hash())


def profiled_traffic(workload: str):
    """DRAM bytes per attention launch of a decode workload (current kernel
    source only)."""
    return _recorded_traffic(f"decode_{workload}", kernel_source_hash())


def profiled_cascade_traffic(workload: str, grouped: bool):
    """DRAM bytes per layer's attention launch of the grouped decode on a
    cascade workload (current kernel source only; None for the three-phase
    path, whose layer is three launches)."""
    if not grouped or os.environ.get("PA_CASCADE", "") == "phases":
        return None
    return _recorded_traffic(f"grouped_decode_{workload}", kernel_source_hash())


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled during the timed
    region, read through NVML (ctypes on libnvidia-ml; reading only).  Falls
    back to ``nvidia-smi`` polling when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: torch.device, period_s: float = 0.002):
        self.device = device
        self.period = period_s
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self._nvml = None
        self._handle = None
        self._smi = None
        self._open()

    def _open(self):
        import ctypes as C
        try:
            nvml = C.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            handle = C.c_void_p()
            props = torch.cuda.get_device_properties(self.device)
            bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0),
                                        getattr(props, "pci_bus_id", 0),
                                        getattr(props, "pci_device_id", 0))
            if nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), C.byref(handle)) != 0:
                if nvml.nvmlDeviceGetHandleByIndex_v2(self.device.index or 0, C.byref(handle)) != 0:
                    return
            mx = C.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(handle, 1, C.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._nvml, self._handle = nvml, handle
        except OSError:
            self._nvml = None

    def _poll(self):
        import ctypes as C
        clk, rs = C.c_uint(), C.c_ulonglong()
        getr = getattr(self._nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, C.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if getr(self._handle, C.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            self._stop.wait(self.period)

    def start(self):
        import threading
        if self._nvml is not None:
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            return
        try:
            self._smi = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index or 0),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self._smi = None

    def stop(self) -> dict:
        source = "nvml"
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        elif self._smi is not None:
            source = "nvidia-smi"
            self._smi.terminate()
            out, _ = self._smi.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except (ValueError, IndexError):
                    continue
                for name, val in zip(names, f[2:6]):
                    if val.lower() == "active":
                        self.reasons.add(name)
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"], "samples": 0}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": source}


# --------------------------------------------------------------------- ours
class Replica:
    """Device-resident inputs of one decode step of the workload."""

    def __init__(self, batch: wl.DecodeBatch, device):
        import pagedattention_decode_attention_gb300 as pa
        self.pa = pa
        self.batch = batch
        self.device = device
        dt = DTYPES[batch.dtype]
        b, hq, hkv, d, nb = (batch.num_seqs, batch.num_q_heads, batch.num_kv_heads,
                             batch.head_dim, batch.num_blocks)
        L = batch.num_layers
        s = batch.seed * 1000
        self.k_cache = [wl.normal((nb, hkv, 16, d), dt, s + 4 * i, device) for i in range(L)]
        self.v_cache = [wl.normal((nb, hkv, 16, d), dt, s + 4 * i + 1, device) for i in range(L)]
        self.q = wl.normal((L, b, hq, d), dt, s + 7, device)
        self.k_new = wl.normal((L, b, hkv, d), dt, s + 8, device)
        self.v_new = wl.normal((L, b, hkv, d), dt, s + 9, device)
        self.out = torch.empty((L, b, hq, d), dtype=dt, device=device)
        self.tables = torch.from_numpy(batch.block_tables).to(device)
        self.lens = torch.from_numpy(batch.context_lens).to(device)
        self.slots = torch.from_numpy(batch.new_token_slots()).to(device)
        self.ws = pa.alloc_workspace(b, hq, hkv, d, batch.max_blocks, device)
        self.scale = batch.scale
        self.launches_per_step = 1 + L   # one plan, then one fused launch per layer
        self.plan_call, self.layer_calls = self.bind(self.inputs())

    # the per-step inputs and the output of a step (the caches and the
    # workspace are the replica's own)
    INPUT_NAMES = ("q", "k_new", "v_new", "tables", "lens", "slots")

    def inputs(self) -> dict:
        return {n: getattr(self, n) for n in self.INPUT_NAMES + ("out",)}

    def spare_inputs(self) -> dict:
        """A second set of step buffers on the device (for double buffering)."""
        return {n: torch.empty_like(t) for n, t in self.inputs().items()}

    def bind(self, io: dict):
        """Calls bound to one set of step buffers (validated once; each step
        only re-issues the C calls)."""
        pa, batch = self.pa, self.batch
        hq, hkv, d = batch.num_q_heads, batch.num_kv_heads, batch.head_dim
        plan = pa.prepare_decode_plan(io["lens"], hq, hkv, d, batch.max_blocks, self.ws)
        layers = [pa.prepare_decode_append_run(
            io["q"][i], io["k_new"][i], io["v_new"][i], io["slots"], self.k_cache[i],
            self.v_cache[i], io["tables"], io["lens"], self.scale, self.ws, io["out"][i])
            for i in range(batch.num_layers)]
        return plan, layers

    def step(self, ev=None):
        """One decode step: the work list is planned once from the context
        lengths (the same for every layer), then each layer appends its new
        K/V rows and runs attention over them, in one launch."""
        self.plan_call()
        for layer in range(self.batch.num_layers):
            if ev is not None:
                ev[layer][0].record()
            self.layer_calls[layer]()
            if ev is not None:
                ev[layer][1].record()

    def kernel_only_ms(self, reps: int = 64) -> float:
        """Mean device time of back-to-back layer-0 launches (no host gaps and
        nothing else between them): a check on the timed-region figure."""
        self.plan_call()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.layer_calls[0]()
        start.record()
        for _ in range(reps):
            self.layer_calls[0]()
        end.record()
        torch.cuda.synchronize()
        return start.elapsed_time(end) / reps


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest x over the ranks (the slowest rank's time).  NCCL reduces a
    device tensor; any other backend (gloo, in the CPU tests) a host one."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank_step: int, world: int, steps: int, secs: float) -> float:
    """Whole-job tokens/s: every rank decodes its own batch each step, and
    the job takes as long as its slowest rank (``secs``, max over ranks)."""
    return tokens_per_rank_step * world * steps / secs


def time_steps(rep: Replica, steps: int, world: int, events: bool):
    """Times `steps` steps between two barriers; returns (seconds, per-launch
    attention durations in ms)."""
    L = rep.batch.num_layers
    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
           for _ in range(L)] for _ in range(steps)] if events else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record()
    for i in range(steps):
        rep.step(ev[i] if ev else None)
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    secs = start.elapsed_time(end) / 1e3
    per = [a.elapsed_time(b) for step_ev in ev for a, b in step_ev] if ev else []
    return secs, per


def time_e2e(rep: Replica, steps: int, world: int):
    """Same steps, end to end: every step's inputs (q, new K/V rows, tables,
    lengths, slots) are copied in from pinned host memory and its outputs read
    back to pinned host memory, inside the timed region.  Two sets of step
    buffers and two copy streams pipeline it: step i+1's inputs load and step
    i-1's outputs drain while step i's kernels run."""
    dev = rep.device
    host_in = {n: t.cpu().pin_memory() for n, t in rep.inputs().items() if n != "out"}
    host_out = [torch.empty(rep.out.shape, dtype=rep.out.dtype).pin_memory() for _ in range(2)]
    sets = [rep.inputs(), rep.spare_inputs()]
    calls = [(rep.plan_call, rep.layer_calls), rep.bind(sets[1])]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    main = torch.cuda.current_stream(dev)
    load_s, drain_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    loaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def load(i):
        j = i % 2
        with torch.cuda.stream(load_s):
            if i >= 2:
                load_s.wait_event(computed[j])    # step i-2 no longer reads set j
            for n, t in host_in.items():
                sets[j][n].copy_(t, non_blocking=True)
            loaded[j].record(load_s)

    barrier(world)
    torch.cuda.synchronize()
    start.record(main)
    load(0)
    for i in range(steps):
        j = i % 2
        if i + 1 < steps:
            load(i + 1)
        main.wait_event(loaded[j])
        if i >= 2:
            main.wait_event(drained[j])           # step i-2's outputs have been read back
        plan, layers = calls[j]
        plan()
        for call in layers:
            call()
        computed[j].record(main)
        with torch.cuda.stream(drain_s):
            drain_s.wait_event(computed[j])
            host_out[j].copy_(sets[j]["out"], non_blocking=True)
            drained[j].record(drain_s)
    main.wait_stream(drain_s)
    end.record(main)
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(end) / 1e3, h2d, d2h


class OracleInputs:
    """Host float32 copies of layer 0 of the workload for the oracle: from the
    device replica when there is one, else drawn on the host."""

    def __init__(self, batch: wl.DecodeBatch, rep: "Replica | None"):
        if rep is not None:
            self.kc = rep.k_cache[0].float().cpu().numpy()
            self.vc = rep.v_cache[0].float().cpu().numpy()
            self.q = rep.q[0].float().cpu().numpy()
        else:
            shape = (batch.num_blocks, batch.num_kv_heads, 16, batch.head_dim)
            gen = np.random.default_rng(batch.seed)
            self.kc = gen.standard_normal(shape, dtype=np.float32)
            self.vc = gen.standard_normal(shape, dtype=np.float32)
            self.q = gen.standard_normal((batch.num_seqs, batch.num_q_heads, batch.head_dim),
                                         dtype=np.float32)
        self.order = np.random.default_rng(7).permutation(batch.num_seqs)
        self.next = 0


def cpu_oracle_sample(batch: wl.DecodeBatch, inp: OracleInputs, seconds: float, step_units=None):
    """Times the oracle on (sequence, layer) units of the workload.  A unit is one
    sequence's attention over all query heads for one layer; ``num_layers``
    units make one decoded token.  Returns (tokens/s, units, elapsed s)."""
    import oracle.attention as oa
    units, t0 = 0, time.perf_counter()
    while True:
        b = int(inp.order[inp.next % batch.num_seqs])
        inp.next += 1
        oa.paged_attention_decode(inp.q, inp.kc, inp.vc, batch.block_tables, batch.context_lens,
                                  batch.scale, seqs=[b])
        units += 1
        el = time.perf_counter() - t0
        if (step_units is not None and units >= step_units) or (step_units is None and el >= seconds):
            break
    return units / batch.num_layers / el, units, el


# ---- the oracle on every host core: worker processes (started with spawn,
# never forked after CUDA is initialised) each time the oracle on their own
# (sequence, layer) units for the same wall time; layer 0's caches reach them
# through a memory-mapped file.
_CPU_STATE = None


def _cpu_worker_init(path, shapes, tables, lens, scale):
    global _CPU_STATE
    mm = np.memmap(path, dtype=np.float32, mode="r")
    parts, at = [], 0
    for shape in shapes:
        n = int(np.prod(shape))
        parts.append(np.asarray(mm[at:at + n]).reshape(shape))
        at += n
    _CPU_STATE = (parts[0], parts[1], parts[2], tables, lens, scale)


def _cpu_worker_run(arg):
    import oracle.attention as oa
    seconds, seed = arg
    kc, vc, q, tables, lens, scale = _CPU_STATE
    order = np.random.default_rng(seed).permutation(len(lens))
    units, t0 = 0, time.perf_counter()
    while True:
        b = int(order[units % len(order)])
        oa.paged_attention_decode(q, kc, vc, tables, lens, scale, seqs=[b])
        units += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return units, el


def cpu_oracle_all_cores(batch: wl.DecodeBatch, inp: OracleInputs, seconds: float):
    """The oracle on every host core at once (one process per core, each
    single-threaded).  Returns (tokens/s, units, elapsed s, cores)."""
    import multiprocessing as mp
    import tempfile
    from concurrent.futures import ProcessPoolExecutor
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    arrays = [np.ascontiguousarray(a, dtype=np.float32) for a in (inp.kc, inp.vc, inp.q)]
    fd, path = tempfile.mkstemp(prefix="pa_oracle_", suffix=".f32")
    os.close(fd)
    try:
        total = sum(a.size for a in arrays)
        mm = np.memmap(path, dtype=np.float32, mode="w+", shape=(total,))
        at = 0
        for a in arrays:
            mm[at:at + a.size] = a.ravel()
            at += a.size
        mm.flush()
        del mm
        # an executor (not a Pool): a worker that dies raises instead of being
        # replaced forever
        with ProcessPoolExecutor(cores, mp_context=mp.get_context("spawn"),
                                 initializer=_cpu_worker_init,
                                 initargs=(path, [a.shape for a in arrays], batch.block_tables,
                                           batch.context_lens, batch.scale)) as pool:
            res = list(pool.map(_cpu_worker_run, [(seconds, 7 + i) for i in range(cores)],
                                timeout=seconds + 300))
    finally:
        os.unlink(path)
    units = sum(r[0] for r in res)
    el = max(r[1] for r in res)
    return units / batch.num_layers / el, units, el, cores


def decode_config(batch: wl.DecodeBatch, world: int) -> dict:
    """The ``config`` of a decode line; the reference arm prints the same."""
    ab = algorithmic_bytes(batch)
    return {
        "workload": batch.name, "num_seqs": batch.num_seqs,
        "num_q_heads": batch.num_q_heads, "num_kv_heads": batch.num_kv_heads,
        "head_dim": batch.head_dim, "block_size": 16, "layers": batch.num_layers,
        "context_tokens": ab["tokens"], "num_blocks_per_layer": batch.num_blocks,
        "l2": (f"inputs larger than L2: {ab['kv'] * batch.num_layers / 1e9:.2f} GB of KV "
               f"read per step across {batch.num_layers} separate layer caches"),
        "step": ("plan the work list once from the context lengths, then per layer one "
                 "launch: kv_append of the new K/V rows fused with paged decode "
                 "attention"),
        "parallelism": f"replicas x{world} (independent batches, no collective)",
    }


def warm_up(step, requested: int, seconds: float, sync_every: int = 8) -> int:
    """At least max(requested, 3) steps and at least ``seconds`` of wall time,
    so the clocks have ramped; returns the steps run."""
    warm, t0 = 0, time.perf_counter()
    while warm < max(requested, 3) or time.perf_counter() - t0 < seconds:
        step()
        warm += 1
        if warm % sync_every == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return warm


def measure_decode(args, batch: wl.DecodeBatch, device, world: int, rank: int,
                   cpu_seconds: float, all_cores: bool) -> dict:
    """One decode workload measured the bench's way; returns its JSON line
    (rank 0) or None."""
    rep = Replica(batch, device)
    warm = warm_up(rep.step, args.warmup, args.warmup_seconds)
    rep.pa.check_status()

    clocks = ClockSampler(device)
    clocks.start()
    h0 = time.perf_counter()
    # The step throughput is timed with nothing between the kernels: an event
    # recorded between two launches would end the programmatic-launch overlap
    # of the next kernel's start with the previous one's end.
    secs, _ = time_steps(rep, args.steps, world, events=False)
    host_secs = time.perf_counter() - h0
    # For comparison only: the same steps again with an event pair around every
    # attention launch (an overestimate: each launch then waits for the event
    # before it and loses its overlap with the previous kernel).
    _, per_launch = time_steps(rep, args.steps, world, events=True)
    clk = clocks.stop()
    rep.pa.check_status()
    kernel_ms = rep.kernel_only_ms()
    secs = max_over_ranks(secs, world)
    tokens_per_step = batch.num_seqs * world
    value = weak_scaling_value(batch.num_seqs, world, args.steps, secs)

    ab = algorithmic_bytes(batch)
    # Average attention launch duration over the timed region: its event-timed
    # length over the attention launches in it (the one plan launch per step is
    # counted against the attention, so this slightly overstates it).
    avg_ms = secs * 1e3 / (args.steps * batch.num_layers)
    events_ms = statistics.mean(per_launch)
    achieved = ab["total"] / (avg_ms / 1e3) / 1e9
    peak, peak_kind = load_peaks()
    workload = next((k for k in ("mha_7b", "gqa_8b") if batch.name.startswith(k)), batch.name)
    traffic = profiled_traffic(workload)

    e2e = None
    if not args.no_e2e:
        for _ in range(2):
            rep.step()
        e_secs, h2d, d2h = time_e2e(rep, args.steps, world)
        e_secs = max_over_ranks(e_secs, world)
        e2e = {"value": tokens_per_step * args.steps / e_secs, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelining": ("two sets of step buffers: step i+1's host-to-device copies and "
                              "step i-1's device-to-host copies overlap step i's kernels")}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp = OracleInputs(batch, rep)
        v1, units1, el1 = cpu_oracle_sample(batch, inp, cpu_seconds)
        one = {"value": v1, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": (f"{units1} (sequence, layer) attention units of layer 0, all "
                          f"{batch.num_q_heads} query heads each, float64 numpy on 1 host "
                          f"thread in {el1:.1f} s; {batch.num_layers} units = 1 token")}
        cpu = one
        if all_cores:
            try:
                vn, unitsn, eln, cores = cpu_oracle_all_cores(batch, inp, cpu_seconds)
                cpu = {"value": vn, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                       "sample": (f"{unitsn} (sequence, layer) attention units of layer 0 on "
                                  f"{cores} single-threaded processes (one per host core) in "
                                  f"{eln:.1f} s; {batch.num_layers} units = 1 token"),
                       "one_thread": one}
            except Exception as exc:  # noqa: BLE001  (no room for the inputs, a worker died, timeout)
                cpu = dict(one, all_cores_unavailable=str(exc)[:200])
        del inp

    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "warmup_steps_run": warm,
            "warmup_rule": (f"at least max(--warmup, 3) steps and at least "
                            f"{args.warmup_seconds:g} s of wall time (clock ramp)"),
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": batch.dtype,
            "data": "synthetic (seeded N(0,1) K/V/Q, seeded lengths and placements)",
            "config": decode_config(batch, world),
            "kv_read_gbs": ab["kv"] / (avg_ms / 1e3) / 1e9,
            "kv_read_gbs_unique": unique_kv_bytes(batch) / (avg_ms / 1e3) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "frac_of_nominal_7900": achieved / 7900.0,
                         "kernel": ("paged_attention_decode_append_run (persistent fused "
                                    "append + attention kernel)"),
                         "algorithmic_bytes_per_launch": ab["total"],
                         "avg_launch_ms": avg_ms, "back_to_back_launch_ms": kernel_ms,
                         "events_around_each_launch_ms": events_ms,
                         # per-launch event times over every timed launch (at
                         # least 20): median and best, and their GB/s
                         "events_launches": len(per_launch),
                         "events_median_ms": statistics.median(per_launch),
                         "events_best_ms": min(per_launch),
                         "events_median_gbs": ab["total"] / (statistics.median(per_launch) / 1e3) / 1e9,
                         "events_best_gbs": ab["total"] / (min(per_launch) / 1e3) / 1e9,
                         "launch_timing": ("timed region / attention launches in it (plan "
                                           "included); events_around_each_launch_ms from a "
                                           "second pass with an event pair per launch")},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": rep.launches_per_step * args.steps,
            "host_ms_per_step": host_secs / args.steps * 1e3,
            "clocks": clk,
        }
    del rep
    torch.cuda.empty_cache()
    return line


def run_ours(args):
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    batch = make_batch(args.workload, rank)
    if args.layers > 0:
        batch.num_layers = args.layers
    line = measure_decode(args, batch, device, world, rank, args.cpu_seconds, all_cores=True)
    if (line is not None and world == 1 and args.workload == "mha_7b" and args.layers == 0
            and not args.no_secondary):
        # the other configurations, each timed the same way in the same run
        sec_cpu = min(args.cpu_seconds, 3.0)
        line["secondary"] = {
            "gqa_8b": measure_decode(args, make_batch("gqa_8b", 0), device, 1, 0, sec_cpu,
                                     all_cores=False),
            "sampling_8b_grouped_cascade": measure_cascade(args, "sampling_8b", device, sec_cpu),
            "prefix_8b_cascade": measure_cascade(args, "prefix_8b", device, sec_cpu),
        }
    if line is not None:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference
def cascade_config(batch: wl.DecodeBatch) -> dict:
    """The ``config`` of a cascade line; the reference arm prints the same."""
    grouped = "group_start" in batch.extra
    return {"workload": batch.name, "num_seqs": batch.num_seqs, "layers": batch.num_layers,
            "prefix_blocks": (int(batch.extra["group_blocks"].min()) if grouped
                              else batch.extra["prefix_blocks"]),
            "context_tokens": int(batch.context_lens.sum()),
            "groups": len(batch.extra["group_start"]) - 1 if grouped else 1,
            "step": "one plan, then per layer: append the new tokens' K/V and attend"}


def run_cascade_bench(args):
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    print(json.dumps(measure_cascade(args, args.workload, device, args.cpu_seconds / 2,
                                     layers=args.layers)))


def cascade_launches_per_step(grouped: bool, layers: int) -> int:
    """Kernel launches of one cascade step: the grouped decode (the default
    for groups, or PA_CASCADE=grouped) is one plan, then one attention launch
    per layer; the three phases are two or three plans (the suffix tables of
    groups, the prefix phase's plan, the suffix decode's plan), then per
    layer the prefix phase, the suffix decode and the combine."""
    impl = os.environ.get("PA_CASCADE", "")
    if impl == "grouped" or (grouped and impl != "phases"):
        return 1 + layers
    return (3 if grouped else 2) + 3 * layers


def measure_cascade(args, workload: str, device, cpu_seconds: float, layers: int = 0) -> dict:
    """Shared-prefix (cascade) decode beside the plain decode of the same
    batch: the prefix-mix batch (one prefix for the whole batch) or the
    parallel-sampling batch (grouped: each prompt's branches share their
    prompt).  Both run as a model step would: one plan, then per layer the
    new tokens' K/V appended and attention over the whole context (the plain
    path in one launch; the grouped cascade in one launch too, over units
    that read a group's shared blocks once for its members; the single-prefix
    cascade as its prefix phase, the suffix decode that also stores the new
    rows, and the combine)."""
    import pagedattention_decode_attention_gb300 as pa
    batch = make_batch(workload, 0)
    if layers > 0:
        batch.num_layers = layers
    rep = Replica(batch, device)
    grouped = "group_start" in batch.extra
    L = batch.num_layers
    hq, hkv, d, mb = batch.num_q_heads, batch.num_kv_heads, batch.head_dim, batch.max_blocks
    dt = DTYPES[batch.dtype]
    size = (pa.grouped_prefix_workspace_size if grouped else pa.shared_prefix_workspace_size)(
        batch.num_seqs, hq, hkv, d, mb)
    ws = torch.empty(max(size, 256), dtype=torch.uint8, device=device)
    if grouped:
        gs = torch.from_numpy(batch.extra["group_start"]).to(device)
        gb = torch.from_numpy(batch.extra["group_blocks"]).to(device)
        P = int(batch.extra["group_blocks"].min())

        def cascade_step():
            pa.grouped_prefix_plan(rep.tables, rep.lens, gs, gb, hq, hkv, d, batch.scale, dt, ws)
            for i in range(L):
                pa.paged_attention_decode_grouped_prefix_append_run(
                    rep.q[i], rep.k_new[i], rep.v_new[i], rep.slots, rep.k_cache[i],
                    rep.v_cache[i], rep.tables, gs, gb, batch.scale, ws, out=rep.out[i])
    else:
        P = batch.extra["prefix_blocks"]

        def cascade_step():
            pa.shared_prefix_plan(rep.lens, P, hq, hkv, d, mb, batch.scale, dt, ws)
            for i in range(L):
                pa.paged_attention_decode_shared_prefix_append_run(
                    rep.q[i], rep.k_new[i], rep.v_new[i], rep.slots, rep.k_cache[i],
                    rep.v_cache[i], rep.tables, rep.lens, P, batch.scale, ws, out=rep.out[i])

    warm = []

    def timed(step):
        warm.append(warm_up(step, args.warmup, args.warmup_seconds))
        pa.check_status()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(args.steps):
            step()
        end.record()
        torch.cuda.synchronize()
        pa.check_status()
        return start.elapsed_time(end) / 1e3 / args.steps

    clocks = ClockSampler(device)
    clocks.start()
    plain_s = timed(rep.step)
    plain_out = rep.out.clone()
    cascade_s = timed(cascade_step)
    clk = clocks.stop()
    # the same attention either way (within rounding of the two merges)
    diff = (plain_out.float() - rep.out.float()).abs().max().item()
    peak, peak_src = load_peaks()
    qo = 2 * batch.num_seqs * hq * d * ELEM[batch.dtype]
    uniq = unique_kv_bytes(batch) + qo
    line = {
        "metric": ("decode tokens/s, grouped shared-prefix (cascade) path, 1 GPU" if grouped
                   else "decode tokens/s, shared-prefix (cascade) path, 1 GPU"),
        "value": batch.num_seqs / cascade_s, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "warmup_steps_run": warm[-1],
        "ms_per_step": cascade_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": batch.dtype,
        "data": "synthetic (seeded N(0,1) Q/K/V; seeded lengths and pool tables)",
        "config": cascade_config(batch),
        "roofline": {"bound": "hbm", "achieved": uniq / (cascade_s / L) / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": uniq / (cascade_s / L) / 1e9 / peak,
                     "traffic": profiled_cascade_traffic(workload, grouped),
                     "peak_source": f"{peak_src} hbm_gbs",
                     "bytes_per_layer": uniq,
                     "bytes": "unique K/V (each physical block once: the prefix once, "
                              "every suffix once), q, out"},
        "cascade_us_per_layer": cascade_s / L * 1e6,
        "plain_us_per_layer": plain_s / L * 1e6,
        "plain_value": batch.num_seqs / plain_s,
        "max_abs_diff_vs_plain": diff,
        "gpu_launches": args.steps * cascade_launches_per_step(grouped, L),
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        # the oracle computes the same attention (the cascade is exact)
        v, units, _ = cpu_oracle_sample(batch, OracleInputs(batch, rep), cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": (f"{units} (sequence, layer) units of layer 0, float64 "
                                           f"numpy, 1 thread; {L} units = 1 token")}
    del rep, ws
    torch.cuda.empty_cache()
    return line


def run_swap_bench(args):
    """Block swap (preemption / offload): a batch of 1024 blocks of every one
    of 32 8B-shaped GQA layers goes to page-locked host memory and back, each
    direction one launch.  The roofline is a plain pinned copy of the same
    bytes in the same direction, measured in the same run."""
    import pagedattention_decode_attention_gb300 as pa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    layers = args.layers if args.layers > 0 else 32
    nb, nblk, hkv, d, dt = 2048, 1024, 8, 128, torch.bfloat16
    gen = np.random.default_rng(wl.SEED_BASE + 7)
    dk = [wl.normal((nb, hkv, 16, d), dt, 4000 + 2 * i, device) for i in range(layers)]
    dv = [wl.normal((nb, hkv, 16, d), dt, 4001 + 2 * i, device) for i in range(layers)]
    hk = [torch.empty((nblk, hkv, 16, d), dtype=dt).pin_memory() for _ in range(layers)]
    hv = [torch.empty((nblk, hkv, 16, d), dtype=dt).pin_memory() for _ in range(layers)]
    out_pairs = torch.from_numpy(np.stack([gen.choice(nb, nblk, replace=False),
                                           gen.permutation(nblk)], 1)).to(device)
    in_pairs = torch.from_numpy(np.stack([gen.permutation(nblk),
                                          gen.choice(nb, nblk, replace=False)], 1)).to(device)
    block_bytes = 2 * hkv * 16 * d * 2                     # K + V of one block of one layer
    moved = block_bytes * nblk * layers                    # payload of one direction
    flat_dev = torch.empty(moved // 2, dtype=dt, device=device)
    flat_host = torch.empty(moved // 2, dtype=dt).pin_memory()

    def timed(fn, reps):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / reps

    reps = max(args.steps, 3)
    clocks = ClockSampler(device)
    clocks.start()
    t_out = timed(lambda: pa.block_swap(dk, dv, hk, hv, out_pairs, pa.PA_SWAP_OUT), reps)
    t_in = timed(lambda: pa.block_swap(dk, dv, hk, hv, in_pairs, pa.PA_SWAP_IN), reps)
    t_d2h = timed(lambda: flat_host.copy_(flat_dev, non_blocking=True), reps)
    t_h2d = timed(lambda: flat_dev.copy_(flat_host, non_blocking=True), reps)
    clk = clocks.stop()
    pa.check_status()
    gbs = lambda t: moved / t / 1e9  # noqa: E731
    line = {
        "metric": "paged KV block swap tokens/s (device <-> page-locked host), 1 GPU",
        "value": nblk * 16 * 2 / (t_out + t_in), "unit": "tokens/s (out + in, all layers)",
        "n_gpus": 1, "steps": reps, "warmup": 1, "ms_per_step": (t_out + t_in) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) caches, random block placement)",
        "config": {"workload": "swap_8b_bf16", "layers": layers, "blocks_per_swap": nblk,
                   "num_kv_heads": hkv, "head_dim": d, "block_size": 16,
                   "bytes_per_direction": moved,
                   "step": "pa_block_swap out (1024 blocks x all layers), then back in"},
        "roofline": {"bound": "link", "unit": "GB/s",
                     "out": {"achieved": gbs(t_out), "peak": gbs(t_d2h), "frac": t_d2h / t_out},
                     "in": {"achieved": gbs(t_in), "peak": gbs(t_h2d), "frac": t_h2d / t_in},
                     "peak_source": "pinned cudaMemcpyAsync of the same bytes, same run"},
        "gpu_launches": 2 * reps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_swap_baseline(layers, args.cpu_seconds / 4)
    print(json.dumps(line))


def cow_divergence(pool, script):
    """Drives a block pool (the native one or the oracle's model, same calls)
    to the divergence point of parallel sampling: every prompt of
    ``prompt_len + shared_extra`` tokens forked into ``branches`` branches,
    then one append per branch.  Returns the branches and the copy-on-write
    pairs, int64 [P, 2]: every branch but the last holder of each shared
    partial block gets its own copy."""
    roots = []
    for p in range(script.prompts):
        s = pool.new_seq()
        for _ in range(script.prompt_len + int(script.shared_extra[p])):
            pool.append_slot(s)
        roots.append(s)
    branches = []
    for s in roots:
        branches.append(s)
        branches.extend(pool.fork(s) for _ in range(script.branches - 1))
    pairs = [cow for _, cow in (pool.append_slot(b) for b in branches) if cow is not None]
    return branches, np.asarray(pairs, dtype=np.int64).reshape(-1, 2)


COPY_METRIC = "paged KV copy-on-write block copies/s (all layers, K and V), 1 GPU"


def run_copy_bench(args):
    """Copy-on-write at the divergence of parallel sampling: 32 prompts of
    1024 + U{1..15} tokens forked 4 ways; the first divergent append of each
    branch copies the shared partial block (96 pairs), in every one of 32
    8B-shaped GQA layers (32 / 8 heads, head_dim 128, bf16), one launch per
    step.  The pairs come from the native pool; consecutive steps use four
    relabellings of the physical ids so each step copies other blocks.
    Roofline: bytes read + written against the measured HBM copy."""
    import pagedattention_decode_attention_gb300 as pa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    layers = args.layers if args.layers > 0 else 32
    hkv, d, dt = 8, 128, torch.bfloat16
    script = wl.sampling_cow()
    nb = script.num_blocks
    pool = pa.BlockPool(nb, 16, script.initial_order)
    _, base = cow_divergence(pool, script)
    npairs = base.shape[0]
    assert npairs == script.prompts * (script.branches - 1)
    gen = np.random.default_rng(wl.SEED_BASE + 8)
    relabel = [np.arange(nb)] + [gen.permutation(nb) for _ in range(3)]
    pair_sets = [torch.from_numpy(r[base]).to(device) for r in relabel]
    kc = [wl.normal((nb, hkv, 16, d), dt, 5000 + 2 * i, device) for i in range(layers)]
    vc = [wl.normal((nb, hkv, 16, d), dt, 5001 + 2 * i, device) for i in range(layers)]
    block_bytes = hkv * 16 * d * 2
    moved = 2 * 2 * block_bytes * npairs * layers       # K and V, read + written, per pair
    # The branches of one prompt copy the same shared block, so a source is
    # read from DRAM once and from L2 after that: the DRAM minimum counts
    # each distinct source once and every destination once.
    n_src = len(np.unique(base[:, 0]))
    unique = 2 * block_bytes * (n_src + npairs) * layers
    caches = pa.LayerCaches(kc, vc)        # checked once; each copy is one C call
    host_sets = [torch.from_numpy(r[base]).pin_memory() for r in relabel]
    staging = torch.empty_like(pair_sets[0])

    warm = max(args.warmup, 3)
    for i in range(warm):
        caches.block_copy(pair_sets[i % 4])
    pa.check_status()
    torch.cuda.synchronize()
    steps = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    clocks = ClockSampler(device)
    clocks.start()
    ev[0].record()
    for i in range(steps):
        caches.block_copy(pair_sets[i % 4])
        ev[i + 1].record()
    torch.cuda.synchronize()
    # end to end: the pool's pairs copied from page-locked host memory, the
    # copy, and the status read back, every step
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        staging.copy_(host_sets[i % 4], non_blocking=True)
        caches.block_copy(staging)
        pa.check_status()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    per = [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(steps)]
    total = ev[0].elapsed_time(ev[steps]) / 1e3
    e2e_s = e0.elapsed_time(e1) / 1e3
    # context: one contiguous device-to-device copy of the same bytes
    flat_src = torch.empty(moved // 2, dtype=torch.uint8, device=device)   # read + written = moved
    flat_dst = torch.empty_like(flat_src)
    for _ in range(3):
        flat_dst.copy_(flat_src)
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    m0.record()
    for _ in range(steps):
        flat_dst.copy_(flat_src)
    m1.record()
    torch.cuda.synchronize()
    memcpy_gbs = moved * steps / (m0.elapsed_time(m1) / 1e3) / 1e9
    del flat_src, flat_dst

    # every destination equals its source afterwards (a fresh destination)
    probe = pair_sets[1]
    for c in (kc[0], vc[-1]):
        c.index_fill_(0, probe[:, 1], 0)
    caches.block_copy(probe)
    pa.check_status()
    for c in (kc[0], vc[-1]):
        assert torch.equal(c.index_select(0, probe[:, 1]), c.index_select(0, probe[:, 0]))

    peak, peak_kind = load_peaks()
    avg = total / steps
    line = {
        "metric": COPY_METRIC, "value": npairs / avg, "unit": "block copies/s",
        "n_gpus": 1, "steps": steps, "warmup": warm, "ms_per_step": avg * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) caches; pairs from the native pool's forks)",
        "config": {"workload": "block_copy_8b", "layers": layers, "pairs": npairs,
                   "prompts": script.prompts, "branches": script.branches,
                   "num_kv_heads": hkv, "head_dim": d, "block_size": 16, "num_blocks": nb,
                   "bytes_per_step": moved, "distinct_sources": n_src,
                   "unique_bytes_per_step": unique,
                   "l2": "inputs larger than L2 (201 MB copied per step, four rotating pair sets)",
                   "step": "pa_block_copy of the 96 divergence pairs in all layers"},
        "roofline": {"bound": "hbm", "achieved": unique / avg / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": unique / avg / 1e9 / peak,
                     "traffic": profiled_copy_traffic(),
                     "bytes": "unique: each distinct source block read once, each destination "
                              "written once (K and V, all layers)",
                     "median_ms": statistics.median(per) * 1e3, "best_ms": min(per) * 1e3,
                     "median_gbs": unique / statistics.median(per) / 1e9,
                     "per_pair_gbs": moved / avg / 1e9,
                     "same_bytes_contiguous_copy_gbs": memcpy_gbs,
                     "peak_source": f"{peak_kind} hbm_gbs (read + written bytes of a copy)"},
        "e2e": {"value": npairs * steps / e2e_s, "unit": "block copies/s",
                "h2d_bytes_per_step": int(staging.numel() * 8), "d2h_bytes_per_step": 4},
        "gpu_launches": steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_copy_sample(script, layers, hkv, d, args.cpu_seconds / 4)
    print(json.dumps(line))


def oracle_copy_inputs(script, layers, hkv, d):
    """The divergence's pairs from the oracle's pool model, renumbered onto
    host caches that hold only the blocks the pairs touch (16-bit words
    standing in for bf16: the copy moves bytes).  Returns (pair count,
    per-layer K caches, V caches, renumbered pairs)."""
    from oracle.pool import BlockPool as ModelPool
    _, pairs = cow_divergence(ModelPool(script.num_blocks, 16, script.initial_order), script)
    ids, compact = np.unique(pairs, return_inverse=True)
    gen = np.random.default_rng(wl.SEED_BASE + 9)
    shape = (len(ids), hkv, 16, d)
    kc = [gen.integers(0, 1 << 16, size=shape, dtype=np.uint16) for _ in range(layers)]
    vc = [gen.integers(0, 1 << 16, size=shape, dtype=np.uint16) for _ in range(layers)]
    return len(pairs), kc, vc, compact.reshape(pairs.shape)


def oracle_copy_sample(script, layers, hkv, d, seconds):
    """The oracle's block copy of the same divergence, repeated for about
    ``seconds``."""
    import oracle.attention as oa
    npairs, kc, vc, compact = oracle_copy_inputs(script, layers, hkv, d)
    oa.block_copy(kc, vc, compact)
    reps, t0 = 0, time.perf_counter()
    while True:
        oa.block_copy(kc, vc, compact)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    secs = time.perf_counter() - t0
    return {"value": npairs * reps / secs, "unit": "block copies/s", "cores": 1,
            "kind": "oracle",
            "sample": (f"{reps} runs of the oracle's block copy of the {npairs} divergence "
                       f"pairs in all {layers} layers, 1 thread")}


def pool_churn_stream(seed: int, n: int):
    """Prefix-mix request stream: three 1024-token system prompts shared by
    all requests, suffixes lognormal (median 128, clipped to [1, 4096]), 8 to
    64 new tokens each, 0-3 arrivals per step."""
    gen = np.random.default_rng(seed)
    systems = [list(range(100_000 * (k + 1), 100_000 * (k + 1) + 1024)) for k in range(3)]
    reqs = []
    for _ in range(n):
        sfx = int(np.clip(round(np.exp(gen.normal(np.log(128), 1.0))), 1, 4096))
        reqs.append((systems[int(gen.integers(3))] + [int(x) for x in gen.integers(0, 50_000, sfx)],
                     int(gen.integers(8, 65))))
    return reqs, gen.integers(0, 4, size=1_000_000)


def drive_pool(pool, reqs, arrivals):
    """Runs the continuous-batching driver until every request retired;
    returns (pool operations, steps, seconds)."""
    from pagedattention_decode_attention_gb300.batching import ContinuousBatcher
    b = ContinuousBatcher(pool, 16, max_running=128)
    pending = list(reqs)
    ops = steps = 0
    tok = lambda r: (r.rid * 7919 + r.generated * 104729) % 50_000  # noqa: E731
    t0 = time.perf_counter()
    while pending or not b.idle:
        for _ in range(int(arrivals[steps])):
            if pending:
                b.submit(*pending.pop(0))
        rep = b.step(tok)
        ops += (len(rep.slots) + len(rep.admitted) + len(rep.retired) + len(rep.swap_out)
                + len(rep.swap_in))
        steps += 1
    return ops, steps, time.perf_counter() - t0


def run_pool_bench(args):
    """Host block pool under continuous-batching churn (no GPU work): pool
    operations per second through the public API."""
    import pagedattention_decode_attention_gb300 as pa
    reqs, arrivals = pool_churn_stream(wl.SEED_BASE + 8, 200)
    pool = pa.BlockPool(4096, 16, np.random.default_rng(1).permutation(4096))
    pool.enable_prefix_cache()
    pool.set_host_blocks(1024)
    ops, steps, secs = drive_pool(pool, reqs, arrivals)
    st = pool.stats()
    print(json.dumps(pool_line(ops, steps, secs, st, impl=None)))


def pool_line(ops, steps, secs, st, impl):
    line = {
        "metric": "host block pool operations/s under continuous batching (prefix cache, swap)",
        "value": ops / secs, "unit": "ops/s", "n_gpus": 1, "steps": steps, "warmup": 0,
        "ms_per_step": secs / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic prefix-mix request stream",
        "config": {"workload": "pool_churn", "requests": 200, "num_blocks": 4096,
                   "host_blocks": 1024, "system_prompts": "3 x 1024 tokens",
                   "prefix_hit_tokens": st["prefix_hit_tokens"], "evictions": st["evictions"],
                   "ops": "one per appended token, admission, retirement, swap"},
    }
    if impl:
        line["impl"] = impl
    return line


def run_reference_pool(args):
    """Reference arm of the pool workload: the pool model driven the same way."""
    from oracle.pool import BlockPool as ModelPool
    reqs, arrivals = pool_churn_stream(wl.SEED_BASE + 8, 200)
    pool = ModelPool(4096, 16, np.random.default_rng(1).permutation(4096))
    pool.enable_prefix_cache()
    pool.set_host_blocks(1024)
    ops, steps, secs = drive_pool(pool, reqs, arrivals)
    line = pool_line(ops, steps, secs, pool.stats(), impl="reference")
    line["cpu_baseline"] = {"value": line["value"], "unit": "ops/s", "cores": 1, "kind": "oracle",
                            "sample": "the whole stream through the Python pool model"}
    line["e2e"] = {"value": line["value"], "unit": "ops/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}
    print(json.dumps(line))


def oracle_prefill_inputs(batch):
    """Host inputs of the chunked-prefill oracle for the workload's shapes:
    (q, k cache, v cache, query starts, row order)."""
    qs = np.concatenate([[0], np.cumsum(batch.extra["query_lens"])]).astype(np.int64)
    total_q = int(qs[-1])
    gen = np.random.default_rng(batch.seed)
    shape = (batch.num_blocks, batch.num_kv_heads, 16, batch.head_dim)
    kc = gen.standard_normal(shape, dtype=np.float32)
    vc = gen.standard_normal(shape, dtype=np.float32)
    q = gen.standard_normal((total_q, batch.num_q_heads, batch.head_dim), dtype=np.float32)
    return q, kc, vc, qs, np.random.default_rng(7).permutation(total_q)


def oracle_prefill_baseline(batch, seconds: float) -> dict:
    """The prefill oracle on 8 query rows at a time for about ``seconds``:
    query tokens/s per layer on one host thread."""
    import oracle.attention as oa
    q, kc, vc, qs, order = oracle_prefill_inputs(batch)
    oa.paged_attention_prefill(q, kc, vc, batch.block_tables, batch.context_lens, qs, batch.scale,
                               rows=order[:8])  # untimed first call
    rows, t0 = 0, time.perf_counter()
    while rows == 0 or time.perf_counter() - t0 < seconds:
        sel = order[rows % len(order):][:8]
        oa.paged_attention_prefill(q, kc, vc, batch.block_tables, batch.context_lens, qs,
                                   batch.scale, rows=sel)
        rows += len(sel)
    value = rows / (time.perf_counter() - t0)
    return {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows} query rows (all heads) of one layer, float64 numpy, 1 thread"}


def run_reference_prefill(args):
    """Reference arm of the chunked-prefill workload: the prefill oracle on a
    bounded sample of query rows per step, scaled to query tokens/s."""
    import oracle.attention as oa
    batch = make_batch("prefill_8b", 0)
    q, kc, vc, qs, order = oracle_prefill_inputs(batch)
    total_q = len(order)
    rows_per_step = 8
    for i in range(max(args.warmup, 3)):
        oa.paged_attention_prefill(q, kc, vc, batch.block_tables, batch.context_lens, qs,
                                   batch.scale, rows=order[i * rows_per_step:(i + 1) * rows_per_step])
    t0 = time.perf_counter()
    for i in range(args.steps):
        sel = order[(i * rows_per_step) % total_q:][:rows_per_step]
        oa.paged_attention_prefill(q, kc, vc, batch.block_tables, batch.context_lens, qs,
                                   batch.scale, rows=sel)
    secs = time.perf_counter() - t0
    value = rows_per_step * args.steps / secs
    line = {
        "impl": "reference", "metric": "paged chunked-prefill attention query tokens/s per layer, 1 GPU",
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": batch.name, "num_seqs": batch.num_seqs},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: {rows_per_step} query rows (all heads), float64 numpy, 1 thread"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_reference_copy(args):
    """Reference arm of the block_copy_8b workload: the oracle's pool model
    and block copy, each step one copy of the 96 divergence pairs in every
    layer (host caches holding only the blocks the pairs touch)."""
    import oracle.attention as oa
    script = wl.sampling_cow()
    layers = args.layers if args.layers > 0 else 32
    npairs, kc, vc, compact = oracle_copy_inputs(script, layers, 8, 128)
    warm = max(args.warmup, 3)
    for _ in range(warm):
        oa.block_copy(kc, vc, compact)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oa.block_copy(kc, vc, compact)
    secs = time.perf_counter() - t0
    value = npairs * args.steps / secs
    line = {
        "impl": "reference", "metric": COPY_METRIC, "value": value, "unit": "block copies/s",
        "n_gpus": 1, "steps": args.steps, "warmup": warm, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16",
        "data": "synthetic", "config": {"workload": "block_copy_8b", "layers": layers,
                                        "pairs": npairs},
        "cpu_baseline": {"value": value, "unit": "block copies/s", "cores": 1, "kind": "oracle",
                         "sample": (f"each step: the {npairs} divergence pairs in all "
                                    f"{layers} layers, numpy, 1 thread")},
        "e2e": {"value": value, "unit": "block copies/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def oracle_swap_step(layers: int, nblk: int = 64):
    """One step of the oracle's block swap: ``nblk`` blocks of every layer out
    to a second set of host caches and back (16-bit words standing in for
    bf16).  Returns (step function, blocks per direction)."""
    import oracle.attention as oa
    hkv, d, nb = 8, 128, 2 * nblk
    gen = np.random.default_rng(wl.SEED_BASE + 7)
    shape = (nb, hkv, 16, d)
    dk = [gen.integers(0, 1 << 16, size=shape, dtype=np.uint16) for _ in range(layers)]
    dv = [gen.integers(0, 1 << 16, size=shape, dtype=np.uint16) for _ in range(layers)]
    hk = [np.empty((nblk, hkv, 16, d), dtype=np.uint16) for _ in range(layers)]
    hv = [np.empty((nblk, hkv, 16, d), dtype=np.uint16) for _ in range(layers)]
    out_pairs = np.stack([gen.choice(nb, nblk, replace=False), gen.permutation(nblk)], 1)
    in_pairs = np.stack([gen.permutation(nblk), gen.choice(nb, nblk, replace=False)], 1)

    def step():
        oa.block_swap(dk, dv, hk, hv, out_pairs)
        oa.block_swap(hk, hv, dk, dv, in_pairs)
    return step, nblk


def oracle_swap_baseline(layers: int, seconds: float) -> dict:
    step, nblk = oracle_swap_step(layers)
    step()
    n, t0 = 0, time.perf_counter()
    while n == 0 or time.perf_counter() - t0 < seconds:
        step()
        n += 1
    value = nblk * 16 * 2 * n / (time.perf_counter() - t0)
    return {"value": value, "unit": "tokens/s (out + in, all layers)", "cores": 1,
            "kind": "oracle",
            "sample": f"{n} steps of {nblk} blocks of all {layers} layers out and back, 1 thread"}


def run_reference_swap(args):
    """Reference arm of the swap_8b workload: the oracle's block swap, each
    step 64 blocks of every layer out to a second set of host caches and back
    (a bounded sample of the 1024-block batch)."""
    layers = args.layers if args.layers > 0 else 32
    step, nblk = oracle_swap_step(layers)

    warm = max(args.warmup, 3)
    for _ in range(warm):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t0
    value = nblk * 16 * 2 * args.steps / secs
    line = {
        "impl": "reference", "metric": "paged KV block swap tokens/s (device <-> page-locked host), 1 GPU",
        "value": value, "unit": "tokens/s (out + in, all layers)", "n_gpus": 1,
        "steps": args.steps, "warmup": warm, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16",
        "data": "synthetic", "config": {"workload": "swap_8b_bf16", "layers": layers},
        "cpu_baseline": {"value": value, "unit": "tokens/s (out + in, all layers)", "cores": 1,
                         "kind": "oracle",
                         "sample": (f"each step: {nblk} blocks of all {layers} layers out and "
                                    "back between host arrays, numpy, 1 thread")},
        "e2e": {"value": value, "unit": "tokens/s (out + in, all layers)",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    if args.workload == "prefill_8b":
        run_reference_prefill(args)
        return
    if args.workload == "pool_churn":
        run_reference_pool(args)
        return
    if args.workload == "block_copy_8b":
        run_reference_copy(args)
        return
    if args.workload == "swap_8b":
        run_reference_swap(args)
        return
    batch = make_batch(args.workload, 0, model_pool=True)
    per_step_units = batch.num_layers          # one token's worth of (sequence, layer) units
    inp = OracleInputs(batch, None)
    for _ in range(max(args.warmup, 3)):
        cpu_oracle_sample(batch, inp, 0.0, step_units=1)
    t0 = time.perf_counter()
    units = 0
    for _ in range(args.steps):
        _, u, _ = cpu_oracle_sample(batch, inp, 0.0, step_units=per_step_units)
        units += u
    secs = time.perf_counter() - t0
    value = units / batch.num_layers / secs
    # with --cascade the measured arm reports the cascade metric; the oracle
    # computes the same attention either way (the cascade is exact)
    metric, config = METRIC, decode_config(batch, world)
    if args.cascade and args.workload in ("prefix_8b", "sampling_8b"):
        metric = ("decode tokens/s, grouped shared-prefix (cascade) path, 1 GPU"
                  if "group_start" in batch.extra
                  else "decode tokens/s, shared-prefix (cascade) path, 1 GPU")
        config = cascade_config(batch)
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "warmup_steps_run": max(args.warmup, 3),
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": (f"each step: {per_step_units} (sequence, layer) units "
                                    "(one token) of the workload, float64 numpy, 1 thread")},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "prefill_8b":
        run_prefill_bench(args)
    elif args.workload in ("prefix_8b", "sampling_8b") and args.cascade:
        run_cascade_bench(args)
    elif args.workload == "swap_8b":
        run_swap_bench(args)
    elif args.workload == "block_copy_8b":
        run_copy_bench(args)
    elif args.workload == "pool_churn":
        run_pool_bench(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
