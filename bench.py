"""Benchmark of the paged decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]

Prints ONE JSON line (rank 0).  Workload (default): 7B-class decode, one layer
-- batch 64, 32 query heads = 32 KV heads, head_dim 128, fp16 cache in blocks
of 16, context lengths uniform integers in [50, 900], pool 1.25x the blocks
needed with tables assigned from a shuffled free list (workloads.decode_7b).

One step = one pass of the whole device hot path over the batch: the
decode step's new token of every sequence is written into its slot (the
block table's position context_len - 1) and paged decode attention runs over
the whole context, in ONE launch (paged_attention_decode_append; split
pieces are merged inside it).  --two-launch runs the write as its own
reshape_and_cache launch before a read-only decode instead.  The workload
has no copy-on-write pair at its decode step, so copy_blocks launches
nothing.  The decode goes through a DecodePlan (validated once; each step is
the launch alone) and the K timed steps go back to back on one stream, CUDA
events only at the two ends of the timed region: with programmatic dependent
launch each launch's prologue overlaps the previous launch's tail, as
consecutive layers of a model step do (--no-graph: the binding's one-shot
calls instead).

* value: KV bytes the decode reads (2 * sum(ctx) * Hkv * D * 2) per step,
  times K steps, over the device-timed K steps (CUDA events, barrier +
  synchronize on both sides, max over ranks), inputs resident in HBM.
  The KV read per step (0.57 GB) is larger than L2 (129 MB), so no L2 flush.
* e2e: the same metric through the public API with host buffers: every step
  the C++ block manager appends one token per sequence and exports the tables
  into the step's pinned staging region (with its queries and new K/V rows);
  one pkv_decode_plan_step_mapped call launches the step, whose kernel reads
  the region straight from host memory over the CPU-GPU link (the lengths and
  tables in its prologue, each piece's query and each new row a few chunks
  ahead of their use), appends the new tokens, attends and writes the output
  straight into a pinned host buffer (--e2e-staged: pkv_decode_plan_step,
  which first copies the region host->device; --e2e-copy-out: a device->host
  copy after the launch instead); the host waits
  for the step (polling an event); the next step's block-manager work
  overlaps the GPU's work on this step; the staging region is a ring of 4
  pinned rows (--e2e-ring).  20 untimed warm-up steps first; the
  line also gives the per-step wall-time percentiles.
* roofline: the decode launch timed alone with CUDA events on its stream
  over the timed region; algorithmic bytes / mean duration vs the
  measured HBM copy bandwidth.
* e2e.breakdown: 50 more serving steps with the step's parts issued as
  separate operations, CUDA events between them and host clocks around them
  (medians): where the e2e step's time outside the kernel goes.
* secondary (the default run on one GPU): the headline launch again, 50
  back-to-back repetitions and 50 with a 256 MB buffer read between
  repetitions (outside the event pair, so each starts with a cold L2); the
  chat, gqa and prefix workloads the same way (prefix also against the bytes
  of the distinct blocks it reaches); identity against shuffled tables (the
  paging overhead); copy_blocks on the prefix workload's first divergent
  step (127 copy-on-write pairs) and reshape_and_cache of the 7B-class
  step's new rows (L2-flushed medians).
* cpu_baseline: the fp64 oracle on the host cores, on a bounded sample of the
  same workload.
* --impl reference: the oracle as the reference arm (rank 0 only).
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
from workloads import BASE_SEED as W_BASE_SEED  # noqa: E402  (numpy only; torch loads lazily)

METRIC = "paged decode attention: KV-read HBM GB/s (% of GB300 peak), seqs/s per layer"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20  # read between flushed repetitions: twice the 129 MB L2
KERNEL_SOURCES = ["pkv_decode_impl.cuh", "pkv_decode_inst.cuh", "pkv_decode.cu", "pkv_device.cuh",
                  "pkv_schedule.h", "pkv_decode_params.h"]

WORKLOAD_TEXT = {
    "7b": "7B-class decode, one layer: batch 64, 32 query heads = 32 KV heads, head_dim 128, fp16, "
          "block_size 16, context uniform integers in [50, 900], pool 1.25x needed, shuffled free list",
    "tiny": "tiny: 4 sequences, context 40/17/100/5, 8 heads, head_dim 64, block 16, pool 64",
    "chat": "chat, one layer: batch 128, prompt U[100,2000] + generated U[50,500], 32 heads, head_dim 128, "
            "block 16, arrival-order allocation with interleaved frees",
    "gqa": "GQA long context, one layer: batch 256, 32 query / 8 KV heads, head_dim 128, block 32, "
           "context log-uniform in [256, 4096], shuffled pool",
    "prefix": "prefix sharing, one layer: 128 sequences sharing a 500-token prefix, suffix U[50,500], "
              "32 heads, head_dim 128, block 16",
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    p.add_argument("--config", choices=list(WORKLOAD_TEXT), default="7b")
    p.add_argument("--seed", type=int, default=None,
                   help="base seed of the workload's draws (lengths, free orders, values); default 152")
    p.add_argument("--num-ctas", type=int, default=0)
    p.add_argument("--block-size", type=int, default=0,
                   help="override the workload's block size (8, 16, 32, 64, 128): the block-size sweep")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-ring", type=int, default=E2E_RING,
                   help="e2e: pinned staging rows used in turn (0: one per step, each touched once)")
    p.add_argument("--e2e-staged", action="store_true",
                   help="e2e: pkv_decode_plan_step, which copies the staged inputs host->device before the launch "
                        "(default: pkv_decode_plan_step_mapped, the kernel reads them from host memory)")
    p.add_argument("--e2e-copy-out", action="store_true",
                   help="e2e: the kernel writes device memory and a D2H copy brings the output back (default: "
                        "the kernel writes the pinned host buffer directly)")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-secondary", action="store_true",
                   help="skip the secondary measurements (other workloads, identity tables, cache ops, "
                        "L2-flushed repetitions) that the default run adds to its line")
    p.add_argument("--two-launch", action="store_true",
                   help="reshape_and_cache, then a decode that only reads (instead of the decode launch "
                        "that writes the new tokens itself)")
    p.add_argument("--no-graph", action="store_true",
                   help="every step through the binding's one-shot calls instead of a DecodePlan launch")
    p.add_argument("--shared", action="store_true",
                   help="decode through the prefix-sharing entry point (paged_attention_decode_shared) with the "
                        "block manager's shared-prefix hints")
    p.add_argument("--identity-tables", action="store_true",
                   help="same workload with each sequence's blocks contiguous and in order")
    p.add_argument("--layers", type=int, default=0,
                   help="measure a model step instead: this many layers, each with its own pools, one "
                        "decode launch per layer, all layers captured as one CUDA graph")
    p.add_argument("--swap", action="store_true",
                   help="measure swapping instead: every sequence's blocks device -> pinned host -> device")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--cpu-worker", default=None, help=argparse.SUPPRESS)
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas, no data-path collective)

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29512")
        dist.init_process_group(backend)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value, device="cpu"):
    """Max of a float over ranks (the timing rule: the slowest rank counts)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value, device="cpu"):
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# environment facts

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the decode kernel's code: its sources without comments and
    blank lines (a recorded ncu figure stays valid across comment edits)."""
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_152_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(line.rstrip() for line in text.splitlines() if line.strip()).encode())
    return h.hexdigest()[:16]


def traffic_file(workload):
    return os.path.join(ROOT, "profiles", f"decode_{workload}_traffic.txt")


def recorded_traffic(workload):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source and this workload (else None)."""
    try:
        kv = {}
        with open(traffic_file(workload)) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_source_hash() or kv.get("workload") != workload:
            return None
        return float(kv["dram_bytes_per_decode_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        from datetime import datetime
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except Exception:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.15 <= r[0] <= self.t1 + 0.15]
        use = inside if inside else rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for name, flag in zip(names, r[3][1:5]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "window": "timed region" if inside else "whole run (timed region shorter than the sampling period)"}


# ---------------------------------------------------------------------------
# the product arm

def build_state(cfg, device, identity_tables=False, e2e_headroom_steps=0, block_size=0, seed=None):
    """Allocator + device tensors of a workload at its decode step."""
    import numpy as np
    import torch
    import paged_kv_cache_152_gb300 as pkv
    import workloads as W

    kw = {"block_size": block_size} if block_size else {}
    if seed is not None:
        kw["base"] = seed
    wl = W.make(cfg, **kw)
    n = wl.num_seqs
    extra = n * (-(-e2e_headroom_steps // wl.block_size) + 1) if e2e_headroom_steps else 0
    nb = wl.num_blocks + extra
    if identity_tables:
        order = np.arange(nb, dtype=np.int32)   # each sequence's blocks contiguous, in order
    else:
        order = np.concatenate([wl.free_order, np.arange(wl.num_blocks, nb, dtype=np.int32)])
    alloc = pkv.BlockAllocator(nb, wl.block_size, order)
    W.replay(alloc, wl.ops)
    slots, pairs = alloc.append_batch(wl.batch)
    mb = wl.max_blocks_per_seq() + (-(-e2e_headroom_steps // wl.block_size) + 1)
    tables, lens = alloc.export(wl.batch, mb)
    assert lens.tolist() == wl.context_lens
    t = W.tensors(wl, device, with_pool=False)
    shape = (nb, wl.num_kv_heads, wl.block_size, wl.head_dim)
    t["key_cache"] = W.normal_fp16_large(shape, wl.seed * 1000 + 4, device)
    t["value_cache"] = W.normal_fp16_large(shape, wl.seed * 1000 + 5, device)
    st = {
        "wl": wl, "alloc": alloc, "mb": mb, "nb": nb, "t": t,
        "shared": torch.from_numpy(alloc.shared_prefix(wl.batch)).to(device),
        "slots": torch.from_numpy(slots.astype(np.int64)).to(device),
        "pairs": torch.from_numpy(pairs.astype(np.int64)).reshape(-1, 2).to(device),
        "tables": torch.from_numpy(tables).to(device),
        "lens": torch.from_numpy(lens).to(device),
        "out": torch.empty((n, wl.num_heads, wl.head_dim), dtype=torch.float16, device=device),
        "status": torch.zeros(1, dtype=torch.int32, device=device),
    }
    # our kernels per step: copy_blocks (only with pairs), reshape_and_cache, decode
    st["launches_per_step"] = (1 if len(pairs) else 0) + 2
    return st


def write_step(pkv, st):
    """copy_blocks (if the step has copy-on-write pairs), then reshape_and_cache
    (unless the decode launch appends the new tokens itself)."""
    t = st["t"]
    if st["pairs"].shape[0]:
        pkv.copy_blocks(t["key_cache"], t["value_cache"], st["pairs"], status=st["status"])
    if not st.get("fused"):
        pkv.reshape_and_cache(t["key"], t["value"], t["key_cache"], t["value_cache"], st["slots"],
                              status=st["status"])


def decode_step(pkv, st, ws, num_ctas):
    t = st["t"]
    if st.get("use_shared"):
        kw = dict(key=t["key"], value=t["value"]) if st.get("fused") else {}
        pkv.paged_attention_decode_shared(st["out"], t["query"], t["key_cache"], t["value_cache"], st["tables"],
                                          st["lens"], st["shared"], st["wl"].scale, num_ctas=num_ctas,
                                          workspace=ws, status=st["status"], **kw)
        return
    if st.get("fused"):
        pkv.paged_attention_decode_append(st["out"], t["query"], t["key"], t["value"], t["key_cache"],
                                          t["value_cache"], st["tables"], st["lens"], st["wl"].scale,
                                          num_ctas=num_ctas, workspace=ws, status=st["status"])
        return
    pkv.paged_attention_decode(st["out"], t["query"], t["key_cache"], t["value_cache"], st["tables"],
                               st["lens"], st["wl"].scale, num_ctas=num_ctas, workspace=ws,
                               status=st["status"])


def device_step(pkv, st, ws, num_ctas, ev=None):
    """One pass of the hot path with inputs resident in HBM; returns launches."""
    write_step(pkv, st)
    if ev is not None:
        ev[0].record()
    decode_step(pkv, st, ws, num_ctas)
    if ev is not None:
        ev[1].record()
    return st["launches_per_step"]


E2E_WARMUP = 20  # untimed serving steps before the timed ones (first-use costs on the host)
E2E_BREAKDOWN = 50  # untimed steps after them, each part timed on its own
E2E_RING = 4  # pinned staging rows, used in turn (a serving loop keeps a few; one fresh row per step
#               costs the device first-touch misses on 350 MB of host pages: p90 step +40-110 us)


def run_e2e(pkv, st, ws, num_ctas, steps, device, dist, warmup=0, breakdown_steps=0, copy_out=False,
            staged=False, ring=0):
    """Serving-loop steps through the public API with host buffers.

    Every step: the C++ block manager appends one token per sequence and
    exports the tables and lengths straight into the step's page-locked
    staging region, which also holds the step's queries and new K/V rows;
    copy-on-write pairs (if any) go through copy_blocks; then ONE library call
    (pkv_decode_plan_step_mapped of a DecodePlan built once on a device
    region of the staging layout: append the new tokens + attend) launches
    the step, whose kernel reads the region from host memory and writes the
    output into pinned host memory (staged: pkv_decode_plan_step copies the
    region host->device first; copy_out: a D2H copy follows); the host waits
    for the step.  The
    block-manager work of step i+1 runs on the host while the GPU runs step
    i (as a serving loop schedules ahead).  The staging region has `ring`
    rows used in turn (0: one row per step); the block manager rewrites a
    row's tables and lengths every step, its queries and new rows were
    drawn once."""
    import numpy as np
    import torch
    wl, alloc = st["wl"], st["alloc"]
    n, h, hkv, d, mb = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim, st["mb"]
    shared = bool(st.get("use_shared"))
    parts = [("q", n * h * d * 2), ("k", n * hkv * d * 2), ("v", n * hkv * d * 2), ("tables", n * mb * 4),
             ("lens", n * 4)] + ([("shared", n * 4)] if shared else [])
    offs, off = {}, 0
    for name, nbytes in parts:
        offs[name] = (off, nbytes)
        off += -(-nbytes // 256) * 256
    step_bytes = off
    timed = steps
    steps = warmup + timed
    rows = ring if ring > 0 else steps  # staging rows, used in turn (default: one per step)
    h_stage = torch.empty((rows, step_bytes), dtype=torch.uint8).pin_memory()
    rng = np.random.default_rng(wl.seed + 77)
    stage_np = h_stage.numpy()
    for name in ("q", "k", "v"):
        o, nbytes = offs[name]
        stage_np[:, o:o + nbytes].view(np.float16)[:] = rng.standard_normal((rows, nbytes // 2)).astype(np.float16)
    tab_np = [stage_np[i % rows, offs["tables"][0]:offs["tables"][0] + offs["tables"][1]].view(np.int32)
              .reshape(n, mb) for i in range(steps)]
    lens_np = [stage_np[i % rows, offs["lens"][0]:offs["lens"][0] + offs["lens"][1]].view(np.int32)
               for i in range(steps)]
    shared_np = [stage_np[i % rows, offs["shared"][0]:offs["shared"][0] + offs["shared"][1]].view(np.int32)
                 for i in range(steps)] if shared else None
    h_rows = [h_stage[i % rows] for i in range(steps)]
    d_stage = torch.empty(step_bytes, dtype=torch.uint8, device=device)

    def dview(name, dtype, shape):
        o, nbytes = offs[name]
        return d_stage[o:o + nbytes].view(dtype).view(*shape)

    d_q = dview("q", torch.float16, (n, h, d))
    d_k = dview("k", torch.float16, (n, hkv, d))
    d_v = dview("v", torch.float16, (n, hkv, d))
    d_tables = dview("tables", torch.int32, (n, mb))
    d_lens = dview("lens", torch.int32, (n,))
    d_shared = dview("shared", torch.int32, (n,)) if shared else None
    t = st["t"]
    h_out = torch.empty((n, h, d), dtype=torch.float16).pin_memory()
    # by default the kernel writes the output straight into the pinned host
    # buffer (over the CPU-GPU link, as rows become final); copy_out: it writes
    # device memory and a D2H copy follows the launch
    plan = pkv.DecodePlan(st["out"] if copy_out else h_out, d_q, t["key_cache"], t["value_cache"], d_tables,
                          d_lens, wl.scale,
                          key=d_k, value=d_v, num_ctas=num_ctas, workspace=ws, status=st["status"],
                          shared_blocks=d_shared)
    h_slots = np.empty(n, dtype=np.int64)
    h_pairs_t = torch.empty((n, 2), dtype=torch.int64).pin_memory()
    h_pairs32 = np.empty((n, 2), dtype=np.int32)
    d_pairs = torch.empty((n, 2), dtype=torch.int64, device=device)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    d_stage_ptr, h_out_ptr = d_stage.data_ptr(), (h_out.data_ptr() if copy_out else None)
    h_row_ptrs = [r.data_ptr() for r in h_rows]
    done = torch.cuda.Event()
    step_fn = plan.step_raw if staged else plan.step_mapped_raw
    batch = np.asarray(wl.batch, dtype=np.int32)
    kv_per_token = 2 * hkv * d * 2
    bytes_total = 0
    h2d = d2h = 0
    def prepare(i):
        """Host work of step i: the block manager appends one token per
        sequence and writes the tables and lengths into step i's region."""
        _, pairs = alloc.append_batch(batch, slots_out=h_slots, pairs_out=h_pairs32)
        alloc.export(batch, mb, tables_out=tab_np[i], lens_out=lens_np[i])
        if shared:
            alloc.shared_prefix(batch, out=shared_np[i])
        return pairs.copy() if len(pairs) else None

    barrier(dist, device)
    torch.cuda.synchronize()
    marks = []  # wall clock at the start of each timed step
    t0 = time.perf_counter()
    pairs = prepare(0)
    for i in range(steps):
        if i == warmup and warmup:
            # the warm-up steps are done (each was waited for): time from here
            barrier(dist, device)
            t0 = time.perf_counter()
        timed_step = i >= warmup
        if timed_step:
            marks.append(time.perf_counter())
        if pairs is not None:
            h_pairs_t.numpy()[:len(pairs)] = pairs
            d_pairs[:len(pairs)].copy_(h_pairs_t[:len(pairs)], non_blocking=True)
            h2d += len(pairs) * 16 if timed_step else 0
            pkv.copy_blocks(t["key_cache"], t["value_cache"], d_pairs[:len(pairs)], status=st["status"])
        # one library call: the launch reading the region from host memory (staged: copied
        # host -> device first), the output into host memory
        step_fn(d_stage_ptr, h_row_ptrs[i], step_bytes, h_out_ptr, sh)
        if timed_step:
            bytes_total += int(lens_np[i].sum()) * kv_per_token
            h2d += step_bytes
            d2h += h_out.numel() * 2
        # the next step's block-manager work runs on the host while the GPU
        # runs this step (it does not depend on this step's output values)
        done.record(stream)
        if i + 1 < steps:
            pairs = prepare(i + 1)
        # wait for the step by polling (a blocking synchronize leaves the
        # waking of this thread to the OS scheduler, which on a busy host adds
        # tens of microseconds per step)
        while not done.query():
            pass
    t_end = time.perf_counter()
    elapsed = max_over_ranks(dist, t_end - t0, device)
    barrier(dist, device)
    marks.append(t_end)
    per = sorted(b - a for a, b in zip(marks, marks[1:]))
    pct = lambda q: round(per[min(len(per) - 1, int(q * len(per)))] * 1e6, 1)
    breakdown = e2e_breakdown(plan, step_fn, prepare, alloc, d_stage, h_rows, h_out if copy_out else None,
                              st["out"], stream, breakdown_steps)
    plan.close()
    return {"bytes": bytes_total, "elapsed": elapsed, "h2d": h2d // timed, "d2h": d2h // timed,
            "step_us": {"p50": pct(0.5), "p90": pct(0.9), "max": round(per[-1] * 1e6, 1)},
            "breakdown": breakdown}


def e2e_breakdown(plan, step_fn, prepare, alloc, d_stage, h_rows, h_out, d_out, stream, steps):
    """Where an e2e step's time goes: the same serving step through the same
    library call (step_fn: pkv_decode_plan_step_mapped, the launch reading the
    inputs from host memory, or pkv_decode_plan_step, the staged inputs in
    and the launch; then the output out), then the step's launch once more
    on its own on the same inputs already in device memory (copied there
    before the first event), CUDA events around both; host clocks around the
    submission, the block manager's work for the next step and the wait.
    Untimed for the e2e value; medians in microseconds.
    device_in_and_out_us = the step's device time minus the kernel's."""
    import torch
    if steps <= 0:
        return None
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    host = {"submit": [], "block_manager": [], "wait_after_block_manager": [], "step_wall": []}
    sh = stream.cuda_stream
    n_rows = len(h_rows)
    step_bytes = d_stage.numel()
    d_ptr = d_stage.data_ptr()
    out_ptr = h_out.data_ptr() if h_out is not None else None
    prepare(0)
    done = torch.cuda.Event()
    for j in range(steps):
        i = j % n_rows
        d_stage.copy_(h_rows[i], non_blocking=True)  # the same inputs in device memory for the launch alone
        ta = time.perf_counter()
        ev[j][0].record(stream)
        step_fn(d_ptr, h_rows[i].data_ptr(), step_bytes, out_ptr, sh)
        ev[j][1].record(stream)
        plan.launch_raw(sh)  # the same launch again, alone (rewrites the same new rows)
        ev[j][2].record(stream)
        done.record(stream)
        tb = time.perf_counter()
        if j + 1 < steps:
            prepare((j + 1) % n_rows)
        tc = time.perf_counter()
        while not done.query():
            pass
        td = time.perf_counter()
        host["submit"].append(tb - ta)
        host["block_manager"].append(tc - tb)
        host["wait_after_block_manager"].append(td - tc)
        host["step_wall"].append(td - ta)
    torch.cuda.synchronize()
    med = lambda xs: round(statistics.median(xs) * 1e6, 2)  # noqa: E731
    step = [e[0].elapsed_time(e[1]) / 1e3 for e in ev]
    kern = [e[1].elapsed_time(e[2]) / 1e3 for e in ev]
    out = {"device_step_us": med(step), "device_kernel_us": med(kern),
           "device_in_and_out_us": med([a - b for a, b in zip(step, kern)])}
    out.update({f"host_{k}_us": med(v) for k, v in host.items()})
    out["outside_device_work_us"] = med([w - a - b for w, a, b in zip(host["step_wall"], step, kern)])
    out["steps"] = steps
    out["how"] = ("each step: the e2e loop's library call (the launch reading its inputs from host memory, or "
                  "the staged copy in and the launch; the output out) between CUDA events, then the same launch "
                  "alone on the same inputs in device memory between events; host clocks around the submission, "
                  "the next step's block-manager work and the wait; outside_device_work_us = wall time minus both "
                  "device intervals")
    return out


def time_launches(fn, reps, stream, flush=None):
    """Device time (ms) of each of `reps` calls of fn(), from CUDA events on
    `stream`.  With `flush` (a buffer larger than L2) the buffer is read
    between calls, outside the event pair: each call starts with nothing of
    its inputs in L2 (clean lines only, so no write-back lands in the timed
    call), and the read also keeps the GPU busy while the host enqueues the
    call, so no host gap falls between the events."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, z in ev:
        if flush is not None:
            flush.amax()
        a.record(stream)
        fn()
        z.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(z) for a, z in ev]

# The longest context each workload's distribution allows: what a contiguous
# KV cache must reserve per request up front (the waste comparison of
# [P1] "The problem": max-length reservations against blocks on demand).
MAX_CONTEXT = {"tiny": 100, "7b": 900, "chat": 2500, "gqa": 4096, "prefix": 1000}


def waste_pct(wl, max_len):
    """KV slots held but unused, in %: paged (the last block of each
    sequence partly filled) and contiguous (max_len reserved per sequence)."""
    used = sum(wl.context_lens)
    paged = wl.block_size * sum(-(-c // wl.block_size) for c in wl.context_lens)
    return {"paged_waste_pct": round(100 * (1 - used / paged), 2),
            "contiguous_waste_pct": round(100 * (1 - used / (max_len * wl.num_seqs)), 2),
            "contiguous_reservation_tokens": max_len}


def period_launches(fn, reps, stream):
    """Mean period (ms) of `reps` calls of fn() issued back to back, CUDA
    events at the two ends only: with programmatic dependent launch each
    launch's prologue overlaps the previous launch's tail."""
    import torch
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    z.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(z) / reps


def unique_kv_bytes(tables, lens, block_size, num_kv_heads, head_dim):
    """K+V bytes of the distinct physical blocks the tables reach (rows in
    use only): what a launch must bring from DRAM when blocks shared between
    sequences are read once."""
    rows = {}
    for s, n in enumerate(lens):
        n = int(n)
        for i in range(-(-n // block_size)):
            b = int(tables[s][i])
            rows[b] = max(rows.get(b, 0), min(block_size, n - i * block_size))
    return 2 * sum(rows.values()) * num_kv_heads * head_dim * 2


def measure_decode(pkv, name, device, peak, reps, flush, identity_tables=False, shared=False):
    """One workload's decode launch (the fused append + attend of the bench
    step, through a DecodePlan; shared: the prefix-sharing plan with the block
    manager's hints): the mean of launches each between its own events, the
    period of launches back to back (events at the ends only) and the
    L2-flushed median."""
    import torch
    stream = torch.cuda.current_stream()
    st = build_state(name, device, identity_tables=identity_tables)
    wl, t = st["wl"], st["t"]
    ws = pkv.new_workspace(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, 0, device,
                           shared=shared)
    plan = pkv.DecodePlan(st["out"], t["query"], t["key_cache"], t["value_cache"], st["tables"], st["lens"],
                          wl.scale, key=t["key"], value=t["value"], workspace=ws, status=st["status"],
                          shared_blocks=st["shared"] if shared else None)
    for _ in range(5):
        plan.launch()
    b2b = time_launches(plan.launch, reps, stream)
    per_us = period_launches(plan.launch, reps, stream) * 1e3
    fl = time_launches(plan.launch, reps, stream, flush)
    assert int(st["status"].item()) == 0, pkv.status_string(int(st["status"].item()))
    kv = wl.kv_read_bytes()
    mean_us, med_us = statistics.fmean(b2b) * 1e3, statistics.median(fl) * 1e3
    r = {"decode_us_mean": round(mean_us, 2), "period_us_back_to_back": round(per_us, 2),
         "GB_s_back_to_back": round(kv / per_us / 1e3, 1), "frac_back_to_back": round(kv / per_us / 1e3 / peak, 4),
         "decode_us_median_l2_flushed": round(med_us, 2), "reps": reps,
         "kv_bytes": kv, "GB_s": round(kv / mean_us / 1e3, 1), "frac": round(kv / mean_us / 1e3 / peak, 4),
         "GB_s_l2_flushed": round(kv / med_us / 1e3, 1), "frac_l2_flushed": round(kv / med_us / 1e3 / peak, 4),
         "seqs_per_s": round(wl.num_seqs / mean_us * 1e6, 1),
         "traffic": None if identity_tables else recorded_traffic(name + ("_shared" if shared else ""))}
    r.update(waste_pct(wl, MAX_CONTEXT[name]))
    if name == "prefix":
        u = unique_kv_bytes(st["tables"].cpu().numpy(), wl.context_lens, wl.block_size, wl.num_kv_heads,
                            wl.head_dim)
        r["logical"] = "kv_bytes counts every sequence's read of the shared prefix"
        r["unique_kv_bytes"] = u
        r["unique_GB_s"] = round(u / mean_us / 1e3, 1)
        r["unique_frac"] = round(u / mean_us / 1e3 / peak, 4)
    plan.close()
    del plan, ws, st, t
    torch.cuda.empty_cache()
    return r


def measure_cache_ops(pkv, device, peak, reps, flush):
    """copy_blocks on the prefix workload's first divergent step (the 127
    copy-on-write copies of the shared tail block) and reshape_and_cache of
    the 7B-class decode step's 64 new tokens: L2-flushed medians."""
    import numpy as np
    import torch
    import workloads as W
    stream = torch.cuda.current_stream()
    status = torch.zeros(1, dtype=torch.int32, device=device)
    wl = W.make("prefix")
    alloc = pkv.BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
    stop = wl.marks["divergence"]
    W.replay(alloc, wl.ops, 0, stop)
    step = [op[1] for op in wl.ops[stop:wl.marks["after_divergence"]]]
    _, pairs = alloc.append_batch(step)
    shape = (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    kc = W.normal_fp16_large(shape, wl.seed * 1000 + 4, device)
    vc = W.normal_fp16_large(shape, wl.seed * 1000 + 5, device)
    dpairs = torch.from_numpy(pairs.astype(np.int64)).to(device)
    block_bytes = kc[0].numel() * kc.element_size()
    moved = 2 * len(pairs) * block_bytes          # per direction (read and written), K and V
    ms = time_launches(lambda: pkv.copy_blocks(kc, vc, dpairs, status=status), reps, stream, flush)
    cb_us = statistics.median(ms) * 1e3
    alloc.close()
    del kc, vc
    st = build_state("7b", device)
    t = st["t"]
    ms = time_launches(lambda: pkv.reshape_and_cache(t["key"], t["value"], t["key_cache"], t["value_cache"],
                                                     st["slots"], status=status), reps, stream, flush)
    rc_us = statistics.median(ms) * 1e3
    rc_bytes = 2 * 2 * t["key"].numel() * 2      # K and V rows, read once and written once
    rc_tokens = int(t["key"].shape[0])
    assert int(status.item()) == 0, pkv.status_string(int(status.item()))
    del st, t
    torch.cuda.empty_cache()
    return {
        "copy_blocks_prefix_divergence": {
            "pairs": int(len(pairs)), "block_bytes_per_cache": block_bytes, "bytes_read": moved,
            "bytes_written": moved, "us_median_l2_flushed": round(cb_us, 2), "reps": reps,
            "GB_s": round(2 * moved / cb_us / 1e3, 1), "frac": round(2 * moved / cb_us / 1e3 / peak, 4),
            "note": "read + written bytes over time, like the copy bandwidth it is compared with"},
        "reshape_and_cache_7b": {
            "tokens": rc_tokens, "bytes_read_plus_written": rc_bytes, "us_median_l2_flushed": round(rc_us, 2),
            "reps": reps, "note": "one decode step's new rows: launch-latency bound"},
    }


def run_secondary(pkv, device, peak, st_main, ws_main, reps=50):
    """The secondary measurements of the default run: the headline launch
    each between its own events, back to back, and with L2 flushed between
    repetitions; the same for chat, gqa and prefix; identity
    against shuffled tables (the paging overhead); copy_blocks and
    reshape_and_cache."""
    import torch
    stream = torch.cuda.current_stream()
    flush = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    wl, t = st_main["wl"], st_main["t"]
    plan = pkv.DecodePlan(st_main["out"], t["query"], t["key_cache"], t["value_cache"], st_main["tables"],
                          st_main["lens"], wl.scale, key=t["key"], value=t["value"], workspace=ws_main,
                          status=st_main["status"])
    b2b = time_launches(plan.launch, reps, stream)
    per_us = period_launches(plan.launch, reps, stream) * 1e3
    fl = time_launches(plan.launch, reps, stream, flush)
    plan.close()
    kv = wl.kv_read_bytes()
    res = {"7b": {"decode_us_mean": round(statistics.fmean(b2b) * 1e3, 2),
                  "period_us_back_to_back": round(per_us, 2),
                  "GB_s_back_to_back": round(kv / per_us / 1e3, 1),
                  "frac_back_to_back": round(kv / per_us / 1e3 / peak, 4),
                  "decode_us_median_l2_flushed": round(statistics.median(fl) * 1e3, 2), "reps": reps,
                  "GB_s_l2_flushed": round(kv / statistics.median(fl) / 1e6, 1),
                  "frac_l2_flushed": round(kv / statistics.median(fl) / 1e6 / peak, 4)}}
    for name in ("chat", "gqa", "prefix"):
        res[name] = measure_decode(pkv, name, device, peak, reps, flush)
    # the prefix workload again, its shared prompt read once per group of 8
    # forks (paged_attention_decode_shared)
    res["prefix_shared"] = measure_decode(pkv, "prefix", device, peak, reps, flush, shared=True)
    ident = measure_decode(pkv, "7b", device, peak, reps, flush, identity_tables=True)
    shuf = res["7b"]["decode_us_mean"]
    res["paging_overhead_7b"] = {
        "identity_tables_us_mean": ident["decode_us_mean"], "shuffled_tables_us_mean": shuf,
        "identity_tables_us_median_l2_flushed": ident["decode_us_median_l2_flushed"],
        "shuffled_tables_us_median_l2_flushed": res["7b"]["decode_us_median_l2_flushed"],
        "pct": round(100 * (shuf - ident["decode_us_mean"]) / ident["decode_us_mean"], 2),
        "note": "shuffled pool vs each sequence's blocks contiguous and in order, same kernel"}
    res.update(measure_cache_ops(pkv, device, peak, reps, flush))
    del flush
    torch.cuda.empty_cache()
    return res


def run_pkv(args):
    import torch
    import paged_kv_cache_152_gb300 as pkv

    rank, local_rank, world = dist_env()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = dist_init(world, "nccl")
    from paged_kv_cache_152_gb300 import build as b
    if rank == 0 or world == 1:
        b.build()
    barrier(dist, device)
    pkv.load()

    # the e2e loop runs its own step count (a step is ~0.1 ms; a short run is at
    # the mercy of one slow host wake-up)
    e2e_steps = 0 if args.no_e2e else max(1, args.e2e_steps)
    st = build_state(args.config, device, args.identity_tables,
                     e2e_headroom_steps=e2e_steps + E2E_WARMUP + E2E_BREAKDOWN if e2e_steps else 0,
                     block_size=args.block_size, seed=args.seed)
    if not args.two_launch:
        st["fused"] = True
        st["launches_per_step"] -= 1
    st["use_shared"] = args.shared
    wl = st["wl"]
    ws = pkv.new_workspace(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                           args.num_ctas, device, shared=args.shared)
    kv_bytes = wl.kv_read_bytes()
    clocks = ClockSampler(local_rank)

    # warm-up (untimed)
    for _ in range(max(3, args.warmup)):
        device_step(pkv, st, ws, args.num_ctas)
    torch.cuda.synchronize()
    assert int(st["status"].item()) == 0, pkv.status_string(int(st["status"].item()))

    # the step as launched in the timed region: the decode through a DecodePlan
    # (validated once; each launch is the launch alone), after the step's
    # cache-write calls when it has any (copy-on-write pairs; reshape_and_cache
    # without the fused decode).  Steps go back to back on one stream: with
    # programmatic dependent launch each launch's prologue and first table
    # loads overlap the previous launch's tail, as consecutive layers of a
    # model step do.  --no-graph: the binding's one-shot calls instead.
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    t = st["t"]
    has_write = bool(st["pairs"].shape[0]) or not st.get("fused")
    plan = None
    if not args.no_graph:
        kw = dict(key=t["key"], value=t["value"]) if st.get("fused") else {}
        plan = pkv.DecodePlan(st["out"], t["query"], t["key_cache"], t["value_cache"], st["tables"], st["lens"],
                              wl.scale, num_ctas=args.num_ctas, workspace=ws, status=st["status"],
                              shared_blocks=st["shared"] if st.get("use_shared") else None, **kw)
        for _ in range(3):
            if has_write:
                write_step(pkv, st)
            plan.launch_raw(sh)
        torch.cuda.synchronize()

    # timed region: K steps back to back, CUDA events at its two ends only,
    # barrier + synchronize both sides
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize()
    clocks.start()
    h0 = time.perf_counter()
    e_start.record(stream)
    launches = 0
    for i in range(args.steps):
        if plan is None:
            launches += device_step(pkv, st, ws, args.num_ctas)
        else:
            if has_write:
                write_step(pkv, st)
            plan.launch_raw(sh)
            launches += st["launches_per_step"]
    e_stop.record(stream)
    host_s = time.perf_counter() - h0
    torch.cuda.synchronize()
    clocks.stop()
    barrier(dist, device)
    elapsed_ms = e_start.elapsed_time(e_stop)
    assert int(st["status"].item()) == 0, pkv.status_string(int(st["status"].item()))
    ms_total = max_over_ranks(dist, elapsed_ms, device)
    # the decode launch on its own (each between its own events: no overlap
    # with a neighbour), for context beside the back-to-back period
    iso = time_launches(plan.launch if plan is not None else (lambda: decode_step(pkv, st, ws, args.num_ctas)),
                        min(50, max(5, args.steps)), stream)
    dec_iso = max_over_ranks(dist, statistics.median(iso), device)
    # the decode's average launch duration over the timed region: the period
    # of the back-to-back launches when a step is the decode launch alone,
    # else the launch on its own
    dec_mean = ms_total / args.steps if st["launches_per_step"] == 1 else dec_iso

    e2e = None
    if e2e_steps:
        e2e = run_e2e(pkv, st, ws, args.num_ctas, e2e_steps, device, dist, warmup=E2E_WARMUP,
                      breakdown_steps=E2E_BREAKDOWN, copy_out=args.e2e_copy_out, staged=args.e2e_staged,
                      ring=args.e2e_ring)
    clock_info = clocks.finish()

    # the secondary measurements: on the default run of one process only
    default_launch = not (args.block_size or args.two_launch or args.identity_tables or args.num_ctas
                          or args.seed not in (None, W_BASE_SEED))
    secondary = None
    peak, peak_kind = measured_hbm_peak()
    if world == 1 and args.config == "7b" and default_launch and not args.no_secondary and not args.no_graph:
        secondary = run_secondary(pkv, device, peak, st, ws)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    value = world * kv_bytes * args.steps / (ms_total / 1e3) / 1e9
    achieved = kv_bytes / (dec_mean / 1e3) / 1e9
    # the ncu record was taken on the default launch of the default inputs
    traffic = recorded_traffic(args.config + ("_shared" if args.shared else "")) if default_launch else None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_total / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "storage_dtype": "f16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config,
                   "seed": args.seed if args.seed is not None else W_BASE_SEED,
                   "num_seqs": wl.num_seqs, "num_heads": wl.num_heads, "num_kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "block_size": wl.block_size, "num_blocks": st["nb"],
                   "sum_context": int(sum(wl.context_lens)), "kv_bytes_per_step": kv_bytes,
                   **waste_pct(wl, MAX_CONTEXT[args.config]),
                   "tables": "identity (contiguous, in order)" if args.identity_tables else "shuffled pool",
                   "num_ctas": args.num_ctas or pkv.decode_default_ctas(wl.num_heads, wl.num_kv_heads,
                                                                        wl.head_dim, wl.block_size),
                   "l2": "no flush: the KV read per step (%.2f GB) is larger than L2 (129 MB)" % (kv_bytes / 1e9),
                   "parallelism": f"replicas x{world} (independent pools and sequences, no collective)"},
        "seqs_per_s_per_layer": round(world * wl.num_seqs * args.steps / (ms_total / 1e3), 1),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "gpu_launches": launches * world,
        "launch_mode": ("direct binding calls" if args.no_graph else
                        "DecodePlan launches, steps back to back on one stream (programmatic dependent launch: "
                        "each launch's prologue overlaps the previous launch's tail); CUDA events at the two ends "
                        "of the timed region only") +
                       ("; reshape_and_cache launch, then a read-only decode launch" if args.two_launch
                        else "; one decode launch per step that also writes the new tokens "
                             "(paged_attention_decode_append)"),
        "host_us_per_step": round(host_s / args.steps * 1e6, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": (("pkv_paged_attention_decode_shared (paged_decode_kernel, grouped: shared "
                                 "blocks read once per group of forks" + ("" if args.two_launch else
                                                                          ", writes the new tokens") + ")")
                                if args.shared else
                                "pkv_paged_attention_decode (paged_decode_kernel, merge fused)" if args.two_launch
                                else "pkv_paged_attention_decode_append (paged_decode_kernel: writes the new "
                                     "tokens, merge fused)"),
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "decode_ms_mean": round(dec_mean, 5),
                     "duration": ("the launch period over the timed region (K launches back to back, events at "
                                  "its ends)" if st["launches_per_step"] == 1 else
                                  "the decode launch on its own, between its own events"),
                     "decode_ms_isolated_median": round(dec_iso, 5)},
        "clocks": clock_info,
    }
    if e2e is not None:
        line["e2e"] = {"value": round(world * e2e["bytes"] / e2e["elapsed"] / 1e9, 2), "unit": UNIT,
                       "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                       "steps": e2e_steps, "warmup_steps": E2E_WARMUP, "step_us": e2e["step_us"],
                       "breakdown": e2e["breakdown"],
                       "output": ("D2H copy after the launch" if args.e2e_copy_out else
                                  "written by the kernel straight into the pinned host buffer over the CPU-GPU "
                                  "link (the plan's out is mapped host memory); no copy after the launch"),
                       "input": ("pkv_decode_plan_step: the region copied host->device, then the launch"
                                 if args.e2e_staged else
                                 "pkv_decode_plan_step_mapped: the kernel reads the region from pinned host memory "
                                 "over the CPU-GPU link (no copy in)"),
                       "staging": (f"{args.e2e_ring} pinned rows used in turn" if args.e2e_ring > 0 else
                                   "one pinned row per step") +
                                  " (tables and lengths rewritten by the block manager every step; queries and "
                                  "new rows drawn once)",
                       "includes": "host block manager append + table export into the step's pinned staging "
                                   "region (queries, new K/V, tables, lengths); one library call per step: the "
                                   "region's bytes into the GPU, the launch (append new tokens + attend), the "
                                   "output into host memory; the host waits for each step (polling an event); "
                                   "the next step's block-manager work overlaps this step's GPU work"}
    if secondary is not None:
        line["secondary"] = secondary
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(args.config, args.cpu_seconds, args.seed)
    if dist is not None:
        dist.destroy_process_group()
    return line


def run_layers(args):
    """A model's decode step over `--layers` layers, each with its own K/V
    pools (same tables: one block id spans all layers): one decode launch per
    layer (the one that also writes the layer's new token), all captured as
    one CUDA graph so that programmatic dependent launch lets each layer's
    prologue overlap the previous layer's tail.  value = KV bytes read by all
    layers per step / step time."""
    import torch
    import paged_kv_cache_152_gb300 as pkv
    import workloads as W

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from paged_kv_cache_152_gb300 import build as b
    b.build()
    pkv.load()
    st = build_state(args.config, device, block_size=args.block_size, seed=args.seed)
    wl, t = st["wl"], st["t"]
    L = args.layers
    shape = tuple(t["key_cache"].shape)
    caches = [(t["key_cache"], t["value_cache"])]
    for layer in range(1, L):
        caches.append((W.normal_fp16_large(shape, wl.seed * 1000 + 100 + 2 * layer, device),
                       W.normal_fp16_large(shape, wl.seed * 1000 + 101 + 2 * layer, device)))
    ws = pkv.new_workspace(wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                           args.num_ctas, device)
    plans = [pkv.DecodePlan(st["out"], t["query"], kc, vc, st["tables"], st["lens"], wl.scale, key=t["key"],
                            value=t["value"], num_ctas=args.num_ctas, workspace=ws, status=st["status"])
             for kc, vc in caches]
    stream = torch.cuda.current_stream()
    for _ in range(3):
        for pl in plans:
            pl.launch()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        for pl in plans:
            pl.launch()
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    assert int(st["status"].item()) == 0, pkv.status_string(int(st["status"].item()))
    steps = max(1, min(args.steps, 200))
    clocks = ClockSampler(0)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        g.replay()
        ev[i][1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    assert int(st["status"].item()) == 0, pkv.status_string(int(st["status"].item()))
    total_ms = e0.elapsed_time(e1)
    step_ms = statistics.fmean(a.elapsed_time(z) for a, z in ev)
    kv = wl.kv_read_bytes() * L
    peak, peak_kind = measured_hbm_peak()
    value = kv * steps / (total_ms / 1e3) / 1e9
    return {
        "metric": METRIC + " (model step over all layers)",
        "value": round(value, 2), "unit": UNIT, "n_gpus": 1, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / steps, 5), "higher_is_better": True, "dtype": "f32",
        "storage_dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config] + f"; {L} layers, each with its own pools",
                   "layers": L, "kv_bytes_per_step": kv, "block_size": wl.block_size,
                   "launch_mode": "one CUDA graph per step: one decode launch per layer (writes the layer's new "
                                  "token, then attends), programmatic dependent launch between layers"},
        "per_layer_us": round(step_ms * 1e3 / L, 3),
        "seqs_per_s_per_layer": round(wl.num_seqs * L * steps / (total_ms / 1e3), 1),
        "pct_of_peak": round(100 * value / peak, 2),
        "peak": peak, "peak_kind": peak_kind,
        "gpu_launches": L * steps,
        "clocks": clocks.finish(),
    }


def run_swap(args):
    """Swapping, measured on its own: the block manager swaps every sequence
    of the workload out to a page-locked host pool and back in; the kernel
    moves the blocks (one launch per direction).  The pair lists of one
    out/in cycle are replayed K times; the copy engine moving the same bytes
    as ONE contiguous buffer is timed beside it as the link's reference."""
    import numpy as np
    import torch
    import paged_kv_cache_152_gb300 as pkv

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from paged_kv_cache_152_gb300 import build as b
    b.build()
    pkv.load()
    st = build_state(args.config, device, block_size=args.block_size, seed=args.seed)
    wl, alloc, t = st["wl"], st["alloc"], st["t"]
    kc, vc = t["key_cache"], t["value_cache"]
    nh = st["nb"]
    hk = torch.empty_like(kc, device="cpu").pin_memory()
    hv = torch.empty_like(vc, device="cpu").pin_memory()
    alloc.host_pool(nh)
    h0 = time.perf_counter()
    out_pairs = alloc.swap_out(wl.batch)
    h1 = time.perf_counter()
    in_pairs = alloc.swap_in(wl.batch)
    h2 = time.perf_counter()
    d_out = torch.from_numpy(out_pairs.astype(np.int64)).to(device)
    d_in = torch.from_numpy(in_pairs.astype(np.int64)).to(device)
    block_bytes = kc[0].numel() * kc.element_size()
    moved = 2 * len(out_pairs) * block_bytes
    status = st["status"]
    stream = torch.cuda.current_stream()
    flat_dev = torch.empty(moved, dtype=torch.uint8, device=device)
    flat_host = torch.empty(moved, dtype=torch.uint8).pin_memory()

    def timed(fn, steps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, z in evs:
            a.record(stream)
            fn()
            z.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(z) for a, z in evs]

    ops = {
        "swap_out_kernel": lambda: pkv.swap_blocks(kc, vc, hk, hv, d_out, status=status),
        "swap_in_kernel": lambda: pkv.swap_blocks(hk, hv, kc, vc, d_in, status=status),
        "copy_engine_d2h": lambda: flat_host.copy_(flat_dev, non_blocking=True),
        "copy_engine_h2d": lambda: flat_dev.copy_(flat_host, non_blocking=True),
    }
    steps = max(1, min(args.steps, 50))
    clocks = ClockSampler(0)
    res = {}
    for name, fn in ops.items():
        timed(fn, max(3, args.warmup))
        if name == "swap_out_kernel":
            clocks.start()
        ms = timed(fn, steps)
        if name == "swap_in_kernel":
            clocks.stop()
        res[name] = {"ms_mean": round(statistics.fmean(ms), 4), "ms_median": round(statistics.median(ms), 4),
                     "GB/s": round(moved / (statistics.fmean(ms) / 1e3) / 1e9, 2)}
    assert int(status.item()) == 0, pkv.status_string(int(status.item()))
    launches = 2 * steps + 2 * max(3, args.warmup)
    return {
        "metric": "swap_blocks: device <-> page-locked host block copies, GB/s",
        "value": round(2 * moved * steps / ((res["swap_out_kernel"]["ms_mean"] + res["swap_in_kernel"]["ms_mean"])
                                            * steps / 1e3) / 1e9, 2),
        "unit": "GB/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup, "higher_is_better": True,
        "dtype": "u8", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config] + "; every sequence swapped out, then in",
                   "blocks_moved_per_direction": int(len(out_pairs)), "block_bytes_per_cache": block_bytes,
                   "bytes_per_direction": moved},
        "kernels": res,
        "kernel_vs_copy_engine": {
            "out": round(res["swap_out_kernel"]["GB/s"] / res["copy_engine_d2h"]["GB/s"], 3),
            "in": round(res["swap_in_kernel"]["GB/s"] / res["copy_engine_h2d"]["GB/s"], 3)},
        "block_manager_us": {"swap_out": round((h1 - h0) * 1e6, 1), "swap_in": round((h2 - h1) * 1e6, 1)},
        "gpu_launches": launches,
        "clocks": clocks.finish(),
    }


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and the reference arm)

def _oracle_worker(cfg, seed, seqs, barrier_, results):
    """Spawned process: build the workload (untimed), wait for the others at
    the barrier, run the oracle on `seqs`, report the elapsed seconds."""
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    import torch
    torch.set_num_threads(1)
    st = _oracle_state(cfg, seed)
    barrier_.wait()
    t0 = time.perf_counter()
    _oracle_decode(st, seqs)
    results.put(time.perf_counter() - t0)


_ORACLE_CACHE = {}


def _oracle_state(cfg, seed=None):
    """The workload at its decode step, with the oracle's own tables (CPU)."""
    if (cfg, seed) in _ORACLE_CACHE:
        return _ORACLE_CACHE[(cfg, seed)]
    import numpy as np
    import workloads as W
    from oracle.block_manager import BlockManagerModel
    wl = W.make(cfg) if seed is None else W.make(cfg, base=seed)
    model = BlockManagerModel(wl.num_blocks, wl.block_size, wl.free_order)
    W.replay(model, wl.ops)
    slots = [model.append_token(s)[0] for s in wl.batch]
    tables, lens = model.export(wl.batch, wl.max_blocks_per_seq())
    t = W.tensors(wl, "cpu")
    st = {"wl": wl, "tables": np.array(tables), "lens": np.array(lens), "slots": np.array(slots),
          "q": t["query"].numpy(), "k": t["key"].numpy(), "v": t["value"].numpy(),
          "kc": t["key_cache"].numpy(), "vc": t["value_cache"].numpy()}
    _ORACLE_CACHE[(cfg, seed)] = st
    return st


def _oracle_decode(st, seqs):
    """One oracle pass over `seqs`: write their new tokens, then attend."""
    from oracle import attention as OA
    from oracle import cache_ops as OC
    idx = list(seqs)
    OC.reshape_and_cache(st["k"][idx], st["v"][idx], st["kc"], st["vc"], st["slots"][idx])
    return OA.paged_decode_attention(st["q"], st["kc"], st["vc"], st["tables"], st["lens"], st["wl"].scale,
                                     seqs=idx)


def _seq_bytes(wl, seqs):
    return sum(2 * wl.context_lens[s] * wl.num_kv_heads * wl.head_dim * 2 for s in seqs)


def cpu_baseline(cfg, seconds, seed=None):
    """Oracle throughput on the host cores, on a bounded sample of the workload.

    Single core: the first sequences of the batch, as many as fit in about
    `seconds` / 2.  All cores: the whole batch split over a spawn pool of
    os.cpu_count() processes (single-threaded BLAS each), timed once.
    """
    import multiprocessing as mp
    st = _oracle_state(cfg, seed)
    wl = st["wl"]
    t0 = time.perf_counter()
    _oracle_decode(st, [0])
    one = max(time.perf_counter() - t0, 1e-4)
    k = int(max(1, min(wl.num_seqs, (seconds / 2) / one)))
    seqs = list(range(k))
    t0 = time.perf_counter()
    _oracle_decode(st, seqs)
    t1 = time.perf_counter() - t0
    v1 = _seq_bytes(wl, seqs) / t1 / 1e9
    cores = os.cpu_count() or 1
    vn, cores_used = None, 1
    if cores > 1:
        chunks = [list(range(i, wl.num_seqs, cores)) for i in range(cores)]
        chunks = [c for c in chunks if c]
        ctx = mp.get_context("spawn")
        bar = ctx.Barrier(len(chunks) + 1)
        results = ctx.Queue()
        procs = [ctx.Process(target=_oracle_worker, args=(cfg, seed, c, bar, results)) for c in chunks]
        for p in procs:
            p.start()
        bar.wait()
        t0 = time.perf_counter()
        for _ in procs:
            results.get()
        tn = time.perf_counter() - t0
        for p in procs:
            p.join()
        vn = _seq_bytes(wl, range(wl.num_seqs)) / tn / 1e9
        cores_used = len(chunks)
    best = vn if vn is not None else v1
    return {"value": round(best, 4), "unit": UNIT, "cores": cores_used if vn is not None else 1,
            "kind": "oracle",
            "sample": (f"all-cores: the whole {wl.num_seqs}-sequence batch split over {cores_used} spawned "
                       f"processes (1 BLAS thread each); single core: first {k} sequences"),
            "single_core_value": round(v1, 4),
            "ms_per_step_all_cores": round(_seq_bytes(wl, range(wl.num_seqs)) / (best * 1e9) * 1e3, 2)}


def run_reference(args):
    """The reference arm: the oracle as it stands, rank 0 only."""
    rank, _, world = dist_env()
    if rank != 0:
        return None
    st = _oracle_state(args.config, args.seed)
    wl = st["wl"]
    t0 = time.perf_counter()
    _oracle_decode(st, [0])
    one = max(time.perf_counter() - t0, 1e-4)
    budget = 90.0 / max(1, args.steps + args.warmup)      # whole run in about 1.5 minutes
    k = int(max(1, min(wl.num_seqs, budget / one)))
    seqs = list(range(k))
    for _ in range(args.warmup):
        _oracle_decode(st, seqs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_decode(st, seqs)
    el = time.perf_counter() - t0
    value = _seq_bytes(wl, seqs) * args.steps / el / 1e9
    sample = f"first {k} of {wl.num_seqs} sequences per step (all heads), 1 process"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config,
                       "seed": args.seed if args.seed is not None else W_BASE_SEED, "sample": sample},
            "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        line = run_reference(args)
    elif args.swap:
        line = run_swap(args)
    elif args.layers:
        line = run_layers(args)
    else:
        line = run_pkv(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
