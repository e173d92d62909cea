"""Benchmark of the R-KV compression event on B300.

One step = one pass of the whole hot path (importance, redundancy Gram,
normalise/blend/select, compaction + freed blocks) over one batch of
synthetic caches resident in HBM. Default workload: the Llama-3-8B-shaped
cache (32 layers x 8 KV heads, d=128, batch 1, N = 1152, budget 1024,
window 8, lambda 0.1): 32 compression events (sequence x layer) per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 0..4] [--impl rkv|reference]

Prints one JSON line. Timing: CUDA events on the launching stream. The timed
region runs K steps of rkv_compress (the public call; `value` and
`ms_per_step` come from these) and then K steps of the four stage calls with
an event between kernels (each kernel's duration, share and roofline
fraction). Before every step the caches are restored from a pristine copy,
L2 is flushed by reading a 512 MiB buffer (so that the restore's dirty lines
are written back there, and the flush leaves only clean lines) and the GPU
runs a short sleep kernel while the host enqueues the step (all outside the
event pairs); barrier + synchronize on both sides of the timed loop; max over
ranks. The same run then measures every workload (dense Gram and closed-form
redundancy) with fewer steps, under the key "workloads".
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "KV compression events/s (seq*layer)"
UNIT = "events/s"
KERNELS = ("rkv_importance", "rkv_redundancy", "rkv_select_compact")          # dense Gram or closed form
KERNELS_FUSED = ("rkv_importance_redundancy", "rkv_select_compact")           # closed form inside importance
METHODS = ("gram", "closed", "closed-fused")
SUFFIX = {"gram": "", "closed": "-closed-form", "closed-fused": "-closed-form-fused"}
KERNEL_SOURCES = {
    "rkv_importance": ("rkv_importance.cuh",),
    "rkv_importance_redundancy": ("rkv_importance.cuh",),
    "rkv_redundancy": ("rkv_redundancy.cuh",),
    "rkv_select_compact": ("rkv_select_compact.cuh", "rkv_select.cuh", "rkv_compact.cuh"),
}


def kernels_of(method: str) -> tuple:
    return KERNELS_FUSED if method == "closed-fused" else KERNELS
L2_FLUSH_BYTES = 512 << 20
SLEEP_CYCLES = 1_000_000  # ~0.5 ms at 2 GHz, outside the timed region


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


def launches_per_pass(shape: synthetic.Shape, method: str) -> int:
    """Kernels one pass of the event launches: one per stage (importance,
    redundancy, select + compact; with the fused closed form, importance and
    redundancy are one launch), except the dense Gram on an odd count of at
    least 17 key tiles of 128, which runs the CTA-pair kernel on the full
    256-row blocks and the single-CTA kernel on the half blocks (two
    launches)."""
    tiles = -(-shape.max_seq_len // 128)
    split = method == "gram" and tiles % 2 == 1 and tiles >= 17
    return len(kernels_of(method)) + (1 if split else 0)


def moved_rows(keep_idx: np.ndarray) -> int:
    """Kept rows that compaction must move (slot j holds token keep[j] != j)."""
    k = keep_idx.reshape(-1, keep_idx.shape[-1])
    slots = np.arange(k.shape[1], dtype=k.dtype)[None, :]
    return int(np.count_nonzero((k >= 0) & (k != slots)))


def algorithmic_work(shape: synthetic.Shape, seq_lens: np.ndarray, keep_idx: np.ndarray,
                     method: str = "gram") -> dict:
    """Per-launch algorithmic bytes / flops of each kernel (all events).
    Compaction counts the rows it must move (read + write of K and V), taken
    from the kept indices of the step, plus reading those indices."""
    d, H, Hq, w, L = shape.head_dim, shape.kv_heads, shape.q_heads, shape.window, shape.layers
    imp_bytes = red_flops = red_bytes = sel_bytes = 0.0
    for n in seq_lens.astype(np.float64):
        kb = min(n, shape.budget)
        imp_bytes += L * (n * H * d * 2 + w * Hq * d * 2 + n * H * 4 * 2)   # K read, Q read, I + 1/|k| written
        red_flops += L * (2.0 * n * n * d * H)                               # dense Gram, as contracted
        red_bytes += L * (n * H * d * 2 + n * H * 4 * 2)
        sel_bytes += L * (n * H * 4 * 2 + kb * H * 4)                        # I, R read; keep_idx written
    # select + compact: the score rows, the kept indices written, and the rows
    # that must move (read + write of K and V)
    cmp_bytes = sel_bytes + moved_rows(keep_idx) * 2.0 * 2 * d * 2
    out = {"rkv_select_compact": dict(bound="hbm", work=cmp_bytes, unit="GB/s")}
    if method == "closed-fused":
        # importance and the rank-one redundancy in one pass over K: the keys
        # and queries read once, I, 1/|k| and R written
        r_bytes = sum(L * n * H * 4.0 for n in seq_lens.astype(np.float64))
        out["rkv_importance_redundancy"] = dict(bound="hbm", work=imp_bytes + r_bytes, unit="GB/s")
    else:
        out["rkv_importance"] = dict(bound="hbm", work=imp_bytes, unit="GB/s")
        if method == "closed":
            # the rank-one identity: the keys and inverse norms read, R written
            out["rkv_redundancy"] = dict(bound="hbm", work=red_bytes, unit="GB/s")
        else:
            out["rkv_redundancy"] = dict(bound="tensor", work=red_flops, unit="TFLOP/s", bytes=red_bytes)
    return out


def job_throughput(local_ms: float, events_per_rank: int, world: int, dist=None, device="cpu"):
    """Whole-job events/s over `world` ranks that each compressed
    `events_per_rank` events: the slowest rank's time (max over ranks) divides
    the events of all ranks. Returns (value, max_ms)."""
    ms = float(local_ms)
    if dist is not None and world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return world * events_per_rank / (ms / 1e3), ms


def source_code_hash(text: str) -> str:
    """Hash of a C++/CUDA source with its comments and whitespace removed: a
    profile taken on the code stays valid when only comments change."""
    code = re.sub(r"//[^\n]*|/\*.*?\*/", " ", text, flags=re.S)
    return hashlib.sha256(" ".join(code.split()).encode()).hexdigest()[:16]


def kernel_source_hash(kernel: str) -> str:
    text = "".join(open(os.path.join(ROOT, "decode_kv_cache_05_b300", "csrc", f)).read()
                   for f in KERNEL_SOURCES[kernel])
    return source_code_hash(text)


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source and this workload; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(kernel)
    if not d or d.get("source_sha") != kernel_source_hash(kernel) or d.get("workload") != workload:
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            self.proc.wait()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [x for x in sm if x > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def run_reference(args) -> None:
    """The oracle (plain fp64 CPU code) timed on the host cores, each step a
    bounded sample of the same workload: one event (one layer of one
    sequence, all KV heads) of a CPU generation of it."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    shape = synthetic.WORKLOADS[args.workload]
    wl = synthetic.generate(args.workload, layers=1, batch=1, device="cpu")
    s = wl.shape
    op = oracle.problem(layers=1, batch=1, kv_heads=s.kv_heads, q_heads=s.q_heads, head_dim=s.head_dim,
                        max_seq_len=s.max_seq_len, budget=s.budget, window=s.window, mix_lambda=s.mix_lambda,
                        paged=s.paged, block_size=s.block_size, num_blocks=wl.num_blocks,
                        max_blocks=s.blocks_per_seq if s.paged else 0)
    k, v = synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache)
    q = synthetic.bf16_bits(wl.q_window)
    lens = wl.seq_lens.numpy()
    bt = None if wl.block_table is None else wl.block_table.numpy()
    closed = args.redundancy != "gram"
    for _ in range(args.warmup):
        oracle.compress(op, k.copy(), v.copy(), q, lens, bt, closed_form=closed)
    t = 0.0
    for _ in range(args.steps):
        kc, vc = k.copy(), v.copy()
        t0 = time.perf_counter()
        oracle.compress(op, kc, vc, q, lens, bt, closed_form=closed)
        t += time.perf_counter() - t0
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    value = args.steps / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": shape.name + SUFFIX[args.redundancy],
                   "redundancy": {"gram": "dense_gram", "closed": "closed_form",
                                  "closed-fused": "closed_form_fused"}[args.redundancy],
                   "sample": "1 event (layer 0 of sequence 0, all KV heads) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "1 event per step, CPU-generated copy of the workload's first layer"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def cpu_baseline(shape: synthetic.Shape, workload_id: int, budget_s: float = 12.0,
                 closed_form: bool = False) -> dict:
    """Oracle events/s on the host cores on a bounded sample (whole events of a
    CPU generation of the workload's first layer, as many as fit the budget);
    closed_form: the oracle's rank-one redundancy instead of the pairwise sum."""
    import oracle
    wl = synthetic.generate(workload_id, layers=1, batch=min(shape.batch, 4), device="cpu")
    s = wl.shape
    k, v = synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache)
    q = synthetic.bf16_bits(wl.q_window)
    lens = wl.seq_lens.numpy()
    bt = None if wl.block_table is None else wl.block_table.numpy()
    op = oracle.problem(layers=1, batch=s.batch, kv_heads=s.kv_heads, q_heads=s.q_heads, head_dim=s.head_dim,
                        max_seq_len=s.max_seq_len, budget=s.budget, window=s.window, mix_lambda=s.mix_lambda,
                        paged=s.paged, block_size=s.block_size, num_blocks=wl.num_blocks,
                        max_blocks=s.blocks_per_seq if s.paged else 0)
    events, t = 0, 0.0
    while t < budget_s:
        kc, vc = k.copy(), v.copy()
        t0 = time.perf_counter()
        oracle.compress(op, kc, vc, q, lens, bt, closed_form=closed_form)
        t += time.perf_counter() - t0
        events += s.batch
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": events / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "redundancy": "closed_form" if closed_form else "pairwise",
            "sample": f"{events} events (layer 0 of {s.batch} sequence(s), all KV heads, repeated), "
                      f"{t:.1f} s of CPU time, OpenMP over heads"}


class Step:
    """One workload resident on the device, with everything a timed step
    needs: the pristine caches to restore from, the outputs and workspace, and
    the L2 flush buffer."""

    def __init__(self, rkv, workload_id: int, dev, method: str, layers=None, batch=None):
        self.rkv = rkv
        self.wl = synthetic.generate(workload_id, device=dev, layers=layers, batch=batch)
        self.method = method
        code = {"gram": rkv.REDUNDANCY_GRAM, "closed": rkv.REDUNDANCY_CLOSED_FORM,
                "closed-fused": rkv.REDUNDANCY_CLOSED_FORM_FUSED}[method]
        self.p = rkv.problem_for(self.wl.shape, self.wl.num_blocks, redundancy=code)
        self.k_pristine, self.v_pristine = self.wl.k_cache.clone(), self.wl.v_cache.clone()
        self.out = rkv.allocate_outputs(self.p, dev)
        stride = rkv.score_stride(self.p)
        heads = self.p.heads
        ws = self.out["workspace"]
        plane = ws.numel() // 3
        self.imp = ws[:plane].view(torch.float32)[: heads * stride]
        self.red = ws[plane:2 * plane].view(torch.float32)[: heads * stride]
        self.inv = ws[2 * plane:].view(torch.float32)[: heads * stride]
        self.freed_ids = self.out["freed_ids"] if self.wl.shape.paged else None
        # L2 flush: the buffer is written once here; every flush only READS it,
        # so the lines it leaves in L2 are clean and the next step pays for no
        # write-back of the flush itself (the restore's dirty lines are pushed
        # out to HBM while the flush runs, outside the timed region)
        self.flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream()

    def stages(self, evs=None):
        """The kernels of rkv_compress, called through their C ABI entries so
        that each can be bracketed by events on the launching stream."""
        rkv, wl, out, st = self.rkv, self.wl, self.out, self.stream
        i = 0
        if evs:
            evs[i].record(st)
        if self.method == "closed-fused":
            rkv.rkv_importance_redundancy(self.p, wl.k_cache, wl.q_window, wl.seq_lens, wl.block_table, self.imp,
                                          self.inv, self.red)
        else:
            rkv.rkv_importance(self.p, wl.k_cache, wl.q_window, wl.seq_lens, wl.block_table, self.imp, self.inv)
            if evs:
                i += 1
                evs[i].record(st)
            rkv.rkv_redundancy(self.p, wl.k_cache, wl.seq_lens, wl.block_table, self.inv, self.red)
        if evs:
            i += 1
            evs[i].record(st)
        rkv.rkv_select_compact(self.p, self.imp, self.red, wl.seq_lens, wl.block_table, wl.k_cache, wl.v_cache,
                               out["keep_idx"], out["freed_off"], self.freed_ids, out["new_seq_lens"], None)
        if evs:
            i += 1
            evs[i].record(st)

    def api(self, evs=None):
        """The whole event through the public entry point (what a caller runs)."""
        wl, out = self.wl, self.out
        if evs:
            evs[0].record(self.stream)
        self.rkv.rkv_compress(self.p, wl.k_cache, wl.v_cache, wl.q_window, wl.seq_lens, wl.block_table,
                              out["keep_idx"], out["freed_off"], self.freed_ids, out["new_seq_lens"], None,
                              out["workspace"])
        if evs:
            evs[1].record(self.stream)

    def reset(self, hot_l2: bool = False):
        self.wl.k_cache.copy_(self.k_pristine)
        self.wl.v_cache.copy_(self.v_pristine)
        if not hot_l2:
            self.flush.max()  # a 512 MiB read: evicts (and writes back) everything the restore left in L2
        # keep the GPU busy while the host enqueues the step, so that host-side
        # launch latency never shows up between the step's kernel events
        torch.cuda._sleep(SLEEP_CYCLES)

    def free(self):
        for name in ("wl", "k_pristine", "v_pristine", "out", "imp", "red", "inv", "freed_ids", "flush"):
            setattr(self, name, None)


def measure(rkv, workload_id: int, dev, steps: int, warmup: int, method: str, world: int, dist, local: int,
            hot_l2: bool = False, layers=None, batch=None, keep: bool = False) -> dict:
    """Times `steps` steps of rkv_compress (the throughput) and then `steps`
    steps of the four stage calls with an event between kernels (each
    kernel's duration; events between kernels keep each launch from
    overlapping its neighbour, so these steps are slower). Barrier +
    synchronize around the timed loop, clocks sampled during it, max over
    ranks."""
    b = Step(rkv, workload_id, dev, method, layers=layers, batch=batch)
    for _ in range(warmup):
        b.reset(hot_l2)
        b.api()
        b.reset(hot_l2)
        b.stages()
    st = rkv.rkv_device_status()
    if st != rkv.RKV_OK:
        raise RuntimeError(f"device error during warm-up: {rkv.status_string(st)}")
    names = kernels_of(method)
    api_events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        for i in range(steps):
            b.reset(hot_l2)
            b.api(api_events[i])
        for i in range(steps):
            b.reset(hot_l2)
            b.stages(events[i])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    st = rkv.rkv_device_status()
    if st != rkv.RKV_OK:
        raise RuntimeError(f"device error in the timed region: {rkv.status_string(st)}")
    per_kernel = {kname: [ev[i].elapsed_time(ev[i + 1]) for ev in events] for i, kname in enumerate(names)}
    step_ms = [ev[0].elapsed_time(ev[1]) for ev in api_events]
    stage_step_ms = float(np.mean([ev[0].elapsed_time(ev[len(names)]) for ev in events]))
    shape = b.wl.shape
    value, total_ms = job_throughput(float(sum(step_ms)), shape.events * steps, world, dist, dev)
    keep_idx = b.out["keep_idx"].cpu().numpy()
    lens = b.wl.seq_lens.cpu().numpy()
    peaks = load_peaks()
    work = algorithmic_work(shape, lens, keep_idx, method=method)
    kern = {}
    for kname in names:
        avg_ms = float(np.mean(per_kernel[kname]))
        w = work[kname]
        achieved = w["work"] / (avg_ms / 1e3) / (1e12 if w["unit"] == "TFLOP/s" else 1e9)
        peak = peaks["bf16_tflops"] if w["unit"] == "TFLOP/s" else peaks["hbm_gbs"]
        kern[kname] = {"avg_ms": avg_ms, "bound": w["bound"], "achieved": achieved, "unit": w["unit"],
                       "frac": achieved / peak, "share": avg_ms / stage_step_ms}
    name = shape.name
    if layers is not None or batch is not None:
        name += f"-L{shape.layers}-B{shape.batch}"
    name += SUFFIX[method] + ("-hot-l2" if hot_l2 else "")
    res = {
        "workload": name, "events_per_step": shape.events, "value": value, "unit": UNIT,
        "ms_per_step": total_ms / steps, "ms_per_step_median": float(np.median(step_ms)),
        "ms_per_step_min": float(np.min(step_ms)), "ms_per_step_stage_calls": stage_step_ms,
        "steps": steps, "warmup": warmup, "gpu_launches": 2 * launches_per_pass(shape, method) * steps,
        "kernels": kern, "clocks": clocks.summary(), "wall_s_timed_loop": t_wall,
        "kv_gb_per_s_compacted": (moved_rows(keep_idx) * 2.0 * 2 * shape.head_dim * 2)
        / (kern["rkv_select_compact"]["avg_ms"] / 1e3) / 1e9,
        "compact_moved_rows_per_step": moved_rows(keep_idx),
    }
    if keep:
        res["_bench"] = b
    else:
        b.free()
        torch.cuda.empty_cache()
    return res


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--impl", choices=["rkv", "reference"], default="rkv")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--hot-l2", action="store_true",
                    help="no L2 flush between steps (inputs stay L2-resident): for the one-layer workload, "
                         "whose 11 MB fit in L2; never the headline number")
    ap.add_argument("--e2e-chunk", type=int, default=0,
                    help="layers per host<->device chunk of the e2e leg (0: the library's choice)")
    ap.add_argument("--redundancy", choices=list(METHODS), default="gram",
                    help="step 2 as the dense key Gram (default), the closed-form identity in a kernel of its "
                         "own, or the closed form fused into the importance kernel")
    ap.add_argument("--layers", type=int, default=None, help="shrink the workload to this many layers")
    ap.add_argument("--batch", type=int, default=None, help="shrink the workload to this many sequences")
    ap.add_argument("--workloads", default="0,1,2,3,4",
                    help="comma-separated workloads also measured in the same run (dense Gram and closed "
                         "form each, and the fused closed form on workloads 1 and 4; fewer steps, no CPU "
                         "baseline or e2e), reported under 'workloads'; 'none' to skip")
    ap.add_argument("--workload-steps", type=int, default=5)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        run_reference(args)
        return

    import decode_kv_cache_05_b300 as rkv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    shape = synthetic.WORKLOADS[args.workload]
    method = args.redundancy
    closed = method != "gram"
    # weak scaling: every rank compresses its own copy of the workload
    head = measure(rkv, args.workload, dev, args.steps, args.warmup, method, world, dist, local,
                   hot_l2=args.hot_l2, layers=args.layers, batch=args.batch, keep=not args.no_e2e)

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        b = head.pop("_bench")
        e2e = run_e2e(rkv, b.wl, b.p, b.k_pristine, b.v_pristine, b.out, args, dev, world, dist)
        b.free()
        torch.cuda.empty_cache()

    # ---- every workload (dense Gram and closed form) in the same run
    extra = []
    if args.workloads != "none" and not args.hot_l2 and args.layers is None and args.batch is None:
        for wid in [int(x) for x in args.workloads.split(",") if x.strip()]:
            for m in ("gram", "closed") + (("closed-fused",) if wid in (1, 4) else ()):
                if wid == args.workload and m == method:
                    continue  # the headline line itself
                extra.append(measure(rkv, wid, dev, args.workload_steps, 3, m, world, dist, local))

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peaks = load_peaks()
    kern = head["kernels"]
    dominant = max(kern, key=lambda k: kern[k]["avg_ms"])
    dk = kern[dominant]
    peak = peaks["bf16_tflops"] if dk["unit"] == "TFLOP/s" else peaks["hbm_gbs"]
    roofline = {"kernel": dominant, "bound": dk["bound"], "achieved": dk["achieved"], "peak": peak,
                "unit": dk["unit"], "frac": dk["achieved"] / peak,
                # the same kernel against the power-capped (seconds-long) bf16 rate, for context
                "frac_of_sustained": (dk["achieved"] / peaks["bf16_tflops_sustained"]
                                      if dk["unit"] == "TFLOP/s" and peaks.get("bf16_tflops_sustained") else None),
                "traffic": (None if (args.hot_l2 or args.layers or args.batch)
                            else ncu_traffic(dominant, head["workload"])),
                "peak_source": f"{peaks['source']} ({'bf16 burst' if dk['unit'] == 'TFLOP/s' else 'HBM copy'})"}
    # DRAM bytes per launch of the other kernels, where an ncu capture of the
    # current source on this workload exists (compaction's writes partly reach
    # HBM only after the kernel ends, when later traffic evicts them from L2)
    for kname in kern:
        t = None if (args.hot_l2 or args.layers or args.batch) else ncu_traffic(kname, head["workload"])
        kern[kname]["ncu_dram_bytes_per_launch"] = t

    cpu = cpu_closed = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(shape, args.workload, closed_form=closed)
        if not closed:
            # the oracle with the rank-one redundancy as well: the CPU's best case
            cpu_closed = cpu_baseline(shape, args.workload, budget_s=5.0, closed_form=True)

    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "ms_per_step_median": head["ms_per_step_median"], "ms_per_step_min": head["ms_per_step_min"],
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": head["workload"],
                   "redundancy": {"gram": "dense_gram", "closed": "closed_form",
                                  "closed-fused": "closed_form_fused"}[method], "layers": args.layers or shape.layers,
                   "batch": args.batch or shape.batch,
                   "kv_heads": shape.kv_heads, "q_heads": shape.q_heads, "head_dim": shape.head_dim,
                   "max_seq_len": shape.max_seq_len, "budget": shape.budget, "window": shape.window,
                   "mix_lambda": shape.mix_lambda, "layout": "paged16" if shape.paged else "contiguous",
                   "events_per_step": head["events_per_step"],
                   "l2": ("hot (no flush; inputs L2-resident)" if args.hot_l2
                          else "flushed before every step by reading a 512 MiB buffer (clean lines)"),
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "cpu_baseline_closed_form": cpu_closed,
        "e2e": e2e,
        "gpu_launches": head["gpu_launches"],
        "ms_per_step_stage_calls": head["ms_per_step_stage_calls"],
        "clocks": head["clocks"],
        "kernels": kern,
        "kv_gb_per_s_compacted": head["kv_gb_per_s_compacted"],
        "compact_moved_rows_per_step": head["compact_moved_rows_per_step"],
        "wall_s_timed_loop": head["wall_s_timed_loop"],
        "workloads": extra,
    }
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def run_e2e(rkv, wl, p, k_pristine, v_pristine, out, args, dev, world, dist) -> dict:
    """The public host-memory call, rkv_compress_host: per step it uploads the
    cache and queries from page-locked host memory, compresses and downloads
    the compacted cache, kept indices, freed blocks and new lengths; the
    library overlaps the chunked copies of both directions with the kernels.
    Events on the caller's stream bracket the steps (the call makes that
    stream wait for its last download)."""
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    hk, hv, hq, hl = pin(k_pristine), pin(v_pristine), pin(wl.q_window), pin(wl.seq_lens)
    ht = pin(wl.block_table) if wl.block_table is not None else None
    rk, rv = torch.empty_like(hk).pin_memory(), torch.empty_like(hv).pin_memory()
    rkeep = torch.empty(out["keep_idx"].shape, dtype=torch.int32).pin_memory()
    roff = torch.empty(out["freed_off"].shape, dtype=torch.int32).pin_memory()
    rids = torch.empty(out["freed_ids"].shape, dtype=torch.int32).pin_memory() if ht is not None else None
    rlen = torch.empty(out["new_seq_lens"].shape, dtype=torch.int32).pin_memory()
    ws = torch.empty(rkv.host_workspace_size(p, args.e2e_chunk), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    h2d = sum(t.numel() * t.element_size() for t in (hk, hv, hq, hl) + ((ht,) if ht is not None else ()))
    d2h = sum(t.numel() * t.element_size() for t in (rk, rv, rkeep, roff, rlen) + ((rids,) if ht is not None else ()))

    def one():
        rkv.rkv_compress_host(p, hk, hv, rk, rv, hq, hl, ht, rkeep, roff, rids, rlen, None, ws,
                              chunk_layers=args.e2e_chunk, stream=stream)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    value, ms = job_throughput(e0.elapsed_time(e1), wl.shape.events * args.steps, world, dist, dev)
    st = rkv.rkv_device_status()
    if st != rkv.RKV_OK:
        raise RuntimeError(f"device error in the e2e loop: {rkv.status_string(st)}")
    return {"value": value, "unit": UNIT, "call": "rkv_compress_host", "chunk_layers": args.e2e_chunk,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / args.steps}


if __name__ == "__main__":
    main()
