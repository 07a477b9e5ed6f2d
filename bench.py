#!/usr/bin/env python
"""Benchmark of the masked-attention forward hot path on GB300.

One step = one pass of the hot path over one batch of synthetic input:
attn_build_tiles (slice list -> CSR tile metadata) + attn_fwd, and, for
workloads that define a KV split, the split partial forwards + attn_merge.
Default workload: the long dense causal problem with grouped-query heads
(S = 131072, 32 query heads over 8 KV heads, d = 128), run whole and as an
8-way KV split whose partials attn_merge combines -- the largest
configuration that fits one GPU.  Metric: valid-pair TFLOPS (4 d FLOPs per
unmasked query-key pair, summed over heads) per second of step time.  The
same JSON line carries, under "configs", the event-timed forward of the
other workloads (packed varlen documents, block-sparse strided grid,
video-generation slice list), measured in the same process.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Prints one JSON line.  N > 1 (torchrun) runs N independent replicas, one per
GPU; the path is not sharded (one GPU per problem), so scaling is "weak".
"""
from __future__ import annotations

import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

METRIC = "masked attn fwd TFLOPS (valid-pair FLOPs) and % of GB300 BF16 dense peak"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
E2E_SLOTS = 2                    # end-to-end device buffer sets (copies of one step overlap another's kernels)
# workloads whose forward is timed alongside the headline one (the "configs" key)
SIDE_WORKLOADS = ["varlen_causal", "block_sparse_strided", "video_gen"]
# a kernel timed for longer than this runs against the sustained tensor peak
# (the power cap settles in), a shorter one against the burst peak
SUSTAINED_AFTER_MS = 10.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gqa_causal")
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"],
                    help="fwd: the forward hot path (default); bwd: attn_bwd alone")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave out the forward timings of the other workloads (the 'configs' key)")
    ap.add_argument("--fwd-tile-q", type=int, default=256, choices=[256, 512],
                    help="query rows per forward work item: 256 = single-CTA kernel (default); "
                         "512 = CTA-pair kernel (two CTAs share each M=256 MMA; head dim 128)")
    ap.add_argument("--exp2-poly", type=int, default=0, choices=[0, 4, 8],
                    help="forward exponentials: 0 all on the special-function unit (default); "
                         "4 / 8 every 4th / 8th pair of a FULL tile on the FMA-pipe polynomial")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK, "fallback"


def slices_of(w):
    from block_sparse_attention_slice_gb300 import attn_slices_from_block_grid
    if w.grid is not None:
        return attn_slices_from_block_grid(w.grid, w.block, w.block)
    return w.slices


class Clocks:
    """Samples SM clock and clock-event reasons during the timed region.

    Reads NVML through ctypes (read-only queries) from a background thread
    every ~2 ms, so that even a timed region of a few milliseconds is
    covered; falls back to an ``nvidia-smi -lms 100`` child process."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        import ctypes
        import threading
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.proc, self.thread = None, None
        self.stop_flag = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            handle = ctypes.c_void_p()
            import torch
            uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle)) != 0:
                cnt = ctypes.c_uint(0)
                nv.nvmlDeviceGetCount_v2(ctypes.byref(cnt))
                if cnt.value != 1 or nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(handle)) != 0:
                    raise OSError("no NVML handle")
            mx = ctypes.c_uint(0)
            nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))
            self.max_mhz = float(mx.value)
            fn_reason = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons

            def loop():
                clk, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
                while not self.stop_flag.is_set():
                    if nv.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0:
                        self.samples.append(float(clk.value))
                    if fn_reason(handle, ctypes.byref(rs)) == 0:
                        self.reasons |= int(rs.value)
                    time.sleep(0.002)
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            self.source = "nvml"
        except (OSError, AttributeError):
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(cuda_index),
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
                     "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                     "clocks_event_reasons.hw_thermal_slowdown",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                time.sleep(0.3)
            except OSError:
                self.source = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
        elif self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            names = ["sw_power_cap", "hw_slowdown", "sw_thermal_slowdown", "hw_thermal_slowdown"]
            bits = [0x4, 0x8, 0x20, 0x40]
            for ln in out.strip().splitlines():
                f = [x.strip() for x in ln.split(",")]
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except (ValueError, IndexError):
                    continue
                for b, v in zip(bits, f[2:6]):
                    if v.lower().startswith("active"):
                        self.reasons |= b
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "samples": len(self.samples), "source": self.source,
                "reasons": sorted(n for b, n in self.REASONS.items() if self.reasons & b)}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def reduce_max(x: float, ws: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity for one rank)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def code_sha16(src: str) -> str:
    """First 16 hex digits of the SHA-256 of a source file's code: the text
    with `//` comments and blank lines removed, so that editing a comment does
    not disown a profile taken on the same compiled kernel."""
    lines = []
    for ln in open(src, encoding="utf-8"):
        cut = ln.find("//")
        if cut >= 0 and '"' not in ln[:cut]:
            ln = ln[:cut]
        ln = ln.rstrip()
        if ln:
            lines.append(ln)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def profile_traffic(kernel: str, workload: str, src: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current code of the kernel (its `code_sha256_16` line);
    else None."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(p):
        return None
    want = code_sha16(src)
    got, traffic = None, None
    for ln in open(p):
        if ln.startswith("code_sha256_16:"):
            got = ln.split(":", 1)[1].split()[0]
        if ln.startswith("dram_bytes_per_launch:"):
            traffic = float(ln.split(":", 1)[1].strip())
    return traffic if got == want else None


# ------------------------------------------------------------------ CPU oracle legs
def run_oracle_timed(w, qf, kf, vf, heads, rows_per_head):
    import oracle
    threads = max(1, len(os.sched_getaffinity(0)))
    if w.grid is not None:
        mask = lambda r: oracle.mask_rows_grid(w.grid, w.block, r, w.S)
    else:
        mask = lambda r: oracle.mask_rows(w.slices, r, w.S)
    rows = None if rows_per_head is None else {h: rows_per_head[h] for h in heads}
    rows_list = None if rows is None else [rows.get(h, np.zeros(0, np.int64)) for h in range(w.H)]
    t0 = time.perf_counter()
    res = oracle.oracle_attention(qf, kf, vf, w.scale, mask, rows=rows_list, heads=heads,
                                  threads=min(threads, len(heads)))
    dt = time.perf_counter() - t0
    pairs = 0
    for h, (rr, O, L) in res.items():
        M = mask(rr)
        pairs += int(M.sum())
    return dt, pairs, min(threads, len(heads))


def cpu_inputs(w):
    from block_sparse_attention_slice_gb300 import workloads as W
    q, k, v = W.draw_qkv(w.S, w.H, w.Hk, w.d, w.seed)
    f = lambda t: t.float().numpy().astype(np.float64)
    return f(q), f(k), f(v)


def sample_plan(w):
    """Bounded oracle sample of a workload: (heads, rows per head or None, text)."""
    threads = max(1, len(os.sched_getaffinity(0)))
    heads = list(range(min(w.H, threads)))
    if w.S <= 16384:
        return heads, None, f"all {w.S} rows of heads 0..{len(heads) - 1} ({len(heads)} of {w.H} heads)"
    from block_sparse_attention_slice_gb300.workloads import sample_rows
    n = 256
    rows = {h: sample_rows(w.S, h, n) for h in heads}
    return heads, rows, (f"{n} seeded sampled rows (default_rng(100+h)) of heads 0..{len(heads) - 1} "
                         f"({len(heads)} of {w.H} heads)")


def reference_arm(args, ws, rank):
    if rank != 0:
        return
    from block_sparse_attention_slice_gb300 import workloads as W
    w = W.ALL[args.workload]()
    qf, kf, vf = cpu_inputs(w)
    heads, rows, text = sample_plan(w)
    steps = args.steps if args.steps is not None else 10
    for _ in range(args.warmup):
        run_oracle_timed(w, qf, kf, vf, heads, rows)
    times, pairs, cores = [], 0, 1
    for _ in range(steps):
        dt, pairs, cores = run_oracle_timed(w, qf, kf, vf, heads, rows)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    val = 4 * w.d * pairs / (ms / 1e3) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "S": w.S, "H": w.H, "Hk": w.Hk, "d": w.d,
                       "sample": text},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": text},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def gpu_arm(args, ws, rank, local):
    import torch

    import block_sparse_attention_slice_gb300 as pkg
    from block_sparse_attention_slice_gb300 import binding as B
    from block_sparse_attention_slice_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.load()
    pkg.attn_set_exp2_poly(args.exp2_poly)
    w = W.ALL[args.workload]()
    sl = slices_of(w)
    q, k, v = W.draw_qkv(w.S, w.H, w.Hk, w.d, w.seed)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    prep = B.host_slices(sl)
    tq = args.fwd_tile_q
    ws_bytes = pkg.attn_tiles_workspace_bytes(sl, w.S, w.S, tq, 128)
    wsbuf = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((w.S, w.H, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.H, w.S), dtype=torch.float32, device=dev)
    split = []
    for s2 in w.kv_splits:
        p2 = B.host_slices(s2)
        b2 = torch.empty(pkg.attn_tiles_workspace_bytes(s2, w.S, w.S, tq, 128), dtype=torch.uint8, device=dev)
        split.append((s2, p2, b2, torch.empty((w.S, w.H, w.d), dtype=torch.float32, device=dev),
                      torch.empty((w.H, w.S), dtype=torch.float32, device=dev)))
    mout = torch.empty_like(out) if split else None
    mlse = torch.empty_like(lse) if split else None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    tiles0 = pkg.attn_build_tiles(sl, w.S, w.S, tq, ws=wsbuf, prepared=prep)
    nnz, nref, pairs_per_head, status = tiles0.totals()
    assert status == 0
    flops = 4.0 * w.d * pairs_per_head * w.H
    # kernels per step: the metadata build (one cooperative launch on these
    # workloads: every query tile's CTA fits at once) and the forward, for
    # the whole problem and for each KV-split part, plus the merge
    launches_per_step = 2 + (len(split) * 2 + 1 if split else 0)

    def step(qx, kx, vx, ev=None):
        if ev is not None:
            ev[0].record(stream)
        t = pkg.attn_build_tiles(sl, w.S, w.S, tq, ws=wsbuf, prepared=prep)
        if ev is not None:
            ev[1].record(stream)
        pkg.attn_fwd(qx, kx, vx, t, w.scale, out=out, lse=lse)
        if ev is not None:
            ev[2].record(stream)
        if split:
            parts = []
            for s2, p2, b2, o2, l2 in split:
                t2 = pkg.attn_build_tiles(s2, w.S, w.S, tq, ws=b2, prepared=p2)
                pkg.attn_fwd(qx, kx, vx, t2, w.scale, out=o2, lse=l2)
                parts.append((o2, l2))
            if ev is not None:
                ev[3].record(stream)
            pkg.attn_merge([p[0] for p in parts], [p[1] for p in parts], out=mout, lse=mlse)
        if ev is not None:
            ev[4].record(stream)

    steps = args.steps
    if steps is None:
        # a timed region of roughly two seconds, for the clock samples
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(3):
            step(qd, kd, vd)
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / 3
        steps = int(min(5000, max(10, 2.0 / max(per, 1e-6))))
    for _ in range(max(3, args.warmup)):
        step(qd, kd, vd)
    torch.cuda.synchronize()
    rc = pkg.attn_last_device_error()
    if rc != 0:
        raise RuntimeError(f"device status {rc} after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    clocks = Clocks(local) if rank == 0 else None
    barrier(ws)
    torch.cuda.synchronize()
    for i in range(steps):
        flush.zero_()                       # L2 flush between timed steps (not timed)
        step(qd, kd, vd, evs[i])
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop() if clocks else None
    rc = pkg.attn_last_device_error()
    if rc != 0:
        raise RuntimeError(f"device status {rc} in the timed region")
    step_ms = [e[0].elapsed_time(e[4]) for e in evs]
    build_ms = [e[0].elapsed_time(e[1]) for e in evs]
    fwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    ms = reduce_max(statistics.mean(step_ms), ws, dev)
    fwd_mean = statistics.mean(fwd_ms)
    split_flops = 0.0
    merge_ms = None
    if split:
        split_flops = flops     # the split partials cover exactly the same valid pairs
        merge_ms = statistics.mean([e[3].elapsed_time(e[4]) for e in evs])
    step_flops = flops + split_flops
    value = ws * step_flops / (ms / 1e3) / 1e12

    # ------------------------------------------------ end to end through host buffers
    # Every step copies its Q, K, V in from pinned host memory, runs the
    # whole path through the public API and reads O and lse back into pinned
    # host memory.  The kernels of all steps run in order on one compute
    # stream (each forward is a persistent kernel that wants every SM); the
    # copies in and out run on two copy streams, so step i+1's inputs arrive
    # and step i-1's result leaves while step i computes.  E2E_SLOTS sets of
    # device buffers rotate; events order each slot's reuse.  The value is
    # valid-pair FLOPs of all steps / the span from the first copy in to the
    # last copy out.
    e2e = None
    if not args.no_e2e:
        nslot = E2E_SLOTS
        s_in, s_comp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        slots = []
        for _ in range(nslot):
            sx = {"q": torch.empty_like(qd), "k": torch.empty_like(kd), "v": torch.empty_like(vd),
                  "ws": torch.empty_like(wsbuf), "out": torch.empty_like(out), "lse": torch.empty_like(lse),
                  "oh": torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
                  "lh": torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True),
                  "split": [(s2, p2, torch.empty_like(b2), torch.empty_like(o2), torch.empty_like(l2))
                            for s2, p2, b2, o2, l2 in split],
                  "in_done": torch.cuda.Event(), "comp_done": torch.cuda.Event(),
                  "out_done": torch.cuda.Event(), "used": False}
            if split:
                sx["mout"], sx["mlse"] = torch.empty_like(mout), torch.empty_like(mlse)
            slots.append(sx)

        def e2e_step(sx):
            # inputs in, once the slot's previous step no longer reads them
            if sx["used"]:
                s_in.wait_event(sx["comp_done"])
            with torch.cuda.stream(s_in):
                sx["q"].copy_(qh, non_blocking=True)
                sx["k"].copy_(kh, non_blocking=True)
                sx["v"].copy_(vh, non_blocking=True)
                sx["in_done"].record(s_in)
            # the path, once the inputs are in and the slot's previous result has left
            s_comp.wait_event(sx["in_done"])
            if sx["used"]:
                s_comp.wait_event(sx["out_done"])
            with torch.cuda.stream(s_comp):
                t = pkg.attn_build_tiles(sl, w.S, w.S, tq, ws=sx["ws"], prepared=prep)
                pkg.attn_fwd(sx["q"], sx["k"], sx["v"], t, w.scale, out=sx["out"], lse=sx["lse"])
                res, resl = sx["out"], sx["lse"]
                if split:
                    parts = []
                    for s2, p2, b2, o2, l2 in sx["split"]:
                        t2 = pkg.attn_build_tiles(s2, w.S, w.S, tq, ws=b2, prepared=p2)
                        pkg.attn_fwd(sx["q"], sx["k"], sx["v"], t2, w.scale, out=o2, lse=l2)
                        parts.append((o2, l2))
                    pkg.attn_merge([x[0] for x in parts], [x[1] for x in parts], out=sx["mout"], lse=sx["mlse"])
                    res, resl = sx["mout"], sx["mlse"]
                sx["comp_done"].record(s_comp)
            # the result out
            s_out.wait_event(sx["comp_done"])
            with torch.cuda.stream(s_out):
                sx["oh"].copy_(res, non_blocking=True)
                sx["lh"].copy_(resl, non_blocking=True)
                sx["out_done"].record(s_out)
            sx["used"] = True

        for i in range(2 * nslot):                       # warm-up
            e2e_step(slots[i % nslot])
        torch.cuda.synchronize()
        n_e2e = max(3 * nslot, min(steps, 48))
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize()
        es.record(s_in)
        s_comp.wait_event(es)
        s_out.wait_event(es)
        for i in range(n_e2e):
            e2e_step(slots[i % nslot])
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_comp)
        ee.record(s_out)
        ee.synchronize()
        barrier(ws)
        rc = pkg.attn_last_device_error()
        if rc != 0:
            raise RuntimeError(f"device status {rc} in the end-to-end region")
        # the last step's result, read back to the host, must equal the
        # device-timed step's (same inputs and kernels): a check of the
        # streams' and events' ordering (outside the timed region)
        last = slots[(n_e2e - 1) % nslot]
        ref_o, ref_l = (mout, mlse) if split else (out, lse)
        if not (torch.equal(last["oh"], ref_o.cpu()) and torch.equal(last["lh"], ref_l.cpu())):
            raise RuntimeError("end-to-end result differs from the device-timed step's")
        e2e_ms = reduce_max(es.elapsed_time(ee) / n_e2e, ws, dev)
        h2d = (q.numel() + k.numel() + v.numel()) * 2 + sum(int(x[1]) * 20 for x in [prep] + [s[1] for s in split])
        d2h = out.numel() * 2 + lse.numel() * 4
        e2e = {"value": ws * step_flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "buffer_slots": nslot, "streams": "one compute stream, copies in and out on two more",
               "steps": n_e2e,
               "l2": "not flushed: each step copies its inputs in from the host"}

    pk, pk_src = peaks()
    fwd_s = fwd_mean / 1e3
    achieved = flops / fwd_s / 1e12
    sustained = fwd_mean > SUSTAINED_AFTER_MS
    peak = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
    src = os.path.join(ROOT, "block_sparse_attention_slice_gb300", "csrc", "fwd_tcgen05.cu")
    # the committed counters were taken with the default exponential path
    traffic = profile_traffic("attn_fwd", w.name, src) if args.exp2_poly == 0 else None
    roof = {"kernel": "attn_fwd", "bound": "tensor", "achieved": achieved,
            "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": traffic,
            "peak_source": (f"bf16_tflops_sustained of {pk_src} (a {fwd_mean:.0f} ms kernel inside a "
                            f"seconds-long run)" if sustained else f"bf16_tflops (burst) of {pk_src}"),
            "frac_of_burst": achieved / pk["bf16_tflops"],
            "frac_of_sustained": achieved / pk["bf16_tflops_sustained"],
            "fwd_ms": fwd_mean, "build_ms": statistics.mean(build_ms),
            "algorithmic_flop_per_launch": flops}
    extra = {}
    if split:
        n = len(split)
        merge_bytes = w.S * w.H * (n * (4 * w.d + 4) + 2 * w.d + 4)
        extra["merge"] = {"kernel": "attn_merge", "bound": "hbm", "ms": merge_ms,
                          "achieved": merge_bytes / (merge_ms / 1e3) / 1e9,
                          "peak": pk["hbm_gbs"], "unit": "GB/s",
                          "frac": merge_bytes / (merge_ms / 1e3) / 1e9 / pk["hbm_gbs"],
                          "bytes": merge_bytes, "parts": n,
                          "peak_source": f"hbm_gbs of {pk_src}",
                          "traffic": profile_traffic("attn_merge", w.name, os.path.join(
                              ROOT, "block_sparse_attention_slice_gb300", "csrc", "merge.cu"))}
        extra["split_fwd_ms"] = statistics.mean([e[2].elapsed_time(e[3]) for e in evs])

    if not args.no_configs:
        extra["configs"] = side_workloads(pkg, W, dev, flush, pk, pk_src,
                                          [x for x in SIDE_WORKLOADS if x != args.workload], tq)
        barrier(ws)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        qf, kf, vf = (t.float().numpy().astype(np.float64) for t in (q, k, v))
        heads, rows, text = sample_plan(w)
        dt, sp, cores = run_oracle_timed(w, qf, kf, vf, heads, rows)
        cpu = {"value": 4 * w.d * sp / dt / 1e12, "unit": "TFLOP/s", "cores": cores,
               "kind": "oracle", "sample": text, "seconds": dt}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": steps,
                "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded numpy normals rounded to bf16)",
                "config": {"workload": w.name, "S": w.S, "H": w.H, "Hk": w.Hk, "d": w.d,
                           "valid_pairs_per_head": pairs_per_head, "tiles_nnz": nnz,
                           "kv_split_parts": len(split),
                           "step": ("build + forward of the whole problem, then build + forward of "
                                    f"each of the {len(split)} KV-split partials and attn_merge; "
                                    "FLOPs of both passes credited") if split else
                                   "build + forward",
                           "l2": "flushed between timed steps",
                           "exp2_poly": args.exp2_poly,
                           "fwd_kernel": ("CTA pair (512-row items, cta_group::2)" if tq == 512
                                          else "single CTA (256-row items)"),
                           "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
                "pct_of_bf16_peak": 100.0 * value / ws / pk["bf16_tflops"],
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * steps, "clocks": clk, **extra}
        print(json.dumps(line), flush=True)


def side_workloads(pkg, W, dev, flush, pk, pk_src, names, tq=256, reps=10):
    """Event-timed forward (inputs resident, L2 flushed before each launch) of
    each named workload: TFLOP/s on valid pairs and its fraction of the burst
    tensor peak (these kernels run for well under a second)."""
    import torch
    res = {}
    for name in names:
        w = W.ALL[name]()
        sl = slices_of(w)
        q, k, v = W.draw_qkv(w.S, w.H, w.Hk, w.d, w.seed)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        tiles = pkg.attn_build_tiles(sl, w.S, w.S, tq)
        nnz, _, pairs, status = tiles.totals()
        assert status == 0
        out = torch.empty((w.S, w.H, w.d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((w.H, w.S), dtype=torch.float32, device=dev)
        for _ in range(3):
            pkg.attn_fwd(qd, kd, vd, tiles, w.scale, out=out, lse=lse)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        torch.cuda.synchronize()
        for a, b in evs:
            flush.zero_()
            a.record()
            pkg.attn_fwd(qd, kd, vd, tiles, w.scale, out=out, lse=lse)
            b.record()
        torch.cuda.synchronize()
        if pkg.attn_last_device_error() != 0:
            raise RuntimeError(f"device status after the {name} forward")
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        tf = 4.0 * w.d * pairs * w.H / (ms / 1e3) / 1e12
        res[name] = {"workload": w.name, "kernel": "attn_fwd", "fwd_ms": ms, "achieved": tf,
                     "unit": "TFLOP/s", "peak": pk["bf16_tflops"],
                     "frac": tf / pk["bf16_tflops"], "peak_source": f"bf16_tflops (burst) of {pk_src}",
                     "valid_pairs_per_head": pairs, "tiles_nnz": nnz, "launches": reps,
                     "l2": "flushed before each launch"}
        del qd, kd, vd, out, lse, tiles
        torch.cuda.empty_cache()
    return res


def bwd_arm(args, ws, rank, local):
    """attn_bwd on one workload, inputs and forward results resident: valid
    pairs x 10 d FLOPs (2.5 x the forward's 4 d, the usual count for five
    GEMMs) per second of attn_bwd time."""
    import torch

    import block_sparse_attention_slice_gb300 as pkg
    from block_sparse_attention_slice_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg.load()
    w = W.ALL[args.workload]()
    sl = slices_of(w)
    q, k, v = W.draw_qkv(w.S, w.H, w.Hk, w.d, w.seed)
    rng = np.random.default_rng(w.seed + 1)
    do = torch.from_numpy(rng.standard_normal((w.S, w.H, w.d), dtype=np.float32)).to(torch.bfloat16)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    tiles = pkg.attn_build_tiles(sl, w.S, w.S)
    pairs = tiles.totals()[2]
    out, lse = pkg.attn_fwd(qd, kd, vd, tiles, w.scale)
    wsb = None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    steps = args.steps if args.steps is not None else 10
    for _ in range(max(3, args.warmup)):
        pkg.attn_bwd(qd, kd, vd, out, dod, lse, tiles, w.scale, grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    clocks = Clocks(local) if rank == 0 else None
    barrier(ws)
    torch.cuda.synchronize()
    for a, b in evs:
        flush.zero_()
        a.record()
        pkg.attn_bwd(qd, kd, vd, out, dod, lse, tiles, w.scale, grad_dtype=torch.bfloat16)
        b.record()
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop() if clocks else None
    if pkg.attn_last_device_error() != 0:
        raise RuntimeError("device status after the timed region")
    ms = reduce_max(statistics.mean(a.elapsed_time(b) for a, b in evs), ws, dev)
    flops = 10.0 * w.d * pairs * w.H
    pk, pk_src = peaks()
    val = flops / (ms / 1e3) / 1e12
    if rank == 0:
        print(json.dumps({
            "metric": "masked attn bwd TFLOPS (valid-pair, 2.5x forward FLOPs) and % of GB300 BF16 dense peak",
            "value": ws * val, "unit": "TFLOP/s", "n_gpus": ws, "steps": steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "S": w.S, "H": w.H, "Hk": w.Hk, "d": w.d,
                       "valid_pairs_per_head": pairs, "l2": "flushed between timed steps"},
            "roofline": {"kernel": "attn_bwd", "bound": "tensor", "achieved": val,
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": val / pk["bf16_tflops"],
                         "traffic": None, "peak_source": f"bf16_tflops (burst) of {pk_src}"},
            "gpu_launches": 5 * steps, "clocks": clk}), flush=True)   # delta, 2 x transposed lists, dK/dV, dQ


def main():
    args = parse()
    ws, rank, local = dist_init()
    if args.impl == "reference":
        reference_arm(args, ws, rank)
    elif args.which == "bwd":
        bwd_arm(args, ws, rank, local)
    else:
        gpu_arm(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
