"""Benchmark of the DSA indexer hot path on GB300.

One step = one decode step of the 32-sequence batch (context lengths
alternating 4500 / 10000, 1 query each, 64 index heads x 128 dims, top-512,
fp8 e4m3 paged keys in blocks of 64): idx_store_keys of the step's 32 new keys
followed by idx_score_topk_decode over every cached key.  The metric is keys
scored and selected per second (232,000 keys per step); microseconds per step
are reported beside it.  Inputs are seeded synthetic data resident in HBM; 9
copies of the paged pool (275 MB, more than twice the L2) are rotated so that
every step reads its keys from HBM.

Also reported, as nested objects of the same JSON line: the long-context decode
batch (8 x 131072 + 1 x 1048576 keys, top-1024) and the 8192-query causal
prefill chunk over 22000 keys (top-1024), each with its own roofline.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch with torch.distributed.run; every rank runs an independent
replica on its own GPU (the indexer has no exchange step on one node).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "indexer keys scored+selected/s (decode, 32 seqs x 4500/10000 keys, top-512, fp8)"
UNIT = "keys/s"
KEY_BYTES_FP8 = 132          # one fp8 index-key record: 128 e4m3 codes + fp32 scale
N_POOL_COPIES = 9

# DRAM bytes per launch of the dominant kernels from ncu captures
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by workload, with the
# hash of the measured kernel's code (its translation unit and every header it
# includes, comments left out) when they were taken; a stale hash reports null.
NCU_TRAFFIC = {
    ("decode", "cd4902da1e770c88"): 31444992 + 0,
    ("longctx", "cd4902da1e770c88"): 277246976 + 2784256,
    ("prefill", "9a835175a16cef1b"): 139506432 + 536455936,   # the scoring kernel
}
KERNEL_TU = {"decode": "decode.cu", "longctx": "decode.cu", "prefill": "prefill.cu"}


def _code_only(text: str) -> str:
    """A source with its comments and blank lines removed (string literals in
    these sources hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(tu: str) -> str:
    """sha256 (first 16 hex digits) of a kernel translation unit and the
    closure of the quoted headers it includes (csrc/ and include/), comments
    and blank lines left out."""
    dirs = [os.path.join(ROOT, "sparse_attention_top_idx_gb300", "csrc"), os.path.join(ROOT, "include")]
    seen, todo = [], [tu]
    while todo:
        name = todo.pop()
        if name in seen:
            continue
        path = next((os.path.join(d, name) for d in dirs if os.path.exists(os.path.join(d, name))), None)
        if path is None:
            continue
        seen.append(name)
        with open(path) as f:
            for line in f:
                t = line.strip()
                if t.startswith("#include \""):
                    todo.append(t.split('"')[1])
    h = hashlib.sha256()
    for name in sorted(seen):
        path = next(os.path.join(d, name) for d in dirs if os.path.exists(os.path.join(d, name)))
        h.update(name.encode())
        with open(path) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_of(workload: str):
    return NCU_TRAFFIC.get((workload, kernel_source_hash(KERNEL_TU[workload])))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU is under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def setup_dist(n_gpus: int):
    """Rank, world size, local rank and the process group of a torchrun launch
    (replicas: the group only carries the barrier and the max-over-ranks of
    the timings).  NCCL on GPUs; gloo where no GPU is present."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local, dist


def whole_job_rate(world: int, keys_per_rank: int, ms_per_step: float) -> float:
    """Keys scored and selected per second by all ranks together: every rank
    processes keys_per_rank keys per step, and a step takes the slowest
    rank's time."""
    return world * keys_per_rank / (ms_per_step * 1e-3)


def max_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------------------
# decode workload
# ----------------------------------------------------------------------------

class DecodeBench:
    def __init__(self, W, device, copies: int):
        import torch
        from sparse_attention_top_idx_gb300 import dsaidx
        from sparse_attention_top_idx_gb300.host import bf16_tensor
        self.W = W
        self.device = device
        self.dsaidx = dsaidx
        B, k = W.batch, W.topk
        k_all = bf16_tensor(W.all_keys(), device)
        slots_all = torch.from_numpy(W.all_slots()).to(device)
        self.caches = []
        for _ in range(copies):
            c = dsaidx.IndexCache.allocate(W.num_blocks, W.bs, dsaidx.FP8, device=device, fill=0)
            dsaidx.store_keys(c, k_all, slots_all)
            self.caches.append(c)
        del k_all
        # the step's new keys: the last position of every sequence
        last = np.concatenate([np.cumsum(W.seq_lens) - 1])
        self.new_k = bf16_tensor(W.all_keys()[last], device)
        self.new_slots = slots_all[torch.from_numpy(last).to(device)].contiguous()
        self.q = bf16_tensor(W.q, device)
        self.w = torch.from_numpy(W.w).to(device)
        self.bt = torch.from_numpy(W.block_table).to(device)
        self.sl = torch.tensor(W.seq_lens, dtype=torch.int32, device=device)
        self.msl = W.max_seq_len
        self.ws = dsaidx.new_workspace(dsaidx.workspace_bytes_decode(self.caches[0], B, self.msl, W.H, k),
                                       device)
        self.out = torch.empty((B, k), dtype=torch.int32, device=device)
        self.keys = int(sum(W.seq_lens))

    def score(self, i):
        c = self.caches[i % len(self.caches)]
        self.dsaidx.score_topk_decode(c, self.q, self.w, self.bt, self.sl, self.msl, self.W.topk, self.out,
                                      self.ws)

    def step(self, i, ev=None):
        c = self.caches[i % len(self.caches)]
        self.dsaidx.store_keys(c, self.new_k, self.new_slots)
        if ev is not None:
            ev[0].record()
        self.score(i)
        if ev is not None:
            ev[1].record()

    def algo_bytes(self):
        W = self.W
        return (self.keys * KEY_BYTES_FP8 + W.q.nbytes + W.w.nbytes + W.batch * W.topk * 4
                + W.block_table.nbytes)


def _timing_events(n):
    """Event pairs that can be recorded inside a captured graph (external
    record nodes); None when this PyTorch cannot make them."""
    import torch
    try:
        return [(torch.cuda.Event(enable_timing=True, external=True),
                 torch.cuda.Event(enable_timing=True, external=True)) for _ in range(n)]
    except TypeError:
        return None


def capture(fn, steps, start, device, evs=None):
    """Capture `steps` calls fn(i, ev) into one CUDA graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.graph(g, stream=side):
        for i in range(steps):
            fn(start + i, evs[i] if evs else None)
    torch.cuda.current_stream(device).wait_stream(side)
    return g


EAGER = False   # --eager: issue the timed steps call by call (for profiler runs)
E2E_REPLAYS = 5  # replays of the end-to-end graph; the median is reported

# fp8-vs-bf16 top-512 overlap the pages report for their synthetic needle test
# ("The Hypothesis That Refused to Die", section "Message 12994: The Synthetic
# Test"): context length -> (Jaccard, positions lost); context only, other data.
PAGES_JACCARD_TOP512 = {2000: (0.395, 222), 4500: (0.382, 229), 10000: (0.299, 276), 22000: (0.267, 296)}


def time_steps(bench, steps, warmup, dist, device):
    """W warm-up steps, then exactly K timed steps replayed from one CUDA graph
    between barriers and synchronisations; per-step events around the scoring
    kernel give its launch durations.  With --eager the steps are issued call
    by call instead (profiler runs)."""
    import torch
    for i in range(warmup):
        bench.step(i)
    torch.cuda.synchronize(device)
    if EAGER:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize(device)
        t0.record()
        for i in range(steps):
            bench.step(warmup + i, evs[i])
        t1.record()
        torch.cuda.synchronize(device)
        barrier(dist)

        class _Replay:
            def replay(self):
                for i in range(steps):
                    bench.step(warmup + i)
        return t0.elapsed_time(t1), [a.elapsed_time(b) for a, b in evs], _Replay()
    # the timed graph has no event node between a step's two kernels, so the
    # decode kernel's set-up may overlap the key store (programmatic launch)
    g = capture(bench.step, steps, warmup, device)
    g.replay()                                # untimed: first replay uploads the graph
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(device)
    t0.record()
    g.replay()
    t1.record()
    torch.cuda.synchronize(device)
    barrier(dist)
    total_ms = t0.elapsed_time(t1)
    # the scoring kernel's durations: the same steps in a second graph with
    # events recorded around every scoring kernel
    kern_ms = None
    evs = _timing_events(steps)
    if evs is not None:
        try:
            ge = capture(bench.step, steps, warmup, device, evs)
            ge.replay()
            torch.cuda.synchronize(device)
            ge.replay()
            torch.cuda.synchronize(device)
            kern_ms = [a.elapsed_time(b) for a, b in evs]
            del ge
        except RuntimeError:
            kern_ms = None
    if kern_ms is None:
        # scoring kernels alone, back to back from a graph, same rotation
        gk = capture(lambda i, ev: bench.score(i), steps, warmup, device)
        gk.replay()
        torch.cuda.synchronize(device)
        t0.record()
        gk.replay()
        t1.record()
        torch.cuda.synchronize(device)
        kern_ms = [t0.elapsed_time(t1) / steps] * steps
    return total_ms, kern_ms, g


def load_padding(graph, seconds, device):
    """Keep replaying the timed graph (untimed) so the clock sampler sees the
    same load for long enough to take samples."""
    import torch
    t_end = time.time() + seconds
    while time.time() < t_end:
        graph.replay()
        torch.cuda.synchronize(device)


def pack_pinned(tensors, device, align=256, pin=True):
    """One pinned host buffer and one device buffer holding `tensors` back to
    back (each at an `align`-byte offset), and device views of every part, so a
    step's inputs cross to the device in a single copy.  Returns (host, dev,
    views)."""
    import torch
    offs, o = [], 0
    for t in tensors:
        o = (o + align - 1) // align * align
        offs.append(o)
        o += t.numel() * t.element_size()
    host = torch.empty(o, dtype=torch.uint8)
    if pin:
        host = host.pin_memory()
    dev = torch.empty(o, dtype=torch.uint8, device=device)
    views = []
    for t, off in zip(tensors, offs):
        n = t.numel() * t.element_size()
        host[off:off + n].copy_(t.detach().cpu().contiguous().reshape(-1).view(torch.uint8))
        views.append(dev[off:off + n].view(t.dtype).view(t.shape))
    return host, dev, views


def e2e_decode(bench, steps, warmup, device):
    """Same decode step through the public API from pinned host memory: every
    step copies the step's inputs host->device (queries, head weights, sequence
    lengths, the new keys and their slots, packed in one pinned buffer and sent
    as one copy), stores the keys, scores and selects, and copies the selected
    indices back to the host.  The copies are the library's copy kernel
    (idx_copy: the GPU reads and writes the pinned buffers over the host link,
    launched like the score calls' kernels); the same steps with the copy
    engine (cudaMemcpyAsync through PyTorch) are timed beside it.  Timed two
    ways: replayed from a CUDA graph (how a serving decode loop issues it;
    E2E_REPLAYS replays of the K steps, the median reported) and issued eagerly
    from Python call by call."""
    import torch
    W = bench.W
    h_in, d_in, (d_q, d_w, d_sl, d_k, d_s) = pack_pinned(
        [bench.q, bench.w, bench.sl, bench.new_k, bench.new_slots], device)
    h_out = torch.empty_like(bench.out, device="cpu").pin_memory()
    h2d = h_in.numel()
    d2h = h_out.numel() * h_out.element_size()
    ds = bench.dsaidx

    def make_one(engine):
        def one(i, ev=None):
            c = bench.caches[i % len(bench.caches)]
            if engine:
                d_in.copy_(h_in, non_blocking=True)
            else:
                ds.copy(d_in, h_in)
            ds.store_keys(c, d_k, d_s)
            ds.score_topk_decode(c, d_q, d_w, bench.bt, d_sl, bench.msl, W.topk, bench.out, bench.ws)
            if engine:
                h_out.copy_(bench.out, non_blocking=True)
            else:
                ds.copy(h_out, bench.out)
        return one

    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    res = {}
    for engine in (False, True):
        one = make_one(engine)
        for i in range(warmup):
            one(i)
        torch.cuda.synchronize(device)
        g = capture(one, steps, warmup, device)
        g.replay()
        torch.cuda.synchronize(device)
        reps = []
        for _ in range(E2E_REPLAYS):
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize(device)
            reps.append(a.elapsed_time(b) / steps)
        del g
        a.record()
        for i in range(steps):
            one(warmup + i)
        b.record()
        torch.cuda.synchronize(device)
        res[engine] = (float(np.median(reps)), a.elapsed_time(b) / steps, reps)
    # the last step's indices, copied by the kernel, equal the device's
    assert torch.equal(h_out, bench.out.cpu())
    return res[False][0], res[False][1], h2d, d2h, res[False][2], res[True][0]


def roofline_hbm(algo_bytes, kern_ms, peak_gbs, traffic):
    avg_ms = float(np.mean(kern_ms))
    ach = algo_bytes / (avg_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": peak_gbs, "unit": "GB/s",
            "frac": round(ach / peak_gbs, 4), "traffic": traffic,
            "kernel_us": round(avg_ms * 1e3, 3), "algorithmic_bytes": int(algo_bytes)}


def bench_long_context(device, steps, warmup, peaks):
    import torch
    from sparse_attention_top_idx_gb300 import workloads as wl
    W = wl.long_context()
    b = DecodeBench(W, device, copies=2)     # 277 MB per copy: larger than L2
    total_ms, kern_ms, g = time_steps(b, steps, warmup, None, device)
    del g
    tr = traffic_of("longctx")
    out = {"workload": W.name, "keys_per_step": b.keys, "ms_per_step": round(total_ms / steps, 5),
           "value": round(b.keys / (total_ms / steps * 1e-3), 1), "unit": UNIT,
           "roofline": roofline_hbm(b.algo_bytes(), kern_ms, peaks["hbm_gbs"], tr)}
    del b
    torch.cuda.empty_cache()
    return out


_TENSOR_PEAKS = None


def tensor_peaks():
    """Dense tcgen05.mma throughput measured on this GPU by the probe library
    (peak/mma_peak.cu): kind::f8f6f4 e4m3 as a burst (one ~5 ms launch) and
    sustained (~0.8 s of launches), kind::f16 bf16 as a burst (checks the
    method against the cuBLAS bf16 figure).  Each run first checks the
    accumulator against its exact value.  Falls back to 2 x the measured
    cuBLAS bf16 peak if the probe cannot run."""
    global _TENSOR_PEAKS
    if _TENSOR_PEAKS is not None:
        return _TENSOR_PEAKS
    import ctypes
    from sparse_attention_top_idx_gb300 import build as bld
    try:
        lib = ctypes.CDLL(bld.build_peak())
        lib.mma_peak_run.argtypes = [ctypes.c_int, ctypes.c_longlong, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
        res = {}
        for name, fp8, iters, launches in (("fp8_tflops", 1, 20000, 1), ("fp8_tflops_sustained", 1, 100000, 30),
                                           ("bf16_tflops_probe", 0, 20000, 1)):
            tf, ms = ctypes.c_double(), ctypes.c_double()
            rc = lib.mma_peak_run(fp8, iters, launches, ctypes.byref(tf), ctypes.byref(ms))
            if rc != 0:
                raise RuntimeError("mma_peak_run rc %d" % rc)
            res[name] = round(tf.value, 1)
        res["source"] = "measured fp8 tcgen05 probe (burst), accumulator checked"
    except Exception as ex:   # no GPU path for the probe: the documented fallback
        pk = measured_peaks()
        res = {"fp8_tflops": round(2.0 * pk["bf16_tflops"], 1), "fp8_tflops_sustained": None,
               "bf16_tflops_probe": None, "source": "2 x measured cuBLAS bf16 (probe failed: %s)" % ex}
    _TENSOR_PEAKS = res
    return res


def bench_prefill(device, steps, warmup, peaks):
    import torch
    from sparse_attention_top_idx_gb300 import dsaidx
    from sparse_attention_top_idx_gb300 import workloads as wl
    from sparse_attention_top_idx_gb300.host import bf16_tensor, build_cache
    W = wl.prefill_chunk()
    cache = build_cache(W, dsaidx.FP8, device=device)
    T, k = W.total_q, W.topk
    q = bf16_tensor(W.q, device)
    w = torch.from_numpy(W.w).to(device)
    cu = torch.from_numpy(W.cu_seqlens_q()).to(device)
    sl = torch.tensor(W.seq_lens, dtype=torch.int32, device=device)
    bt = torch.from_numpy(W.block_table).to(device)
    ws = dsaidx.new_workspace(dsaidx.workspace_bytes_prefill(cache, 1, T, W.max_seq_len, W.H, k), device)
    oi = torch.empty((T, k), dtype=torch.int32, device=device)
    for _ in range(warmup):
        dsaidx.score_topk_prefill(cache, q, w, cu, sl, bt, W.max_seq_len, k, oi, ws)
    torch.cuda.synchronize(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    # per-kernel events on the call's stream: the scoring kernel, then the row select
    dsaidx.kernel_timing(2 * steps)
    a.record()
    for _ in range(steps):
        dsaidx.score_topk_prefill(cache, q, w, cu, sl, bt, W.max_seq_len, k, oi, ws)
    b.record()
    torch.cuda.synchronize(device)
    times = dsaidx.kernel_times(2 * steps)
    dsaidx.kernel_timing(0)
    ms = a.elapsed_time(b) / steps
    score_ms = float(np.mean(times[0::2])) if len(times) >= 2 else ms
    select_ms = float(np.mean(times[1::2])) if len(times) >= 2 else 0.0
    pairs = int(np.sum(W.row_pos() + 1))
    flops = 2.0 * pairs * W.H * W.d
    tp = tensor_peaks()
    fp8_peak = tp["fp8_tflops"]
    ach = flops / (score_ms * 1e-3) / 1e12
    out = {"workload": W.name, "pairs_per_step": pairs, "ms_per_step": round(ms, 4),
           "value": round(pairs / (ms * 1e-3), 1), "unit": "query-key pairs/s",
           "kernels_us": {"score": round(score_ms * 1e3, 1), "select": round(select_ms * 1e3, 1)},
           "roofline": {"bound": "tensor", "achieved": round(ach, 1), "peak": round(fp8_peak, 1),
                        "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 4),
                        "traffic": traffic_of("prefill"),
                        "kernel_us": round(score_ms * 1e3, 1),
                        "algorithmic_flop": flops,
                        "whole_call_frac": round(flops / (ms * 1e-3) / 1e12 / fp8_peak, 4),
                        "note": "the scoring kernel (events around its launch); peak: " + tp["source"]},
           "tensor_peaks": tp}
    del cache, ws
    torch.cuda.empty_cache()
    return out


def bench_precision(device):
    """Key formats against bf16 keys on the precision workload (4 sequences of
    2000 / 4500 / 10000 / 22000 keys, one query each, planted needle), from the
    GPU's own outputs: fp8 keys, fp8 keys after the fp4 round trip ("fp4"),
    and the same with the Walsh-Hadamard rotation of keys (store) and queries
    (caller side, fp64 on the device) ("rot_fp4").  Per format: the needle's
    rank in each top-k (None: not selected), the Jaccard overlap with the
    bf16 index set and the bf16 positions it lost, at top-512 and top-1024.
    The pages' numbers for their own synthetic test are attached as context."""
    import torch
    from sparse_attention_top_idx_gb300 import dsaidx
    from sparse_attention_top_idx_gb300 import workloads as wl
    from sparse_attention_top_idx_gb300.host import bf16_tensor, build_cache, hadamard_rotate_bf16
    rows = []
    formats = (("bf16", dsaidx.BF16, False, False), ("fp8", dsaidx.FP8, False, False),
               ("fp4", dsaidx.FP8, False, True), ("rot_fp4", dsaidx.FP8, True, True))
    for k in (512, 1024):
        W = wl.precision_compare(topk=k)
        idx = {}
        for name, mode, rot, fp4 in formats:
            cache = build_cache(W, mode, device=device, rotate=rot, fp4=fp4)
            B = W.batch
            q = bf16_tensor(W.q, device)
            if rot:
                q = hadamard_rotate_bf16(q)
            ws = dsaidx.new_workspace(dsaidx.workspace_bytes_decode(cache, B, W.max_seq_len, W.H, k), device)
            oi = torch.empty((B, k), dtype=torch.int32, device=device)
            dsaidx.score_topk_decode(cache, q, torch.from_numpy(W.w).to(device),
                                     torch.from_numpy(W.block_table).to(device),
                                     torch.tensor(W.seq_lens, dtype=torch.int32, device=device),
                                     W.max_seq_len, k, oi, ws)
            idx[name] = oi.cpu().numpy()
            del cache, ws
        for b, S in enumerate(W.seq_lens):
            nd = int(W.needle_pos[b])
            sel = {n: [int(x) for x in idx[n][b] if x >= 0] for n, _, _, _ in formats}
            Hs = set(sel["bf16"])
            row = {"S": int(S), "topk": k,
                   "needle_rank_bf16": sel["bf16"].index(nd) + 1 if nd in Hs else None}
            for n in ("fp8", "fp4", "rot_fp4"):
                F = set(sel[n])
                row["needle_rank_" + n] = sel[n].index(nd) + 1 if nd in F else None
                row["jaccard_%s_vs_bf16" % n] = round(len(F & Hs) / max(1, len(F | Hs)), 4)
                row["lost_bf16_to_" + n] = len(Hs - F)
            if k == 512 and int(S) in PAGES_JACCARD_TOP512:
                row["pages_jaccard"], row["pages_lost"] = PAGES_JACCARD_TOP512[int(S)]
            rows.append(row)
    torch.cuda.empty_cache()
    return {"workload": "precision_s2000_4500_10000_22000", "source": "GPU outputs, every key format",
            "pages_context": "fp8-vs-bf16 top-512 Jaccard 0.395/0.382/0.299/0.267 at 2k/4.5k/10k/22k "
                             "from the pages' own synthetic test (different data)",
            "rows": rows}


# ----------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ----------------------------------------------------------------------------

def cpu_baselines(W):
    """The oracle, as it stands, on this host's cores: the decode workload with
    every core and with one thread (the headline value is the all-core one),
    a 64-query subset of the prefill chunk and one 131072-key row of the
    long-context workload, each rate labelled with its sample."""
    import oracle
    from sparse_attention_top_idx_gb300 import workloads as wl
    rate, cores, reps, el = oracle_decode_rate(W, 8.0)
    out = {"value": round(rate, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": "%d whole decode steps (32 rows, all 232,000 keys) in %.1f s" % (reps, el)}
    nt = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        r1, c1, reps1, el1 = oracle_decode_rate(W, 6.0)
    finally:
        oracle.set_num_threads(nt)
    out["single_thread"] = {"value": round(r1, 1), "unit": UNIT, "cores": 1,
                            "sample": "%d whole decode steps in %.1f s" % (reps1, el1)}
    P = wl.prefill_chunk()
    rows = np.linspace(0, P.total_q - 1, 64).astype(np.int64)
    keys = [oracle.quantize_rows(k) for k in P.keys]
    pairs = int(np.sum(P.row_pos()[rows] + 1))
    t0 = time.perf_counter()
    oracle.score_topk(oracle.FP8, P.topk, P.q[rows], P.w[rows], P.row_seq()[rows], P.row_pos()[rows], keys)
    elp = time.perf_counter() - t0
    total_pairs = int(np.sum(P.row_pos() + 1))
    out["prefill"] = {"value": round(pairs / elp, 1), "unit": "query-key pairs/s", "cores": cores,
                      "sample": "64 evenly spaced queries of the 8192-query chunk (%d pairs) in %.2f s; "
                                "the whole chunk extrapolates to %.0f s" % (pairs, elp, total_pairs / (pairs / elp))}
    L = wl.long_context()
    kq = [oracle.quantize_rows(L.keys[0])]
    t0 = time.perf_counter()
    oracle.score_topk(oracle.FP8, L.topk, L.q[:1], L.w[:1], np.zeros(1, np.int32),
                      np.array([L.seq_lens[0] - 1], np.int64), kq)
    ell = time.perf_counter() - t0
    out["long_context"] = {"value": round(L.seq_lens[0] / ell, 1), "unit": "keys/s", "cores": cores,
                           "sample": "one 131072-key row (top-1024) in %.2f s; the whole batch "
                                     "(2,097,152 keys) extrapolates to %.1f s" % (ell, sum(L.seq_lens) / (L.seq_lens[0] / ell))}
    return out


def oracle_decode_rate(W, budget_s: float):
    """Time the oracle on whole decode steps of the workload (keys already
    quantised, as they sit in the cache) until about budget_s has passed."""
    import oracle
    keys = [oracle.quantize_rows(k) for k in W.keys]
    pos = np.asarray(W.seq_lens, np.int64) - 1
    rows = np.arange(W.batch, dtype=np.int32)
    last = np.cumsum(W.seq_lens) - 1
    newk = W.all_keys()[last]
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.quantize_rows(newk)                  # the step's new keys
        oracle.score_topk(oracle.FP8, W.topk, W.q, W.w, rows, pos, keys)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    keys_total = reps * int(sum(W.seq_lens))
    return keys_total / el, oracle.num_threads(), reps, el


def oracle_decode_steps(W, steps: int, warmup: int, budget_s: float = 90.0):
    """The oracle on decode steps of the workload (keys already quantised, as
    they sit in the cache): `warmup` untimed steps (the first of them also
    times a whole step), then exactly `steps` timed ones.  A step is every
    row of the batch when steps + warmup of those fit in about budget_s,
    else the same bounded sample of the first r rows (r even where it can
    be, so that the 4500/10000-key alternation stays balanced).  Returns
    (keys/s over the timed steps, threads, rows per step, seconds)."""
    import oracle
    keys = [oracle.quantize_rows(k) for k in W.keys]
    pos = np.asarray(W.seq_lens, np.int64) - 1
    last = np.cumsum(W.seq_lens) - 1
    newk = W.all_keys()[last]

    def step(r):
        oracle.quantize_rows(newk[:r])              # the step's new keys
        oracle.score_topk(oracle.FP8, W.topk, W.q[:r], W.w[:r], np.arange(r, dtype=np.int32), pos[:r], keys[:r])

    t0 = time.perf_counter()
    step(W.batch)
    full = time.perf_counter() - t0
    r = W.batch
    if full * (steps + warmup) > budget_s:
        r = max(1, int(W.batch * budget_s / (full * (steps + warmup))))
        if r >= 2:
            r -= r % 2
    for _ in range(warmup - 1):
        step(r)
    t0 = time.perf_counter()
    for _ in range(steps):
        step(r)
    el = time.perf_counter() - t0
    return steps * int(sum(W.seq_lens[:r])) / el, oracle.num_threads(), r, el


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from sparse_attention_top_idx_gb300 import workloads as wl
    W = wl.decode_batch()
    rate, cores, r, el = oracle_decode_steps(W, args.steps, args.warmup)
    sample = ("%d timed decode steps of %d rows (%d keys each) after %d warm-up steps, %.1f s"
              % (args.steps, r, int(sum(W.seq_lens[:r])), args.warmup, el))
    line = {"impl": "reference", "metric": METRIC, "value": round(rate, 1), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * el / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulation)", "data": "synthetic",
            "config": config_dict(W),
            "cpu_baseline": {"value": round(rate, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(rate, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def config_dict(W):
    return {"workload": W.name, "batch": W.batch, "seq_lens": "4500/10000 alternating",
            "keys_per_step": int(sum(W.seq_lens)), "heads": W.H, "head_dim": W.d, "topk": W.topk,
            "block_size": W.bs, "key_format": "fp8 e4m3 + fp32 scale (132 B/token)",
            "step": "idx_store_keys(32 new keys) + idx_score_topk_decode",
            "l2": "rotating %d pool copies (%.0f MB) so each step reads its keys from HBM"
                  % (N_POOL_COPIES, N_POOL_COPIES * sum(W.seq_lens) * KEY_BYTES_FP8 / 1e6)}


# ----------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the long-context and prefill objects")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    ap.add_argument("--eager", action="store_true", help="no CUDA graphs (for profiler runs)")
    ap.add_argument("--only", choices=["longctx", "prefill", "precision"], default=None,
                    help="run just one secondary workload and print its object (for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    global EAGER
    EAGER = args.eager
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import __graft_entry__
    rank, world, local, dist = setup_dist(args.gpus)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        __graft_entry__.build()
    barrier(dist)
    from sparse_attention_top_idx_gb300 import dsaidx, workloads as wl
    dsaidx.load()
    peaks = measured_peaks()
    if args.only == "longctx":
        print(json.dumps(bench_long_context(device, args.steps, args.warmup, peaks)))
        return 0
    if args.only == "prefill":
        print(json.dumps(bench_prefill(device, args.steps, args.warmup, peaks)))
        return 0
    if args.only == "precision":
        print(json.dumps(bench_precision(device)))
        return 0

    W = wl.decode_batch()
    bench = DecodeBench(W, device, N_POOL_COPIES)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    total_ms, kern_ms, graph = time_steps(bench, args.steps, args.warmup, dist, device)
    load_padding(graph, 1.0, device)
    del graph
    clocks = sampler.stop()
    total_ms = max_over_ranks(total_ms, dist, device)
    ms_step = total_ms / args.steps
    value = whole_job_rate(world, bench.keys, ms_step)

    e2e_ms, e2e_eager_ms, h2d, d2h, e2e_reps, e2e_engine_ms = e2e_decode(bench, args.steps, args.warmup, device)
    e2e_ms = max_over_ranks(e2e_ms, dist, device)
    e2e_eager_ms = max_over_ranks(e2e_eager_ms, dist, device)
    e2e_engine_ms = max_over_ranks(e2e_engine_ms, dist, device)

    tr = traffic_of("decode")
    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "us_per_step": round(ms_step * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulation)",
            "data": "synthetic (seeded iid N(0,1) keys, planted needle)",
            "config": config_dict(W),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "roofline": dict(roofline_hbm(bench.algo_bytes(), kern_ms, peaks["hbm_gbs"], tr),
                             note="kernel_us: events around each scoring kernel in a second graph of the "
                                  "same steps (event nodes stop the programmatic overlap, so it includes the "
                                  "kernel's launch and set-up); the timed steps overlap them with the key store",
                             frac_of_step=round(bench.algo_bytes() / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)),
            "peaks_source": peaks["source"],
            "e2e": {"value": round(whole_job_rate(world, bench.keys, e2e_ms), 1), "unit": UNIT,
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "issue": "public API calls replayed from a CUDA graph",
                    "copies": "idx_copy kernel (the GPU reads and writes the pinned host buffers)",
                    "copy_engine_ms_per_step": round(e2e_engine_ms, 5),
                    "replays": len(e2e_reps), "ms_per_step_each_replay": [round(x, 5) for x in e2e_reps],
                    "eager_value": round(whole_job_rate(world, bench.keys, e2e_eager_ms), 1),
                    "eager_ms_per_step": round(e2e_eager_ms, 5)},
            "timing": "K steps replayed from one CUDA graph (no event between a step's kernels); "
                      "scoring-kernel durations from events recorded around each scoring kernel in a "
                      "second graph of the same steps",
            "gpu_launches": 2 * args.steps,
            "clocks": clocks}
    del bench
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_extra:
        line["long_context"] = bench_long_context(device, max(10, args.steps // 4), args.warmup, peaks)
        line["prefill"] = bench_prefill(device, max(3, args.steps // 40), 3, peaks)
    if rank == 0 and not args.no_extra:
        line["precision"] = bench_precision(device)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baselines(W)
    if rank == 0:
        print(json.dumps(line))
    barrier(dist)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
