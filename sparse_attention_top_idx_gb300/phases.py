"""Per-phase timeline of the decode kernel, from %globaltimer stamps.

Builds the diagnostic library libdsaidx_phases.so (the library's sources
compiled with -DDSAIDX_PHASE_STAMPS: the decode kernel stores a timestamp per
CTA and unit at each phase boundary), runs the decode batch (32 sequences of
4500 / 10000 keys, top-512) and the long-context workload (8 x 131072 +
1 x 1048576 keys, top-1024), both fp8, and prints per phase the median and the
largest over CTAs of the time since the earliest CTA finished its set-up, for
the first unit of every CTA.  Needs a GPU.

    python -m sparse_attention_top_idx_gb300.phases
"""
from __future__ import annotations

import ctypes
import sys

import numpy as np
import torch

from . import build as _build
from . import dsaidx
from . import workloads as wl
from .host import bf16_tensor, build_cache

CTAS, UNITS, SLOTS = 2048, 4, 16
NAMES = ["entry", "set-up done", "unit located", "query rows landed", "B tile complete",
         "first key tile", "stream done", "window sent", "windows received", "boundary known",
         "pool complete", "ranks written", "unit end", "loop done", "exit"]


def _run(L, W, warm: int = 50):
    cache = build_cache(W, dsaidx.FP8)
    dev = "cuda"
    q, w = bf16_tensor(W.q, dev), torch.from_numpy(W.w).to(dev)
    bt, sl = torch.from_numpy(W.block_table).to(dev), torch.tensor(W.seq_lens, dtype=torch.int32, device=dev)
    ws = dsaidx.new_workspace(dsaidx.workspace_bytes_decode(cache, W.batch, W.max_seq_len, W.H, W.topk))
    oi = torch.empty((W.batch, W.topk), dtype=torch.int32, device=dev)
    for _ in range(warm):
        dsaidx.score_topk_decode(cache, q, w, bt, sl, W.max_seq_len, W.topk, oi, ws)
    torch.cuda.synchronize()
    buf = np.zeros((CTAS, UNITS, SLOTS), np.uint64)
    L.idx_phase_stamps(None, 1)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    dsaidx.score_topk_decode(cache, q, w, bt, sl, W.max_seq_len, W.topk, oi, ws)
    b.record()
    torch.cuda.synchronize()
    if L.idx_phase_stamps(buf.ctypes.data_as(ctypes.c_void_p), 0) != 0:
        raise RuntimeError("idx_phase_stamps failed")
    st = buf.astype(np.int64)
    ctas = np.nonzero(st[:, 0, 1])[0]
    t0 = st[ctas, 0, 1].min()
    print("%s: %d CTAs, kernel %.2f us (events, one launch)" % (W.name, len(ctas), a.elapsed_time(b) * 1e3))
    print("  %-18s %10s %10s   (us since the earliest set-up end; unit 0 of each CTA)" % ("phase", "median", "max"))
    for k in range(15):
        u = 0
        v = np.array([st[c, u, k] - t0 for c in ctas if st[c, u, k] > 0], np.float64) / 1e3
        if v.size:
            print("  %-18s %10.2f %10.2f" % (NAMES[k], np.median(v), v.max()))
    cache.close()   # while this library is the loaded one


def main() -> int:
    if not torch.cuda.is_available():
        print("needs a GPU")
        return 1
    L = dsaidx.load(_build.build_phases())
    L.idx_phase_stamps.argtypes = [ctypes.c_void_p, ctypes.c_int]
    L.idx_phase_stamps.restype = ctypes.c_int
    saved = dsaidx._lib
    dsaidx._lib = L
    try:
        _run(L, wl.decode_batch())
        _run(L, wl.long_context(), warm=10)
    finally:
        dsaidx._lib = saved
    return 0


if __name__ == "__main__":
    sys.exit(main())
