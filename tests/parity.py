"""Helpers shared by the GPU parity tests, the smoke check and the benchmark's
parity leg: run the CUDA path on a synthetic workload through the C ABI, and
compare its rows with the CPU oracle.

Comparison rule (tolerance tol = 1e-3 on fp32 scores):
* every row selects exactly min(k, visible) distinct visible indices, padded
  with -1; scores are non-increasing and equal scores list lower indices first;
* each returned score is within tol relative (plus 1e-6 of the row's largest
  oracle score, which only matters for exact zeros) of the oracle's score of
  that index;
* when the oracle's k-th and (k+1)-th scores differ by more than tol * |k-th|,
  the selected set equals the oracle's set exactly; otherwise (near-ties at the
  boundary) every index scoring above tau * (1 + tol) is selected and every
  selected index scores at least tau * (1 - tol), tau the oracle's k-th score.
"""
from __future__ import annotations

import numpy as np
import torch

from sparse_attention_top_idx_gb300 import dsaidx
from sparse_attention_top_idx_gb300 import workloads as wl
from sparse_attention_top_idx_gb300.host import bf16_tensor, build_cache  # noqa: F401 (re-exported)

TOL = 1e-3


def decode_inputs(W: wl.Workload, device="cuda"):
    assert all(n == 1 for n in W.nq)
    return dict(q=bf16_tensor(W.q, device), w=torch.from_numpy(W.w).to(device),
                block_table=torch.from_numpy(W.block_table).to(device),
                seq_lens=torch.tensor(W.seq_lens, dtype=torch.int32, device=device))


def run_decode(W: wl.Workload, mode: int, cache=None, max_seq_len=None, reps: int = 1,
               device="cuda", expect_status: int = 0):
    cache = cache or build_cache(W, mode, device=device)
    ins = decode_inputs(W, device)
    msl = W.max_seq_len if max_seq_len is None else max_seq_len
    B, k = W.batch, W.topk
    ws = dsaidx.new_workspace(dsaidx.workspace_bytes_decode(cache, B, msl, W.H, k), device)
    outs = []
    for _ in range(reps):
        oi = torch.full((B, k), -7, dtype=torch.int32, device=device)
        osc = torch.full((B, k), float("nan"), dtype=torch.float32, device=device)
        dsaidx.score_topk_decode(cache, ins["q"], ins["w"], ins["block_table"], ins["seq_lens"], msl, k,
                                 oi, ws, out_score=osc)
        outs.append({"idx": oi.cpu().numpy(), "score": osc.cpu().numpy()})
    st = dsaidx.read_device_status(ws)
    assert st == expect_status, "device status %d" % st
    return outs[0] if reps == 1 else outs


def run_prefill(W: wl.Workload, mode: int, cache=None, device="cuda", expect_status: int = 0):
    cache = cache or build_cache(W, mode, device=device)
    T, k = W.total_q, W.topk
    q = bf16_tensor(W.q, device)
    w = torch.from_numpy(W.w).to(device)
    cu = torch.from_numpy(W.cu_seqlens_q()).to(device)
    sl = torch.tensor(W.seq_lens, dtype=torch.int32, device=device)
    bt = torch.from_numpy(W.block_table).to(device)
    ws = dsaidx.new_workspace(dsaidx.workspace_bytes_prefill(cache, W.batch, T, W.max_seq_len, W.H, k),
                              device)
    oi = torch.full((T, k), -7, dtype=torch.int32, device=device)
    osc = torch.full((T, k), float("nan"), dtype=torch.float32, device=device)
    dsaidx.score_topk_prefill(cache, q, w, cu, sl, bt, W.max_seq_len, k, oi, ws, out_score=osc)
    st = dsaidx.read_device_status(ws)
    assert st == expect_status, "device status %d" % st
    return {"idx": oi.cpu().numpy(), "score": osc.cpu().numpy()}


def check_row(gi, gs, o, k, tol=TOL):
    """Check one GPU row (indices gi, scores gs) against oracle scores o of its
    visible keys.  Returns True when the selected set equals the oracle's."""
    nv = len(o)
    m = min(k, nv)
    assert np.all(gi[:m] >= 0), "missing selections"
    assert np.all(gi[m:] == -1), "bad padding"
    assert np.all(np.isneginf(gs[m:])), "bad score padding"
    sel = gi[:m].astype(np.int64)
    assert len(np.unique(sel)) == m, "duplicate indices"
    assert sel.max(initial=-1) < nv, "index beyond the visible keys"
    if m == 0:
        return True
    g = gs[:m].astype(np.float64)
    ov = o[sel].astype(np.float64)
    floor = 1e-6 * np.max(np.abs(o))
    err = np.abs(g - ov)
    assert np.all(err <= tol * np.abs(ov) + floor), "score mismatch, max rel %g" % (
        np.max(err / np.maximum(np.abs(ov), 1e-30)))
    assert np.all(np.diff(g) <= 0), "scores not in descending order"
    eq = np.diff(g) == 0
    assert np.all(np.diff(sel)[eq] > 0), "equal scores not in ascending index order"
    if nv <= k:
        assert set(sel.tolist()) == set(range(nv))
        return True
    order = np.argsort(-o.astype(np.float64), kind="stable")
    tau = float(o[order[k - 1]])
    nxt = float(o[order[k]])
    ref = set(order[:k].tolist())
    got = set(sel.tolist())
    if tau - nxt > tol * abs(tau):
        assert got == ref, "set differs although the boundary gap exceeds the tolerance"
        return True
    must = np.nonzero(o > tau + tol * abs(tau))[0]
    assert set(must.tolist()) <= got, "a clearly-above-boundary index is missing"
    assert np.all(o[sel] >= tau - tol * abs(tau)), "a clearly-below-boundary index was selected"
    return got == ref


def check_rows(got, ref, nvis, k, rows=None, tol=TOL):
    """Check GPU rows against oracle output from oracle.score_topk(..., full_scores=True).
    rows: which GPU rows the oracle rows correspond to (default: all, in order).
    Returns the number of rows whose set equals the oracle's exactly."""
    rows = range(len(nvis)) if rows is None else rows
    exact = 0
    for i, r in enumerate(rows):
        nv = int(nvis[i])
        exact += bool(check_row(got["idx"][r], got["score"][r], ref["scores"][i, :nv], k, tol))
    return exact
