"""Pins for the oracle's causal mask and top-k selection.

The selection keeps the index_topk best-scoring positions of each query row
(ROCm/ATOM issue #1507, sections "Environment" and "How it was isolated":
index_topk 512/1024, per-row top-k checked by set overlap against a library
top-k).  Readings taken where the pages are silent: ties go to the lower
position, the list is in descending score order, rows with fewer visible keys
than k are padded with -1, and a query at position p sees keys 0..p.

Pins: brute force over all k-subsets on tiny rows, numpy's stable argsort,
the selection invariants, and the Jaccard identity against the table printed
in "The Hypothesis That Refused to Die", section "Message 12994: The
Synthetic Test" (tests/golden/jaccard_synthetic_test.txt).
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from sparse_attention_top_idx_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_topk(scores, k):
    """The unique k-subset whose every member beats every non-member under
    (score desc, index asc)."""
    n = len(scores)
    keyf = lambda i: (-float(scores[i]), i)
    for sub in itertools.combinations(range(n), min(k, n)):
        inside = set(sub)
        worst_in = max((keyf(i) for i in inside), default=None)
        best_out = min((keyf(i) for i in range(n) if i not in inside), default=None)
        if worst_in is None or best_out is None or worst_in < best_out:
            return sorted(inside, key=keyf)
    raise AssertionError("no valid subset")


@pytest.mark.parametrize("n,k", [(1, 1), (5, 3), (8, 8), (9, 4), (12, 5), (6, 10)])
def test_topk_brute_force(n, k):
    rng = np.random.default_rng(n * 31 + k)
    for trial in range(20):
        # few distinct values so that ties are common
        s = rng.integers(0, 4, n).astype(np.float32) * np.float32(0.25)
        if trial % 2:
            s = rng.standard_normal(n).astype(np.float32)
        idx, sc = oracle.topk_row(s, k)
        want = brute_topk(s, k)
        m = min(k, n)
        assert idx[:m].tolist() == want
        assert np.all(idx[m:] == -1) and np.all(np.isneginf(sc[m:]))
        assert np.array_equal(sc[:m], s[want])


def test_topk_against_stable_argsort():
    rng = np.random.default_rng(1)
    for n, k in [(2000, 512), (10000, 1024), (777, 1024)]:
        s = rng.standard_normal(n).astype(np.float32)
        s[rng.integers(0, n, n // 10)] = 0.5   # plant ties
        idx, _ = oracle.topk_row(s, k)
        order = np.argsort(-s.astype(np.float64), kind="stable")[:k]
        m = min(k, n)
        assert np.array_equal(idx[:m], order[:m].astype(np.int32))


def test_selection_invariants_and_causal_mask():
    W = wl.tiny_prefill()
    kc_ks = oracle.quantize_rows(W.keys[0])
    out = oracle.score_topk(oracle.FP8, W.topk, W.q, W.w, W.row_seq(), W.row_pos(),
                            [kc_ks], full_scores=True)
    for r, pos in enumerate(W.row_pos()):
        idx = out["idx"][r]
        vis = pos + 1
        sel = idx[idx >= 0]
        assert len(sel) == min(W.topk, vis)
        assert len(np.unique(sel)) == len(sel)
        assert sel.max() <= pos                       # causal: nothing after pos
        sc = out["scores"][r, :vis]
        assert np.all(np.isnan(out["scores"][r, vis:]))
        mask = np.zeros(vis, bool)
        mask[sel] = True
        assert sc[mask].min() >= sc[~mask].max()      # selected beat unselected
        assert np.all(np.diff(out["score"][r][:len(sel)]) <= 0)


def test_short_rows_are_padded():
    W = wl.make_workload("short", [40], [40], topk=32, seed=3)
    out = oracle.score_topk(oracle.BF16, 32, W.q, W.w, W.row_seq(), W.row_pos(), W.keys)
    for r, pos in enumerate(W.row_pos()):
        idx = out["idx"][r]
        nv = min(32, pos + 1)
        assert np.all(idx[:nv] >= 0) and np.all(idx[nv:] == -1)
        assert set(idx[:nv].tolist()) <= set(range(pos + 1))


def test_decode_row_equals_last_prefill_row():
    # Decode is the causal chunk with one query: the last row of a chunk and a
    # one-query call at the same position must agree bit for bit.
    W = wl.make_workload("x", [700], [9], topk=64, seed=5)
    kk = [oracle.quantize_rows(W.keys[0])]
    full = oracle.score_topk(oracle.FP8, 64, W.q, W.w, W.row_seq(), W.row_pos(), kk)
    last = oracle.score_topk(oracle.FP8, 64, W.q[-1:], W.w[-1:], np.zeros(1, np.int32),
                             np.array([699]), kk)
    assert np.array_equal(full["idx"][-1], last["idx"][0])
    assert np.array_equal(full["score"][-1], last["score"][0])


def _read_golden_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def test_jaccard_identity_against_printed_table():
    # The printed table's columns satisfy jaccard = (k - lost) / (k + lost)
    # for two top-k sets of equal size k that differ in `lost` positions.
    rows = _read_golden_table("jaccard_synthetic_test.txt")
    assert len(rows) == 4
    k = 512
    for S, jac, lost in rows:
        lost = int(lost)
        a = np.arange(k)
        b = np.concatenate([np.arange(lost, k), np.arange(k, k + lost)])
        assert oracle.lost(a, b) == lost
        assert abs(oracle.jaccard(a, b) - float(jac)) < 5e-4
        assert abs((k - lost) / (k + lost) - float(jac)) < 5e-4


def test_needle_rank_definition():
    s = np.array([0.1, 0.9, 0.5, 0.9, 0.2], np.float32)
    assert oracle.needle_rank(s, 1) == 1
    assert oracle.needle_rank(s, 2) == 3
    assert oracle.needle_rank(s, 0) == 5
