"""Randomised parity sweep: seeded random shapes for the decode and prefill
calls -- batch sizes, ragged and empty lengths, sequences across segment
boundaries, k from 1 to 2048, block sizes 32 and 64, both key formats --
each checked against the oracle row by row.  The cases are drawn from a
fixed seed, so a failure reproduces."""
import numpy as np
import pytest

import oracle
from sparse_attention_top_idx_gb300 import workloads as wl
from tests.parity import check_rows, run_decode, run_prefill

pytestmark = pytest.mark.gpu


def _decode_case(c):
    rng = np.random.default_rng(1000 + c)
    B = int(rng.integers(1, 12))
    lens = []
    for _ in range(B):
        r = rng.random()
        if r < 0.1:
            lens.append(0)
        elif r < 0.25:
            lens.append(int(rng.integers(1, 300)))
        elif r < 0.85:
            lens.append(int(rng.integers(300, 20000)))
        else:
            lens.append(int(rng.integers(65000, 140000)))   # one or two segments past 65536
    if max(lens) == 0:
        lens[0] = int(rng.integers(1, 5000))   # a pool needs at least one block
    k = int(rng.choice([1, 7, 64, 257, 512, 1000, 1024, 2048]))
    bs = int(rng.choice([32, 64]))
    mode = int(rng.integers(0, 2))
    return lens, k, bs, mode


def _prefill_case(c):
    rng = np.random.default_rng(2000 + c)
    B = int(rng.integers(1, 4))
    lens = [int(rng.integers(1, 6000)) for _ in range(B)]
    nq = [int(rng.integers(1, min(l, 40) + 1)) for l in lens]
    k = int(rng.choice([1, 33, 256, 512, 1024, 2048]))
    bs = int(rng.choice([32, 64]))
    mode = int(rng.integers(0, 2))
    return lens, nq, k, bs, mode


@pytest.mark.parametrize("case", range(40))
def test_decode_random_shapes(case):
    lens, k, bs, mode = _decode_case(case)
    W = wl.make_workload("fuzzdec%d" % case, lens, [1] * len(lens), topk=k, bs=bs, seed=300 + case)
    got = run_decode(W, mode)
    rows = [b for b in range(W.batch) if W.seq_lens[b] > 0]
    keys = [oracle.quantize_rows(W.keys[b]) if mode == oracle.FP8 else W.keys[b] for b in rows]
    pos = np.asarray([W.seq_lens[b] - 1 for b in rows], np.int64)
    if rows:
        ref = oracle.score_topk(mode, k, W.q[rows], W.w[rows], np.arange(len(rows), dtype=np.int32), pos, keys,
                                full_scores=True)
        check_rows(got, ref, pos + 1, k, rows=rows)
    for b in range(W.batch):
        if W.seq_lens[b] == 0:
            assert np.all(got["idx"][b] == -1)
        else:
            n = min(k, W.seq_lens[b])
            assert np.all(got["idx"][b][:n] >= 0) and np.all(got["idx"][b][n:] == -1)


@pytest.mark.parametrize("case", range(16))
def test_prefill_random_shapes(case):
    lens, nq, k, bs, mode = _prefill_case(case)
    W = wl.make_workload("fuzzpre%d" % case, lens, nq, topk=k, bs=bs, seed=400 + case)
    got = run_prefill(W, mode)
    keys = [oracle.quantize_rows(kk) if mode == oracle.FP8 else kk for kk in W.keys]
    ref = oracle.score_topk(mode, k, W.q, W.w, W.row_seq(), W.row_pos(), keys, full_scores=True)
    check_rows(got, ref, W.row_pos() + 1, k)
