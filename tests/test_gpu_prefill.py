"""GPU parity of idx_score_topk_prefill (causal query chunks) against the CPU
oracle: the tiny workload in full, ragged multi-sequence chunks, the long
prefill chunk at full size (sampled rows against the oracle, every row against
the selection invariants), and decode / prefill agreement."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_idx_gb300 import dsaidx
from sparse_attention_top_idx_gb300 import workloads as wl
from tests.parity import build_cache, check_rows, run_decode, run_prefill

pytestmark = pytest.mark.gpu


def oracle_ref(W, mode, rows=None):
    R = W.total_q
    rows = list(range(R)) if rows is None else list(rows)
    keys = [oracle.quantize_rows(k) if mode == oracle.FP8 else k for k in W.keys]
    ref = oracle.score_topk(mode, W.topk, W.q[rows], W.w[rows], W.row_seq()[rows], W.row_pos()[rows],
                            keys, full_scores=True)
    return ref, W.row_pos()[rows] + 1


@pytest.mark.parametrize("mode", [0, 1])
def test_tiny_prefill(mode):
    # 1 sequence of 2000 keys, queries at its last 16 positions, top-512
    W = wl.tiny_prefill()
    got = run_prefill(W, mode)
    ref, nvis = oracle_ref(W, mode)
    exact = check_rows(got, ref, nvis, W.topk)
    assert exact >= 14
    for r in range(W.total_q):
        assert got["idx"][r][0] == W.needle_pos[0]


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("mode", [0, 1])
def test_ragged_chunks(bs, mode):
    # several sequences, chunk sizes not multiples of 4 queries, rows that see
    # fewer keys than k, a one-query chunk
    W = wl.make_workload("rag", [300, 1000, 129, 70], [7, 130, 1, 70], topk=128, bs=bs,
                         seed=40 + bs + mode)
    got = run_prefill(W, mode)
    ref, nvis = oracle_ref(W, mode)
    check_rows(got, ref, nvis, W.topk)


def test_prefill_chunk_full_size_sampled():
    # 1 sequence of 22000 keys, queries at its last 8192 positions, top-1024
    W = wl.prefill_chunk()
    got = run_prefill(W, dsaidx.FP8)
    T = W.total_q
    rows = sorted(set([0, 1, 2, 3, 4, 5, 127, 128, 129, 4095, 4096, T - 5, T - 4, T - 3, T - 2, T - 1]
                      + list(range(7, T, 613))))
    ref, nvis = oracle_ref(W, dsaidx.FP8, rows)
    check_rows(got, ref, nvis, W.topk, rows=rows)
    pos = W.row_pos()
    idx = got["idx"]
    assert np.all(idx >= 0)
    assert np.all(idx.max(axis=1) <= pos)
    s = np.sort(idx, axis=1)
    assert np.all(np.diff(s, axis=1) > 0)                 # no duplicates in any row
    assert np.all(np.diff(got["score"], axis=1) <= 0)     # descending in every row


def test_prefill_chunk_full_size_dense_rows_and_scores():
    # the full-size chunk (22000 keys, 8192 causal queries, top-1024): rows
    # 4090..4200, the last 64 and every 4th row against the oracle -- the
    # selections, and every visible fp32 score the scoring kernel left in the
    # workspace (its layout: 256-byte header, one flag word per row rounded up
    # to 256 bytes, then the score rows of max_seq_len rounded up to 4 floats)
    from sparse_attention_top_idx_gb300.host import bf16_tensor
    W = wl.prefill_chunk()
    cache = build_cache(W, dsaidx.FP8)
    T, k = W.total_q, W.topk
    nbytes = dsaidx.workspace_bytes_prefill(cache, W.batch, T, W.max_seq_len, W.H, k)
    ws = dsaidx.new_workspace(nbytes)
    oi = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    osc = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    dsaidx.score_topk_prefill(cache, bf16_tensor(W.q), torch.from_numpy(W.w).cuda(),
                              torch.from_numpy(W.cu_seqlens_q()).cuda(),
                              torch.tensor(W.seq_lens, dtype=torch.int32, device="cuda"),
                              torch.from_numpy(W.block_table).cuda(), W.max_seq_len, k, oi, ws, out_score=osc)
    assert dsaidx.read_device_status(ws) == 0
    got = {"idx": oi.cpu().numpy(), "score": osc.cpu().numpy()}
    rows = sorted(set(list(range(4090, 4201)) + list(range(T - 64, T)) + list(range(0, T, 4))))
    ref, nvis = oracle_ref(W, dsaidx.FP8, rows)
    exact = check_rows(got, ref, nvis, W.topk, rows=rows)
    assert exact >= len(rows) - 8
    align = lambda x, a: (x + a - 1) // a * a
    off = align(256 + T * 4, 256)
    stride = align(W.max_seq_len, 4)
    scores = ws[off: off + T * stride * 4].view(torch.float32).view(T, stride)
    sub = scores[torch.tensor(rows, device="cuda")].cpu().numpy()
    for i, r in enumerate(rows):
        nv = int(nvis[i])
        want = ref["scores"][i, :nv].astype(np.float64)
        have = sub[i, :nv].astype(np.float64)
        tol = 1e-3 * np.abs(want) + 1e-6 * np.abs(want).max()
        bad = np.nonzero(np.abs(have - want) > tol)[0]
        assert bad.size == 0, "row %d: %d of %d scores off, first at key %d" % (r, bad.size, nv, bad[0])


@pytest.mark.parametrize("mode", [0, 1])
def test_last_prefill_row_equals_decode(mode):
    # decode is the one-query chunk: same scores and selection for the last row
    W = wl.make_workload("x", [3000, 1500], [9, 4], topk=256, seed=12)
    cache = build_cache(W, mode)
    pre = run_prefill(W, mode, cache=cache)
    cu = W.cu_seqlens_q()
    D = wl.Workload("x1", W.seq_lens, [1, 1], W.H, W.d, W.topk, W.bs, W.keys,
                    W.q[cu[1:] - 1], W.w[cu[1:] - 1], W.needle_pos, W.block_table, W.num_blocks)
    dec = run_decode(D, mode, cache=cache)
    for b in range(2):
        r = cu[b + 1] - 1
        assert np.array_equal(pre["idx"][r], dec["idx"][b])
        assert np.array_equal(pre["score"][r].view(np.uint32), dec["score"][b].view(np.uint32))


def test_bad_block_id_flags_rows():
    W = wl.make_workload("bad", [500, 400], [5, 6], topk=64, seed=13)
    cache = build_cache(W, dsaidx.FP8)
    W.block_table[0, 2] = -3
    got = run_prefill(W, dsaidx.FP8, cache=cache, expect_status=5)
    assert np.all(got["idx"][:5] == -1)
    ref, nvis = oracle_ref(W, dsaidx.FP8, range(5, 11))
    check_rows(got, ref, nvis, 64, rows=range(5, 11))


def test_kernel_timing_records_each_kernel():
    # prefill launches the scoring kernel and the row select; decode one kernel
    W = wl.make_workload("ktime", [700, 300], [5, 3], topk=64, seed=91)
    cache = build_cache(W, dsaidx.FP8)
    dsaidx.kernel_timing(16)
    run_prefill(W, dsaidx.FP8, cache=cache)
    t = dsaidx.kernel_times()
    assert len(t) == 2 and all(x > 0.0 for x in t)
    D = wl.make_workload("ktime_dec", [700, 300], [1, 1], topk=64, seed=92)
    run_decode(D, dsaidx.FP8)
    t = dsaidx.kernel_times()
    assert len(t) == 1 and t[0] > 0.0
    dsaidx.kernel_timing(0)
    run_decode(D, dsaidx.FP8)
    assert dsaidx.kernel_times() == []


def test_prefill_slot_output_is_the_block_table_translate():
    W = wl.make_workload("pslots", [2500, 300], [40, 7], topk=128, bs=32, seed=81)
    cache = build_cache(W, dsaidx.FP8)
    T, k = W.total_q, W.topk
    from sparse_attention_top_idx_gb300.host import bf16_tensor
    ws = dsaidx.new_workspace(dsaidx.workspace_bytes_prefill(cache, W.batch, T, W.max_seq_len, W.H, k))
    oi = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    osl = torch.full((T, k), -7, dtype=torch.int64, device="cuda")
    dsaidx.score_topk_prefill(cache, bf16_tensor(W.q), torch.from_numpy(W.w).cuda(),
                              torch.from_numpy(W.cu_seqlens_q()).cuda(),
                              torch.tensor(W.seq_lens, dtype=torch.int32, device="cuda"),
                              torch.from_numpy(W.block_table).cuda(), W.max_seq_len, k, oi, ws, out_slot=osl)
    idx, slots = oi.cpu().numpy(), osl.cpu().numpy()
    ref = run_prefill(W, dsaidx.FP8, cache=cache)
    assert np.array_equal(idx, ref["idx"])
    for r, b in enumerate(W.row_seq()):
        assert np.array_equal(slots[r], oracle.translate_slots(W.block_table[b], W.bs, idx[r]))
