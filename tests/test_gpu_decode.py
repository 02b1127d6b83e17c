"""GPU parity of idx_score_topk_decode (fused score + top-k, one query per
sequence) against the CPU oracle, on the decode workloads at full size and on
ragged / degenerate cases."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_idx_gb300 import dsaidx
from sparse_attention_top_idx_gb300 import workloads as wl
from tests.parity import build_cache, check_rows, decode_inputs, run_decode

pytestmark = pytest.mark.gpu


def oracle_ref(W, mode, rows=None):
    rows = list(range(W.batch)) if rows is None else rows
    keys = [oracle.quantize_rows(W.keys[b]) if mode == oracle.FP8 else W.keys[b] for b in rows]
    q = W.q[rows]
    w = W.w[rows]
    pos = np.asarray([W.seq_lens[b] - 1 for b in rows], np.int64)
    ref = oracle.score_topk(mode, W.topk, q, w, np.arange(len(rows), dtype=np.int32), pos, keys,
                            full_scores=True)
    return ref, pos + 1


def check(W, mode, got, rows=None):
    rows = list(range(W.batch)) if rows is None else rows
    ref, nvis = oracle_ref(W, mode, rows)
    return check_rows(got, ref, nvis, W.topk, rows=rows)


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("mode", [0, 1])
def test_ragged_small(bs, mode):
    # lengths around tile / block / k boundaries, k larger than some sequences
    W = wl.make_workload("ragged", [700, 129, 1, 128, 64, 2049, 513, 0], [1] * 8, topk=128, bs=bs,
                         seed=31 + bs + mode)
    got = run_decode(W, mode)
    check(W, mode, got)
    assert np.all(got["idx"][7] == -1)           # empty sequence


@pytest.mark.parametrize("k", [512, 1024])
@pytest.mark.parametrize("mode", [0, 1])
def test_precision_workload(mode, k):
    # 4 sequences of 2000 / 4500 / 10000 / 22000 keys with a planted needle
    W = wl.precision_compare(topk=k)
    got = run_decode(W, mode)
    check(W, mode, got)
    for b in range(W.batch):
        assert got["idx"][b][0] == W.needle_pos[b]      # the needle ranks first


def test_decode_batch_full_size():
    # 32 sequences alternating 4500 / 10000 keys, top-512, fp8, blocks of 64
    W = wl.decode_batch()
    got = run_decode(W, dsaidx.FP8)
    exact = check(W, dsaidx.FP8, got)
    assert exact >= 30
    for b in range(W.batch):
        assert got["idx"][b][0] == W.needle_pos[b]


def test_long_context_full_size_sampled():
    # 8 x 131072 + 1 x 1048576 keys, top-1024: the GPU runs the whole batch;
    # the oracle checks one 131072-key row and the 1M-key row
    W = wl.long_context()
    got = run_decode(W, dsaidx.FP8)
    check(W, dsaidx.FP8, got, rows=[3, 8])
    for b in range(W.batch):
        idx = got["idx"][b]
        assert len(np.unique(idx)) == 1024 and idx.min() >= 0 and idx.max() < W.seq_lens[b]
        assert idx[0] == W.needle_pos[b]


@pytest.mark.parametrize("mode", [0, 1])
def test_ties_go_to_lower_index(mode):
    # every key identical: all scores tie, so the top-k is the first k positions
    W = wl.make_workload("ties", [3000, 300], [1, 1], topk=256, seed=4)
    for b in range(W.batch):
        W.keys[b][:] = W.keys[b][0]
    got = run_decode(W, mode)
    assert np.array_equal(got["idx"][0], np.arange(256))
    assert np.array_equal(got["idx"][1], np.arange(256))
    assert np.all(got["score"][0] == got["score"][0][0])
    # more tied candidates than the selection keeps in shared memory
    W3 = wl.make_workload("ties3", [10000], [1], topk=100, seed=6)
    W3.keys[0][:] = W3.keys[0][0]
    got3 = run_decode(W3, mode)
    assert np.array_equal(got3["idx"][0], np.arange(100))
    # groups of duplicates: many exact ties at the boundary
    W2 = wl.make_workload("ties2", [5000], [1], topk=300, seed=5)
    W2.keys[0][:] = W2.keys[0][np.arange(5000) % 37]
    got2 = run_decode(W2, mode)
    check(W2, mode, got2)


@pytest.mark.parametrize("k", [512, 2048])
@pytest.mark.parametrize("mode", [0, 1])
def test_multisegment_ties(mode, k):
    # every key identical in a sequence of two segments: each CTA's whole
    # chunk is candidates (fp8: more than a CTA's candidate list holds), the
    # refinement runs through the index bits, and for k = 2048 the merge of
    # the tied runs refines as well; the top-k is the first k positions
    W = wl.make_workload("mties", [70000, 3000], [1, 1], topk=k, seed=41 + mode)
    for b in range(W.batch):
        W.keys[b][:] = W.keys[b][0]
    got = run_decode(W, mode)
    assert np.array_equal(got["idx"][0], np.arange(k))
    assert np.array_equal(got["idx"][1], np.arange(k))
    assert np.all(got["score"][0] == got["score"][0][0])


@pytest.mark.parametrize("k", [512, 1024])
@pytest.mark.parametrize("mode", [0, 1])
def test_multisegment_random(mode, k):
    # lengths at and just past a segment (8 chunks of 8192 keys), a 5-segment
    # sequence and a short one in the same batch: every row against the oracle
    W = wl.make_workload("mseg", [65536, 65537, 300000, 131073, 777], [1] * 5, topk=k, seed=51 + mode + k)
    got = run_decode(W, mode)
    check(W, mode, got)
    for b in range(W.batch):
        assert got["idx"][b][0] == W.needle_pos[b]


def test_topk_2048_one_and_two_segments():
    # the largest k over a one-segment and a two-segment sequence
    W = wl.make_workload("k2048", [20000, 70000], [1, 1], topk=2048, seed=43)
    got = run_decode(W, dsaidx.FP8)
    check(W, dsaidx.FP8, got)


def test_bf16_many_segments_merge_reads_runs_from_memory():
    # bf16 chunks hold at most 2048 keys, so 300000 keys take 19 segments;
    # with k = 1024 a merging CTA's share of the runs exceeds the shared
    # staging area and the merge reads the runs from global memory
    W = wl.make_workload("bf16long", [300000, 5000], [1, 1], topk=1024, seed=44)
    got = run_decode(W, dsaidx.BF16)
    check(W, dsaidx.BF16, got)
    assert got["idx"][0][0] == W.needle_pos[0]


def test_many_sequences_and_a_one_key_segment():
    # 300 sequences (the grid's cluster ids come from a scan over more than
    # one sequence per thread), one of 65537 keys whose second segment holds a
    # single key (its run is one entry and padding), one empty, and k larger
    # than the short sequences
    lens = [90 + (7 * i) % 50 for i in range(300)]
    lens[17] = 65537
    lens[200] = 0
    W = wl.make_workload("many", lens, [1] * 300, topk=256, seed=45)
    got = run_decode(W, dsaidx.FP8)
    check(W, dsaidx.FP8, got, rows=[0, 17, 99, 199, 201, 299])
    assert np.all(got["idx"][200] == -1)


def test_deterministic_and_workspace_reuse():
    W = wl.make_workload("det", [4500, 10000, 300, 7777], [1] * 4, topk=512, seed=8)
    outs = run_decode(W, dsaidx.FP8, reps=5)
    for o in outs[1:]:
        assert np.array_equal(o["idx"], outs[0]["idx"])
        assert np.array_equal(o["score"].view(np.uint32), outs[0]["score"].view(np.uint32))
    check(W, dsaidx.FP8, outs[-1])


def test_bad_block_id_flags_row():
    W = wl.make_workload("bad", [1000, 1000], [1, 1], topk=64, seed=9)
    cache = build_cache(W, dsaidx.FP8)
    W.block_table[1, 3] = W.num_blocks + 5       # outside the pool
    got = run_decode(W, dsaidx.FP8, cache=cache, expect_status=5)
    assert np.all(got["idx"][1] == -1)
    ref, nvis = oracle_ref(W, dsaidx.FP8, [0])
    check_rows(got, ref, nvis, 64, rows=[0])


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("mode", [0, 1])
def test_bad_block_ids_on_either_key_issuer(bs, mode):
    # Two lanes issue a decode tile's key copies: one the first half of its
    # blocks (and the tile's byte count), the other the second half.  A bad
    # id in either half flags only its own sequence.  2000 keys over 8 CTAs
    # give 256-key chunks, two tiles each; the ids hit rank 0's second tile.
    W = wl.make_workload("bad2", [2000, 2000, 1000], [1, 1, 1], topk=64, bs=bs, seed=12 + bs + mode)
    cache = build_cache(W, mode)
    per_tile = 128 // bs
    W.block_table[0, per_tile + per_tile // 2 - 1] = W.num_blocks + 3   # last of the first half
    W.block_table[1, per_tile + per_tile // 2] = -2                     # first of the second half
    got = run_decode(W, mode, cache=cache, expect_status=5)
    assert np.all(got["idx"][0] == -1)
    assert np.all(got["idx"][1] == -1)
    ref, nvis = oracle_ref(W, mode, [2])
    check_rows(got, ref, nvis, 64, rows=[2])


def test_seq_len_above_bound_flags_row():
    W = wl.make_workload("over", [1000, 600], [1, 1], topk=64, seed=10)
    got = run_decode(W, dsaidx.FP8, max_seq_len=800, expect_status=5)
    assert np.all(got["idx"][0] == -1)
    ref, nvis = oracle_ref(W, dsaidx.FP8, [1])
    check_rows(got, ref, nvis, 64, rows=[1])


def test_workspace_too_small_is_rejected():
    W = wl.make_workload("ws", [300], [1], topk=64, seed=11)
    cache = build_cache(W, dsaidx.FP8)
    ins = decode_inputs(W)
    need = dsaidx.workspace_bytes_decode(cache, 1, 300, 64, 64)
    ws = dsaidx.new_workspace(need - 256)
    oi = torch.empty((1, 64), dtype=torch.int32, device="cuda")
    with pytest.raises(dsaidx.IdxError) as e:
        dsaidx.score_topk_decode(cache, ins["q"], ins["w"], ins["block_table"], ins["seq_lens"], 300, 64,
                                 oi, ws)
    assert e.value.code == 4


def test_timeout_path_flags_rows_and_the_next_call_recovers():
    # The test hook shortens the pipeline waits to 2 ms and makes each CTA's
    # MMA issuer withhold the signal of its first accumulator, so every CTA's
    # epilogue wait runs out (no GPU fault, trap or hang: the wait is bounded).
    # The call must record IDX_ERR_TIMEOUT, write -1 rows, drain its copies
    # and MMAs and free TMEM; a normal call afterwards must pass parity.
    W = wl.make_workload("tmo", [4500, 10000, 30000], [1, 1, 1], topk=512, seed=71)
    cache = build_cache(W, dsaidx.FP8)
    dsaidx.test_set_wait_limit(2_000_000)
    try:
        got = run_decode(W, dsaidx.FP8, cache=cache, expect_status=6)
    finally:
        dsaidx.test_set_wait_limit(0)
    assert np.all(got["idx"] == -1)
    assert np.all(np.isneginf(got["score"]))
    again = run_decode(W, dsaidx.FP8, cache=cache)
    check(W, dsaidx.FP8, again)


@pytest.mark.parametrize("mode", [0, 1])
def test_slot_output_is_the_block_table_translate(mode):
    # idx_score_topk_decode_slots: out_slot equals the oracle's translate of the
    # returned indices (bit for bit), -1 where out_idx is -1; one- and
    # multi-segment rows, an empty row, blocks of 32 and 64
    for bs in (32, 64):
        W = wl.make_workload("slots", [3000, 70000, 0, 129], [1] * 4, topk=512, bs=bs, seed=71 + bs + mode)
        cache = build_cache(W, mode)
        ins = decode_inputs(W)
        B, k = W.batch, W.topk
        ws = dsaidx.new_workspace(dsaidx.workspace_bytes_decode(cache, B, W.max_seq_len, W.H, k))
        oi = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
        osl = torch.full((B, k), -7, dtype=torch.int64, device="cuda")
        dsaidx.score_topk_decode(cache, ins["q"], ins["w"], ins["block_table"], ins["seq_lens"], W.max_seq_len, k,
                                 oi, ws, out_slot=osl)
        idx, slots = oi.cpu().numpy(), osl.cpu().numpy()
        ref = run_decode(W, mode, cache=cache)
        assert np.array_equal(idx, ref["idx"])
        for b in range(B):
            assert np.array_equal(slots[b], oracle.translate_slots(W.block_table[b], bs, idx[b]))
        assert np.all(slots[2] == -1)


@pytest.mark.parametrize("mode", [0, 1])
def test_large_batch_many_units_per_cluster(mode):
    # 300 sequences (more than one per scanning thread), random lengths with
    # empty ones and two multi-segment ones: each cluster takes about nine
    # units from the counter, alternating the next-unit barrier slots
    rng = np.random.default_rng(131 + mode)
    lens = rng.integers(0, 5000, 300)
    lens[::37] = 0
    lens[5], lens[200] = 70000, 131073
    W = wl.make_workload("many", [int(x) for x in lens], [1] * 300, topk=256, seed=133 + mode)
    got = run_decode(W, mode)
    rows = [b for b in range(W.batch) if W.seq_lens[b] > 0]
    check(W, mode, got, rows=rows)
    for b in range(W.batch):
        if W.seq_lens[b] == 0:
            assert np.all(got["idx"][b] == -1)


@pytest.mark.parametrize("mode", [0, 1])
def test_two_segment_merge_one_run_empty(mode):
    # two-segment sequences whose second (first) segment's keys are scaled
    # down a hundredfold, so one run contributes no candidate to the merge,
    # a balanced one, and k not a multiple of 32
    W = wl.make_workload("twoseg", [100000, 100000, 70000], [1, 1, 1], topk=1000, seed=61 + mode)
    seg = 65536
    for b, sl in ((0, slice(seg, None)), (1, slice(0, seg))):
        kf = wl.bf16_bits_to_f32(W.keys[b])
        kf[sl] *= np.float32(0.01)
        W.keys[b] = wl.f32_to_bf16_bits(kf)
    got = run_decode(W, mode)
    check(W, mode, got)
    assert np.all(got["idx"][0][got["idx"][0] >= 0] < seg)
    # the first segment of row 1 holds the planted needle: at most it survives
    assert np.sum(got["idx"][1][got["idx"][1] >= 0] < seg) <= 1
