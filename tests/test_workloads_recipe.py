"""The synthetic-input recipe (the seeded generators both the oracle and the
CUDA path are fed from): workload shapes, seeding, value distributions, the
planted needle and the paged block tables.  CPU only; the long-context
workload (about 1 GB of keys) is checked through the generator it calls,
on its sequence lengths, without generating its keys."""
import math

import numpy as np
import pytest

from sparse_attention_top_idx_gb300 import workloads as wl


def _f32(bits):
    return wl.bf16_bits_to_f32(bits)


@pytest.fixture(scope="module")
def decode():
    return wl.decode_batch()


def test_workload_shapes(decode):
    assert decode.batch == 32 and decode.topk == 512 and decode.H == 64 and decode.d == 128
    assert decode.seq_lens == [4500 if i % 2 == 0 else 10000 for i in range(32)]
    assert decode.nq == [1] * 32 and decode.q.shape == (32, 64, 128) and decode.w.shape == (32, 64)
    t = wl.tiny_prefill()
    assert t.seq_lens == [2000] and t.nq == [16] and t.topk == 512
    p = wl.precision_compare()
    assert p.seq_lens == [2000, 4500, 10000, 22000] and p.nq == [1] * 4


def test_long_context_lengths(monkeypatch):
    seen = {}

    def fake(name, seq_lens, nq, **kw):
        seen.update(name=name, seq_lens=list(seq_lens), nq=list(nq), **kw)
        return None

    monkeypatch.setattr(wl, "make_workload", fake)
    wl.long_context()
    assert seen["seq_lens"] == [131072] * 8 + [1048576] and seen["nq"] == [1] * 9 and seen["topk"] == 1024


def test_seeding_is_deterministic_and_per_seed():
    a = wl.make_workload("s", [300, 500], [2, 1], seed=5)
    b = wl.make_workload("s", [300, 500], [2, 1], seed=5)
    c = wl.make_workload("s", [300, 500], [2, 1], seed=6)
    for x, y in zip(a.keys + [a.q, a.w, a.block_table], b.keys + [b.q, b.w, b.block_table]):
        assert np.array_equal(x, y)
    assert not np.array_equal(a.keys[0], c.keys[0])
    # one sub-stream per sequence: the first sequence does not depend on the second's length
    d = wl.make_workload("s", [300, 900], [2, 1], seed=5)
    assert np.array_equal(a.keys[0], d.keys[0]) and np.array_equal(a.q[:2], d.q[:2])


def test_value_distributions(decode):
    k = _f32(decode.keys[1]).astype(np.float64)
    needle_row = decode.needle_pos[1]
    k = np.delete(k, needle_row, axis=0)
    assert abs(k.mean()) < 0.01 and abs(k.std() - 1.0) < 0.01              # N(0, 1)
    q = _f32(decode.q).astype(np.float64)
    assert abs(q.std() * math.sqrt(128) - 1.0) < 0.02                      # N(0, 1) / sqrt(128)
    w = decode.w
    assert w.dtype == np.float32 and w.min() >= 0.0 and w.max() < 1.0 / 8.0   # U[0, 1) / sqrt(64)
    assert abs(w.mean() * 16.0 - 1.0) < 0.05


def test_needle(decode):
    for b in (0, 1):
        S = decode.seq_lens[b]
        pos = decode.needle_pos[b]
        assert pos == math.floor(0.55 * S)
        v = _f32(decode.keys[b][pos]).astype(np.float64)
        assert abs(np.linalg.norm(v) - 4.0 * math.sqrt(128)) < 0.05 * 4.0 * math.sqrt(128)
        m = _f32(decode.q[b]).astype(np.float64).reshape(-1, 128).mean(axis=0)
        cos = v @ m / (np.linalg.norm(v) * np.linalg.norm(m))
        assert cos > 0.99                                                  # along the queries' mean


def test_block_tables_are_a_permutation_with_padding(decode):
    bt, bs = decode.block_table, decode.bs
    used = []
    for b, S in enumerate(decode.seq_lens):
        n = (S + bs - 1) // bs
        assert np.all(bt[b, :n] >= 0) and np.all(bt[b, n:] == -1)
        used.extend(bt[b, :n].tolist())
    assert sorted(used) == list(range(decode.num_blocks))                  # every block once, none shared
    assert used != sorted(used)                                            # shuffled


def test_prefill_rows_are_the_last_positions():
    t = wl.make_workload("p", [50, 80], [3, 5], seed=2)
    assert t.row_seq().tolist() == [0] * 3 + [1] * 5
    assert t.row_pos().tolist() == [47, 48, 49, 75, 76, 77, 78, 79]
    assert t.cu_seqlens_q().tolist() == [0, 3, 8]
