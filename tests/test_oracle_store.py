"""Pins for the oracle's paged key store and gather.

"DeepSeek-V4 index_topk=1024 sparse indexer can't recall verbatim lines"
(ROCm/ATOM issue #1507), section "How it was isolated": index keys are
quantised and scattered into a paged cache (block sizes 32 and 64) and read
back through a gather, with the write/read round trip exact (zero error in
codes, scales and keys).  The record sizes are those of "The Pivot: A Single
Edit That Finally Fixed DeepSeek V4's Long-Context Recall Failure", section
"Assumptions and Input Knowledge": 132 bytes per token in fp8, 256 in bf16.
"""
import numpy as np
import pytest

import oracle
from sparse_attention_top_idx_gb300 import workloads as wl


def test_block_bytes():
    assert oracle.block_bytes(oracle.FP8, 64) == 64 * 132 == 8448
    assert oracle.block_bytes(oracle.FP8, 32) == 32 * 132
    assert oracle.block_bytes(oracle.BF16, 64) == 64 * 256


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("mode", [0, 1])
def test_store_gather_roundtrip(bs, mode):
    W = wl.make_workload("rt", [130, 64, 1, 257], [1, 1, 1, 1], bs=bs, seed=bs + mode,
                         extra_blocks=3)
    bb = oracle.block_bytes(mode, bs)
    pool = np.full(W.num_blocks * bb, 0xA5, np.uint8)
    n = oracle.store_keys(pool, W.all_keys(), W.all_slots(), bs, mode)
    assert n == sum(W.seq_lens)
    for b, S in enumerate(W.seq_lens):
        got = oracle.gather_keys(pool, W.block_table[b], S, bs, mode)
        if mode == oracle.FP8:
            c, s = oracle.quantize_rows(W.keys[b])
            assert np.array_equal(got[0], c) and np.array_equal(got[1].view(np.uint32),
                                                                s.view(np.uint32))
        else:
            assert np.array_equal(got, W.keys[b])
    # the untouched tail of partially filled blocks and the spare blocks keep
    # their canary bytes
    written = np.zeros(W.num_blocks * bs, bool)
    written[W.all_slots()] = True
    blocks = pool.reshape(W.num_blocks, bb)
    for blk in range(W.num_blocks):
        for off in range(bs):
            if written[blk * bs + off]:
                continue
            if mode == oracle.FP8:
                assert np.all(blocks[blk, off * 128:(off + 1) * 128] == 0xA5)
                assert np.all(blocks[blk, bs * 128 + off * 4: bs * 128 + off * 4 + 4] == 0xA5)
            else:
                assert np.all(blocks[blk, off * 256:(off + 1) * 256] == 0xA5)


def test_fp8_block_layout():
    # A block holds bs rows of 128 codes followed by bs fp32 scales.
    bs = 64
    rng = np.random.default_rng(0)
    k = wl.f32_to_bf16_bits(rng.standard_normal((3, 128)).astype(np.float32))
    pool = np.zeros(2 * 8448, np.uint8)
    oracle.store_keys(pool, k, np.array([64 + 5, 2, -1], np.int64), bs, oracle.FP8)
    c, s = oracle.quantize_rows(k)
    assert np.array_equal(pool[8448 + 5 * 128: 8448 + 6 * 128], c[0])
    assert np.array_equal(pool[8448 + 8192 + 20: 8448 + 8192 + 24].view(np.float32), s[:1])
    assert np.array_equal(pool[2 * 128: 3 * 128], c[1])
    # slot -1 is skipped: nothing else in the pool is written
    mask = np.ones(pool.size, bool)
    for a, b in [(8448 + 640, 8448 + 768), (8448 + 8212, 8448 + 8216), (256, 384),
                 (8192 + 8, 8192 + 12)]:
        mask[a:b] = False
    assert np.all(pool[mask] == 0)


def test_store_rejects_out_of_range_slot():
    pool = np.zeros(8448, np.uint8)
    k = np.zeros((1, 128), np.uint16)
    with pytest.raises(ValueError):
        oracle.store_keys(pool, k, np.array([64], np.int64), 64, oracle.FP8)


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("dtype", [oracle.FP8, oracle.BF16])
def test_translate_is_the_block_table_gather(bs, dtype):
    # the token at physical slot translate(s) is the key the block-table gather
    # returns for logical index s (ROCm/ATOM #1507, "How it was isolated": the
    # translate feeds sparse attention the rows the indexer selected)
    W = wl.make_workload("tr", [700, 129], [1, 1], bs=bs, seed=61 + bs + dtype, extra_blocks=3)
    bb = oracle.block_bytes(dtype, bs)
    pool = np.zeros(W.num_blocks * bb, np.uint8)
    oracle.store_keys(pool, W.all_keys(), W.all_slots(), bs, dtype)
    for b in range(W.batch):
        S = W.seq_lens[b]
        idx = np.concatenate([np.arange(S), [-1, -1]]).astype(np.int32)
        slots = oracle.translate_slots(W.block_table[b], bs, idx)
        assert np.all(slots[-2:] == -1)
        g = oracle.gather_keys(pool, W.block_table[b], S, bs, dtype)
        for s, sl in zip(idx[:-2], slots[:-2]):
            blk, off = divmod(int(sl), bs)
            base = blk * bb
            if dtype == oracle.FP8:
                codes = pool[base + off * 128: base + off * 128 + 128]
                scale = pool[base + bs * 128 + off * 4: base + bs * 128 + off * 4 + 4].view(np.float32)[0]
                assert np.array_equal(codes, g[0][s]) and scale == g[1][s]
            else:
                assert np.array_equal(pool[base + off * 256: base + off * 256 + 256].view(np.uint16), g[s])
    # an index whose block lies past the table row
    assert oracle.translate_slots(np.array([3, 4], np.int32), bs, np.array([2 * bs], np.int32))[0] == -1
