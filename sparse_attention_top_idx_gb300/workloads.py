"""Seeded synthetic inputs for the indexer path (shared by tests and bench).

This module holds no arithmetic of the method -- no quantisation, no scores,
no selection -- only the random inputs and the paging structure a caller would
hold: bf16 index keys per sequence, bf16 index queries, fp32 head weights, a
planted needle key, a block table and the slot mapping derived from it.

The shapes follow the workloads the pages describe:

* contexts of 2000, 4500, 10000 and 22000 tokens with top-512 selection and a
  planted needle -- "The Hypothesis That Refused to Die", section "Message
  12994: The Synthetic Test" (the needle is a key aligned with the query
  direction and scaled up, section "The Reasoning");
* the needle 55% of the way into the context -- "DeepSeek-V4 index_topk=1024
  sparse indexer can't recall verbatim lines" (ROCm/ATOM issue #1507), section
  "Reproduction (self-contained)";
* index_topk 512 and 1024, block sizes 64 and 32, max model length 1,048,576
  -- the same issue, sections "Environment" and "How it was isolated".

Distributions: keys iid N(0, 1); queries iid N(0, 1) / sqrt(d); head weights
U[0, 1) / sqrt(H); all rounded to bf16 (round to nearest even) where the path
takes bf16.  The needle is 4 * sqrt(d) * u, u the unit vector along the mean of
the sequence's fp32 queries over all (query, head) rows, placed at
floor(0.55 * S).  Block tables are random permutations of the physical blocks.
The pages' own data (real prompts, "realistic data") is not available; these
iid inputs stand in for it at the pages' context lengths.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

FP8 = 0
BF16 = 1


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    """One synthetic batch.

    seq_lens[b] keys per sequence; queries of sequence b are its last nq[b]
    positions (position = seq_len - nq + i).  keys[b]: bf16 bits [S_b, d].
    q: bf16 bits [sum(nq), H, d]; w: fp32 [sum(nq), H].
    block_table: int32 [B, max_blocks] (-1 where unused), num_blocks physical
    blocks of bs tokens.
    """
    name: str
    seq_lens: List[int]
    nq: List[int]
    H: int
    d: int
    topk: int
    bs: int
    keys: List[np.ndarray]
    q: np.ndarray
    w: np.ndarray
    needle_pos: List[int]
    block_table: np.ndarray
    num_blocks: int

    @property
    def batch(self) -> int:
        return len(self.seq_lens)

    @property
    def total_q(self) -> int:
        return int(sum(self.nq))

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(max(self.seq_lens)) if self.seq_lens else 0

    def cu_seqlens_q(self) -> np.ndarray:
        c = np.zeros(self.batch + 1, np.int32)
        c[1:] = np.cumsum(self.nq)
        return c

    def row_seq(self) -> np.ndarray:
        return np.repeat(np.arange(self.batch, dtype=np.int32), self.nq)

    def row_pos(self) -> np.ndarray:
        out = []
        for S, n in zip(self.seq_lens, self.nq):
            out.extend(range(S - n, S))
        return np.asarray(out, np.int64)

    def all_keys(self) -> np.ndarray:
        """Keys of every sequence concatenated, [sum(S), d] bf16 bits."""
        if not self.keys:
            return np.zeros((0, self.d), np.uint16)
        return np.concatenate(self.keys)

    def all_slots(self) -> np.ndarray:
        """Slot of every key of every sequence (same order as all_keys)."""
        return np.concatenate([slot_mapping(self.block_table[b], np.arange(S), self.bs)
                               for b, S in enumerate(self.seq_lens)]
                              ) if self.seq_lens else np.zeros(0, np.int64)


def slot_mapping(table_row: np.ndarray, positions: np.ndarray, bs: int) -> np.ndarray:
    """slot = physical block * bs + offset for logical positions of one sequence."""
    positions = np.asarray(positions, np.int64)
    return table_row[positions // bs].astype(np.int64) * bs + positions % bs


def make_block_table(rng: np.random.Generator, seq_lens, bs: int, extra_blocks: int = 0,
                     max_blocks: Optional[int] = None, permute: bool = True):
    """Random permutation of physical blocks handed out to the sequences."""
    nblk = [(S + bs - 1) // bs for S in seq_lens]
    total = int(sum(nblk)) + extra_blocks
    mb = max(max(nblk) if nblk else 1, 1) if max_blocks is None else max_blocks
    perm = rng.permutation(total).astype(np.int32) if permute else np.arange(total, dtype=np.int32)
    table = np.full((len(seq_lens), mb), -1, np.int32)
    o = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[o:o + n]
        o += n
    return table, max(total, 1)


def make_workload(name: str, seq_lens, nq, *, H: int = 64, d: int = 128, topk: int = 512,
                  bs: int = 64, seed: int = 0, needle: bool = True, permute: bool = True,
                  extra_blocks: int = 0, max_blocks: Optional[int] = None) -> Workload:
    seq_lens = [int(s) for s in seq_lens]
    nq = [int(n) for n in (nq if hasattr(nq, "__len__") else [nq] * len(seq_lens))]
    ss = np.random.SeedSequence(seed)
    kids = ss.spawn(len(seq_lens) + 1)
    keys, qs, ws, npos = [], [], [], []
    for b, (S, n) in enumerate(zip(seq_lens, nq)):
        rng = np.random.Generator(np.random.PCG64(kids[b]))
        k32 = rng.standard_normal((S, d), dtype=np.float32)
        q32 = rng.standard_normal((n, H, d), dtype=np.float32) / np.float32(math.sqrt(d))
        w32 = (rng.random((n, H), dtype=np.float32) / np.float32(math.sqrt(H))).astype(np.float32)
        pos = int(math.floor(0.55 * S))
        if needle and S > 0 and n > 0:
            m = q32.reshape(-1, d).astype(np.float64).mean(axis=0)
            u = m / np.linalg.norm(m)
            k32[pos] = (4.0 * math.sqrt(d) * u).astype(np.float32)
        keys.append(f32_to_bf16_bits(k32))
        qs.append(f32_to_bf16_bits(q32))
        ws.append(w32)
        npos.append(pos)
    rng = np.random.Generator(np.random.PCG64(kids[-1]))
    table, nblocks = make_block_table(rng, seq_lens, bs, extra_blocks, max_blocks, permute)
    q = np.concatenate(qs) if qs else np.zeros((0, H, d), np.uint16)
    w = np.concatenate(ws) if ws else np.zeros((0, H), np.float32)
    return Workload(name, seq_lens, nq, H, d, topk, bs, keys, q, w, npos, table, nblocks)


# The five workloads: a tiny causal chunk, a decode batch, a long causal
# prefill chunk, the fp8-vs-bf16 precision comparison and a long-context
# decode batch.  Seeds are 1000 + the workload number.
def tiny_prefill(seed: int = 1001) -> Workload:
    """1 sequence of 2000 keys, its last 16 positions as queries, top-512."""
    return make_workload("tiny_s2000_t16_top512", [2000], [16], topk=512, seed=seed)


def decode_batch(seed: int = 1002) -> Workload:
    """32 sequences alternating 4500 / 10000 keys, 1 query each, top-512."""
    lens = [4500 if i % 2 == 0 else 10000 for i in range(32)]
    return make_workload("decode_b32_s4500_10000_top512", lens, [1] * 32, topk=512, seed=seed)


def prefill_chunk(seed: int = 1003, T: int = 8192, S: int = 22000) -> Workload:
    """1 sequence of 22000 keys, queries at its last 8192 positions, top-1024."""
    return make_workload("prefill_s22000_t8192_top1024", [S], [T], topk=1024, seed=seed)


def precision_compare(seed: int = 1004, topk: int = 512) -> Workload:
    """4 sequences of 2000 / 4500 / 10000 / 22000 keys, 1 query each."""
    return make_workload("precision_s2000_4500_10000_22000", [2000, 4500, 10000, 22000],
                         [1] * 4, topk=topk, seed=seed)


def long_context(seed: int = 1005) -> Workload:
    """8 sequences of 131072 keys plus 1 of 1048576, 1 query each, top-1024."""
    lens = [131072] * 8 + [1048576]
    return make_workload("longctx_b8x131072_1x1048576_top1024", lens, [1] * 9, topk=1024,
                         seed=seed)


WORKLOADS = {
    "tiny": tiny_prefill,
    "decode": decode_batch,
    "prefill": prefill_chunk,
    "precision": precision_compare,
    "longctx": long_context,
}
