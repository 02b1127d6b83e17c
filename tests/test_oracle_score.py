"""Pins for the oracle's indexer scores.

The score is the one "The Hypothesis That Refused to Die" (section "The
Context") describes as a compressed query-key dot product used to rank every
cached position, written out as

    score[t, s] = sum_h w[t, h] * ReLU(q[t, h] . k[s])

accumulated in fp32.  With fp8 keys each key carries a per-token fp32 scale
(the 132-byte record of "The Pivot: A Single Edit That Finally Fixed
DeepSeek V4's Long-Context Recall Failure", section "Assumptions and Input
Knowledge"), and the query is fp8 as well (ROCm/ATOM issue #1507, "Root cause
found": RoPE + Hadamard + fp8 quant of the index query), its per-(t, h) scale
folded into w.

Pins used here, none of which re-runs the oracle's own loops (the fp32
results are held to the standard rounding-error bound of a length-n fp32
sum, (n + 1) u times the sum of magnitudes):
* an exact integer shadow: e4m3 values are multiples of 2^-9, so code values
  times 512 are integers and the dot products are exact int64 matmuls (numpy),
  with the codes decoded by PyTorch's float8_e4m3fn, not by the oracle;
* closed forms: a one-hot key with one head reduces the score to w * ReLU(q_j)
  (bf16, exact) or to w' * q-code * 448 * key-scale (fp8);
* invariants: scaling a key by 2 doubles its score exactly, a key opposite
  every query scores exactly 0, linearity in w;
* a planted needle ranks first.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_idx_gb300 import workloads as wl
from sparse_attention_top_idx_gb300.workloads import f32_to_bf16_bits


def torch_decode(c):
    return torch.from_numpy(np.ascontiguousarray(c, np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def rand_case(rng, S, H, d=128):
    k = f32_to_bf16_bits(rng.standard_normal((S, d)).astype(np.float32))
    q = f32_to_bf16_bits((rng.standard_normal((H, d)) / np.sqrt(d)).astype(np.float32))
    w = (rng.random(H) / np.sqrt(H)).astype(np.float32)
    return k, q, w


@pytest.mark.parametrize("H", [1, 7, 64])
def test_fp8_scores_against_integer_shadow(H):
    rng = np.random.default_rng(11 + H)
    S = 300
    k, q, w = rand_case(rng, S, H)
    kc, ks = oracle.quantize_rows(k)
    qc, sq = oracle.quantize_rows(q)
    got, ex = oracle.scores_row(oracle.FP8, q, w, (kc, ks), S, exact=True)
    # integer shadow of the code dot products
    ki = np.rint(torch_decode(kc) * 512).astype(np.int64)
    qi = np.rint(torch_decode(qc) * 512).astype(np.int64)
    dots = (ki @ qi.T).astype(np.float64) / (512.0 * 512.0)       # [S, H], exact
    wq = (w * sq).astype(np.float32).astype(np.float64)           # w' = fl32(w * sq)
    shadow = ks.astype(np.float64) * (np.maximum(dots, 0.0) @ wq)
    assert np.allclose(ex, shadow, rtol=1e-12, atol=0)
    # fp32 evaluation error bound (Higham, sums of d products then H terms)
    bound = ks.astype(np.float64) * ((np.abs(ki) @ np.abs(qi).T / 512.0 ** 2) @ wq)
    assert np.all(np.abs(got - shadow) <= (128 + H + 3) * 2.0 ** -24 * bound)


@pytest.mark.parametrize("H", [1, 5, 64])
def test_bf16_scores_against_fp64(H):
    rng = np.random.default_rng(21 + H)
    S = 300
    k, q, w = rand_case(rng, S, H)
    got, ex = oracle.scores_row(oracle.BF16, q, w, k, S, exact=True)
    kf = wl.bf16_bits_to_f32(k).astype(np.float64)
    qf = wl.bf16_bits_to_f32(q).astype(np.float64)
    ref = np.maximum(kf @ qf.T, 0.0) @ w.astype(np.float64)
    assert np.allclose(ex, ref, rtol=1e-12, atol=1e-300)
    bound = (np.abs(kf) @ np.abs(qf).T) @ w.astype(np.float64)
    assert np.all(np.abs(got - ref) <= (128 + H + 3) * 2.0 ** -24 * bound)


def test_one_hot_key_closed_form():
    rng = np.random.default_rng(5)
    d = 128
    q32 = (rng.standard_normal((1, d)) / np.sqrt(d)).astype(np.float32)
    q = f32_to_bf16_bits(q32)
    qf = wl.bf16_bits_to_f32(q)[0]
    w = np.array([0.75], np.float32)
    keys = np.zeros((d, d), np.float32)
    keys[np.arange(d), np.arange(d)] = 1.0
    kb = f32_to_bf16_bits(keys)
    # bf16: score = w * ReLU(q_j), exact
    got = oracle.scores_row(oracle.BF16, q, w, kb, d)
    want = (w[0] * np.maximum(qf, 0)).astype(np.float32)
    assert np.array_equal(got, want)
    # fp8: the key's only code is 448 (0x7E) with scale 1/448; the score is
    # fl32(ks * fl32(w' * fl32(qcode_j * 448)))
    kc, ks = oracle.quantize_rows(kb)
    assert np.all(kc[np.arange(d), np.arange(d)] == 0x7E)
    assert np.all(ks == np.float32(1.0) / np.float32(448.0))
    qc, sq = oracle.quantize_rows(q)
    qv = torch_decode(qc[0]).astype(np.float32)
    wq = np.float32(w[0] * sq[0])
    got8 = oracle.scores_row(oracle.FP8, q, w, (kc, ks), d)
    dot = (qv * np.float32(448.0)).astype(np.float32)
    want8 = (ks * (wq * np.maximum(dot, np.float32(0)))).astype(np.float32)
    assert np.array_equal(got8, want8)
    # and it approximates w * ReLU(q_j) within the query's fp8 error
    assert np.allclose(got8, w[0] * np.maximum(qf, 0), rtol=0.07, atol=float(sq[0]) * 0.75)


def test_invariants_scale_relu_linearity():
    rng = np.random.default_rng(9)
    S, H = 64, 16
    k, q, w = rand_case(rng, S, H)
    kf = wl.bf16_bits_to_f32(k)
    # doubling a key (exact in bf16) doubles its score exactly, in both modes
    k2 = f32_to_bf16_bits(kf * 2)
    for mode in (oracle.FP8, oracle.BF16):
        def sc(kk):
            keys = oracle.quantize_rows(kk) if mode == oracle.FP8 else kk
            return oracle.scores_row(mode, q, w, keys, S)
        assert np.array_equal(sc(k2), 2 * sc(k))
    # a key opposite to every query head scores exactly zero
    qf = wl.bf16_bits_to_f32(q)
    anti = f32_to_bf16_bits(-np.sign(qf.sum(0))[None, :] * np.ones((1, 128), np.float32))
    qpos = f32_to_bf16_bits(np.abs(qf) * np.sign(qf.sum(0))[None, :])
    for mode in (oracle.FP8, oracle.BF16):
        keys = oracle.quantize_rows(anti) if mode == oracle.FP8 else anti
        assert oracle.scores_row(mode, qpos, w, keys, 1)[0] == 0.0
    # linear in w (to fp32 rounding)
    w1 = (rng.random(H) * 0.1).astype(np.float32)
    w2 = (rng.random(H) * 0.1).astype(np.float32)
    for mode in (oracle.FP8, oracle.BF16):
        keys = oracle.quantize_rows(k) if mode == oracle.FP8 else k
        a = oracle.scores_row(mode, q, w1, keys, S)
        b = oracle.scores_row(mode, q, w2, keys, S)
        c = oracle.scores_row(mode, q, (w1 + w2).astype(np.float32), keys, S)
        assert np.allclose(a + b, c, rtol=2e-5)
    # a head with zero weight contributes nothing: dropping it changes nothing
    wz = w.copy()
    wz[3] = 0
    keep = [h for h in range(H) if h != 3]
    for mode in (oracle.FP8, oracle.BF16):
        keys = oracle.quantize_rows(k) if mode == oracle.FP8 else k
        a = oracle.scores_row(mode, q, wz, keys, S)
        b = oracle.scores_row(mode, q[keep], wz[keep], keys, S)
        assert np.array_equal(a, b)


@pytest.mark.parametrize("mode", [0, 1])
def test_needle_ranks_first(mode):
    W = wl.precision_compare()
    for b, S in enumerate(W.seq_lens):
        keys = oracle.quantize_rows(W.keys[b]) if mode == oracle.FP8 else W.keys[b]
        sc = oracle.scores_row(mode, W.q[b], W.w[b], keys, S)
        assert oracle.needle_rank(sc, W.needle_pos[b]) == 1
