"""Pins of the oracle's Walsh-Hadamard key rotation (orc_wht_row) and of the
rotated key store.

"DeepSeek-V4 index_topk=1024 sparse indexer can't recall verbatim lines"
(ROCm/ATOM issue #1507), section "Root cause": the index query is
Walsh-Hadamard rotated and fix (B) rotates the key the same way on the store
path; the rotation is orthogonal, so (Hq).(Hk) = q.k.  Reading: H is the
orthonormal 128-point transform in Sylvester order, H = S / sqrt(128) with
S = [[1, 1], [1, -1]] Kronecker-multiplied by itself seven times.

The checks do not retype the oracle's formula: the matrix is built here by
Kronecker products, values are compared with exact integer sums and
50-digit decimals, and the store is compared through numpy's and torch's
own rounding."""
import decimal

import numpy as np
import torch

import oracle
from sparse_attention_top_idx_gb300 import workloads as wl

D = 128


def sylvester(n: int) -> np.ndarray:
    S = np.ones((1, 1), np.int64)
    while S.shape[0] < n:
        S = np.kron(np.array([[1, 1], [1, -1]], np.int64), S)
    return S


def identity_rows():
    E = np.zeros((D, D), np.uint16)
    E[np.arange(D), np.arange(D)] = 0x3F80      # bf16 1.0
    return E


def test_sylvester_helper_is_a_hadamard_matrix():
    S = sylvester(D)
    assert np.array_equal(S @ S.T, D * np.eye(D, dtype=np.int64))
    assert np.all(S[0] == 1) and np.all(S[:, 0] == 1)


def test_rotation_matrix_is_sylvester_over_sqrt_d():
    # row j of the output is H applied to unit vector e_j, i.e. column j of H
    M = oracle.wht_rows(identity_rows())
    want = (sylvester(D).astype(np.float64) / np.sqrt(D)).astype(np.float32)
    assert np.array_equal(M, want.T)
    Mf = M.astype(np.float64)
    assert np.abs(Mf @ Mf.T - np.eye(D)).max() < 1e-6


def test_dot_products_are_invariant():
    rng = np.random.default_rng(5)
    q = wl.f32_to_bf16_bits(rng.standard_normal((64, D)).astype(np.float32))
    k = wl.f32_to_bf16_bits(rng.standard_normal((64, D)).astype(np.float32))
    qf, kf = wl.bf16_bits_to_f32(q).astype(np.float64), wl.bf16_bits_to_f32(k).astype(np.float64)
    qr, kr = oracle.wht_rows(q).astype(np.float64), oracle.wht_rows(k).astype(np.float64)
    ref = qf @ kf.T
    got = qr @ kr.T
    bound = np.linalg.norm(qf, axis=1)[:, None] * np.linalg.norm(kf, axis=1)[None, :]
    assert np.all(np.abs(got - ref) <= 1e-6 * bound)
    assert np.allclose(np.linalg.norm(qr, axis=1), np.linalg.norm(qf, axis=1), rtol=1e-6)


def _ulp32(x: float) -> float:
    return float(np.spacing(np.float32(abs(x)))) if x != 0.0 else 2.0 ** -149


def test_exact_rational_inputs():
    # small integers are exact in bf16; S x is an exact integer vector and the
    # result must be within half an fp32 ulp (plus the double rounding of the
    # constant, far below that) of S x / sqrt(128), exactly 0 where S x is 0
    cases = [np.arange(D), np.ones(D, np.int64), (np.arange(D) % 7) - 3, np.eye(D, dtype=np.int64)[5] * 96]
    decimal.getcontext().prec = 50
    inv = decimal.Decimal(1) / decimal.Decimal(D).sqrt()
    for x in cases:
        bits = wl.f32_to_bf16_bits(x.astype(np.float32))
        assert np.array_equal(wl.bf16_bits_to_f32(bits), x.astype(np.float32))
        y = oracle.wht_rows(bits[None, :])[0]
        exact = sylvester(D) @ x.astype(np.int64)
        for i in range(D):
            e = decimal.Decimal(int(exact[i])) * inv
            if exact[i] == 0:
                assert y[i] == 0.0
            else:
                assert abs(decimal.Decimal(float(y[i])) - e) <= decimal.Decimal(0.5 * _ulp32(float(e)) * (1 + 2.0 ** -20))
    # all-ones: the energy moves to entry 0, sqrt(128)
    ones = oracle.wht_rows(wl.f32_to_bf16_bits(np.ones((1, D), np.float32)))[0]
    assert np.all(ones[1:] == 0.0) and abs(float(ones[0]) - 128 ** 0.5) <= 0.5 * _ulp32(128 ** 0.5)


def test_bf16_rounding_matches_numpy_rne():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(50000) * 10.0 ** rng.uniform(-5, 5, 50000)).astype(np.float32)
    # exact halfway cases: low 16 bits 0x8000 with both parities of bit 16
    tie = (np.arange(1, 2001, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, tie, -tie])
    assert np.array_equal(oracle.f32_to_bf16(x), wl.f32_to_bf16_bits(x))


def test_rotated_store_fp8_and_bf16():
    W = wl.make_workload("rot", [150, 70], [1, 1], bs=64, seed=12)
    for dtype in (oracle.FP8, oracle.BF16):
        pool = np.zeros(W.num_blocks * oracle.block_bytes(dtype, 64), np.uint8)
        assert oracle.store_keys(pool, W.all_keys(), W.all_slots(), 64, dtype, rotate=True) == 220
        for b in range(W.batch):
            y = oracle.wht_rows(W.keys[b])
            got = oracle.gather_keys(pool, W.block_table[b], W.seq_lens[b], 64, dtype)
            if dtype == oracle.FP8:
                codes, scales = got
                amax = np.abs(y).max(1)
                assert np.array_equal(scales, (amax / np.float32(448)).astype(np.float32))
                ratio = (y / scales[:, None]).astype(np.float32)
                want = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                assert np.array_equal(codes, want)
            else:
                assert np.array_equal(got, wl.f32_to_bf16_bits(y))
