"""Pins of the oracle's fp4 (e2m1) round trip with block-32 scales.

The round trip is the key-path step fp4_act_quant_inplace(kv, 32) of
"DeepSeek-V4 index_topk=1024 sparse indexer can't recall verbatim lines"
(ROCm/ATOM issue #1507, section "Where (main 0c7d50f9)").  The e2m1 values
are derived here from the format's bit fields (1 sign, 2 exponent bits with
bias 1, 1 mantissa bit; exponent field 0 is the subnormal 0.5 * m), not
copied from the oracle's table, and the encoder is checked against the
decision boundaries (midpoints between neighbours) rather than against a
second nearest-value search.
"""
from fractions import Fraction

import numpy as np

import oracle
from sparse_attention_top_idx_gb300 import workloads as wl

O = oracle._default()


def e2m1_value(code: int) -> float:
    """Value of a 4-bit e2m1 code from its bit fields."""
    sign = -1.0 if code & 8 else 1.0
    e, m = (code >> 1) & 3, code & 1
    mag = 0.5 * m if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return sign * mag


GRID = np.array([e2m1_value(c) for c in range(8)])
MIDS = (GRID[:-1] + GRID[1:]) / 2          # decision boundaries 0.25 .. 5


def encode_by_boundaries(x):
    """e2m1 code from the boundaries: the number of midpoints below |x|; a
    value exactly on a midpoint goes to the even one of its two codes."""
    a = np.abs(x.astype(np.float64))
    k = np.searchsorted(MIDS, a, side="left")          # midpoints strictly below
    on = (k < len(MIDS)) & (a == MIDS[np.minimum(k, len(MIDS) - 1)])
    code = np.where(on & (k % 2 == 1), k + 1, k)       # tie between k and k + 1: the even one
    return (code | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def test_grid_from_bit_fields():
    assert GRID.tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_grid_points_are_fixed():
    for c in range(16):
        v = np.float32(e2m1_value(c))
        if c == 8:
            v = np.float32(-0.0)
        assert O.e2m1_encode(np.array([v]))[0] == c


def test_encode_every_bf16_pattern():
    # every finite bf16 value (both signs), as fp32
    b = np.arange(1 << 16, dtype=np.uint32)
    x = (b << 16).view(np.float32)
    x = x[np.isfinite(x)]
    assert np.array_equal(O.e2m1_encode(x), encode_by_boundaries(x))


def test_encode_around_each_boundary():
    # 4096 fp32 neighbours on each side of every midpoint, and the midpoints
    xs = []
    for m in MIDS:
        c = np.float32(m).view(np.uint32)
        xs.append((c + np.arange(-4096, 4097, dtype=np.int64)).astype(np.uint32).view(np.float32))
    x = np.concatenate(xs)
    x = np.concatenate([x, -x])
    assert np.array_equal(O.e2m1_encode(x), encode_by_boundaries(x))


def test_ties_go_to_the_even_code():
    got = O.e2m1_encode(MIDS.astype(np.float32))
    # 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0, 5 -> 4.0
    assert [e2m1_value(int(c)) for c in got] == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_saturation_and_sign():
    x = np.array([6.0, 6.5, 100.0, 3.0e38, -7.0, -0.1], np.float32)
    assert O.e2m1_encode(x).tolist() == [7, 7, 7, 7, 15, 8]


def _rows(seed, R=64):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, 128)) * 10.0 ** rng.uniform(-3, 3, (R, 4)).repeat(32, axis=1)
    return x.astype(np.float32)


def test_roundtrip_scale_is_block_amax_over_6():
    x = _rows(1)
    y = O.fp4_roundtrip_rows(x)
    for r in range(8):
        for b in range(4):
            blk = x[r, 32 * b:32 * b + 32]
            s = np.float32(np.abs(blk).max()) / np.float32(6)
            # the block's largest magnitude is 6 * s after the round trip
            j = int(np.argmax(np.abs(blk)))
            assert y[r, 32 * b + j] == np.float32(np.copysign(np.float64(6.0) * np.float64(s), blk[j]))
            # every output is a grid value times s
            q = y[r, 32 * b:32 * b + 32].astype(np.float64) / np.float64(s)
            assert np.all(np.isin(np.round(np.abs(q), 6), GRID))


def test_roundtrip_error_bound():
    # nearest grid point: |x - y| <= half the widest gap (1, between 4 and 6)
    # times s, and <= s / 4 where |x / s| <= 2 (gaps of 0.5 there)
    x = _rows(2)
    y = O.fp4_roundtrip_rows(x)
    s = (np.abs(x).reshape(-1, 4, 32).max(2) / np.float32(6)).astype(np.float32).repeat(32, axis=1)
    err = np.abs(x.astype(np.float64) - y) / s
    assert np.all(err <= 1.0 + 1e-6)
    small = np.abs(x) / s <= 2.0
    assert np.all(err[small] <= 0.25 + 1e-6)


def test_roundtrip_blocks_are_independent_and_32_wide():
    x = _rows(3, R=4)
    y = O.fp4_roundtrip_rows(x)
    x2 = x.copy()
    x2[:, 32] *= np.float32(1000.0)        # an outlier in the second block
    y2 = O.fp4_roundtrip_rows(x2)
    assert np.array_equal(y2[:, :32], y[:, :32])
    assert np.array_equal(y2[:, 64:], y[:, 64:])
    assert not np.array_equal(y2[:, 33:64], y[:, 33:64])


def test_roundtrip_fixed_points_zero_blocks_and_signs():
    rng = np.random.default_rng(4)
    # rows already on the grid with power-of-two block scales survive exactly
    codes = rng.integers(0, 16, (16, 128))
    codes[:, ::32] = 7                        # each block reaches 6, so s = 2^e exactly
    e = rng.integers(-20, 20, (16, 4)).repeat(32, axis=1)
    x = (np.vectorize(e2m1_value)(codes) * 2.0 ** e).astype(np.float32)
    assert np.array_equal(O.fp4_roundtrip_rows(x), x)
    z = np.zeros((2, 128), np.float32)
    z[0, :32] = -0.0
    y = O.fp4_roundtrip_rows(z)
    assert np.array_equal(y.view(np.uint32), z.view(np.uint32))
    v = _rows(5, R=8)
    assert np.array_equal(O.fp4_roundtrip_rows(-v), -O.fp4_roundtrip_rows(v))


def test_roundtrip_brute_force_exact_rationals():
    # tiny case in exact arithmetic: fl32 scale and quotient, nearest grid
    # value with ties to the even code, fl32 product
    x = _rows(6, R=2)
    y = O.fp4_roundtrip_rows(x)
    for r in range(2):
        for b in range(4):
            blk = x[r, 32 * b:32 * b + 32]
            s = np.float32(np.abs(blk).max()) / np.float32(6)
            for j in range(32):
                v = Fraction(float(np.float32(blk[j]) / s))
                best = min(range(8), key=lambda c: (abs(abs(v) - Fraction(GRID[c])), c & 1))
                want = np.float32(float(Fraction(GRID[best]) * Fraction(float(s))) * (1 if blk[j] >= 0 else -1))
                assert y[r, 32 * b + j] == want


def test_store_with_fp4_roundtrip_keeps_the_quantised_roundtrip():
    W = wl.make_workload("fp4st", [70], [1], bs=32, seed=7)
    for dt in (oracle.FP8, oracle.BF16):
        for rot in (False, True):
            bb = O.block_bytes(dt, 32)
            pool = np.zeros(W.num_blocks * bb, np.uint8)
            O.store_keys(pool, W.all_keys(), W.all_slots(), 32, dt, rotate=rot, fp4=True)
            got = O.gather_keys(pool, W.block_table[0], 70, 32, dt)
            y = O.wht_rows(W.keys[0]) if rot else wl.bf16_bits_to_f32(W.keys[0])
            want = (O.quantize_rows_f32(O.fp4_roundtrip_rows(y)) if dt == oracle.FP8
                    else O.f32_to_bf16(O.fp4_roundtrip_rows(y)))
            if dt == oracle.FP8:
                assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
            else:
                assert np.array_equal(got, want)
