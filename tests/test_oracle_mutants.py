"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/orc.c (a dropped term, a
wrong constant, a transposed index, a reversed tie rule, an off-by-one in
the causal mask...), compiles it on the CPU and checks that the battery of
pin checks below -- the same kinds of checks as the other oracle tests --
rejects it, while the real oracle passes.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_idx_gb300 import workloads as wl
from tests import test_oracle_fp4 as fp4pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "orc.c")

MUTANTS = {
    "relu_dropped": ("float r = dot > 0.0f ? dot : 0.0f;", "float r = dot;"),
    "scale_constant": ("scale = amax / 448.0f;", "scale = amax / 447.0f;"),
    "q_transposed": ("float p = qf[h * d + i] * kf[i];", "float p = qf[i * H + h] * kf[i];"),
    "key_scale_dropped": ("acc = ks[s] * acc;", "acc = acc;"),
    "weight_dropped": ("float t = wq[h] * r;", "float t = r;"),
    "q_scale_not_folded": ("wq[h] = w[h] * sq;", "wq[h] = w[h];"),
    "ties_reversed": ("return (x->idx < y->idx) ? -1 : (x->idx > y->idx);",
                      "return (x->idx > y->idx) ? -1 : (x->idx < y->idx);"),
    "round_half_up": ("return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;", "return f + 1.0;"),
    "causal_off_by_one": ("int64_t nvis = row_pos[r] + 1 > 0 ? row_pos[r] + 1 : 0;",
                          "int64_t nvis = row_pos[r] > 0 ? row_pos[r] : 0;"),
    "scale_slot_stride": ("memcpy(base + (int64_t)bs * d + off * 4, &sc, 4);",
                          "memcpy(base + (int64_t)bs * d + off, &sc, 4);"),
    "subnormal_step": ("q = ldexp(1.0, -9);", "q = ldexp(1.0, -8);"),
    "wht_sign": ("s += orc_odd_parity((unsigned)(i & j)) ? -v : v;",
                 "s += orc_odd_parity((unsigned)(i & j)) ? v : -v;"),
    "wht_no_normalisation": ("const double c = 1.0 / sqrt((double)d);", "const double c = 1.0;"),
    "wht_index_or": ("s += orc_odd_parity((unsigned)(i & j)) ? -v : v;",
                     "s += orc_odd_parity((unsigned)(i | j)) ? -v : v;"),
    "bf16_round_half_up": ("u = u + 0x7FFFu + ((u >> 16) & 1u);", "u = u + 0x8000u;"),
    "translate_offset_dropped": ("out[i] = (int64_t)table_row[s / bs] * bs + s % bs;",
                                 "out[i] = (int64_t)table_row[s / bs] * bs;"),
    "e2m1_ties_odd": ("if (dist < bd || (dist == bd && (c & 1) == 0)) {",
                      "if (dist < bd || (dist == bd && (c & 1) == 1)) {"),
    "e2m1_no_saturation": ("if (a >= orc_e2m1_mag[7])", "if (a > 1e30)"),
    "fp4_block_64": ("#define ORC_FP4_BLOCK 32", "#define ORC_FP4_BLOCK 64"),
    "fp4_max_4": ("s = amax / 6.0f;", "s = amax / 4.0f;"),
    "fp4_scale_not_reapplied": ("y[b + j] = (float)(orc_e2m1_decode(orc_e2m1_encode(v)) * (double)s);",
                                "y[b + j] = (float)(orc_e2m1_decode(orc_e2m1_encode(v)));"),
}


def _torch_enc(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_dec(c):
    return torch.from_numpy(np.ascontiguousarray(c, np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def battery(O) -> bool:
    """True when every check passes for oracle instance O."""
    rng = np.random.default_rng(123)
    # encode against torch on a wide sample of magnitudes, incl. subnormals and ties
    x = np.concatenate([rng.standard_normal(20000) * 10 ** rng.uniform(-4, 2.6, 20000),
                        np.arange(1, 64) * 2.0 ** -10]).astype(np.float32)
    x = x[np.abs(x) < 464]
    if not np.array_equal(O.e4m3_encode(x), _torch_enc(x)):
        return False
    # quantisation: scale is amax / 448
    kb = wl.f32_to_bf16_bits(rng.standard_normal((200, 128)).astype(np.float32))
    kc, ks = O.quantize_rows(kb)
    kf = wl.bf16_bits_to_f32(kb)
    if not np.array_equal(ks, (np.abs(kf).max(1) / np.float32(448)).astype(np.float32)):
        return False
    # integer shadow of fp8 scores, H = 8
    q = wl.f32_to_bf16_bits((rng.standard_normal((8, 128)) / 11.3).astype(np.float32))
    w = rng.random(8).astype(np.float32)
    got = O.scores_row(O_FP8, q, w, (kc, ks), 200)
    qc, sq = O.quantize_rows(q)
    ki = np.rint(_torch_dec(kc) * 512)
    qi = np.rint(_torch_dec(qc) * 512)
    wq = (w * sq).astype(np.float32).astype(np.float64)
    shadow = ks * (np.maximum(ki @ qi.T / 512.0 ** 2, 0) @ wq)
    bound = ks * ((np.abs(ki) @ np.abs(qi).T / 512.0 ** 2) @ wq)
    if not np.all(np.abs(got - shadow) <= 140 * 2.0 ** -24 * bound + 1e-30):
        return False
    # brute-force top-k with ties
    s = (rng.integers(0, 3, 10) * 0.5).astype(np.float32)
    idx, _ = O.topk_row(s, 4)
    want = sorted(range(10), key=lambda i: (-float(s[i]), i))[:4]
    if idx.tolist() != want:
        return False
    # causal: the row at position p sees exactly p + 1 keys
    W = wl.make_workload("m", [20], [20], topk=8, seed=2)
    out = O.score_topk(O_BF16, 8, W.q, W.w, W.row_seq(), W.row_pos(), W.keys)
    for r, p in enumerate(W.row_pos()):
        sel = out["idx"][r][out["idx"][r] >= 0]
        if len(sel) != min(8, p + 1) or (len(sel) and sel.max() > p):
            return False
        if p + 1 <= 8 and set(sel.tolist()) != set(range(p + 1)):
            return False
    # Walsh-Hadamard rotation: the Kronecker-built Sylvester matrix over sqrt(d)
    E = np.zeros((128, 128), np.uint16)
    E[np.arange(128), np.arange(128)] = 0x3F80
    S = np.ones((1, 1))
    while S.shape[0] < 128:
        S = np.kron(np.array([[1.0, 1.0], [1.0, -1.0]]), S)
    if not np.array_equal(O.wht_rows(E), (S / np.sqrt(128.0)).astype(np.float32)):
        return False
    # float -> bf16 rounding against numpy, ties included
    xt = np.concatenate([rng.standard_normal(5000).astype(np.float32),
                         (np.arange(1, 500, dtype=np.uint32) << 16 | 0x8000).view(np.float32)])
    if not np.array_equal(O.f32_to_bf16(xt), wl.f32_to_bf16_bits(xt)):
        return False
    # store round trip at bs 64
    Wk = wl.make_workload("st", [100], [1], bs=64, seed=4)
    pool = np.zeros(Wk.num_blocks * 8448, np.uint8)
    O.store_keys(pool, Wk.all_keys(), Wk.all_slots(), 64, O_FP8)
    c2, s2 = O.gather_keys(pool, Wk.block_table[0], 100, 64, O_FP8)
    c1, s1 = O.quantize_rows(Wk.keys[0])
    if not (np.array_equal(c1, c2) and np.array_equal(s1, s2)):
        return False
    # translate: the slot of logical index s holds the gathered key s
    sl = O.translate_slots(Wk.block_table[0], 64, np.arange(100, dtype=np.int32))
    for s_, slot in enumerate(sl):
        blk, off = divmod(int(slot), 64)
        if not np.array_equal(pool[blk * 8448 + off * 128: blk * 8448 + off * 128 + 128], c2[s_]):
            return False
    # e2m1: every bf16 pattern against the decision boundaries
    b = np.arange(1 << 16, dtype=np.uint32)
    xb = (b << 16).view(np.float32)
    xb = xb[np.isfinite(xb)]
    if not np.array_equal(O.e2m1_encode(xb), fp4pins.encode_by_boundaries(xb)):
        return False
    # fp4 round trip: grid rows with power-of-two block scales are fixed points
    codes = rng.integers(0, 16, (8, 128))
    codes[:, ::32] = 7
    e = rng.integers(-10, 10, (8, 4)).repeat(32, axis=1)
    xg = (np.vectorize(fp4pins.e2m1_value)(codes) * 2.0 ** e).astype(np.float32)
    if not np.array_equal(O.fp4_roundtrip_rows(xg), xg):
        return False
    # blocks are 32 wide and independent
    xr = rng.standard_normal((4, 128)).astype(np.float32)
    yr = O.fp4_roundtrip_rows(xr)
    xo = xr.copy()
    xo[:, 32] *= np.float32(1000.0)
    if not np.array_equal(O.fp4_roundtrip_rows(xo)[:, :32], yr[:, :32]):
        return False
    return True


O_FP8, O_BF16 = oracle.FP8, oracle.BF16


def test_real_oracle_passes_battery():
    assert battery(oracle._default())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not found: " + old
    mpath = tmp_path / "orc_mut.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "liborc_mut.so"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c99",
                    "-D_DEFAULT_SOURCE", str(mpath), "-o", str(so), "-lm"], check=True)
    assert not battery(oracle.load_variant(str(so)))
