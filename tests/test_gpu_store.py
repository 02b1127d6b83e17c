"""GPU parity of idx_store_keys against the oracle's store: every byte of the
pool (codes, scales, untouched canary bytes) must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_idx_gb300 import dsaidx
from sparse_attention_top_idx_gb300 import workloads as wl
from tests.parity import bf16_tensor

pytestmark = pytest.mark.gpu


def oracle_pool(W, mode, k_bits, slots, fill=0xA5):
    bb = oracle.block_bytes(mode, W.bs)
    pool = np.full(W.num_blocks * bb, fill, np.uint8)
    oracle.store_keys(pool, k_bits, slots, W.bs, mode)
    return pool


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("mode", [0, 1])
def test_store_bit_exact(bs, mode):
    W = wl.make_workload("st", [1000, 77, 64, 3000], [1, 1, 1, 1], bs=bs, seed=10 + bs + mode,
                         extra_blocks=5)
    k = W.all_keys().copy()
    slots = W.all_slots().copy()
    # some tokens skipped with a negative slot
    slots[::17] = -1
    # keys over a wide range of magnitudes, including tiny rows that hit the
    # e4m3 subnormals and an all-zero row
    rng = np.random.default_rng(bs + mode)
    scale = (10.0 ** rng.uniform(-30, 30, (k.shape[0], 1))).astype(np.float32)
    kf = wl.bf16_bits_to_f32(k) * scale
    kf[5] = 0.0
    k = wl.f32_to_bf16_bits(kf)
    cache = dsaidx.IndexCache.allocate(W.num_blocks, bs, mode, fill=0xA5)
    dsaidx.store_keys(cache, bf16_tensor(k), torch.from_numpy(slots).cuda())
    got = cache.pool.cpu().numpy()
    want = oracle_pool(W, mode, k, slots)
    diff = np.nonzero(got != want)[0]
    assert diff.size == 0, "first differing byte %d of %d" % (diff[0], diff.size)


@pytest.mark.parametrize("amax", [448.0, 1344.0, 336.0, 1000.0])
def test_e4m3_convert_every_bf16_below_amax(amax):
    # Every finite bf16 magnitude up to amax, both signs, in rows whose
    # largest magnitude is amax, against the oracle's encoder.  amax = 448
    # gives scale exactly 1 (the codes are the e4m3 encodings of the bf16
    # values themselves); 1344, 336 and 1000 give scales 3, 0.75 and 1000/448,
    # where x / scale is inexact and its correct rounding decides ties.
    top = int(wl.f32_to_bf16_bits(np.array([amax], np.float32))[0])
    pos = np.arange(0, top + 1, dtype=np.uint16)
    vals = np.concatenate([pos, pos | 0x8000])
    per = 127
    nrows = (len(vals) + per - 1) // per
    rows = np.zeros((nrows, 128), np.uint16)
    rows[:, 0] = top
    flat = np.zeros(nrows * per, np.uint16)
    flat[:len(vals)] = vals
    rows[:, 1:] = flat.reshape(nrows, per)
    bs = 64
    nblk = (nrows + bs - 1) // bs
    cache = dsaidx.IndexCache.allocate(nblk, bs, dsaidx.FP8, fill=0)
    slots = np.arange(nrows, dtype=np.int64)
    dsaidx.store_keys(cache, bf16_tensor(rows), torch.from_numpy(slots).cuda())
    got = cache.pool.cpu().numpy().reshape(nblk, 8448)
    codes = np.concatenate([got[b, :bs * 128].reshape(bs, 128) for b in range(nblk)])[:nrows]
    scales = np.concatenate([got[b, bs * 128:].view(np.float32) for b in range(nblk)])[:nrows]
    want, want_s = oracle.quantize_rows(rows)
    assert np.array_equal(scales.view(np.uint32), want_s.view(np.uint32))
    if amax == 448.0:
        assert np.all(scales == 1.0)
    assert np.array_equal(codes, want)


def test_out_of_range_slot_sets_status_and_skips():
    bs = 64
    cache = dsaidx.IndexCache.allocate(2, bs, dsaidx.FP8, fill=0x11)
    k = bf16_tensor(wl.f32_to_bf16_bits(np.ones((3, 128), np.float32)))
    slots = torch.tensor([0, 2 * bs, 5], dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsaidx.store_keys(cache, k, slots, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5
    pool = cache.pool.cpu().numpy()
    assert np.all(pool[:128] == 0x7E) and np.all(pool[5 * 128:6 * 128] == 0x7E)
    # nothing else written
    mask = np.ones(pool.size, bool)
    mask[:128] = mask[5 * 128:6 * 128] = False
    mask[8192:8196] = mask[8192 + 20:8192 + 24] = False
    assert np.all(pool[mask] == 0x11)


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("mode", [0, 1])
def test_rotated_store_bit_exact(bs, mode):
    # idx_store_keys_rotated against the oracle's rotated store, every byte
    W = wl.make_workload("strot", [1000, 77, 64, 3000], [1, 1, 1, 1], bs=bs, seed=20 + bs + mode,
                         extra_blocks=5)
    k = W.all_keys().copy()
    slots = W.all_slots().copy()
    slots[::13] = -1
    rng = np.random.default_rng(100 + bs + mode)
    scale = (10.0 ** rng.uniform(-30, 30, (k.shape[0], 1))).astype(np.float32)
    kf = wl.bf16_bits_to_f32(k) * scale
    kf[7] = 0.0
    kf[9] = 1.0                       # all-ones row: its energy moves to entry 0
    k = wl.f32_to_bf16_bits(kf)
    cache = dsaidx.IndexCache.allocate(W.num_blocks, bs, mode, fill=0xA5)
    dsaidx.store_keys(cache, bf16_tensor(k), torch.from_numpy(slots).cuda(), rotate=True)
    got = cache.pool.cpu().numpy()
    bb = oracle.block_bytes(mode, W.bs)
    want = np.full(W.num_blocks * bb, 0xA5, np.uint8)
    oracle.store_keys(want, k, slots, W.bs, mode, rotate=True)
    diff = np.nonzero(got != want)[0]
    assert diff.size == 0, "first differing byte %d of %d" % (diff[0], diff.size)


@pytest.mark.parametrize("mode", [0, 1])
def test_rotated_keys_and_queries_score_parity(mode):
    # keys stored rotated, queries rotated by the caller (here with the
    # oracle's rotation, rounded to bf16): decode parity against the oracle on
    # the same rotated operands, and the planted needle still ranks first
    from tests.parity import check_rows, decode_inputs
    W = wl.make_workload("rotdec", [3000, 9000, 129], [1, 1, 1], topk=256, seed=31 + mode)
    B, H, d = W.q.shape
    qr = oracle.f32_to_bf16(oracle.wht_rows(W.q.reshape(B * H, d))).reshape(B, H, d)
    cache = dsaidx.IndexCache.allocate(W.num_blocks, W.bs, mode, fill=0)
    dsaidx.store_keys(cache, bf16_tensor(W.all_keys()), torch.from_numpy(W.all_slots()).cuda(), rotate=True)
    ins = decode_inputs(W)
    ws = dsaidx.new_workspace(dsaidx.workspace_bytes_decode(cache, B, W.max_seq_len, H, W.topk))
    oi = torch.full((B, W.topk), -7, dtype=torch.int32, device="cuda")
    osc = torch.full((B, W.topk), float("nan"), dtype=torch.float32, device="cuda")
    dsaidx.score_topk_decode(cache, bf16_tensor(qr), ins["w"], ins["block_table"], ins["seq_lens"],
                             W.max_seq_len, W.topk, oi, ws, out_score=osc)
    got = {"idx": oi.cpu().numpy(), "score": osc.cpu().numpy()}
    keys = [oracle.rotated_key_rows(W.keys[b], mode) for b in range(B)]
    pos = np.asarray(W.seq_lens, np.int64) - 1
    ref = oracle.score_topk(mode, W.topk, qr, W.w, np.arange(B, dtype=np.int32), pos, keys, full_scores=True)
    check_rows(got, ref, pos + 1, W.topk)
    for b in range(B):
        assert got["idx"][b][0] == W.needle_pos[b]


@pytest.mark.parametrize("rot", [False, True])
@pytest.mark.parametrize("mode", [0, 1])
def test_fp4_roundtrip_store_bit_exact(mode, rot):
    # idx_store_keys_ex with the fp4 round trip (after the rotation when rot)
    # against the oracle's store, every byte; magnitudes spread over blocks
    # and rows, zero blocks, a block whose values sit on e2m1 midpoints
    W = wl.make_workload("stfp4", [1000, 77, 3000], [1, 1, 1], bs=64, seed=40 + mode + 2 * rot,
                         extra_blocks=3)
    k = W.all_keys().copy()
    slots = W.all_slots().copy()
    slots[::11] = -1
    rng = np.random.default_rng(200 + mode + 2 * rot)
    # per-block magnitudes without the rotation; with it one scale per row (the
    # double-precision rotation is exact for rows within 38 binades)
    scale = (10.0 ** rng.uniform(-20, 20, (k.shape[0], 1 if rot else 4))).astype(np.float32)
    scale = scale.repeat(128 if rot else 32, axis=1)
    kf = wl.bf16_bits_to_f32(k) * scale
    kf[5] = 0.0
    kf[6, 32:64] = 0.0
    kf[8, :32] = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4, np.float32) * np.float32(0.5)
    k = wl.f32_to_bf16_bits(kf)
    cache = dsaidx.IndexCache.allocate(W.num_blocks, 64, mode, fill=0x5A)
    dsaidx.store_keys(cache, bf16_tensor(k), torch.from_numpy(slots).cuda(), rotate=rot, fp4=True)
    got = cache.pool.cpu().numpy()
    want = np.full(W.num_blocks * oracle.block_bytes(mode, 64), 0x5A, np.uint8)
    oracle.store_keys(want, k, slots, 64, mode, rotate=rot, fp4=True)
    diff = np.nonzero(got != want)[0]
    assert diff.size == 0, "first differing byte %d of %d" % (diff[0], diff.size)


def test_store_ex_rejects_unknown_flags():
    W = wl.make_workload("stflag", [10], [1], bs=64, seed=3)
    cache = dsaidx.IndexCache.allocate(W.num_blocks, 64, 0, fill=0)
    rc = dsaidx.load().idx_store_keys_ex(cache.handle, bf16_tensor(W.all_keys()).data_ptr(),
                                         torch.from_numpy(W.all_slots()).cuda().data_ptr(), 10, 4, None, None)
    assert rc == 1


@pytest.mark.parametrize("rot", [False, True])
def test_fp4_keys_score_parity(rot):
    # keys stored through the fp4 round trip (fp8 pool), queries rotated by
    # the caller when the keys are: decode parity against the oracle on the
    # same operands
    from tests.parity import check_rows, decode_inputs
    W = wl.make_workload("fp4dec", [3000, 9000, 129], [1, 1, 1], topk=256, seed=51 + rot)
    B, H, d = W.q.shape
    q = oracle.f32_to_bf16(oracle.wht_rows(W.q.reshape(B * H, d))).reshape(B, H, d) if rot else W.q
    cache = dsaidx.IndexCache.allocate(W.num_blocks, W.bs, 0, fill=0)
    dsaidx.store_keys(cache, bf16_tensor(W.all_keys()), torch.from_numpy(W.all_slots()).cuda(), rotate=rot,
                      fp4=True)
    ins = decode_inputs(W)
    ws = dsaidx.new_workspace(dsaidx.workspace_bytes_decode(cache, B, W.max_seq_len, H, W.topk))
    oi = torch.full((B, W.topk), -7, dtype=torch.int32, device="cuda")
    osc = torch.full((B, W.topk), float("nan"), dtype=torch.float32, device="cuda")
    dsaidx.score_topk_decode(cache, bf16_tensor(q), ins["w"], ins["block_table"], ins["seq_lens"],
                             W.max_seq_len, W.topk, oi, ws, out_score=osc)
    got = {"idx": oi.cpu().numpy(), "score": osc.cpu().numpy()}
    keys = [oracle.stored_key_rows(W.keys[b], 0, rotate=rot, fp4=True) for b in range(B)]
    pos = np.asarray(W.seq_lens, np.int64) - 1
    ref = oracle.score_topk(0, W.topk, q, W.w, np.arange(B, dtype=np.int32), pos, keys, full_scores=True)
    check_rows(got, ref, pos + 1, W.topk)


def test_copy_kernel_host_device_round_trip():
    # idx_copy from pinned host memory to the device and back, and device to
    # device, byte for byte
    rng = np.random.default_rng(5)
    h = torch.from_numpy(rng.integers(0, 256, 541184, dtype=np.uint8)).pin_memory()
    d = torch.empty(h.numel(), dtype=torch.uint8, device="cuda")
    d2 = torch.empty_like(d)
    back = torch.empty_like(h).pin_memory()
    dsaidx.copy(d, h)
    dsaidx.copy(d2, d)
    dsaidx.copy(back, d2)
    torch.cuda.synchronize()
    assert torch.equal(back, h)
    assert torch.equal(d.cpu(), h)
