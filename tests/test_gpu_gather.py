"""The gather read (idx_gather_blocks) and the paged-versus-gathered cross-check
of "DeepSeek-V4 index_topk=1024 sparse indexer can't recall verbatim lines"
(ROCm/ATOM issue #1507, section "How it was isolated"): the same cache read
through its block table and read contiguously after a gather must give the
same scores and the same top-k, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_idx_gb300 import dsaidx
from sparse_attention_top_idx_gb300 import workloads as wl
from sparse_attention_top_idx_gb300.host import build_cache
from tests.parity import check_rows, decode_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("mode", [0, 1])
def test_gathered_blocks_equal_the_oracle_pool(bs, mode):
    W = wl.make_workload("gath", [700, 0, 129, 3000], [1] * 4, bs=bs, seed=91 + bs + mode, extra_blocks=4)
    cache = build_cache(W, mode)
    bb = oracle.block_bytes(mode, bs)
    B, mbps = W.block_table.shape
    dst = torch.full((B * mbps * bb,), 0x5A, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsaidx.gather_blocks(cache, torch.from_numpy(W.block_table).cuda(),
                         torch.tensor(W.seq_lens, dtype=torch.int32, device="cuda"), dst, status=st)
    got = dst.cpu().numpy().reshape(B, mbps, bb)
    ref = np.full(W.num_blocks * bb, 0xA5, np.uint8)
    oracle.store_keys(ref, W.all_keys(), W.all_slots(), bs, mode)
    ref = ref.reshape(W.num_blocks, bb)
    assert int(st.item()) == 0
    for b in range(B):
        nb = (W.seq_lens[b] + bs - 1) // bs
        for j in range(mbps):
            if j < nb:
                assert np.array_equal(got[b, j], ref[W.block_table[b][j]]), (b, j)
            else:
                assert np.all(got[b, j] == 0x5A)      # past the sequence: untouched


@pytest.mark.parametrize("mode", [0, 1])
def test_gathered_read_equals_paged_read(mode):
    # decode on the paged pool and on the gathered grid (identity block table):
    # identical indices and identical fp32 scores, one- and two-segment rows
    W = wl.make_workload("gxc", [4500, 70000, 10000], [1] * 3, topk=512, seed=95 + mode)
    cache = build_cache(W, mode)
    B, mbps = W.block_table.shape
    bb = dsaidx.block_bytes(mode, W.bs)
    grid = torch.zeros(B * mbps * bb, dtype=torch.uint8, device="cuda")
    ins = decode_inputs(W)
    dsaidx.gather_blocks(cache, ins["block_table"], ins["seq_lens"], grid)
    gcache = dsaidx.IndexCache(grid, W.bs, mode)
    ident = torch.arange(B * mbps, dtype=torch.int32, device="cuda").view(B, mbps)

    def run(c, bt):
        ws = dsaidx.new_workspace(dsaidx.workspace_bytes_decode(c, B, W.max_seq_len, W.H, W.topk))
        oi = torch.empty((B, W.topk), dtype=torch.int32, device="cuda")
        osc = torch.empty((B, W.topk), dtype=torch.float32, device="cuda")
        dsaidx.score_topk_decode(c, ins["q"], ins["w"], bt, ins["seq_lens"], W.max_seq_len, W.topk, oi, ws,
                                 out_score=osc)
        assert dsaidx.read_device_status(ws) == 0
        return oi.cpu().numpy(), osc.cpu().numpy()

    pi, ps = run(cache, ins["block_table"])
    gi, gs = run(gcache, ident)
    assert np.array_equal(pi, gi)
    assert np.array_equal(ps.view(np.uint32), gs.view(np.uint32))
    # and both are the oracle's
    keys = [oracle.quantize_rows(W.keys[b]) if mode == oracle.FP8 else W.keys[b] for b in range(B)]
    pos = np.asarray(W.seq_lens, np.int64) - 1
    ref = oracle.score_topk(mode, W.topk, W.q, W.w, np.arange(B, dtype=np.int32), pos, keys, full_scores=True)
    check_rows({"idx": gi, "score": gs}, ref, pos + 1, W.topk)
